/*
 * moe.h -- C ABI of libmoe_gb300: the Mixture-of-Experts token path on one
 * NVIDIA GB300 (sm_103a): router top-k, per-expert count and scan, dispatch
 * into expert-major capacity-padded buffers, and top-k weighted combine; the
 * experts between them as a synthetic stand-in or as grouped fp8 / bf16 GEMMs
 * on the tensor cores; fused route + dispatch for decode batches; expert and
 * combine with per-row readiness; a two-stream dual-batch-overlap step and its
 * multi-layer schedule with CUDA-graph capture; and the whole path with host
 * buffers in one call.
 *
 * Pages the operations follow (title, section):
 *   [PMC] "Efficient and portable mixture-of-experts communication"
 *         (Perplexity, 2025-04-02), read in its Indonesian translation
 *         "Komunikasi mixture-of-experts yang efisien dan portabel".
 *   [DBO] "Dual Batch Overlap" (vLLM design documentation).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every buffer pointer is a DEVICE pointer (cudaMalloc / PyTorch CUDA
 *   tensor) on the current device, allocated and owned by the caller, unless a
 *   parameter says "host". The library never allocates, frees or synchronises
 *   inside these calls, which matches [PMC §Portable kernels] (buffers are
 *   sized once and reused across layers) and [PMC §Combine] (the result goes to
 *   an externally allocated tensor).
 * Streams.  `stream` is a cudaStream_t passed as void*; NULL is the legacy
 *   default stream. Work is enqueued asynchronously on it, in argument order.
 * Errors.  Arguments are checked on the host before anything is launched. A
 *   failing call returns a negative moe_status and launches nothing. A launch
 *   failure reported by the CUDA runtime returns MOE_ERR_CUDA. No call aborts.
 * Sizes.  T = num_tokens, H = hidden, E = num_experts, k = top_k,
 *   R = num_ranks, C = capacity, Er = E/R experts per virtual rank.
 *   Limits: 0 <= T <= 2^24, 8 <= H <= 65536 with H % 8 == 0 (H % 128 == 0 for
 *   fp8), 1 <= E <= 1024, 1 <= k <= min(E, 16), 1 <= R <= E with E % R == 0,
 *   1 <= C <= 2^24, and T*k, E*C below 2^31. T == 0 is a valid empty batch:
 *   the call returns MOE_OK after writing the all-zero counts it implies.
 * Alignment.  Row buffers (x, recv, recv_scale, y, out) must be 16-byte
 *   aligned, logits too when E % 4 == 0 (4-byte otherwise); int32/float
 *   arrays 4-byte aligned; the route workspace 16-byte aligned.
 * Layouts (row-major, C order):
 *   logits[T][E] f32; topk_idx[T][k] i32; topk_w[T][k] f32; slot[T][k] i32;
 *   x[T][H] bf16; recv[E][C][H] bf16 or e4m3; recv_scale[E][C][H/128] f32;
 *   recv_src[E][C] i32; y[E][C][H] bf16; out[T][H] bf16.
 *   Expert e belongs to virtual expert-parallel rank e / Er and owns rows
 *   [e*C, (e+1)*C) of recv / y, so [R][Er][C][H] and [E][C][H] are the same
 *   memory: the receive buffer of [PMC §Portable kernels] for every rank at
 *   once, in this one GPU's HBM.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,   /* a size, pointer or alignment check failed       */
    MOE_ERR_UNSUPPORTED = -2,   /* valid request outside what this build supports  */
    MOE_ERR_CUDA = -3,          /* the CUDA runtime reported an error               */
    MOE_ERR_DEVICE_CHECK = -4,  /* a device-side consistency check failed           */
    MOE_ERR_TIMEOUT = -5        /* a bounded device wait gave up (moe_device_status)  */
} moe_status;

typedef enum moe_dispatch_dtype {
    MOE_DTYPE_BF16 = 0,         /* rows are copied as bf16                          */
    MOE_DTYPE_FP8_E4M3_B128 = 1 /* rows are quantised to e4m3, one f32 scale / 128  */
} moe_dispatch_dtype;

/* The problem statement: hidden states of T tokens, their router logits over
 * E experts, top-k, R virtual expert-parallel ranks and a per-expert capacity
 * C ([PMC §Portable kernels]: the maximum number of tokens is fixed, which
 * bounds what each expert can receive). */
typedef struct moe_problem {
    int32_t num_tokens;      /* T */
    int32_t hidden;          /* H */
    int32_t num_experts;     /* E */
    int32_t top_k;           /* k */
    int32_t num_ranks;       /* R */
    int32_t capacity;        /* C */
    int32_t dispatch_dtype;  /* moe_dispatch_dtype */
    int32_t max_blocks;      /* 0: library default grid; > 0: at most this many
                                thread blocks for dispatch / expert / combine and
                                the persistent GEMM and readiness grids, so that
                                kernels on another stream stay co-resident */
    int32_t tokens_per_src_rank; /* tokens each virtual data-parallel source rank
                                contributes: token t comes from source rank
                                t / tokens_per_src_rank, S = max(1, ceil(T /
                                tokens_per_src_rank)) ranks (the last may hold
                                fewer); 0 means one source rank of all T tokens.
                                Used by moe_src_offsets only. */
} moe_problem;

/* Human-readable name of a moe_status value. Never NULL; static storage. */
const char *moe_status_string(int status);

/* Device status of this library on the current device. Kernels that wait
 * on their own asynchronous copies (mbarrier waits on bulk loads) bound every
 * wait; a wait that gives up records it in a status word on the device, drains
 * what it still has in flight and returns, leaving its outputs incomplete.
 * This call synchronises with the device (a blocking copy: keep it out of
 * timed or captured regions), returns MOE_ERR_TIMEOUT if such a wait gave up
 * since the last call, MOE_OK otherwise, and clears the word. */
int moe_device_status(void);

/* Host-only validation of a problem (no CUDA call). Returns MOE_OK or
 * MOE_ERR_INVALID_ARG. */
int moe_validate(const moe_problem *p);

/* Bytes of device workspace moe_route needs for this problem (host-only, no
 * CUDA call); 0 if the problem is invalid. For decode-sized batches (T <= 4096
 * and E * ceil(ceil(T/8) / 16) <= 2048: 1024 tokens at E = 256, 4096 at
 * E <= 64) the workspace holds one byte per (expert, tile of 8 tokens), each
 * expert's row rounded up to 16 bytes: E * 16 * ceil(ceil(T/8) / 16) bytes.
 * Otherwise it holds one 32-bit count per (tile of 32 tokens, expert) and, for
 * large batches (more than 2^22 / E tiles squared), two 32-bit values per
 * (chunk of 32 tiles, expert) for a two-level scan of those counts. Always a
 * multiple of 256 and at least 256. Its contents need no initialisation. */
size_t moe_route_workspace_bytes(const moe_problem *p);

/* Step 1 and 2: router top-k with renormalised softmax weights, then the
 * per-expert histogram, its exclusive scan and every pair's slot.
 *
 *  [PMC §Introduction]: the router gives a probability distribution over the
 *  experts; the top-K experts are chosen and the output is their weighted
 *  average with weights from that distribution. Here, per token t:
 *    topk_idx[t][0..k-1]: the k largest logits, largest first; equal logits go
 *                         to the lower expert index (-0.0 equals +0.0);
 *    topk_w[t][j] = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0)  (fp32).
 *  [PMC §Dispatch]: tokens are counted per destination expert; [PMC §Portable
 *  kernels]: a fixed per-expert bound gives every row a unique address with no
 *  synchronisation between senders. Here:
 *    counts[e]      = number of pairs (t, j) with topk_idx[t][j] == e;
 *    offsets[e]     = sum_{e' < e} counts[e'], offsets[E] = T*k  (E+1 entries);
 *    slot[t][j]     = number of tokens t' < t that chose the same expert, or -1
 *                     when that number is >= C (the pair is dropped);
 *    rank_counts[r] = sum over experts e of rank r of min(counts[e], C);
 *    dropped[0]     = sum_e max(0, counts[e] - C).
 *  Capacity overflow is not an error: it shows in dropped and slot == -1.
 *  Results are deterministic and independent of the launch configuration.
 *  NaN logits give unspecified (but in-range) indices.
 *  workspace: device scratch of at least moe_route_workspace_bytes(p) bytes,
 *  16-byte aligned, not shared with a concurrent call. */
int moe_route(const moe_problem *p, const float *logits,
              int32_t *topk_idx, float *topk_w,
              int32_t *counts, int32_t *offsets, int32_t *slot,
              int32_t *rank_counts, int32_t *dropped,
              void *workspace, size_t workspace_bytes, void *stream);

/* moe_route without a workspace argument, for callers that cannot allocate
 * device memory: code running while a stream is captured into a CUDA graph
 * (cudaMalloc is not allowed during capture), runtimes that forbid device
 * allocation once started, and plugin interfaces that pass a kernel only its
 * inputs and outputs. The paper (the pages cited above) has no counterpart of
 * this call; it computes exactly what moe_route computes, on the same kernels.
 *  Scratch: a 1 MiB array in device memory, defined in the library, which
 *  every GPU that loads the library holds until the process exits. The call
 *  returns MOE_ERR_UNSUPPORTED, launching nothing, when the problem needs more
 *  (moe_route_workspace_bytes(p) > 1 MiB, about E x 4.25 bytes per tile of 32
 *  tokens; for instance more than 30784 tokens at E = 256).
 *  Set-up: the first call in a CUDA context looks up the array's device
 *  address with that context current (cudaGetSymbolAddress); make that first
 *  call before any stream capture on the device. The address is kept per
 *  context: after cudaDeviceReset the re-created context looks it up again on
 *  its first call. Later calls in the same context make no CUDA call other
 *  than the kernel launches and the lock-free lookup of the current device
 *  and context (cudaGetDevice, cuCtxGetCurrent, cuCtxGetId).
 *  Sharing: all calls on a device use the same array, which keeps the last
 *  call's contents (the route kernels overwrite what they read, so nothing
 *  needs clearing). Calls whose executions overlap on the GPU (other streams,
 *  other threads) race on the array: order them on one stream.
 *  Arguments, outputs and errors are otherwise those of moe_route. */
int moe_route_noalloc(const moe_problem *p, const float *logits,
                      int32_t *topk_idx, float *topk_w,
                      int32_t *counts, int32_t *offsets, int32_t *slot,
                      int32_t *rank_counts, int32_t *dropped, void *stream);

/* Step 3: dispatch. [PMC §Dispatch]: rows are placed into one tensor for the
 * downstream grouped GEMM, all tokens of one expert grouped together whatever
 * their source, and each row's origin is stored so that combine can send it
 * back. For every pair with slot[t][j] >= 0 and e = topk_idx[t][j]:
 *   MOE_DTYPE_BF16:          recv[e][slot][:] = x[t][:] (bit copy);
 *   MOE_DTYPE_FP8_E4M3_B128: per block b of 128 elements of x[t]:
 *       scale = amax_b / 448 (fp32 division; 1.0 if amax_b == 0),
 *       recv[e][slot][i] = e4m3(x[t][i] / scale) (round to nearest even,
 *       saturating to +-448), recv_scale[e][slot][b] = scale
 *     ([PMC §Dispatch]: tokens travel with their block scaling factors);
 *   recv_src[e][slot] = t.
 * Rows at slots >= min(counts[e], C) are not written. recv_scale must be NULL
 * for bf16 and non-NULL for fp8. topk_idx and slot are moe_route's outputs. */
int moe_dispatch(const moe_problem *p, const void *x,
                 const int32_t *topk_idx, const int32_t *slot,
                 void *recv, float *recv_scale, int32_t *recv_src, void *stream);

/* Where each source rank's tokens sit inside each expert's rows.
 * [PMC §Dispatch]: the receiver unpacks the tokens into one tensor for the
 * grouped GEMM, all tokens of one expert grouped together across the
 * data-parallel ranks that sent them. Here a token's slot ascends with its
 * index, so the kept rows of expert e are ordered by source rank
 * s(t) = t / tokens_per_src_rank, and
 *   src_offsets[e][s] = number of kept rows of expert e whose token comes from
 *                       a source rank below s,   s = 0 .. S,
 * so rows [src_offsets[e][s], src_offsets[e][s+1]) of expert e came from
 * source rank s, and src_offsets[e][S] = min(counts[e], C).
 * counts and recv_src are moe_route's and moe_dispatch's outputs for the same
 * problem. src_offsets: device i32[E][S+1] (S from tokens_per_src_rank; S = 1
 * when it is 0). One block per expert; a programmatic dependent of the
 * previous kernel. */
int moe_src_offsets(const moe_problem *p, const int32_t *counts, const int32_t *recv_src,
                    int32_t *src_offsets, void *stream);

/* moe_route followed by moe_dispatch in one call, with the same outputs bit
 * for bit, for decode: [PMC §Dispatch] counts tokens per destination inside
 * the dispatch kernel. For at most 1024 tokens, H <= 16384, max_blocks == 0
 * and a decode-sized route (see moe_route_workspace_bytes; every E <= 256 at
 * 1024 tokens), for fp8 or bf16 dispatch, it runs in two launches instead of
 * three: the route's top-k kernel, then one kernel with a block per token
 * that forms the token's slots from the per-tile counts and dispatches its
 * row (launched as a programmatic dependent of the first). Otherwise it calls
 * moe_route and moe_dispatch. workspace: device scratch of at least
 * moe_route_dispatch_workspace_bytes(p) bytes (equal to
 * moe_route_workspace_bytes(p)), 16-byte aligned, contents needing no
 * initialisation, not shared with a concurrent call. */
size_t moe_route_dispatch_workspace_bytes(const moe_problem *p);
int moe_route_dispatch(const moe_problem *p, const float *logits, const void *x,
                       int32_t *topk_idx, float *topk_w,
                       int32_t *counts, int32_t *offsets, int32_t *slot,
                       int32_t *rank_counts, int32_t *dropped,
                       void *recv, float *recv_scale, int32_t *recv_src,
                       void *workspace, size_t workspace_bytes, void *stream);

/* Stand-in for the grouped expert GEMM that [PMC §Dispatch] feeds: on rows
 * r < min(counts[e], C) of every expert,
 *   bf16 recv:  y[e][r] = bf16(x * s[e]);
 *   fp8 recv:   y[e][r] = bf16((e4m3_value * recv_scale) * s[e]);
 * fp32 products, bf16 round to nearest even. Other rows of y are not written.
 * s: device float[E]. recv_scale: NULL for bf16, the dispatch scales for fp8. */
int moe_expert_synthetic(const moe_problem *p, const void *recv, const float *recv_scale,
                         const int32_t *counts, const float *s, void *y, void *stream);

/* Grouped expert GEMM on the fp8 dispatch layout, on the tensor cores: the
 * experts that consume the block-scaled dispatched tokens of [PMC §Dispatch],
 * one H -> H linear map per expert with random weights (no activation):
 *   y[e][r][n] = bf16( sum_b recv_scale[e][r][b] * w_scale[e][n/128][b]
 *                      * sum_{i in block b} recv_q[e][r][i] * w_q[e][n][i] )
 * for r < min(counts[e], C), n < H, blocks b of 128 inputs; other rows of y
 * are not written. Each block's sum runs on the tensor cores in fp32, is
 * multiplied by fl(recv_scale * w_scale) and accumulated with one fp32 FMA per
 * block in ascending b, then rounded to bf16 (nearest even).
 * Layouts (device, row-major): recv_q u8[E][C][H] and recv_scale f32[E][C][H/128]
 * as moe_dispatch writes them; w_q u8[E][H][H] e4m3 codes, output index major
 * (row n holds the H inputs of output n); w_scale f32[E][H/128][H/128]; y bf16
 * [E][C][H]; counts i32[E] as moe_route writes them. recv_q, w_q and y 16-byte
 * aligned. Requires dispatch_dtype == MOE_DTYPE_FP8_E4M3_B128 (else
 * MOE_ERR_UNSUPPORTED); max_blocks caps the persistent grid (one CTA per SM
 * by default). Launched as a programmatic dependent of the previous kernel. */
int moe_expert_gemm_fp8(const moe_problem *p, const void *recv_q, const float *recv_scale,
                        const int32_t *counts, const void *w_q, const float *w_scale,
                        void *y, void *stream);

/* Grouped expert GEMM on the bf16 dispatch layout, on the tensor cores: the
 * same expert stand-in for bf16 rows, one H -> H linear map per expert with
 * random bf16 weights (no activation):
 *   y[e][r][n] = bf16( sum_i recv_x[e][r][i] * w[e][n][i] )
 * for r < min(counts[e], C); other rows of y are not written. The products
 * are exact and summed on the tensor cores in fp32 (tcgen05.mma kind::f16),
 * then rounded to bf16 (nearest even). recv_x bf16 [E][C][H] as moe_dispatch
 * writes it; w bf16 [E][H][H], output index major; y bf16 [E][C][H]; all
 * 16-byte aligned. Requires dispatch_dtype == MOE_DTYPE_BF16 and H % 64 == 0
 * (else MOE_ERR_UNSUPPORTED); max_blocks caps the persistent grid. Launched as
 * a programmatic dependent of the previous kernel. */
int moe_expert_gemm_bf16(const moe_problem *p, const void *recv_x, const int32_t *counts,
                         const void *w, void *y, void *stream);

/* Synthetic expert and combine in one kernel, readiness tracked per expert
 * row instead of per kernel: [PMC §Further Improvements] notes that buffers
 * shared across devices allow synchronisation per token instead of per batch.
 * Every warp first computes its units of y (kept row, segment of 32 x 4
 * sixteen-byte input pieces; the arithmetic of moe_expert_synthetic) and
 * publishes each with a release store of `epoch` into its flag, then combines
 * tokens in order (the arithmetic of moe_combine), each unit once the flags
 * of the row segments it reads hold `epoch`. y and out come out bit for bit
 * as moe_expert_synthetic followed by moe_combine write them.
 * flags: device u32[E*C*segments] (moe_ready_flags_bytes(p) bytes), owned by the
 * caller, zero-filled before first use, not shared with a concurrent call.
 * epoch: nonzero, never repeated since the flags were last zero-filled (an
 * incrementing counter). The grid is launched cooperatively (all blocks
 * resident; not a programmatic dependent); max_blocks caps it (>= 2).
 * A consumer wait that gives up after 100 ms (inputs inconsistent with counts)
 * raises the device status word (moe_device_status: MOE_ERR_TIMEOUT) and that
 * unit of out is not written. */
size_t moe_ready_flags_bytes(const moe_problem *p);
int moe_expert_combine(const moe_problem *p, const void *recv, const float *recv_scale,
                       const int32_t *counts, const float *s, void *y,
                       const int32_t *topk_idx, const float *topk_w, const int32_t *slot,
                       void *out, uint32_t *flags, size_t flags_bytes, uint32_t epoch,
                       void *stream);

/* Step 4: combine. [PMC §Combine]: the expert outputs are read back through
 * the routing table and summed with the router weights into an externally
 * allocated tensor:
 *   out[t] = bf16( sum_j topk_w[t][j] * y[topk_idx[t][j]][slot[t][j]] )
 * accumulated in fp32, one fused multiply-add per j in ascending j, from 0;
 * pairs with slot == -1 are skipped (no renormalisation). */
int moe_combine(const moe_problem *p, const void *y,
                const int32_t *topk_idx, const float *topk_w, const int32_t *slot,
                void *out, void *stream);

/* ---- Dual batch overlap ------------------------------------------------- */

/* Buffers of one micro-batch, each sized for its token count (see dbo_step). */
typedef struct moe_ubatch_bufs {
    int32_t *topk_idx;     /* [Tu][k]   */
    float *topk_w;         /* [Tu][k]   */
    int32_t *counts;       /* [E]       */
    int32_t *offsets;      /* [E+1]     */
    int32_t *slot;         /* [Tu][k]   */
    int32_t *rank_counts;  /* [R]       */
    int32_t *dropped;      /* [1]       */
    void *recv;            /* [E][C][H] bf16 or e4m3 */
    float *recv_scale;     /* [E][C][H/128] for fp8, else NULL */
    int32_t *recv_src;     /* [E][C]    */
    void *y;               /* [E][C][H] bf16 */
    void *workspace;       /* route workspace for Tu tokens */
    size_t workspace_bytes;
} moe_ubatch_bufs;

/* The whole path for one batch whose inputs and output live in HOST memory,
 * in one call (the serving-loop form of the path; the paper has no
 * counterpart: its path starts and ends in device memory). On `stream`, all
 * asynchronous: copy x_host (bf16 [T][H]) into x_dev and logits_host
 * (f32 [T][E]) into logits_dev, then moe_route, moe_dispatch,
 * moe_expert_synthetic and moe_combine into out_dev (bf16 [T][H]), then copy
 * out_dev into out_host. bufs: the device buffers of one batch (as for
 * dbo_step, sized for T tokens); s: device f32[E]. Host buffers should be
 * page-locked, or the copies do not overlap other streams' work. The call
 * returns before the work completes: synchronise `stream` before reading
 * out_host or reusing x_host, logits_host or the device buffers. Two streams
 * with two buffer sets, used alternately, overlap one batch's copies with
 * the neighbouring batch's kernels. Errors: MOE_ERR_INVALID_ARG for any
 * argument one of the four calls would reject, or a null host buffer (when
 * T > 0), checked before the first copy is enqueued, so a rejected call
 * enqueues nothing; MOE_ERR_CUDA if a copy or launch fails. */
int moe_path_host(const moe_problem *p, const void *x_host, const float *logits_host,
                  const float *s, void *x_dev, float *logits_dev,
                  const moe_ubatch_bufs *bufs, void *out_dev, void *out_host, void *stream);

/* Event timing of the overlapped pair of the last dbo_step that recorded it
 * (milliseconds, from CUDA events). overlap_fraction = time both kernels were
 * running / the shorter kernel's duration, in [0, 1]. */
typedef struct moe_dbo_timing {
    float step_ms;              /* first to last event of the step            */
    float dispatch_ub1_ms;      /* dispatch of micro-batch 1 (comm stream)    */
    float combine_ub0_ms;       /* combine of micro-batch 0 (compute stream)  */
    float overlap_ms;           /* time both were running                     */
    float overlap_fraction;
} moe_dbo_timing;

typedef struct moe_dbo_ctx moe_dbo_ctx;   /* owns CUDA events only */

/* Creates a context on the current device (cudaEventCreate only). */
int dbo_create(moe_dbo_ctx **ctx);
/* Destroys a context and its events. NULL is a no-op. */
void dbo_destroy(moe_dbo_ctx *ctx);

/* One dual-batch-overlap step over T = full->num_tokens tokens.
 * [DBO §UBatchRunner]: the batch is split at its midpoint; micro-batch 0 is
 * tokens [0, T/2) and micro-batch 1 is [T/2, T) (floor); a micro-batch with
 * no tokens is run as an empty batch. [DBO §Introduction]: while one
 * micro-batch computes, the other communicates. Here the two micro-batches
 * run the whole path on their own buffers (bufs[0], bufs[1]; recv_src and
 * slot hold micro-batch-local token indices) and the dispatch of micro-batch 1
 * on `comm` overlaps the combine of micro-batch 0 on `compute`:
 *   compute: route(0) route(1) dispatch(0) expert(0) | combine(0) | wait(D1) expert(1) combine(1)
 *   comm:                      wait(route(1), expert(0)) dispatch(1) -> D1
 * `comm` first waits for the work already on `compute`; at return all work of
 * the step is ordered before later work on `compute`. out[T][H] receives both
 * micro-batches' rows in token order and equals two single-shot runs.
 * record_timing != 0 records events for dbo_read_timing. */
int dbo_step(moe_dbo_ctx *ctx, const moe_problem *full,
             const void *x, const float *logits, const float *s,
             const moe_ubatch_bufs *bufs /* [2] */, void *out,
             void *compute_stream, void *comm_stream, int record_timing);

/* Waits for the events of the last step that recorded timing (host
 * synchronisation: call it outside a timed or captured region) and fills *t. */
int dbo_read_timing(moe_dbo_ctx *ctx, moe_dbo_timing *t /* host */);

/* ---- Dual batch overlap over layers ------------------------------------- */

/* Stand-in for the layer compute around the MoE block (the qkv projection,
 * the core attention and out projection, and the shared expert of [DBO
 * §Introduction]'s schedule, whose weights are out of scope):
 *   out[i] = bf16(float(in[i]) * a)   (fp32 product, round to nearest even),
 * over n_elements bf16 values (a multiple of 8; in and out 16-byte aligned,
 * not overlapping), plus busy_fmas (0 .. 2^20) dependent fp32 FMAs of busy
 * work per 8 elements that do not change the output: a tunable compute cost
 * standing in for the GEMMs. */
int moe_layer_stand_in(const void *in, void *out, int64_t n_elements, float a,
                       int32_t busy_fmas, void *stream);

/* Arguments of dbo_layers. Micro-batch u of T = full.num_tokens tokens is
 * rows [0, T/2) (u = 0) or [T/2, T) (u = 1); bufs[u] is sized for T - T/2
 * tokens (as for dbo_step). full.dispatch_dtype must be MOE_DTYPE_BF16. */
typedef struct moe_dbo_layers_args {
    moe_problem full;         /* T = both micro-batches                               */
    int32_t n_layers;         /* L >= 1                                               */
    int32_t busy_fmas;        /* busy work of the A0 and S stand-ins                  */
    float alpha;              /* A0 stand-in: h = bf16(x * alpha)                      */
    float sigma;              /* S stand-in: shared = bf16(h * sigma)                  */
    const void *x;            /* [T][H] bf16: input of layer 0                         */
    const float *logits;      /* [L][T][E] f32: router logits of every layer           */
    const float *s;           /* [E] f32: synthetic expert scales                      */
    moe_ubatch_bufs bufs[2];  /* per micro-batch route / dispatch / expert buffers    */
    void *h;                  /* [T][H] bf16 scratch: A0 output, dispatched rows      */
    void *shared;             /* [T][H] bf16: S output of the last layer             */
    void *out;                /* [T][H] bf16: layer activations; layer L's output    */
    const void *expert_w;     /* NULL: MLP = moe_expert_synthetic with s; else [E][H][H] bf16
                                 weights (output-major, shared by every layer): MLP =
                                 moe_expert_gemm_bf16 (needs H % 64 == 0)               */
    int32_t mlp_max_blocks;   /* with expert_w: at most this many CTAs for the GEMM (0: one
                                 per SM), leaving SMs to the comm-stream kernels         */
} moe_dbo_layers_args;

/* L layers of the [DBO §Introduction] schedule on two streams of one GPU.
 * Per layer l and micro-batch u: A0 (h = bf16(x_u * alpha), x_u the layer's
 * input), A1 (moe_route on logits[l]), D (moe_dispatch of h), MLP
 * (moe_expert_synthetic, or the grouped bf16 GEMM with expert_w), S
 * (shared = bf16(h * sigma)) and C (moe_combine, whose output is the next
 * layer's input). A0, A1, MLP and S run on
 * `compute`, D and C on `comm`, enqueued in the page's order:
 *   D_1 | A0_0 A1_0 | D_0 | MLP_1 | C_1 | S_1 | MLP_0 | C_0 | S_0 | A0_1 A1_1 (next layer)
 * with each receive as an event wait; a prologue runs layer 0's A0_1 A1_1.
 * `comm` first waits for the work already on `compute`; at return every step
 * is ordered before later work on `compute`. With compute == comm the same
 * work runs in the same order on one stream (the no-overlap baseline). No
 * host synchronisation, no allocation: the call can be captured into a CUDA
 * graph (dbo_layers_capture). */
int dbo_layers(moe_dbo_ctx *ctx, const moe_dbo_layers_args *a, void *compute_stream, void *comm_stream);

/* Captures dbo_layers(ctx, a, compute, comm) into a CUDA graph owned by ctx
 * (relaxed stream capture; `compute` must not be the legacy default stream),
 * replacing any graph captured before. Make one eager call with the same
 * shapes first: first calls look up device properties. The graph keeps the
 * pointers of `a`. */
int dbo_layers_capture(moe_dbo_ctx *ctx, const moe_dbo_layers_args *a, void *compute_stream, void *comm_stream);

/* Launches the graph last captured by dbo_layers_capture on `stream`. */
int dbo_graph_launch(moe_dbo_ctx *ctx, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
