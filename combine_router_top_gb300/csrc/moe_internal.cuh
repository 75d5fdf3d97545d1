// moe_internal.cuh -- internal helpers of libmoe_gb300 (not part of the ABI).
//
// Page abbreviations used in this library's comments:
//   [PMC] "Efficient and portable mixture-of-experts communication" (Perplexity blog)
//   [DBO] "Dual Batch Overlap" (vLLM design documentation)
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <initializer_list>
#include <mutex>

#include "moe.h"

namespace moe {

constexpr int kTileTokens = 32;    // tokens per route tile: one 32-bit mask word per expert
constexpr int kChunkTiles = 32;    // route tiles per chunk of the two-level scan of tile counts

// Batches of up to kRouteSmallMaxTokens tokens take the small-batch route: tiles
// of kSmallTileTokens tokens (one warp each, one 256-thread block per tile), and
// the count of every (expert, tile) stored as one byte in an expert-major
// workspace cnt8[E][stride] (a tile holds at most 8 pairs of one expert). The
// counts of all tiles before tile b of expert e are then the first b bytes of
// row e: at most 512 bytes, one 16-byte piece per lane of a warp.
constexpr int kSmallTileTokens = 8;
constexpr int kRouteSmallMaxTokens = 4096;
// 16-byte pieces of the byte counts the totals block reads: E rows of
// ceil(tiles / 16) pieces. The small-batch route runs while that is at most
// 8 pieces per thread of the block (1024 tokens at E = 256, 4096 at E <= 64);
// beyond, one block reading them is slower than the 32-token tiles.
constexpr int kRouteSmallMaxPieces = 8 * 256;
inline bool route_small(long long T, int E) {
    const long long tiles = (T + kSmallTileTokens - 1) / kSmallTileTokens;
    return T <= kRouteSmallMaxTokens && (long long)E * ((tiles + 15) / 16) <= kRouteSmallMaxPieces;
}
// Bytes per expert row of the small-batch workspace: the tile count rounded up to 16.
inline size_t route_small_stride(long long T) {
    const size_t tiles = ((size_t)T + kSmallTileTokens - 1) / kSmallTileTokens;
    return (tiles + 15) & ~(size_t)15;
}

// The route finaliser sums the counts of all earlier tiles directly, about
// n_tiles^2 * E / 2 loads in all; above 2^22 of them (128 tiles at E = 256)
// the two-level scan, two launches more but linear, is faster.
inline bool route_two_level(size_t n_tiles, int E) { return n_tiles * n_tiles * (size_t)E > ((size_t)1 << 22); }
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kMaxHidden = 65536;
constexpr int kMaxTokens = 1 << 24;
constexpr int kMaxCapacity = 1 << 24;
constexpr unsigned kFull = 0xFFFFFFFFu;

// Validated sizes of one call.
struct Dims {
    int T, H, E, k, R, C, dtype, max_blocks;
};

// Host-side checks (moe_abi.cu).
int check_problem(const moe_problem *p, Dims *d);
// Device address of this library's status word on the current device
// (moe_abi.cu); nullptr if it cannot be looked up.
unsigned *device_status_word();

// Bits of the device status word.
constexpr unsigned kStatusWaitGaveUp = 1u;     // a bounded wait on a copy gave up
inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int sm_count();                         // SMs of the current device (cached per context)

// The CUDA context current on the calling thread: its device and its unique
// id (cuCtxGetId). A context created again after cudaDeviceReset gets a new
// id. Returns false if there is no current context or the lookup fails.
struct CtxKey {
    int dev;
    unsigned long long id;
};
bool current_ctx(CtxKey *key);

// A value computed once per CUDA context and read without a lock afterwards.
// Device addresses of this library's __device__ arrays, function attributes
// and occupancy all belong to the context they were obtained in, so a
// context re-created after cudaDeviceReset (or another context on the same
// device) computes its own. `make` returns the value; a value equal to T{}
// (0, nullptr) means failure and is returned without being cached. Records
// are never freed (a reader may still hold one); there is one per context
// seen, chained per device.
template <typename T>
class PerContext {
    static constexpr int kDevices = 64;
    struct Rec {
        unsigned long long id;
        T val;
        const Rec *next;
    };
    std::atomic<const Rec *> head_[kDevices] = {};
    std::mutex mu_;

    const Rec *find(int dev, unsigned long long id) const {
        for (const Rec *r = head_[dev].load(std::memory_order_acquire); r != nullptr; r = r->next)
            if (r->id == id) return r;
        return nullptr;
    }

  public:
    template <typename F>
    T get(F make) {
        CtxKey k;
        if (!current_ctx(&k) || k.dev < 0 || k.dev >= kDevices) return make();
        if (const Rec *r = find(k.dev, k.id)) return r->val;
        std::lock_guard<std::mutex> lock(mu_);
        if (const Rec *r = find(k.dev, k.id)) return r->val;
        const T v = make();
        if (v == T{}) return v;
        head_[k.dev].store(new Rec{k.id, v, head_[k.dev].load(std::memory_order_relaxed)}, std::memory_order_release);
        return v;
    }
};

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) once per
// context; false if the runtime refuses it.
template <typename Kernel>
bool set_smem_once(PerContext<int> &done, Kernel kernel, int bytes) {
    return done.get([&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess ? 1 : 0;
    }) == 1;
}
// The small-batch route's top-k kernel alone (moe_route.cu), for
// 0 < T <= kRouteSmallMaxTokens: indices, weights, each pair's rank within its
// tile of 8 tokens, and the byte counts cnt8[E][route_small_stride(T)].
int launch_route_topk_small(const Dims &d, cudaStream_t st, const float *logits, int32_t *topk_idx, float *topk_w,
                            int32_t *rank, uint8_t *cnt8);
// moe_layer_stand_in with a cap on its grid (moe_layers.cu).
int layer_stand_in(const void *in, void *out, int64_t n_elements, float a, int32_t busy_fmas, int max_blocks,
                   cudaStream_t st);
inline int launch_status(void) {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Thread blocks of `kernel` that fit on the whole GPU at once (occupancy x SMs).
template <typename Kernel>
int resident_blocks(Kernel kernel, int block, size_t smem = 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, smem) != cudaSuccess || n < 1) n = 1;
    return n * sm_count();
}

// resident_blocks, computed once per context into `cache`.
template <typename Kernel>
int resident_blocks_cached(PerContext<int> &cache, Kernel kernel, int block, size_t smem = 0) {
    return cache.get([&] { return resident_blocks(kernel, block, smem); });
}

// Grid of a persistent kernel over `units` work units: one wave of resident
// blocks, or fewer when max_blocks caps it or there is less work.
inline int persistent_grid(long long units, int resident, int max_blocks) {
    long long g = resident;
    if (max_blocks > 0 && max_blocks < g) g = max_blocks;
    if (units < g) g = units;
    return g < 1 ? 1 : (int)g;
}

// Tasks per lane per work unit: the largest of 8, 7, 4, 2, 1 for which units of
// 32*U tasks tile a row of n_tasks exactly (else 4).
inline int lane_tasks(int n_tasks) {
    for (int u : {8, 7, 4, 2, 1})
        if (n_tasks % (32 * u) == 0) return u;
    return 4;
}

// Launches `kernel` on `st` allowing programmatic dependent launch: the grid
// may be scheduled while the previous kernel on the stream finishes. Every
// kernel of this library starts with pdl_wait(), so none touches global memory
// before its predecessor has completed and flushed.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), int grid, int block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// launch_pdl with `smem` bytes of dynamic shared memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl_smem(void (*kernel)(Params...), int grid, int block, size_t smem, cudaStream_t st,
                            Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// ---- device helpers -------------------------------------------------------

// ---- TMA bulk copies and mbarriers -------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of
// 16), completing `bytes` of transaction on the mbarrier.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst_smem)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// Shared -> global bulk copy, tracked by this thread's bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src_smem, unsigned bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src_smem)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed group of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until every committed group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later async-proxy (bulk copy) reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Waits for phase `parity` of the mbarrier, giving up after a bounded number
// of polls (each poll may itself suspend for a short, hardware-defined time).
constexpr unsigned kMbarPollLimit = 1u << 20;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity) {
    const uint32_t a = smem_u32(bar);
    for (unsigned i = 0; i < kMbarPollLimit; ++i) {
        uint32_t done;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done)
                     : "r"(a), "r"(parity)
                     : "memory");
        if (done) return true;
    }
    return false;
}

// Programmatic dependent launch: wait until the previous grid on the stream
// has completed and its memory is visible, then let the next grid launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_launch_dependents();
}

// Exclusive scan of min(counts[e], C) over e into off[0..E] (off[E] = kept rows).
__device__ __forceinline__ void kept_row_offsets(const int32_t *__restrict__ counts, int E, int C, int32_t *off, int32_t *warp_tot) {
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (E + nt - 1) / nt;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int local = 0;
    for (int e = e0; e < e1; ++e) {
        const int c = __ldg(counts + e);
        local += c < C ? c : C;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < (nt >> 5) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += n;
        }
        warp_tot[lane] = v;
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? warp_tot[warp - 1] : 0);
    for (int e = e0; e < e1; ++e) {
        off[e] = run;
        const int c = __ldg(counts + e);
        run += c < C ? c : C;
    }
    if (tid == nt - 1) off[E] = run;
    __syncthreads();
}

// Expert of kept row p: the last e with off[e] <= p (off is non-decreasing).
__device__ __forceinline__ int expert_of_row(const int32_t *off, int E, int p) {
    int lo = 0, hi = E;        // off[lo] <= p < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= p) lo = mid; else hi = mid;
    }
    return lo;
}

// Walks the work units unit0, unit0 + stride, ... of a (row, segment) grid
// with `segs` segments per row, keeping (row, seg) without any division in
// the loop.
struct UnitWalk {
    unsigned row, seg, drow, dseg, segs;
    __device__ __forceinline__ UnitWalk(unsigned unit0, unsigned stride, unsigned segs_)
        : row(unit0 / segs_), seg(unit0 % segs_), drow(stride / segs_), dseg(stride % segs_), segs(segs_) {}
    __device__ __forceinline__ void next() {
        row += drow;
        seg += dseg;
        if (seg >= segs) { seg -= segs; row += 1; }
    }
};

// 16-byte load through the read-only path, not kept in L1 (each row is read
// once). Only for data no kernel writes while this one runs.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w));
}

// bf16 pair in a 32-bit word -> two floats (exact: bf16 is the upper half of a binary32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Elementwise max of |a| and |b| on bf16 pairs (exact: no rounding involved).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    const __nv_bfloat162 r = __hmax2(__habs2(*reinterpret_cast<const __nv_bfloat162 *>(&a)),
                                     __habs2(*reinterpret_cast<const __nv_bfloat162 *>(&b)));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Two floats -> bf16 pair, round to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Two floats -> two e4m3 codes (round to nearest even, saturating to +-448), lo in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
    __nv_fp8x2_storage_t s = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(s);
}

// Block scale of the fp8 dispatch: amax / 448 in fp32 (IEEE division), 1 for
// an all-zero block.
__device__ __forceinline__ float e4m3_block_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// Scales for which quantise16_e4m3 takes the FMA-corrected quotient.
constexpr float kQuotientFastMin = 0x1p-100f, kQuotientFastMax = 0x1p120f;

// The e4m3 codes of 16 bf16 elements of one block (wv: 8 bf16 pairs, lo
// first) with block scale sc: code = e4m3(x / sc) of the IEEE fp32 quotient,
// as four words of four codes. Inside [kQuotientFastMin, kQuotientFastMax]
// (every finite scale of a block whose amax is at least about 2^-91) one
// correctly rounded reciprocal r = 1/sc replaces the 16 divisions: per
// element q0 = x*r, the remainder x - sc*q0 by FMA and one correction
// q0 + rem*r (Markstein's FMA-based division: P. Markstein, IBM J. Res. Dev.
// 34(1), 1990). That q can be one
// fp32 ulp off the IEEE quotient, but never across an e4m3 rounding boundary:
// an exhaustive host check over every bf16 amax whose scale is in the range
// and every bf16 x with |x| <= amax finds the same code in every case. A zero
// remainder keeps q0, which carries the sign of x (so -0 stays -0). Outside
// the range (tiny blocks, an infinite amax, NaN) the IEEE division is used.
__device__ __forceinline__ float fma_corrected_quotient(float x, float sc, float r) {
    const float q0 = __fmul_rn(x, r);
    const float rem = __fmaf_rn(-q0, sc, x);
    return rem == 0.0f ? q0 : __fmaf_rn(rem, r, q0);
}
__device__ __forceinline__ void quantise16_e4m3(const uint32_t wv[8], float sc, uint32_t q[4]) {
    if (sc >= kQuotientFastMin && sc <= kQuotientFastMax) {
        const float r = __frcp_rn(sc);
#pragma unroll
        for (int h = 0; h < 4; ++h)
            q[h] = pack_e4m3x2(fma_corrected_quotient(bf16_lo(wv[2 * h]), sc, r),
                               fma_corrected_quotient(bf16_hi(wv[2 * h]), sc, r)) |
                   (pack_e4m3x2(fma_corrected_quotient(bf16_lo(wv[2 * h + 1]), sc, r),
                                fma_corrected_quotient(bf16_hi(wv[2 * h + 1]), sc, r)) << 16);
    } else {
#pragma unroll
        for (int h = 0; h < 4; ++h)
            q[h] = pack_e4m3x2(__fdiv_rn(bf16_lo(wv[2 * h]), sc), __fdiv_rn(bf16_hi(wv[2 * h]), sc)) |
                   (pack_e4m3x2(__fdiv_rn(bf16_lo(wv[2 * h + 1]), sc), __fdiv_rn(bf16_hi(wv[2 * h + 1]), sc)) << 16);
    }
}

// Total order on fp32 logits as unsigned keys: larger logit -> larger key,
// -0.0 folded onto +0.0, NaN mapped to 1 (below every number), 0 reserved
// for "no candidate".
// ---- small-batch route helpers ------------------------------------------------

// acc + the sum of the bytes of v (the 16 bytes at row offsets first .. first+15)
// whose row offset is below limit, by shifts and masks.
__device__ __forceinline__ unsigned add_bytes_below(uint4 v, int first, int limit, unsigned acc) {
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int n = limit - (first + 4 * i);                  // valid bytes of word i
        const unsigned m = n >= 4 ? 0xFFFFFFFFu : (n <= 0 ? 0u : (1u << (8 * n)) - 1u);
        const unsigned x = w[i] & m;
        const unsigned h = (x & 0x00FF00FFu) + ((x >> 8) & 0x00FF00FFu);    // two 16-bit partial sums
        acc += (h & 0xFFFFu) + (h >> 16);
    }
    return acc;
}

// Sum of v over the 32 lanes of a warp, by a butterfly of shuffles; every lane
// returns it. The byte sums of the small-batch route are reduced this way: in a
// probe on sm_103a (nvcc 13.0) the same sums reduced with redux.sync
// (__reduce_add_sync) came out wrong, while each lane's value was right.
__device__ __forceinline__ unsigned warp_sum(unsigned v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Sum of bytes [0, limit) of a 16-byte aligned row, limit <= 512, over one warp:
// lane l reads bytes [16 l, 16 l + 16). Every lane returns the sum.
__device__ __forceinline__ int warp_row_prefix(const uint8_t *__restrict__ row, int limit) {
    const int c = (threadIdx.x & 31) * 16;
    unsigned acc = 0;
    if (c < limit) acc = add_bytes_below(__ldcg(reinterpret_cast<const uint4 *>(row + c)), c, limit, 0u);
    return (int)warp_sum(acc);
}

// One block (any multiple of 32 threads, at most 1024) turns the byte counts
// cnt8[E][stride] of n_tiles tiles into the totals: counts[e], offsets[0..E]
// (exclusive scan), rank_counts[r] (kept rows of the experts of rank r) and
// dropped. tot: E ints, wsum: 32 ints, both shared. Each thread issues up to
// BATCH loads before it uses any.
template <int BATCH>
__device__ inline void small_route_totals(const uint8_t *__restrict__ cnt8, size_t stride, int n_tiles, int E, int R,
                                          int C, int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                          int32_t *__restrict__ rank_counts, int32_t *__restrict__ dropped, int *tot,
                                          int *wsum) {
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // every (expert, 16-byte piece) pair is one load, spread over all threads
    // (so that a few experts with long rows still use the whole block); the
    // pieces of a row meet in an integer sum, whose order does not matter
    const int pieces = (n_tiles + 15) / 16;
    for (int e = tid; e < E; e += nt) tot[e] = 0;
    __syncthreads();
    const int pairs = E * pieces;
    for (int base = 0; base < pairs; base += BATCH * nt) {  // one pass while pairs <= BATCH * threads
        uint4 v[BATCH];
        int ex[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {                  // all loads issued before any is used
            const int i = base + j * nt + tid;
            ex[j] = -1;
            if (i < pairs) {
                ex[j] = i / pieces;
                v[j] = __ldcg(reinterpret_cast<const uint4 *>(cnt8 + (size_t)ex[j] * stride +
                                                              (size_t)(i - ex[j] * pieces) * 16));
            }
        }
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            if (ex[j] < 0) continue;
            const int c = (base + j * nt + tid - ex[j] * pieces) * 16;
            const unsigned sum = add_bytes_below(v[j], c, n_tiles, 0u);
            if (sum != 0) atomicAdd(&tot[ex[j]], (int)sum);
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += nt) counts[e] = tot[e];
    // exclusive scan of tot over e: each thread a run of consecutive experts
    const int per = (E + nt - 1) / nt;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int local = 0, lost = 0;
    for (int e = e0; e < e1; ++e) {
        local += tot[e];
        lost += tot[e] > C ? tot[e] - C : 0;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    lost = (int)warp_sum((unsigned)lost);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < (nt >> 5) ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += n;
        }
        wsum[lane] = v;
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? wsum[warp - 1] : 0);
    for (int e = e0; e < e1; ++e) {
        offsets[e] = run;
        run += tot[e];
    }
    if (tid == nt - 1) offsets[E] = run;
    const int per_rank = E / R;
    for (int r = tid; r < R; r += nt) {
        int kept = 0;
        for (int e = r * per_rank; e < (r + 1) * per_rank; ++e) kept += tot[e] < C ? tot[e] : C;
        rank_counts[r] = kept;
    }
    __syncthreads();                           // every read of wsum above is done
    if (lane == 0) wsum[warp] = lost;
    __syncthreads();
    if (tid == 0) {
        int d = 0;
        for (int w = 0; w < (nt >> 5); ++w) d += wsum[w];
        *dropped = d;
    }
}

__device__ __forceinline__ uint32_t logit_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f != f) return 1u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

}  // namespace moe
