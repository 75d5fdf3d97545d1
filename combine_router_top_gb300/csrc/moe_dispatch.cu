// moe_dispatch.cu -- step 3: scatter token rows into the expert-major,
// capacity-padded receive buffer recv[E][C][H] (virtual EP rank r owns experts
// [r*E/R, (r+1)*E/R), i.e. a contiguous range of rows), as bf16 or as e4m3
// with one fp32 scale per 128 elements.
//
// [PMC §Dispatch]: the sender packs each token's activations, scale factors
// and indices and sends the same packed token to every expert it was routed
// to; the receiver groups all tokens of one expert into the grouped-GEMM
// input and keeps each row's origin. On one GPU the "send" is a store into
// the expert's rows of this HBM, at the address the slot fixes; no counts have
// to be awaited because moe_route already produced them.
//
// Kernels, chosen by moe_dispatch from the dtype and H:
//   fp8, H % 1024 == 0: dispatch_fp8_seg, one 64-thread CTA per (token,
//     1024-element segment), loads and stores straight from registers;
//   bf16, rows of at most 32 KB: dispatch_bf16_tma, one warp per token, one
//     bulk copy in and one bulk copy out per destination;
//   otherwise the persistent register kernels below: one wave of resident
//     thread blocks, every warp walking its own work units (token, segment of
//     its row) with no block-wide barrier, the next unit's routing and row
//     data loaded before the current unit is stored.
// In all of them lanes j < k hold the token's destination rows (ascending j)
// and recv_src is written once per kept pair. moe_route_dispatch fuses the
// slot computation of moe_route into the fp8 and bf16 dispatch for decode
// batches (route_dispatch_kernel, at the end of this file).
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBlock = 256;             // 8 warps; every warp walks its own work units
constexpr int kWarps = kBlock / 32;

// Lane j < k holds choice j of the token: its destination row e*C + slot
// (< 2^31), or -1 when the pair was dropped.
__device__ __forceinline__ int load_dest(unsigned t, int k, int C, const int32_t *__restrict__ topk_idx,
                                         const int32_t *__restrict__ slot) {
    const int lane = threadIdx.x & 31;
    if (lane >= k) return -1;
    const int s = __ldg(slot + (size_t)t * k + lane);
    const int e = __ldg(topk_idx + (size_t)t * k + lane);
    return s >= 0 ? e * C + s : -1;
}

template <int U>
__device__ __forceinline__ void load_fp8_tasks(const uint4 *__restrict__ x, int H, unsigned n_tasks,
                                               const UnitWalk &at, int lane, uint4 (&v)[2 * U]) {
    const uint4 *src = x + (size_t)at.row * (H / 8) + 2 * ((size_t)at.seg * 32 * U + lane);
#pragma unroll
    for (int i = 0; i < U; ++i) {
        if (at.seg * 32 * U + 32 * i + lane < n_tasks) {
            v[2 * i] = ld_stream_v4(src + 64 * i);
            v[2 * i + 1] = ld_stream_v4(src + 64 * i + 1);
        } else {
            v[2 * i] = v[2 * i + 1] = make_uint4(0, 0, 0, 0);
        }
    }
}

template <int U>
__device__ __forceinline__ void load_bf16_chunks(const uint4 *__restrict__ x, int H8, const UnitWalk &at, int lane,
                                                 uint4 (&v)[U]) {
    const uint4 *src = x + (size_t)at.row * H8 + (size_t)at.seg * 32 * U + lane;
#pragma unroll
    for (int i = 0; i < U; ++i)
        if (at.seg * 32 * U + 32 * i + lane < (unsigned)H8) v[i] = ld_stream_v4(src + 32 * i);
}

// bf16: a unit is (token, 32*U consecutive 16-byte chunks); lane l owns
// chunks 32*(U*seg + i) + l, i < U.
template <int U>
__global__ void __launch_bounds__(kBlock)
dispatch_bf16_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                     const int32_t *__restrict__ slot, uint4 *__restrict__ recv,
                     int32_t *__restrict__ recv_src, int T, int H8, int k, int C, int segs) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    UnitWalk w(blockIdx.x * kWarps + (threadIdx.x >> 5), gridDim.x * kWarps, segs);
    if (w.row >= (unsigned)T) return;                                  // warp-uniform
    int dest = load_dest(w.row, k, C, topk_idx, slot);
    uint4 a[U];
    load_bf16_chunks<U>(x, H8, w, lane, a);
    for (;;) {
        UnitWalk nw = w;
        nw.next();
        const bool more = nw.row < (unsigned)T;
        int ndest = -1;
        uint4 b[U];
        if (more) {
            ndest = load_dest(nw.row, k, C, topk_idx, slot);
            load_bf16_chunks<U>(x, H8, nw, lane, b);
        }
        if (w.seg == 0 && dest >= 0) recv_src[dest] = (int32_t)w.row;
        const unsigned c0 = w.seg * 32 * U + lane;
        unsigned rem = __ballot_sync(kFull, dest >= 0);
        while (rem) {                                                  // warp-uniform
            const int src = __ffs(rem) - 1;
            rem &= rem - 1;
            uint4 *dst = recv + (size_t)__shfl_sync(kFull, dest, src) * H8 + c0;
#pragma unroll
            for (int i = 0; i < U; ++i)
                if (c0 + 32 * i < (unsigned)H8) st_v4(dst + 32 * i, a[i]);
        }
        if (!more) break;
        w = nw;
        dest = ndest;
#pragma unroll
        for (int i = 0; i < U; ++i) a[i] = b[i];
    }
}

// fp8: a task is 16 consecutive elements (32 bytes of bf16 in, 16 bytes of
// e4m3 out); a unit is (token, 32*U tasks); lane l owns tasks
// 32*(U*seg + i) + l, i < U. The 8 lanes of one 128-element block agree on
// its amax with 3 shuffles; scale = amax/448 (1 for an all-zero block);
// codes are e4m3(x / scale), round to nearest even, saturating.
template <int U>
__global__ void __launch_bounds__(kBlock)
dispatch_fp8_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                    const int32_t *__restrict__ slot, uint4 *__restrict__ recv_q,
                    float *__restrict__ recv_scale, int32_t *__restrict__ recv_src, int T, int H,
                    int k, int C, int segs) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const unsigned n_tasks = H / 16, nb = H / 128;
    UnitWalk w(blockIdx.x * kWarps + (threadIdx.x >> 5), gridDim.x * kWarps, segs);
    if (w.row >= (unsigned)T) return;                                  // warp-uniform
    int dest = load_dest(w.row, k, C, topk_idx, slot);
    uint4 a[2 * U];
    load_fp8_tasks<U>(x, H, n_tasks, w, lane, a);
    for (;;) {
        UnitWalk nw = w;
        nw.next();
        const bool more = nw.row < (unsigned)T;
        int ndest = -1;
        uint4 b[2 * U];
        if (more) {
            ndest = load_dest(nw.row, k, C, topk_idx, slot);
            load_fp8_tasks<U>(x, H, n_tasks, nw, lane, b);
        }
        uint4 qv[U];
        float scale[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const uint32_t wv[8] = {a[2 * i].x, a[2 * i].y, a[2 * i].z, a[2 * i].w,
                                    a[2 * i + 1].x, a[2 * i + 1].y, a[2 * i + 1].z, a[2 * i + 1].w};
            // |x| max of the 16 values on packed bf16 pairs (exact), then over the 8 lanes
            uint32_t m = 0;
#pragma unroll
            for (int h = 0; h < 8; ++h) m = bf16x2_absmax(m, wv[h]);
            float amax = fmaxf(bf16_lo(m), bf16_hi(m));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
            const float sc = e4m3_block_scale(amax);
            uint32_t q[4];
            quantise16_e4m3(wv, sc, q);
            qv[i] = make_uint4(q[0], q[1], q[2], q[3]);
            scale[i] = sc;
        }
        if (w.seg == 0 && dest >= 0) recv_src[dest] = (int32_t)w.row;
        const unsigned task0 = w.seg * 32 * U + lane;
        unsigned rem = __ballot_sync(kFull, dest >= 0);
        while (rem) {                                                  // warp-uniform
            const int src = __ffs(rem) - 1;
            rem &= rem - 1;
            const size_t row = (size_t)__shfl_sync(kFull, dest, src);
            uint4 *dq = recv_q + row * n_tasks + task0;
            float *ds = recv_scale + row * nb + (task0 >> 3);
#pragma unroll
            for (int i = 0; i < U; ++i) {
                if (task0 + 32 * i < n_tasks) {
                    st_v4(dq + 32 * i, qv[i]);
                    if ((lane & 7) == 0) ds[4 * i] = scale[i];
                }
            }
        }
        if (!more) break;
        w = nw;
        dest = ndest;
#pragma unroll
        for (int i = 0; i < 2 * U; ++i) a[i] = b[i];
    }
}

// ---- segment (fp8) and bulk-copy (bf16) dispatch ------------------------------
//
// fp8: a CTA of 64 threads takes a unit (token, 1024-element segment): each
// thread loads its 16 elements with two 16-byte loads (2 KB, coalesced
// across the CTA), quantises them in registers, and for every kept
// destination the CTA writes the 1 KB of codes as one coalesced pass of
// 16-byte stores and the 8 scales as 4-byte stores. bf16: a warp takes a
// token: one bulk copy of the row in, one bulk store per destination out
// (each lane j < k stores its own destination), no per-element instruction.
// Both loop grid-stride over their units when max_blocks caps the grid.

constexpr int kFp8Seg = 1024;                    // fp8 unit: elements
constexpr int kFp8SegThreads = kFp8Seg / 16;     // one 16-element task per thread
constexpr int kTmaBf16MaxRowBytes = 32768;       // bf16 rows staged whole (H <= 16384)

__global__ void __launch_bounds__(kFp8SegThreads, 32)     // 32 CTAs (2048 threads) resident per SM
dispatch_fp8_seg_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ topk_idx,
                        const int32_t *__restrict__ slot, uint8_t *__restrict__ recv_q,
                        float *__restrict__ recv_scale, int32_t *__restrict__ recv_src, int T, int H, int k,
                        int C) {
    __shared__ __align__(16) float ss[kFp8Seg / 128];
    __shared__ int s_row[kMaxTopK];
    __shared__ int s_n;
    pdl_enter();
    const int tid = threadIdx.x, lane = tid & 31;
    const int segs = H / kFp8Seg, nb = H / 128;
    // T * segs <= 2^24 * 64 = 2^30: unit indices and their split stay in 32 bits
    const unsigned units = (unsigned)T * (unsigned)segs;
    for (unsigned u = blockIdx.x; u < units; u += gridDim.x) {
        const unsigned t32 = u / (unsigned)segs;
        const int t = (int)t32, seg = (int)(u - t32 * (unsigned)segs);
        // the 16 elements of task tid: two 16-byte loads, coalesced across the CTA
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H + (size_t)seg * kFp8Seg) + 2 * tid;
        const uint4 a = ld_stream_v4(src), c = ld_stream_v4(src + 1);
        if (tid < 32) {
            const int dest = load_dest(t, k, C, topk_idx, slot);
            const unsigned kept = __ballot_sync(kFull, dest >= 0);
            if (dest >= 0) {
                s_row[__popc(kept & ((1u << lane) - 1u))] = dest;
                if (seg == 0) recv_src[dest] = t;
            }
            if (lane == 0) s_n = __popc(kept);
        }
        // quantise the 16 elements (lanes 8g .. 8g+7 share a 128-element block)
        const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        uint32_t m = 0;
#pragma unroll
        for (int h = 0; h < 8; ++h) m = bf16x2_absmax(m, wv[h]);
        float amax = fmaxf(bf16_lo(m), bf16_hi(m));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
        const float sc = e4m3_block_scale(amax);
        uint32_t q[4];
        quantise16_e4m3(wv, sc, q);
        if ((tid & 7) == 0) ss[tid >> 3] = sc;
        __syncthreads();
        // every thread stores its 16 codes to each kept destination (the CTA
        // writes each destination's segment of codes in one coalesced pass),
        // and thread kSegBlocks*j + b the scale of block b to destination j
        const int nd = s_n;
        const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
        for (int j = 0; j < nd; ++j)
            st_v4(recv_q + (size_t)s_row[j] * H + (size_t)seg * kFp8Seg + (size_t)tid * 16, qv);
        constexpr int kSegBlocks = kFp8Seg / 128;            // scales per segment
        for (int i = tid; i < nd * kSegBlocks; i += kFp8SegThreads)
            recv_scale[(size_t)s_row[i / kSegBlocks] * nb + (size_t)seg * kSegBlocks + (i % kSegBlocks)] =
                ss[i % kSegBlocks];
        __syncthreads();                     // ss and s_row are rewritten by the next unit
    }
}

__global__ void __launch_bounds__(32)
dispatch_bf16_tma_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ topk_idx,
                         const int32_t *__restrict__ slot, uint16_t *__restrict__ recv,
                         int32_t *__restrict__ recv_src, int T, int H, int k, int C, unsigned *status) {
    extern __shared__ __align__(128) unsigned char rowbuf[];
    __shared__ __align__(8) uint64_t bar;
    pdl_enter();
    const int lane = threadIdx.x;
    const unsigned bytes = (unsigned)H * 2u;
    if (lane == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    unsigned phase = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, phase ^= 1u) {
        if (lane == 0) {
            mbar_expect_tx(&bar, bytes);
            bulk_g2s(rowbuf, x + (size_t)t * H, bytes, &bar);
        }
        const int dest = load_dest(t, k, C, topk_idx, slot);
        if (dest >= 0) recv_src[dest] = t;
        const bool ok = mbar_wait_bounded(&bar, phase);
        if (!__all_sync(kFull, ok)) {
            if (lane == 0) {
                atomicOr(status, kStatusWaitGaveUp);
                mbar_wait_bounded(&bar, phase);
            }
            bulk_wait_all();
            return;
        }
        if (dest >= 0) {                     // lane j stores the row to its own destination
            bulk_s2g(recv + (size_t)dest * H, rowbuf, bytes);
            bulk_commit();
            bulk_wait_read_all();
        }
        __syncwarp();
    }
    bulk_wait_all();                         // every store complete before the grid ends
}

// ---- fused route finalisation + dispatch, for decode-sized batches -----------
//
// The small-batch top-k kernel of moe_route leaves, per pair, its rank within
// its tile of 8 tokens (in slot[]) and, per (expert, tile), the tile's count as
// one byte of cnt8[E][stride]. Here one block per token t stages t's bf16 row
// in shared memory (one bulk copy, issued before the wait on the top-k kernel:
// x is an input of the call, final when this grid starts), forms the slots of
// t's k choices while the copy is in flight (slot_j = rank_j + the first
// t/8 bytes of row e_j, one warp per choice), writes slot[] and recv_src,
// then writes the row to each kept destination: for an fp8 dispatch each
// thread stores the 16 codes it has just quantised (16-byte stores, coalesced
// across the block), for a bf16 one the staged row leaves by one bulk store
// per destination. Block 0 forms counts, offsets, rank_counts and dropped
// from the byte counts.
constexpr int kFusedMaxTokens = 1024;          // decode-sized batches
constexpr int kFusedThreads = 256;             // two quantise passes at H 7168; 128, 384 and 512 measured no faster
constexpr int kFusedMaxHidden = 16384;         // staged bf16 row: 2 * H bytes of shared memory
static_assert(kFusedMaxTokens <= kRouteSmallMaxTokens, "the fused path runs on the small-batch top-k kernel");

constexpr size_t fused_smem_bytes(int H, int E) {
    return 2 * (size_t)H > 4 * (size_t)E ? 2 * (size_t)H : 4 * (size_t)E;
}

// FP8: quantise the staged row and store codes and scales; bf16: store the
// staged row itself to each kept destination.
template <bool FP8>
__global__ void __launch_bounds__(kFusedThreads, 6)     // 6 blocks (40 registers a thread) per SM, as before the byte-count totals
route_dispatch_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ topk_idx,
                          const uint8_t *__restrict__ cnt8, int stride,
                          int32_t *__restrict__ slot, uint8_t *__restrict__ recv_q, float *__restrict__ recv_scale,
                          int32_t *__restrict__ recv_src, int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                          int32_t *__restrict__ rank_counts, int32_t *__restrict__ dropped, int H, int E, int k,
                          int C, int R, int n_tiles, unsigned *status) {
    // the bf16 row (2H bytes); block 0: the E totals
    extern __shared__ __align__(128) uint4 fused_smem[];
    __shared__ float ss[kFusedMaxHidden / 128];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_base[kMaxTopK];
    __shared__ int s_row[kMaxTopK];
    __shared__ int s_wsum[32];
    __shared__ int s_n;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0) {          // the totals block: first, so that it is no tail of the grid
        pdl_enter();
        // (not on the critical path: it runs beside the token blocks; 4 loads a
        // thread in flight keep it within the 40 registers of the token blocks)
        small_route_totals<4>(cnt8, (size_t)stride, n_tiles, E, R, C, counts, offsets, rank_counts, dropped,
                           reinterpret_cast<int *>(fused_smem), s_wsum);
        return;
    }
    const int t = blockIdx.x - 1;
    const int nb = H / 128, tasks = H / 16;
    uint4 *xs = fused_smem;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_expect_tx(&bar, (uint32_t)H * 2);
        bulk_g2s(xs, x + (size_t)t * H, (uint32_t)H * 2, &bar);
    }
    pdl_wait();                 // top-k kernel complete from here on; dependents launch at the end
    // slot of each choice j: its rank in t's tile (in slot[]) + the pairs of e_j
    // in the tiles before t's tile, the first t/8 bytes of row e_j (warp j % 8)
    const int tile = t / kSmallTileTokens;
    for (int j = warp; j < k; j += kFusedThreads / 32) {
        const int ej = __ldg(topk_idx + (size_t)t * k + j);
        const int pre = warp_row_prefix(cnt8 + (size_t)ej * stride, tile);
        if (lane == 0) s_base[j] = pre;
    }
    const int e = lane < k ? __ldg(topk_idx + (size_t)t * k + lane) : 0;
    const int my_rank = (tid < k) ? slot[(size_t)t * k + tid] : 0;
    __syncthreads();
    if (tid < 32) {
        int dest = -1;
        if (lane < k) {
            const int base = s_base[lane] + my_rank;
            const int sl = base < C ? base : -1;
            slot[(size_t)t * k + lane] = sl;
            if (sl >= 0) dest = e * C + sl;
        }
        const unsigned kept = __ballot_sync(kFull, dest >= 0);
        if (dest >= 0) {
            s_row[__popc(kept & ((1u << lane) - 1u))] = dest;
            recv_src[dest] = t;
        }
        if (lane == 0) s_n = __popc(kept);
    }
    const bool ok = mbar_wait_bounded(&bar, 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            atomicOr(status, kStatusWaitGaveUp);
            mbar_wait_bounded(&bar, 0);
        }
        return;
    }
    if constexpr (!FP8) {
        // bf16: the staged row goes out as it is (recv_q holds bf16 rows here)
        pdl_launch_dependents();
        if (tid == 0) {
            const int nd = s_n;
            for (int j = 0; j < nd; ++j)
                bulk_s2g(recv_q + (size_t)s_row[j] * H * 2, xs, (uint32_t)H * 2);
            bulk_commit();
            bulk_wait_all();
        }
    } else {
        // 16 elements per task; the 8 tasks of a 128-element block sit in 8
        // neighbouring lanes of one pass (the stride is a multiple of 8 and
        // tasks % 8 == 0), so a pass is active or idle for a whole block
        const int nd = s_n;
        for (int pass = 0; pass < tasks; pass += kFusedThreads) {
            const int task = pass + tid;
            const bool on = task < tasks;
            uint32_t wv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (on) {
                const uint4 a = xs[2 * task], c = xs[2 * task + 1];
                wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
                wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
            }
            uint32_t m = 0;
    #pragma unroll
            for (int h = 0; h < 8; ++h) m = bf16x2_absmax(m, wv[h]);
            float amax = fmaxf(bf16_lo(m), bf16_hi(m));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
            if (on) {
                const float sc = e4m3_block_scale(amax);
                uint32_t q[4];
                quantise16_e4m3(wv, sc, q);
                const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
                for (int j = 0; j < nd; ++j) st_v4(recv_q + (size_t)s_row[j] * H + (size_t)task * 16, qv);
                if ((task & 7) == 0) ss[task >> 3] = sc;
            }
        }
        __syncthreads();
        for (int i = tid; i < nd * nb; i += kFusedThreads) {
            const int j = i / nb, blk = i - j * nb;
            recv_scale[(size_t)s_row[j] * nb + blk] = ss[blk];
        }
        pdl_launch_dependents();
    }
}

template <int U>
int launch_fp8(const Dims &d, cudaStream_t st, const void *x, const int32_t *idx, const int32_t *slot, void *recv,
               float *scale, int32_t *src) {
    static PerContext<int> resident_cache;
    const int resident = resident_blocks_cached(resident_cache, dispatch_fp8_kernel<U>, kBlock);
    const int n_tasks = d.H / 16;
    const int segs = (n_tasks + 32 * U - 1) / (32 * U);
    const long long units = (long long)d.T * segs;
    if (units >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    const int grid = persistent_grid((units + kWarps - 1) / kWarps, resident, d.max_blocks);
    if (launch_pdl(dispatch_fp8_kernel<U>, grid, kBlock, st, static_cast<const uint4 *>(x), idx, slot,
                   static_cast<uint4 *>(recv), scale, src, d.T, d.H, d.k, d.C, segs) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

template <int U>
int launch_bf16(const Dims &d, cudaStream_t st, const void *x, const int32_t *idx, const int32_t *slot, void *recv,
                int32_t *src) {
    static PerContext<int> resident_cache;
    const int resident = resident_blocks_cached(resident_cache, dispatch_bf16_kernel<U>, kBlock);
    const int H8 = d.H / 8;
    const int segs = (H8 + 32 * U - 1) / (32 * U);
    const long long units = (long long)d.T * segs;
    if (units >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    const int grid = persistent_grid((units + kWarps - 1) / kWarps, resident, d.max_blocks);
    if (launch_pdl(dispatch_bf16_kernel<U>, grid, kBlock, st, static_cast<const uint4 *>(x), idx, slot,
                   static_cast<uint4 *>(recv), src, d.T, H8, d.k, d.C, segs) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_dispatch(const moe_problem *p, const void *x, const int32_t *topk_idx,
                            const int32_t *slot, void *recv, float *recv_scale, int32_t *recv_src,
                            void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    const bool fp8 = d.dtype == MOE_DTYPE_FP8_E4M3_B128;
    if (fp8 != (recv_scale != nullptr)) return MOE_ERR_INVALID_ARG;
    if (d.T == 0) return MOE_OK;
    if (!x || !topk_idx || !slot || !recv || !recv_src) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(topk_idx, 4) || !aligned(slot, 4) ||
        !aligned(recv_src, 4) || (fp8 && !aligned(recv_scale, 16)))
        return MOE_ERR_INVALID_ARG;

    cudaStream_t st = as_stream(stream);
    unsigned *status = device_status_word();
    if (status == nullptr) return MOE_ERR_CUDA;
    if (fp8 && d.H % kFp8Seg == 0) {
        static PerContext<int> resident_cache;
        const int resident = resident_blocks_cached(resident_cache, dispatch_fp8_seg_kernel, kFp8SegThreads);
        const long long units = (long long)d.T * (d.H / kFp8Seg);
        const int grid = d.max_blocks > 0 ? persistent_grid(units, resident, d.max_blocks)
                                          : (int)std::min<long long>(units, 1LL << 30);
        if (launch_pdl(dispatch_fp8_seg_kernel, grid, kFp8SegThreads, st, static_cast<const uint16_t *>(x), topk_idx,
                       slot, static_cast<uint8_t *>(recv), recv_scale, recv_src, d.T, d.H, d.k, d.C) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (!fp8 && d.H * 2 <= kTmaBf16MaxRowBytes) {
        const size_t smem = (size_t)d.H * 2;
        const int grid = d.max_blocks > 0 ? std::min(d.T, d.max_blocks) : d.T;
        if (launch_pdl_smem(dispatch_bf16_tma_kernel, grid, 32, smem, st, static_cast<const uint16_t *>(x), topk_idx,
                            slot, static_cast<uint16_t *>(recv), recv_src, d.T, d.H, d.k, d.C, status) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (fp8) {
        // two tasks per lane per unit: 64 tasks = 1024 elements; the next unit's rows are prefetched
        const int n_tasks = d.H / 16;
        if (n_tasks % 64 == 0) return launch_fp8<2>(d, st, x, topk_idx, slot, recv, recv_scale, recv_src);
        return launch_fp8<1>(d, st, x, topk_idx, slot, recv, recv_scale, recv_src);
    }
    switch (lane_tasks(d.H / 8)) {
        case 8: return launch_bf16<8>(d, st, x, topk_idx, slot, recv, recv_src);
        case 7: return launch_bf16<7>(d, st, x, topk_idx, slot, recv, recv_src);
        case 2: return launch_bf16<2>(d, st, x, topk_idx, slot, recv, recv_src);
        case 1: return launch_bf16<1>(d, st, x, topk_idx, slot, recv, recv_src);
        default: return launch_bf16<4>(d, st, x, topk_idx, slot, recv, recv_src);
    }
}

extern "C" size_t moe_route_dispatch_workspace_bytes(const moe_problem *p) {
    moe::Dims d;
    if (moe::check_problem(p, &d) != MOE_OK) return 0;
    // the fused path uses the small-batch route's byte counts, the same workspace as moe_route
    return moe_route_workspace_bytes(p);
}

extern "C" int moe_route_dispatch(const moe_problem *p, const float *logits, const void *x, int32_t *topk_idx,
                                  float *topk_w, int32_t *counts, int32_t *offsets, int32_t *slot,
                                  int32_t *rank_counts, int32_t *dropped, void *recv, float *recv_scale,
                                  int32_t *recv_src, void *workspace, size_t workspace_bytes, void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    if (workspace_bytes < moe_route_dispatch_workspace_bytes(p)) return MOE_ERR_INVALID_ARG;
    const bool fp8 = d.dtype == MOE_DTYPE_FP8_E4M3_B128;
    const int n_tiles = (d.T + kSmallTileTokens - 1) / kSmallTileTokens;
    const bool fused = d.H <= kFusedMaxHidden && d.T <= kFusedMaxTokens && route_small(d.T, d.E) && d.max_blocks == 0;
    if (!fused) {
        rc = moe_route(p, logits, topk_idx, topk_w, counts, offsets, slot, rank_counts, dropped, workspace,
                       workspace_bytes, stream);
        if (rc != MOE_OK) return rc;
        return moe_dispatch(p, x, topk_idx, slot, recv, recv_scale, recv_src, stream);
    }
    // the same argument checks as moe_route and moe_dispatch
    if (!counts || !offsets || !rank_counts || !dropped || !workspace) return MOE_ERR_INVALID_ARG;
    if (fp8 != (recv_scale != nullptr)) return MOE_ERR_INVALID_ARG;
    if (d.T > 0 && (!logits || !x || !topk_idx || !topk_w || !slot || !recv || !recv_src)) return MOE_ERR_INVALID_ARG;
    const size_t logit_align = (d.E % 4 == 0) ? 16 : 4;
    if (!aligned(workspace, 16) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(rank_counts, 4) ||
        !aligned(dropped, 4) || (fp8 && !aligned(recv_scale, 16)))
        return MOE_ERR_INVALID_ARG;
    if (d.T > 0 && (!aligned(logits, logit_align) || !aligned(x, 16) || !aligned(recv, 16) ||
                    !aligned(topk_idx, 4) || !aligned(topk_w, 4) || !aligned(slot, 4) || !aligned(recv_src, 4)))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    unsigned *status = device_status_word();
    if (status == nullptr) return MOE_ERR_CUDA;
    uint8_t *cnt8 = static_cast<uint8_t *>(workspace);
    if (n_tiles > 0) {
        rc = launch_route_topk_small(d, st, logits, topk_idx, topk_w, slot, cnt8);
        if (rc != MOE_OK) return rc;
    }
    static PerContext<int> smem_done[2];
    auto kernel = fp8 ? route_dispatch_kernel<true> : route_dispatch_kernel<false>;
    if (!set_smem_once(smem_done[fp8], kernel, (int)fused_smem_bytes(kFusedMaxHidden, kMaxExperts)))
        return MOE_ERR_CUDA;
    if (launch_pdl_smem(kernel, d.T + 1, kFusedThreads, fused_smem_bytes(d.H, d.E), st,
                        static_cast<const uint16_t *>(x), static_cast<const int32_t *>(topk_idx),
                        static_cast<const uint8_t *>(cnt8), (int)route_small_stride(d.T), slot,
                        static_cast<uint8_t *>(recv), recv_scale, recv_src, counts, offsets, rank_counts, dropped, d.H,
                        d.E, d.k, d.C, d.R, n_tiles, status) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

// ---- per-source-rank row offsets inside each expert ---------------------------
//
// Rows of expert e are ordered by token, so by source rank: for every s the
// first row whose token comes from source s or later is a lower bound over
// recv_src. One block per expert, one thread per source rank (looping), each
// a binary search over the expert's kept rows.
namespace moe {
namespace {
__global__ void __launch_bounds__(256)
src_offsets_kernel(const int32_t *__restrict__ counts, const int32_t *__restrict__ recv_src, int32_t *__restrict__ out,
                   int C, int tps, int S) {
    pdl_enter();
    const int e = blockIdx.x;
    const int kept = min(__ldg(counts + e), C);
    const int32_t *src = recv_src + (size_t)e * C;
    for (int s = threadIdx.x; s <= S; s += blockDim.x) {
        int lo = 0, hi = kept;                              // first row with src[row] / tps >= s
        const long long first_token = (long long)s * tps;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((long long)__ldg(src + mid) < first_token) lo = mid + 1; else hi = mid;
        }
        out[(size_t)e * (S + 1) + s] = lo;
    }
}
}  // namespace
}  // namespace moe

extern "C" int moe_src_offsets(const moe_problem *p, const int32_t *counts, const int32_t *recv_src,
                               int32_t *src_offsets, void *stream) {
    using namespace moe;
    Dims d;
    const int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    if (!counts || !recv_src || !src_offsets) return MOE_ERR_INVALID_ARG;
    if (!aligned(counts, 4) || !aligned(recv_src, 4) || !aligned(src_offsets, 4)) return MOE_ERR_INVALID_ARG;
    const int tps = p->tokens_per_src_rank > 0 ? p->tokens_per_src_rank : (d.T > 0 ? d.T : 1);
    const int S = d.T > 0 ? (int)(((long long)d.T + tps - 1) / tps) : 1;
    if (launch_pdl(src_offsets_kernel, d.E, 256, as_stream(stream), counts, recv_src, src_offsets, d.C, tps, S) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
