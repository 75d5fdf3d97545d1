// moe_combine.cu -- step 4 (top-k weighted combine) and the synthetic expert
// that stands in for the grouped GEMM between dispatch and combine.
//
// [PMC §Combine]: the receiver reads each expert's 16-bit output row through
// the routing table, weights it with the router weight of that expert and sums
// the contributions into an externally allocated tensor. Here the "receive"
// is a gather from y[E][C][H] in this GPU's HBM:
//   out[t] = bf16( fma-accumulate_{j ascending, slot >= 0} w[t][j] * y[e_j][slot_j] )
//
// Both kernels are persistent: one wave of resident thread blocks walks a
// list of small work units, so that no partial second wave idles SMs, and
// no block-wide barrier sits in the steady-state loop.
//   combine: every warp walks its own units (token, 32*U chunks of 16 bytes,
//     U = 4, 2 or 1 for top-2, top-4 and above); the routing of a token is
//     held by lanes j < k and broadcast by shuffle.
//   expert: tasks (kept row, 16-byte piece) are numbered over the kept rows
//     only, through an exclusive scan of min(counts[e], C) held in shared
//     memory, so no thread walks empty capacity rows; the fp8 expert writes
//     its bf16 output through per-warp shared-memory buffers and bulk copies.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBlock = 256;                  // 8 warps; every warp walks its own work units
constexpr int kWarps = kBlock / 32;

// Lane j < k holds choice j of token t: its source row e*C + slot (< 2^31)
// or -1 when the pair was dropped, and its weight.
__device__ __forceinline__ int load_choice(unsigned t, int k, int C, const int32_t *__restrict__ topk_idx,
                                           const float *__restrict__ topk_w, const int32_t *__restrict__ slot,
                                           float &w) {
    const int lane = threadIdx.x & 31;
    w = 0.0f;
    if (lane >= k) return -1;
    const int s = __ldg(slot + (size_t)t * k + lane);
    const int e = __ldg(topk_idx + (size_t)t * k + lane);
    w = __ldg(topk_w + (size_t)t * k + lane);
    return s >= 0 ? e * C + s : -1;
}

// Unit = (token, 32*U consecutive 16-byte chunks of its row): lane l owns
// chunks 32*(U*seg + i) + l, i < U. The warp broadcasts each kept choice
// (ascending j) by shuffle, issues all KMAX*U gathers, then accumulates each
// chunk in fp32 in ascending j. U > 1 for small k keeps as many loads in
// flight per lane as top-8 has. The next unit's routing is loaded before the
// current unit's gathers are issued.
template <int KMAX, int U>
__global__ void __launch_bounds__(kBlock, KMAX * U <= 8 ? 4 : 2)
combine_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ topk_idx,
               const float *__restrict__ topk_w, const int32_t *__restrict__ slot,
               uint4 *__restrict__ out, int T, int H8, int k, int C, int segs) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    UnitWalk wk(blockIdx.x * kWarps + (threadIdx.x >> 5), gridDim.x * kWarps, segs);
    if (wk.row >= (unsigned)T) return;                         // warp-uniform
    float w;
    int src_row = load_choice(wk.row, k, C, topk_idx, topk_w, slot, w);
    for (;;) {
        UnitWalk nw = wk;
        nw.next();
        const bool more = nw.row < (unsigned)T;
        float nwt = 0.0f;
        int nrow = -1;
        if (more) nrow = load_choice(nw.row, k, C, topk_idx, topk_w, slot, nwt);
        const unsigned c0 = wk.seg * (32 * U) + lane;
        const unsigned kept = __ballot_sync(kFull, src_row >= 0);
        const int n_kept = __popc(kept);
        uint4 v[KMAX][U];
        unsigned rem = kept;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < n_kept) {                                  // warp-uniform
                const int src = __ffs(rem) - 1;
                rem &= rem - 1;
                const uint4 *yr = y + (size_t)__shfl_sync(kFull, src_row, src) * H8;
#pragma unroll
                for (int i = 0; i < U; ++i)
                    if (c0 + 32 * i < (unsigned)H8) v[j][i] = ld_stream_v4(yr + c0 + 32 * i);
            }
        }
        float wj[KMAX];
        rem = kept;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            wj[j] = 0.0f;
            if (j < n_kept) {                                  // warp-uniform
                const int src = __ffs(rem) - 1;
                rem &= rem - 1;
                wj[j] = __shfl_sync(kFull, w, src);
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j < n_kept) {                              // warp-uniform
                    const uint32_t wv[4] = {v[j][i].x, v[j][i].y, v[j][i].z, v[j][i].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = __fmaf_rn(wj[j], bf16_lo(wv[q]), acc[2 * q]);
                        acc[2 * q + 1] = __fmaf_rn(wj[j], bf16_hi(wv[q]), acc[2 * q + 1]);
                    }
                }
            }
            const unsigned c = c0 + 32 * i;
            if (c < (unsigned)H8)
                st_v4(out + (size_t)wk.row * H8 + c,
                      make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                 pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
        }
        if (!more) break;
        wk = nw;
        src_row = nrow;
        w = nwt;
    }
}

// Synthetic expert, bf16 rows. A unit is (kept row p, 32*U consecutive
// 16-byte chunks); kept rows are numbered through the scan above, so no
// warp walks an empty capacity row. Lane l owns chunks 32*(U*seg + i) + l.
template <int U>
__global__ void __launch_bounds__(kBlock)
expert_bf16_kernel(const uint4 *__restrict__ recv, const int32_t *__restrict__ counts,
                   const float *__restrict__ s, uint4 *__restrict__ y, int E, int C, int H8, int segs) {
    __shared__ int32_t off[kMaxExperts + 1];
    __shared__ int32_t warp_tot[32];
    pdl_enter();
    kept_row_offsets(counts, E, C, off, warp_tot);
    const int lane = threadIdx.x & 31;
    const unsigned rows = off[E];
    for (UnitWalk wk(blockIdx.x * kWarps + (threadIdx.x >> 5), gridDim.x * kWarps, segs); wk.row < rows;
         wk.next()) {
        const int e = expert_of_row(off, E, (int)wk.row);
        const size_t row = (size_t)e * C + (wk.row - off[e]);
        const float se = __ldg(s + e);
        const unsigned c0 = wk.seg * 32 * U + lane;
        const uint4 *in = recv + row * H8 + c0;
        uint4 *o = y + row * H8 + c0;
        uint4 v[U];
#pragma unroll
        for (int i = 0; i < U; ++i)
            if (c0 + 32 * i < (unsigned)H8) v[i] = ld_stream_v4(in + 32 * i);
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (c0 + 32 * i < (unsigned)H8) {
                const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t ov[4];
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    ov[h] = pack_bf16x2(__fmul_rn(bf16_lo(wv[h]), se), __fmul_rn(bf16_hi(wv[h]), se));
                st_v4(o + 32 * i, make_uint4(ov[0], ov[1], ov[2], ov[3]));
            }
        }
    }
}

// e4m3 code pair -> two floats, exact (every e4m3 value is a binary16 value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Synthetic expert, fp8 rows: a task is 16 codes (16 bytes in, 32 bytes of
// bf16 out) with its block scale; a unit is (kept row, 32*U tasks). The
// unit's output (32*U*32 contiguous bytes of one row) is converted into a
// per-warp shared-memory buffer and written by one bulk copy, so that the
// 117 MB of output at the DeepSeek-V3 shape leave as bulk copies instead of
// 16-byte stores (40.6 -> 28.7 us). A warp waits until its previous bulk copy
// has read the buffer before overwriting it.
template <int U>
__global__ void __launch_bounds__(kBlock)
expert_fp8_bulk_kernel(const uint4 *__restrict__ recv_q, const float *__restrict__ recv_scale,
                       const int32_t *__restrict__ counts, const float *__restrict__ s,
                       uint4 *__restrict__ y, int E, int C, int H, int segs) {
    extern __shared__ __align__(128) uint4 expert_stage[];   // kWarps x (32 * U * 2) uint4
    __shared__ int32_t off[kMaxExperts + 1];
    __shared__ int32_t warp_tot[32];
    pdl_enter();
    kept_row_offsets(counts, E, C, off, warp_tot);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint4 *buf = expert_stage + (size_t)warp * (32 * U * 2);
    const unsigned n_tasks = H / 16, nb = H / 128, rows = off[E];
    for (UnitWalk wk(blockIdx.x * kWarps + warp, gridDim.x * kWarps, segs); wk.row < rows; wk.next()) {
        const int e = expert_of_row(off, E, (int)wk.row);
        const size_t row = (size_t)e * C + (wk.row - off[e]);
        const float se = __ldg(s + e);
        const unsigned first = wk.seg * 32 * U;
        const unsigned t0 = first + lane;
        uint4 q[U];
        float sc[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (t0 + 32 * i < n_tasks) {
                q[i] = ld_stream_v4(recv_q + row * n_tasks + t0 + 32 * i);
                sc[i] = __ldg(recv_scale + row * nb + ((t0 + 32 * i) >> 3));
            }
        }
        if (lane == 0) bulk_wait_read_all();             // the previous unit's copy has read the buffer
        __syncwarp();
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (t0 + 32 * i < n_tasks) {
                const uint32_t qw[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
                uint32_t ov[8];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float2 lo = e4m3x2_to_float2(qw[h]);
                    const float2 hi = e4m3x2_to_float2(qw[h] >> 16);
                    ov[2 * h] = pack_bf16x2(__fmul_rn(__fmul_rn(lo.x, sc[i]), se), __fmul_rn(__fmul_rn(lo.y, sc[i]), se));
                    ov[2 * h + 1] = pack_bf16x2(__fmul_rn(__fmul_rn(hi.x, sc[i]), se), __fmul_rn(__fmul_rn(hi.y, sc[i]), se));
                }
                buf[2 * (32 * i + lane)] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                buf[2 * (32 * i + lane) + 1] = make_uint4(ov[4], ov[5], ov[6], ov[7]);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const unsigned n = min(32u * U, n_tasks - first);
            bulk_s2g(y + row * (H / 8) + 2 * first, buf, n * 32);
            bulk_commit();
        }
    }
    if (lane == 0) bulk_wait_all();
}

template <int U>
int launch_expert_fp8(const Dims &d, long long max_rows, cudaStream_t st, const void *recv, const float *scale,
                      const int32_t *counts, const float *s, void *y) {
    const int segs = (d.H / 16 + 32 * U - 1) / (32 * U);
    const long long units = max_rows * segs;
    if (units >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    const size_t smem = (size_t)kWarps * 32 * U * 32;
    static PerContext<int> smem_done, resident_cache;
    if (!set_smem_once(smem_done, expert_fp8_bulk_kernel<U>, (int)smem)) return MOE_ERR_CUDA;
    const int resident = resident_blocks_cached(resident_cache, expert_fp8_bulk_kernel<U>, kBlock, smem);
    const int grid = persistent_grid((units + kWarps - 1) / kWarps, resident, d.max_blocks);
    if (launch_pdl_smem(expert_fp8_bulk_kernel<U>, grid, kBlock, smem, st, static_cast<const uint4 *>(recv), scale,
                        counts, s, static_cast<uint4 *>(y), d.E, d.C, d.H, segs) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

template <int U>
int launch_expert_bf16(const Dims &d, long long max_rows, cudaStream_t st, const void *recv,
                       const int32_t *counts, const float *s, void *y) {
    static PerContext<int> resident_cache;
    const int resident = resident_blocks_cached(resident_cache, expert_bf16_kernel<U>, kBlock);
    const int segs = (d.H / 8 + 32 * U - 1) / (32 * U);
    const long long units = max_rows * segs;
    if (units >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    const int grid = persistent_grid((units + kWarps - 1) / kWarps, resident, d.max_blocks);
    if (launch_pdl(expert_bf16_kernel<U>, grid, kBlock, st, static_cast<const uint4 *>(recv), counts, s,
                   static_cast<uint4 *>(y), d.E, d.C, d.H / 8, segs) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_expert_synthetic(const moe_problem *p, const void *recv, const float *recv_scale,
                                    const int32_t *counts, const float *s, void *y, void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    const bool fp8 = d.dtype == MOE_DTYPE_FP8_E4M3_B128;
    if (fp8 != (recv_scale != nullptr)) return MOE_ERR_INVALID_ARG;
    if (!recv || !counts || !s || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned(recv, 16) || !aligned(y, 16) || !aligned(counts, 4) || !aligned(s, 4) ||
        (fp8 && !aligned(recv_scale, 16)))
        return MOE_ERR_INVALID_ARG;
    // the kept-row count is known only on the device: size the grid for the
    // largest possible one, min(T*k, E*C) rows
    const long long max_rows = std::min<long long>((long long)d.T * d.k, (long long)d.E * d.C);
    cudaStream_t st = as_stream(stream);
    if (fp8) {
        switch (lane_tasks(d.H / 16)) {
            case 8: return launch_expert_fp8<8>(d, max_rows, st, recv, recv_scale, counts, s, y);
            case 7: return launch_expert_fp8<7>(d, max_rows, st, recv, recv_scale, counts, s, y);
            case 2: return launch_expert_fp8<2>(d, max_rows, st, recv, recv_scale, counts, s, y);
            case 1: return launch_expert_fp8<1>(d, max_rows, st, recv, recv_scale, counts, s, y);
            default: return launch_expert_fp8<4>(d, max_rows, st, recv, recv_scale, counts, s, y);
        }
    }
    switch (lane_tasks(d.H / 8)) {
        case 8: return launch_expert_bf16<8>(d, max_rows, st, recv, counts, s, y);
        case 7: return launch_expert_bf16<7>(d, max_rows, st, recv, counts, s, y);
        case 2: return launch_expert_bf16<2>(d, max_rows, st, recv, counts, s, y);
        case 1: return launch_expert_bf16<1>(d, max_rows, st, recv, counts, s, y);
        default: return launch_expert_bf16<4>(d, max_rows, st, recv, counts, s, y);
    }
}

namespace {
template <int KMAX, int U = (KMAX < 8 ? 8 / KMAX : 1)>
int launch_combine(const moe::Dims &d, cudaStream_t st, const uint4 *y, const int32_t *idx, const float *w,
                   const int32_t *slot, uint4 *out) {
    using namespace moe;
    static PerContext<int> resident_cache;
    const int resident = resident_blocks_cached(resident_cache, combine_kernel<KMAX, U>, kBlock);
    const int H8 = d.H / 8;
    const int segs = (H8 + 32 * U - 1) / (32 * U);
    const long long units = (long long)d.T * segs;
    if (units >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    const int grid = persistent_grid((units + kWarps - 1) / kWarps, resident, d.max_blocks);
    if (launch_pdl(combine_kernel<KMAX, U>, grid, kBlock, st, y, idx, w, slot, out, d.T, H8, d.k, d.C, segs) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
}  // namespace

extern "C" int moe_combine(const moe_problem *p, const void *y, const int32_t *topk_idx,
                           const float *topk_w, const int32_t *slot, void *out, void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    if (d.T == 0) return MOE_OK;
    if (!y || !topk_idx || !topk_w || !slot || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
        !aligned(slot, 4))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    const uint4 *yy = static_cast<const uint4 *>(y);
    uint4 *oo = static_cast<uint4 *>(out);
    if (d.k <= 2) return launch_combine<2>(d, st, yy, topk_idx, topk_w, slot, oo);
    if (d.k <= 4) return launch_combine<4>(d, st, yy, topk_idx, topk_w, slot, oo);
    if (d.k <= 8) return launch_combine<8>(d, st, yy, topk_idx, topk_w, slot, oo);
    return launch_combine<16>(d, st, yy, topk_idx, topk_w, slot, oo);
}
