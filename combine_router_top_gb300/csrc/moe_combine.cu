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
// list of small work units, so that no partial second wave idles SMs.
//   combine: unit = (token, 128 consecutive 16-byte chunks of its row). A
//     thread owns one chunk: it issues the k gathers, then k fp32 FMAs in
//     ascending j, then one 16-byte bf16 store. Warp 0 loads the next unit's
//     routing (row, weight) into the other half of a double buffer while the
//     block works on the current one.
//   expert: unit = (kept row, segment of the row). Kept rows are enumerated
//     compactly through an exclusive scan of min(counts[e], C) held in
//     shared memory, so no block walks empty capacity rows.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kCombineBlock = 128;

// Warp 0: compacted (row offset in 16-byte units, weight) of token t's kept
// choices, ascending j. The three loads of a lane are independent.
template <int KMAX>
__device__ __forceinline__ void combine_routing(int t, int k, int C, int H8, const int32_t *__restrict__ topk_idx,
                                                const float *__restrict__ topk_w, const int32_t *__restrict__ slot,
                                                long long *rows, float *ws, int *n) {
    const int lane = threadIdx.x;
    int s = -1, e = 0;
    float w = 0.0f;
    if (lane < k) {
        s = __ldg(slot + (size_t)t * k + lane);
        e = __ldg(topk_idx + (size_t)t * k + lane);
        w = __ldg(topk_w + (size_t)t * k + lane);
    }
    const unsigned kept = __ballot_sync(kFull, s >= 0);
    if (s >= 0) {
        const int pos = __popc(kept & ((1u << lane) - 1u));
        rows[pos] = ((long long)e * C + s) * H8;
        ws[pos] = w;
    }
    if (lane == 0) *n = __popc(kept);
}

template <int KMAX>
__global__ void __launch_bounds__(kCombineBlock)
combine_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ topk_idx,
               const float *__restrict__ topk_w, const int32_t *__restrict__ slot,
               uint4 *__restrict__ out, int T, int H8, int k, int C, int segs) {
    __shared__ long long s_row[2][KMAX];
    __shared__ float s_w[2][KMAX];
    __shared__ int s_n[2];
    const long long n_units = (long long)T * segs;
    long long u = blockIdx.x;
    if (u >= n_units) return;
    if (threadIdx.x < 32)
        combine_routing<KMAX>((int)(u / segs), k, C, H8, topk_idx, topk_w, slot, s_row[0], s_w[0], &s_n[0]);
    __syncthreads();
    int b = 0;
    for (; u < n_units; u += gridDim.x) {
        const long long un = u + gridDim.x;
        if (un < n_units && threadIdx.x < 32)
            combine_routing<KMAX>((int)(un / segs), k, C, H8, topk_idx, topk_w, slot, s_row[b ^ 1], s_w[b ^ 1],
                                  &s_n[b ^ 1]);
        const int t = (int)(u / segs);
        const int c = (int)(u % segs) * kCombineBlock + threadIdx.x;
        const int ns = s_n[b];
        if (c < H8) {
            uint4 v[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < ns) v[j] = ld_stream_v4(y + s_row[b][j] + c);
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j < ns) {
                    const float w = s_w[b][j];
                    const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] = __fmaf_rn(w, bf16_lo(wv[i]), acc[2 * i]);
                        acc[2 * i + 1] = __fmaf_rn(w, bf16_hi(wv[i]), acc[2 * i + 1]);
                    }
                }
            }
            st_v4(out + (size_t)t * H8 + c,
                  make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                             pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
        }
        __syncthreads();   // current buffer consumed, next one filled
        b ^= 1;
    }
}

// Exclusive scan of min(counts[e], C) over e into off[0..E] (off[E] = kept rows).
__device__ void kept_row_offsets(const int32_t *__restrict__ counts, int E, int C, int32_t *off, int32_t *warp_tot) {
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

// Expert e of kept row p: the last e with off[e] <= p (off is non-decreasing).
__device__ __forceinline__ int expert_of_row(const int32_t *off, int E, int p) {
    int lo = 0, hi = E;        // off[lo] <= p < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= p) lo = mid; else hi = mid;
    }
    return lo;
}

constexpr int kExpertBf16Block = 128;   // one 16-byte chunk (8 bf16) per thread per unit
constexpr int kExpertFp8Block = 64;     // 16 e4m3 codes per thread per unit

__global__ void __launch_bounds__(kExpertBf16Block)
expert_bf16_kernel(const uint4 *__restrict__ recv, const int32_t *__restrict__ counts,
                   const float *__restrict__ s, uint4 *__restrict__ y, int E, int C, int H8, int segs) {
    __shared__ int32_t off[kMaxExperts + 1];
    __shared__ int32_t warp_tot[32];
    kept_row_offsets(counts, E, C, off, warp_tot);
    const long long n_units = (long long)off[E] * segs;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int p = (int)(u / segs);
        const int e = expert_of_row(off, E, p);
        const long long row = (long long)e * C + (p - off[e]);
        const int c = (int)(u % segs) * kExpertBf16Block + threadIdx.x;
        if (c < H8) {
            const float se = __ldg(s + e);
            const uint4 v = ld_stream_v4(recv + row * H8 + c);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            uint32_t ov[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                ov[i] = pack_bf16x2(__fmul_rn(bf16_lo(wv[i]), se), __fmul_rn(bf16_hi(wv[i]), se));
            st_v4(y + row * H8 + c, make_uint4(ov[0], ov[1], ov[2], ov[3]));
        }
    }
}

// e4m3 code -> float, exact (every e4m3 value is a binary16 and a binary32 value).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
    return __half2float(*reinterpret_cast<const __half *>(&h));
}

__global__ void __launch_bounds__(kExpertFp8Block)
expert_fp8_kernel(const uint4 *__restrict__ recv_q, const float *__restrict__ recv_scale,
                  const int32_t *__restrict__ counts, const float *__restrict__ s,
                  uint4 *__restrict__ y, int E, int C, int H, int segs) {
    __shared__ int32_t off[kMaxExperts + 1];
    __shared__ int32_t warp_tot[32];
    kept_row_offsets(counts, E, C, off, warp_tot);
    const int n_tasks = H / 16, nb = H / 128;
    const long long n_units = (long long)off[E] * segs;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int p = (int)(u / segs);
        const int e = expert_of_row(off, E, p);
        const long long row = (long long)e * C + (p - off[e]);
        const int task = (int)(u % segs) * kExpertFp8Block + threadIdx.x;
        if (task < n_tasks) {
            const float se = __ldg(s + e);
            const uint4 q = ld_stream_v4(recv_q + row * n_tasks + task);
            const float sc = __ldg(recv_scale + row * nb + (task >> 3));
            const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
            uint32_t ov[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t two = qw[i] >> (16 * h);
                    const float a = __fmul_rn(__fmul_rn(e4m3_to_float(two & 0xFFu), sc), se);
                    const float b = __fmul_rn(__fmul_rn(e4m3_to_float((two >> 8) & 0xFFu), sc), se);
                    ov[2 * i + h] = pack_bf16x2(a, b);
                }
            }
            uint4 *o = y + row * (H / 8) + 2 * task;
            st_v4(o, make_uint4(ov[0], ov[1], ov[2], ov[3]));
            st_v4(o + 1, make_uint4(ov[4], ov[5], ov[6], ov[7]));
        }
    }
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
        static int resident = resident_blocks(expert_fp8_kernel, kExpertFp8Block);
        const int segs = (d.H / 16 + kExpertFp8Block - 1) / kExpertFp8Block;
        const int grid = persistent_grid(max_rows * segs, resident, d.max_blocks);
        expert_fp8_kernel<<<grid, kExpertFp8Block, 0, st>>>(static_cast<const uint4 *>(recv), recv_scale, counts, s,
                                                            static_cast<uint4 *>(y), d.E, d.C, d.H, segs);
    } else {
        static int resident = resident_blocks(expert_bf16_kernel, kExpertBf16Block);
        const int segs = (d.H / 8 + kExpertBf16Block - 1) / kExpertBf16Block;
        const int grid = persistent_grid(max_rows * segs, resident, d.max_blocks);
        expert_bf16_kernel<<<grid, kExpertBf16Block, 0, st>>>(static_cast<const uint4 *>(recv), counts, s,
                                                              static_cast<uint4 *>(y), d.E, d.C, d.H / 8, segs);
    }
    return launch_status();
}

namespace {
template <int KMAX>
int launch_combine(const moe::Dims &d, cudaStream_t st, const uint4 *y, const int32_t *idx, const float *w,
                   const int32_t *slot, uint4 *out) {
    using namespace moe;
    static int resident = resident_blocks(combine_kernel<KMAX>, kCombineBlock);
    const int H8 = d.H / 8;
    const int segs = (H8 + kCombineBlock - 1) / kCombineBlock;
    const int grid = persistent_grid((long long)d.T * segs, resident, d.max_blocks);
    combine_kernel<KMAX><<<grid, kCombineBlock, 0, st>>>(y, idx, w, slot, out, d.T, H8, d.k, d.C, segs);
    return launch_status();
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
