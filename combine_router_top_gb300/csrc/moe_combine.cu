// moe_combine.cu -- step 4 (top-k weighted combine) and the synthetic expert
// that stands in for the grouped GEMM between dispatch and combine.
//
// [PMC §Combine]: the receiver reads each expert's 16-bit output row through
// the routing table, weights it with the router weight of that expert and sums
// the contributions into an externally allocated tensor. Here the "receive"
// is a gather from y[E][C][H] in this GPU's HBM:
//   out[t] = bf16( fma-accumulate_{j ascending, slot >= 0} w[t][j] * y[e_j][slot_j] )
// One CTA per token (grid-stride under max_blocks). Warp 0 compacts the kept
// (row, weight) pairs; each thread owns 16-byte chunks of the row, issues all
// k gathers of a chunk before the first FMA, accumulates in fp32 and stores
// 16 bytes of bf16.
#include "moe_internal.cuh"

namespace moe {
namespace {

template <int KMAX>
__global__ void __launch_bounds__(256)
combine_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ topk_idx,
               const float *__restrict__ topk_w, const int32_t *__restrict__ slot,
               uint4 *__restrict__ out, int T, int H8, int k, int C) {
    __shared__ long long src_row[KMAX];
    __shared__ float src_w[KMAX];
    __shared__ int n_src;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            long long row = -1;
            float w = 0.0f;
            if (lane < k) {
                const int s = slot[(size_t)t * k + lane];
                if (s >= 0) {
                    row = (long long)topk_idx[(size_t)t * k + lane] * C + s;
                    w = topk_w[(size_t)t * k + lane];
                }
            }
            const unsigned kept = __ballot_sync(kFull, row >= 0);
            if (row >= 0) {
                const int pos = __popc(kept & ((1u << lane) - 1u));
                src_row[pos] = row * H8;
                src_w[pos] = w;
            }
            if (lane == 0) n_src = __popc(kept);
        }
        __syncthreads();
        const int ns = n_src;
        uint4 *dst = out + (size_t)t * H8;
        for (int c = threadIdx.x; c < H8; c += blockDim.x) {
            uint4 v[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < ns) v[j] = ld_stream_v4(y + src_row[j] + c);
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j < ns) {
                    const float w = src_w[j];
                    const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] = __fmaf_rn(w, bf16_lo(wv[i]), acc[2 * i]);
                        acc[2 * i + 1] = __fmaf_rn(w, bf16_hi(wv[i]), acc[2 * i + 1]);
                    }
                }
            }
            st_v4(dst + c, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                      pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
        }
        __syncthreads();
    }
}

// Synthetic expert, bf16 rows: one warp per row (grid-stride over all E*C rows,
// rows at or past min(counts[e], C) skipped).
__global__ void __launch_bounds__(256)
expert_bf16_kernel(const uint4 *__restrict__ recv, const int32_t *__restrict__ counts,
                   const float *__restrict__ s, uint4 *__restrict__ y, int E, int C, int H8) {
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < (long long)E * C;
         row += warps) {
        const int e = (int)(row / C), r = (int)(row % C);
        if (r >= __ldg(counts + e)) continue;          // warp-uniform
        const float se = __ldg(s + e);
        const uint4 *in = recv + row * H8;
        uint4 *o = y + row * H8;
        for (int c = lane; c < H8; c += 32) {
            const uint4 v = ld_stream_v4(in + c);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            uint32_t ov[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ov[i] = pack_bf16x2(__fmul_rn(bf16_lo(wv[i]), se), __fmul_rn(bf16_hi(wv[i]), se));
            st_v4(o + c, make_uint4(ov[0], ov[1], ov[2], ov[3]));
        }
    }
}

// e4m3 code -> float, exact (every e4m3 value is a binary32 value).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
    const __nv_fp8_storage_t b = static_cast<__nv_fp8_storage_t>(byte);
    const __half_raw h = __nv_cvt_fp8_to_halfraw(b, __NV_E4M3);
    return __half2float(*reinterpret_cast<const __half *>(&h));
}

// Synthetic expert, fp8 rows: a lane handles 16 codes (one 16-byte load) and
// writes 16 bf16 (two 16-byte stores); 8 lanes share one block scale.
__global__ void __launch_bounds__(256)
expert_fp8_kernel(const uint4 *__restrict__ recv_q, const float *__restrict__ recv_scale,
                  const int32_t *__restrict__ counts, const float *__restrict__ s,
                  uint4 *__restrict__ y, int E, int C, int H) {
    const int lane = threadIdx.x & 31;
    const int n_tasks = H / 16, nb = H / 128;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < (long long)E * C;
         row += warps) {
        const int e = (int)(row / C), r = (int)(row % C);
        if (r >= __ldg(counts + e)) continue;
        const float se = __ldg(s + e);
        for (int task = lane; task < n_tasks; task += 32) {
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

int pick_block(int work) {
    for (int b = 256; b >= 32; b -= 32)
        if (work % b == 0) return b;
    return 128;
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
    const long long rows = (long long)d.E * d.C;
    long long grid = (rows + 7) / 8;
    const long long cap = d.max_blocks > 0 ? d.max_blocks : (long long)sm_count() * 8;
    if (grid > cap) grid = cap;
    cudaStream_t st = as_stream(stream);
    if (fp8)
        expert_fp8_kernel<<<(int)grid, 256, 0, st>>>(static_cast<const uint4 *>(recv), recv_scale, counts, s,
                                                     static_cast<uint4 *>(y), d.E, d.C, d.H);
    else
        expert_bf16_kernel<<<(int)grid, 256, 0, st>>>(static_cast<const uint4 *>(recv), counts, s,
                                                      static_cast<uint4 *>(y), d.E, d.C, d.H / 8);
    return launch_status();
}

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
    const int H8 = d.H / 8;
    const int block = pick_block(H8);
    const int grid = d.max_blocks > 0 && d.max_blocks < d.T ? d.max_blocks : d.T;
    cudaStream_t st = as_stream(stream);
    const uint4 *yy = static_cast<const uint4 *>(y);
    uint4 *oo = static_cast<uint4 *>(out);
    if (d.k <= 2) combine_kernel<2><<<grid, block, 0, st>>>(yy, topk_idx, topk_w, slot, oo, d.T, H8, d.k, d.C);
    else if (d.k <= 4) combine_kernel<4><<<grid, block, 0, st>>>(yy, topk_idx, topk_w, slot, oo, d.T, H8, d.k, d.C);
    else if (d.k <= 8) combine_kernel<8><<<grid, block, 0, st>>>(yy, topk_idx, topk_w, slot, oo, d.T, H8, d.k, d.C);
    else combine_kernel<16><<<grid, block, 0, st>>>(yy, topk_idx, topk_w, slot, oo, d.T, H8, d.k, d.C);
    return launch_status();
}
