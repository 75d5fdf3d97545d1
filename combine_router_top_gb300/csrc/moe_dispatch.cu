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
// One CTA per token (grid-stride when max_blocks caps the grid): warp 0
// gathers the token's kept destinations (ascending j) into shared memory and
// writes recv_src; every thread then reads its 16-byte chunks of the row once
// and stores them to all destinations. fp8: a lane quantises 16 elements, the
// 8 lanes of a 128-element block agree on amax with 3 shuffles.
#include "moe_internal.cuh"

namespace moe {
namespace {

// Warp 0 compacts the kept destination rows of token t (ascending j) into
// dst_row[0..*n_dst) and records the origin of each. Ends with a CTA barrier.
__device__ __forceinline__ void token_destinations(int t, int k, int C, const int32_t *__restrict__ topk_idx,
                                                   const int32_t *__restrict__ slot, long long *dst_row,
                                                   int *n_dst, int32_t *__restrict__ recv_src) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        long long row = -1;
        if (lane < k) {
            const int s = slot[(size_t)t * k + lane];
            if (s >= 0) row = (long long)topk_idx[(size_t)t * k + lane] * C + s;
        }
        const unsigned kept = __ballot_sync(kFull, row >= 0);
        if (row >= 0) {
            dst_row[__popc(kept & ((1u << lane) - 1u))] = row;
            recv_src[row] = t;
        }
        if (lane == 0) *n_dst = __popc(kept);
    }
    __syncthreads();
}

constexpr int kDispatchUnroll = 4;

__global__ void __launch_bounds__(256)
dispatch_bf16_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                     const int32_t *__restrict__ slot, uint4 *__restrict__ recv,
                     int32_t *__restrict__ recv_src, int T, int H8, int k, int C) {
    __shared__ long long dst_row[kMaxTopK];
    __shared__ int n_dst;
    const int step = blockDim.x * kDispatchUnroll;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        token_destinations(t, k, C, topk_idx, slot, dst_row, &n_dst, recv_src);
        const int nd = n_dst;
        const uint4 *src = x + (size_t)t * H8;
        for (int c0 = threadIdx.x; c0 < H8; c0 += step) {
            uint4 v[kDispatchUnroll];
#pragma unroll
            for (int u = 0; u < kDispatchUnroll; ++u) {
                const int c = c0 + u * blockDim.x;
                if (c < H8) v[u] = ld_stream_v4(src + c);
            }
            for (int j = 0; j < nd; ++j) {
                uint4 *d = recv + dst_row[j] * H8;
#pragma unroll
                for (int u = 0; u < kDispatchUnroll; ++u) {
                    const int c = c0 + u * blockDim.x;
                    if (c < H8) st_v4(d + c, v[u]);
                }
            }
        }
        __syncthreads();   // dst_row is rewritten for the next token
    }
}

// A task is 16 consecutive elements of a row: 32 bytes of bf16 in, 16 bytes of e4m3 out.
__global__ void __launch_bounds__(256)
dispatch_fp8_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                    const int32_t *__restrict__ slot, uint4 *__restrict__ recv_q,
                    float *__restrict__ recv_scale, int32_t *__restrict__ recv_src, int T, int H,
                    int k, int C) {
    __shared__ long long dst_row[kMaxTopK];
    __shared__ int n_dst;
    const int n_tasks = H / 16, nb = H / 128;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        token_destinations(t, k, C, topk_idx, slot, dst_row, &n_dst, recv_src);
        const int nd = n_dst;
        const uint4 *src = x + (size_t)t * (H / 8);
        for (int base = 0; base < n_tasks; base += blockDim.x) {     // uniform trip count
            const int task = base + threadIdx.x;
            const bool on = task < n_tasks;
            uint4 a = make_uint4(0, 0, 0, 0), b = a;
            if (on) {
                a = ld_stream_v4(src + 2 * task);
                b = ld_stream_v4(src + 2 * task + 1);
            }
            const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            float f[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                f[2 * i] = bf16_lo(wv[i]);
                f[2 * i + 1] = bf16_hi(wv[i]);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
            // the 8 lanes of one 128-element block (lanes 8g .. 8g+7)
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
            const float scale = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = pack_e4m3x2(__fdiv_rn(f[4 * i], scale), __fdiv_rn(f[4 * i + 1], scale));
                const uint32_t hi = pack_e4m3x2(__fdiv_rn(f[4 * i + 2], scale), __fdiv_rn(f[4 * i + 3], scale));
                q[i] = lo | (hi << 16);
            }
            if (on) {
                const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
                for (int j = 0; j < nd; ++j) {
                    st_v4(recv_q + dst_row[j] * n_tasks + task, qv);
                    if ((threadIdx.x & 7) == 0) recv_scale[dst_row[j] * nb + (task >> 3)] = scale;
                }
            }
        }
        __syncthreads();
    }
}

// Threads per CTA: the largest multiple of 32 (<= 256) dividing `work`, else 128.
int pick_block(int work) {
    for (int b = 256; b >= 32; b -= 32)
        if (work % b == 0) return b;
    return 128;
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

    const int grid = d.max_blocks > 0 && d.max_blocks < d.T ? d.max_blocks : d.T;
    cudaStream_t st = as_stream(stream);
    if (fp8) {
        const int block = pick_block(d.H / 16);
        dispatch_fp8_kernel<<<grid, block, 0, st>>>(static_cast<const uint4 *>(x), topk_idx, slot,
                                                    static_cast<uint4 *>(recv), recv_scale, recv_src,
                                                    d.T, d.H, d.k, d.C);
    } else {
        const int H8 = d.H / 8;
        int block = pick_block((H8 + kDispatchUnroll - 1) / kDispatchUnroll);
        dispatch_bf16_kernel<<<grid, block, 0, st>>>(static_cast<const uint4 *>(x), topk_idx, slot,
                                                     static_cast<uint4 *>(recv), recv_src, d.T, H8,
                                                     d.k, d.C);
    }
    return launch_status();
}
