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
// Persistent kernels: one wave of resident thread blocks walks the work units
// (token, 1024-element segment of its row), so no partial second wave idles
// SMs. Warp 0 gathers the kept destination rows (ascending j) of the next
// unit into the other half of a shared-memory double buffer while the block
// copies the current one, and writes recv_src on a token's first segment.
// A thread reads its part of the row once and stores it to every
// destination. fp8: a thread quantises 16 elements; the 8 threads of one
// 128-element block agree on amax with 3 shuffles.
#include "moe_internal.cuh"

namespace moe {
namespace {

// Warp 0: compacted destination rows (ascending j) of token t; on the token's
// first segment also records the origin of each row.
__device__ __forceinline__ void dispatch_routing(int t, bool first_seg, int k, int C,
                                                 const int32_t *__restrict__ topk_idx,
                                                 const int32_t *__restrict__ slot, long long *rows, int *n,
                                                 int32_t *__restrict__ recv_src) {
    const int lane = threadIdx.x;
    int s = -1, e = 0;
    if (lane < k) {
        s = __ldg(slot + (size_t)t * k + lane);
        e = __ldg(topk_idx + (size_t)t * k + lane);
    }
    const unsigned kept = __ballot_sync(kFull, s >= 0);
    if (s >= 0) {
        const long long row = (long long)e * C + s;
        rows[__popc(kept & ((1u << lane) - 1u))] = row;
        if (first_seg) recv_src[row] = t;
    }
    if (lane == 0) *n = __popc(kept);
}

constexpr int kDispatchBf16Block = 128;   // 16-byte chunk (8 elements) per thread per unit
constexpr int kDispatchFp8Block = 64;     // 16 elements per thread per unit

__global__ void __launch_bounds__(kDispatchBf16Block)
dispatch_bf16_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                     const int32_t *__restrict__ slot, uint4 *__restrict__ recv,
                     int32_t *__restrict__ recv_src, int T, int H8, int k, int C, int segs) {
    __shared__ long long s_row[2][kMaxTopK];
    __shared__ int s_n[2];
    const long long n_units = (long long)T * segs;
    long long u = blockIdx.x;
    if (u >= n_units) return;
    if (threadIdx.x < 32)
        dispatch_routing((int)(u / segs), u % segs == 0, k, C, topk_idx, slot, s_row[0], &s_n[0], recv_src);
    __syncthreads();
    int b = 0;
    for (; u < n_units; u += gridDim.x) {
        const long long un = u + gridDim.x;
        if (un < n_units && threadIdx.x < 32)
            dispatch_routing((int)(un / segs), un % segs == 0, k, C, topk_idx, slot, s_row[b ^ 1], &s_n[b ^ 1],
                             recv_src);
        const int t = (int)(u / segs);
        const int c = (int)(u % segs) * kDispatchBf16Block + threadIdx.x;
        if (c < H8) {
            const uint4 v = ld_stream_v4(x + (size_t)t * H8 + c);
            const int nd = s_n[b];
            for (int j = 0; j < nd; ++j) st_v4(recv + s_row[b][j] * H8 + c, v);
        }
        __syncthreads();
        b ^= 1;
    }
}

// A task is 16 consecutive elements of a row: 32 bytes of bf16 in, 16 bytes of e4m3 out.
__global__ void __launch_bounds__(kDispatchFp8Block)
dispatch_fp8_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                    const int32_t *__restrict__ slot, uint4 *__restrict__ recv_q,
                    float *__restrict__ recv_scale, int32_t *__restrict__ recv_src, int T, int H,
                    int k, int C, int segs) {
    __shared__ long long s_row[2][kMaxTopK];
    __shared__ int s_n[2];
    const int n_tasks = H / 16, nb = H / 128;
    const long long n_units = (long long)T * segs;
    long long u = blockIdx.x;
    if (u >= n_units) return;
    if (threadIdx.x < 32)
        dispatch_routing((int)(u / segs), u % segs == 0, k, C, topk_idx, slot, s_row[0], &s_n[0], recv_src);
    __syncthreads();
    int b = 0;
    for (; u < n_units; u += gridDim.x) {
        const long long un = u + gridDim.x;
        if (un < n_units && threadIdx.x < 32)
            dispatch_routing((int)(un / segs), un % segs == 0, k, C, topk_idx, slot, s_row[b ^ 1], &s_n[b ^ 1],
                             recv_src);
        const int t = (int)(u / segs);
        const int task = (int)(u % segs) * kDispatchFp8Block + threadIdx.x;
        const bool on = task < n_tasks;            // uniform over each 8-thread block group
        uint4 a = make_uint4(0, 0, 0, 0), c = a;
        if (on) {
            const uint4 *src = x + (size_t)t * (H / 8) + 2 * task;
            a = ld_stream_v4(src);
            c = ld_stream_v4(src + 1);
        }
        const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        float f[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            f[2 * i] = bf16_lo(wv[i]);
            f[2 * i + 1] = bf16_hi(wv[i]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
        // the 8 threads of one 128-element block (lanes 8g .. 8g+7)
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
            const int nd = s_n[b];
            for (int j = 0; j < nd; ++j) {
                const long long row = s_row[b][j];
                st_v4(recv_q + row * n_tasks + task, qv);
                if ((threadIdx.x & 7) == 0) recv_scale[row * nb + (task >> 3)] = scale;
            }
        }
        __syncthreads();
        b ^= 1;
    }
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
    if (fp8) {
        static int resident = resident_blocks(dispatch_fp8_kernel, kDispatchFp8Block);
        const int segs = (d.H / 16 + kDispatchFp8Block - 1) / kDispatchFp8Block;
        const int grid = persistent_grid((long long)d.T * segs, resident, d.max_blocks);
        dispatch_fp8_kernel<<<grid, kDispatchFp8Block, 0, st>>>(static_cast<const uint4 *>(x), topk_idx, slot,
                                                                static_cast<uint4 *>(recv), recv_scale, recv_src,
                                                                d.T, d.H, d.k, d.C, segs);
    } else {
        static int resident = resident_blocks(dispatch_bf16_kernel, kDispatchBf16Block);
        const int H8 = d.H / 8;
        const int segs = (H8 + kDispatchBf16Block - 1) / kDispatchBf16Block;
        const int grid = persistent_grid((long long)d.T * segs, resident, d.max_blocks);
        dispatch_bf16_kernel<<<grid, kDispatchBf16Block, 0, st>>>(static_cast<const uint4 *>(x), topk_idx, slot,
                                                                  static_cast<uint4 *>(recv), recv_src, d.T, H8,
                                                                  d.k, d.C, segs);
    }
    return launch_status();
}
