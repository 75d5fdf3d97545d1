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
// Persistent kernels: one wave of resident thread blocks; every warp walks
// its own work units (token, segment of its row) with no block-wide barrier.
// Lanes j < k hold the token's destination rows and broadcast them by
// shuffle (ascending j). The next unit's routing and row data are loaded
// before the current unit is stored, so that two units' loads are in flight.
// recv_src is written on a token's first segment.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBlock = 256;             // 8 warps; every warp walks its own work units
constexpr int kWarps = kBlock / 32;

// Lane j < k holds choice j of token t (slot, expert).
struct Dest {
    int s, e;
};
__device__ __forceinline__ Dest load_dest(int t, int k, const int32_t *__restrict__ topk_idx,
                                          const int32_t *__restrict__ slot) {
    Dest d{-1, 0};
    const int lane = threadIdx.x & 31;
    if (lane < k) {
        d.s = __ldg(slot + (size_t)t * k + lane);
        d.e = __ldg(topk_idx + (size_t)t * k + lane);
    }
    return d;
}

// bf16: unit = (token, 64 consecutive 16-byte chunks); lane l owns chunks
// 64*seg + l and 64*seg + 32 + l.
__global__ void __launch_bounds__(kBlock)
dispatch_bf16_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                     const int32_t *__restrict__ slot, uint4 *__restrict__ recv,
                     int32_t *__restrict__ recv_src, int T, int H8, int k, int C, int segs) {
    const int lane = threadIdx.x & 31;
    const long long n_units = (long long)T * segs;
    const long long stride = (long long)gridDim.x * kWarps;
    long long u = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (u >= n_units) return;                                      // warp-uniform
    auto load_row = [&](long long unit, uint4 &a, uint4 &b) {
        const int t = (int)(unit / segs), c = (int)(unit % segs) * 64 + lane;
        const uint4 *src = x + (size_t)t * H8;
        if (c < H8) a = ld_stream_v4(src + c);
        if (c + 32 < H8) b = ld_stream_v4(src + c + 32);
    };
    Dest cur = load_dest((int)(u / segs), k, topk_idx, slot);
    uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
    load_row(u, a0, a1);
    for (; u < n_units; u += stride) {
        const long long un = u + stride;
        Dest nxt{-1, 0};
        uint4 b0 = make_uint4(0, 0, 0, 0), b1 = b0;
        if (un < n_units) {
            nxt = load_dest((int)(un / segs), k, topk_idx, slot);
            load_row(un, b0, b1);
        }
        const int t = (int)(u / segs);
        const int sg = (int)(u % segs);
        const int c = sg * 64 + lane;
        const long long my_row = (long long)cur.e * C + (cur.s >= 0 ? cur.s : 0);
        if (sg == 0 && cur.s >= 0) recv_src[my_row] = t;
        unsigned rem = __ballot_sync(kFull, cur.s >= 0);
        while (rem) {                                              // warp-uniform
            const int src = __ffs(rem) - 1;
            rem &= rem - 1;
            uint4 *dst = recv + __shfl_sync(kFull, my_row, src) * H8;
            if (c < H8) st_v4(dst + c, a0);
            if (c + 32 < H8) st_v4(dst + c + 32, a1);
        }
        cur = nxt;
        a0 = b0;
        a1 = b1;
    }
}

// fp8: unit = (token, 32 tasks of 16 elements = 512 elements); lane l owns
// task 32*seg + l. The 8 lanes of one 128-element block agree on its amax
// with 3 shuffles; scale = amax/448 (1 for an all-zero block); codes are
// e4m3(x / scale), round to nearest even, saturating.
__global__ void __launch_bounds__(kBlock)
dispatch_fp8_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx,
                    const int32_t *__restrict__ slot, uint4 *__restrict__ recv_q,
                    float *__restrict__ recv_scale, int32_t *__restrict__ recv_src, int T, int H,
                    int k, int C, int segs) {
    const int lane = threadIdx.x & 31;
    const int n_tasks = H / 16, nb = H / 128;
    const long long n_units = (long long)T * segs;
    const long long stride = (long long)gridDim.x * kWarps;
    long long u = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (u >= n_units) return;                                      // warp-uniform
    auto load_task = [&](long long unit, uint4 &a, uint4 &b) {
        const int t = (int)(unit / segs), task = (int)(unit % segs) * 32 + lane;
        if (task < n_tasks) {
            const uint4 *src = x + (size_t)t * (H / 8) + 2 * task;
            a = ld_stream_v4(src);
            b = ld_stream_v4(src + 1);
        }
    };
    Dest cur = load_dest((int)(u / segs), k, topk_idx, slot);
    uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
    load_task(u, a0, a1);
    for (; u < n_units; u += stride) {
        const long long un = u + stride;
        Dest nxt{-1, 0};
        uint4 b0 = make_uint4(0, 0, 0, 0), b1 = b0;
        if (un < n_units) {
            nxt = load_dest((int)(un / segs), k, topk_idx, slot);
            load_task(un, b0, b1);
        }
        const int t = (int)(u / segs);
        const int sg = (int)(u % segs);
        const int task = sg * 32 + lane;
        const bool on = task < n_tasks;                            // uniform per 8-lane block
        const uint32_t wv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float f[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            f[2 * i] = bf16_lo(wv[i]);
            f[2 * i + 1] = bf16_hi(wv[i]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
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
        const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
        const long long my_row = (long long)cur.e * C + (cur.s >= 0 ? cur.s : 0);
        if (sg == 0 && cur.s >= 0) recv_src[my_row] = t;
        unsigned rem = __ballot_sync(kFull, cur.s >= 0);
        while (rem) {                                              // warp-uniform
            const int src = __ffs(rem) - 1;
            rem &= rem - 1;
            const long long row = __shfl_sync(kFull, my_row, src);
            if (on) {
                st_v4(recv_q + row * n_tasks + task, qv);
                if ((lane & 7) == 0) recv_scale[row * nb + (task >> 3)] = scale;
            }
        }
        cur = nxt;
        a0 = b0;
        a1 = b1;
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
        static int resident = resident_blocks(dispatch_fp8_kernel, kBlock);
        const int segs = (d.H / 16 + 31) / 32;
        const long long units = (long long)d.T * segs;
        const int grid = persistent_grid((units + kWarps - 1) / kWarps, resident, d.max_blocks);
        dispatch_fp8_kernel<<<grid, kBlock, 0, st>>>(static_cast<const uint4 *>(x), topk_idx, slot,
                                                     static_cast<uint4 *>(recv), recv_scale, recv_src, d.T, d.H,
                                                     d.k, d.C, segs);
    } else {
        static int resident = resident_blocks(dispatch_bf16_kernel, kBlock);
        const int H8 = d.H / 8;
        const int segs = (H8 + 63) / 64;
        const long long units = (long long)d.T * segs;
        const int grid = persistent_grid((units + kWarps - 1) / kWarps, resident, d.max_blocks);
        dispatch_bf16_kernel<<<grid, kBlock, 0, st>>>(static_cast<const uint4 *>(x), topk_idx, slot,
                                                      static_cast<uint4 *>(recv), recv_src, d.T, H8, d.k, d.C,
                                                      segs);
    }
    return launch_status();
}
