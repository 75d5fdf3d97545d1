// moe_ready.cu -- synthetic expert and combine in one kernel, with readiness
// tracked per expert row instead of per kernel.
//
// "Efficient and portable mixture-of-experts communication" (§Further
// Improvements) notes that buffers shared across devices would allow
// synchronisation per individual token instead of per batch of tokens. On
// one GPU the batch boundary is the kernel boundary between the expert and
// combine; here it is replaced by one flag per (expert row, segment):
//
//   phase 1   every warp computes its units of the synthetic expert (kept
//             row, segment of 32 x 4 sixteen-byte pieces; the arithmetic of
//             moe_expert_synthetic); after a unit's stores, one release store
//             sets its flag to the call's epoch;
//   phase 2   every warp then takes combine units (token, 32 chunks of 8
//             outputs) in token order; the lanes holding the token's kept
//             choices acquire the flags of the segments the unit reads, then
//             the warp gathers and accumulates exactly as moe_combine does.
//
// A warp that finishes its expert units early starts combining the tokens
// whose rows are complete instead of waiting for the whole expert pass.
// Phase 1 never waits, and the grid is launched cooperatively, so every block
// is resident: every segment a consumer waits for is being produced by a
// running warp. Waits are bounded all the same: a wait that gives up (100 ms)
// raises the device status word, that unit is not written, and the warp
// waits no more.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRBlock = 256;
constexpr int kRWarps = kRBlock / 32;
constexpr unsigned long long kReadyWaitNs = 100ull * 1000 * 1000;   // a wait gives up after 100 ms

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// 16-byte load cached in L2 only: y is written by other SMs during this kernel.
__device__ __forceinline__ uint4 ld_cg_v4(const uint4 *p) { return __ldcg(p); }

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Expert work is cut into segments of kSegTasks 16-byte input pieces per
// lane (one warp unit, as in moe_expert_synthetic); each (kept row, segment)
// has its own flag. A combine unit (token, 32 chunks of 8 outputs) lies inside
// one segment of each row it reads: a segment spans 32 * kSegTasks pieces, a
// multiple of 32 chunks for fp8 (2 chunks per piece) and bf16 (1 per piece).
constexpr int kSegTasks = 4;

__host__ __device__ __forceinline__ int ready_segments(int H, bool fp8) {
    const int pieces = fp8 ? H / 16 : H / 8;
    return (pieces + 32 * kSegTasks - 1) / (32 * kSegTasks);
}

template <int KMAX, bool FP8>
__global__ void __launch_bounds__(kRBlock)
expert_combine_kernel(const uint4 *__restrict__ recv, const float *__restrict__ recv_scale,
                      const int32_t *__restrict__ counts, const float *__restrict__ s, uint4 *__restrict__ y,
                      const int32_t *__restrict__ topk_idx, const float *__restrict__ topk_w,
                      const int32_t *__restrict__ slot, uint4 *__restrict__ out, unsigned *__restrict__ flags,
                      unsigned epoch, int T, int H, int E, int k, int C, unsigned *status) {
    __shared__ int32_t off[kMaxExperts + 1];
    __shared__ int32_t warp_tot[32];
    // fp8: per-warp output buffer of one unit (32 * kSegTasks pieces of 32 bytes)
    extern __shared__ __align__(128) uint4 ready_stage[];
    uint4 *stage = ready_stage + (size_t)(threadIdx.x >> 5) * (32 * kSegTasks * 2);
    kept_row_offsets(counts, E, C, off, warp_tot);
    const int lane = threadIdx.x & 31;
    const unsigned gw = blockIdx.x * kRWarps + (threadIdx.x >> 5), G = gridDim.x * kRWarps;
    const int H8 = H / 8;
    const unsigned pieces = FP8 ? H / 16 : H8, nb = H / 128;
    const int esegs = ready_segments(H, FP8);
    const unsigned rows = off[E];

    // ---- phase 1: every warp computes its (kept row, segment) units; no waiting
    for (UnitWalk wk(gw, G, esegs); wk.row < rows; wk.next()) {
        const int e = expert_of_row(off, E, (int)wk.row);
        const size_t row = (size_t)e * C + (wk.row - off[e]);
        const float se = __ldg(s + e);
        const unsigned first = wk.seg * 32 * kSegTasks;
        const unsigned p0 = first + lane;
        uint4 v[kSegTasks];
        float sc[kSegTasks];
#pragma unroll
        for (int i = 0; i < kSegTasks; ++i) {
            const unsigned pc = p0 + 32 * i;
            if (pc < pieces) {
                v[i] = ld_stream_v4(recv + row * pieces + pc);
                if (FP8) sc[i] = __ldg(recv_scale + row * nb + (pc >> 3));
            }
        }
#pragma unroll
        for (int i = 0; i < kSegTasks; ++i) {
            const unsigned pc = p0 + 32 * i;
            if (pc >= pieces) continue;
            const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            if (FP8) {
                uint32_t ov[8];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float2 lo = e4m3x2_to_float2(wv[h]);
                    const float2 hi = e4m3x2_to_float2(wv[h] >> 16);
                    ov[2 * h] =
                        pack_bf16x2(__fmul_rn(__fmul_rn(lo.x, sc[i]), se), __fmul_rn(__fmul_rn(lo.y, sc[i]), se));
                    ov[2 * h + 1] =
                        pack_bf16x2(__fmul_rn(__fmul_rn(hi.x, sc[i]), se), __fmul_rn(__fmul_rn(hi.y, sc[i]), se));
                }
                // fp8: into this warp's buffer; one bulk copy writes the unit
                stage[2 * (pc - first)] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                stage[2 * (pc - first) + 1] = make_uint4(ov[4], ov[5], ov[6], ov[7]);
            } else {
                uint32_t ov[4];
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    ov[h] = pack_bf16x2(__fmul_rn(bf16_lo(wv[h]), se), __fmul_rn(bf16_hi(wv[h]), se));
                st_v4(y + row * H8 + pc, make_uint4(ov[0], ov[1], ov[2], ov[3]));
            }
        }
        if (FP8) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const unsigned n = min((unsigned)(32 * kSegTasks), pieces - first);
                bulk_s2g(y + row * H8 + 2 * first, stage, n * 32);
                bulk_commit();
                bulk_wait_all();                          // the unit's rows are written ...
                asm volatile("fence.proxy.async.global;" ::: "memory");   // ... and ordered before the flag
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            st_release_u32(flags + row * esegs + wk.seg, epoch);
        }
    }

    // ---- phase 2: combine units in token order, each waiting only for the
    // segments of its own kept rows
    const int csegs = (H8 + 31) / 32;
    const int chunks_per_eseg = 32 * kSegTasks * (FP8 ? 2 : 1);
    bool gave_up = false;                                       // after one timeout, no more waiting
    for (UnitWalk wk(gw, G, csegs); wk.row < (unsigned)T; wk.next()) {
        const unsigned t = wk.row;
        int src_row = -1;
        float w = 0.0f;
        if (lane < k) {
            const int sl = __ldg(slot + (size_t)t * k + lane);
            const int e = __ldg(topk_idx + (size_t)t * k + lane);
            w = __ldg(topk_w + (size_t)t * k + lane);
            if (sl >= 0) src_row = e * C + sl;
        }
        bool ready = true;
        if (src_row >= 0) {
            const unsigned *f = flags + (size_t)src_row * esegs + (wk.seg * 32) / chunks_per_eseg;
            unsigned ns = 32;
            const unsigned long long t0 = global_ns();
            while (ld_acquire_u32(f) != epoch) {
                if (gave_up || global_ns() - t0 > kReadyWaitNs) {
                    ready = false;
                    break;
                }
                __nanosleep(ns);
                if (ns < 1024) ns <<= 1;
            }
        }
        if (!__all_sync(kFull, ready)) {
            gave_up = true;
            if (lane == 0) atomicOr(status, kStatusWaitGaveUp);
            continue;
        }
        const unsigned c = wk.seg * 32 + lane;
        const bool on = c < (unsigned)H8;
        const unsigned kept = __ballot_sync(kFull, src_row >= 0);
        const int n_kept = __popc(kept);
        uint4 v[KMAX];
        unsigned rem = kept;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < n_kept) {                                  // warp-uniform
                const int src = __ffs(rem) - 1;
                rem &= rem - 1;
                const size_t row = (size_t)__shfl_sync(kFull, src_row, src);
                if (on) v[j] = ld_cg_v4(y + row * H8 + c);
            }
        }
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        rem = kept;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < n_kept) {
                const int src = __ffs(rem) - 1;
                rem &= rem - 1;
                const float wj = __shfl_sync(kFull, w, src);
                const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = __fmaf_rn(wj, bf16_lo(wv[i]), acc[2 * i]);
                    acc[2 * i + 1] = __fmaf_rn(wj, bf16_hi(wv[i]), acc[2 * i + 1]);
                }
            }
        }
        if (on)
            st_v4(out + (size_t)t * H8 + c,
                  make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                             pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
    }
}

template <int KMAX, bool FP8>
int launch_expert_combine(const Dims &d, cudaStream_t st, const void *recv, const float *recv_scale,
                          const int32_t *counts, const float *s, void *y, const int32_t *topk_idx,
                          const float *topk_w, const int32_t *slot, void *out, unsigned *flags, unsigned epoch,
                          unsigned *status) {
    auto kernel = expert_combine_kernel<KMAX, FP8>;
    const size_t smem = FP8 ? (size_t)kRWarps * 32 * kSegTasks * 32 : 0;
    static PerContext<int> resident_cache;     // blocks resident on the whole GPU
    const int resident = resident_blocks_cached(resident_cache, kernel, kRBlock, smem);
    int grid = resident;
    if (d.max_blocks > 0 && d.max_blocks < grid) grid = d.max_blocks;
    if (grid < 2) return MOE_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kRBlock);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;        // every block resident: consumers may wait on producers
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, static_cast<const uint4 *>(recv), recv_scale, counts, s,
                           static_cast<uint4 *>(y), topk_idx, topk_w, slot, static_cast<uint4 *>(out), flags, epoch,
                           d.T, d.H, d.E, d.k, d.C, status) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

template <bool FP8>
int dispatch_kmax(const Dims &d, cudaStream_t st, const void *recv, const float *recv_scale, const int32_t *counts,
                  const float *s, void *y, const int32_t *topk_idx, const float *topk_w, const int32_t *slot,
                  void *out, unsigned *flags, unsigned epoch, unsigned *status) {
    if (d.k <= 2)
        return launch_expert_combine<2, FP8>(d, st, recv, recv_scale, counts, s, y, topk_idx, topk_w, slot, out,
                                             flags, epoch, status);
    if (d.k <= 4)
        return launch_expert_combine<4, FP8>(d, st, recv, recv_scale, counts, s, y, topk_idx, topk_w, slot, out,
                                             flags, epoch, status);
    if (d.k <= 8)
        return launch_expert_combine<8, FP8>(d, st, recv, recv_scale, counts, s, y, topk_idx, topk_w, slot, out,
                                             flags, epoch, status);
    return launch_expert_combine<16, FP8>(d, st, recv, recv_scale, counts, s, y, topk_idx, topk_w, slot, out, flags,
                                          epoch, status);
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_ready_flags_bytes(const moe_problem *p) {
    moe::Dims d;
    if (moe::check_problem(p, &d) != MOE_OK) return 0;
    return (size_t)d.E * d.C * moe::ready_segments(d.H, d.dtype == MOE_DTYPE_FP8_E4M3_B128) * sizeof(uint32_t);
}

extern "C" int moe_expert_combine(const moe_problem *p, const void *recv, const float *recv_scale,
                                  const int32_t *counts, const float *s, void *y, const int32_t *topk_idx,
                                  const float *topk_w, const int32_t *slot, void *out, uint32_t *flags,
                                  size_t flags_bytes, uint32_t epoch, void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    const bool fp8 = d.dtype == MOE_DTYPE_FP8_E4M3_B128;
    if (fp8 != (recv_scale != nullptr)) return MOE_ERR_INVALID_ARG;
    if (epoch == 0 || flags == nullptr || flags_bytes < moe_ready_flags_bytes(p)) return MOE_ERR_INVALID_ARG;
    if (d.T == 0) return MOE_OK;
    if (!recv || !counts || !s || !y || !topk_idx || !topk_w || !slot || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(recv, 16) || !aligned(y, 16) || !aligned(out, 16) || !aligned(counts, 4) || !aligned(s, 4) ||
        !aligned(topk_idx, 4) || !aligned(topk_w, 4) || !aligned(slot, 4) || !aligned(flags, 4) ||
        (fp8 && !aligned(recv_scale, 16)))
        return MOE_ERR_INVALID_ARG;
    unsigned *status = device_status_word();
    if (status == nullptr) return MOE_ERR_CUDA;
    cudaStream_t st = as_stream(stream);
    if (fp8)
        return dispatch_kmax<true>(d, st, recv, recv_scale, counts, s, y, topk_idx, topk_w, slot, out, flags, epoch,
                                   status);
    return dispatch_kmax<false>(d, st, recv, nullptr, counts, s, y, topk_idx, topk_w, slot, out, flags, epoch,
                                status);
}
