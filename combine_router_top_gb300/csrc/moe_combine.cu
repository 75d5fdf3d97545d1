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
//   combine: every warp walks its own units (token, 32 chunks of 16 bytes);
//     the routing of a token is held by lanes j < k and broadcast by shuffle.
//   expert: tasks (kept row, 16-byte piece) are numbered over the kept rows
//     only, through an exclusive scan of min(counts[e], C) held in shared
//     memory, so no thread walks empty capacity rows.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBlock = 256;                  // 8 warps; every warp walks its own work units
constexpr int kWarps = kBlock / 32;

// Lane j < k of a warp holds choice j of token t: slot, expert, weight.
struct Choice {
    int s, e;
    float w;
};
__device__ __forceinline__ Choice load_choice(int t, int k, const int32_t *__restrict__ topk_idx,
                                              const float *__restrict__ topk_w, const int32_t *__restrict__ slot) {
    Choice c{-1, 0, 0.0f};
    const int lane = threadIdx.x & 31;
    if (lane < k) {
        c.s = __ldg(slot + (size_t)t * k + lane);
        c.e = __ldg(topk_idx + (size_t)t * k + lane);
        c.w = __ldg(topk_w + (size_t)t * k + lane);
    }
    return c;
}

// Unit = (token, 32 consecutive 16-byte chunks of its row): lane l owns chunk
// 32*seg + l. The warp broadcasts each kept choice (ascending j) by shuffle,
// issues all gathers, then accumulates in fp32 in ascending j. The next
// unit's routing is loaded before the current unit's gathers are issued.
template <int KMAX>
__global__ void __launch_bounds__(kBlock, KMAX <= 8 ? 4 : 2)
combine_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ topk_idx,
               const float *__restrict__ topk_w, const int32_t *__restrict__ slot,
               uint4 *__restrict__ out, int T, int H8, int k, int C, int segs) {
    const int lane = threadIdx.x & 31;
    const long long n_units = (long long)T * segs;
    const long long stride = (long long)gridDim.x * kWarps;
    long long u = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (u >= n_units) return;                                  // warp-uniform
    Choice cur = load_choice((int)(u / segs), k, topk_idx, topk_w, slot);
    for (; u < n_units; u += stride) {
        const long long un = u + stride;
        Choice nxt{-1, 0, 0.0f};
        if (un < n_units) nxt = load_choice((int)(un / segs), k, topk_idx, topk_w, slot);
        const int t = (int)(u / segs);
        const int c = (int)(u % segs) * 32 + lane;
        const bool on = c < H8;
        const long long my_row = ((long long)cur.e * C + (cur.s >= 0 ? cur.s : 0)) * H8;
        const unsigned kept = __ballot_sync(kFull, cur.s >= 0);
        const int n_kept = __popc(kept);
        uint4 v[KMAX];
        unsigned rem = kept;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < n_kept) {                                  // warp-uniform
                const int src = __ffs(rem) - 1;
                rem &= rem - 1;
                const long long row = __shfl_sync(kFull, my_row, src);
                if (on) v[j] = ld_stream_v4(y + row + c);
            }
        }
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        rem = kept;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < n_kept) {                                  // warp-uniform
                const int src = __ffs(rem) - 1;
                rem &= rem - 1;
                const float w = __shfl_sync(kFull, cur.w, src);
                const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = __fmaf_rn(w, bf16_lo(wv[i]), acc[2 * i]);
                    acc[2 * i + 1] = __fmaf_rn(w, bf16_hi(wv[i]), acc[2 * i + 1]);
                }
            }
        }
        if (on) {
            st_v4(out + (size_t)t * H8 + c,
                  make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                             pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
        }
        cur = nxt;
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

// Expert of kept row p: the last e with off[e] <= p (off is non-decreasing).
__device__ __forceinline__ int expert_of_row(const int32_t *off, int E, int p) {
    int lo = 0, hi = E;        // off[lo] <= p < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= p) lo = mid; else hi = mid;
    }
    return lo;
}

constexpr int kExpertBatch = 4;   // tasks per thread whose loads are in flight together

// Synthetic expert, bf16 rows. Tasks (kept row, 16-byte chunk) are numbered
// row-major over the kept rows; consecutive threads take consecutive tasks
// (coalesced), a thread issues kExpertBatch loads before its first store.
__global__ void __launch_bounds__(kBlock)
expert_bf16_kernel(const uint4 *__restrict__ recv, const int32_t *__restrict__ counts,
                   const float *__restrict__ s, uint4 *__restrict__ y, int E, int C, int H8) {
    __shared__ int32_t off[kMaxExperts + 1];
    __shared__ int32_t warp_tot[32];
    kept_row_offsets(counts, E, C, off, warp_tot);
    const long long total = (long long)off[E] * H8;
    const long long stride = (long long)gridDim.x * kBlock;
    for (long long g0 = (long long)blockIdx.x * kBlock + threadIdx.x; g0 < total; g0 += stride * kExpertBatch) {
        uint4 v[kExpertBatch];
        long long at[kExpertBatch];
        float se[kExpertBatch];
#pragma unroll
        for (int i = 0; i < kExpertBatch; ++i) {
            const long long g = g0 + i * stride;
            at[i] = -1;
            if (g < total) {
                const int p = (int)(g / H8);
                const int e = expert_of_row(off, E, p);
                at[i] = ((long long)e * C + (p - off[e])) * H8 + (g % H8);
                se[i] = __ldg(s + e);
                v[i] = ld_stream_v4(recv + at[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < kExpertBatch; ++i) {
            if (at[i] >= 0) {
                const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t ov[4];
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    ov[h] = pack_bf16x2(__fmul_rn(bf16_lo(wv[h]), se[i]), __fmul_rn(bf16_hi(wv[h]), se[i]));
                st_v4(y + at[i], make_uint4(ov[0], ov[1], ov[2], ov[3]));
            }
        }
    }
}

// e4m3 code -> float, exact (every e4m3 value is a binary16 and a binary32 value).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
    return __half2float(*reinterpret_cast<const __half *>(&h));
}

// Synthetic expert, fp8 rows: a task is 16 codes (16 bytes in, 32 bytes of bf16 out).
__global__ void __launch_bounds__(kBlock)
expert_fp8_kernel(const uint4 *__restrict__ recv_q, const float *__restrict__ recv_scale,
                  const int32_t *__restrict__ counts, const float *__restrict__ s,
                  uint4 *__restrict__ y, int E, int C, int H) {
    __shared__ int32_t off[kMaxExperts + 1];
    __shared__ int32_t warp_tot[32];
    kept_row_offsets(counts, E, C, off, warp_tot);
    const int n_tasks = H / 16, nb = H / 128;
    const long long total = (long long)off[E] * n_tasks;
    const long long stride = (long long)gridDim.x * kBlock;
    for (long long g0 = (long long)blockIdx.x * kBlock + threadIdx.x; g0 < total; g0 += stride * kExpertBatch) {
        uint4 q[kExpertBatch];
        float sc[kExpertBatch], se[kExpertBatch];
        long long row[kExpertBatch];
        int task[kExpertBatch];
#pragma unroll
        for (int i = 0; i < kExpertBatch; ++i) {
            const long long g = g0 + i * stride;
            row[i] = -1;
            if (g < total) {
                const int p = (int)(g / n_tasks);
                task[i] = (int)(g % n_tasks);
                const int e = expert_of_row(off, E, p);
                row[i] = (long long)e * C + (p - off[e]);
                se[i] = __ldg(s + e);
                q[i] = ld_stream_v4(recv_q + row[i] * n_tasks + task[i]);
                sc[i] = __ldg(recv_scale + row[i] * nb + (task[i] >> 3));
            }
        }
#pragma unroll
        for (int i = 0; i < kExpertBatch; ++i) {
            if (row[i] >= 0) {
                const uint32_t qw[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
                uint32_t ov[8];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t two = qw[w] >> (16 * h);
                        const float a = __fmul_rn(__fmul_rn(e4m3_to_float(two & 0xFFu), sc[i]), se[i]);
                        const float b = __fmul_rn(__fmul_rn(e4m3_to_float((two >> 8) & 0xFFu), sc[i]), se[i]);
                        ov[2 * w + h] = pack_bf16x2(a, b);
                    }
                }
                uint4 *o = y + row[i] * (H / 8) + 2 * task[i];
                st_v4(o, make_uint4(ov[0], ov[1], ov[2], ov[3]));
                st_v4(o + 1, make_uint4(ov[4], ov[5], ov[6], ov[7]));
            }
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
        static int resident = resident_blocks(expert_fp8_kernel, kBlock);
        const long long tasks = max_rows * (d.H / 16);
        const int grid = persistent_grid((tasks + (long long)kBlock * kExpertBatch - 1) / ((long long)kBlock * kExpertBatch),
                                         resident, d.max_blocks);
        expert_fp8_kernel<<<grid, kBlock, 0, st>>>(static_cast<const uint4 *>(recv), recv_scale, counts, s,
                                                   static_cast<uint4 *>(y), d.E, d.C, d.H);
    } else {
        static int resident = resident_blocks(expert_bf16_kernel, kBlock);
        const long long tasks = max_rows * (d.H / 8);
        const int grid = persistent_grid((tasks + (long long)kBlock * kExpertBatch - 1) / ((long long)kBlock * kExpertBatch),
                                         resident, d.max_blocks);
        expert_bf16_kernel<<<grid, kBlock, 0, st>>>(static_cast<const uint4 *>(recv), counts, s,
                                                    static_cast<uint4 *>(y), d.E, d.C, d.H / 8);
    }
    return launch_status();
}

namespace {
template <int KMAX>
int launch_combine(const moe::Dims &d, cudaStream_t st, const uint4 *y, const int32_t *idx, const float *w,
                   const int32_t *slot, uint4 *out) {
    using namespace moe;
    static int resident = resident_blocks(combine_kernel<KMAX>, kBlock);
    const int H8 = d.H / 8;
    const int segs = (H8 + 31) / 32;
    const long long units = (long long)d.T * segs;
    const int grid = persistent_grid((units + kWarps - 1) / kWarps, resident, d.max_blocks);
    combine_kernel<KMAX><<<grid, kBlock, 0, st>>>(y, idx, w, slot, out, d.T, H8, d.k, d.C, segs);
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
