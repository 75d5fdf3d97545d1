// moe_gemm.cu -- grouped fp8 GEMM on the dispatch layout, on the tcgen05
// tensor cores: the experts that consume the block-scaled tokens of
// "Efficient and portable mixture-of-experts communication" (§Dispatch), with
// random weights standing in for trained ones.
//
//   y[e][r][n] = bf16( sum_b a_scale[e][r][b] * w_scale[e][n/128][b]
//                      * sum_{i in block b} q[e][r][i] * w[e][n][i] )
//
// for r < min(counts[e], C), n < H, blocks b of 128 inputs. q and w are e4m3.
//
// A persistent grid (one CTA per SM) walks the list of 128 x 256 output tiles
// (128 rows of one expert, 256 outputs) that hold kept rows; each CTA builds
// that list from counts in shared memory. In each CTA:
//   warp 0       one lane issues the TMA loads of the A (rows, 128 x 128 B) and
//                B (weights, 256 x 128 B) tiles, 128-byte swizzled, into a
//                4-stage ring;
//   warp 1       allocates all 512 TMEM columns; one lane issues, per block b
//                of 128 inputs, four tcgen05.mma kind::f8f6f4 (128 x 256 x 32)
//                into one of two 256-column fp32 accumulators, fresh for every b;
//   warps 2..17  read the block's accumulator (tcgen05.ld), release it, and add
//                it times a_scale[r][b] * w_scale[n/128][b] into 64 registers per
//                thread (four warps per 32-lane TMEM quadrant, 64 columns each);
//                after a tile's last block they round to bf16 and store its rows
//                while the tensor cores start on the next tile;
//   warps 18, 19 idle: registers are granted per four warps, so 20 warps of
//                96 registers fit where 18 warps of 112 do not.
// The fp32 scales of both operands change with b, so the per-block partial
// sums are scaled outside the tensor core (the hardware block-scaled MMA
// takes power-of-two scales per 32 elements, not these).
//
// Every mbarrier wait is bounded. A wait that gives up raises the device
// status word and a CTA-wide abort flag; the CTA then drains its copies and
// MMAs in flight (again bounded), frees its TMEM and returns.
#include "moe_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

namespace moe {
namespace {

constexpr int kBM = 128;                         // rows of one MMA (and of one TMA load of A)
constexpr int kBN = 256;                         // outputs per tile (128 or 256)
constexpr int kBK = 128;                         // bytes of input per row and block: 128 e4m3 (one scale) or 64 bf16
constexpr int kNumAcc = 512 / kBN;               // fp32 accumulators that fill the 512 TMEM columns
constexpr int kGemmEpiWarps = 16;
constexpr int kGemmThreads = 32 * (2 + kGemmEpiWarps + 2);   // + 2 idle warps: 20 warps, 96 registers each
constexpr uint32_t kATileBytes = kBM * kBK;      // 16 KB
constexpr uint32_t kBTileBytes = kBN * kBK;      // 32 KB
constexpr uint32_t kGemmTmemCols = kNumAcc * kBN;   // all 512 columns
constexpr int kEpiCols = kBN / 4;                // columns per promotion warp (4 per TMEM lane quadrant)

// Tile geometry. Tiles of 128 rows (one MMA row block): stages of A 16 KB +
// B 32 KB, four of them. WIDE (bf16 only): tiles of up to 256 rows, two
// 128-row MMAs sharing each B tile, so a third fewer operand bytes per FLOP
// and each weight tile read once per pair of row blocks; stages of A 32 KB +
// B 32 KB, three of them. Chosen on the host for experts that average 512
// rows or more; with about 256 rows per expert the narrow tiles are faster
// (the wide tile's epilogue cannot overlap the next tile, since its two
// halves fill TMEM, and its ragged one-half remainders lose the fourth stage).
template <bool WIDE>
struct GemmGeom {
    static constexpr int kTileRows = WIDE ? 2 * kBM : kBM;
    static constexpr uint32_t kARegion = (uint32_t)kTileRows * kBK;
    static constexpr uint32_t kStageBytes = kARegion + kBTileBytes;
    static constexpr int kStages = (196 * 1024) / kStageBytes;
};
constexpr size_t kGemmSmemBytes =
    (GemmGeom<false>::kStages * GemmGeom<false>::kStageBytes > GemmGeom<true>::kStages * GemmGeom<true>::kStageBytes
         ? GemmGeom<false>::kStages * GemmGeom<false>::kStageBytes
         : GemmGeom<true>::kStages * GemmGeom<true>::kStageBytes) +
    1024;                                        // + alignment slack
constexpr int kWideMinRows = 512;               // mean kept rows per expert from which bf16 takes wide tiles
constexpr unsigned kGemmPollLimit = 1u << 20;

// Shared-memory matrix descriptor of a K-major tile whose rows are 128 bytes,
// 128-byte swizzled (as TMA writes it): 8-row swizzle atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);           // start address
    d |= (uint64_t)(1024u >> 4) << 32;                           // stride byte offset
    d |= (uint64_t)1 << 46;                                      // descriptor version
    d |= (uint64_t)2 << 61;                                      // 128-byte swizzle
    return d;
}

// Instruction descriptors, both operands K-major, fp32 accumulator, M = 128,
// N = kBN: kind::f8f6f4 with A and B e4m3 (format 0), kind::f16 with A and B
// bf16 (format 1).
constexpr uint32_t kIdescShape = (1u << 4)                          // D format f32
                                 | ((uint32_t)(kBN >> 3) << 17)     // N / 8
                                 | ((uint32_t)(kBM >> 4) << 24);    // M / 16
constexpr uint32_t kIdescF8 = kIdescShape | (0u << 7) | (0u << 10);
constexpr uint32_t kIdescBF16 = kIdescShape | (1u << 7) | (1u << 10);

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// One MMA of 32 bytes of K per row: 32 e4m3 (kind::f8f6f4) or 16 bf16 (kind::f16).
template <bool FP8>
__device__ __forceinline__ void mma_k32b(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t accumulate) {
    if constexpr (FP8)
        asm volatile(
            "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(tmem_d),
            "l"(a), "l"(b), "r"(kIdescF8), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem_d),
            "l"(a), "l"(b), "r"(kIdescBF16), "r"(accumulate)
            : "memory");
}

// Arrives once on the mbarrier when every MMA this thread issued so far is complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded wait on phase `parity`; gives up early once another role aborted.
__device__ __forceinline__ bool gemm_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    for (unsigned i = 0; i < kGemmPollLimit; ++i) {
        uint32_t done;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done)
                     : "r"(bar), "r"(parity)
                     : "memory");
        if (done) return true;
        if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
    *abort_flag = 1;
    return false;
}

// The tiles holding kept rows, in the order (expert, output tile, row tile):
// s_first[e] = index of expert e's first tile, s_first[E] = the total.
struct TileList {
    const int *first, *kept;
    int E, n_tiles, tile_rows;
    __device__ __forceinline__ void decode(int t, int &e, int &nt, int &mt, int &rows) const {
        int lo = 0, hi = E;                          // first[lo] <= t < first[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (first[mid] <= t) lo = mid; else hi = mid;
        }
        e = lo;
        const int mtiles = (first[e + 1] - first[e]) / n_tiles;
        const int local = t - first[e];
        nt = local / mtiles;
        mt = local - nt * mtiles;
        rows = min(kept[e] - mt * tile_rows, tile_rows);
    }
};

// FP8: per-block promotion (fresh accumulator per block of 128 inputs, scaled
// in registers). BF16: no scales, so one accumulator holds a whole tile and
// the promotion warps only convert and store it.
template <bool FP8, bool WIDE>
__global__ void __launch_bounds__(kGemmThreads, 1)
expert_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                       const float *__restrict__ a_scale, const int32_t *__restrict__ counts,
                       const float *__restrict__ w_scale, uint16_t *__restrict__ y, int H, int C, int E,
                       unsigned *status) {
    static_assert(!(FP8 && WIDE), "wide tiles are for bf16 rows");
    constexpr int kStages = GemmGeom<WIDE>::kStages, TR = GemmGeom<WIDE>::kTileRows;
    constexpr uint32_t kStageBytes = GemmGeom<WIDE>::kStageBytes, kARegion = GemmGeom<WIDE>::kARegion;
    extern __shared__ uint8_t gemm_smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
    __shared__ __align__(8) uint64_t tfull_bar[kNumAcc], tempty_bar[kNumAcc];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_first[kMaxExperts + 1];
    __shared__ int s_kept[kMaxExperts];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = FP8 ? H / kBK : H / (kBK / 2), nb = H / 128;
    const int kb_elems = FP8 ? kBK : kBK / 2;           // inputs per block (TMA x coordinate step)
    const int n_tiles = (H + kBN - 1) / kBN;
    const uint32_t smem0 = (smem_u32(gemm_smem_raw) + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < kNumAcc; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], kGemmEpiWarps);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    pdl_wait();                                   // counts and the dispatched rows are final from here on
    if (warp == 0) {                              // tile list: lane l scans experts [l*per, l*per + per)
        const int per = (E + 31) / 32;
        int sum = 0;
        for (int e = lane * per; e < min(E, lane * per + per); ++e) {
            const int kept = min(__ldg(counts + e), C);
            s_kept[e] = kept;
            sum += (kept + TR - 1) / TR * n_tiles;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int e = lane * per; e < min(E, lane * per + per); ++e) {
            s_first[e] = run;
            run += (s_kept[e] + TR - 1) / TR * n_tiles;
        }
        if (lane == 31) s_first[E] = incl;
    }
    __syncthreads();
    const int total = s_first[E];
    if ((int)blockIdx.x >= total) {               // no tile for this CTA
        pdl_launch_dependents();
        return;
    }
    const TileList tiles{s_first, s_kept, E, n_tiles, TR};
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kGemmTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    uint32_t issued = 0;                          // producer: stages loaded
    uint32_t last_tfull = 0, last_tfull_par = 0;  // MMA issuer: the last accumulator commit
    bool committed = false;
    if (warp == 0) {
        if (lane == 0) {
            uint32_t g = 0;
            for (int t = blockIdx.x; t < total && !s_abort; t += gridDim.x) {
                int e, nt, mt, rows;
                tiles.decode(t, e, nt, mt, rows);
                const int row_a = e * C + mt * TR;
                const int row_b = e * H + nt * kBN;
                const int a_boxes = rows > kBM ? 2 : 1;      // 128-row A loads this tile needs
                for (int kb = 0; kb < nkb; ++kb, ++g) {
                    const int s = g % kStages;
                    if (g >= kStages && !gemm_wait(smem_u32(&empty_bar[s]), ((g / kStages) + 1) & 1, &s_abort))
                        break;
                    const uint32_t sa = smem0 + s * kStageBytes, sb = sa + kARegion;
                    mbar_expect_tx(&full_bar[s], a_boxes * kATileBytes + kBTileBytes);
                    for (int h = 0; h < a_boxes; ++h)
                        tma_load_2d(sa + h * kATileBytes, &map_a, smem_u32(&full_bar[s]), kb * kb_elems,
                                    row_a + h * kBM);
                    tma_load_2d(sb, &map_b, smem_u32(&full_bar[s]), kb * kb_elems, row_b);
                    issued = g + 1;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t g = 0;                       // blocks consumed (stage ring)
            uint32_t a = 0;                       // accumulators used: FP8 one per block, BF16 one per tile
            uint32_t uses[kNumAcc] = {};          // WIDE: commits of each TMEM half (accumulator)
            int next_h = 0;                       // WIDE: the half a one-half tile takes next
            bool stop = false;
            for (int t = blockIdx.x; t < total && !stop && !s_abort; t += gridDim.x) {
                // WIDE: the tile takes halves h0 .. h0 + halves - 1 (one per 128 rows);
                // one-half tiles alternate, as the issuer and the epilogue both count
                int halves = 1, h0 = 0;
                if constexpr (WIDE) {
                    int e, nt, mt, rows;
                    tiles.decode(t, e, nt, mt, rows);
                    halves = rows > kBM ? 2 : 1;
                    h0 = halves == 2 ? 0 : next_h;
                    next_h = halves == 2 ? 0 : 1 - h0;
                }
                for (int kb = 0; kb < nkb; ++kb, ++g) {
                    const int s = g % kStages;
                    if (!gemm_wait(smem_u32(&full_bar[s]), (g / kStages) & 1, &s_abort)) { stop = true; break; }
                    const uint32_t sa = smem0 + s * kStageBytes, sb = sa + kARegion;
                    if constexpr (FP8) {
                        const int buf = a % kNumAcc;
                        if (a >= kNumAcc &&
                            !gemm_wait(smem_u32(&tempty_bar[buf]), ((a / kNumAcc) + 1) & 1, &s_abort)) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem + buf * kBN;
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            mma_k32b<FP8>(d, umma_desc_sw128(sa + 32 * k), umma_desc_sw128(sb + 32 * k),
                                          k > 0 ? 1u : 0u);
                        mma_commit(smem_u32(&empty_bar[s]));
                        mma_commit(smem_u32(&tfull_bar[buf]));
                        last_tfull = smem_u32(&tfull_bar[buf]);
                        last_tfull_par = (a / kNumAcc) & 1;
                        committed = true;
                        ++a;
                    } else if constexpr (!WIDE) {
                        // one accumulator per tile, alternating (a counts tiles)
                        const int buf = a % kNumAcc;
                        if (kb == 0 && a >= kNumAcc &&
                            !gemm_wait(smem_u32(&tempty_bar[buf]), ((a / kNumAcc) + 1) & 1, &s_abort)) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem + buf * kBN;
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            mma_k32b<FP8>(d, umma_desc_sw128(sa + 32 * k), umma_desc_sw128(sb + 32 * k),
                                          (k > 0 || kb > 0) ? 1u : 0u);
                        mma_commit(smem_u32(&empty_bar[s]));
                        if (kb == nkb - 1) {
                            mma_commit(smem_u32(&tfull_bar[buf]));
                            last_tfull = smem_u32(&tfull_bar[buf]);
                            last_tfull_par = (a / kNumAcc) & 1;
                            committed = true;
                            ++a;
                        }
                    } else {
                        if (kb == 0) {            // the halves' previous tiles must have been read
                            for (int hh = 0; hh < halves && !stop; ++hh) {
                                const int h = h0 + hh;
                                if (uses[h] > 0 &&
                                    !gemm_wait(smem_u32(&tempty_bar[h]), (uses[h] - 1) & 1, &s_abort))
                                    stop = true;
                            }
                            if (stop) break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            for (int hh = 0; hh < halves; ++hh)
                                mma_k32b<FP8>(tmem + (h0 + hh) * kBN, umma_desc_sw128(sa + hh * kATileBytes + 32 * k),
                                              umma_desc_sw128(sb + 32 * k), (k > 0 || kb > 0) ? 1u : 0u);
                        mma_commit(smem_u32(&empty_bar[s]));
                        if (kb == nkb - 1) {
                            for (int hh = 0; hh < halves; ++hh) {
                                const int h = h0 + hh;
                                mma_commit(smem_u32(&tfull_bar[h]));
                                last_tfull = smem_u32(&tfull_bar[h]);
                                last_tfull_par = uses[h] & 1;
                                ++uses[h];
                            }
                            committed = true;
                        }
                    }
                }
            }
        }
    } else if (warp < 2 + kGemmEpiWarps) {
        const int quad = warp & 3;                        // TMEM lanes this warp may read
        const int cg = (warp - 2) >> 2;                   // which quarter of the tile's columns
        const int r = quad * 32 + lane;                   // row within a 128-row block of the tile
        uint32_t g = 0;
        uint32_t uses[kNumAcc] = {};                      // WIDE: reads of each TMEM half, as the issuer counts
        int next_h = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
            int e, nt, mt, rows;
            tiles.decode(t, e, nt, mt, rows);
            const int col0 = nt * kBN + cg * kEpiCols;         // this warp's first output column
            const int nblk = col0 / 128;                       // its 128-output weight-scale block
            const bool live = r < rows && col0 < H;
            const size_t grow = (size_t)e * C + (size_t)mt * TR + r;
            if constexpr (!FP8 && !WIDE) {
                // the tile's whole sum is in one accumulator: convert and store
                const int buf = g % kNumAcc;
                int got = 0;
                if (lane == 0) got = gemm_wait(smem_u32(&tfull_bar[buf]), (g / kNumAcc) & 1, &s_abort) ? 1 : 0;
                if (!__shfl_sync(kFull, got, 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + buf * kBN + cg * kEpiCols;
                uint4 *dst = reinterpret_cast<uint4 *>(y + grow * H + (size_t)nt * kBN + cg * kEpiCols);
#pragma unroll
                for (int c = 0; c < kEpiCols / 16; ++c) {
                    uint32_t v[16];
                    tmem_ld16(taddr + 16 * c, v);
                    tmem_ld_wait();
                    if (live) {
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            dst[2 * c + q] = make_uint4(
                                pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty_bar[buf]);
                ++g;
                continue;
            }
            if constexpr (WIDE) {
                // the tile's whole sum is in one TMEM half per 128 rows: convert and store
                const int halves = rows > kBM ? 2 : 1;
                const int h0 = halves == 2 ? 0 : next_h;
                next_h = halves == 2 ? 0 : 1 - h0;
                for (int hh = 0; hh < halves; ++hh) {
                    const int h = h0 + hh;
                    int got = 0;
                    if (lane == 0) got = gemm_wait(smem_u32(&tfull_bar[h]), uses[h] & 1, &s_abort) ? 1 : 0;
                    if (!__shfl_sync(kFull, got, 0)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const bool live_h = hh * kBM + r < rows && col0 < H;
                    const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + h * kBN + cg * kEpiCols;
                    uint4 *dst = reinterpret_cast<uint4 *>(y + (grow + (size_t)hh * kBM) * H + (size_t)nt * kBN +
                                                           cg * kEpiCols);
#pragma unroll
                    for (int c = 0; c < kEpiCols / 16; ++c) {
                        uint32_t v[16];
                        tmem_ld16(taddr + 16 * c, v);
                        tmem_ld_wait();
                        if (live_h) {
#pragma unroll
                            for (int q = 0; q < 2; ++q)
                                dst[2 * c + q] = make_uint4(
                                    pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                                    pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                    pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                    pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty_bar[h]);
                    ++uses[h];
                }
                continue;
            }
            const float *sa_row = a_scale + grow * nb;
            const float *sw_row = w_scale + ((size_t)e * nb + (live ? nblk : 0)) * nb;
            float acc[kEpiCols];
#pragma unroll
            for (int j = 0; j < kEpiCols; ++j) acc[j] = 0.0f;
            float f_next = live ? __ldg(sa_row) * __ldg(sw_row) : 0.0f;
            for (int kb = 0; kb < nkb; ++kb, ++g) {
                const int buf = g % kNumAcc;
                const float f = f_next;
                if (kb + 1 < nkb) f_next = live ? __ldg(sa_row + kb + 1) * __ldg(sw_row + kb + 1) : 0.0f;
                int got = 0;
                if (lane == 0) got = gemm_wait(smem_u32(&tfull_bar[buf]), (g / kNumAcc) & 1, &s_abort) ? 1 : 0;
                if (!__shfl_sync(kFull, got, 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + buf * kBN + cg * kEpiCols;
#pragma unroll
                for (int c = 0; c < kEpiCols / 16; ++c) {     // 16 columns at a time
                    uint32_t v[16];
                    tmem_ld16(taddr + 16 * c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[c * 16 + j] = fmaf(__uint_as_float(v[j]), f, acc[c * 16 + j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty_bar[buf]);
            }
            if (ok && live) {
                uint4 *dst = reinterpret_cast<uint4 *>(y + grow * H + (size_t)nt * kBN + cg * kEpiCols);
#pragma unroll
                for (int c = 0; c < kEpiCols / 8; ++c)
                    dst[c] = make_uint4(pack_bf16x2(acc[8 * c + 0], acc[8 * c + 1]),
                                        pack_bf16x2(acc[8 * c + 2], acc[8 * c + 3]),
                                        pack_bf16x2(acc[8 * c + 4], acc[8 * c + 5]),
                                        pack_bf16x2(acc[8 * c + 6], acc[8 * c + 7]));
            }
        }
    }
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (s_abort) {
        // drain: the loads and MMAs this CTA started must land before its
        // shared memory and TMEM are released
        volatile int no_abort = 0;
        if (warp == 0 && lane == 0) {
            atomicOr(status, kStatusWaitGaveUp);
            for (uint32_t g = (issued > kStages ? issued - kStages : 0); g < issued; ++g)
                gemm_wait(smem_u32(&full_bar[g % kStages]), (g / kStages) & 1, &no_abort);
        }
        if (warp == 1 && lane == 0 && committed)   // the last commit: every MMA before it is complete with it
            gemm_wait(last_tfull, last_tfull_par, &no_abort);
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kGemmTmemCols)
                     : "memory");
    }
}

// ---- host: tensor maps --------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A [rows][cols] matrix of 1- or 2-byte elements read in tiles of box_rows x
// 128 bytes, 128-byte swizzled; rows past the end read as zero.
bool encode_tile_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     int elem_bytes) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(kBK / elem_bytes), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8, bool WIDE>
int launch_gemm(const Dims &d, const void *recv, const float *recv_scale, const int32_t *counts, const void *w,
                const float *w_scale, void *y, void *stream) {
    const int eb = FP8 ? 1 : 2;
    CUtensorMap map_a, map_b;
    if (!encode_tile_map(&map_a, recv, (uint64_t)d.E * d.C, (uint64_t)d.H, kBM, eb) ||
        !encode_tile_map(&map_b, w, (uint64_t)d.E * d.H, (uint64_t)d.H, kBN, eb))
        return MOE_ERR_CUDA;
    unsigned *status = device_status_word();
    if (status == nullptr) return MOE_ERR_CUDA;
    static PerContext<int> smem_done;
    if (!set_smem_once(smem_done, expert_gemm_kernel<FP8, WIDE>, (int)kGemmSmemBytes)) return MOE_ERR_CUDA;
    int grid = sm_count();                        // persistent: one CTA per SM
    if (d.max_blocks > 0 && d.max_blocks < grid) grid = d.max_blocks;
    if (launch_pdl_smem(expert_gemm_kernel<FP8, WIDE>, grid, kGemmThreads, kGemmSmemBytes, as_stream(stream), map_a,
                        map_b, recv_scale, counts, w_scale, static_cast<uint16_t *>(y), d.H, d.C, d.E, status) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_expert_gemm_fp8(const moe_problem *p, const void *recv_q, const float *recv_scale,
                                   const int32_t *counts, const void *w_q, const float *w_scale, void *y,
                                   void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    if (d.dtype != MOE_DTYPE_FP8_E4M3_B128) return MOE_ERR_UNSUPPORTED;
    if (!recv_q || !recv_scale || !counts || !w_q || !w_scale || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned(recv_q, 16) || !aligned(w_q, 16) || !aligned(y, 16) || !aligned(recv_scale, 4) ||
        !aligned(w_scale, 4) || !aligned(counts, 4))
        return MOE_ERR_INVALID_ARG;
    return launch_gemm<true, false>(d, recv_q, recv_scale, counts, w_q, w_scale, y, stream);
}

extern "C" int moe_expert_gemm_bf16(const moe_problem *p, const void *recv_x, const int32_t *counts,
                                    const void *w, void *y, void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    if (d.dtype != MOE_DTYPE_BF16 || d.H % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (!recv_x || !counts || !w || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned(recv_x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(counts, 4))
        return MOE_ERR_INVALID_ARG;
    // wide tiles when the experts average kWideMinRows kept rows or more
    // (counts are on the device: the mean follows from the problem's sizes)
    const long long mean_rows = std::min<long long>((long long)d.T * d.k / d.E, (long long)d.C);
    if (mean_rows >= kWideMinRows) return launch_gemm<false, true>(d, recv_x, nullptr, counts, w, nullptr, y, stream);
    return launch_gemm<false, false>(d, recv_x, nullptr, counts, w, nullptr, y, stream);
}
