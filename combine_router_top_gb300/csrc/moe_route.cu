// moe_route.cu -- steps 1 and 2 of the path: router top-k with renormalised
// softmax weights, then the per-expert histogram, its exclusive scan and the
// slot of every (token, choice) pair.
//
// [PMC §Introduction]: the router's probability distribution picks the top-K
// experts and weights their outputs. [PMC §Dispatch]: a counting warp tallies
// tokens per destination expert. [PMC §Portable kernels]: a fixed per-expert
// bound lets every sender compute a unique destination address.
//
// Two launches (the second a programmatic dependent of the first, so its
// launch latency hides behind the first), no atomics that decide an order.
// Small batches (T <= kRouteSmallMaxTokens, every decode batch):
//   K1 route_topk_small: one 256-thread CTA per tile of 8 tokens, one warp per
//      token (warp_topk: k rounds of a warp arg-max). Each chosen expert sets
//      the token's bit in a per-expert shared-memory mask: a pair's rank within
//      the tile is the popcount of the lower bits, the tile's count of expert e
//      the popcount, stored as byte cnt8[e][tile].
//   K2 route_slots_small: block 0 forms counts, offsets, rank_counts and
//      dropped from the byte counts; block 1 + b takes tile b, one warp per
//      token: the pairs of e_j in earlier tiles are the first b bytes of row
//      e_j, summed by the warp in one 16-byte load per lane and a shuffle sum.
// Large batches: the same top-k on tiles of 32 tokens (route_topk_tile) with
// 32-bit counts per (tile, expert), then route_finalize, one CTA per tile,
// adds the earlier tiles' counts; the last CTA forms the totals. That sum
// grows with the square of the batch; once it is large (route_two_level), two
// more launches between them make it a two-level scan: route_chunk_sums adds
// each chunk of kChunkTiles tiles, route_chunk_scan turns the chunk sums into
// exclusive bases, and route_finalize adds to its chunk's base only the tiles
// before it in its own chunk.
#include "moe_internal.cuh"

namespace moe {
namespace {

// Top-k of one token by its warp. Lane l owns experts [l*V, l*V + V) (clipped
// to E) of the token's logit row. k rounds of a warp arg-max: redux.sync max on
// an order-preserving 32-bit key (-0 folded onto +0, NaN below every number),
// then a ballot picks the lowest tied lane, which holds the lowest index.
// Lane j < k returns choice j: its expert and its weight
// w_j = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0) (expf, one IEEE division).
template <int V>
__device__ __forceinline__ void warp_topk(const float *__restrict__ row, int E, int k, int lane, int &my_e,
                                          float &my_w) {
    const int e0 = lane * V;
    uint32_t key[V];
    if ((V % 4) == 0 && (E % 4) == 0 && e0 + V <= E) {
#pragma unroll
        for (int i = 0; i < V; i += 4) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(row + e0 + i));
            key[i] = logit_key(f.x);
            key[i + 1] = logit_key(f.y);
            key[i + 2] = logit_key(f.z);
            key[i + 3] = logit_key(f.w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) key[i] = (e0 + i < E) ? logit_key(__ldg(row + e0 + i)) : 0u;
    }

    uint32_t my_key = 0, top_key = 0;
    my_e = 0;
    for (int j = 0; j < k; ++j) {
        // the lane's best remaining candidate (lowest index among equals)
        uint32_t best = 0;
        int bi = 0;
#pragma unroll
        for (int i = 0; i < V; ++i)
            if (key[i] > best) { best = key[i]; bi = i; }
        const uint32_t m = __reduce_max_sync(kFull, best);
        // lanes own ascending index ranges: the lowest tied lane holds the lowest index
        const int wl = __ffs(__ballot_sync(kFull, best == m)) - 1;
        const int e = __shfl_sync(kFull, e0 + bi, wl);
        if (lane == wl) {
#pragma unroll
            for (int i = 0; i < V; ++i)
                if (i == bi) key[i] = 0u;
        }
        if (lane == j) { my_key = m; my_e = e; }
        if (j == 0) top_key = m;
    }

    float ex = 0.0f;
    if (lane < k) ex = expf(key_logit(my_key) - key_logit(top_key));
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    my_w = __fdiv_rn(ex, sum);
}

// Large batches, K1: one CTA per tile of 32 tokens, one warp per token. Each
// chosen expert sets the token's bit in a per-expert 32-bit shared-memory
// mask; a pair's rank within the tile is the popcount of the lower bits, the
// tile's count per expert the popcount.
template <int V>
__global__ void __launch_bounds__(1024, 1)
route_topk_tile_kernel(const float *__restrict__ logits, int T, int E, int k,
                       int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                       int32_t *__restrict__ slot_rank, int32_t *__restrict__ tile_counts) {
    __shared__ uint32_t mask[kMaxExperts];
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int wt = threadIdx.x >> 5;                 // token within the tile
    const int tile = blockIdx.x;
    const int t = tile * kTileTokens + wt;
    const bool active = t < T;                       // warp-uniform
    for (int e = threadIdx.x; e < E; e += blockDim.x) mask[e] = 0u;
    __syncthreads();

    int my_e = 0;
    if (active) {
        float my_w;
        warp_topk<V>(logits + (size_t)t * E, E, k, lane, my_e, my_w);
        if (lane < k) {
            topk_idx[(size_t)t * k + lane] = my_e;
            topk_w[(size_t)t * k + lane] = my_w;
            atomicOr(&mask[my_e], 1u << wt);
        }
    }
    __syncthreads();
    if (active && lane < k)
        slot_rank[(size_t)t * k + lane] = __popc(mask[my_e] & ((1u << wt) - 1u));
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        tile_counts[(size_t)tile * E + e] = __popc(mask[e]);
}

// Small batches, K1: one 256-thread CTA per tile of 8 tokens, one warp per
// token, so that a decode batch spreads over most SMs. As the large-batch K1,
// with 8-bit masks; the tile's count of expert e goes to byte cnt8[e][tile].
template <int V>
__global__ void __launch_bounds__(kSmallTileTokens * 32)
route_topk_small_kernel(const float *__restrict__ logits, int T, int E, int k, int32_t *__restrict__ topk_idx,
                        float *__restrict__ topk_w, int32_t *__restrict__ slot_rank, uint8_t *__restrict__ cnt8,
                        int stride) {
    __shared__ uint32_t mask[kMaxExperts];
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int wt = threadIdx.x >> 5;                 // token within the tile
    const int tile = blockIdx.x;
    const int t = tile * kSmallTileTokens + wt;
    const bool active = t < T;                       // warp-uniform
    for (int e = threadIdx.x; e < E; e += blockDim.x) mask[e] = 0u;
    __syncthreads();

    int my_e = 0;
    if (active) {
        float my_w;
        warp_topk<V>(logits + (size_t)t * E, E, k, lane, my_e, my_w);
        if (lane < k) {
            topk_idx[(size_t)t * k + lane] = my_e;
            topk_w[(size_t)t * k + lane] = my_w;
            atomicOr(&mask[my_e], 1u << wt);
        }
    }
    __syncthreads();
    if (active && lane < k)
        slot_rank[(size_t)t * k + lane] = __popc(mask[my_e] & ((1u << wt) - 1u));
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cnt8[(size_t)e * stride + tile] = (uint8_t)__popc(mask[e]);
}

// Small batches, K2: block 0 forms the totals (counts, offsets, rank_counts,
// dropped) from all tiles' byte counts; block 1 + b finalises tile b, one warp
// per token: for each choice j the warp sums the first b bytes of row e_j (the
// pairs of e_j in earlier tiles), and slot = that + the rank within the tile,
// or -1 at or past the capacity.
__global__ void __launch_bounds__(kSmallTileTokens * 32)
route_slots_small_kernel(int T, int n_tiles, int E, int k, int R, int C, const uint8_t *__restrict__ cnt8, int stride,
                         const int32_t *__restrict__ topk_idx, int32_t *__restrict__ slot,
                         int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                         int32_t *__restrict__ rank_counts, int32_t *__restrict__ dropped) {
    __shared__ int tot[kMaxExperts];
    __shared__ int wsum[32];
    pdl_enter();
    if (blockIdx.x == 0) {             // first, so that it is no tail of the grid
        small_route_totals<8>(cnt8, (size_t)stride, n_tiles, E, R, C, counts, offsets, rank_counts, dropped, tot, wsum);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int tile = blockIdx.x - 1;
    const int t = tile * kSmallTileTokens + (threadIdx.x >> 5);
    if (t >= T) return;                              // warp-uniform
    const int e = lane < k ? __ldg(topk_idx + (size_t)t * k + lane) : 0;
    const int rank = lane < k ? slot[(size_t)t * k + lane] : 0;
    const int limit = tile;                          // bytes [0, tile) of a row: the earlier tiles
    const int c = lane * 16;
    unsigned part[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        part[j] = 0;
        if (j < k) {                                 // warp-uniform
            const int ej = __shfl_sync(kFull, e, j);
            if (c < limit)
                part[j] = add_bytes_below(__ldcg(reinterpret_cast<const uint4 *>(cnt8 + (size_t)ej * stride + c)),
                                          c, limit, 0u);
        }
    }
    int base = 0;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k) {
            const int sj = (int)warp_sum(part[j]);
            if (lane == j) base = sj;
        }
    }
    if (lane < k) {
        const int sl = base + rank;
        slot[(size_t)t * k + lane] = sl < C ? sl : -1;
    }
}

// Chunk c of kChunkTiles tiles: chunk_sums[c][e] = the sum of its tiles'
// counts of expert e.
__global__ void __launch_bounds__(1024)
route_chunk_sums_kernel(int n_tiles, int E, const int32_t *__restrict__ tile_counts, int32_t *__restrict__ chunk_sums) {
    pdl_enter();
    const int c = blockIdx.x;
    const int t0 = c * kChunkTiles, t1 = min(n_tiles, t0 + kChunkTiles);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int s = 0;
#pragma unroll 8
        for (int t = t0; t < t1; ++t) s += __ldg(tile_counts + (size_t)t * E + e);
        chunk_sums[(size_t)c * E + e] = s;
    }
}

// One CTA: chunk_base[c][e] = the sum of chunk_sums[c'][e] over c' < c.
// 1024 / E thread groups split the chunks into contiguous ranges; each group
// starts from the sums of the groups before it.
__global__ void __launch_bounds__(1024)
route_chunk_scan_kernel(int n_chunks, int E, const int32_t *__restrict__ chunk_sums, int32_t *__restrict__ chunk_base) {
    __shared__ int32_t part[1024];
    pdl_enter();
    const int G = (1024 / E) > 0 ? (1024 / E) : 1;
    const int tid = threadIdx.x, g = tid / E, e = tid % E;
    const int per = (n_chunks + G - 1) / G;
    const int c0 = g * per, c1 = min(n_chunks, c0 + per);
    if (g < G) {
        int s = 0;
        for (int c = c0; c < c1; ++c) s += chunk_sums[(size_t)c * E + e];
        part[tid] = s;
    }
    __syncthreads();
    if (g < G) {
        int run = 0;
        for (int gg = 0; gg < g; ++gg) run += part[gg * E + e];
        for (int c = c0; c < c1; ++c) {
            chunk_base[(size_t)c * E + e] = run;
            run += chunk_sums[(size_t)c * E + e];
        }
    }
}

// CTA b finalises tile b: its per-expert base is the sum of the counts of
// tiles 0..b-1 (read from the workspace; 1024/E thread groups split the
// tiles), or with chunk_base its chunk's base plus the tiles before b in the
// chunk; slot = base + rank in tile (or -1 at or past C). The last CTA also
// adds its own tile to get the totals and writes counts, offsets,
// rank_counts and dropped.
__global__ void __launch_bounds__(1024, 1)
route_finalize_kernel(int T, int n_tiles, int E, int k, int R, int C, const int32_t *__restrict__ tile_counts,
                      const int32_t *__restrict__ chunk_base,
                      const int32_t *__restrict__ topk_idx, int32_t *__restrict__ slot,
                      int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                      int32_t *__restrict__ rank_counts, int32_t *__restrict__ dropped) {
    __shared__ int32_t part[1024];
    __shared__ int32_t base[kMaxExperts];
    __shared__ int32_t racc[kMaxExperts];
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t dacc;
    pdl_enter();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const bool last = b == (int)gridDim.x - 1;
    const int G = (1024 / E) > 0 ? (1024 / E) : 1;
    const int g = tid / E, e = tid % E;
    const int from = chunk_base != nullptr ? b / kChunkTiles * kChunkTiles : 0;
    if (g < G) {
        int s = 0;
#pragma unroll 8
        for (int tt = from + g; tt < b; tt += G) s += __ldg(tile_counts + (size_t)tt * E + e);
        part[tid] = s;
    }
    if (last) {
        for (int i = tid; i < E; i += blockDim.x) racc[i] = 0;
        if (tid == 0) dacc = 0;
    }
    __syncthreads();
    if (tid < E) {
        int s = chunk_base != nullptr ? chunk_base[(size_t)(b / kChunkTiles) * E + tid] : 0;
        for (int gg = 0; gg < G; ++gg) s += part[gg * E + tid];
        base[tid] = s;
    }
    __syncthreads();
    const int t0 = b * kTileTokens;
    const int n_pairs = (min(T - t0, kTileTokens) > 0 ? min(T - t0, kTileTokens) : 0) * k;
    for (int i = tid; i < n_pairs; i += blockDim.x) {
        const size_t gi = (size_t)t0 * k + i;
        const int s = base[__ldg(topk_idx + gi)] + slot[gi];
        slot[gi] = s < C ? s : -1;
    }
    if (!last) return;                                   // block-uniform

    // totals = base of this (last) tile + its own counts
    const int v = tid < E ? base[tid] + (b < n_tiles ? __ldg(tile_counts + (size_t)b * E + tid) : 0) : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int ws = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, ws, o);
            if (lane >= o) ws += n;
        }
        warp_sums[lane] = ws;
    }
    __syncthreads();
    const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (tid < E) {
        counts[tid] = v;
        offsets[tid] = excl;
        if (tid == E - 1) offsets[E] = excl + v;
        atomicAdd(&racc[tid / (E / R)], v < C ? v : C);          // integer sums: order-free
        if (v > C) atomicAdd(&dacc, v - C);
    }
    __syncthreads();
    for (int r = tid; r < R; r += blockDim.x) rank_counts[r] = racc[r];
    if (tid == 0) *dropped = dacc;
}

template <int V>
cudaError_t launch_topk(int n_tiles, cudaStream_t st, const float *logits, const Dims &d, int32_t *idx,
                        float *w, int32_t *slot, int32_t *wc) {
    return launch_pdl(route_topk_tile_kernel<V>, n_tiles, 1024, st, logits, d.T, d.E, d.k, idx, w, slot, wc);
}

template <int V>
cudaError_t launch_topk_small(int n_tiles, cudaStream_t st, const float *logits, const Dims &d, int32_t *idx,
                              float *w, int32_t *rank, uint8_t *cnt8, int stride) {
    return launch_pdl(route_topk_small_kernel<V>, n_tiles, kSmallTileTokens * 32, st, logits, d.T, d.E, d.k, idx, w,
                      rank, cnt8, stride);
}

}  // namespace

// The small-batch top-k kernel alone (T <= kRouteSmallMaxTokens, T > 0): top-k
// indices and weights, each pair's rank within its tile of 8 tokens into
// `rank`, and the byte counts cnt8[E][route_small_stride(T)] of every tile.
int launch_route_topk_small(const Dims &d, cudaStream_t st, const float *logits, int32_t *topk_idx, float *topk_w,
                            int32_t *rank, uint8_t *cnt8) {
    const int n_tiles = (d.T + kSmallTileTokens - 1) / kSmallTileTokens;
    const int stride = (int)route_small_stride(d.T);
    const int per_lane = (d.E + 31) / 32;
    cudaError_t e;
    if (per_lane <= 1) e = launch_topk_small<1>(n_tiles, st, logits, d, topk_idx, topk_w, rank, cnt8, stride);
    else if (per_lane <= 2) e = launch_topk_small<2>(n_tiles, st, logits, d, topk_idx, topk_w, rank, cnt8, stride);
    else if (per_lane <= 4) e = launch_topk_small<4>(n_tiles, st, logits, d, topk_idx, topk_w, rank, cnt8, stride);
    else if (per_lane <= 8) e = launch_topk_small<8>(n_tiles, st, logits, d, topk_idx, topk_w, rank, cnt8, stride);
    else if (per_lane <= 16) e = launch_topk_small<16>(n_tiles, st, logits, d, topk_idx, topk_w, rank, cnt8, stride);
    else e = launch_topk_small<32>(n_tiles, st, logits, d, topk_idx, topk_w, rank, cnt8, stride);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

extern "C" int moe_route(const moe_problem *p, const float *logits, int32_t *topk_idx, float *topk_w,
                         int32_t *counts, int32_t *offsets, int32_t *slot, int32_t *rank_counts,
                         int32_t *dropped, void *workspace, size_t workspace_bytes, void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    if (!counts || !offsets || !rank_counts || !dropped || !workspace) return MOE_ERR_INVALID_ARG;
    if (d.T > 0 && (!logits || !topk_idx || !topk_w || !slot)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < moe_route_workspace_bytes(p)) return MOE_ERR_INVALID_ARG;
    if (!aligned(workspace, 16) || !aligned(counts, 4) || !aligned(offsets, 4) ||
        !aligned(rank_counts, 4) || !aligned(dropped, 4))
        return MOE_ERR_INVALID_ARG;
    // 16-byte vector loads of logit rows are used only when E % 4 == 0
    const size_t logit_align = (d.E % 4 == 0) ? 16 : 4;
    if (d.T > 0 && (!aligned(logits, logit_align) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
                    !aligned(slot, 4)))
        return MOE_ERR_INVALID_ARG;

    cudaStream_t st = as_stream(stream);
    if (route_small(d.T, d.E)) {
        // small batches: top-k per tile of 8 tokens, then slots and totals; the
        // second kernel is a programmatic dependent of the first
        uint8_t *cnt8 = static_cast<uint8_t *>(workspace);
        const int n_tiles = (d.T + kSmallTileTokens - 1) / kSmallTileTokens;
        if (n_tiles > 0) {
            rc = launch_route_topk_small(d, st, logits, topk_idx, topk_w, slot, cnt8);
            if (rc != MOE_OK) return rc;
        }
        // an empty batch still runs the totals block: it writes the zero counts
        if (launch_pdl(route_slots_small_kernel, n_tiles + 1, kSmallTileTokens * 32, st, d.T, n_tiles, d.E, d.k, d.R,
                       d.C, static_cast<const uint8_t *>(cnt8), (int)route_small_stride(d.T),
                       static_cast<const int32_t *>(topk_idx), slot, counts, offsets, rank_counts,
                       dropped) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    int32_t *wc = static_cast<int32_t *>(workspace);
    const int n_tiles = (d.T + kTileTokens - 1) / kTileTokens;
    {
        const int per_lane = (d.E + 31) / 32;
        cudaError_t e;
        if (per_lane <= 1) e = launch_topk<1>(n_tiles, st, logits, d, topk_idx, topk_w, slot, wc);
        else if (per_lane <= 2) e = launch_topk<2>(n_tiles, st, logits, d, topk_idx, topk_w, slot, wc);
        else if (per_lane <= 4) e = launch_topk<4>(n_tiles, st, logits, d, topk_idx, topk_w, slot, wc);
        else if (per_lane <= 8) e = launch_topk<8>(n_tiles, st, logits, d, topk_idx, topk_w, slot, wc);
        else if (per_lane <= 16) e = launch_topk<16>(n_tiles, st, logits, d, topk_idx, topk_w, slot, wc);
        else e = launch_topk<32>(n_tiles, st, logits, d, topk_idx, topk_w, slot, wc);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    // many tiles: the two-level scan of the tile counts (chunk sums, then
    // their exclusive bases), each kernel a programmatic dependent of the last
    const int32_t *chunk_base = nullptr;
    if (route_two_level((size_t)n_tiles, d.E)) {
        const int n_chunks = (n_tiles + kChunkTiles - 1) / kChunkTiles;
        int32_t *sums = wc + (size_t)n_tiles * d.E;
        int32_t *bases = sums + (size_t)n_chunks * d.E;
        const int threads = d.E < 1024 ? (d.E + 31) / 32 * 32 : 1024;
        if (launch_pdl(route_chunk_sums_kernel, n_chunks, threads, st, n_tiles, d.E,
                       static_cast<const int32_t *>(wc), sums) != cudaSuccess ||
            launch_pdl(route_chunk_scan_kernel, 1, 1024, st, n_chunks, d.E, static_cast<const int32_t *>(sums),
                       bases) != cudaSuccess)
            return MOE_ERR_CUDA;
        chunk_base = bases;
    }
    // launched as a programmatic dependent of the kernel before it: its launch
    // latency overlaps that kernel's run
    if (launch_pdl(route_finalize_kernel, n_tiles, 1024, st, d.T, n_tiles, d.E, d.k, d.R, d.C,
                   static_cast<const int32_t *>(wc), chunk_base, static_cast<const int32_t *>(topk_idx), slot,
                   counts, offsets, rank_counts, dropped) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

// ---- allocation-free variant ---------------------------------------------
//
// Some callers cannot call cudaMalloc at all: code that runs while a stream is
// being captured into a CUDA graph (allocation is not allowed then), runtimes
// that forbid device allocation after start-up, and plugin interfaces that hand
// a kernel only its input and output buffers. For them moe_route_noalloc keeps
// the route workspace in a file-scope device array instead of a caller buffer.

namespace {

constexpr size_t kStaticRouteScratchBytes = 1u << 20;     // 1 MiB on every GPU that loads the library

__device__ __align__(256) unsigned char g_route_scratch[kStaticRouteScratchBytes];

// Device address of g_route_scratch in the current context, looked up once
// per context (the host-side name of the array is not a device address, and
// a context created again after cudaDeviceReset may load the array
// elsewhere); nullptr if the lookup fails.
void *route_scratch_address() {
    static moe::PerContext<void *> cache;
    return cache.get([] {
        void *p = nullptr;
        return cudaGetSymbolAddress(&p, g_route_scratch) == cudaSuccess ? p : nullptr;
    });
}

}  // namespace

extern "C" int moe_route_noalloc(const moe_problem *p, const float *logits, int32_t *topk_idx, float *topk_w,
                                 int32_t *counts, int32_t *offsets, int32_t *slot, int32_t *rank_counts,
                                 int32_t *dropped, void *stream) {
    using namespace moe;
    const int rc = check_problem(p, nullptr);
    if (rc != MOE_OK) return rc;
    if (moe_route_workspace_bytes(p) > kStaticRouteScratchBytes) return MOE_ERR_UNSUPPORTED;
    void *scratch = route_scratch_address();
    if (scratch == nullptr) return MOE_ERR_CUDA;
    return moe_route(p, logits, topk_idx, topk_w, counts, offsets, slot, rank_counts, dropped, scratch,
                     kStaticRouteScratchBytes, stream);
}
