// moe_route.cu -- steps 1 and 2 of the path: router top-k with renormalised
// softmax weights, then the per-expert histogram, its exclusive scan and the
// slot of every (token, choice) pair.
//
// [PMC §Introduction]: the router's probability distribution picks the top-K
// experts and weights their outputs. [PMC §Dispatch]: a counting warp tallies
// tokens per destination expert. [PMC §Portable kernels]: a fixed per-expert
// bound lets every sender compute a unique destination address.
//
// One launch, no atomic that decides an order, no waiting:
//   Every CTA takes a tile of 32 tokens, one warp per token. Top-k by k rounds
//   of a warp arg-max (redux.sync max on an order-preserving 32-bit key,
//   ballot for the lowest tied lane). Weights by expf and one IEEE division.
//   Each chosen expert sets the token's bit in a per-expert 32-bit shared-
//   memory mask: a pair's rank within the tile is the popcount of the lower
//   bits, the tile's count per expert the popcount. The CTA writes its counts,
//   fences, and takes a ticket (atomicInc, which wraps back to 0 on the last
//   one). The CTA that draws the last ticket sees every tile's counts: it
//   scans them per expert over the tiles (tile bases), writes every pair's
//   slot = base + rank (or -1 at or past C), and the totals, offsets, rank
//   counts and drops.
//
// Workspace: [ticket counter, 16 bytes][tile counts: max(tiles,1) x E int32].
// The counter must be zero before the first call; every call that completes
// leaves it zero.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

// Lane l of a token's warp owns experts [l*V, l*V + V) (clipped to E).
template <int V>
__global__ void __launch_bounds__(1024, 1)
route_kernel(const float *__restrict__ logits, int T, int E, int k, int R, int C, int n_tiles,
             int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int32_t *__restrict__ slot,
             unsigned *__restrict__ ticket, int32_t *__restrict__ tile_counts, int32_t *__restrict__ counts,
             int32_t *__restrict__ offsets, int32_t *__restrict__ rank_counts, int32_t *__restrict__ dropped) {
    __shared__ uint32_t mask[kMaxExperts];
    __shared__ int32_t part[1024];
    __shared__ int32_t racc[kMaxExperts];
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t dacc;
    __shared__ unsigned s_ticket;
    pdl_enter();
    const int tid = threadIdx.x, lane = tid & 31;
    const int wt = tid >> 5;                          // token within the tile
    const int tile = blockIdx.x;
    const int t = tile * kTileTokens + wt;
    const bool active = t < T;                        // warp-uniform
    for (int e = tid; e < E; e += blockDim.x) mask[e] = 0u;
    __syncthreads();

    int my_e = 0;
    if (active) {
        const int e0 = lane * V;
        const float *row = logits + (size_t)t * E;
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

        // w_j = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0)
        float ex = 0.0f;
        if (lane < k) ex = expf(key_logit(my_key) - key_logit(top_key));
        float sum = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
        if (lane < k) {
            topk_idx[(size_t)t * k + lane] = my_e;
            topk_w[(size_t)t * k + lane] = __fdiv_rn(ex, sum);
            atomicOr(&mask[my_e], 1u << wt);
        }
    }
    __syncthreads();
    if (active && lane < k)
        slot[(size_t)t * k + lane] = __popc(mask[my_e] & ((1u << wt) - 1u));   // rank within the tile
    for (int e = tid; e < E; e += blockDim.x) tile_counts[(size_t)tile * E + e] = __popc(mask[e]);

    // the last CTA to finish finalises every tile
    __threadfence();
    __syncthreads();
    if (tid == 0) s_ticket = atomicInc(ticket, (unsigned)gridDim.x - 1u);
    __syncthreads();
    if (s_ticket != gridDim.x - 1u) return;           // block-uniform
    __threadfence();

    // exclusive scan over tiles per expert; 1024/E thread groups split the tiles
    const int G = (1024 / E) > 0 ? (1024 / E) : 1;
    const int g = tid / E, e = tid % E;
    const int per = (n_tiles + G - 1) / G;
    const int b0 = min(n_tiles, g * per), b1 = min(n_tiles, b0 + per);
    if (g < G) {
        int sum = 0;
#pragma unroll 8
        for (int b = b0; b < b1; ++b) sum += __ldcg(tile_counts + (size_t)b * E + e);
        part[tid] = sum;
    }
    for (int i = tid; i < E; i += blockDim.x) racc[i] = 0;
    if (tid == 0) dacc = 0;
    __syncthreads();
    int v = 0;                                         // total of expert tid (tid < E)
    if (g < G) {
        int run = 0;
        for (int gg = 0; gg < g; ++gg) run += part[gg * E + e];
        for (int b = b0; b < b1; ++b) {
            const int c = __ldcg(tile_counts + (size_t)b * E + e);
            tile_counts[(size_t)b * E + e] = run;       // becomes the tile's base for expert e
            run += c;
        }
    }
    if (tid < E)
        for (int gg = 0; gg < G; ++gg) v += part[gg * E + tid];
    __syncthreads();                                   // bases visible to the whole CTA

    // slots of every pair
    const int n_pairs = T * k;
    for (int i = tid; i < n_pairs; i += blockDim.x) {
        const int b = (i / k) / kTileTokens;
        const int sl = __ldcg(tile_counts + (size_t)b * E + __ldcg(topk_idx + i)) + __ldcg(slot + i);
        slot[i] = sl < C ? sl : -1;
    }

    // offsets = exclusive scan of the totals over experts
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    const int warp = tid >> 5;
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
int launch_route(int grid, cudaStream_t st, const float *logits, const Dims &d, int n_tiles, int32_t *idx,
                 float *w, int32_t *slot, void *workspace, int32_t *counts, int32_t *offsets, int32_t *rank_counts,
                 int32_t *dropped) {
    unsigned *ticket = static_cast<unsigned *>(workspace);
    int32_t *tile_counts = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + 16);
    if (launch_pdl(route_kernel<V>, grid, 1024, st, logits, d.T, d.E, d.k, d.R, d.C, n_tiles, idx, w, slot,
                   ticket, tile_counts, counts, offsets, rank_counts, dropped) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace
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
    const int n_tiles = (d.T + kTileTokens - 1) / kTileTokens;
    // an empty batch still runs one block: it writes the zero counts
    const int grid = n_tiles > 0 ? n_tiles : 1;
    const int per_lane = (d.E + 31) / 32;
    int rc2;
    if (per_lane <= 1) rc2 = launch_route<1>(grid, st, logits, d, n_tiles, topk_idx, topk_w, slot, workspace, counts, offsets, rank_counts, dropped);
    else if (per_lane <= 2) rc2 = launch_route<2>(grid, st, logits, d, n_tiles, topk_idx, topk_w, slot, workspace, counts, offsets, rank_counts, dropped);
    else if (per_lane <= 4) rc2 = launch_route<4>(grid, st, logits, d, n_tiles, topk_idx, topk_w, slot, workspace, counts, offsets, rank_counts, dropped);
    else if (per_lane <= 8) rc2 = launch_route<8>(grid, st, logits, d, n_tiles, topk_idx, topk_w, slot, workspace, counts, offsets, rank_counts, dropped);
    else if (per_lane <= 16) rc2 = launch_route<16>(grid, st, logits, d, n_tiles, topk_idx, topk_w, slot, workspace, counts, offsets, rank_counts, dropped);
    else rc2 = launch_route<32>(grid, st, logits, d, n_tiles, topk_idx, topk_w, slot, workspace, counts, offsets, rank_counts, dropped);
    return rc2;
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
constexpr int kMaxScratchDevices = 64;

__device__ __align__(256) unsigned char g_route_scratch[kStaticRouteScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxScratchDevices] = {};

// Device address of g_route_scratch on the current device, looked up once per
// device (the host-side name of the array is not a device address).
int route_scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxScratchDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_route_noalloc(const moe_problem *p, const float *logits, int32_t *topk_idx, float *topk_w,
                                 int32_t *counts, int32_t *offsets, int32_t *slot, int32_t *rank_counts,
                                 int32_t *dropped, void *stream) {
    using namespace moe;
    const int rc = check_problem(p, nullptr);
    if (rc != MOE_OK) return rc;
    if (moe_route_workspace_bytes(p) > kStaticRouteScratchBytes) return MOE_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const int ac = route_scratch_address(&scratch);
    if (ac != MOE_OK) return ac;
    return moe_route(p, logits, topk_idx, topk_w, counts, offsets, slot, rank_counts, dropped, scratch,
                     kStaticRouteScratchBytes, stream);
}
