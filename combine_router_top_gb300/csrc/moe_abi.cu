// moe_abi.cu -- status strings, argument validation and workspace sizing.
// Host code only; nothing here touches the GPU except the cached SM count,
// the status word's address and the current context's identity.
#include "moe_internal.cuh"

#include <cuda.h>

namespace moe {

namespace {
__device__ unsigned g_device_status;    // kStatus* bits, set by kernels whose bounded waits gave up

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}
}  // namespace

bool current_ctx(CtxKey *key) {
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (get_current == nullptr || get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (cudaGetDevice(&key->dev) != cudaSuccess) return false;
    // before the runtime's first call on this thread no context may be current yet
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, &key->id) == CUDA_SUCCESS;
}

unsigned *device_status_word() {
    static PerContext<unsigned *> cache;
    return cache.get([] {
        void *p = nullptr;
        return cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess ? static_cast<unsigned *>(p) : nullptr;
    });
}

int check_problem(const moe_problem *p, Dims *d) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    const long long T = p->num_tokens, H = p->hidden, E = p->num_experts, k = p->top_k;
    const long long R = p->num_ranks, C = p->capacity;
    if (T < 0 || T > kMaxTokens) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > kMaxExperts) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > kMaxTopK || k > E) return MOE_ERR_INVALID_ARG;
    if (R < 1 || R > E || E % R != 0) return MOE_ERR_INVALID_ARG;
    if (C < 1 || C > kMaxCapacity) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > kMaxHidden || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (p->dispatch_dtype != MOE_DTYPE_BF16 && p->dispatch_dtype != MOE_DTYPE_FP8_E4M3_B128)
        return MOE_ERR_INVALID_ARG;
    if (p->dispatch_dtype == MOE_DTYPE_FP8_E4M3_B128 && H % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (p->max_blocks < 0 || p->tokens_per_src_rank < 0) return MOE_ERR_INVALID_ARG;
    if (T * k >= (1LL << 31) || E * C >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
    if (d) {
        d->T = (int)T; d->H = (int)H; d->E = (int)E; d->k = (int)k;
        d->R = (int)R; d->C = (int)C; d->dtype = p->dispatch_dtype; d->max_blocks = p->max_blocks;
    }
    return MOE_OK;
}

int sm_count() {
    static PerContext<int> cache;
    const int n = cache.get([] {
        int dev = 0, m = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || m <= 0)
            return 0;
        return m;
    });
    return n > 0 ? n : 1;
}

}  // namespace moe

extern "C" {

const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: a size, pointer or alignment check failed";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: request outside what this build supports";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: the CUDA runtime reported an error";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK: a device-side consistency check failed";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait gave up";
        default: return "unknown moe_status";
    }
}

int moe_validate(const moe_problem *p) { return moe::check_problem(p, nullptr); }

int moe_device_status(void) {
    unsigned *w = moe::device_status_word();
    if (w == nullptr) return MOE_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (v == 0) return MOE_OK;
    const unsigned zero = 0;
    if (cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
    return (v & moe::kStatusWaitGaveUp) ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE_CHECK;
}

size_t moe_route_workspace_bytes(const moe_problem *p) {
    moe::Dims d;
    if (moe::check_problem(p, &d) != MOE_OK) return 0;
    size_t bytes;
    if (moe::route_small(d.T, d.E)) {
        bytes = (size_t)d.E * moe::route_small_stride(d.T);              // one byte per (expert, tile of 8)
    } else {
        const size_t tiles = ((size_t)d.T + moe::kTileTokens - 1) / moe::kTileTokens;
        bytes = tiles * (size_t)d.E * sizeof(int32_t);                 // counts per (tile of 32, expert)
        if (moe::route_two_level(tiles, d.E)) {                        // + sums and bases per (chunk, expert)
            const size_t chunks = (tiles + moe::kChunkTiles - 1) / moe::kChunkTiles;
            bytes += 2 * chunks * (size_t)d.E * sizeof(int32_t);
        }
    }
    bytes = (bytes + 255) & ~(size_t)255;
    return bytes < 256 ? 256 : bytes;
}

}  // extern "C"
