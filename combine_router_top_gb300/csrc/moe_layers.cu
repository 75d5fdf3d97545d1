// moe_layers.cu -- stand-in for the layer compute around the MoE block, used
// by the multi-layer dual-batch-overlap schedule.
//
// [DBO §Introduction] names the compute of a layer: A0 (qkv projection), A1
// (core attention, out projection and the MoE gate) and S (the shared
// expert). Their weights are out of scope; this kernel stands in for them:
//   out[i] = bf16(float(in[i]) * a)      (fp32 product, round to nearest even)
// plus `busy` dependent fp32 FMAs per 16-byte chunk of busy work that cannot
// change the output, so that the stand-in can be made compute-bound like the
// GEMMs it replaces.
#include "moe_internal.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256)
stand_in_kernel(const uint4 *__restrict__ in, uint4 *__restrict__ out, long long n16, float a, int busy) {
    pdl_enter();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint4 v = in[i];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t ov[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) ov[h] = pack_bf16x2(__fmul_rn(bf16_lo(wv[h]), a), __fmul_rn(bf16_hi(wv[h]), a));
        // busy work: z stays finite for a finite input, so the test below never
        // changes the output (a NaN input gives a NaN output either way); it
        // only keeps the compiler from dropping the loop
        float z = bf16_lo(v.x);
        for (int r = 0; r < busy; ++r) z = __fmaf_rn(z, 0.999999f, 1e-6f);
        if (z != z) ov[0] |= 0x7FC0u;
        out[i] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
    }
}

}  // namespace
}  // namespace moe

namespace moe {
// moe_layer_stand_in with at most max_blocks thread blocks (0: one resident wave).
int layer_stand_in(const void *in, void *out, int64_t n_elements, float a, int32_t busy_fmas, int max_blocks,
                   cudaStream_t st) {
    if (n_elements < 0 || n_elements % 8 != 0 || busy_fmas < 0 || busy_fmas > (1 << 20)) return MOE_ERR_INVALID_ARG;
    if (n_elements == 0) return MOE_OK;
    if (!in || !out || !aligned(in, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
    static PerContext<int> resident_cache;
    const int resident = resident_blocks_cached(resident_cache, stand_in_kernel, 256);
    const long long n16 = n_elements / 8;
    const int grid = persistent_grid((n16 + 255) / 256, resident, max_blocks);
    if (launch_pdl(stand_in_kernel, grid, 256, st, static_cast<const uint4 *>(in), static_cast<uint4 *>(out), n16, a,
                   (int)busy_fmas) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
}  // namespace moe

extern "C" int moe_layer_stand_in(const void *in, void *out, int64_t n_elements, float a, int32_t busy_fmas,
                                  void *stream) {
    return moe::layer_stand_in(in, out, n_elements, a, busy_fmas, 0, moe::as_stream(stream));
}
