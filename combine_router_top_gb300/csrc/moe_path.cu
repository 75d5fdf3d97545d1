// moe_path.cu -- the whole path for one batch whose inputs and output live in
// host memory, in one call: the serving-loop form of the path.
//
// On `stream`, in order: copy x and the router logits from host memory into
// device staging buffers, route, dispatch, synthetic expert, combine, copy the
// output back to host memory. Every step is asynchronous; one call issues
// the whole batch. With two streams and two buffer sets used alternately,
// one batch's copies run under the neighbouring batch's kernels.
#include "moe_internal.cuh"

extern "C" int moe_path_host(const moe_problem *p, const void *x_host, const float *logits_host, const float *s,
                             void *x_dev, float *logits_dev, const moe_ubatch_bufs *bufs, void *out_dev,
                             void *out_host, void *stream) {
    using namespace moe;
    Dims d;
    int rc = check_problem(p, &d);
    if (rc != MOE_OK) return rc;
    if (bufs == nullptr) return MOE_ERR_INVALID_ARG;
    // every check the four calls make, before anything is enqueued, so that a
    // failing call launches nothing
    const moe_ubatch_bufs &c = *bufs;
    const bool fp8 = d.dtype == MOE_DTYPE_FP8_E4M3_B128;
    if (!c.counts || !c.offsets || !c.rank_counts || !c.dropped || !c.workspace || !s || !c.recv || !c.y)
        return MOE_ERR_INVALID_ARG;
    if (c.workspace_bytes < moe_route_workspace_bytes(p) || fp8 != (c.recv_scale != nullptr)) return MOE_ERR_INVALID_ARG;
    if (!aligned(c.counts, 4) || !aligned(c.offsets, 4) || !aligned(c.rank_counts, 4) || !aligned(c.dropped, 4) ||
        !aligned(c.workspace, 16) || !aligned(s, 4) || !aligned(c.recv, 16) || !aligned(c.y, 16) ||
        (fp8 && !aligned(c.recv_scale, 16)))
        return MOE_ERR_INVALID_ARG;
    if (d.T > 0) {
        if (!x_host || !logits_host || !x_dev || !logits_dev || !out_dev || !out_host || !c.topk_idx || !c.topk_w ||
            !c.slot || !c.recv_src)
            return MOE_ERR_INVALID_ARG;
        const size_t logit_align = (d.E % 4 == 0) ? 16 : 4;
        if (!aligned(x_dev, 16) || !aligned(logits_dev, logit_align) || !aligned(out_dev, 16) ||
            !aligned(c.topk_idx, 4) || !aligned(c.topk_w, 4) ||
            !aligned(c.slot, 4) || !aligned(c.recv_src, 4))
            return MOE_ERR_INVALID_ARG;
    }
    cudaStream_t st = as_stream(stream);
    const size_t x_bytes = (size_t)d.T * d.H * sizeof(uint16_t);
    const size_t l_bytes = (size_t)d.T * d.E * sizeof(float);
    if (d.T > 0) {
        if (cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaMemcpyAsync(logits_dev, logits_host, l_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    rc = moe_route(p, logits_dev, c.topk_idx, c.topk_w, c.counts, c.offsets, c.slot, c.rank_counts, c.dropped,
                   c.workspace, c.workspace_bytes, stream);
    if (rc != MOE_OK) return rc;
    rc = moe_dispatch(p, x_dev, c.topk_idx, c.slot, c.recv, c.recv_scale, c.recv_src, stream);
    if (rc != MOE_OK) return rc;
    rc = moe_expert_synthetic(p, c.recv, c.recv_scale, c.counts, s, c.y, stream);
    if (rc != MOE_OK) return rc;
    rc = moe_combine(p, c.y, c.topk_idx, c.topk_w, c.slot, out_dev, stream);
    if (rc != MOE_OK) return rc;
    if (d.T > 0 && cudaMemcpyAsync(out_host, out_dev, x_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
