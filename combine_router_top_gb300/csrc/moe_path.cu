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
    if (d.T > 0 && (!x_host || !logits_host || !x_dev || !logits_dev || !out_dev || !out_host))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    const size_t x_bytes = (size_t)d.T * d.H * sizeof(uint16_t);
    const size_t l_bytes = (size_t)d.T * d.E * sizeof(float);
    if (d.T > 0) {
        if (cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaMemcpyAsync(logits_dev, logits_host, l_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    const moe_ubatch_bufs &b = *bufs;
    rc = moe_route(p, logits_dev, b.topk_idx, b.topk_w, b.counts, b.offsets, b.slot, b.rank_counts, b.dropped,
                   b.workspace, b.workspace_bytes, stream);
    if (rc != MOE_OK) return rc;
    rc = moe_dispatch(p, x_dev, b.topk_idx, b.slot, b.recv, b.recv_scale, b.recv_src, stream);
    if (rc != MOE_OK) return rc;
    rc = moe_expert_synthetic(p, b.recv, b.recv_scale, b.counts, s, b.y, stream);
    if (rc != MOE_OK) return rc;
    rc = moe_combine(p, b.y, b.topk_idx, b.topk_w, b.slot, out_dev, stream);
    if (rc != MOE_OK) return rc;
    if (d.T > 0 && cudaMemcpyAsync(out_host, out_dev, x_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
