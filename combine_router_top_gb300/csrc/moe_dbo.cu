// moe_dbo.cu -- the dual-batch-overlap step on two CUDA streams of one GPU.
//
// [DBO §Introduction]: the batch is split into two micro-batches so that while
// one computes, the other communicates. [DBO §UBatchRunner]: the split is at
// the midpoint; a micro-batch with no tokens runs as a dummy (empty) batch.
// [DBO §UBatchContext, §Interfaces]: the two micro-batch threads hand over at
// yield points and a receive hook waits on the all-to-all. Here no host
// threads are needed: the hand-over is a cudaEvent recorded on one stream and
// waited on by the other, and the "all-to-all" of a micro-batch is its
// dispatch (rows into the expert-major buffer) and its combine.
//
// Schedule (compute = caller's compute stream, comm = caller's comm stream):
//   compute: route(0) route(1) dispatch(0) expert(0) [E0] combine(0) wait(D1) expert(1) combine(1)
//   comm:    wait(entry) ........................ wait(E0) dispatch(1) [D1]
// so dispatch of micro-batch 1 runs while micro-batch 0 combines. Combine(0)
// gets a capped grid (grid-stride loop) so that dispatch(1)'s blocks find
// room on every SM at the same time.
#include <new>

#include "moe_internal.cuh"

struct moe_dbo_ctx {
    int device;
    cudaEvent_t entry, expert0, dispatch1;                 // ordering only
    cudaEvent_t t_start, t_d1_start, t_d1_end, t_c0_start, t_c0_end, t_end;   // timing
    bool timed;
    // multi-layer schedule: per micro-batch, end of A1 (gate), dispatch, experts, combine
    cudaEvent_t a1[2], d[2], mlp[2], c[2];
    cudaGraphExec_t graph;                                 // captured multi-layer schedule, or nullptr
};

namespace {

const char *byte_ptr(const void *p, size_t off) { return static_cast<const char *>(p) + off; }

}  // namespace

extern "C" int dbo_create(moe_dbo_ctx **out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    moe_dbo_ctx *c = new (std::nothrow) moe_dbo_ctx();
    if (!c) return MOE_ERR_CUDA;
    if (cudaGetDevice(&c->device) != cudaSuccess) { delete c; return MOE_ERR_CUDA; }
    cudaEvent_t *sync_ev[] = {&c->entry, &c->expert0, &c->dispatch1, &c->a1[0], &c->a1[1], &c->d[0], &c->d[1],
                              &c->mlp[0], &c->mlp[1], &c->c[0], &c->c[1]};
    c->graph = nullptr;
    cudaEvent_t *time_ev[] = {&c->t_start, &c->t_d1_start, &c->t_d1_end, &c->t_c0_start, &c->t_c0_end, &c->t_end};
    bool ok = true;
    for (auto e : sync_ev) ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    for (auto e : time_ev) ok = ok && cudaEventCreate(e) == cudaSuccess;
    c->timed = false;
    if (!ok) { dbo_destroy(c); return MOE_ERR_CUDA; }
    *out = c;
    return MOE_OK;
}

extern "C" void dbo_destroy(moe_dbo_ctx *c) {
    if (!c) return;
    cudaEvent_t evs[] = {c->entry, c->expert0, c->dispatch1, c->t_start, c->t_d1_start, c->t_d1_end,
                         c->t_c0_start, c->t_c0_end, c->t_end, c->a1[0], c->a1[1], c->d[0], c->d[1],
                         c->mlp[0], c->mlp[1], c->c[0], c->c[1]};
    for (auto e : evs)
        if (e) cudaEventDestroy(e);
    if (c->graph) cudaGraphExecDestroy(c->graph);
    delete c;
}

extern "C" int dbo_step(moe_dbo_ctx *ctx, const moe_problem *full, const void *x, const float *logits,
                        const float *s, const moe_ubatch_bufs *bufs, void *out, void *compute_stream,
                        void *comm_stream, int record_timing) {
    using namespace moe;
    Dims d;
    int rc = check_problem(full, &d);
    if (rc != MOE_OK) return rc;
    if (!ctx || !bufs || !s) return MOE_ERR_INVALID_ARG;
    if (d.T > 0 && (!x || !logits || !out)) return MOE_ERR_INVALID_ARG;
    if (compute_stream == comm_stream) return MOE_ERR_INVALID_ARG;

    const int T0 = d.T / 2, T1 = d.T - T0;
    moe_problem p[2] = {*full, *full};
    p[0].num_tokens = T0;
    p[1].num_tokens = T1;
    // overlapped pair: combine(0) keeps two 256-thread blocks per SM (half the
    // register file); dispatch(1), whose bulk-copy blocks are small and
    // short-lived, is not capped: its blocks fill what combine leaves free
    moe_problem p_overlap[2] = {p[0], p[1]};
    p_overlap[0].max_blocks = full->max_blocks > 0 ? full->max_blocks : 2 * sm_count();
    p_overlap[1].max_blocks = full->max_blocks;

    const size_t xrow = (size_t)d.H * 2, lrow = (size_t)d.E * sizeof(float);
    const void *x_ub[2] = {x, d.T ? byte_ptr(x, xrow * T0) : nullptr};
    const float *l_ub[2] = {logits, d.T ? reinterpret_cast<const float *>(byte_ptr(logits, lrow * T0)) : nullptr};
    void *o_ub[2] = {out, d.T ? static_cast<char *>(out) + xrow * T0 : nullptr};

    cudaStream_t cs = as_stream(compute_stream), ms = as_stream(comm_stream);
    const bool timed = record_timing != 0;
#define MOE_TRY(call)                      \
    do {                                   \
        int _r = (call);                   \
        if (_r != MOE_OK) return _r;       \
    } while (0)
#define MOE_CUDA(call)                                   \
    do {                                                 \
        if ((call) != cudaSuccess) return MOE_ERR_CUDA;  \
    } while (0)

    MOE_CUDA(cudaEventRecord(ctx->entry, cs));
    MOE_CUDA(cudaStreamWaitEvent(ms, ctx->entry, 0));
    if (timed) MOE_CUDA(cudaEventRecord(ctx->t_start, cs));

    for (int u = 0; u < 2; ++u) {
        const moe_ubatch_bufs &b = bufs[u];
        MOE_TRY(moe_route(&p[u], l_ub[u], b.topk_idx, b.topk_w, b.counts, b.offsets, b.slot, b.rank_counts,
                          b.dropped, b.workspace, b.workspace_bytes, compute_stream));
    }
    const moe_ubatch_bufs &b0 = bufs[0], &b1 = bufs[1];
    MOE_TRY(moe_dispatch(&p[0], x_ub[0], b0.topk_idx, b0.slot, b0.recv, b0.recv_scale, b0.recv_src, compute_stream));
    MOE_TRY(moe_expert_synthetic(&p[0], b0.recv, b0.recv_scale, b0.counts, s, b0.y, compute_stream));
    MOE_CUDA(cudaEventRecord(ctx->expert0, cs));

    // comm stream: dispatch of micro-batch 1
    MOE_CUDA(cudaStreamWaitEvent(ms, ctx->expert0, 0));
    if (timed) MOE_CUDA(cudaEventRecord(ctx->t_d1_start, ms));
    MOE_TRY(moe_dispatch(&p_overlap[1], x_ub[1], b1.topk_idx, b1.slot, b1.recv, b1.recv_scale, b1.recv_src,
                         comm_stream));
    if (timed) MOE_CUDA(cudaEventRecord(ctx->t_d1_end, ms));
    MOE_CUDA(cudaEventRecord(ctx->dispatch1, ms));

    // compute stream: combine of micro-batch 0 overlaps the dispatch above
    if (timed) MOE_CUDA(cudaEventRecord(ctx->t_c0_start, cs));
    MOE_TRY(moe_combine(&p_overlap[0], b0.y, b0.topk_idx, b0.topk_w, b0.slot, o_ub[0], compute_stream));
    if (timed) MOE_CUDA(cudaEventRecord(ctx->t_c0_end, cs));

    MOE_CUDA(cudaStreamWaitEvent(cs, ctx->dispatch1, 0));
    MOE_TRY(moe_expert_synthetic(&p[1], b1.recv, b1.recv_scale, b1.counts, s, b1.y, compute_stream));
    MOE_TRY(moe_combine(&p[1], b1.y, b1.topk_idx, b1.topk_w, b1.slot, o_ub[1], compute_stream));
    if (timed) MOE_CUDA(cudaEventRecord(ctx->t_end, cs));
    ctx->timed = timed;
#undef MOE_TRY
#undef MOE_CUDA
    return MOE_OK;
}

extern "C" int dbo_read_timing(moe_dbo_ctx *ctx, moe_dbo_timing *t) {
    if (!ctx || !t) return MOE_ERR_INVALID_ARG;
    if (!ctx->timed) return MOE_ERR_INVALID_ARG;
    if (cudaEventSynchronize(ctx->t_end) != cudaSuccess) return MOE_ERR_CUDA;
    float sd, ed, sc, ec, step;
    if (cudaEventElapsedTime(&step, ctx->t_start, ctx->t_end) != cudaSuccess ||
        cudaEventElapsedTime(&sd, ctx->t_start, ctx->t_d1_start) != cudaSuccess ||
        cudaEventElapsedTime(&ed, ctx->t_start, ctx->t_d1_end) != cudaSuccess ||
        cudaEventElapsedTime(&sc, ctx->t_start, ctx->t_c0_start) != cudaSuccess ||
        cudaEventElapsedTime(&ec, ctx->t_start, ctx->t_c0_end) != cudaSuccess)
        return MOE_ERR_CUDA;
    const float dd = ed - sd, dc = ec - sc;
    float ov = (ed < ec ? ed : ec) - (sd > sc ? sd : sc);
    if (ov < 0.0f) ov = 0.0f;
    const float shorter = dd < dc ? dd : dc;
    float frac = shorter > 0.0f ? ov / shorter : 0.0f;
    if (frac > 1.0f) frac = 1.0f;
    t->step_ms = step;
    t->dispatch_ub1_ms = dd;
    t->combine_ub0_ms = dc;
    t->overlap_ms = ov;
    t->overlap_fraction = frac;
    return MOE_OK;
}

// ---- the schedule over layers -------------------------------------------------
//
// [DBO §Introduction] gives the steady-state schedule of one layer for two
// micro-batches (S = shared expert, A0 = qkv projection, A1 = core attention
// + out projection + MoE gate, D = dispatch, C = combine):
//   compute: A0_0 A1_0 | MLP_1 | S_1 MLP_0 | S_0 A0_1 A1_1
//   comm:    D_1       | D_0   | C_1       | C_0
// in the order D_1 send, A0_0, A1_0, D_1 recv, D_0 send, MLP_1, D_0 recv,
// C_1 send, S_1, MLP_0, C_1 recv, C_0 send, S_0, A0_1, A1_1, C_0 recv.
// A0_1 A1_1 at the end of a layer belong to the next layer. Here A0 and S are
// moe_layer_stand_in, A1 is moe_route on the layer's logits, MLP is the
// synthetic expert, D and C are moe_dispatch and moe_combine, and every
// "recv" is an event wait. A prologue runs A0_1 A1_1 of layer 0; the
// combine output of a layer is the next layer's input (in args->out).

extern "C" int dbo_layers(moe_dbo_ctx *ctx, const moe_dbo_layers_args *a, void *compute_stream, void *comm_stream) {
    using namespace moe;
    if (!ctx || !a) return MOE_ERR_INVALID_ARG;
    Dims d;
    int rc = check_problem(&a->full, &d);
    if (rc != MOE_OK) return rc;
    if (a->n_layers < 1 || !a->s || !a->h || !a->shared || !a->out) return MOE_ERR_INVALID_ARG;
    if (d.dtype != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;       // layer inputs are bf16 rows
    if (d.T > 0 && (!a->x || !a->logits)) return MOE_ERR_INVALID_ARG;
    if (a->mlp_max_blocks < 0) return MOE_ERR_INVALID_ARG;
    if (a->expert_w != nullptr && d.H % 64 != 0) return MOE_ERR_UNSUPPORTED;

    const int T0 = d.T / 2, T1 = d.T - T0;
    const int Tu[2] = {T0, T1}, row0[2] = {0, T0};
    moe_problem p[2] = {a->full, a->full};
    p[0].num_tokens = T0;
    p[1].num_tokens = T1;
    // combine (comm stream) keeps at most two 256-thread blocks per SM so that
    // compute-stream blocks find room beside it; the compute-stream kernels run
    // full waves (capping them as well was measured slower: each kernel loses
    // more throughput than the overlap wins back) and dispatch's small
    // bulk-copy blocks fill what is left
    const int cap = a->full.max_blocks > 0 ? a->full.max_blocks : 2 * sm_count();
    moe_problem pc[2] = {p[0], p[1]};
    pc[0].max_blocks = pc[1].max_blocks = cap;
    moe_problem pe[2] = {p[0], p[1]};
    if (a->expert_w != nullptr && a->mlp_max_blocks > 0) pe[0].max_blocks = pe[1].max_blocks = a->mlp_max_blocks;
    const int compute_cap = a->full.max_blocks;

    const size_t rowb = (size_t)d.H * 2;
    auto rows = [&](const void *base, int u) { return static_cast<const char *>(base) + rowb * row0[u]; };
    auto rows_w = [&](void *base, int u) { return static_cast<char *>(base) + rowb * row0[u]; };
    auto logits = [&](int l, int u) {
        return a->logits + ((size_t)l * d.T + row0[u]) * d.E;
    };
    cudaStream_t cs = as_stream(compute_stream), ms = as_stream(comm_stream);
#define MOE_TRY(call)                      \
    do {                                   \
        int _r = (call);                   \
        if (_r != MOE_OK) return _r;       \
    } while (0)
#define MOE_CUDA(call)                                   \
    do {                                                 \
        if ((call) != cudaSuccess) return MOE_ERR_CUDA;  \
    } while (0)

    // A0 and A1 of micro-batch u for layer l (compute stream), then mark the gate done
    auto attention = [&](int l, int u) -> int {
        const void *in = l == 0 ? rows(a->x, u) : rows(a->out, u);
        const moe_ubatch_bufs &b = a->bufs[u];
        int r = layer_stand_in(in, rows_w(a->h, u), (int64_t)Tu[u] * d.H, a->alpha, a->busy_fmas, compute_cap, cs);
        if (r != MOE_OK) return r;
        r = moe_route(&p[u], logits(l, u), b.topk_idx, b.topk_w, b.counts, b.offsets, b.slot, b.rank_counts,
                      b.dropped, b.workspace, b.workspace_bytes, compute_stream);
        if (r != MOE_OK) return r;
        return cudaEventRecord(ctx->a1[u], cs) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    };
    auto dispatch = [&](int u) -> int {                    // comm stream
        const moe_ubatch_bufs &b = a->bufs[u];
        if (cudaStreamWaitEvent(ms, ctx->a1[u], 0) != cudaSuccess) return MOE_ERR_CUDA;
        const int r = moe_dispatch(&p[u], rows(a->h, u), b.topk_idx, b.slot, b.recv, b.recv_scale, b.recv_src,
                                   comm_stream);
        if (r != MOE_OK) return r;
        return cudaEventRecord(ctx->d[u], ms) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    };
    auto experts = [&](int u) -> int {                     // compute stream, after this micro-batch's dispatch
        const moe_ubatch_bufs &b = a->bufs[u];
        if (cudaStreamWaitEvent(cs, ctx->d[u], 0) != cudaSuccess) return MOE_ERR_CUDA;
        const int r = a->expert_w != nullptr
                          ? moe_expert_gemm_bf16(&pe[u], b.recv, b.counts, a->expert_w, b.y, compute_stream)
                          : moe_expert_synthetic(&pe[u], b.recv, b.recv_scale, b.counts, a->s, b.y, compute_stream);
        if (r != MOE_OK) return r;
        return cudaEventRecord(ctx->mlp[u], cs) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    };
    auto combine = [&](int u) -> int {                     // comm stream, after the experts
        const moe_ubatch_bufs &b = a->bufs[u];
        if (cudaStreamWaitEvent(ms, ctx->mlp[u], 0) != cudaSuccess) return MOE_ERR_CUDA;
        const int r = moe_combine(&pc[u], b.y, b.topk_idx, b.topk_w, b.slot, rows_w(a->out, u), comm_stream);
        if (r != MOE_OK) return r;
        return cudaEventRecord(ctx->c[u], ms) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    };
    auto shared_expert = [&](int u) -> int {               // compute stream
        return layer_stand_in(rows(a->h, u), rows_w(a->shared, u), (int64_t)Tu[u] * d.H, a->sigma, a->busy_fmas,
                              compute_cap, cs);
    };

    MOE_CUDA(cudaEventRecord(ctx->entry, cs));
    MOE_CUDA(cudaStreamWaitEvent(ms, ctx->entry, 0));
    MOE_TRY(attention(0, 1));                              // prologue: A0_1 A1_1 of layer 0
    for (int l = 0; l < a->n_layers; ++l) {
        MOE_TRY(dispatch(1));                              // D_1
        if (l > 0) MOE_CUDA(cudaStreamWaitEvent(cs, ctx->c[0], 0));   // layer input of micro-batch 0
        MOE_TRY(attention(l, 0));                          // A0_0 A1_0
        MOE_TRY(dispatch(0));                              // D_0
        MOE_TRY(experts(1));                               // MLP_1 (D_1 recv)
        MOE_TRY(combine(1));                               // C_1
        MOE_TRY(shared_expert(1));                         // S_1
        MOE_TRY(experts(0));                               // MLP_0 (D_0 recv)
        MOE_TRY(combine(0));                               // C_0
        MOE_TRY(shared_expert(0));                         // S_0
        if (l + 1 < a->n_layers) {
            MOE_CUDA(cudaStreamWaitEvent(cs, ctx->c[1], 0));          // C_1 recv: next layer's input
            MOE_TRY(attention(l + 1, 1));                  // A0_1 A1_1 of the next layer
        }
    }
    MOE_CUDA(cudaStreamWaitEvent(cs, ctx->c[0], 0));       // C_0 recv, and C_1 of the last layer
    MOE_CUDA(cudaStreamWaitEvent(cs, ctx->c[1], 0));
#undef MOE_TRY
#undef MOE_CUDA
    return MOE_OK;
}

extern "C" int dbo_layers_capture(moe_dbo_ctx *ctx, const moe_dbo_layers_args *a, void *compute_stream,
                                  void *comm_stream) {
    if (!ctx || !a) return MOE_ERR_INVALID_ARG;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(compute_stream);
    if (cs == nullptr) return MOE_ERR_INVALID_ARG;         // the legacy stream cannot be captured
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) return MOE_ERR_CUDA;
    const int rc = dbo_layers(ctx, a, compute_stream, comm_stream);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(cs, &g);
    if (rc != MOE_OK) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess || g == nullptr) return MOE_ERR_CUDA;
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, g, 0);
    cudaGraphDestroy(g);
    if (ie != cudaSuccess) return MOE_ERR_CUDA;
    if (ctx->graph) cudaGraphExecDestroy(ctx->graph);
    ctx->graph = exec;
    return MOE_OK;
}

extern "C" int dbo_graph_launch(moe_dbo_ctx *ctx, void *stream) {
    if (!ctx || !ctx->graph) return MOE_ERR_INVALID_ARG;
    return cudaGraphLaunch(ctx->graph, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
