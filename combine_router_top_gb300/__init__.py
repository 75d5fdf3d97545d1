"""Python binding of libmoe_gb300, the MoE route / dispatch / combine path on
one GB300 (sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels, reached through ctypes with the same entry-point names as the C ABI in
``include/moe.h``. PyTorch supplies device memory and streams. There is no CPU
fallback: if the library is not built, or a tensor is not on a CUDA device,
the call raises.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_DEVICE_CHECK = -4
MOE_ERR_TIMEOUT = -5

MOE_DTYPE_BF16 = 0
MOE_DTYPE_FP8_E4M3_B128 = 1


class moe_problem(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("num_tokens", "hidden", "num_experts", "top_k", "num_ranks",
                                         "capacity", "dispatch_dtype", "max_blocks", "tokens_per_src_rank")]


class moe_ubatch_bufs(C.Structure):
    _fields_ = [("topk_idx", C.c_void_p), ("topk_w", C.c_void_p), ("counts", C.c_void_p),
                ("offsets", C.c_void_p), ("slot", C.c_void_p), ("rank_counts", C.c_void_p),
                ("dropped", C.c_void_p), ("recv", C.c_void_p), ("recv_scale", C.c_void_p),
                ("recv_src", C.c_void_p), ("y", C.c_void_p), ("workspace", C.c_void_p),
                ("workspace_bytes", C.c_size_t)]


class moe_dbo_timing(C.Structure):
    _fields_ = [(n, C.c_float) for n in ("step_ms", "dispatch_ub1_ms", "combine_ub0_ms", "overlap_ms",
                                         "overlap_fraction")]


class moe_dbo_layers_args(C.Structure):
    _fields_ = [("full", moe_problem), ("n_layers", C.c_int32), ("busy_fmas", C.c_int32), ("alpha", C.c_float),
                ("sigma", C.c_float), ("x", C.c_void_p), ("logits", C.c_void_p), ("s", C.c_void_p),
                ("bufs", moe_ubatch_bufs * 2), ("h", C.c_void_p), ("shared", C.c_void_p), ("out", C.c_void_p),
                ("expert_w", C.c_void_p), ("mlp_max_blocks", C.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {moe_status_string(status)} ({status})")
        self.status = status


_lib = None


def lib() -> C.CDLL:
    """The loaded library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        P, i = C.c_void_p, C.c_int
        pp = C.POINTER(moe_problem)
        sig = {
            "moe_status_string": ([i], C.c_char_p),
            "moe_validate": ([pp], i),
            "moe_device_status": ([], i),
            "moe_route_workspace_bytes": ([pp], C.c_size_t),
            "moe_route": ([pp, P, P, P, P, P, P, P, P, P, C.c_size_t, P], i),
            "moe_route_noalloc": ([pp, P, P, P, P, P, P, P, P, P], i),
            "moe_dispatch": ([pp, P, P, P, P, P, P, P], i),
            "moe_src_offsets": ([pp, P, P, P, P], i),
            "moe_route_dispatch_workspace_bytes": ([pp], C.c_size_t),
            "moe_route_dispatch": ([pp, P, P, P, P, P, P, P, P, P, P, P, P, P, C.c_size_t, P], i),
            "moe_expert_synthetic": ([pp, P, P, P, P, P, P], i),
            "moe_expert_gemm_fp8": ([pp, P, P, P, P, P, P, P], i),
            "moe_expert_gemm_bf16": ([pp, P, P, P, P, P], i),
            "moe_ready_flags_bytes": ([pp], C.c_size_t),
            "moe_path_host": ([pp, P, P, P, P, P, C.POINTER(moe_ubatch_bufs), P, P, P], i),
            "moe_expert_combine": ([pp, P, P, P, P, P, P, P, P, P, P, C.c_size_t, C.c_uint32, P], i),
            "moe_combine": ([pp, P, P, P, P, P, P], i),
            "dbo_create": ([C.POINTER(P)], i),
            "dbo_destroy": ([P], None),
            "dbo_step": ([P, pp, P, P, P, C.POINTER(moe_ubatch_bufs), P, P, P, i], i),
            "dbo_read_timing": ([P, C.POINTER(moe_dbo_timing)], i),
            "moe_layer_stand_in": ([P, P, C.c_int64, C.c_float, C.c_int32, P], i),
            "dbo_layers": ([P, C.POINTER(moe_dbo_layers_args), P, P], i),
            "dbo_layers_capture": ([P, C.POINTER(moe_dbo_layers_args), P, P], i),
            "dbo_graph_launch": ([P, P], i),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes, f.restype = args, res
        _lib = L
    return _lib


EXPORTS = ("moe_status_string", "moe_validate", "moe_device_status", "moe_route_workspace_bytes", "moe_route", "moe_route_noalloc",
           "moe_dispatch", "moe_src_offsets", "moe_route_dispatch_workspace_bytes", "moe_route_dispatch",
           "moe_expert_synthetic", "moe_expert_gemm_fp8", "moe_expert_gemm_bf16", "moe_ready_flags_bytes", "moe_expert_combine", "moe_path_host",
           "moe_combine", "dbo_create", "dbo_destroy", "dbo_step", "dbo_read_timing",
           "moe_layer_stand_in", "dbo_layers", "dbo_layers_capture", "dbo_graph_launch")


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def problem(T, H, E, k, R, Cap, dtype=MOE_DTYPE_BF16, max_blocks=0, tokens_per_src_rank=0) -> moe_problem:
    return moe_problem(T, H, E, k, R, Cap, dtype, max_blocks, tokens_per_src_rank)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe_gb300 takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libmoe_gb300 takes contiguous tensors only")
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def moe_device_status() -> int:
    """MOE_OK, or MOE_ERR_TIMEOUT if a bounded device wait gave up since the last call (synchronises)."""
    return lib().moe_device_status()


def moe_validate(p: moe_problem) -> int:
    return lib().moe_validate(C.byref(p))


def moe_route_workspace_bytes(p: moe_problem) -> int:
    return lib().moe_route_workspace_bytes(C.byref(p))


def moe_route(p, logits, topk_idx, topk_w, counts, offsets, slot, rank_counts, dropped, workspace, stream=None):
    rc = lib().moe_route(C.byref(p), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(offsets),
                         _ptr(slot), _ptr(rank_counts), _ptr(dropped), _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check("moe_route", rc)


def moe_route_noalloc(p, logits, topk_idx, topk_w, counts, offsets, slot, rank_counts, dropped, stream=None):
    """moe_route with the library's own static scratch instead of a workspace
    (for callers that cannot allocate device memory)."""
    rc = lib().moe_route_noalloc(C.byref(p), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
                                 _ptr(offsets), _ptr(slot), _ptr(rank_counts), _ptr(dropped), _stream(stream))
    _check("moe_route_noalloc", rc)


def src_ranks(p) -> int:
    """S, the number of virtual data-parallel source ranks of problem p."""
    T, tps = p.num_tokens, p.tokens_per_src_rank
    return max(1, (T + tps - 1) // tps) if tps > 0 else 1


def moe_src_offsets(p, counts, recv_src, src_offsets, stream=None):
    """src_offsets [E][S+1]: per expert, the first row of each source rank's tokens."""
    rc = lib().moe_src_offsets(C.byref(p), _ptr(counts), _ptr(recv_src), _ptr(src_offsets), _stream(stream))
    _check("moe_src_offsets", rc)


def moe_dispatch(p, x, topk_idx, slot, recv, recv_scale, recv_src, stream=None):
    rc = lib().moe_dispatch(C.byref(p), _ptr(x), _ptr(topk_idx), _ptr(slot), _ptr(recv), _ptr(recv_scale),
                            _ptr(recv_src), _stream(stream))
    _check("moe_dispatch", rc)


def moe_route_dispatch_workspace_bytes(p: moe_problem) -> int:
    return lib().moe_route_dispatch_workspace_bytes(C.byref(p))


def moe_route_dispatch(p, logits, x, topk_idx, topk_w, counts, offsets, slot, rank_counts, dropped, recv,
                       recv_scale, recv_src, workspace, stream=None):
    """moe_route then moe_dispatch in one call (fused into two launches for fp8 decode batches)."""
    rc = lib().moe_route_dispatch(C.byref(p), _ptr(logits), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
                                  _ptr(offsets), _ptr(slot), _ptr(rank_counts), _ptr(dropped), _ptr(recv),
                                  _ptr(recv_scale), _ptr(recv_src), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check("moe_route_dispatch", rc)


def moe_expert_synthetic(p, recv, recv_scale, counts, s, y, stream=None):
    rc = lib().moe_expert_synthetic(C.byref(p), _ptr(recv), _ptr(recv_scale), _ptr(counts), _ptr(s), _ptr(y),
                                    _stream(stream))
    _check("moe_expert_synthetic", rc)


def moe_expert_gemm_fp8(p, recv_q, recv_scale, counts, w_q, w_scale, y, stream=None):
    """Grouped fp8 GEMM on the dispatch layout (tensor cores): y[e][r] = bf16(row . W_e^T) on kept rows."""
    rc = lib().moe_expert_gemm_fp8(C.byref(p), _ptr(recv_q), _ptr(recv_scale), _ptr(counts), _ptr(w_q),
                                   _ptr(w_scale), _ptr(y), _stream(stream))
    _check("moe_expert_gemm_fp8", rc)


def moe_expert_gemm_bf16(p, recv_x, counts, w, y, stream=None):
    """Grouped bf16 GEMM on the dispatch layout (tensor cores): y[e][r] = bf16(row . W_e^T) on kept rows."""
    rc = lib().moe_expert_gemm_bf16(C.byref(p), _ptr(recv_x), _ptr(counts), _ptr(w), _ptr(y), _stream(stream))
    _check("moe_expert_gemm_bf16", rc)


def moe_ready_flags_bytes(p: moe_problem) -> int:
    return lib().moe_ready_flags_bytes(C.byref(p))


def moe_expert_combine(p, recv, recv_scale, counts, s, y, topk_idx, topk_w, slot, out, flags, epoch: int,
                       stream=None):
    """Synthetic expert + combine in one kernel with per-row readiness flags (epoch: nonzero, fresh per call)."""
    rc = lib().moe_expert_combine(C.byref(p), _ptr(recv), _ptr(recv_scale), _ptr(counts), _ptr(s), _ptr(y),
                                  _ptr(topk_idx), _ptr(topk_w), _ptr(slot), _ptr(out), _ptr(flags),
                                  flags.numel() * flags.element_size(), epoch, _stream(stream))
    _check("moe_expert_combine", rc)


def moe_combine(p, y, topk_idx, topk_w, slot, out, stream=None):
    rc = lib().moe_combine(C.byref(p), _ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(slot), _ptr(out),
                           _stream(stream))
    _check("moe_combine", rc)


class DboContext:
    """Owns a moe_dbo_ctx (CUDA events only)."""

    def __init__(self):
        h = C.c_void_p()
        _check("dbo_create", lib().dbo_create(C.byref(h)))
        self.handle = h

    def close(self):
        if self.handle:
            lib().dbo_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dbo_create() -> DboContext:
    return DboContext()


def dbo_destroy(ctx: DboContext):
    ctx.close()


def ubatch_bufs(b: dict) -> moe_ubatch_bufs:
    """moe_ubatch_bufs from a dict of tensors laid out as alloc_buffers() makes them."""
    return moe_ubatch_bufs(_ptr(b["topk_idx"]), _ptr(b["topk_w"]), _ptr(b["counts"]), _ptr(b["offsets"]),
                           _ptr(b["slot"]), _ptr(b["rank_counts"]), _ptr(b["dropped"]), _ptr(b["recv"]),
                           _ptr(b.get("recv_scale")), _ptr(b["recv_src"]), _ptr(b["y"]), _ptr(b["workspace"]),
                           b["workspace"].numel() * b["workspace"].element_size())


def _host_ptr(t):
    if t.is_cuda:
        raise ValueError("moe_path_host takes host tensors for x_host, logits_host and out_host")
    if not t.is_contiguous():
        raise ValueError("libmoe_gb300 takes contiguous tensors only")
    return t.data_ptr()


class HostPath:
    """moe_path_host with its arguments marshalled once: every call() issues
    one batch (H2D of x and logits, the four stages, D2H of out) on `stream`."""

    def __init__(self, p: moe_problem, x_host, logits_host, s, x_dev, logits_dev, bufs: dict, out_dev, out_host,
                 stream=None):
        self.p = p
        self.ub = ubatch_bufs(bufs)
        self.args = (C.byref(self.p), _host_ptr(x_host), _host_ptr(logits_host), _ptr(s), _ptr(x_dev),
                     _ptr(logits_dev), C.byref(self.ub), _ptr(out_dev), _host_ptr(out_host), _stream(stream))
        self.fn = lib().moe_path_host
        self._keep = (x_host, logits_host, s, x_dev, logits_dev, bufs, out_dev, out_host)

    def __call__(self):
        _check("moe_path_host", self.fn(*self.args))


def moe_path_host(p, x_host, logits_host, s, x_dev, logits_dev, bufs: dict, out_dev, out_host, stream=None):
    """The whole path with host inputs and output, in one call (asynchronous on `stream`)."""
    HostPath(p, x_host, logits_host, s, x_dev, logits_dev, bufs, out_dev, out_host, stream)()


def dbo_step(ctx: DboContext, p_full, x, logits, s, bufs2, out, compute_stream, comm_stream, record_timing=False):
    arr = (moe_ubatch_bufs * 2)(ubatch_bufs(bufs2[0]), ubatch_bufs(bufs2[1]))
    rc = lib().dbo_step(ctx.handle, C.byref(p_full), _ptr(x), _ptr(logits), _ptr(s), arr, _ptr(out),
                        _stream(compute_stream), _stream(comm_stream), int(bool(record_timing)))
    _check("dbo_step", rc)


def dbo_read_timing(ctx: DboContext) -> dict:
    t = moe_dbo_timing()
    _check("dbo_read_timing", lib().dbo_read_timing(ctx.handle, C.byref(t)))
    return {n: getattr(t, n) for n, _ in moe_dbo_timing._fields_}


def alloc_buffers(p: moe_problem, device="cuda") -> dict:
    """Device buffers of every output of the path for problem p (torch.empty:
    contents undefined until written). Row buffers are bf16 stored as int16
    (or uint8 e4m3 codes)."""
    import torch
    T, H, E, k, R, Cap = p.num_tokens, p.hidden, p.num_experts, p.top_k, p.num_ranks, p.capacity
    fp8 = p.dispatch_dtype == MOE_DTYPE_FP8_E4M3_B128
    i32 = dict(dtype=torch.int32, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    ws = max(moe_route_workspace_bytes(p), moe_route_dispatch_workspace_bytes(p))
    if ws == 0:
        raise MoeError("moe_route_workspace_bytes", MOE_ERR_INVALID_ARG)
    b = {
        "topk_idx": torch.empty((T, k), **i32), "topk_w": torch.empty((T, k), **f32),
        "counts": torch.empty(E, **i32), "offsets": torch.empty(E + 1, **i32),
        "slot": torch.empty((T, k), **i32), "rank_counts": torch.empty(R, **i32),
        "dropped": torch.empty(1, **i32),
        "recv": torch.empty((E, Cap, H), dtype=torch.uint8 if fp8 else torch.int16, device=device),
        "recv_scale": torch.empty((E, Cap, H // 128), **f32) if fp8 else None,
        "recv_src": torch.empty((E, Cap), **i32),
        "y": torch.empty((E, Cap, H), dtype=torch.int16, device=device),
        "workspace": torch.empty(ws, dtype=torch.uint8, device=device),
        # per-row readiness flags of moe_expert_combine: zero-filled once, then epoch-tagged
        "ready_flags": torch.zeros(max(moe_ready_flags_bytes(p) // 4, 1), **i32),
    }
    return b


def run_path(p: moe_problem, x, logits, s, bufs: dict, out, stream=None, fused=False):
    """route -> dispatch -> synthetic expert -> combine for one batch, on one stream
    (fused: route and dispatch through moe_route_dispatch)."""
    if fused:
        moe_route_dispatch(p, logits, x, bufs["topk_idx"], bufs["topk_w"], bufs["counts"], bufs["offsets"],
                           bufs["slot"], bufs["rank_counts"], bufs["dropped"], bufs["recv"], bufs.get("recv_scale"),
                           bufs["recv_src"], bufs["workspace"], stream)
    else:
        moe_route(p, logits, bufs["topk_idx"], bufs["topk_w"], bufs["counts"], bufs["offsets"], bufs["slot"],
                  bufs["rank_counts"], bufs["dropped"], bufs["workspace"], stream)
        moe_dispatch(p, x, bufs["topk_idx"], bufs["slot"], bufs["recv"], bufs.get("recv_scale"), bufs["recv_src"],
                     stream)
    moe_expert_synthetic(p, bufs["recv"], bufs.get("recv_scale"), bufs["counts"], s, bufs["y"], stream)
    moe_combine(p, bufs["y"], bufs["topk_idx"], bufs["topk_w"], bufs["slot"], out, stream)


def moe_layer_stand_in(x, out, a: float, busy_fmas: int = 0, stream=None):
    """out = bf16(x * a) (+ busy work that does not change the output)."""
    _check("moe_layer_stand_in", lib().moe_layer_stand_in(_ptr(x), _ptr(out), x.numel(), float(a), int(busy_fmas),
                                                          _stream(stream)))


def dbo_layers_args(p_full, n_layers, x, logits, s, bufs2, h, shared, out, alpha=1.0, sigma=1.0, busy_fmas=0,
                    expert_w=None, mlp_max_blocks=0):
    """moe_dbo_layers_args from tensors (the struct keeps raw pointers: keep the tensors alive).
    expert_w: [E][H][H] bf16 weights for the grouped GEMM as the MLP, or None for the synthetic expert."""
    a = moe_dbo_layers_args()
    a.full = p_full
    a.n_layers, a.busy_fmas, a.alpha, a.sigma = int(n_layers), int(busy_fmas), float(alpha), float(sigma)
    a.x, a.logits, a.s = _ptr(x), _ptr(logits), _ptr(s)
    a.bufs[0], a.bufs[1] = ubatch_bufs(bufs2[0]), ubatch_bufs(bufs2[1])
    a.h, a.shared, a.out = _ptr(h), _ptr(shared), _ptr(out)
    a.expert_w, a.mlp_max_blocks = _ptr(expert_w), int(mlp_max_blocks)
    return a


def dbo_layers(ctx: DboContext, args, compute_stream, comm_stream):
    _check("dbo_layers", lib().dbo_layers(ctx.handle, C.byref(args), _stream(compute_stream), _stream(comm_stream)))


def dbo_layers_capture(ctx: DboContext, args, compute_stream, comm_stream):
    _check("dbo_layers_capture", lib().dbo_layers_capture(ctx.handle, C.byref(args), _stream(compute_stream),
                                                          _stream(comm_stream)))


def dbo_graph_launch(ctx: DboContext, stream=None):
    _check("dbo_graph_launch", lib().dbo_graph_launch(ctx.handle, _stream(stream)))
