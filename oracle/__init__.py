"""CPU oracle for the MoE route / dispatch / combine path (numpy front end).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (``bench.py --impl reference`` and the
``cpu_baseline`` object) may import this package. The product path never does:
the CUDA library and its binding share no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain, single-threaded C); this module
only marshals numpy arrays. Page citations are in the C source:
  [PMC] "Efficient and portable mixture-of-experts communication"
  [DBO] "Dual Batch Overlap"
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        # MOE_ORACLE_LIB: a separately compiled copy of the oracle (the mutation
        # tests plant one mistake in a copy and check that the pins catch it)
        path = os.environ.get("MOE_ORACLE_LIB") or _build()
        L = C.CDLL(path)
        P = C.c_void_p
        i32, i64 = C.c_int32, C.c_int64
        for name, args in {
            "oracle_bf16_encode": [P, P, i64],
            "oracle_bf16_decode": [P, P, i64],
            "oracle_e4m3_encode": [P, P, i64],
            "oracle_e4m3_decode": [P, P, i64],
            "oracle_route": [i32, i32, i32, P, P, P, P],
            "oracle_count": [i32, i32, i32, i32, i32, P, P, P, P, P, P],
            "oracle_dispatch_bf16": [i32, i32, i32, i32, i32, P, P, P, P, P],
            "oracle_dispatch_fp8": [i32, i32, i32, i32, i32, P, P, P, P, P, P],
            "oracle_expert_synthetic": [i32, i32, i32, i32, P, P, P, P, P],
            "oracle_combine": [i32, i32, i32, i32, i32, P, P, P, P, P],
            "oracle_src_offsets": [i32, i32, i32, i32, P, P, P],
            "oracle_scale_rows": [i64, P, C.c_float, P],
            "oracle_gemm_fp8_row": [i32, i32, P, P, P, P, P],
            "oracle_expert_gemm_fp8": [i32, i32, i32, i32, P, P, P, P, P, P],
            "oracle_gemm_bf16_row": [i32, i32, P, P, P],
            "oracle_expert_gemm_bf16": [i32, i32, i32, i32, P, P, P, P],
        }.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = None if name.startswith(("oracle_bf16", "oracle_e4m3")) else C.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: invalid argument")


# ---- codecs -----------------------------------------------------------------

def bf16_encode(f32: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(f32, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_bf16_encode(_p(a), _p(out), a.size)
    return out


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(a.shape, dtype=np.float32)
    lib().oracle_bf16_decode(_p(a), _p(out), a.size)
    return out


def e4m3_encode(f32: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(f32, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode(_p(a), _p(out), a.size)
    return out


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(a.shape, dtype=np.float32)
    lib().oracle_e4m3_decode(_p(a), _p(out), a.size)
    return out


# ---- the path, step by step ---------------------------------------------------

def route(logits: np.ndarray, k: int, with_double: bool = False):
    """Top-k of each row of logits[T][E] and the renormalised softmax weights."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    w64 = np.empty((T, k), dtype=np.float64) if with_double else None
    _check(lib().oracle_route(T, E, k, _p(lg), _p(idx), _p(w), _p(w64)), "oracle_route")
    return (idx, w, w64) if with_double else (idx, w)


def count(topk_idx: np.ndarray, E: int, R: int, Cap: int) -> dict:
    """Histogram, exclusive scan, slots, per-rank row counts and drops."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    slot = np.empty((T, k), dtype=np.int32)
    rank_counts = np.empty(R, dtype=np.int32)
    dropped = np.zeros(1, dtype=np.int32)
    _check(lib().oracle_count(T, E, k, R, Cap, _p(idx), _p(counts), _p(offsets), _p(slot),
                              _p(rank_counts), _p(dropped)), "oracle_count")
    return {"counts": counts, "offsets": offsets, "slot": slot,
            "rank_counts": rank_counts, "dropped": int(dropped[0])}


def dispatch_bf16(x: np.ndarray, topk_idx, slot, E: int, Cap: int, fill: int = 0):
    xb = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = xb.shape
    k = topk_idx.shape[1]
    # untouched pages of np.zeros stay unallocated: only written rows cost memory
    recv_x = np.zeros((E, Cap, H), dtype=np.uint16) if fill == 0 else np.full((E, Cap, H), fill, dtype=np.uint16)
    recv_src = np.full((E, Cap), -1, dtype=np.int32)
    _check(lib().oracle_dispatch_bf16(T, H, E, k, Cap, _p(xb), _p(np.ascontiguousarray(topk_idx, dtype=np.int32)),
                                      _p(np.ascontiguousarray(slot, dtype=np.int32)), _p(recv_x), _p(recv_src)),
           "oracle_dispatch_bf16")
    return recv_x, recv_src


def dispatch_fp8(x: np.ndarray, topk_idx, slot, E: int, Cap: int):
    xb = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = xb.shape
    k = topk_idx.shape[1]
    recv_q = np.zeros((E, Cap, H), dtype=np.uint8)
    recv_scale = np.zeros((E, Cap, H // 128), dtype=np.float32)
    recv_src = np.full((E, Cap), -1, dtype=np.int32)
    _check(lib().oracle_dispatch_fp8(T, H, E, k, Cap, _p(xb), _p(np.ascontiguousarray(topk_idx, dtype=np.int32)),
                                     _p(np.ascontiguousarray(slot, dtype=np.int32)), _p(recv_q), _p(recv_scale),
                                     _p(recv_src)), "oracle_dispatch_fp8")
    return recv_q, recv_scale, recv_src


def src_offsets(topk_idx, slot, E: int, tokens_per_src_rank: int):
    """[E][S+1]: per expert, the number of kept pairs from source ranks below s (s = 0 .. S)."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    tps = int(tokens_per_src_rank)
    S = max(1, -(-T // tps)) if tps > 0 else 1
    out = np.empty((E, S + 1), dtype=np.int32)
    _check(lib().oracle_src_offsets(T, E, k, tps, _p(idx), _p(np.ascontiguousarray(slot, dtype=np.int32)), _p(out)),
           "oracle_src_offsets")
    return out


def expert_synthetic(recv, recv_scale, counts, s):
    """y = bf16(x * s_e) (bf16 recv) or bf16((q * scale) * s_e) (fp8 recv); valid rows only."""
    E, Cap, H = recv.shape
    fp8 = recv.dtype == np.uint8
    y = np.zeros((E, Cap, H), dtype=np.uint16)
    rs = np.ascontiguousarray(recv_scale, dtype=np.float32) if fp8 else None
    _check(lib().oracle_expert_synthetic(H, E, Cap, int(fp8), _p(np.ascontiguousarray(recv)), _p(rs),
                                         _p(np.ascontiguousarray(counts, dtype=np.int32)),
                                         _p(np.ascontiguousarray(s, dtype=np.float32)), _p(y)),
           "oracle_expert_synthetic")
    return y


def expert_gemm_fp8(recv_q, recv_scale, counts, w_q, w_scale):
    """Grouped fp8 GEMM on the dispatch layout: y[e][r] = bf16(sum over 128-blocks of
    a_scale * w_scale * (q . w[e][n])) for r < min(counts[e], C); other rows zero.
    recv_q [E][C][K] u8, recv_scale [E][C][K/128] f32, w_q [E][N][K] u8,
    w_scale [E][N/128][K/128] f32 -> y [E][C][N] bf16 bits."""
    E, Cap, K = recv_q.shape
    N = w_q.shape[1]
    y = np.zeros((E, Cap, N), dtype=np.uint16)
    _check(lib().oracle_expert_gemm_fp8(K, N, E, Cap, _p(np.ascontiguousarray(recv_q, dtype=np.uint8)),
                                        _p(np.ascontiguousarray(recv_scale, dtype=np.float32)),
                                        _p(np.ascontiguousarray(counts, dtype=np.int32)),
                                        _p(np.ascontiguousarray(w_q, dtype=np.uint8)),
                                        _p(np.ascontiguousarray(w_scale, dtype=np.float32)), _p(y)),
           "oracle_expert_gemm_fp8")
    return y


def gemm_fp8_row(q_row, a_scale_row, w_q_e, w_scale_e):
    """One output row of the grouped GEMM: q_row [K] u8, a_scale_row [K/128] f32,
    w_q_e [N][K] u8, w_scale_e [N/128][K/128] f32 -> [N] bf16 bits."""
    N, K = w_q_e.shape
    y = np.empty(N, dtype=np.uint16)
    _check(lib().oracle_gemm_fp8_row(K, N, _p(np.ascontiguousarray(q_row, dtype=np.uint8)),
                                     _p(np.ascontiguousarray(a_scale_row, dtype=np.float32)),
                                     _p(np.ascontiguousarray(w_q_e, dtype=np.uint8)),
                                     _p(np.ascontiguousarray(w_scale_e, dtype=np.float32)), _p(y)),
           "oracle_gemm_fp8_row")
    return y


def expert_gemm_bf16(recv_x, counts, w):
    """Grouped bf16 GEMM on the dispatch layout: y[e][r] = bf16(sum_i x[e][r][i] * w[e][n][i]) (double sums)
    for r < min(counts[e], C); other rows zero. recv_x [E][C][K], w [E][N][K] bf16 bits -> y [E][C][N]."""
    E, Cap, K = recv_x.shape
    N = w.shape[1]
    y = np.zeros((E, Cap, N), dtype=np.uint16)
    _check(lib().oracle_expert_gemm_bf16(K, N, E, Cap, _p(np.ascontiguousarray(recv_x, dtype=np.uint16)),
                                         _p(np.ascontiguousarray(counts, dtype=np.int32)),
                                         _p(np.ascontiguousarray(w, dtype=np.uint16)), _p(y)),
           "oracle_expert_gemm_bf16")
    return y


def gemm_bf16_row(x_row, w_e):
    """One output row of the bf16 grouped GEMM: x_row [K], w_e [N][K] bf16 bits -> [N] bf16 bits."""
    N, K = w_e.shape
    y = np.empty(N, dtype=np.uint16)
    _check(lib().oracle_gemm_bf16_row(K, N, _p(np.ascontiguousarray(x_row, dtype=np.uint16)),
                                      _p(np.ascontiguousarray(w_e, dtype=np.uint16)), _p(y)), "oracle_gemm_bf16_row")
    return y


def combine(y: np.ndarray, topk_idx, topk_w, slot, T: int):
    E, Cap, H = y.shape
    k = topk_idx.shape[1]
    out = np.empty((T, H), dtype=np.uint16)
    _check(lib().oracle_combine(T, H, E, k, Cap, _p(np.ascontiguousarray(y, dtype=np.uint16)),
                                _p(np.ascontiguousarray(topk_idx, dtype=np.int32)),
                                _p(np.ascontiguousarray(topk_w, dtype=np.float32)),
                                _p(np.ascontiguousarray(slot, dtype=np.int32)), _p(out)), "oracle_combine")
    return out


def run_path(x, logits, s, k: int, R: int, Cap: int, fp8: bool, expert_w=None) -> dict:
    """Route -> count -> dispatch -> experts -> combine on one batch. The experts are the
    synthetic stand-in y = x * s_e, or with expert_w ([E][H][H] bf16 bits, bf16 rows only)
    the grouped GEMM y[e][r] = bf16(sum_i x_i w[e][n][i])."""
    T, E = logits.shape
    idx, w = route(logits, k)
    c = count(idx, E, R, Cap)
    if fp8:
        assert expert_w is None, "GEMM experts on fp8 rows take block-scaled weights: expert_gemm_fp8"
        rq, rs, src = dispatch_fp8(x, idx, c["slot"], E, Cap)
        y = expert_synthetic(rq, rs, c["counts"], s)
        res = {"recv_q": rq, "recv_scale": rs}
    else:
        rx, src = dispatch_bf16(x, idx, c["slot"], E, Cap)
        y = expert_synthetic(rx, None, c["counts"], s) if expert_w is None else expert_gemm_bf16(rx, c["counts"], expert_w)
        res = {"recv_x": rx}
    out = combine(y, idx, w, c["slot"], T)
    res.update(c)
    res.update({"topk_idx": idx, "topk_w": w, "recv_src": src, "y": y, "out": out})
    return res


def micro_batches(T: int):
    """[DBO §UBatchRunner]: the batch is split at its midpoint into two
    micro-batches; a micro-batch with no tokens runs as an empty (dummy) batch.
    Returns the token ranges [(0, T//2), (T//2, T)]."""
    m = T // 2
    return [(0, m), (m, T)]


def run_dbo(x, logits, s, k: int, R: int, Cap: int, fp8: bool) -> dict:
    """The two-micro-batch step: each half runs the whole path on its own
    buffers; the output is the two halves' outputs in token order."""
    T, E = logits.shape
    H = x.shape[1]
    outs, parts = [], []
    for (a, b) in micro_batches(T):
        if b == a:
            parts.append(None)
            outs.append(np.empty((0, H), dtype=np.uint16))
            continue
        r = run_path(x[a:b], logits[a:b], s, k, R, Cap, fp8)
        parts.append(r)
        outs.append(r["out"])
    return {"out": np.concatenate(outs, axis=0), "parts": parts}


def scale_rows(x: np.ndarray, a: float) -> np.ndarray:
    """bf16(float(x) * a), the stand-in for the layer compute around the MoE block."""
    xb = np.ascontiguousarray(x, dtype=np.uint16)
    out = np.empty_like(xb)
    _check(lib().oracle_scale_rows(xb.size, _p(xb), float(np.float32(a)), _p(out)), "oracle_scale_rows")
    return out


def run_dbo_layers(x, logits_layers, s, k: int, R: int, Cap: int, alpha: float, sigma: float,
                   expert_w=None) -> dict:
    """Layers of the dual-batch-overlap schedule, micro-batch by micro-batch.
    [DBO §Introduction]: per layer and micro-batch u, A0 (here h = bf16(x a)),
    A1 (the MoE gate: route on the layer's logits), dispatch of h, the experts
    (the synthetic stand-in, or the grouped GEMM with expert_w), S (shared
    expert: bf16(h s)) and combine, whose output is the next layer's input.
    Returns the last layer's output and shared-expert output."""
    L, T, E = logits_layers.shape
    H = x.shape[1]
    out = np.empty((T, H), dtype=np.uint16)
    shared = np.empty((T, H), dtype=np.uint16)
    for (a, b) in micro_batches(T):
        if b == a:
            continue
        xu = np.ascontiguousarray(x[a:b])
        for l in range(L):
            h = scale_rows(xu, alpha)
            r = run_path(h, logits_layers[l, a:b], s, k, R, Cap, False, expert_w)
            shared[a:b] = scale_rows(h, sigma)
            xu = r["out"]
        out[a:b] = xu
    return {"out": out, "shared": shared}
