"""Pins of the CPU oracle's path: route, count, dispatch, expert, combine.

Each pin ties the oracle to something other than itself: brute force on tiny
inputs, library routines (numpy stable argsort, torch float64 softmax, torch
casts), closed forms, invariants, and a worked example derived by hand
(tests/golden/worked_tiny.json).

Pages: [PMC] "Efficient and portable mixture-of-experts communication";
[DBO] "Dual Batch Overlap".
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(vals):
    return torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def bf16_ulp_distance(a_bits, b_bits):
    """Distance in representable bf16 steps between two bit patterns (finite values)."""
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + (b & 0x7FFF))
    return np.abs(ordered(a_bits) - ordered(b_bits))


# ---- worked example -----------------------------------------------------------

def test_worked_example_by_hand():
    with open(os.path.join(GOLDEN, "worked_tiny.json")) as fh:
        g = json.load(fh)
    lg = np.array([[float(v) for v in row] for row in g["logits"]], dtype=np.float32)
    assert np.signbit(lg[2, 0])
    x = bf16_bits(g["x"])
    s = np.array(g["s"], dtype=np.float32)
    ex = g["expected"]
    r = O.run_path(x, lg, s, g["k"], g["R"], g["C"], fp8=False)
    assert r["topk_idx"].tolist() == ex["topk_idx"]
    assert np.allclose(r["topk_w"], np.array(ex["topk_w"]), rtol=1e-6, atol=0)
    assert r["counts"].tolist() == ex["counts"]
    assert r["offsets"].tolist() == ex["offsets"]
    assert r["slot"].tolist() == ex["slot"]
    assert r["rank_counts"].tolist() == ex["rank_counts"]
    assert r["dropped"] == ex["dropped"]
    assert r["recv_src"].tolist() == ex["recv_src"]
    assert np.array_equal(r["out"], bf16_bits(ex["out"]))


# ---- route ------------------------------------------------------------------

def brute_force_topk(l, k):
    """The k-subset whose keys (logit, -index), sorted descending, are
    lexicographically largest; returned in that order."""
    E = len(l)
    best = None
    for sub in itertools.combinations(range(E), k):
        keys = sorted(((float(l[e]) + 0.0, -e) for e in sub), reverse=True)
        if best is None or keys > best:
            best = keys
    return [-e for (_, e) in best]


@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (8, 3), (6, 6), (9, 4)])
def test_topk_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 100 + k)
    # few distinct values -> many ties; include signed zeros
    vals = np.array([-1.0, -0.0, 0.0, 0.5, 2.0], dtype=np.float32)
    lg = vals[rng.integers(0, len(vals), size=(200, E))]
    idx, _ = O.route(lg, k)
    for t in range(lg.shape[0]):
        assert idx[t].tolist() == brute_force_topk(lg[t], k), (t, lg[t])


def test_topk_matches_numpy_stable_argsort(inputs_of):
    for name in ["v2lite", "dsv3_fp8", "mixtral_skew"]:
        w = W.WORKLOADS[name]
        lg = inputs_of(name)["logits"]
        idx, _ = O.route(lg, w.k)
        ref = np.argsort(-lg, axis=1, kind="stable")[:, :w.k]
        assert np.array_equal(idx, ref), name


def test_topk_signed_zero_is_a_tie():
    lg = np.array([[0.0, -0.0, -1.0], [-0.0, 0.0, -1.0]], dtype=np.float32)
    idx, w = O.route(lg, 1)
    assert idx[:, 0].tolist() == [0, 0]
    assert w[:, 0].tolist() == [1.0, 1.0]


def test_all_equal_logits():
    lg = np.full((3, 16), 0.25, dtype=np.float32)
    idx, w = O.route(lg, 8)
    assert idx.tolist() == [list(range(8))] * 3
    assert np.all(w == np.float32(1 / 8))


def test_k1_weight_is_exactly_one(inputs_of):
    lg = inputs_of("v2lite")["logits"]
    idx, w = O.route(lg, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(idx[:, 0], np.argmax(lg, axis=1))


def test_k_equals_E_is_full_softmax_float64():
    rng = np.random.default_rng(3)
    lg = (rng.standard_normal((64, 16)) * 3).astype(np.float32)
    idx, w, w64 = O.route(lg, 16, with_double=True)
    assert np.array_equal(idx, np.argsort(-lg, axis=1, kind="stable"))
    p = torch.softmax(torch.from_numpy(lg.astype(np.float64)), dim=1).numpy()
    assert np.allclose(w64, np.take_along_axis(p, idx, axis=1), rtol=1e-12, atol=0)


def test_weights_are_renormalised_full_softmax(inputs_of):
    """Softmax over all E experts restricted to the chosen k and renormalised
    equals the oracle's k-only form (exact-arithmetic identity)."""
    for name in ["v2lite", "dsv3_fp8", "mixtral_skew"]:
        w = W.WORKLOADS[name]
        lg = inputs_of(name)["logits"]
        idx, wf, w64 = O.route(lg, w.k, with_double=True)
        p = torch.softmax(torch.from_numpy(lg.astype(np.float64)), dim=1).numpy()
        sel = np.take_along_axis(p, idx, axis=1)
        ref = sel / sel.sum(axis=1, keepdims=True)
        assert np.allclose(w64, ref, rtol=1e-12, atol=0), name
        assert np.all(np.abs(w64.sum(axis=1) - 1.0) <= 4 * np.finfo(np.float64).eps)
        assert np.array_equal(wf, w64.astype(np.float32))
        # descending weights follow descending logits
        assert np.all(np.diff(w64, axis=1) <= 0)


# ---- count / scan / slot --------------------------------------------------------

def brute_force_count(idx, E, R, Cap):
    T, k = idx.shape
    counts = np.zeros(E, np.int64)
    slot = np.zeros((T, k), np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            pos = sum(1 for tt in range(t) if e in idx[tt].tolist())
            slot[t, j] = pos if pos < Cap else -1
            counts[e] += 1
    offsets = np.concatenate([[0], np.cumsum(counts)])
    per = E // R
    rank_counts = [int(np.minimum(counts[r * per:(r + 1) * per], Cap).sum()) for r in range(R)]
    dropped = int(np.maximum(counts - Cap, 0).sum())
    return counts, offsets, slot, rank_counts, dropped


@pytest.mark.parametrize("T,E,k,R,Cap", [(40, 8, 2, 2, 64), (40, 8, 3, 4, 6), (33, 6, 6, 3, 20), (0, 4, 2, 2, 4), (1, 4, 4, 1, 1)])
def test_count_brute_force(T, E, k, R, Cap):
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = O.route(lg, k)
    c = O.count(idx, E, R, Cap)
    counts, offsets, slot, rank_counts, dropped = brute_force_count(idx, E, R, Cap)
    assert c["counts"].tolist() == counts.tolist()
    assert c["offsets"].tolist() == offsets.tolist()
    assert c["slot"].tolist() == slot.tolist()
    assert c["rank_counts"].tolist() == rank_counts
    assert c["dropped"] == dropped


def test_count_invariants_at_workload_sizes(inputs_of):
    for name in ["v2lite", "mixtral_skew", "dsv3_fp8"]:
        w = W.WORKLOADS[name]
        idx, _ = O.route(inputs_of(name)["logits"], w.k)
        c = O.count(idx, w.E, w.R, w.C)
        assert c["counts"].tolist() == np.bincount(idx.ravel(), minlength=w.E).tolist()
        assert c["offsets"][-1] == w.T * w.k
        assert np.array_equal(np.diff(c["offsets"]), c["counts"])
        for e in range(w.E):
            t_of, j_of = np.nonzero(idx == e)          # row-major: ascending t
            sl = c["slot"][t_of, j_of]
            kept = min(c["counts"][e], w.C)
            assert sl[:kept].tolist() == list(range(kept))
            assert np.all(sl[kept:] == -1)
        # a token never selects one expert twice
        assert all(len(set(r)) == w.k for r in idx.tolist())


def test_skewed_workload_is_skewed(inputs_of):
    """The Zipf-biased logits put most tokens on expert 0 (hot expert)."""
    w = W.WORKLOADS["mixtral_skew"]
    idx, _ = O.route(inputs_of("mixtral_skew")["logits"], w.k)
    c = O.count(idx, w.E, w.R, w.C)
    assert c["counts"][0] > 3000 and np.all(np.diff(c["counts"]) <= 0)
    assert c["dropped"] == 0


# ---- dispatch ----------------------------------------------------------------

def test_dispatch_bf16_is_a_bit_copy_and_src_inverts_slot(inputs_of):
    w = W.WORKLOADS["v2lite"]
    d = inputs_of("v2lite")
    idx, _ = O.route(d["logits"], w.k)
    c = O.count(idx, w.E, w.R, w.C)
    rx, src = O.dispatch_bf16(d["x"], idx, c["slot"], w.E, w.C, fill=0xFFFF)
    for t in range(w.T):
        for j in range(w.k):
            e, s = idx[t, j], c["slot"][t, j]
            assert s >= 0
            assert np.array_equal(rx[e, s], d["x"][t])
            assert src[e, s] == t
    for e in range(w.E):   # rows past the count are never written
        n = c["counts"][e]
        assert np.all(rx[e, n:] == 0xFFFF) and np.all(src[e, n:] == -1)


def test_dispatch_rows_grouped_by_source_rank(inputs_of):
    """[PMC §Dispatch]: the tokens of one expert are grouped together across
    the DP source ranks. With slots ascending in token order, an expert's rows
    come from source rank 0 first, then 1, and so on."""
    w = W.WORKLOADS["dsv3_fp8"]
    idx, _ = O.route(inputs_of("dsv3_fp8")["logits"], w.k)
    c = O.count(idx, w.E, w.R, w.C)
    per_src = w.T // w.src_ranks
    for e in range(w.E):
        t_of = np.nonzero(idx == e)[0]
        assert np.all(np.diff(t_of // per_src) >= 0)


@pytest.mark.parametrize("name,tps", [("dsv3_fp8", 128), ("dsv3_fp8", 100), ("v2lite", 0), ("v2lite", 1),
                                      ("mixtral_skew", 512)])
def test_src_offsets_bound_each_source_ranks_rows(name, tps, inputs_of):
    """[PMC §Dispatch] groups one expert's tokens across the DP ranks that sent them. The offsets,
    counted over the pairs, must cut the dispatched rows (placed by the slots) at the source-rank
    boundaries: numpy's searchsorted over recv_src // tps finds the same cuts; the last offset is the
    expert's kept rows; per source, the rows over all experts are that source's kept pairs."""
    w = W.WORKLOADS[name]
    d = inputs_of(name)
    T = w.T if name != "mixtral_skew" else 1000              # a partial last source rank too
    r = O.run_path(d["x"][:T], d["logits"][:T], d["s"], w.k, w.R, min(w.C, 200), False)
    Cap = min(w.C, 200)
    off = O.src_offsets(r["topk_idx"], r["slot"], w.E, tps)
    S = max(1, -(-T // tps)) if tps > 0 else 1
    per = tps if tps > 0 else T
    assert off.shape == (w.E, S + 1)
    kept = np.minimum(r["counts"], Cap)
    assert np.array_equal(off[:, 0], np.zeros(w.E)) and np.array_equal(off[:, S], kept)
    for e in range(w.E):
        src_rank = r["recv_src"][e, :kept[e]] // per
        assert np.all(np.diff(src_rank) >= 0)
        assert np.array_equal(off[e], np.searchsorted(src_rank, np.arange(S + 1), side="left"))
    for s_ in range(S):
        rows = int(np.sum(off[:, s_ + 1] - off[:, s_]))
        assert rows == int(np.sum(r["slot"][s_ * per:(s_ + 1) * per] >= 0))


def test_dispatch_fp8_against_torch_and_bounds(inputs_of):
    w = W.WORKLOADS["dsv3_fp8"]
    d = inputs_of("dsv3_fp8")
    T = 64
    x = d["x"][:T]
    idx, _ = O.route(d["logits"][:T], w.k)
    c = O.count(idx, w.E, w.R, w.C)
    rq, rs, src = O.dispatch_fp8(x, idx, c["slot"], w.E, w.C)
    xf = bf16_vals(x).reshape(T, -1, 128)
    amax = np.abs(xf).max(axis=2)
    scale_ref = np.where(amax == 0, np.float32(1), amax / np.float32(448)).astype(np.float32)
    q_ref = torch.from_numpy(xf / scale_ref[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t in range(T):
        for j in range(w.k):
            e, s = idx[t, j], c["slot"][t, j]
            assert np.array_equal(rs[e, s], scale_ref[t])
            assert np.array_equal(rq[e, s], q_ref[t].reshape(-1))
            assert src[e, s] == t
    # dequantisation error bound of round-to-nearest e4m3 within each block
    e0, s0 = idx[:, 0], c["slot"][:, 0]
    deq = O.e4m3_decode(rq[e0, s0]).reshape(T, -1, 128) * rs[e0, s0][:, :, None]
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, rs[e0, s0][:, :, None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(deq - xf) <= bound)
    # the largest element of every block maps to +-448
    qa = np.abs(O.e4m3_decode(rq[e0, s0]).reshape(T, -1, 128)).max(axis=2)
    assert np.all(qa == 448.0)


def test_dispatch_fp8_zero_block():
    x = np.zeros((2, 256), dtype=np.uint16)
    x[1, 128:] = bf16_bits(np.linspace(-3, 3, 128))
    idx = np.array([[0], [1]], np.int32)
    slot = np.array([[0], [0]], np.int32)
    rq, rs, _ = O.dispatch_fp8(x, idx, slot, 2, 1)
    assert rs[0, 0].tolist() == [1.0, 1.0] and np.all(rq[0, 0] == 0)
    assert rs[1, 0, 0] == 1.0 and rs[1, 0, 1] == np.float32(3) / np.float32(448)


# ---- synthetic expert ----------------------------------------------------------

def test_expert_identity_and_power_of_two(inputs_of):
    d = inputs_of("tiny")
    E, Cap, H = 4, 16, 256
    rx = d["x"][:E * Cap].reshape(E, Cap, H).copy()
    counts = np.array([16, 3, 0, 40], np.int32)
    y1 = O.expert_synthetic(rx, None, counts, np.ones(E, np.float32))
    y2 = O.expert_synthetic(rx, None, counts, np.full(E, 2.0, np.float32))
    for e in range(E):
        n = min(counts[e], Cap)
        assert np.array_equal(y1[e, :n], rx[e, :n])
        assert np.array_equal(bf16_vals(y2[e, :n]), 2 * bf16_vals(rx[e, :n]))
        assert np.all(y1[e, n:] == 0)


def test_expert_rounding_bound(inputs_of):
    w = W.WORKLOADS["tiny"]
    d = inputs_of("tiny")
    rx = d["x"].reshape(w.E, w.T // w.E, w.H)
    counts = np.full(w.E, w.T // w.E, np.int32)
    y = O.expert_synthetic(rx, None, counts, d["s"])
    exact = bf16_vals(rx).astype(np.float64) * d["s"][:, None, None]
    # bf16 keeps 8 significant bits: rounding to nearest moves a value by at most 2^-8 of it
    assert np.all(np.abs(bf16_vals(y) - exact) <= np.abs(exact) * 2.0 ** -8)


# ---- combine -----------------------------------------------------------------

def test_combine_k1_unit_scale_returns_x(inputs_of):
    w = W.WORKLOADS["v2lite"]
    d = inputs_of("v2lite")
    r = O.run_path(d["x"], d["logits"], np.ones(w.E, np.float32), 1, w.R, w.C, fp8=False)
    assert np.array_equal(r["out"], d["x"])


def test_combine_unit_scale_within_one_ulp_of_x(inputs_of):
    w = W.WORKLOADS["v2lite"]
    d = inputs_of("v2lite")
    r = O.run_path(d["x"], d["logits"], np.ones(w.E, np.float32), w.k, w.R, w.C, fp8=False)
    assert bf16_ulp_distance(r["out"], d["x"]).max() <= 1


@pytest.mark.parametrize("name", ["tiny", "v2lite", "mixtral_skew"])
def test_combine_closed_form(name, inputs_of):
    """out_t = sum_j w_j * s_{e_j} * x_t (closed form of the synthetic expert):
    the exact model sum_j w_j * bf16(x*s_e) in float64, rounded to bf16, is
    within 1 ulp; the unmodelled closed form within 2 ulps (every term has
    the sign of x_t, so nothing cancels)."""
    w = W.WORKLOADS[name]
    d = inputs_of(name)
    r = O.run_path(d["x"], d["logits"], d["s"], w.k, w.R, w.C, fp8=False)
    assert r["dropped"] == 0
    xf = bf16_vals(d["x"]).astype(np.float64)
    wv = r["topk_w"].astype(np.float64)
    se = d["s"][r["topk_idx"]].astype(np.float64)
    closed = xf * (wv * se).sum(axis=1, keepdims=True)
    ys = np.stack([bf16_vals(bf16_bits((xf * se[:, j:j + 1]).astype(np.float32))) for j in range(w.k)], axis=1)
    model = (wv[:, :, None] * ys.astype(np.float64)).sum(axis=1)
    assert bf16_ulp_distance(r["out"], bf16_bits(model.astype(np.float32))).max() <= 1
    assert bf16_ulp_distance(r["out"], bf16_bits(closed.astype(np.float32))).max() <= 2


def test_combine_fp8_closed_form_bound(inputs_of):
    w = W.WORKLOADS["dsv3_fp8"]
    d = inputs_of("dsv3_fp8")
    T = 128
    r = O.run_path(d["x"][:T], d["logits"][:T], d["s"], w.k, w.R, w.C, fp8=True)
    xf = bf16_vals(d["x"][:T]).astype(np.float64)
    coef = (r["topk_w"].astype(np.float64) * d["s"][r["topk_idx"]]).sum(axis=1, keepdims=True)
    out = bf16_vals(r["out"]).astype(np.float64)
    # per element: e4m3 error (<= 2^-4 |x| or 2^-10 scale) plus bf16 rounding
    sc = np.repeat(r["recv_scale"][r["topk_idx"][:, 0], r["slot"][:, 0]], 128, axis=1)
    bound = coef * np.maximum(np.abs(xf) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 2.0 ** -7) + np.abs(coef * xf) * 2.0 ** -7
    assert np.all(np.abs(out - coef * xf) <= bound + 1e-30)


def test_combine_skips_dropped_pairs_without_renormalising():
    rng = np.random.default_rng(5)
    T, E, k, H, Cap = 24, 4, 2, 16, 3
    lg = rng.standard_normal((T, E)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((T, H)))
    s = np.ones(E, np.float32)
    r = O.run_path(x, lg, s, k, 1, Cap, fp8=False)
    assert r["dropped"] > 0
    xf = bf16_vals(x).astype(np.float64)
    keep = (r["slot"] >= 0).astype(np.float64)
    model = xf * (r["topk_w"].astype(np.float64) * keep).sum(axis=1, keepdims=True)
    assert bf16_ulp_distance(r["out"], bf16_bits(model.astype(np.float32))).max() <= 1
    gone = np.all(r["slot"] < 0, axis=1)
    assert np.all(bf16_vals(r["out"][gone]) == 0)


def _exact(expr: str) -> float:
    """Value of a golden file's exact expression such as "2033633*2^-29", "1+2^-8" or "257/256"
    (every one of them is exactly representable in float64)."""
    return float(eval(expr.replace("^", "**"), {"__builtins__": {}}, {}))


def _f32_from_hex(h: str) -> np.float32:
    return np.array([int(h, 16)], dtype=np.uint32).view(np.float32)[0]


def _order_golden():
    with open(os.path.join(GOLDEN, "combine_fp32_order.json")) as fh:
        return json.load(fh)


@pytest.mark.parametrize("case", [c["name"] for c in _order_golden()["combine"]])
def test_combine_fp32_ascending_fma_order_by_hand(case):
    """[PMC §Combine] weighted sum, read as fp32 fused multiply-adds in ascending j from +0 and one
    bf16 rounding: hand-derived cases on which descending j, an unfused product, a double
    accumulator or a -0 start each give another bf16 result."""
    c = next(c for c in _order_golden()["combine"] if c["name"] == case)
    k = c["k"]
    w = np.array([[_f32_from_hex(h) for h in c["w_f32_bits"]]], dtype=np.float32)
    # the bit patterns are the exact values the derivation names
    assert [float(v) for v in w[0]] == [_exact(e) for e in c["w"]]
    y = np.array([int(h, 16) for h in c["y_bf16_bits"]], dtype=np.uint16).reshape(k, 1, 1)
    idx = np.arange(k, dtype=np.int32).reshape(1, k)
    slot = np.zeros((1, k), dtype=np.int32)
    out = O.combine(y, idx, w, slot, 1)
    assert int(out[0, 0]) == int(c["out_bf16_bits"], 16)


def test_expert_fp8_dequantise_then_scale_by_hand():
    """The synthetic expert on fp8 rows, y = bf16((q * scale) * s_e) in two fp32 products in that
    order ("dequant(x) * s_e"): a hand-derived element whose result differs from q * (scale * s_e)."""
    c = _order_golden()["expert_fp8"][0]
    H = c["H"]
    scale = _f32_from_hex(c["scale_f32_bits"])
    s_e = _f32_from_hex(c["s_e_f32_bits"])
    assert float(scale) == _exact(c["scale"]) and float(s_e) == _exact(c["s_e"])
    code = int(c["code"], 16)
    assert float(O.e4m3_decode(np.array([code], np.uint8))[0]) == _exact(c["q"])
    recv = np.zeros((2, 1, H), dtype=np.uint8)
    recv[1, 0, 0] = code
    recv[1, 0, 1] = code | 0x80                  # the same value negated: the result's negation
    recv_scale = np.full((2, 1, H // 128), scale, dtype=np.float32)
    counts = np.array([0, 1], dtype=np.int32)
    s = np.array([1.0, s_e], dtype=np.float32)
    y = O.expert_synthetic(recv, recv_scale, counts, s)
    want = int(c["y_bf16_bits"], 16)
    assert int(y[1, 0, 0]) == want
    assert int(y[1, 0, 1]) == want | 0x8000
    assert np.all(y[1, 0, 2:] == 0)


# ---- dual batch overlap split ------------------------------------------------------

def test_micro_batch_split_at_midpoint():
    assert O.micro_batches(8192) == [(0, 4096), (4096, 8192)]
    assert O.micro_batches(7) == [(0, 3), (3, 7)]
    assert O.micro_batches(1) == [(0, 0), (0, 1)]
    assert O.micro_batches(0) == [(0, 0), (0, 0)]


def test_dbo_output_is_the_two_halves_in_order(inputs_of):
    w = W.WORKLOADS["v2lite"]
    d = inputs_of("v2lite")
    r = O.run_dbo(d["x"], d["logits"], d["s"], w.k, w.R, w.C, fp8=False)
    a = O.run_path(d["x"][:128], d["logits"][:128], d["s"], w.k, w.R, w.C, False)
    b = O.run_path(d["x"][128:], d["logits"][128:], d["s"], w.k, w.R, w.C, False)
    assert np.array_equal(r["out"], np.concatenate([a["out"], b["out"]]))
    # splitting changes the slot layout but not the result of a token:
    # combine is per-token, so the single-shot output matches too
    full = O.run_path(d["x"], d["logits"], d["s"], w.k, w.R, w.C, False)
    assert np.array_equal(r["out"], full["out"])


# ---- layers of the dual-batch-overlap schedule ------------------------------------

def test_scale_rows_is_exact_for_powers_of_two_and_rounds_otherwise(inputs_of):
    x = inputs_of("tiny")["x"]
    assert np.array_equal(bf16_vals(O.scale_rows(x, 2.0)), 2 * bf16_vals(x))
    assert np.array_equal(O.scale_rows(x, 1.0), x)
    y = bf16_vals(O.scale_rows(x, 1.1)).astype(np.float64)
    exact = bf16_vals(x).astype(np.float64) * np.float64(np.float32(1.1))
    assert np.all(np.abs(y - exact) <= np.abs(exact) * 2.0 ** -8)


def test_dbo_layers_one_layer_reduces_to_the_path(inputs_of):
    """With one layer and alpha = 1 the layer is exactly the MoE path of its
    micro-batches; the shared-expert output is bf16(x sigma)."""
    w = W.WORKLOADS["v2lite"]
    d = inputs_of("v2lite")
    r = O.run_dbo_layers(d["x"], d["logits"][None], d["s"], w.k, w.R, w.C, 1.0, 0.5)
    ref = O.run_dbo(d["x"], d["logits"], d["s"], w.k, w.R, w.C, False)
    assert np.array_equal(r["out"], ref["out"])
    assert np.array_equal(bf16_vals(r["shared"]), 0.5 * bf16_vals(d["x"]))


def test_dbo_layers_closed_form_two_layers():
    """Two layers with unit expert scales: each layer multiplies a token by
    alpha * sum_j w_j (= alpha, no drops) up to rounding: out ~ alpha^2 x."""
    rng = np.random.default_rng(9)
    T, H, E, k = 64, 256, 8, 2
    x = bf16_bits(rng.standard_normal((T, H)))
    lg = rng.standard_normal((2, T, E)).astype(np.float32)
    r = O.run_dbo_layers(x, lg, np.ones(E, np.float32), k, 2, T, 0.5, 1.0)
    xf = bf16_vals(x).astype(np.float64)
    got = bf16_vals(r["out"]).astype(np.float64)
    assert np.all(np.abs(got - 0.25 * xf) <= np.abs(0.25 * xf) * 4 * 2.0 ** -8 + 1e-30)
