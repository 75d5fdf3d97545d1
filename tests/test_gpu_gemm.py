"""GPU parity of the grouped fp8 GEMM on the tensor cores against the oracle.

The kernel is fed the oracle's own dispatch output (rows past each expert's
count filled with random codes, NaN codes included, which must not leak into
kept rows), and the seeded weights.

Tolerance, from the arithmetic: the kernel sums each 128-input block on the
tensor cores in fp32 (products of two e4m3 values are exact; the sum rounds),
scales it by fl(a_scale * w_scale) and accumulates blocks with one fp32 FMA
each, then rounds to bf16; the oracle is exact until one final bf16 rounding.
With S = sum_b |a_scale * w_scale| * sum_i |q_i * w_i| the bound is
    |y_gpu - y_oracle| <= 2^-12 * S + 2^-20 * S + 1 bf16 ulp of y_oracle,
granting the block sum 12 correct bits relative to its absolute sum, the
scale product and FMA chain 2^-20, and one ulp for the two bf16 roundings.
A wrong element, block, scale or transposition is off by O(S).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SENTINEL = 0xFFFF


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_top_gb300 import build as B
    B.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def e4m3_abs(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).abs().numpy()


def bf16_f64(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def abs_bound_row(q_row, sa_row, w_e, sw_e):
    """S[n] for one row: sum_b |sa_b * sw[n/128][b]| * sum_{i in b} |q_i| |w[n][i]|."""
    N, K = w_e.shape
    qa, wa = e4m3_abs(q_row), e4m3_abs(w_e)
    S = np.zeros(N)
    for b in range(K // 128):
        blk = wa[:, b * 128:(b + 1) * 128] @ qa[b * 128:(b + 1) * 128]
        S += blk * np.abs(sa_row[b] * np.repeat(sw_e[:, b].astype(np.float64), 128))
    return S


def check_row(y_gpu, y_ref, S):
    g, r = bf16_f64(y_gpu), bf16_f64(y_ref)
    assert np.all(np.isfinite(g)), "non-finite output"
    a = np.abs(r)
    ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7), 2.0 ** -133)
    tol = (2.0 ** -12 + 2.0 ** -20) * S + ulp
    err = np.abs(g - r)
    assert np.all(err <= tol), f"max err/S {np.max(err / np.maximum(S, 1e-300)):.3g}"
    return float(np.max(err / np.maximum(S, 1e-300)))


def oracle_dispatch(w: W.Workload):
    x, lg = W.make_x(w), W.make_logits(w)
    idx, _ = O.route(lg, w.k)
    c = O.count(idx, w.E, w.R, w.C)
    rq, rs, _ = O.dispatch_fp8(x, idx, c["slot"], w.E, w.C)
    return rq, rs, c["counts"]


def run_gemm(w: W.Workload, rq, rs, counts, wq, ws, max_blocks=0):
    import combine_router_top_gb300 as M
    E, C, H = rq.shape
    rng = np.random.default_rng(w.seed)
    rq_dev = rq.copy()
    rs_dev = rs.copy()
    for e in range(E):                        # rows past the count: garbage, NaN codes included
        kept = min(int(counts[e]), C)
        rq_dev[e, kept:] = rng.integers(0, 256, size=(C - kept, H), dtype=np.uint8)
        rs_dev[e, kept:] = np.nan
    p = M.problem(w.T, H, E, w.k, w.R, C, M.MOE_DTYPE_FP8_E4M3_B128, max_blocks)
    y = torch.full((E, C, H), SENTINEL, dtype=torch.int32, device=DEV).to(torch.int16)
    M.moe_expert_gemm_fp8(p, torch.from_numpy(rq_dev).to(DEV), torch.from_numpy(rs_dev).to(DEV),
                          torch.from_numpy(np.ascontiguousarray(counts, dtype=np.int32)).to(DEV),
                          torch.from_numpy(wq).to(DEV), torch.from_numpy(ws).to(DEV), y)
    torch.cuda.synchronize()
    assert M.moe_device_status() == M.MOE_OK
    return y.cpu().numpy().view(np.uint16)


CASES = {
    # one input block; partial last tile (C = 40 < 128)
    "H128": (W.Workload("g128", T=60, H=128, E=3, k=2, R=1, C=40, dtype=1, seed=201), None),
    # as many blocks as pipeline stages
    "H384": (W.Workload("g384", T=100, H=384, E=4, k=2, R=2, C=64, dtype=1, seed=202), None),
    # two row tiles per expert (C = 160), the stage ring wrapping
    "H512_two_row_tiles": (W.Workload("g512", T=150, H=512, E=2, k=2, R=1, C=160, dtype=1, seed=203), None),
    # many blocks
    "H2048": (W.Workload("g2048", T=24, H=2048, E=2, k=2, R=2, C=32, dtype=1, seed=204), None),
    # overflowing experts (counts > C) and experts forced empty
    "overflow_and_empty": (W.Workload("gov", T=64, H=256, E=8, k=2, R=4, C=8, dtype=1, seed=205), [1, 6]),
}


@pytest.mark.parametrize("max_blocks", [0, 1, 3])
@pytest.mark.parametrize("case", sorted(CASES))
def test_gemm_matches_oracle(case, max_blocks):
    """Small grids (one CTA, three CTAs) walk many tiles per CTA, so the two
    TMEM accumulators alternate across blocks and tiles within one CTA."""
    w, empty = CASES[case]
    rq, rs, counts = oracle_dispatch(w)
    counts = counts.copy()
    if empty:
        counts[empty] = 0
    wq, ws = W.make_weights(w)
    y_ref = O.expert_gemm_fp8(rq, rs, counts, wq, ws)
    y = run_gemm(w, rq, rs, counts, wq, ws, max_blocks)
    worst = 0.0
    for e in range(w.E):
        kept = min(int(counts[e]), w.C)
        assert np.all(y[e, kept:] == SENTINEL), f"expert {e}: rows past the count were written"
        for r in range(kept):
            worst = max(worst, check_row(y[e, r], y_ref[e, r], abs_bound_row(rq[e, r], rs[e, r], wq[e], ws[e])))
    print(f"{case} max_blocks={max_blocks}: max |err| / S = {worst:.3g}")


@pytest.mark.parametrize("name", ["dsv3_decode", "dsv3_prefill"])
def test_gemm_full_size_sampled_rows(name):
    """The two shapes the benchmark times: DeepSeek-V3 decode (1024 tokens, H
    7168, 256 experts, C 128) and an 8192-token prefill (C 1024: several row
    tiles per expert). The whole chain route -> dispatch -> GEMM on the GPU,
    13 GB of device-drawn weights; sampled rows against the oracle's row entry
    fed by the oracle's own dispatch; every row past a count untouched."""
    import combine_router_top_gb300 as M
    w = W.WORKLOADS["dsv3_fp8"] if name == "dsv3_decode" else W.WORKLOADS["dbo"].with_(dtype=W.DTYPE_FP8_E4M3_B128)
    rq, rs, counts = oracle_dispatch(w)
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
    b = M.alloc_buffers(p, DEV)
    x = torch.from_numpy(W.make_x(w).view(np.int16)).to(DEV)
    lg = torch.from_numpy(W.make_logits(w)).to(DEV)
    M.moe_route(p, lg, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"], b["rank_counts"],
                b["dropped"], b["workspace"])
    M.moe_dispatch(p, x, b["topk_idx"], b["slot"], b["recv"], b["recv_scale"], b["recv_src"])
    wq, ws = W.make_weights_device(w, DEV)
    y = torch.full((w.E, w.C, w.H), SENTINEL, dtype=torch.int32, device=DEV).to(torch.int16)
    M.moe_expert_gemm_fp8(p, b["recv"], b["recv_scale"], b["counts"], wq, ws, y)
    torch.cuda.synchronize()
    assert M.moe_device_status() == M.MOE_OK
    assert np.array_equal(b["counts"].cpu().numpy(), counts)
    yh = y.cpu().numpy().view(np.uint16)
    kept = np.minimum(counts, w.C)
    for e in range(w.E):
        assert np.all(yh[e, kept[e]:] == SENTINEL)
    live = [e for e in range(w.E) if kept[e] > 0]
    picks = [(live[0], 0), (live[0], kept[live[0]] - 1), (live[len(live) // 2], 1 % kept[live[len(live) // 2]]),
             (live[-1], kept[live[-1]] - 1), (live[-1], 0), (live[len(live) // 3], kept[live[len(live) // 3]] // 2)]
    if name == "dsv3_prefill":                     # rows in the second and last row tiles
        e = int(np.argmax(kept))
        picks = [(e, 128), (e, kept[e] - 1), (live[1], min(200, kept[live[1]] - 1))] + picks[:3]
    worst = 0.0
    for e, r in picks:
        wq_e, ws_e = wq[e].cpu().numpy(), ws[e].cpu().numpy()
        ref = O.gemm_fp8_row(rq[e, r], rs[e, r], wq_e, ws_e)
        worst = max(worst, check_row(yh[e, r], ref, abs_bound_row(rq[e, r], rs[e, r], wq_e, ws_e)))
    print(f"{name} sampled rows: max |err| / S = {worst:.3g}")


# ---- bf16 rows, bf16 weights (tcgen05 kind::f16) --------------------------------
#
# Tolerance: bf16 x bf16 products are exact in fp32 and the tensor cores sum
# them in fp32; the worst case of a sequential fp32 sum of K <= 8192 terms is
# K * 2^-24 * S <= 2^-11 * S with S = sum_i |x_i * w_i|. Bar:
#     |y_gpu - y_oracle| <= 2^-11 * S + 1 bf16 ulp of y_oracle.

def bf16_abs(bits):
    return np.abs(bf16_f64(bits))


def check_row_bf16(y_gpu, y_ref, x_row, w_e):
    S = bf16_abs(w_e) @ bf16_abs(x_row)
    g, r = bf16_f64(y_gpu), bf16_f64(y_ref)
    assert np.all(np.isfinite(g)), "non-finite output"
    a = np.abs(r)
    ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7), 2.0 ** -133)
    err = np.abs(g - r)
    assert np.all(err <= 2.0 ** -11 * S + ulp), f"max err/S {np.max(err / np.maximum(S, 1e-300)):.3g}"
    return float(np.max(err / np.maximum(S, 1e-300)))


def oracle_dispatch_bf16(w: W.Workload):
    x, lg = W.make_x(w), W.make_logits(w)
    idx, _ = O.route(lg, w.k)
    c = O.count(idx, w.E, w.R, w.C)
    rx, _ = O.dispatch_bf16(x, idx, c["slot"], w.E, w.C)
    return rx, c["counts"]


CASES_BF16 = {
    # one block of 64 inputs; 64 valid outputs of a 256-output tile
    "H64": (W.Workload("b64", T=40, H=64, E=3, k=2, R=1, C=32, seed=301), None),
    # 192 of 256 outputs valid in the only output tile; 3 blocks
    "H192": (W.Workload("b192", T=60, H=192, E=4, k=2, R=2, C=40, seed=302), None),
    # two row tiles per expert, the stage ring wrapping
    "H512_two_row_tiles": (W.Workload("b512", T=150, H=512, E=2, k=2, R=1, C=160, seed=303), None),
    "H2048": (W.Workload("b2048", T=24, H=2048, E=2, k=2, R=2, C=32, seed=304), None),
    "overflow_and_empty": (W.Workload("bov", T=64, H=256, E=8, k=2, R=4, C=8, seed=305), [2, 5]),
    # 600 rows per expert on average: the host picks 256-row tiles (two TMEM
    # halves per tile, 256 + 256 + a one-half remainder of 88 rows)
    "H256_wide_600": (W.Workload("b600", T=600, H=256, E=2, k=2, R=1, C=640, seed=307), None),
    # about 300 rows per expert: three 128-row tiles, the last one ragged
    "H256_three_row_blocks": (W.Workload("b300", T=300, H=256, E=2, k=2, R=1, C=320, seed=306), None),
}


@pytest.mark.parametrize("max_blocks", [0, 1, 3])
@pytest.mark.parametrize("case", sorted(CASES_BF16))
def test_gemm_bf16_matches_oracle(case, max_blocks):
    """Small grids (one CTA, three CTAs) walk many tiles per CTA, so the two
    TMEM accumulators alternate and are reused across tiles within one CTA."""
    import combine_router_top_gb300 as M
    w, empty = CASES_BF16[case]
    rx, counts = oracle_dispatch_bf16(w)
    counts = counts.copy()
    if empty:
        counts[empty] = 0
    wb = W.make_weights_bf16(w)
    y_ref = O.expert_gemm_bf16(rx, counts, wb)
    rng = np.random.default_rng(w.seed)
    rx_dev = rx.copy()
    for e in range(w.E):                      # rows past the count: garbage bits, NaNs included
        kept = min(int(counts[e]), w.C)
        rx_dev[e, kept:] = rng.integers(0, 1 << 16, size=(w.C - kept, w.H), dtype=np.uint16)
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, M.MOE_DTYPE_BF16, max_blocks)
    y = torch.full((w.E, w.C, w.H), SENTINEL, dtype=torch.int32, device=DEV).to(torch.int16)
    M.moe_expert_gemm_bf16(p, torch.from_numpy(rx_dev.view(np.int16)).to(DEV),
                           torch.from_numpy(np.ascontiguousarray(counts, dtype=np.int32)).to(DEV),
                           torch.from_numpy(wb.view(np.int16)).to(DEV), y)
    torch.cuda.synchronize()
    assert M.moe_device_status() == M.MOE_OK
    yh = y.cpu().numpy().view(np.uint16)
    worst = 0.0
    for e in range(w.E):
        kept = min(int(counts[e]), w.C)
        assert np.all(yh[e, kept:] == SENTINEL), f"expert {e}: rows past the count were written"
        for r in range(kept):
            worst = max(worst, check_row_bf16(yh[e, r], y_ref[e, r], rx[e, r], wb[e]))
    print(f"bf16 {case} max_blocks={max_blocks}: max |err| / S = {worst:.3g}")


@pytest.mark.parametrize("name", ["v2lite", "dbo_prefill", "prefill_32_wide"])
def test_gemm_bf16_full_size_sampled_rows(name):
    """DeepSeek-V2-Lite decode (256 tokens, H 2048, 64 experts), the 8192-token
    dual-batch prefill shape (H 7168, 256 experts, C 1024; 26 GB of device-drawn
    weights) and the same prefill over 32 experts (1024 kept rows each: the
    256-row tiles): route -> dispatch -> GEMM on the GPU, sampled rows against
    the oracle fed by its own dispatch."""
    import combine_router_top_gb300 as M
    w = {"v2lite": W.WORKLOADS["v2lite"], "dbo_prefill": W.WORKLOADS["dbo"],
         "prefill_32_wide": W.WORKLOADS["dbo"].with_(E=32)}[name]
    rx, counts = oracle_dispatch_bf16(w)
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, M.MOE_DTYPE_BF16)
    b = M.alloc_buffers(p, DEV)
    x = torch.from_numpy(W.make_x(w).view(np.int16)).to(DEV)
    lg = torch.from_numpy(W.make_logits(w)).to(DEV)
    M.moe_route(p, lg, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"], b["rank_counts"],
                b["dropped"], b["workspace"])
    M.moe_dispatch(p, x, b["topk_idx"], b["slot"], b["recv"], None, b["recv_src"])
    wb = W.make_weights_bf16_device(w, DEV)
    y = torch.full((w.E, w.C, w.H), SENTINEL, dtype=torch.int32, device=DEV).to(torch.int16)
    M.moe_expert_gemm_bf16(p, b["recv"], b["counts"], wb, y)
    torch.cuda.synchronize()
    assert M.moe_device_status() == M.MOE_OK
    assert np.array_equal(b["counts"].cpu().numpy(), counts)
    kept = np.minimum(counts, w.C)
    live = [e for e in range(w.E) if kept[e] > 0]
    emax = int(np.argmax(kept))
    picks = [(live[0], 0), (live[-1], kept[live[-1]] - 1), (emax, kept[emax] - 1), (emax, min(130, kept[emax] - 1)),
             (emax, min(255, kept[emax] - 1)), (emax, min(256, kept[emax] - 1)), (emax, min(383, kept[emax] - 1))]
    worst = 0.0
    for e, r in picks:
        yr = y[e, r].cpu().numpy().view(np.uint16)
        assert np.all(y[e, kept[e]:].cpu().numpy().view(np.uint16) == SENTINEL)
        w_e = wb[e].cpu().numpy().view(np.uint16)
        ref = O.gemm_bf16_row(rx[e, r], w_e)
        worst = max(worst, check_row_bf16(yr, ref, rx[e, r], w_e))
    print(f"bf16 {name} sampled rows: max |err| / S = {worst:.3g}")
