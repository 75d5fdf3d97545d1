"""GPU parity of the grouped fp8 and bf16 GEMMs on the tensor cores against the oracle.

The kernel is fed the oracle's own dispatch output (rows past each expert's
count filled with random codes, NaN codes included, which must not leak into
kept rows), and the seeded weights; at full size the whole chain runs on the
GPU and one row of every expert (decode) or of every 128-row tile (prefill) is
checked.

Tolerance, from the arithmetic. The oracle is exact until one bf16 rounding of
y. The kernels take exact products (e4m3 x e4m3 and bf16 x bf16 are exact in
fp32) and sum them on the tensor cores into an fp32 accumulator, one MMA
instruction per 32 fp8 inputs or 16 bf16 inputs; the order and number of
roundings inside one instruction are not documented, so the bars grant each
instruction step up to r fp32 roundings of a partial sum bounded by the
absolute sum S:
  fp8:  S = sum_b |a_scale * w_scale| * sum_{i in b} |q_i * w_i| over the K/128
        blocks; per block 4 steps of 32 inputs (r = 8), the product
        fl(a_scale * w_scale) and one fp32 FMA per block:
            |y_gpu - y_oracle| <= (4 r + 1 + K/128) * 2^-24 * S + ulp(y_oracle)
        = (33 + K/128) * 2^-24 * S + ulp; at K = 7168 about 2^-17.5 * S.
  bf16: S = sum_i |x_i * w_i|; K/16 steps (r = 2: the step's sum and its add
        into the accumulator):
            |y_gpu - y_oracle| <= (K/8) * 2^-24 * S + ulp(y_oracle)
        at K = 7168 about 2^-14.2 * S.
The ulp covers the two bf16 roundings. Measured on GB300 (the tests print it):
the error beyond that ulp is at most 5.5e-9 * S (fp8, full size) and 3.2e-7 * S
(bf16, K = 7168), far inside both bars. A wrong element, block, scale or
transposition is off by about S / K or more, which both bars catch.
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


def fp8_rel_bar(K):
    return (33 + K // 128) * 2.0 ** -24


def bf16_rel_bar(K):
    return (K / 8) * 2.0 ** -24


def check_row(y_gpu, y_ref, S, K):
    """(max err/S, max (err - ulp)/S) of one fp8 GEMM row of K inputs, asserting the bar."""
    return err_over_bound(y_gpu, y_ref, S, fp8_rel_bar(K))


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
    worst = [0.0, 0.0]
    for e in range(w.E):
        kept = min(int(counts[e]), w.C)
        assert np.all(y[e, kept:] == SENTINEL), f"expert {e}: rows past the count were written"
        for r in range(kept):
            a, x_ = check_row(y[e, r], y_ref[e, r], abs_bound_row(rq[e, r], rs[e, r], wq[e], ws[e]), w.H)
            worst = [max(worst[0], a), max(worst[1], x_)]
    print(f"{case} max_blocks={max_blocks}: max |err| / S = {worst[0]:.3g}, max (|err| - ulp) / S = {worst[1]:.3g}")


def rows_in_every_tile(kept, tile_rows=128):
    """(e, r): one kept row in every 128-row tile of every expert, its place in the tile varying."""
    picks = []
    for e, n in enumerate(kept.tolist()):
        for mt in range((n + tile_rows - 1) // tile_rows):
            in_tile = min(tile_rows, n - mt * tile_rows)
            picks.append((e, mt * tile_rows + (37 * e + 11 * mt) % in_tile))
    return picks


def host_workers():
    import os
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:
        return 4


def check_rows_threaded(picks, y_rows, one_expert):
    """Checks y_rows[i] (GPU output of row picks[i]) against the oracle, expert by expert on a pool of
    host threads (the oracle's C code and numpy release the GIL). one_expert(e, rows, y) returns the
    worst (err/S, excess over the ulp / S) of those rows. Returns the worst of both over all rows."""
    import collections
    import concurrent.futures as cf
    by_e = collections.defaultdict(list)
    for i, (e, r) in enumerate(picks):
        by_e[e].append((r, y_rows[i]))
    worst = [0.0, 0.0]
    with cf.ThreadPoolExecutor(host_workers()) as ex:
        for a, b in ex.map(lambda item: one_expert(item[0], [r for r, _ in item[1]], [y for _, y in item[1]]),
                           sorted(by_e.items())):
            worst = [max(worst[0], a), max(worst[1], b)]
    return worst


def err_over_bound(y_gpu, y_ref, S, rel):
    """(max err/S, max (err - ulp)/S) of one row; asserts err <= rel * S + ulp(y_ref)."""
    g, r = bf16_f64(y_gpu), bf16_f64(y_ref)
    assert np.all(np.isfinite(g)), "non-finite output"
    a = np.abs(r)
    ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7), 2.0 ** -133)
    err = np.abs(g - r)
    Sg = np.maximum(S, 1e-300)
    assert np.all(err <= rel * S + ulp), f"max err/S {np.max(err / Sg):.3g}"
    return float(np.max(err / Sg)), float(np.max(np.maximum(err - ulp, 0.0) / Sg))


def sentinel_rows_untouched(y, kept):
    """Every row at or past an expert's count still holds the sentinel (checked on the device)."""
    E, C, _ = y.shape
    past = torch.arange(C, device=y.device)[None, :] >= torch.from_numpy(kept).to(y.device)[:, None]
    return bool((y[past] == torch.tensor(SENTINEL, dtype=torch.int32).to(torch.int16).to(y.device)).all())


@pytest.mark.parametrize("name", ["dsv3_decode", "dsv3_prefill"])
def test_gemm_full_size_rows_of_every_expert_and_tile(name):
    """The two shapes the benchmark times: DeepSeek-V3 decode (1024 tokens, H
    7168, 256 experts, C 128) and an 8192-token prefill (C 1024: several row
    tiles per expert). The whole chain route -> dispatch -> GEMM on the GPU,
    13 GB of device-drawn weights; one kept row of every expert at decode (all
    256) and one row in every 128-row tile at prefill, each against the
    oracle's row entry fed by the oracle's own dispatch; every row past a count
    untouched."""
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
    kept = np.minimum(counts, w.C)
    assert sentinel_rows_untouched(y, kept)
    picks = rows_in_every_tile(kept)
    assert len(picks) >= 256
    ei = torch.tensor([e for e, _ in picks], device=DEV)
    ri = torch.tensor([r for _, r in picks], device=DEV)
    y_rows = y[ei, ri].cpu().numpy().view(np.uint16)

    def one_expert(e, rows, ys):
        wq_e, ws_e = wq[e].cpu().numpy(), ws[e].cpu().numpy()
        wa = e4m3_abs(wq_e).astype(np.float32)                      # |w| exactly; sums below need no precision
        worst = [0.0, 0.0]
        for r, yg in zip(rows, ys):
            ref = O.gemm_fp8_row(rq[e, r], rs[e, r], wq_e, ws_e)
            qa = e4m3_abs(rq[e, r]).astype(np.float32)
            S = np.zeros(w.H)
            for blk in range(w.H // 128):
                sl = slice(blk * 128, (blk + 1) * 128)
                S += (wa[:, sl] @ qa[sl]).astype(np.float64) * np.abs(rs[e, r, blk] * np.repeat(ws_e[:, blk].astype(np.float64), 128))
            a, x_ = err_over_bound(yg, ref, S, fp8_rel_bar(w.H))
            worst = [max(worst[0], a), max(worst[1], x_)]
        return worst[0], worst[1]

    worst = check_rows_threaded(picks, y_rows, one_expert)
    print(f"{name}: {len(picks)} rows, max |err| / S = {worst[0]:.3g}, max (|err| - ulp) / S = {worst[1]:.3g}")


# ---- bf16 rows, bf16 weights (tcgen05 kind::f16): bar in the module docstring ----

def bf16_abs(bits):
    return np.abs(bf16_f64(bits))


def check_row_bf16(y_gpu, y_ref, x_row, w_e):
    """(max err/S, max (err - ulp)/S) of one bf16 GEMM row, asserting the bar."""
    S = bf16_abs(w_e) @ bf16_abs(x_row)
    return err_over_bound(y_gpu, y_ref, S, bf16_rel_bar(len(x_row)))


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
    worst = [0.0, 0.0]
    for e in range(w.E):
        kept = min(int(counts[e]), w.C)
        assert np.all(yh[e, kept:] == SENTINEL), f"expert {e}: rows past the count were written"
        for r in range(kept):
            a, x_ = check_row_bf16(yh[e, r], y_ref[e, r], rx[e, r], wb[e])
            worst = [max(worst[0], a), max(worst[1], x_)]
    print(f"bf16 {case} max_blocks={max_blocks}: max |err| / S = {worst[0]:.3g}, max (|err| - ulp) / S = {worst[1]:.3g}")


@pytest.mark.parametrize("name", ["v2lite", "dbo_prefill", "prefill_32_wide"])
def test_gemm_bf16_full_size_rows_of_every_tile(name):
    """DeepSeek-V2-Lite decode (256 tokens, H 2048, 64 experts), the 8192-token
    dual-batch prefill shape (H 7168, 256 experts, C 1024; 26 GB of device-drawn
    weights) and the same prefill over 32 experts (1024 kept rows each: the
    256-row tiles): route -> dispatch -> GEMM on the GPU; one row in every
    128-row block of every expert against the oracle fed by its own dispatch;
    every row past a count untouched."""
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
    assert sentinel_rows_untouched(y, kept)
    picks = rows_in_every_tile(kept)
    assert len(picks) >= min(256, int(np.count_nonzero(kept)))
    ei = torch.tensor([e for e, _ in picks], device=DEV)
    ri = torch.tensor([r for _, r in picks], device=DEV)
    y_rows = y[ei, ri].cpu().numpy().view(np.uint16)

    def one_expert(e, rows, ys):
        w_e = wb[e].cpu().numpy().view(np.uint16)
        wa = bf16_abs(w_e).astype(np.float32)
        worst = [0.0, 0.0]
        for r, yg in zip(rows, ys):
            ref = O.gemm_bf16_row(rx[e, r], w_e)
            S = (wa @ bf16_abs(rx[e, r]).astype(np.float32)).astype(np.float64)
            a, x_ = err_over_bound(yg, ref, S, bf16_rel_bar(w.H))
            worst = [max(worst[0], a), max(worst[1], x_)]
        return worst[0], worst[1]

    worst = check_rows_threaded(picks, y_rows, one_expert)
    print(f"bf16 {name}: {len(picks)} rows, max |err| / S = {worst[0]:.3g}, max (|err| - ulp) / S = {worst[1]:.3g}")
