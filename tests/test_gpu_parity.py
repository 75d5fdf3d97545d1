"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle
on the same seeded inputs.

Bars: indices, counts, offsets, slots, rank counts, drops and dispatched
buffers (bf16 rows, e4m3 codes, fp32 scales, recv_src) bit-exact; routing
weights within 1e-6 relative; combine output within 1 bf16 ulp of the oracle's
chained result, and bit-exact when the CUDA combine is given the oracle's own
expert output and routing (both accumulate with one fp32 FMA per expert in
selection order).
"""
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from combine_router_top_gb300 import build as B
    B.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_both(w: W.Workload, x=None, logits=None, s=None, max_blocks=0, isolate=True):
    from gpu_path import run_stages
    x = W.make_x(w) if x is None else x
    logits = W.make_logits(w) if logits is None else logits
    s = W.expert_scale(w) if s is None else s
    fp8 = w.dtype == W.DTYPE_FP8_E4M3_B128
    o = O.run_path(x, logits, s, w.k, w.R, w.C, fp8)
    g = run_stages(x, logits, s, w.k, w.R, w.C, fp8, max_blocks=max_blocks, oracle_inputs=o if isolate else None)
    return g, o


@pytest.mark.parametrize("name", ["tiny", "v2lite", "mixtral_skew", "dsv3_fp8"])
def test_workload_parity(name):
    from gpu_path import compare
    w = W.WORKLOADS[name]
    g, o = run_both(w)
    compare(g, o, w.C, w.dtype == W.DTYPE_FP8_E4M3_B128)


GRID_CASES = {
    "fp8_top8": W.WORKLOADS["dsv3_fp8"].with_(T=300),
    # combine units of 4 and 2 chunk groups (top-2, top-4), rows ragged against them
    "bf16_top2": W.WORKLOADS["mixtral_skew"].with_(T=300, H=1800, C=400),
    "bf16_top4": W.WORKLOADS["v2lite"].with_(T=300, k=4, H=2056),
}


@pytest.mark.parametrize("max_blocks", [1, 7, 152, 1000])
@pytest.mark.parametrize("case", list(GRID_CASES))
def test_results_do_not_depend_on_the_grid(case, max_blocks):
    """Capped grids (grid-stride loops, as the overlapped kernels of the
    dual-batch step use) give bit-identical results."""
    from gpu_path import run_stages
    w = GRID_CASES[case]
    fp8 = w.dtype == W.DTYPE_FP8_E4M3_B128
    x, lg, s = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    a = run_stages(x, lg, s, w.k, w.R, w.C, fp8)
    b = run_stages(x, lg, s, w.k, w.R, w.C, fp8, max_blocks=max_blocks)
    for key in a:
        assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), key


EDGE = {
    # ragged token counts: partial 32-token tiles, partial waves
    "T1": W.WORKLOADS["v2lite"].with_(T=1),
    "T77": W.WORKLOADS["v2lite"].with_(T=77),
    "T33_fp8": W.WORKLOADS["dsv3_fp8"].with_(T=33),
    # capacity overflow: pairs dropped and counted
    "overflow_bf16": W.WORKLOADS["v2lite"].with_(C=3),
    "overflow_fp8": W.WORKLOADS["dsv3_fp8"].with_(T=200, C=2),
    "overflow_skew": W.WORKLOADS["mixtral_skew"].with_(T=512, C=100),
    # k extremes
    "k1": W.WORKLOADS["v2lite"].with_(k=1),
    "k_eq_E": W.WORKLOADS["tiny"].with_(k=8),
    # expert counts not a multiple of 32 / of 4, smallest and largest
    "E100": W.Workload("E100", T=130, H=64, E=100, k=5, R=4, C=40, seed=7),
    "E1": W.Workload("E1", T=40, H=16, E=1, k=1, R=1, C=64, seed=8),
    "E6": W.Workload("E6", T=50, H=8, E=6, k=3, R=3, C=50, seed=9),
    "E1024_k16_fp8": W.Workload("E1024", T=100, H=128, E=1024, k=16, R=8, C=16, dtype=1, seed=10),
    "k16_H2048_fp8": W.Workload("k16h2048", T=50, H=2048, E=64, k=16, R=4, C=50, dtype=1, seed=16),
    # hidden extremes
    "H8": W.Workload("H8", T=64, H=8, E=8, k=2, R=2, C=64, seed=11),
    "H65536": W.Workload("H65536", T=3, H=65536, E=4, k=2, R=2, C=4, seed=12),
    "H65536_fp8": W.Workload("H65536f", T=5, H=65536, E=4, k=2, R=2, C=4, dtype=1, seed=19),
    "H128_fp8": W.Workload("H128", T=64, H=128, E=16, k=4, R=4, C=64, dtype=1, seed=13),
    # decode-sized batches count per tile of 8 tokens in bytes: E = 1024 (more
    # experts than threads in the totals block, the most it takes: 256 tokens),
    # E = 500 (not a multiple of 32) and the largest batch (4096 tokens at E 8)
    "T256_E1024_k16_small": W.Workload("t256", T=256, H=64, E=1024, k=16, R=8, C=64, seed=20),
    "T300_E500_small": W.Workload("t300", T=300, H=64, E=500, k=5, R=4, C=100, seed=18),
    "T4096_E8_small_max": W.Workload("t4096", T=4096, H=64, E=8, k=2, R=2, C=4096, seed=25),
    # beyond, tiles of 32 tokens: one token past the byte counts at E 256
    # (33 tiles, direct sum), at E = 1024 (65 tiles: the two-level scan) and
    # E = 500 (102 tiles, a ragged last chunk, two thread groups in the chunk scan)
    "T1025_E256_direct": W.Workload("t1025", T=1025, H=64, E=256, k=8, R=8, C=128, seed=26),
    "T2049_E1024_chunked": W.Workload("t2049", T=2049, H=64, E=1024, k=6, R=8, C=64, seed=17),
    "T3239_E500_chunked": W.Workload("t3239", T=3239, H=64, E=500, k=5, R=4, C=100, seed=19),
    # 129 tiles at E = 256 (two-level, ragged last chunk), the direct sum of
    # earlier tiles (256 tiles at E = 8), and the two-level scan at 8193 and 5000 tokens
    "T4097_E256_chunked": W.Workload("t4097", T=4097, H=64, E=256, k=8, R=8, C=256, seed=21),
    "T8192_E8_direct": W.Workload("t8192", T=8192, H=64, E=8, k=2, R=2, C=4096, seed=22),
    "T8193_E1024_chunked": W.Workload("t8193", T=8193, H=64, E=1024, k=6, R=8, C=64, seed=23),
    "T5000_E500_chunked": W.Workload("t5000", T=5000, H=64, E=500, k=5, R=4, C=100, seed=24),
    # large token counts and capacities: 131072 route tiles; one expert with a million slots
    "T4M": W.Workload("T4M", T=1 << 22, H=8, E=8, k=2, R=2, C=1 << 21, seed=14),
    "E1_C1M": W.Workload("E1_C1M", T=1 << 20, H=8, E=1, k=1, R=1, C=1 << 20, seed=15),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_case_parity(case):
    from gpu_path import compare
    w = EDGE[case]
    g, o = run_both(w)
    compare(g, o, w.C, w.dtype == W.DTYPE_FP8_E4M3_B128)
    if case.startswith("overflow"):
        assert o["dropped"] > 0


FUSED = {
    # fused kernel: H <= 16384, at most 32 tiles of 32 tokens
    "dsv3_fp8": W.WORKLOADS["dsv3_fp8"],
    "T1": W.WORKLOADS["dsv3_fp8"].with_(T=1),
    "T33": W.WORKLOADS["dsv3_fp8"].with_(T=33),
    "T1000": W.WORKLOADS["dsv3_fp8"].with_(T=1000, C=64),
    "overflow": W.WORKLOADS["dsv3_fp8"].with_(T=500, C=3),
    "k16_E1024": W.Workload("k16", T=97, H=1024, E=1024, k=16, R=8, C=8, dtype=1, seed=31),
    "k3_E6": W.Workload("k3", T=45, H=2048, E=6, k=3, R=3, C=20, dtype=1, seed=32),
    "H128_E1024": W.Workload("h128", T=70, H=128, E=1024, k=8, R=8, C=4, dtype=1, seed=34),
    "H16384": W.Workload("h16384", T=40, H=16384, E=32, k=4, R=4, C=16, dtype=1, seed=35),
    "H1152": W.Workload("h1152", T=64, H=1152, E=16, k=4, R=4, C=64, dtype=1, seed=33),
    # bf16 dispatch: the staged row goes out as it is
    "bf16_v2lite": W.WORKLOADS["v2lite"],
    "bf16_T33_overflow": W.WORKLOADS["v2lite"].with_(T=33, C=2),
    "bf16_H8_E1": W.Workload("h8e1", T=40, H=8, E=1, k=1, R=1, C=64, seed=37),
    # separate calls behind the same entry point
    "fallback_T1025": W.WORKLOADS["dsv3_fp8"].with_(T=1025, C=256),
    "fallback_H16512": W.Workload("h16512", T=20, H=16512, E=16, k=2, R=4, C=16, dtype=1, seed=36),
    "fallback_bf16_T2048": W.WORKLOADS["v2lite"].with_(T=2048),
}


@pytest.mark.parametrize("case", sorted(FUSED))
def test_fused_route_dispatch_equals_separate_calls_and_the_oracle(case):
    """moe_route_dispatch writes exactly what moe_route then moe_dispatch
    write, and the whole path built on it matches the oracle."""
    from gpu_path import compare, run_stages
    w = FUSED[case]
    fp8 = w.dtype == W.DTYPE_FP8_E4M3_B128
    x, lg, s = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    a = run_stages(x, lg, s, w.k, w.R, w.C, fp8)
    b = run_stages(x, lg, s, w.k, w.R, w.C, fp8, fused=True)
    for key in a:
        assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), key
    o = O.run_path(x, lg, s, w.k, w.R, w.C, fp8)
    compare(b, o, w.C, fp8)
    if case == "overflow":
        assert o["dropped"] > 0


def test_fused_route_dispatch_empty_batch():
    import torch
    import combine_router_top_gb300 as M
    p = M.problem(0, 7168, 256, 8, 8, 16, M.MOE_DTYPE_FP8_E4M3_B128)
    b = M.alloc_buffers(p, "cuda:0")
    for key in ["counts", "offsets", "rank_counts", "dropped"]:
        b[key].fill_(-7)
    e = torch.empty(0, device="cuda:0")
    M.moe_route_dispatch(p, e, e, e, e, b["counts"], b["offsets"], e, b["rank_counts"], b["dropped"], e,
                         b["recv_scale"], e, b["workspace"])
    torch.cuda.synchronize()
    for key in ["counts", "offsets", "rank_counts", "dropped"]:
        assert int(b[key].abs().sum()) == 0, key


def test_ties_and_signed_zeros():
    from gpu_path import compare
    w = W.Workload("ties", T=256, H=256, E=64, k=6, R=4, C=256, seed=21)
    rng = np.random.default_rng(21)
    vals = np.array([-1.0, -0.0, 0.0, 0.5, 2.0], dtype=np.float32)
    lg = vals[rng.integers(0, len(vals), size=(w.T, w.E))]
    g, o = run_both(w, logits=lg)
    compare(g, o, w.C, False)


def test_all_equal_logits_and_k_eq_E_fp8():
    from gpu_path import compare
    w = W.Workload("flat", T=40, H=256, E=16, k=16, R=2, C=40, dtype=1, seed=22)
    lg = np.zeros((w.T, w.E), dtype=np.float32)
    g, o = run_both(w, logits=lg)
    compare(g, o, w.C, True)
    assert np.array_equal(g["topk_idx"], np.tile(np.arange(16, dtype=np.int32), (w.T, 1)))


def test_fp8_zero_and_tiny_blocks():
    """All-zero blocks (scale 1, codes 0), blocks of subnormal-range values
    and negative zeros."""
    from gpu_path import compare
    import torch
    w = W.Workload("zeros", T=64, H=512, E=8, k=2, R=2, C=64, dtype=1, seed=23)
    x = W.make_x(w)
    x[:, :128] = 0
    x[1::2, 128:256] = 0x8000                                   # -0.0
    tiny = torch.tensor(np.random.default_rng(3).standard_normal((w.T, 128)) * 1e-30, dtype=torch.float32)
    x[:, 256:384] = tiny.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    x[:, 384] = 0x3F80                                           # 1.0 next to tiny values
    g, o = run_both(w, x=x)
    compare(g, o, w.C, True)



def test_fp8_codes_over_every_bf16_value():
    """The quantiser on every bf16 bit pattern, codes and scales bit-exact
    against the oracle. Rows 0-63: all 65536 patterns sorted by magnitude, 128
    to a block, so blocks of NaNs, infinities, subnormals and tiny values (the
    IEEE-division path) sit beside blocks of one binade each (the
    FMA-corrected path). Rows 64-127: blocks whose amax is a random finite
    bf16 and whose other values are random patterns of either sign at or
    below it, so x / sc spans the whole e4m3 range and below."""
    from gpu_path import valid_rows
    w = W.Workload("allbf16", T=128, H=1024, E=8, k=2, R=2, C=128, dtype=1, seed=25)
    pats = np.arange(1 << 16, dtype=np.uint32)
    order = np.lexsort((pats >> 15, pats & 0x7FFF))
    x = np.empty((w.T, w.H), dtype=np.uint16)
    x[:64] = pats[order].astype(np.uint16).reshape(64, w.H)
    rng = np.random.default_rng(25)
    blocks = x[64:].reshape(-1, 128)
    for b in blocks:
        amax = int(rng.integers(1, 0x7F80))
        b[:] = rng.integers(0, amax + 1, size=128) | (rng.integers(0, 2, size=128) << 15)
        b[int(rng.integers(0, 128))] = amax | (int(rng.integers(0, 2)) << 15)
    g, o = run_both(w, x=x)
    assert np.array_equal(g["slot"], o["slot"]) and int(o["dropped"]) == 0
    e, r = valid_rows(o["counts"], w.C)
    assert len(e) == w.T * w.k
    assert np.array_equal(g["recv_src"][e, r], o["recv_src"][e, r])
    assert np.array_equal(g["recv_q"][e, r], o["recv_q"][e, r]), "codes"
    assert np.array_equal(g["recv_scale"][e, r].view(np.uint32), o["recv_scale"][e, r].view(np.uint32)), "scales"
    # the two paths were both taken: infinite / tiny scales and ordinary ones
    sc = o["recv_scale"][e, r]
    assert np.isinf(sc).any() and (sc < 2.0**-100).any() and ((sc > 1e-3) & (sc < 1e3)).any()


def _amax_x_chunks(blocks_per_chunk=1 << 17, H=7168):
    """Every pair (amax, x) of bf16 values with |x| <= amax, for every positive
    finite amax (subnormal ones included) and both signs of x, as 128-element
    blocks: amax first, then 127 of its x values (zero-padded). Yields
    [T, H] arrays of whole rows, blocks_per_chunk blocks at a time."""
    per_row = H // 128
    pending, n = [], 0
    for a in range(1, 0x7F80):
        v = np.arange(a + 1, dtype=np.uint16)
        vals = np.concatenate([v, v | np.uint16(0x8000)])
        vals = np.concatenate([vals, np.zeros(-len(vals) % 127, dtype=np.uint16)]).reshape(-1, 127)
        b = np.empty((len(vals), 128), dtype=np.uint16)
        b[:, 0] = a
        b[:, 1:] = vals
        pending.append(b)
        n += len(b)
        if n >= blocks_per_chunk or a == 0x7F7F:
            blk = np.concatenate(pending)
            blk = np.concatenate([blk, np.zeros((-len(blk) % per_row, 128), dtype=np.uint16)])
            yield blk.reshape(-1, H)
            pending, n = [], 0


def test_fp8_quantiser_on_every_amax_x_pair():
    """moe_dispatch quantises every (amax, x) pair of bf16 values, |x| <= amax,
    x of either sign, amax over every positive finite bf16 (so blocks of
    subnormal and tiny amax take the IEEE-division path and the rest the
    FMA-corrected quotient): codes and scales bit-exact against the oracle's
    dispatch of the same rows."""
    import concurrent.futures as cf
    import torch
    import combine_router_top_gb300 as M
    H = 7168

    def expect(x):
        T = x.shape[0]
        q, sc, _ = O.dispatch_fp8(x, np.zeros((T, 1), np.int32), np.arange(T, dtype=np.int32).reshape(T, 1), 1, T)
        return x, q[0], sc[0]

    pairs = 0
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 2)) as ex:
        for x, q_ref, sc_ref in ex.map(expect, _amax_x_chunks(H=H)):
            T = x.shape[0]
            p = M.problem(T, H, 1, 1, 1, T, M.MOE_DTYPE_FP8_E4M3_B128)
            xd = torch.from_numpy(x.view(np.int16)).to("cuda:0")
            idx = torch.zeros((T, 1), dtype=torch.int32, device="cuda:0")
            sl = torch.arange(T, dtype=torch.int32, device="cuda:0").reshape(T, 1)
            recv = torch.empty((T, H), dtype=torch.uint8, device="cuda:0")
            scale = torch.empty((T, H // 128), dtype=torch.float32, device="cuda:0")
            src = torch.empty((T,), dtype=torch.int32, device="cuda:0")
            M.moe_dispatch(p, xd, idx, sl, recv, scale, src)
            torch.cuda.synchronize()
            assert np.array_equal(recv.cpu().numpy(), q_ref), "codes"
            assert np.array_equal(scale.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32)), "scales"
            pairs += int((x.reshape(-1, 128)[:, 0] != 0).sum()) * 127
    assert pairs > 10**9

def test_nan_logits_give_in_range_distinct_indices():
    """NaN logits: the order is unspecified, but the indices stay valid."""
    from gpu_path import run_stages
    w = W.Workload("nan", T=64, H=64, E=32, k=4, R=2, C=64, seed=24)
    lg = W.make_logits(w)
    lg[::3, ::5] = np.nan
    g = run_stages(W.make_x(w), lg, W.expert_scale(w), w.k, w.R, w.C, False)
    assert np.all((g["topk_idx"] >= 0) & (g["topk_idx"] < w.E))
    assert all(len(set(r)) == w.k for r in g["topk_idx"].tolist())
    assert int(g["counts"].sum()) == w.T * w.k


def test_empty_batch_writes_zero_counts():
    import torch
    import combine_router_top_gb300 as M
    p = M.problem(0, 256, 8, 2, 2, 16)
    b = M.alloc_buffers(p, "cuda:0")
    for key in ["counts", "offsets", "rank_counts", "dropped"]:
        b[key].fill_(-7)
    empty = torch.empty(0, device="cuda:0")
    M.moe_route(p, empty, empty, empty, b["counts"], b["offsets"], empty, b["rank_counts"], b["dropped"], b["workspace"])
    torch.cuda.synchronize()
    for key in ["counts", "offsets", "rank_counts", "dropped"]:
        assert int(b[key].abs().sum()) == 0, key


def test_dbo_step_equals_two_single_shot_runs_and_the_oracle():
    """[DBO §UBatchRunner] midpoint split; each micro-batch runs the whole path
    on its own buffers, dispatch(1) on the comm stream overlapping combine(0)
    on the compute stream. The step's output is bit-identical to two single-
    stream runs of the halves and within 1 ulp of the oracle."""
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev, to_host, ulp_distance
    w = W.WORKLOADS["dbo"]
    x, lg, s = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    T0, T1 = w.T // 2, w.T - w.T // 2
    pf = M.problem(w.T, w.H, w.E, w.k, w.R, w.C)
    bufs = [M.alloc_buffers(M.problem(T1, w.H, w.E, w.k, w.R, w.C), "cuda:0") for _ in range(2)]
    xd, ld, sd = to_dev(x), to_dev(lg), to_dev(s)
    out = torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0")
    comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
    ctx = M.dbo_create()
    comp.wait_stream(torch.cuda.current_stream())
    M.dbo_step(ctx, pf, xd, ld, sd, bufs, out, comp, comm, record_timing=True)
    t = M.dbo_read_timing(ctx)
    torch.cuda.synchronize()
    got = to_host(out, np.uint16)
    assert 0.0 <= t["overlap_fraction"] <= 1.0 and t["step_ms"] > 0
    # two single-shot runs of the halves on one stream
    ref = torch.empty_like(out)
    for (a, b) in [(0, T0), (T0, w.T)]:
        p = M.problem(b - a, w.H, w.E, w.k, w.R, w.C)
        bb = M.alloc_buffers(p, "cuda:0")
        M.run_path(p, xd[a:b], ld[a:b], sd, bb, ref[a:b])
    torch.cuda.synchronize()
    assert np.array_equal(got, to_host(ref, np.uint16))
    # the oracle, micro-batch by micro-batch
    o = O.run_dbo(x, lg, s, w.k, w.R, w.C, False)
    assert ulp_distance(got, o["out"]).max() <= 1
    for u in range(2):
        assert np.array_equal(to_host(bufs[u]["topk_idx"])[: o["parts"][u]["topk_idx"].shape[0]], o["parts"][u]["topk_idx"])
        assert np.array_equal(to_host(bufs[u]["counts"]), o["parts"][u]["counts"])
        assert np.array_equal(to_host(bufs[u]["slot"])[: o["parts"][u]["slot"].shape[0]], o["parts"][u]["slot"])
    ctx.close()


@pytest.mark.parametrize("T", [1, 7, 64])
def test_dbo_small_and_odd_batches(T):
    """Odd T puts the extra token in micro-batch 1; T = 1 leaves micro-batch 0
    empty, which runs as an empty batch."""
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev, to_host, ulp_distance
    w = W.WORKLOADS["tiny"].with_(T=T)
    x, lg, s = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    pf = M.problem(T, w.H, w.E, w.k, w.R, w.C)
    T1 = T - T // 2
    bufs = [M.alloc_buffers(M.problem(T1, w.H, w.E, w.k, w.R, w.C), "cuda:0") for _ in range(2)]
    out = torch.empty((T, w.H), dtype=torch.int16, device="cuda:0")
    comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
    ctx = M.dbo_create()
    comp.wait_stream(torch.cuda.current_stream())
    M.dbo_step(ctx, pf, to_dev(x), to_dev(lg), to_dev(s), bufs, out, comp, comm)
    torch.cuda.synchronize()
    o = O.run_dbo(x, lg, s, w.k, w.R, w.C, False)
    assert ulp_distance(to_host(out, np.uint16), o["out"]).max() <= 1
    if T == 1:
        assert int(to_host(bufs[0]["counts"]).sum()) == 0
    ctx.close()



def test_dbo_step_fp8_dispatch():
    """The dual-batch step with fp8 dispatch (DeepSeek-V3 shape, two micro-batches
    of 256 tokens): output within 1 ulp of the oracle's, each micro-batch's codes
    and scales bit-exact."""
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev, to_host, ulp_distance, valid_rows
    w = W.WORKLOADS["dsv3_fp8"].with_(T=512)
    x, lg, s = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    dt = M.MOE_DTYPE_FP8_E4M3_B128
    pf = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, dt)
    bufs = [M.alloc_buffers(M.problem(w.T // 2, w.H, w.E, w.k, w.R, w.C, dt), "cuda:0") for _ in range(2)]
    out = torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0")
    comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
    ctx = M.dbo_create()
    comp.wait_stream(torch.cuda.current_stream())
    M.dbo_step(ctx, pf, to_dev(x), to_dev(lg), to_dev(s), bufs, out, comp, comm)
    torch.cuda.synchronize()
    o = O.run_dbo(x, lg, s, w.k, w.R, w.C, True)
    assert ulp_distance(to_host(out, np.uint16), o["out"]).max() <= 1
    for u in range(2):
        ref = o["parts"][u]
        e, r = valid_rows(ref["counts"], w.C)
        assert np.array_equal(to_host(bufs[u]["recv"])[e, r], ref["recv_q"][e, r])
        assert np.array_equal(to_host(bufs[u]["recv_scale"])[e, r].view(np.uint32), ref["recv_scale"][e, r].view(np.uint32))
    ctx.close()


def test_repeated_runs_are_bit_identical():
    """The paths whose kernels run concurrently or signal one another, repeated:
    the PDL-chained step (separate and fused route + dispatch, alternately), the
    readiness kernel with a new epoch each time, and the two-stream dual-batch
    step; every run equals the first bit for bit."""
    import torch
    import combine_router_top_gb300 as M
    w = W.WORKLOADS["dsv3_fp8"]
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
    b = M.alloc_buffers(p, "cuda:0")
    x = torch.from_numpy(W.make_x(w).view(np.int16)).to("cuda:0")
    lg = torch.from_numpy(W.make_logits(w)).to("cuda:0")
    s = torch.from_numpy(W.expert_scale(w)).to("cuda:0")
    out = torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0")
    M.run_path(p, x, lg, s, b, out)
    torch.cuda.synchronize()
    ref = out.clone()
    for i in range(200):
        out.zero_()
        M.run_path(p, x, lg, s, b, out, fused=(i % 2 == 1))
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"step, run {i}"
        out.zero_()
        M.moe_expert_combine(p, b["recv"], b["recv_scale"], b["counts"], s, b["y"], b["topk_idx"], b["topk_w"],
                             b["slot"], out, b["ready_flags"], i + 1)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"readiness kernel, run {i}"
    assert M.moe_device_status() == M.MOE_OK
    w = W.WORKLOADS["v2lite"].with_(T=2048)
    pf = M.problem(w.T, w.H, w.E, w.k, w.R, w.C)
    x = torch.from_numpy(W.make_x(w).view(np.int16)).to("cuda:0")
    lg = torch.from_numpy(W.make_logits(w)).to("cuda:0")
    s = torch.from_numpy(W.expert_scale(w)).to("cuda:0")
    bufs = [M.alloc_buffers(M.problem(w.T // 2, w.H, w.E, w.k, w.R, w.C), "cuda:0") for _ in range(2)]
    out = torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0")
    comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
    ctx = M.dbo_create()
    comp.wait_stream(torch.cuda.current_stream())
    M.dbo_step(ctx, pf, x, lg, s, bufs, out, comp, comm)
    torch.cuda.synchronize()
    ref = out.clone()
    for i in range(200):
        out.zero_()
        torch.cuda.synchronize()
        M.dbo_step(ctx, pf, x, lg, s, bufs, out, comp, comm)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"dual-batch step, run {i}"
    ctx.close()


def _layers_setup(w, L, alpha, sigma, busy=0):
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev
    rng = np.random.default_rng(w.seed)
    x = W.make_x(w)
    lg = np.stack([W.make_logits(w.with_(seed=w.seed + 31 * l)) for l in range(L)])
    s = W.expert_scale(w)
    T1 = w.T - w.T // 2
    pf = M.problem(w.T, w.H, w.E, w.k, w.R, w.C)
    bufs = [M.alloc_buffers(M.problem(T1, w.H, w.E, w.k, w.R, w.C), "cuda:0") for _ in range(2)]
    t = {"x": to_dev(x), "lg": to_dev(lg), "s": to_dev(s),
         "h": torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0"),
         "shared": torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0"),
         "out": torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0")}
    args = M.dbo_layers_args(pf, L, t["x"], t["lg"], t["s"], bufs, t["h"], t["shared"], t["out"], alpha, sigma, busy)
    return x, lg, s, t, bufs, args


def _layers_sequential(w, L, alpha, sigma, t):
    """The same kernels, micro-batch after micro-batch and layer after layer, on one stream."""
    import torch
    import combine_router_top_gb300 as M
    out = torch.empty_like(t["out"])
    shared = torch.empty_like(t["out"])
    for (a, b) in [(0, w.T // 2), (w.T // 2, w.T)]:
        if b == a:
            continue
        p = M.problem(b - a, w.H, w.E, w.k, w.R, w.C)
        bb = M.alloc_buffers(p, "cuda:0")
        xu = t["x"][a:b].clone()
        h = torch.empty_like(xu)
        for l in range(L):
            M.moe_layer_stand_in(xu, h, alpha)
            M.run_path(p, h, t["lg"][l, a:b].contiguous(), t["s"], bb, xu)
            M.moe_layer_stand_in(h, shared[a:b], sigma)
        out[a:b] = xu
    torch.cuda.synchronize()
    return out, shared


@pytest.mark.parametrize("name,L,busy", [("tiny", 3, 0), ("v2lite", 2, 64), ("mixtral_skew", 2, 0)])
def test_dbo_layers_match_sequential_and_oracle(name, L, busy):
    """[DBO §Introduction] schedule over L layers on two streams: bit-identical
    to the same kernels run one after another on one stream, and within L+1
    bf16 ulps of the oracle (the routing is identical, each layer's combine is
    within 1 ulp)."""
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_host, ulp_distance
    w = W.WORKLOADS[name]
    alpha, sigma = 0.75, 1.5
    x, lg, s, t, bufs, args = _layers_setup(w, L, alpha, sigma, busy)
    comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
    comp.wait_stream(torch.cuda.current_stream())
    ctx = M.dbo_create()
    M.dbo_layers(ctx, args, comp, comm)
    torch.cuda.synchronize()
    got, got_sh = to_host(t["out"], np.uint16), to_host(t["shared"], np.uint16)
    ref, ref_sh = _layers_sequential(w, L, alpha, sigma, t)
    assert np.array_equal(got, to_host(ref, np.uint16))
    assert np.array_equal(got_sh, to_host(ref_sh, np.uint16))
    o = O.run_dbo_layers(x, lg, s, w.k, w.R, w.C, alpha, sigma)
    assert ulp_distance(got, o["out"]).max() <= L + 1
    assert ulp_distance(got_sh, o["shared"]).max() <= L + 1
    ctx.close()


def test_dbo_layers_graph_replay_equals_eager():
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_host
    w = W.WORKLOADS["v2lite"]
    x, lg, s, t, bufs, args = _layers_setup(w, 3, 0.5, 2.0, 16)
    comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
    comp.wait_stream(torch.cuda.current_stream())
    ctx = M.dbo_create()
    M.dbo_layers(ctx, args, comp, comm)                 # eager first
    torch.cuda.synchronize()
    eager = to_host(t["out"], np.uint16).copy()
    eager_sh = to_host(t["shared"], np.uint16).copy()
    M.dbo_layers_capture(ctx, args, comp, comm)
    for _ in range(2):
        t["out"].fill_(0)
        t["shared"].fill_(0)
        torch.cuda.synchronize()
        M.dbo_graph_launch(ctx, comp)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(t["out"], np.uint16), eager)
        assert np.array_equal(to_host(t["shared"], np.uint16), eager_sh)
    ctx.close()


def test_dbo_layers_full_size_as_benchmarked():
    """The 8192-token dual-batch workload in the configuration the benchmark
    times (4 layers, 256 busy FMAs per 8 elements): two streams eager, graph
    replay and the sequential one-stream run agree bit for bit. (The oracle
    pins the same kernels at this size through the dual-batch step test and
    the layer schedule at smaller sizes.)"""
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_host
    w = W.WORKLOADS["dbo"]
    L, alpha, sigma = 4, 0.75, 1.5
    x, lg, s, t, bufs, args = _layers_setup(w, L, alpha, sigma, 256)
    comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
    comp.wait_stream(torch.cuda.current_stream())
    ctx = M.dbo_create()
    M.dbo_layers(ctx, args, comp, comm)
    torch.cuda.synchronize()
    got, got_sh = to_host(t["out"], np.uint16).copy(), to_host(t["shared"], np.uint16).copy()
    M.dbo_layers_capture(ctx, args, comp, comm)
    t["out"].fill_(0)
    torch.cuda.synchronize()
    M.dbo_graph_launch(ctx, comp)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(t["out"], np.uint16), got)
    ref, ref_sh = _layers_sequential(w, L, alpha, sigma, t)
    assert np.array_equal(got, to_host(ref, np.uint16))
    assert np.array_equal(got_sh, to_host(ref_sh, np.uint16))
    assert np.isfinite(torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float().numpy()).all()
    ctx.close()


def test_dbo_layers_with_gemm_experts():
    """[DBO §Introduction] schedule with the grouped bf16 GEMM as the MLP (random bf16 weights, shared by
    the layers): two streams give bit for bit what one stream gives; the GEMM grid capped to leave SMs to
    the comm stream gives the same bits; and one layer is within the GEMM's bound of the oracle's
    composition (A0 is exact and the routing identical, so out differs only through y):
        |out - out_oracle| <= sum_j w_j ((K/8) 2^-24 S_j + ulp(y_oracle_j)) + 2 ulp(out_oracle),
    S_j = sum_i |x_i w[e_j][n][i]|, the GEMM's bar for row j (see the GEMM tests)."""
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev, to_host
    w = W.Workload("dbo_gemm", T=150, H=512, E=16, k=4, R=4, C=96, seed=808)
    alpha, sigma = 0.75, 1.5
    wb = W.make_weights_bf16(w)
    wd = to_dev(wb)
    results = {}
    for L in [1, 2]:
        x, lg, s, t, bufs, args = _layers_setup(w, L, alpha, sigma, 0)
        comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
        comp.wait_stream(torch.cuda.current_stream())
        ctx = M.dbo_create()
        for mode, (streams, cap) in {"two": ((comp, comm), 0), "one": ((comp, comp), 0),
                                     "two_capped": ((comp, comm), 100)}.items():
            a = M.dbo_layers_args(args.full, L, t["x"], t["lg"], t["s"], bufs, t["h"], t["shared"], t["out"], alpha,
                                  sigma, 0, expert_w=wd, mlp_max_blocks=cap)
            t["out"].fill_(0)
            torch.cuda.synchronize()
            M.dbo_layers(ctx, a, *streams)
            torch.cuda.synchronize()
            results[(L, mode)] = to_host(t["out"], np.uint16).copy()
        ctx.close()
        assert np.array_equal(results[(L, "two")], results[(L, "one")])
        assert np.array_equal(results[(L, "two")], results[(L, "two_capped")])
        if L == 1:
            got = results[(1, "two")]

            def f64(bits):
                return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()

            def ulp(v):
                a = np.abs(v)
                return np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7), 2.0 ** -133)
            absw = np.abs(f64(wb))                                   # [E][H][H]
            bound = np.zeros((w.T, w.H))
            o = O.run_dbo_layers(x, lg, s, w.k, w.R, w.C, alpha, sigma, expert_w=wb)
            for (a0, a1) in [(0, w.T // 2), (w.T // 2, w.T)]:
                h = O.scale_rows(np.ascontiguousarray(x[a0:a1]), alpha)
                r = O.run_path(h, lg[0, a0:a1], s, w.k, w.R, w.C, False, wb)
                assert np.array_equal(r["out"], o["out"][a0:a1])
                habs = np.abs(f64(h))
                for tt in range(a1 - a0):
                    for j in range(w.k):
                        sl = r["slot"][tt, j]
                        if sl < 0:
                            continue
                        e = r["topk_idx"][tt, j]
                        S = absw[e] @ habs[tt]
                        bound[a0 + tt] += r["topk_w"][tt, j] * ((w.H / 8) * 2.0 ** -24 * S + ulp(f64(r["y"][e, sl])))
            oo = f64(o["out"])
            err = np.abs(f64(got) - oo)
            assert np.all(err <= bound + 2 * ulp(oo)), f"max excess {np.max(err - bound - 2 * ulp(oo))}"


@pytest.mark.parametrize("name", ["tiny", "dsv3_fp8"])
def test_path_host_equals_the_device_path(name):
    """moe_path_host (host x and logits in, host out, one call per batch),
    alternated over two streams and buffer sets as a serving loop would:
    every batch's host output equals the device-resident path's output."""
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev
    w = W.WORKLOADS[name]
    x, lg, s = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
    b = M.alloc_buffers(p, "cuda:0")
    sd = to_dev(s)
    ref = torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0")
    M.run_path(p, to_dev(x), to_dev(lg), sd, b, ref)
    torch.cuda.synchronize()
    ref_h = ref.cpu()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    paths, outs = [], []
    for j in range(2):
        xp = torch.from_numpy(x.view(np.int16)).pin_memory()
        lp = torch.from_numpy(lg).pin_memory()
        op = torch.full((w.T, w.H), 7, dtype=torch.int16).pin_memory()
        outs.append(op)
        paths.append(M.HostPath(p, xp, lp, sd, torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0"),
                                torch.empty((w.T, w.E), dtype=torch.float32, device="cuda:0"),
                                M.alloc_buffers(p, "cuda:0"), torch.empty_like(ref), op, streams[j]))
    for i in range(4):
        paths[i % 2]()
    torch.cuda.synchronize()
    for op in outs:
        assert torch.equal(op, ref_h)


def test_layer_stand_in_is_exact():
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev, to_host
    w = W.WORKLOADS["tiny"]
    x = W.make_x(w)
    out = torch.empty((w.T, w.H), dtype=torch.int16, device="cuda:0")
    for a, busy in [(1.1, 0), (0.3, 100)]:
        M.moe_layer_stand_in(to_dev(x), out, a, busy)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(out, np.uint16), O.scale_rows(x, a))


def test_fp32_order_cases_by_hand():
    """The hand-derived cases that fix combine's fp32 accumulation (fused multiply-adds in ascending j
    from +0) and the fp8 stand-in's product order ((q * scale) * s_e): the kernels give the derived
    bits, where any other order would not."""
    import json
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev, to_host
    with open(os.path.join(os.path.dirname(__file__), "golden", "combine_fp32_order.json")) as fh:
        g = json.load(fh)
    H = 8
    for c in g["combine"]:
        k = c["k"]
        p = M.problem(1, H, k, k, 1, 1, M.MOE_DTYPE_BF16)
        y = np.repeat(np.array([int(h, 16) for h in c["y_bf16_bits"]], np.uint16).reshape(k, 1, 1), H, axis=2)
        w = np.array([[int(h, 16) for h in c["w_f32_bits"]]], np.uint32).view(np.float32)
        out = torch.full((1, H), 0x7777, dtype=torch.int16, device="cuda:0")
        M.moe_combine(p, to_dev(y), to_dev(np.arange(k, dtype=np.int32).reshape(1, k)), to_dev(w),
                      to_dev(np.zeros((1, k), np.int32)), out)
        torch.cuda.synchronize()
        assert np.all(to_host(out, np.uint16) == int(c["out_bf16_bits"], 16)), c["name"]
    c = g["expert_fp8"][0]
    Hq = c["H"]
    p = M.problem(1, Hq, 2, 1, 1, 1, M.MOE_DTYPE_FP8_E4M3_B128)
    recv = np.zeros((2, 1, Hq), np.uint8)
    recv[1, 0, :] = int(c["code"], 16)
    scale = np.array([int(c["scale_f32_bits"], 16)], np.uint32).view(np.float32)[0]
    s = np.array([1.0, np.array([int(c["s_e_f32_bits"], 16)], np.uint32).view(np.float32)[0]], np.float32)
    yd = torch.zeros((2, 1, Hq), dtype=torch.int16, device="cuda:0")
    M.moe_expert_synthetic(p, to_dev(recv), to_dev(np.full((2, 1, Hq // 128), scale, np.float32)),
                           to_dev(np.array([0, 1], np.int32)), to_dev(s), yd)
    torch.cuda.synchronize()
    assert np.all(to_host(yd, np.uint16)[1, 0] == int(c["y_bf16_bits"], 16))


@pytest.mark.parametrize("name,T,tps,Cap", [("dsv3_fp8", 1024, 128, 128), ("v2lite", 256, 0, 256),
                                           ("mixtral_skew", 1000, 512, 200), ("dsv3_fp8", 77, 10, 4),
                                           ("dsv3_fp8", 0, 128, 128)])
def test_src_offsets_match_the_oracle(name, T, tps, Cap):
    """moe_src_offsets on the GPU's own route and dispatch output: bit for bit the oracle's offsets,
    which it counts over the pairs (ragged last source rank, drops and an empty batch included)."""
    import torch
    import combine_router_top_gb300 as M
    from gpu_path import to_dev, to_host
    w = W.WORKLOADS[name].with_(T=T, C=Cap) if T > 0 else W.WORKLOADS[name].with_(T=1, C=Cap)
    x, lg = W.make_x(w), W.make_logits(w)
    x, lg = x[:T], lg[:T]
    p = M.problem(T, w.H, w.E, w.k, w.R, Cap, w.dtype, 0, tps)
    b = M.alloc_buffers(p, "cuda:0")
    M.run_path(p, to_dev(np.ascontiguousarray(x)), to_dev(np.ascontiguousarray(lg)),
               to_dev(W.expert_scale(w)), b, torch.empty((max(T, 1), w.H), dtype=torch.int16, device="cuda:0"))
    S = M.src_ranks(p)
    off = torch.full((w.E, S + 1), -5, dtype=torch.int32, device="cuda:0")
    M.moe_src_offsets(p, b["counts"], b["recv_src"], off)
    torch.cuda.synchronize()
    idx, _ = O.route(np.ascontiguousarray(lg), w.k)
    c = O.count(idx, w.E, w.R, Cap)
    assert np.array_equal(to_host(off), O.src_offsets(idx, c["slot"], w.E, tps))


def _random_shapes(n, seed=2468):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        E = int(rng.choice([1, 2, 3, 6, 8, 16, 33, 64, 100, 256, 500, 1024]))
        divisors = [r for r in range(1, E + 1) if E % r == 0]
        R = int(rng.choice(divisors[:8]))
        k = int(rng.integers(1, min(16, E) + 1))
        fp8 = bool(rng.integers(0, 2))
        H = int(rng.choice([128, 256, 1024, 2048, 3072])) if fp8 else int(rng.choice([8, 64, 200, 1024, 2056]))
        T = int(rng.choice([1, 7, 31, 33, 100, 257, 1000, 1025, 2048, 3000]))
        if T * E > 2_000_000 or T * H > 2_000_000:
            continue
        C = int(max(1, rng.integers(1, 2 * max(1, T * k // E) + 8)))
        out.append(W.Workload(f"rnd{len(out)}", T=T, H=H, E=E, k=k, R=R, C=C, dtype=int(fp8),
                              seed=int(rng.integers(0, 1 << 30))))
    return out


@pytest.mark.parametrize("w", _random_shapes(40), ids=lambda w: f"{w.name}-T{w.T}-H{w.H}-E{w.E}-k{w.k}-R{w.R}-C{w.C}-{'fp8' if w.dtype else 'bf16'}")
def test_random_shapes_parity(w):
    """Seeded random shapes (ragged token counts, 1 to 1024 experts, any k, capacities that drop pairs,
    bf16 and fp8): both route paths (byte counts and 32-token tiles), every dispatch kernel, expert and
    combine against the oracle at the usual bars; and the fused route + dispatch equals the separate calls."""
    from gpu_path import compare, run_stages
    g, o = run_both(w)
    compare(g, o, w.C, w.dtype == W.DTYPE_FP8_E4M3_B128)
    x, lg, s = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    f = run_stages(x, lg, s, w.k, w.R, w.C, w.dtype == W.DTYPE_FP8_E4M3_B128, fused=True)
    for key in ["topk_idx", "slot", "counts", "offsets", "rank_counts", "out"]:
        assert np.array_equal(np.asarray(f[key]), np.asarray(g[key])), key
