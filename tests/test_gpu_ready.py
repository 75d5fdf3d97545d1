"""GPU tests of moe_expert_combine: the synthetic expert and combine in one
kernel, with readiness per expert row ("Efficient and portable
mixture-of-experts communication", §Further Improvements: synchronisation
per token instead of per batch).

Bars: y (kept rows) and out bit-identical to moe_expert_synthetic followed by
moe_combine on the same device inputs; y bit-exact against the oracle and out
within 1 bf16 ulp of the oracle's chained result (the same bars as the
separate calls). The timeout test makes consumers wait for rows that no
producer writes (counts forced to zero): the bounded waits run out and the
device status reports it, with the context still usable.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from combine_router_top_gb300 import build as B
    B.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def setup(w: W.Workload):
    import combine_router_top_gb300 as M
    fp8 = w.dtype == W.DTYPE_FP8_E4M3_B128
    x, lg, s = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
    b = M.alloc_buffers(p, DEV)
    xd = torch.from_numpy(x.view(np.int16)).to(DEV)
    ld = torch.from_numpy(lg).to(DEV)
    sd = torch.from_numpy(s).to(DEV)
    M.moe_route(p, ld, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"], b["rank_counts"],
                b["dropped"], b["workspace"])
    M.moe_dispatch(p, xd, b["topk_idx"], b["slot"], b["recv"], b.get("recv_scale"), b["recv_src"])
    out = torch.empty((w.T, w.H), dtype=torch.int16, device=DEV)
    b["y"].zero_()
    M.moe_expert_synthetic(p, b["recv"], b.get("recv_scale"), b["counts"], sd, b["y"])
    M.moe_combine(p, b["y"], b["topk_idx"], b["topk_w"], b["slot"], out)
    torch.cuda.synchronize()
    return dict(p=p, b=b, s=sd, y_sep=b["y"].clone(), out_sep=out.clone(), x=x, lg=lg, s_h=s, fp8=fp8)


def run_fused(w, st, epoch, max_blocks=0):
    import combine_router_top_gb300 as M
    b = st["b"]
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype, max_blocks)
    b["y"].fill_(0x5555)
    out = torch.full((w.T, w.H), 0x5555, dtype=torch.int16, device=DEV)
    M.moe_expert_combine(p, b["recv"], b.get("recv_scale"), b["counts"], st["s"], b["y"], b["topk_idx"],
                         b["topk_w"], b["slot"], out, b["ready_flags"], epoch)
    torch.cuda.synchronize()
    assert M.moe_device_status() == M.MOE_OK
    return b["y"], out


def kept_mask(b, C):
    counts = b["counts"].cpu().numpy()
    E = counts.shape[0]
    m = np.zeros((E, C), dtype=bool)
    for e in range(E):
        m[e, :min(int(counts[e]), C)] = True
    return torch.from_numpy(m).to(DEV)


CASES = {
    "tiny": W.WORKLOADS["tiny"],
    "v2lite": W.WORKLOADS["v2lite"],
    "mixtral_skew": W.WORKLOADS["mixtral_skew"].with_(T=1024),
    "dsv3_fp8": W.WORKLOADS["dsv3_fp8"],
    "k16_E1024_fp8": W.Workload("k16", T=100, H=128, E=1024, k=16, R=8, C=16, dtype=1, seed=41),
    "T1": W.WORKLOADS["v2lite"].with_(T=1),
    "overflow_fp8": W.WORKLOADS["dsv3_fp8"].with_(T=300, C=3),
    "H8": W.Workload("H8", T=64, H=8, E=8, k=2, R=2, C=64, seed=42),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fused_equals_separate_calls_and_oracle(case):
    from gpu_path import ulp_distance
    w = CASES[case]
    st = setup(w)
    y, out = run_fused(w, st, epoch=1)
    m = kept_mask(st["b"], w.C)
    assert torch.equal(y[m], st["y_sep"][m]), "y differs from moe_expert_synthetic"
    assert torch.equal(out, st["out_sep"]), "out differs from moe_combine"
    o = O.run_path(st["x"], st["lg"], st["s_h"], w.k, w.R, w.C, st["fp8"])
    yh = y.cpu().numpy().view(np.uint16)
    mh = m.cpu().numpy()
    assert np.array_equal(yh[mh], o["y"][mh])
    assert ulp_distance(out.cpu().numpy().view(np.uint16), o["out"]).max() <= 1


@pytest.mark.parametrize("max_blocks", [2, 3, 17])
def test_fused_small_grids_and_repeated_epochs(max_blocks):
    """One producer block and one or two consumer blocks still finish (every
    block is resident); flags carried over from earlier epochs are not mistaken
    for ready rows."""
    w = W.WORKLOADS["dsv3_fp8"].with_(T=256)
    st = setup(w)
    m = kept_mask(st["b"], w.C)
    for epoch in (1, 2, 9):
        y, out = run_fused(w, st, epoch, max_blocks=max_blocks)
        assert torch.equal(y[m], st["y_sep"][m])
        assert torch.equal(out, st["out_sep"])


def test_fused_wait_that_runs_out_reports_timeout():
    """counts forced to zero: no producer writes a row, every consumer wait
    runs out (100 ms each, then the warp stops waiting), the status word says
    so, and the next, consistent call succeeds."""
    import combine_router_top_gb300 as M
    w = W.WORKLOADS["tiny"]
    st = setup(w)
    b = st["b"]
    zero = torch.zeros_like(b["counts"])
    out = torch.empty((w.T, w.H), dtype=torch.int16, device=DEV)
    assert M.moe_device_status() == M.MOE_OK
    M.moe_expert_combine(st["p"], b["recv"], b.get("recv_scale"), zero, st["s"], b["y"], b["topk_idx"],
                         b["topk_w"], b["slot"], out, b["ready_flags"], 5)
    torch.cuda.synchronize()
    assert M.moe_device_status() == M.MOE_ERR_TIMEOUT
    assert M.moe_device_status() == M.MOE_OK                  # reading clears it
    y, out = run_fused(w, st, epoch=6)
    assert torch.equal(out, st["out_sep"])
