"""moe_route_noalloc: the route entry point for callers that cannot allocate
device memory (code inside a CUDA-graph capture, runtimes that forbid
allocation after start-up, plugin interfaces that pass only inputs and
outputs). It keeps its scratch in a static device array of the library, so
the test checks that it gives exactly what moe_route gives with a caller
workspace, on two calls in a row (the second reuses the array as the first
left it), and that a problem needing more scratch than the array holds is
refused before anything is launched.

This file is collected last on purpose: if it fails, a run stopped at the
first failure has already run every other test."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def route_outputs(M, p, logits, use_noalloc):
    import torch
    b = M.alloc_buffers(p, DEV)
    for key in ["topk_idx", "topk_w", "counts", "offsets", "slot", "rank_counts", "dropped"]:
        b[key].fill_(-3)
    if use_noalloc:
        M.moe_route_noalloc(p, logits, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"],
                            b["rank_counts"], b["dropped"])
    else:
        M.moe_route(p, logits, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"],
                    b["rank_counts"], b["dropped"], b["workspace"])
    torch.cuda.synchronize()
    return {k: b[k].cpu().numpy() for k in ["topk_idx", "topk_w", "counts", "offsets", "slot", "rank_counts",
                                           "dropped"]}


@pytest.mark.parametrize("name", ["dsv3_fp8", "v2lite", "mixtral_skew"])
def test_noalloc_route_matches_route_on_two_calls_in_a_row(name):
    import torch
    from combine_router_top_gb300 import build as B
    B.build()
    import combine_router_top_gb300 as M
    w = W.WORKLOADS[name]
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
    logits = torch.from_numpy(W.make_logits(w)).to(DEV)
    ref = route_outputs(M, p, logits, use_noalloc=False)
    # a second, different problem in between, so that the second no-alloc call
    # starts from scratch contents another call left behind
    w2 = w.with_(T=max(1, w.T // 3), seed=w.seed + 77)
    p2 = M.problem(w2.T, w2.H, w2.E, w2.k, w2.R, w2.C, w2.dtype)
    logits2 = torch.from_numpy(W.make_logits(w2)).to(DEV)
    for _ in range(2):
        got = route_outputs(M, p, logits, use_noalloc=True)
        for key in ["topk_idx", "counts", "offsets", "slot", "rank_counts", "dropped"]:
            assert np.array_equal(got[key], ref[key]), key
        rel = np.abs(got["topk_w"].astype(np.float64) - ref["topk_w"]) / np.abs(ref["topk_w"].astype(np.float64))
        assert rel.max() <= 1e-6
        ref2 = route_outputs(M, p2, logits2, use_noalloc=False)
        got2 = route_outputs(M, p2, logits2, use_noalloc=True)
        assert np.array_equal(got2["slot"], ref2["slot"]) and np.array_equal(got2["counts"], ref2["counts"])


def test_noalloc_route_at_the_exact_scratch_limit():
    """30784 tokens at 256 experts fill the array exactly: 962 tiles of 32 tokens take the two-level scan,
    whose chunk sums and bases sit at the end of the 1 MiB. Bit for bit as moe_route, twice in a row."""
    import torch
    from combine_router_top_gb300 import build as B
    B.build()
    import combine_router_top_gb300 as M
    w = W.WORKLOADS["dsv3_fp8"].with_(T=30784, C=2048, seed=4242)
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
    assert M.moe_route_workspace_bytes(p) == (1 << 20)
    logits = torch.from_numpy(W.make_logits(w)).to(DEV)
    ref = route_outputs(M, p, logits, use_noalloc=False)
    for _ in range(2):
        got = route_outputs(M, p, logits, use_noalloc=True)
        for key in ["topk_idx", "counts", "offsets", "slot", "rank_counts", "dropped"]:
            assert np.array_equal(got[key], ref[key]), key
        assert np.array_equal(got["topk_w"].view(np.uint32), ref["topk_w"].view(np.uint32))


def test_noalloc_route_refuses_problems_beyond_its_scratch():
    import torch
    from combine_router_top_gb300 import build as B
    B.build()
    import combine_router_top_gb300 as M
    # 131072 tokens at 256 experts need 4096 tiles x 256 x 4 bytes = 4 MiB > 1 MiB; 30785 tokens (963 tiles)
    # need 1 KiB more than the array, one token past the largest batch that fits
    t = torch.zeros(16, dtype=torch.int32, device=DEV)
    for T in [131072, 30785]:
        p = M.problem(T, 7168, 256, 8, 8, 1024)
        assert M.moe_route_workspace_bytes(p) > (1 << 20)
        with pytest.raises(M.MoeError) as err:
            M.moe_route_noalloc(p, t, t, t, t, t, t, t, t)
        assert err.value.status == M.MOE_ERR_UNSUPPORTED
