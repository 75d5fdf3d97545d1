"""Helpers of the GPU parity tests: run the CUDA path through the C ABI on
seeded host inputs and bring every output back as numpy arrays."""
import numpy as np
import torch

import combine_router_top_gb300 as M

DEV = "cuda:0"


def to_dev(a: np.ndarray):
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def to_host(t, dtype=None):
    a = t.cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def run_stages(x, logits, s, k, R, Cap, fp8, max_blocks=0, oracle_inputs=None, fused=False):
    """The whole path on the GPU, stage by stage. With oracle_inputs (a result
    of oracle.run_path), also runs the expert and combine kernels on the
    oracle's own upstream results, so that each stage can be compared alone.
    fused: route and dispatch through the one call moe_route_dispatch."""
    T, E = logits.shape
    H = x.shape[1]
    p = M.problem(T, H, E, k, R, Cap, M.MOE_DTYPE_FP8_E4M3_B128 if fp8 else M.MOE_DTYPE_BF16, max_blocks)
    b = M.alloc_buffers(p, DEV)
    b["recv"].zero_()
    b["y"].zero_()
    b["recv_src"].fill_(-1)
    if fp8:
        b["recv_scale"].zero_()
    b["workspace"].fill_(0x55)             # the workspace needs no initialisation
    xd, ld, sd = to_dev(x), to_dev(logits), to_dev(s)
    out = torch.empty((T, H), dtype=torch.int16, device=DEV)
    M.run_path(p, xd, ld, sd, b, out, fused=fused)
    torch.cuda.synchronize()
    r = {
        "topk_idx": to_host(b["topk_idx"]), "topk_w": to_host(b["topk_w"]), "counts": to_host(b["counts"]),
        "offsets": to_host(b["offsets"]), "slot": to_host(b["slot"]), "rank_counts": to_host(b["rank_counts"]),
        "dropped": int(to_host(b["dropped"])[0]), "recv_src": to_host(b["recv_src"]),
        "y": to_host(b["y"], np.uint16), "out": to_host(out, np.uint16),
    }
    if fp8:
        r["recv_q"] = to_host(b["recv"])
        r["recv_scale"] = to_host(b["recv_scale"])
    else:
        r["recv_x"] = to_host(b["recv"], np.uint16)
    if oracle_inputs is not None:
        o = oracle_inputs
        # synthetic expert on the oracle's dispatch output
        recv_o = to_dev(o["recv_q"] if fp8 else o["recv_x"])
        rs_o = to_dev(o["recv_scale"]) if fp8 else None
        y2 = torch.zeros((E, Cap, H), dtype=torch.int16, device=DEV)
        M.moe_expert_synthetic(p, recv_o, rs_o, to_dev(o["counts"]), sd, y2)
        # combine on the oracle's expert output and routing
        out2 = torch.empty((T, H), dtype=torch.int16, device=DEV)
        M.moe_combine(p, to_dev(o["y"]), to_dev(o["topk_idx"]), to_dev(o["topk_w"]), to_dev(o["slot"]), out2)
        torch.cuda.synchronize()
        r["y_from_oracle"] = to_host(y2, np.uint16)
        r["out_from_oracle"] = to_host(out2, np.uint16)
    return r


def ulp_distance(a_bits, b_bits):
    """Distance in representable bf16 steps between two arrays of bit patterns."""
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + (b & 0x7FFF))
    return np.abs(ordered(a_bits) - ordered(b_bits))


def valid_rows(counts, Cap):
    """(e, r) of every written row of the expert-major buffers."""
    es, rs = [], []
    for e, c in enumerate(counts.tolist()):
        n = min(c, Cap)
        es.extend([e] * n)
        rs.extend(range(n))
    return np.array(es, dtype=np.int64), np.array(rs, dtype=np.int64)


def compare(g, o, Cap, fp8, combine_ulp=1, w_rtol=1e-6):
    """Asserts the CUDA results g equal the oracle's o within the stated bars."""
    assert np.array_equal(g["topk_idx"], o["topk_idx"]), "topk_idx"
    gw, ow = g["topk_w"].astype(np.float64), o["topk_w"].astype(np.float64)
    rel = np.divide(np.abs(gw - ow), np.abs(ow), out=np.where(gw == ow, 0.0, np.inf), where=ow != 0)
    assert rel.max(initial=0.0) <= w_rtol, f"topk_w rel err {rel.max()}"
    for key in ["counts", "offsets", "slot", "rank_counts"]:
        assert np.array_equal(g[key], o[key]), key
    assert g["dropped"] == o["dropped"]
    e, r = valid_rows(o["counts"], Cap)
    assert np.array_equal(g["recv_src"][e, r], o["recv_src"][e, r]), "recv_src"
    if fp8:
        assert np.array_equal(g["recv_q"][e, r], o["recv_q"][e, r]), "recv_q"
        assert np.array_equal(g["recv_scale"][e, r], o["recv_scale"][e, r]), "recv_scale"
    else:
        assert np.array_equal(g["recv_x"][e, r], o["recv_x"][e, r]), "recv_x"
    # dispatched buffers are bit-exact, so the expert output is too
    assert np.array_equal(g["y"][e, r], o["y"][e, r]), "y"
    d = ulp_distance(g["out"], o["out"])
    assert d.max(initial=0) <= combine_ulp, f"combine max ulp {d.max()}"
    if "out_from_oracle" in g:
        assert np.array_equal(g["y_from_oracle"][e, r], o["y"][e, r]), "expert on oracle input"
        assert np.array_equal(g["out_from_oracle"], o["out"]), "combine on oracle input"
    return int(d.max(initial=0))
