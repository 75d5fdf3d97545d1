"""The C-ABI library loads, exports every entry point include/moe.h declares,
and validates arguments on the host (no GPU needed: every call here returns
before anything is launched)."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from combine_router_top_gb300 import build as B
    B.build()
    import combine_router_top_gb300 as M
    return M


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*([a-z_][a-z_0-9]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path(moe):
    names = declared_functions()
    for n in ["moe_route", "moe_dispatch", "moe_combine", "moe_expert_synthetic", "dbo_step", "dbo_create",
              "dbo_destroy", "dbo_read_timing", "moe_status_string", "moe_validate", "moe_route_workspace_bytes"]:
        assert n in names


def test_library_exports_every_declared_symbol(moe):
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (\S+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(moe.lib(), n)
    assert set(moe.EXPORTS) == set(declared_functions())


def test_library_does_not_export_cuda_runtime(moe):
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True, check=True).stdout
    assert not re.search(r" T cuda", out)


def test_status_strings(moe):
    for s in [0, -1, -2, -3, -4, -5]:
        assert moe.moe_status_string(s).startswith("MOE_")
    assert moe.moe_status_string(12345) == "unknown moe_status"


GOOD = dict(T=1024, H=7168, E=256, k=8, R=8, Cap=128, dtype=1)


def mk(moe, **kw):
    a = dict(GOOD)
    a.update(kw)
    return moe.problem(a["T"], a["H"], a["E"], a["k"], a["R"], a["Cap"], a["dtype"], a.get("mb", 0))


@pytest.mark.parametrize("bad", [
    dict(k=0), dict(k=17), dict(E=4, k=5, R=4), dict(E=1025, R=1), dict(E=0), dict(R=0), dict(R=3),
    dict(Cap=0), dict(T=-1), dict(H=12, dtype=0), dict(H=0), dict(H=7168 + 8), dict(dtype=2),
    dict(H=65536 + 8, dtype=0), dict(mb=-1), dict(T=(1 << 24) + 1),
])
def test_validate_rejects(moe, bad):
    assert moe.moe_validate(mk(moe, **bad)) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_route_workspace_bytes(mk(moe, **bad)) == 0


def test_validate_accepts_workloads(moe):
    import workloads as W
    for w in W.WORKLOADS.values():
        p = moe.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
        assert moe.moe_validate(p) == moe.MOE_OK
    assert moe.moe_validate(mk(moe, T=0)) == moe.MOE_OK
    assert moe.moe_validate(mk(moe, H=8, dtype=0, E=1, k=1, R=1)) == moe.MOE_OK


def test_route_workspace_bytes(moe):
    # decode-sized batches (T <= 4096 and E * ceil(tiles8 / 16) <= 2048): one byte per
    # (expert, tile of 8 tokens), each expert's row rounded up to 16 bytes
    assert moe.moe_route_workspace_bytes(mk(moe)) == 256 * 128                  # 1024 tokens, E 256
    assert moe.moe_route_workspace_bytes(mk(moe, T=4096, E=64, R=8)) == 64 * 512
    assert moe.moe_route_workspace_bytes(mk(moe, T=4096, E=8, k=2, R=8)) == 8 * 512
    assert moe.moe_route_workspace_bytes(mk(moe, T=9, E=3, k=1, R=1)) == 256
    assert moe.moe_route_workspace_bytes(mk(moe, T=256, E=1024, k=8, R=8)) == 1024 * 32
    # beyond: int32 counts per (tile of 32 tokens, expert); while tiles^2 * E <= 2^22
    # the finaliser sums earlier tiles directly, beyond that the two-level scan adds
    # a sum and a base per (chunk of 32 tiles, expert)
    assert moe.moe_route_workspace_bytes(mk(moe, T=1025)) == 33 * 256 * 4        # 1025 tokens, E 256
    assert moe.moe_route_workspace_bytes(mk(moe, T=4096)) == 128 * 256 * 4
    assert moe.moe_route_workspace_bytes(mk(moe, T=4097)) == (129 + 2 * 5) * 256 * 4
    assert moe.moe_route_workspace_bytes(mk(moe, T=4097, E=8, R=8)) == (129 * 8 * 4 + 255) // 256 * 256
    assert moe.moe_route_workspace_bytes(mk(moe, T=3239, E=500, k=5, R=4)) == ((102 + 2 * 4) * 500 * 4 + 255) // 256 * 256
    assert moe.moe_route_workspace_bytes(mk(moe, T=3239, E=100, k=5, R=4)) == (102 * 100 * 4 + 255) // 256 * 256
    assert moe.moe_route_workspace_bytes(mk(moe, T=0)) == 256
    assert moe.moe_route_workspace_bytes(mk(moe, T=33, E=8, R=2)) % 256 == 0


def test_route_dispatch_workspace_bytes(moe):
    p = mk(moe)        # the fused path keeps its ranks in slot[]: the route's own workspace
    assert moe.moe_route_dispatch_workspace_bytes(p) == moe.moe_route_workspace_bytes(p) == 256 * 128
    assert moe.moe_route_dispatch_workspace_bytes(mk(moe, T=0)) == 256
    assert moe.moe_route_dispatch_workspace_bytes(mk(moe, k=0)) == 0
    L = moe.lib()
    fake = C.c_void_p(1 << 40)
    args = [fake] * 12
    assert L.moe_route_dispatch(C.byref(p), *args, fake, 16, None) == moe.MOE_ERR_INVALID_ARG
    odd = C.c_void_p((1 << 40) + 4)
    assert L.moe_route_dispatch(C.byref(p), odd, *args[1:], fake, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG


def test_gemm_rejects_bad_arguments_before_any_launch(moe):
    L = moe.lib()
    p, pb = mk(moe), mk(moe, dtype=0)
    fake = C.c_void_p(1 << 40)
    odd = C.c_void_p((1 << 40) + 8)
    args = [fake] * 6
    assert L.moe_expert_gemm_fp8(C.byref(pb), *args, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_expert_gemm_fp8(None, *args, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_expert_gemm_fp8(C.byref(p), None, *args[1:], None) == moe.MOE_ERR_INVALID_ARG
    for i in (0, 3, 5):                      # recv_q, w_q, y need 16-byte alignment
        a = list(args)
        a[i] = odd
        assert L.moe_expert_gemm_fp8(C.byref(p), *a, None) == moe.MOE_ERR_INVALID_ARG


def test_expert_combine_rejects_bad_arguments_before_any_launch(moe):
    L = moe.lib()
    p = mk(moe)
    assert moe.moe_ready_flags_bytes(p) == 256 * 128 * 4 * 4        # 448 fp8 pieces per row: 4 segments of 128
    assert moe.moe_ready_flags_bytes(mk(moe, dtype=0)) == 256 * 128 * 7 * 4   # 896 bf16 pieces: 7 segments
    assert moe.moe_ready_flags_bytes(mk(moe, k=0)) == 0
    fake = C.c_void_p(1 << 40)
    args = [fake] * 9
    fb = 256 * 128 * 4 * 4
    # epoch 0, flags too small, missing flags
    assert L.moe_expert_combine(C.byref(p), *args, fake, fb, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_expert_combine(C.byref(p), *args, fake, fb - 4, 1, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_expert_combine(C.byref(p), *args, None, fb, 1, None) == moe.MOE_ERR_INVALID_ARG
    # fp8 needs recv_scale
    a = list(args)
    a[1] = None
    assert L.moe_expert_combine(C.byref(p), *a, fake, fb, 1, None) == moe.MOE_ERR_INVALID_ARG
    # misaligned y
    a = list(args)
    a[4] = C.c_void_p((1 << 40) + 8)
    assert L.moe_expert_combine(C.byref(p), *a, fake, fb, 1, None) == moe.MOE_ERR_INVALID_ARG
    # empty batch: nothing to do
    assert L.moe_expert_combine(C.byref(mk(moe, T=0)), *args, fake, fb, 1, None) == moe.MOE_OK


def test_gemm_bf16_and_route_dispatch_argument_checks(moe):
    L = moe.lib()
    fake = C.c_void_p(1 << 40)
    odd = C.c_void_p((1 << 40) + 8)
    pb, pf = mk(moe, dtype=0), mk(moe)
    args = [fake] * 4                                    # recv_x, counts, w, y
    assert L.moe_expert_gemm_bf16(C.byref(pf), *args, None) == moe.MOE_ERR_UNSUPPORTED      # fp8 problem
    assert L.moe_expert_gemm_bf16(C.byref(mk(moe, dtype=0, H=7168 + 8)), *args, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_expert_gemm_bf16(C.byref(pb), None, *args[1:], None) == moe.MOE_ERR_INVALID_ARG
    for i in (0, 2, 3):                                  # recv_x, w, y need 16-byte alignment
        a = list(args)
        a[i] = odd
        assert L.moe_expert_gemm_bf16(C.byref(pb), *a, None) == moe.MOE_ERR_INVALID_ARG
    # moe_route_dispatch: a scale buffer exactly when the dispatch is fp8
    ws = moe.moe_route_dispatch_workspace_bytes(pb)
    a = [fake] * 12
    a[10] = fake                                         # recv_scale given for a bf16 dispatch
    assert L.moe_route_dispatch(C.byref(pb), *a, fake, ws, None) == moe.MOE_ERR_INVALID_ARG
    a[10] = None                                         # and missing for an fp8 one
    assert L.moe_route_dispatch(C.byref(pf), *a, fake, moe.moe_route_dispatch_workspace_bytes(pf), None) == \
        moe.MOE_ERR_INVALID_ARG


def test_calls_reject_bad_arguments_before_any_launch(moe):
    L = moe.lib()
    p = mk(moe)
    fake = C.c_void_p(1 << 40)           # never dereferenced: checks fail first
    # null problem
    assert L.moe_route(None, fake, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    assert L.moe_route(C.byref(p), fake, fake, fake, fake, fake, fake, fake, fake, fake, 16, None) == moe.MOE_ERR_INVALID_ARG
    # misaligned logits
    odd = C.c_void_p((1 << 40) + 4)
    assert L.moe_route(C.byref(p), odd, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    # fp8 dispatch needs recv_scale; bf16 must not have one
    assert L.moe_dispatch(C.byref(p), fake, fake, fake, fake, None, fake, None) == moe.MOE_ERR_INVALID_ARG
    pb = mk(moe, dtype=0)
    assert L.moe_dispatch(C.byref(pb), fake, fake, fake, fake, fake, fake, None) == moe.MOE_ERR_INVALID_ARG
    # misaligned row buffer
    assert L.moe_combine(C.byref(p), odd, fake, fake, fake, fake, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine(C.byref(p), fake, fake, fake, fake, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_expert_synthetic(C.byref(p), fake, None, fake, fake, fake, None) == moe.MOE_ERR_INVALID_ARG
    # dbo: null context, same stream for both roles
    arr = (moe.moe_ubatch_bufs * 2)()
    assert L.dbo_step(None, C.byref(p), fake, fake, fake, arr, fake, None, None, 0) == moe.MOE_ERR_INVALID_ARG
    assert L.dbo_read_timing(None, None) == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("field", ["counts", "offsets", "rank_counts", "dropped", "workspace", "recv", "y",
                                   "recv_scale", "topk_idx", "topk_w", "slot", "recv_src"])
@pytest.mark.parametrize("how", ["null", "odd"])
def test_path_host_checks_every_buffer_before_any_copy(moe, field, how):
    """moe_path_host makes every check its four calls make before it enqueues
    the first copy: one bad buffer fails the whole call with nothing launched."""
    L = moe.lib()
    p = mk(moe)
    fake = 1 << 40
    b = moe.moe_ubatch_bufs()
    for n, _ in moe.moe_ubatch_bufs._fields_:
        setattr(b, n, fake)
    b.workspace_bytes = moe.moe_route_workspace_bytes(p)
    setattr(b, field, None if how == "null" else fake + 2)
    f = C.c_void_p(fake)
    assert L.moe_path_host(C.byref(p), f, f, f, f, f, C.byref(b), f, f, None) == moe.MOE_ERR_INVALID_ARG


def test_path_host_rejects_small_workspace_and_null_host_buffers(moe):
    L = moe.lib()
    p = mk(moe)
    fake = 1 << 40
    b = moe.moe_ubatch_bufs()
    for n, _ in moe.moe_ubatch_bufs._fields_:
        setattr(b, n, fake)
    b.workspace_bytes = moe.moe_route_workspace_bytes(p) - 1
    f = C.c_void_p(fake)
    assert L.moe_path_host(C.byref(p), f, f, f, f, f, C.byref(b), f, f, None) == moe.MOE_ERR_INVALID_ARG
    b.workspace_bytes += 1
    # x_host, logits_host, s, x_dev, logits_dev, bufs, out_dev, out_host: each one null
    for i in range(8):
        args = [f, f, f, f, f, C.byref(b), f, f]
        args[i] = None
        assert L.moe_path_host(C.byref(p), *args, None) == moe.MOE_ERR_INVALID_ARG, i


def test_empty_batch_calls_are_noops_without_gpu(moe):
    """T == 0: dispatch and combine return MOE_OK without launching anything."""
    L = moe.lib()
    p = mk(moe, T=0)
    fake = C.c_void_p(1 << 40)
    assert L.moe_dispatch(C.byref(p), None, None, None, None, fake, None, None) == moe.MOE_OK
    assert L.moe_combine(C.byref(p), None, None, None, None, None, None) == moe.MOE_OK


def test_binding_refuses_cpu_tensors(moe):
    import torch
    p = mk(moe, T=4, H=256, E=8, k=2, R=2, Cap=4, dtype=0)
    t = torch.zeros(16, dtype=torch.int32)
    with pytest.raises(ValueError):
        moe.moe_combine(p, t, t, t, t, t)
