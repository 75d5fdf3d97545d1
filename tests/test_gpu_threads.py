"""The library outside the usual single-threaded Python caller. Host threads
calling the library at once, from the very first call of a
process: the per-context host caches (device addresses of the library's
arrays, shared-memory attributes, occupancy) are filled under concurrency,
and every thread's results must equal a single-threaded run bit for bit.
Each thread has its own stream and buffers (calls on distinct buffers may
run concurrently). Runs in a fresh child process, so that no earlier test
has filled the caches."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, threading, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import combine_router_top_gb300 as M, workloads as W
torch.cuda.init()
dev = "cuda:0"
w = W.WORKLOADS["dsv3_fp8"].with_(T=256)
x = torch.from_numpy(W.make_x(w).view(np.int16)).to(dev)
lg = torch.from_numpy(W.make_logits(w)).to(dev)
s = torch.from_numpy(W.expert_scale(w)).to(dev)
p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
n = 8
bufs = [M.alloc_buffers(p, dev) for _ in range(n)]
outs = [torch.empty((w.T, w.H), dtype=torch.int16, device=dev) for _ in range(n)]
streams = [torch.cuda.Stream() for _ in range(n)]
torch.cuda.synchronize()
start = threading.Barrier(n)
errors = []
def worker(i):
    try:
        start.wait()
        with torch.cuda.stream(streams[i]):
            M.run_path(p, x, lg, s, bufs[i], outs[i], streams[i])
            M.moe_route_dispatch(p, lg, x, bufs[i]["topk_idx"], bufs[i]["topk_w"], bufs[i]["counts"], bufs[i]["offsets"],
                                 bufs[i]["slot"], bufs[i]["rank_counts"], bufs[i]["dropped"], bufs[i]["recv"],
                                 bufs[i]["recv_scale"], bufs[i]["recv_src"], bufs[i]["workspace"], streams[i])
        streams[i].synchronize()
    except Exception as e:
        errors.append(repr(e))
ts = [threading.Thread(target=worker, args=(i,)) for i in range(n)]
for t in ts: t.start()
for t in ts: t.join()
assert not errors, errors
ref = M.alloc_buffers(p, dev)
out_ref = torch.empty_like(outs[0])
M.run_path(p, x, lg, s, ref, out_ref)
torch.cuda.synchronize()
assert M.moe_device_status() == M.MOE_OK
for i in range(n):
    assert torch.equal(outs[i], out_ref), f"thread {i}: out"
    for key in ["topk_idx", "slot", "counts", "offsets", "recv_src"]:
        assert torch.equal(bufs[i][key], ref[key]), f"thread {i}: {key}"
    for e, c in enumerate(ref["counts"].cpu().tolist()):
        kk = min(c, w.C)
        assert torch.equal(bufs[i]["recv"][e, :kk], ref["recv"][e, :kk]), f"thread {i}: recv rows of expert {e}"
print("threads ok")
'''


def test_concurrent_first_calls_from_host_threads():
    from combine_router_top_gb300 import build as B
    B.build()
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout


def test_c_abi_from_plain_c():
    """The C ABI from a plain C program (tests/c_abi_check.c): cudaMalloc'd buffers, route -> dispatch ->
    synthetic expert -> combine for a bf16 and an fp8 batch, and the allocation-free route, each result
    checked against the C oracle linked into the same program. No Python or PyTorch in that process."""
    import shutil
    import tempfile
    from combine_router_top_gb300 import build as B
    lib = B.build()
    cuda = os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"))
    libdir = os.path.dirname(lib)
    exe = os.path.join(tempfile.mkdtemp(), "c_abi_check")
    subprocess.run(["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c_abi_check.c"),
                    os.path.join(ROOT, "oracle", "moe_oracle.c"), "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), "-L", libdir, "-lmoe_gb300",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm", "-Wl,-rpath," + libdir,
                    "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "c abi ok" in r.stdout
