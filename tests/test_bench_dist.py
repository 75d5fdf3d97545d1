"""Multi-rank plumbing of bench.py, on CPU with the gloo backend and two
ranks: the max-over-ranks timing and the barrier that bracket the replicas'
timed region (N GPUs run N independent replicas of the step)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        bench.barrier(world)
        mx = bench.reduce_max(1.5 + rank, world)
        # the slowest rank's dispatch+combine time sets the whole-job rate
        dc_ms = bench.reduce_max(0.040 if rank == 0 else 0.050, world)
        q.put((rank, mx, world * 1024 / (dc_ms * 1e-3)))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [2.5, 2.5]
    assert all(abs(g[2] - 2 * 1024 / 50e-6) < 1e-3 for g in got)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)


def test_traffic_records_follow_code_not_comments(tmp_path, monkeypatch):
    """A recorded ncu traffic figure stays valid through comment edits and
    lapses when the kernel's code changes."""
    import bench
    csrc = tmp_path / "combine_router_top_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "k.cu").write_text("// kernel\n__global__ void k(int *p) { p[0] = 1; }\n")
    a = bench.kernel_source_sha(["k.cu"])
    (csrc / "k.cu").write_text("/* the\n kernel */\n__global__ void k(int *p)\n{\n    p[0] = 1;   // store\n}\n")
    assert bench.kernel_source_sha(["k.cu"]) == a
    (csrc / "k.cu").write_text("__global__ void k(int *p) { p[0] = 2; }\n")
    assert bench.kernel_source_sha(["k.cu"]) != a


@pytest.mark.parametrize("name,T,threads", [("dsv3_fp8", 200, 7), ("v2lite", 256, 5), ("tiny", 64, 64)])
def test_threaded_oracle_baseline_equals_the_oracle_path(name, T, threads):
    """The CPU baseline's threaded harness (the oracle's functions over disjoint token and expert
    ranges) computes exactly what the single-threaded oracle path computes."""
    import numpy as np
    import bench
    import oracle as O
    import workloads as W
    w = W.WORKLOADS[name]
    x, lg, s = W.make_x(w, 0, T), W.make_logits(w, 0, T), W.expert_scale(w)
    fp8 = w.dtype == W.DTYPE_FP8_E4M3_B128
    ref = O.run_path(x, lg, s, w.k, w.R, w.C, fp8)
    to = bench.ThreadedOracle(O, x, lg, s, w, threads)
    try:
        for _ in range(2):
            to.step()
            assert np.array_equal(to.idx, ref["topk_idx"]) and np.array_equal(to.wt, ref["topk_w"])
            for key in ["counts", "offsets", "slot", "rank_counts"]:
                assert np.array_equal(getattr(to, key), ref[key]), key
            assert int(to.dropped[0]) == ref["dropped"]
            assert np.array_equal(to.out, ref["out"])
            for e, c in enumerate(ref["counts"].tolist()):
                n = min(c, w.C)
                assert np.array_equal(to.recv_src[e, :n], ref["recv_src"][e, :n])
                assert np.array_equal(to.y[e, :n], ref["y"][e, :n])
                assert np.array_equal(to.recv[e, :n], ref["recv_q" if fp8 else "recv_x"][e, :n])
            to.recv_src.fill(-1)
    finally:
        to.close()
