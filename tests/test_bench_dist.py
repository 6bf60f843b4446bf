"""The multi-process path of bench.py on CPU: two gloo ranks, as torchrun would start
them on two GPUs (replicas only: the ranks exchange nothing but the timing barrier and
the max over ranks)."""
import json
import multiprocessing as mp
import os
import socket
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_env(rank: int, world: int, port: int):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "QZ_BENCH_BACKEND": "gloo"})
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)


def _helpers_child(rank, world, port, q):
    _rank_env(rank, world, port)
    import bench
    r, w, lr = bench.dist_setup(world)
    bench.barrier(w)
    m = bench.reduce_max(1.5 * (r + 1), w, device="cpu")
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, lr, m))


def _reference_child(rank, world, port, q):
    _rank_env(rank, world, port)
    import io
    import contextlib
    import bench
    calls = []

    def fake_baseline(budget_s=12.0):           # stands in for the oracle's seconds of work
        calls.append(budget_s)
        return {"value": 0.5, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "stub"}

    bench.cpu_baseline = fake_baseline
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.main(["--impl", "reference", "--gpus", str(world), "--steps", "2", "--warmup", "3"])
    q.put((rank, len(calls), out.getvalue()))


def _run(target, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_two_ranks_barrier_and_max_over_ranks():
    res = _run(_helpers_child)
    assert [r[:3] for r in res] == [(0, 2, 0), (1, 2, 1)]
    assert all(r[3] == 3.0 for r in res)      # both ranks see the slowest rank's time


def test_reference_arm_runs_on_rank_zero_only():
    res = _run(_reference_child)
    (r0, calls0, out0), (r1, calls1, out1) = res
    assert calls1 == 0 and out1.strip() == ""
    assert calls0 == 5                         # 3 warm-up + 2 timed samples
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] == 0.5 and line["e2e"]["h2d_bytes_per_step"] == 0
