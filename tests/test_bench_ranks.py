"""bench.py's multi-rank plumbing on CPU: two gloo ranks reduce a step time
by max over ranks, the reference arm prints on rank 0 only, and this
one-GPU build's own arm prints its "unavailable" line on rank 0 only and
launches nothing."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.dist_barrier(w)
    q.put((rank, bench.dist_max(1.0 + rank * 2.5, w)))
    dist.destroy_process_group()


def test_two_ranks_take_the_max_step_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert got == [(0, 3.5), (1, 3.5)]


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload, batch, n_keys, cpu_sample, steps, warmup = "tiny", None, None, 8, 1, 0

    bench.run_reference(A, rank=1, world=2)
    assert capsys.readouterr().out == ""
    bench.run_reference(A, rank=0, world=1)
    line = capsys.readouterr().out.strip()
    assert '"impl": "reference"' in line and '"kind": "oracle"' in line


def test_own_arm_with_several_ranks_prints_unavailable_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import json
    import bench

    class A:
        workload, batch, n_keys = "tiny", None, None

    bench.run_ours(A, rank=1, world=2, local=1)
    assert capsys.readouterr().out == ""
    bench.run_ours(A, rank=0, world=2, local=0)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "ours" and line["n_gpus"] == 2 and "unavailable" in line
