"""The multi-rank timing path of bench.py on CPU: two gloo ranks (one process each, as torchrun
starts them) exchange their step times with the max-over-ranks reduction and meet at the
barriers; the reference arm runs on rank 0 only.  Every layer is an independent problem per
rank, so this reduction is the only collective."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    r, w, _ = bench._dist()
    assert (r, w) == (rank, world)
    bench._barrier(w)
    got = bench._max_over_ranks(10.0 + rank, w, torch.device("cpu"))
    bench._barrier(w)
    out.put((rank, got))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 11.0, 1: 11.0}


@pytest.mark.parametrize("rank,expect_line", [(0, True), (1, False)])
def test_reference_arm_prints_on_rank0_only(rank, expect_line):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny", "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if expect_line:
        d = json.loads(lines[-1])
        assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["cpu_baseline"]["kind"] == "oracle"
    else:
        assert not lines
