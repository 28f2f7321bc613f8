"""The benchmark's multi-process host logic on CPU (gloo, world size 2).

The path runs as independent replicas (no data-path collective): ranks only
meet at a barrier and take the maximum of their timings.  The reference arm
runs on rank 0 alone; other ranks exit without work."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist("gloo")
    d.barrier()
    m = d.max(1.5 * (rank + 1))
    q.put((rank, d.world, m))
    d.close()


def test_replicas_barrier_and_max_over_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r for r, _, _ in res] == [0, 1]
    assert all(w == 2 and m == 3.0 for _, w, m in res)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank0_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--config", "tiny", "--ref-tokens", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank != 0:
        assert lines == []
    else:
        out = json.loads(lines[-1])
        assert out["impl"] == "reference" and out["unit"] == "TFLOP/s" and out["value"] > 0
        assert out["cpu_baseline"]["kind"] == "oracle"
        assert out["e2e"]["h2d_bytes_per_step"] == 0
