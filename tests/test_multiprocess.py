"""The bench's multi-process path on CPU, world size 2 over gloo (127.0.0.1):
the rendezvous, the barrier and the max-over-ranks timing that every N > 1
bench line is built on, and the reference arm launched by torchrun exactly as
for N GPUs (rank 0 alone prints one JSON line; the other rank exits 0 without
work).  No GPU is involved."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    w, r, _, pg = bench.dist_setup()
    bench.barrier(pg)
    slowest = bench.max_over_ranks(pg, 10.0 * (rank + 1))   # rank 1 is "slower"
    bench.barrier(pg)
    q.put((r, w, slowest))
    pg.destroy_process_group()


def test_gloo_rendezvous_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in procs)
    assert [r for r, _, _ in res] == [0, 1]
    assert all(w == 2 for _, w, _ in res)
    assert all(m == 20.0 for _, _, m in res), "every rank must see the slowest rank's time"


def test_single_process_helpers_are_identity():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5) == 3.5
    bench.barrier(None)


def test_reference_arm_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "dense_tiny", "--steps", "1", "--warmup", "0", "--gpus",
           "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
