"""The N > 1 path of bench.py on CPU: two gloo ranks, one replica each.

The forward pass is independent per (batch, head), so ranks run replicas
with no collective on the data path; the only cross-rank operations are the
barrier around the timed region and the max over ranks of the step time.
These run here with the gloo backend (no GPU)."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports its own "step time"; every rank must see the max
    out[rank] = bench.max_over_ranks(1.5 + rank, w)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_step_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched by torchrun with 2 ranks: rank 0
    alone runs the oracle and prints one JSON line; rank 1 exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=280,
                         env=env, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    import json
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert rec["n_gpus"] == 2 and rec["e2e"]["h2d_bytes_per_step"] == 0
