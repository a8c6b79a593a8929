"""The N > 1 launch path on the CPU (gloo, world size 2): the bench's
barrier and max-over-ranks timing, and a torchrun launch of the reference arm
in which rank 0 alone prints its JSON line and every rank exits 0.  The GPU
path runs one independent replica per rank (no data-path collective)."""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(world)
    out[rank] = bench.max_over_ranks(float(rank + 1) * 1.5, world)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_with_gloo():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, free_port(), out), nprocs=world, join=True)
        assert dict(out) == {0: 3.0, 1: 3.0}


def test_torchrun_reference_arm_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--config",
           "tiny_fp32"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_oracle_pool_spreads_the_batch_over_workers():
    """The CPU baseline's process pool (spawn context) covers every sequence
    once per pass and reports the workers it used."""
    import bench
    g, passes, el, cores, g1 = bench.parallel_oracle("tiny_fp32", 0.5, cores=2)
    assert cores == 2 and passes >= 1 and el >= 0.5 and g > 0 and g1 > 0
    p = bench.OraclePool("tiny_fp32", cores=3)
    try:
        assert sorted(r for c in p.chunks for r in c) == list(range(p.w.num_seqs))
        assert p.one_pass() > 0
    finally:
        p.close()
