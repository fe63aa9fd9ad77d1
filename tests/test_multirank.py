"""The multi-GPU path on the CPU: two gloo ranks.

Sequences are independent, so the path shards over the batch with no
exchange: every rank verifies a batch of its own (weak scaling), and the only
collectives are the timing barrier and the max over ranks.  Here the ranks
verify with the oracle (no GPU), reduce their times the way bench.py does, and
rank 0 alone reports; the reference arm under torchrun prints one line from
rank 0 while the other rank exits without work."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        inp = bench.rank_inputs("b1_k4_v32000_f32", rank)
        out = oracle.verify_inputs(inp)
        # a stand-in local time per rank; the job time is the slowest rank's
        local = 10.0 * (rank + 1)
        job = bench.max_over_ranks(local, dist, device="cpu")
        gathered = [None] * world
        dist.all_gather_object(gathered, (int(out["accept_len"][0]), inp.uniforms.tolist(),
                                          int(out["status"][0])))
        q.put((rank, job, gathered))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_verify_their_own_batches_and_agree_on_the_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    (r0, job0, g0), (r1, job1, g1) = res
    assert (r0, r1) == (0, 1)
    assert job0 == job1 == 20.0                       # the slower rank's time, on both
    assert g0 == g1                                   # both see both ranks' results
    (al0, u0, st0), (al1, u1, st1) = g0
    assert st0 == st1 == 0 and 1 <= al0 <= 5 and 1 <= al1 <= 5
    assert u0 != u1                                   # each rank verified its own batch


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "b1_k4_v32000_f32", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["gpu_launches"] == 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_weak_scaling_value():
    """value = units all ranks processed / the slowest rank's time."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    a = bench.rank_inputs("b1_k4_v32000_f32", 0)
    b = bench.rank_inputs("b1_k4_v32000_f32", 1)
    assert a.logits.shape == b.logits.shape and not np.array_equal(a.logits, b.logits)
