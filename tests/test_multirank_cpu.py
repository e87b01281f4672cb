"""The N > 1 launch path of bench.py on CPU, with two gloo ranks.

Every (batch, head) sequence of the recurrence is independent, so N GPUs run N
independent replicas of the workload and meet only to agree on the timing:
a barrier on both sides of the timed region and the maximum over ranks.
These tests run that host logic with world_size 2 on the gloo backend, and
check that the reference arm prints from rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from state_space_sequence_04_b300 import synth

    ws, r, local = bench.dist_env()
    d = bench.init_dist(ws, local, "gloo")
    assert dist.get_world_size() == world and dist.get_rank() == rank
    # each rank draws its own replica of the workload
    w = synth.Workload("replica", 1, 2, 32, 16, 16, 1, 16, "fp32")
    x = synth.make_inputs(w, seed=r)["x"]
    bench.barrier(d)
    # timing: the slowest rank decides
    t = bench.max_over_ranks(d, 1.0 + 2.0 * r, "cpu")
    # total tokens: every rank processed batch x T tokens
    tokens = w.batch * w.seqlen * ws
    q.put((r, float(x[0, 0, 0, 0, 0]), t, tokens))
    bench.barrier(d)
    dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_max_timing():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    out = sorted(q.get(timeout=10) for _ in range(2))
    (r0, x0, t0, n0), (r1, x1, t1, n1) = out
    assert (r0, r1) == (0, 1)
    assert x0 != x1, "replicas must be drawn with different seeds"
    assert t0 == t1 == 3.0, "timing is the maximum over ranks on every rank"
    assert n0 == n1 == 2 * 32


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3", "--workload", "tiny_fp32_b1_h2_T256_P16_N16_R1_Q64"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--workload", "tiny_fp32_b1_h2_T256_P16_N16_R1_Q64"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
