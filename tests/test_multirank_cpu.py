"""The bench's multi-GPU path on the CPU: two ranks over gloo (127.0.0.1).
Ranks serve independent batches (weak scaling, no data exchanged); the
step time reported is the slowest rank's; the whole-job rate counts every
rank's units; the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.5 + rank, world, device="cpu")  # rank 1 is slower
        w = bench.rank_workload("tiny", rank)
        q, _, _ = w.step_inputs()
        out.put((rank, slowest, w.seed, q.tobytes()[:64], bench.whole_job_rate(w.batch_size, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_to_the_slowest_and_serve_independent_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, seed0, q0, rate0), (r1, s1, seed1, q1, rate1) = res
    assert s0 == s1 == 2.5  # both ranks report the slowest rank's time
    assert (seed0, seed1) == (0, 1) and q0 != q1  # independent, rank-seeded batches
    assert rate0 == rate1 == 4 * 2 / 2.5e-3  # every rank's sequences over the slowest time


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", LOCAL_RANK="0", MASTER_ADDR="127.0.0.1")
    lines = {}
    for rank in (0, 1):
        env["RANK"] = str(rank)
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                            "tiny", "--gpus", "2", "--steps", "1", "--warmup", "1"],
                           capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        lines[rank] = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert lines[1] == []
    (line,) = lines[0]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert np.isfinite(d["ms_per_step"])
