"""Benchmark of one paged decode step on GB300.

A step is the whole hot path for one batch: copy-on-write block copies (when
the step has any), the append of each sequence's new token, and decode
attention over every sequence's full context, for one attention layer.
Default workload (the headline): Llama-3.3-70B geometry (64 q / 8 kv heads,
d_h 128, bf16, 16-token blocks), batch 256, lognormal(4096, 1.2) contexts
clipped to [16, 131072] with four sequences at 131,072, permuted pool with
10% free blocks. The same run also times the Llama-3-8B-geometry batch of 64
(lognormal(1024, 1.0) contexts in [1, 8192]) and reports it under
per_workload.

value = decode tokens per second = sequences per step / step time (all ranks'
sequences over the slowest rank's time). Timing: CUDA events on the launch
stream, L2 flushed before every timed launch (256 MiB written, then 256 MiB
read, so L2 is cold and clean), outside the events. e2e: the same step
through the public API from pinned host buffers, host->device copies of the
step inputs and the device->host copy of the output inside the timed region.

cpu_baseline and --impl reference time the oracle (plain numpy, float64) on
the same sample of the workload's sequences, one process per host core.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention tokens/s and achieved HBM GB/s (% of GB300 peak)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
# The decode kernel's device code: a recorded ncu capture applies while these
# are unchanged.
KERNEL_SOURCES = [os.path.join(ROOT, "paged_kv_cache_49_gb300", "csrc", f)
                  for f in ("pkv_decode_kernel.cuh", "pkv_ptx.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_dram_traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama33_70b_b256")
    ap.add_argument("--also", default="llama3_8b_b64",
                    help="comma-separated workloads also timed in the same run (per_workload); 'none' for none")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="least wall time of the timed oracle passes")
    ap.add_argument("--num-ctas", type=int, default=0)
    ap.add_argument("--block-tokens", type=int, default=16, help="cache block size (8, 16, 32 or 64)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-math-ab", action="store_true",
                    help="skip timing the CUDA-core variant of the attention math beside the tensor-core kernel")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device="cuda") -> float:
    """The largest value over all ranks (the slowest rank's time); the value
    itself for one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(name: str, rank: int, **kw):
    """Weak scaling: every rank serves its own independent batch, seeded by
    its rank (no data is exchanged between ranks)."""
    from workloads import make_workload
    return make_workload(name, seed=rank, **kw)


def whole_job_rate(units_per_rank: int, world: int, ms: float) -> float:
    """Units per second over all ranks: every rank processes its own units
    in ms (the slowest rank's time)."""
    return units_per_rank * world / (ms * 1e-3)


def algorithmic_bytes(ctx, hq, hkv, d=128, block_tokens=16):
    """Decode attention's bytes per launch: every context token's K and V
    rows once, q and out, the table entries read and the lengths."""
    ctx = np.asarray(ctx, dtype=np.int64)
    kv = int(ctx.sum()) * hkv * d * 2 * 2
    qo = 2 * len(ctx) * hq * d * 2
    bt = int(((ctx + block_tokens - 1) // block_tokens).sum()) * 4
    return kv + qo + bt + len(ctx) * 4


def unique_kv_bytes(tables, ctx, hkv, d=128, block_tokens=16):
    """K and V bytes of the distinct physical blocks the launch reads: below
    the algorithmic bytes when sequences share blocks (prefix groups, forks),
    where the shared blocks can be served from L2 after their first read."""
    used = set()
    for row, c in zip(tables, np.asarray(ctx)):
        used.update(int(b) for b in row[: (int(c) + block_tokens - 1) // block_tokens])
    return len(used) * hkv * block_tokens * d * 2 * 2


def tail_waste_tokens(ctx, block_tokens=16):
    """Slots of the batch's last blocks that hold no token: a sequence of n
    tokens occupies ceil(n / b) blocks, wasting b * ceil(n / b) - n slots."""
    ctx = np.asarray(ctx, dtype=np.int64)
    return int((((ctx + block_tokens - 1) // block_tokens) * block_tokens - ctx)[ctx > 0].sum())


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, units):
    """DRAM bytes per launch from a committed ncu capture of this workload,
    (value, "measured"); else one of another workload scaled to this launch by
    context tokens, (value, "scaled from <workload>"); else (None, reason).
    Nothing applies once the kernel's device code has changed."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, "no traffic record"
    if rec.get("kernel_sha256_16") != kernel_hash():
        return None, "kernel changed since the traffic record"
    records = rec.get("records", {})
    if workload in records:
        return float(records[workload]["dram_bytes_per_launch"]), "measured"
    for name, r in sorted(records.items()):
        if r.get("context_tokens"):
            return float(r["dram_bytes_per_launch"]) * units / float(r["context_tokens"]), f"scaled from {name}"
    return None, "no traffic record"


# ---------------------------------------------------------------------------
# The oracle on the host cores: cpu_baseline and the reference arm.

def oracle_sample(ctx):
    """Rows the oracle baseline times: every 4th sequence by context length,
    plus the longest contexts (up to four rows at the maximum)."""
    ctx = np.asarray(ctx)
    order = np.argsort(ctx, kind="stable")
    rows = set(int(r) for r in order[::4])
    rows.update(int(r) for r in np.flatnonzero(ctx == ctx.max())[:4])
    return sorted(rows)


def split_rows(rows, ctx, n):
    """Rows dealt to n workers, longest first to the least loaded (about
    equal context tokens each); empty shares are dropped."""
    shares = [[] for _ in range(n)]
    load = [0] * n
    for r in sorted(rows, key=lambda r: -int(ctx[r])):
        i = load.index(min(load))
        shares[i].append(r)
        load[i] += int(ctx[r]) + 1
    return [sorted(x) for x in shares if x]


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_batch_ctx(w):
    """Context lengths of the workload's decode step, from the oracle's block
    manager (bookkeeping only, no pool)."""
    from oracle import scenario
    from oracle.block_manager import BlockManager
    bm = BlockManager(w.pool_blocks, w.block_tokens, w.free_order)
    scenario._apply_events(w, bm)
    bm.prepare_append(w.batch)
    return np.array([bm.context_len(s) for s in w.batch], dtype=np.int64)


def _oracle_worker(conn, name, seed, rows, extra):
    """One host core's share of the oracle step: its rows' inputs are built
    once (untimed), then each request runs the step -- the block copies, the
    rows' appends and their attention -- and answers with its duration."""
    from oracle import cache_ops, paged_attention, scenario
    from workloads import make_workload
    try:
        w = make_workload(name, seed=seed, **extra)
        if any(ev[0] == "history" for ev in w.events):
            ref = scenario.replay(w, attend=False)  # small pools: the whole pool
            q, k_new, v_new = w.step_inputs()
            inp = dict(q=q[rows], k_new=k_new[rows], v_new=v_new[rows], k_pool=ref["k_pool"], v_pool=ref["v_pool"],
                       pairs=ref["pairs"], slots=[ref["slots"][r] for r in rows], tables=ref["tables"][rows],
                       ctx=ref["ctx"][rows])
        else:
            inp = scenario.sampled_inputs(w, rows)
        conn.send(("ready", int(np.sum(inp["ctx"]))))
        while True:
            cmd = conn.recv()
            if cmd == "stop":
                break
            t0 = time.perf_counter()
            cache_ops.copy_blocks(inp["k_pool"], inp["v_pool"], inp["pairs"])
            cache_ops.append_kv(inp["k_pool"], inp["v_pool"], inp["k_new"], inp["v_new"], inp["slots"])
            out = paged_attention.paged_decode_attention(inp["q"], inp["k_pool"], inp["v_pool"], inp["tables"],
                                                         inp["ctx"], w.scale)
            el = time.perf_counter() - t0
            conn.send(("done", el, out if cmd == "out" else None))
    except Exception as e:  # reported to the parent, which raises
        conn.send(("error", repr(e)))
    finally:
        conn.close()


class OracleCores:
    """The oracle step on a sample of a workload's sequences, one spawned
    process per host core (each builds its rows' inputs once). step() runs
    one pass over the sample on every worker at once and returns its wall
    time and the sum of the workers' busy times (what one core would take)."""

    def __init__(self, name, seed, rows, ctx, workers, extra=None):
        import multiprocessing as mp
        env = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in env:
            os.environ[k] = "1"  # one thread per worker process
        ctxm = mp.get_context("spawn")
        self.rows = list(rows)
        self.shares = split_rows(self.rows, ctx, max(1, workers))
        self.procs, self.conns = [], []
        try:
            for share in self.shares:
                a, b = ctxm.Pipe()
                p = ctxm.Process(target=_oracle_worker, args=(b, name, seed, share, extra or {}), daemon=True)
                p.start()
                self.procs.append(p)
                self.conns.append(a)
        finally:
            for k, v in env.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.context_tokens = None

    @property
    def workers(self):
        return len(self.shares)

    def _recv(self, c):
        msg = c.recv()
        if msg[0] == "error":
            raise RuntimeError(f"oracle worker failed: {msg[1]}")
        return msg

    def wait_ready(self):
        if self.context_tokens is None:
            self.context_tokens = sum(self._recv(c)[1] for c in self.conns)
        return self

    def step(self, want_out=False):
        self.wait_ready()
        t0 = time.perf_counter()
        for c in self.conns:
            c.send("out" if want_out else "run")
        msgs = [self._recv(c) for c in self.conns]
        wall = time.perf_counter() - t0
        busy = sum(m[1] for m in msgs)
        if want_out:
            out = {}
            for share, m in zip(self.shares, msgs):
                for i, r in enumerate(share):
                    out[r] = m[2][i]
            return wall, busy, out
        return wall, busy

    def close(self):
        for c in self.conns:
            try:
                c.send("stop")
            except OSError:
                pass
        for p in self.procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()

    def describe(self, w):
        return (f"{len(self.rows)} of {w.batch_size} sequences (every 4th by context length and the longest; "
                f"{self.context_tokens} context tokens), one process per host core ({self.workers}); "
                "numpy float64 oracle, as committed")


def time_oracle(pool, min_seconds, w):
    """Passes of the oracle step over the sample until min_seconds of wall
    time; the cpu_baseline record."""
    pool.wait_ready()
    pool.step()  # warm-up pass
    walls, busy = [], []
    while sum(walls) < min_seconds:
        a, b = pool.step()
        walls.append(a)
        busy.append(b)
    n = len(pool.rows)
    return {"value": n * len(walls) / sum(walls), "unit": UNIT, "cores": pool.workers, "kind": "oracle",
            "sample": pool.describe(w), "timing": f"{len(walls)} timed passes over the sample, {sum(walls):.1f} s",
            "single_core_value": n * len(busy) / sum(busy),
            "single_core_note": "the same passes' summed per-process busy time (the time one core would take)"}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    from workloads import make_workload

    w = make_workload(args.workload)
    ctx = oracle_batch_ctx(w)
    rows = oracle_sample(ctx)
    pool = OracleCores(args.workload, 0, rows, ctx, min(host_cores(), len(rows)))
    try:
        pool.wait_ready()
        for _ in range(args.warmup):
            pool.step()
        walls, busy = [], []
        for _ in range(args.steps):
            a, b = pool.step()
            walls.append(a)
            busy.append(b)
    finally:
        pool.close()
    el = sum(walls)
    value = len(rows) * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch_size, "q_heads": w.num_q_heads,
                   "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_tokens": 16,
                   "sample_sequences": len(rows), "sample_context_tokens": pool.context_tokens},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
                         "sample": pool.describe(w), "timing": "one pass over the sample per step",
                         "single_core_value": len(rows) * args.steps / sum(busy)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class L2Flush:
    """Leaves L2 cold and clean: write a buffer twice the L2 size, then read
    another one, so that the lines the timed kernel finds in L2 are clean
    (evicting them costs no DRAM write-back) and none of them is its data."""

    def __init__(self):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def __call__(self, i: int):
        self.w.fill_(i & 0xFF)
        self.r.max()


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled every ~1 ms from
    NVML (read-only queries through libnvidia-ml) in a background thread
    while the timed region runs; nvidia-smi at 200 ms if NVML is missing."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index):
        self.device_index = device_index
        self.samples = []
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self._nvml = None
        self._handle = None
        self._smi = None
        self._smi_path = None

    def _open_nvml(self):
        import ctypes
        import torch
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if nv.nvmlInit_v2() != 0:
            return False
        p = torch.cuda.get_device_properties(self.device_index)
        bus = f"{getattr(p, 'pci_domain_id', 0):08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            return False
        mx = ctypes.c_uint(0)
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nvml, self._handle = nv, h
        return True

    def _poll(self):
        import ctypes
        nv, h = self._nvml, self._handle
        mhz, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and \
                    get_reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(0.001)

    def __enter__(self):
        import threading
        if self._open_nvml():
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            time.sleep(0.01)
        else:
            fd, self._smi_path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.device_index}",
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=open(self._smi_path, "w"), stderr=subprocess.DEVNULL)
            except OSError:
                self._smi = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        if self._smi is not None:
            self._smi.terminate()
            self._smi.wait(timeout=5)
            with open(self._smi_path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    try:
                        self.samples.append((float(parts[0]), int(parts[2], 16)))
                        self.max_mhz = float(parts[1])
                    except (ValueError, IndexError):
                        pass
        if self._smi_path:
            os.unlink(self._smi_path)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"], "samples": 0}
        mask = 0
        for _, r in self.samples:
            mask |= r
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for bit, n in self.REASONS.items() if mask & bit),
                "samples": len(self.samples), "source": "nvml" if self._nvml else "nvidia-smi"}


def measure(pkv, name, args, rank, world, local, flush, e2e_on=True):
    """One workload on this rank's GPU: the timed decode steps, the step's
    kernels alone, end to end through the host-buffer call, and the roofline
    of the attention launch. Returns the measurements for the JSON line."""
    import torch
    import torch.distributed as dist

    extra = {} if args.block_tokens == 16 else {"block_tokens": args.block_tokens}
    w = rank_workload(name, rank, **extra)
    eng = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim, free_order=w.free_order,
                            block_tokens=w.block_tokens)
    eng.load_workload_pool(w)
    eng.replay_events(w, with_content=True)
    q_bits, k_bits, v_bits = w.step_inputs()
    sb = eng.prepare_step(w.batch, q_bits, k_bits, v_bits)
    ctx = sb.ctx.cpu().numpy()
    B = w.batch_size
    stream = torch.cuda.current_stream()
    pool = dict(eng.bm.stats(), num_blocks=w.pool_blocks,
                tail_waste_tokens=tail_waste_tokens(ctx, w.block_tokens))  # the block manager's counters

    for _ in range(args.warmup):
        eng.run_step(sb, w.scale, args.num_ctas)
    torch.cuda.synchronize()
    if eng.read_errors(sb):
        raise RuntimeError("device error word set during warm-up")

    # Timed region: K decode steps (one pkv_decode_step call each: copies,
    # append, attention), then K attention launches alone for the roofline.
    # L2 is flushed before every timed launch, outside its events. A spin
    # kernel issued first keeps the GPU busy while the host enqueues all of
    # it, so host submission latency does not land inside device timings
    # (the effect CUDA-graph replay of a decode step has in a server).
    ev = lambda n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    ev_step, ev_attn, ev_app = ev(args.steps), ev(args.steps), ev(args.steps)
    ev_copy = ev(args.steps if sb.num_pairs else 0)
    # batches whose shared prefixes save enough reads: cascade attention too
    cas = eng.cascade_for(sb)
    cas_out = torch.empty_like(sb.out) if cas else None
    ev_cas = ev(args.steps if cas else 0)
    # the same attention with its per-tile math on the CUDA cores (group sizes
    # 4 and 8): the measured alternative to the tensor cores
    fma_ok = not args.no_math_ab and w.block_tokens == 16 and w.num_q_heads // w.num_kv_heads in (4, 8)
    fma_out = torch.empty_like(sb.out) if fma_ok else None
    ev_fma = ev(args.steps if fma_ok else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        torch.cuda._sleep(int(2.0e9 * (0.003 + 400e-6 * args.steps)))
        flush(0)  # one untimed step after the spin kernel, so the first timed one is not the first to run
        eng.run_step(sb, w.scale, args.num_ctas)
        for i in range(args.steps):
            flush(i)
            ev_step[i][0].record(stream)
            eng.run_step(sb, w.scale, args.num_ctas)
            ev_step[i][1].record(stream)
        for i in range(args.steps):
            flush(i + 1)
            ev_attn[i][0].record(stream)
            pkv.attn_decode(sb.q, eng.k_cache, eng.v_cache, sb.tables, sb.ctx, w.scale, sb.out,
                            sb.workspace, args.num_ctas)
            ev_attn[i][1].record(stream)
        for i, (e0, e1) in enumerate(ev_app):  # the step's cache kernels alone (idempotent for fixed inputs)
            flush(i + 2)
            e0.record(stream)
            pkv.append(sb.k, sb.v, sb.slots, eng.k_cache, eng.v_cache, eng.error)
            e1.record(stream)
        for i, (e0, e1) in enumerate(ev_copy):
            flush(i + 3)
            e0.record(stream)
            pkv.block_copy(eng.k_cache, eng.v_cache, sb.pairs, eng.error)
            e1.record(stream)
        for i, (e0, e1) in enumerate(ev_cas):
            flush(i + 4)
            e0.record(stream)
            cas.decode(sb.q, eng.k_cache, eng.v_cache, sb.tables, sb.ctx, w.scale, cas_out)
            e1.record(stream)
        for i, (e0, e1) in enumerate(ev_fma):
            flush(i + 5)
            e0.record(stream)
            pkv.attn_decode_cuda_cores(sb.q, eng.k_cache, eng.v_cache, sb.tables, sb.ctx, w.scale, fma_out,
                                       sb.workspace, args.num_ctas)
            e1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    attn_ms = [a.elapsed_time(b) for a, b in ev_attn]
    ms = max_over_ranks(statistics.mean(step_ms), world)

    def stats_of(evs):
        t = [a.elapsed_time(b) for a, b in evs]
        return {"min": min(t), "median": statistics.median(t), "max": max(t)} if t else None

    launches = (args.steps * (2 + (1 if sb.num_pairs else 0)) + args.steps + len(ev_app) + len(ev_copy)
                + 3 * len(ev_cas) + len(ev_fma))
    if fma_ok and (fma_out.float() - sb.out.float()).abs().max().item() > 4e-2:
        raise RuntimeError("the CUDA-core variant differs from the tensor-core kernel")
    if cas is not None:
        if cas.read_error():
            raise RuntimeError("device error word set by the cascade attention")
        if (cas_out.float() - sb.out.float()).abs().max().item() > 4e-2:
            raise RuntimeError("cascade attention differs from the plain kernel")
    if eng.read_errors(sb):
        raise RuntimeError("device error word set during the timed steps")

    # ---- end to end through the C ABI's host-buffer step ----
    # Every step (pkv_decode_step_host): the packed inputs brought from pinned
    # host memory (a staging kernel reads them across the host link), the
    # step's kernels, and the output rows written back to pinned host memory
    # by the attention itself.
    e2e = None
    if e2e_on:
        hs = pkv.HostStep(eng, B, sb.tables.shape[1], max_pairs=max(1, sb.num_pairs))
        hs.pack(sb.q.cpu(), sb.k.cpu(), sb.v.cpu(), sb.slots.cpu(), sb.tables.cpu(), sb.ctx.cpu(),
                sb.pairs.cpu() if sb.num_pairs else None)
        h2d = hs.h2d_bytes()  # what crosses the host link each step (table rows up to their live entries)
        d2h = hs.out_host.numel() * hs.out_host.element_size()

        def timed(run):
            ts = []
            for i in range(args.warmup + args.steps):
                flush(i)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run()
                e1.record(stream)
                e1.synchronize()
                if i >= args.warmup:
                    ts.append(e0.elapsed_time(e1))
            return max_over_ranks(statistics.mean(ts), world)

        e2e_ms = timed(lambda: hs.run(w.scale, args.num_ctas))
        if not torch.equal(hs.out_host, sb.out.cpu()):
            raise RuntimeError("host-buffer step output differs from the device step")
        e2e = {"value": whole_job_rate(B, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "call": "pkv_decode_step_host"}
        # The same call captured once in a CUDA graph and replayed (as a server does).
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            hs.run(w.scale, args.num_ctas)
        g_ms = timed(graph.replay)
        e2e["graph_replay"] = {"value": whole_job_rate(B, world, g_ms), "ms_per_step": g_ms}
        # timed calls, eager and replayed: staging, block copy (if any), append, attention
        launches += 2 * args.steps * (3 + (1 if sb.num_pairs else 0))

    abytes = algorithmic_bytes(ctx, w.num_q_heads, w.num_kv_heads, block_tokens=w.block_tokens)
    ubytes = unique_kv_bytes(sb.tables.cpu().numpy(), ctx, w.num_kv_heads, block_tokens=w.block_tokens)
    attn_s = statistics.mean(attn_ms) * 1e-3
    peak, peak_kind = measured_peak_gbs()
    achieved = abytes / attn_s / 1e9
    traffic, traffic_src = recorded_traffic(w.name, int(ctx.sum()))
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_src,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs copy bandwidth)",
                "kernel": "pkv::attn::decode_kernel", "algorithmic_bytes_per_launch": abytes,
                "attn_ms": attn_s * 1e3, "attn_ms_min": min(attn_ms), "frac_of_nominal_8tbs": achieved / 8000.0,
                "unique_kv_bytes_per_launch": ubytes, "unique_kv_gbs": ubytes / attn_s / 1e9}
    if cas is not None:
        cas_s = statistics.mean(a.elapsed_time(b) for a, b in ev_cas) * 1e-3
        roofline["cascade"] = {"attn_ms": cas_s * 1e3, "groups": len(cas.groups),
                               "saved_kv_bytes": pkv.cascade_saved_bytes(cas.groups, w.num_kv_heads),
                               "logical_gbs": abytes / cas_s / 1e9, "unique_kv_gbs": ubytes / cas_s / 1e9,
                               "frac_unique_of_measured": ubytes / cas_s / 1e9 / peak}
    if fma_ok:
        fma_s = statistics.mean(a.elapsed_time(b) for a, b in ev_fma) * 1e-3
        roofline["cuda_core_variant"] = {
            "kernel": "pkv::attn::decode_kernel, per-tile math on FP32 FMA", "attn_ms": fma_s * 1e3,
            "achieved": abytes / fma_s / 1e9, "frac": abytes / fma_s / 1e9 / peak,
            "tensor_core_speedup": fma_s / attn_s}
    res = {
        "w": w, "value": whole_job_rate(B, world, ms), "ms_per_step": ms, "e2e": e2e, "gpu_launches": launches,
        "roofline": roofline, "clocks": clk.summary(), "pool": pool,
        "timing_ms": {"step": stats_of(ev_step), "attention_alone": stats_of(ev_attn),
                      "append_alone": stats_of(ev_app), "block_copy_alone": stats_of(ev_copy),
                      "attention_cascade": stats_of(ev_cas), "attention_cuda_cores": stats_of(ev_fma)},
        "config": {"workload": w.name, "batch": B, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "block_tokens": w.block_tokens, "context_tokens": int(ctx.sum()),
                   "pool_blocks": w.pool_blocks, "cow_pairs_per_step": sb.num_pairs,
                   "num_ctas": args.num_ctas or pkv.launch_ctas(B, w.num_kv_heads, int(sb.tables.shape[1]),
                                                                 w.block_tokens),
                   "l2": "flushed before each timed launch (256 MiB write, then 256 MiB read: cold and clean)",
                   "parallelism": f"replicas x{world}"},
    }
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_info()
    # The oracle's host processes (rank 0, one GPU) are spawned first, so
    # that they build their inputs while the GPU side loads its pool.
    pool = None
    if not args.no_cpu_baseline and world == 1:
        from workloads import make_workload
        w0 = make_workload(args.workload) if args.block_tokens == 16 else None
        if w0 is not None:
            ctx0 = oracle_batch_ctx(w0)
            rows = oracle_sample(ctx0)
            pool = OracleCores(args.workload, 0, rows, ctx0, min(host_cores(), len(rows)))
    try:
        torch.cuda.set_device(local)
        if world > 1:
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        if rank == 0 or world == 1:
            from __graft_entry__ import _build_module
            _build_module().build()
        if world > 1:
            dist.barrier()
        import paged_kv_cache_49_gb300 as pkv

        flush = L2Flush()
        head = measure(pkv, args.workload, args, rank, world, local, flush, e2e_on=not args.no_e2e)
        others = {}
        for name in [x for x in args.also.split(",") if x and x != "none" and x != args.workload]:
            torch.cuda.empty_cache()  # the previous workload's pool
            m = measure(pkv, name, args, rank, world, local, flush, e2e_on=not args.no_e2e)
            others[name] = {k: m[k] for k in ("value", "ms_per_step", "e2e", "roofline", "timing_ms", "clocks",
                                              "config", "gpu_launches", "pool")}
        cpu = time_oracle(pool, args.cpu_seconds, head["w"]) if pool is not None and rank == 0 else None
    finally:
        if pool is not None:
            pool.close()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": head["config"],
        "clocks": head["clocks"], "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"] + sum(o["gpu_launches"] for o in others.values()),
        "roofline": head["roofline"], "timing_ms": head["timing_ms"], "pool": head["pool"], "cpu_baseline": cpu,
        "per_workload": others,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
