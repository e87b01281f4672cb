"""Benchmark of the Mamba-3 SSM layer recurrence on B300.

One JSON line on rank 0.  A step is one chunked prefill (m3_scan_fwd: every
hot-path step from coefficients to the final state) over the SISO workload at
~1.5B layer width: batch 4, 64 heads, P=64, N=128, R=1, T=4096, chunk 64,
bf16 x/B/C, fp32 dt/lambda/omega/A and fp32 final state.  Inputs (1.09 GB
per step) are larger than L2, so no flush is needed between steps.

value       prefill Mtok/s (tokens = batch x T; each token covers all heads),
            inputs resident in HBM, CUDA events on the launch stream.
e2e         the same through the C ABI with pinned HOST buffers: host-to-device
            copies of the step's inputs and device-to-host copies of y and the
            final state are inside the timed region.
roofline    algorithmic bytes of one m3_scan_fwd call / its event-timed
            duration, against the measured HBM copy bandwidth.
decode      the decode sweep (batch 1/8/64/256 x R 1/4, H=64, P=64, N=128):
            1024 carried m3_decode_step calls each, steps/s and HBM roofline.
cpu_baseline  the float64 oracle on a bounded sample of the same workload,
            on this host's cores.

Launch: python bench.py [--gpus N --steps K --warmup W] [--impl reference];
for N > 1 under torch.distributed.run, one rank per GPU, each rank an
independent replica of the workload (the (batch, head) sequences are
independent: no collective on the data path), timing max-reduced over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from state_space_sequence_04_b300 import synth  # noqa: E402

METRIC = "Mamba-3 SSM prefill Mtok/s & decode steps/s on 1 B300; % of roofline"
KEYS = ("x", "B", "C", "dt", "A", "lam", "omega")
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0


def peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# algorithmic cost model (bytes that must cross HBM once; FLOPs of the chunked form)
def io_bytes(io: str) -> int:
    return 2 if io == "bf16" else 4


def prefill_bytes(w: synth.Workload) -> int:
    """x, B, C, omega, dt, lambda read once; y written once; final state written once."""
    e = io_bytes(w.io)
    R, P, N = w.rank, w.headdim, w.dstate
    per_ht = R * P * e + 2 * R * N * e + (N // 2) * 4 + 8 + R * P * e
    return per_ht * w.batch * w.seqlen * w.heads + w.batch * w.heads * N * P * 4 + w.heads * 4


def prefill_tc_flops(w: synth.Workload) -> float:
    """Tensor-core FLOPs of the chunked form per call: causal half of the (QR)^2 score
    square times N and P, plus chunk state (N x P x QR) and inter output (QR x N x P)."""
    Q, R, N, P = w.chunk, w.rank, w.dstate, w.headdim
    nchunk_tok = w.batch * w.heads * w.seqlen / Q
    qr = Q * R
    causal = qr * (qr + R) / 2.0
    per_chunk = 2 * causal * N + 2 * causal * P + 2 * N * P * qr + 2 * qr * N * P
    return per_chunk * nchunk_tok


def decode_bytes(b: int, H: int, P: int, N: int, R: int, io: str = "bf16") -> int:
    """State read + write (fp32), inputs and cache read, cache and y written."""
    e = io_bytes(io)
    per = 8 * N * P + (R * P + 2 * R * N) * e + (N // 2) * 4 + 8 + 2 * R * (N + P) * e + R * P * e
    return b * H * per + H * 4


# ---------------------------------------------------------------------------
class ClockSampler:
    """Samples SM clocks and throttle reasons through NVML while running (read only)."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.01):
        self.samples = []
        self.period = period_s
        self._stop = threading.Event()
        self._thread = None
        self.max_mhz = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
        except Exception as exc:  # NVML missing: report no clocks rather than guess
            self._nv = None
            self.error = str(exc)

    def _run(self):
        nv = self._nv
        while not self._stop.is_set():
            try:
                mhz = nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM)
                rs = nv.nvmlDeviceGetCurrentClocksEventReasons(self._h)
                self.samples.append((mhz, int(rs)))
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self._nv is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()

    def summary(self):
        if self._nv is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        reasons = sorted({name for _, r in busy for bit, name in self.REASONS.items() if r & bit})
        mhz = statistics.median([m for m, _ in busy]) if busy else None
        return {"sm_mhz": mhz, "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(busy)}


# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, local, backend):
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
def time_prefill(binding, w, d, stream, steps, warmup, dist, device):
    """Device-resident prefill: returns (total seconds max over ranks, per-call event ms list)."""
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.batch, w.heads, w.dstate, w.headdim), dtype=torch.float32, device=device)
    ws = binding.alloc_workspace(d["x"].shape, w.dstate, w.rank, w.chunk, d["x"].dtype, device)
    args = [d[k] for k in KEYS]

    def call():
        st = binding.m3_scan_fwd(*args, w.rank, w.chunk, y, fin, ws, stream)
        if st != 0:
            raise binding.M3Error(st, "m3_scan_fwd")

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(dist)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    total_ms = start.elapsed_time(end)
    per = [a.elapsed_time(b) for a, b in ev]
    return max_over_ranks(dist, total_ms, device) / 1e3, per, (y, fin)


def time_prefill_e2e(binding, w, host, stream, steps, warmup, dist, device):
    """Host pinned buffers in, y and final state back to host, all inside the timed region."""
    dev = {k: torch.empty_like(host[k], device=device) for k in KEYS}
    y = torch.empty_like(dev["x"])
    fin = torch.empty((w.batch, w.heads, w.dstate, w.headdim), dtype=torch.float32, device=device)
    y_h = torch.empty_like(y, device="cpu").pin_memory()
    fin_h = torch.empty_like(fin, device="cpu").pin_memory()
    ws = binding.alloc_workspace(dev["x"].shape, w.dstate, w.rank, w.chunk, dev["x"].dtype, device)
    h2d = sum(host[k].numel() * host[k].element_size() for k in KEYS)
    d2h = y.numel() * y.element_size() + fin.numel() * fin.element_size()

    def step():
        for k in KEYS:
            dev[k].copy_(host[k], non_blocking=True)
        st = binding.m3_scan_fwd(*[dev[k] for k in KEYS], w.rank, w.chunk, y, fin, ws, stream)
        if st != 0:
            raise binding.M3Error(st, "m3_scan_fwd")
        y_h.copy_(y, non_blocking=True)
        fin_h.copy_(fin, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        barrier(dist)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            step()
        t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    sec = max_over_ranks(dist, t0.elapsed_time(t1), device) / 1e3
    return sec, h2d, d2h


def time_decode(binding, b, R, stream, device, steps=synth.DECODE_STEPS, ring=32, warmup=16):
    """``steps`` carried decode calls at batch b, rank R (H=64, P=64, N=128); per-step
    inputs cycle through ``ring`` pre-drawn sets.  Returns seconds for all steps."""
    H, P, N = 64, 64, 128
    state = synth.make_decode_state(b, H, N, P, seed=0, device=device)
    ins = synth.make_decode_steps(b, H, P, N, R, ring, io="bf16", seed=1, device=device)
    cache = binding.new_decode_cache(b, H, N, P, R, torch.bfloat16, device)
    y_t = torch.empty((b, H, R, P), dtype=torch.bfloat16, device=device)
    A = ins["A"]
    per = [[ins[k][i] for k in ("x", "B", "C", "dt", "lam", "omega")] for i in range(ring)]

    def call(i):
        a = per[i % ring]
        st = binding.m3_decode_step(state, a[0], a[1], cache, a[2], a[3], A, a[4], a[5], y_t, R, stream)
        if st != 0:
            raise binding.M3Error(st, "m3_decode_step")

    with torch.cuda.stream(stream):
        for i in range(warmup):
            call(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        call(i)
    t1.record(stream)
    torch.cuda.synchronize()
    ok = bool(torch.isfinite(state).all())
    return t0.elapsed_time(t1) / 1e3, ok


# ---------------------------------------------------------------------------
def cpu_baseline_run(w, target_s: float = 12.0, max_s: float = 40.0):
    """Time the float64 oracle on a bounded sample of the workload: whole sequences
    (one (batch, head) of T tokens each), doubling the sample until it runs
    >= target_s.  Returns (Mtok/s, threads, sample description, seconds)."""
    import oracle
    threads = oracle.num_threads()
    inp = synth.make_inputs(w, seed=0, batch=1)   # batch row 0 of the workload: H sequences
    n = max(1, min(w.heads, threads))
    while True:
        heads = list(range(n))
        args = [inp["x"][:, :, heads], inp["B"][:, :, heads], inp["C"][:, :, heads], inp["dt"][:, :, heads],
                inp["A"][heads], inp["lam"][:, :, heads], inp["omega"][:, :, heads]]
        args = [oracle.f64(a) for a in args]
        t0 = time.perf_counter()
        oracle.scan(*args)
        el = time.perf_counter() - t0
        if el >= target_s or n >= w.heads or el * 2 > max_s:
            break
        n = min(w.heads, n * 2)
    tokens = n * w.seqlen / w.heads          # token-equivalents (a token covers all heads)
    sample = f"{n} of {w.heads * w.batch} (batch, head) sequences x {w.seqlen} tokens, float64"
    return tokens / el / 1e6, threads, sample, el


def run_reference(args):
    """--impl reference: the float64 oracle timed as it stands on the host cores."""
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = synth.SISO_1P5B
    threads = oracle.num_threads()
    inp = synth.make_inputs(w, seed=0, batch=1)
    n = max(1, min(w.heads, threads))
    heads = list(range(n))
    a = [oracle.f64(v) for v in (inp["x"][:, :, heads], inp["B"][:, :, heads], inp["C"][:, :, heads],
                                 inp["dt"][:, :, heads], inp["A"][heads], inp["lam"][:, :, heads],
                                 inp["omega"][:, :, heads])]
    for _ in range(args.warmup):
        oracle.scan(*a)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan(*a)
    el = time.perf_counter() - t0
    tokens = n * w.seqlen / w.heads * args.steps
    val = tokens / el / 1e6
    sample = f"per step {n} of {w.heads * w.batch} (batch, head) sequences x {w.seqlen} tokens, float64"
    line = {
        "metric": METRIC, "value": val, "unit": "Mtok/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name},
        "cpu_baseline": {"value": val, "unit": "Mtok/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "Mtok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default=synth.SISO_1P5B.name, choices=sorted(synth.WORKLOADS))
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(ws, local, "nccl")
    from state_space_sequence_04_b300 import binding
    binding.load()
    pk = peaks()
    w = synth.WORKLOADS[args.workload]
    stream = torch.cuda.Stream(device=device)

    # every rank draws its own replica of the workload (seeded by rank)
    d = synth.make_inputs(w, seed=rank, device=device)
    path, launches = binding.m3_scan_fwd_plan(w.batch, w.seqlen, w.heads, w.headdim, w.dstate, w.rank, w.chunk,
                                              binding.io_code(d["x"].dtype))
    with ClockSampler(local) as clk:
        sec, per_ms, _ = time_prefill(binding, w, d, stream, args.steps, args.warmup, dist, device)
    clocks = clk.summary()
    tokens = w.batch * w.seqlen * ws
    value = tokens / sec / 1e6
    avg_call_ms = sum(per_ms) / len(per_ms)
    nbytes = prefill_bytes(w)
    achieved_gbs = nbytes / (avg_call_ms * 1e-3) / 1e9
    tflops = prefill_tc_flops(w) / (avg_call_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "Mtok/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if path == 1 else "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "heads": w.heads,
                   "headdim": w.headdim, "dstate": w.dstate, "rank": w.rank, "chunk": w.chunk, "io": w.io,
                   "parallelism": f"replicas x{ws} (independent (batch, head) sequences, no collective)",
                   "l2": f"inputs larger than L2 ({nbytes / 1e9:.2f} GB per step), no flush"},
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved_gbs / pk["hbm_gbs"], "traffic": None,
                     "kernel": "m3_scan_fwd (" + ("tensor-core" if path == 1 else "CUDA-core") +
                               f" path, {launches} launches per call)",
                     "algorithmic_bytes_per_call": nbytes, "peak_source": pk["source"],
                     "tc_tflops": tflops, "tc_frac_of_bf16_peak": tflops / pk["bf16_tflops"]},
        "clocks": clocks,
    }

    if not args.no_e2e:
        host = {k: d[k].to("cpu").pin_memory() for k in KEYS}
        esec, h2d, d2h = time_prefill_e2e(binding, w, host, stream, max(3, args.steps // 4), 3, dist, device)
        line["e2e"] = {"value": tokens / (esec / max(3, args.steps // 4)) / 1e6, "unit": "Mtok/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        del host

    if not args.no_decode and rank == 0:
        dec = {}
        for R in synth.DECODE_RANKS:
            for b in synth.DECODE_BATCHES:
                dsec, ok = time_decode(binding, b, R, stream, device)
                per_step = dsec / synth.DECODE_STEPS
                gbs = decode_bytes(b, 64, 64, 128, R) / per_step / 1e9
                dec[f"b{b}_R{R}"] = {"steps_per_s": 1.0 / per_step, "us_per_step": per_step * 1e6,
                                     "tokens_per_s": b / per_step, "achieved_gbs": gbs,
                                     "frac_of_measured_hbm": gbs / pk["hbm_gbs"], "frac_of_8tbs": gbs / 8000.0,
                                     "finite": ok}
        line["decode"] = {"unit": "steps/s", "steps": synth.DECODE_STEPS, "heads": 64, "headdim": 64,
                          "dstate": 128, "eager": True, "sweep": dec}

    if not args.no_cpu_baseline and rank == 0 and ws == 1:
        v, threads, sample, el = cpu_baseline_run(w)
        line["cpu_baseline"] = {"value": v, "unit": "Mtok/s", "cores": threads, "kind": "oracle",
                                "sample": sample, "seconds": el}

    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
