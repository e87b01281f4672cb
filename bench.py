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
            1024 carried m3_decode_step calls each, steps/s and HBM roofline,
            and the float64 oracle's decode steps on the host cores.
cpu_baseline  the float64 oracle on a bounded sample of the same workload,
            on this host's cores.
workloads   the other prefill workloads, each with the same keys (value,
            roofline with ncu traffic, cpu_baseline): the tiny fp32 check
            (batch 1, 2 heads, T=256, P=N=16), MIMO prefill (batch 2, 32 heads,
            T=8192, P=N=64, R=4) and long-context MIMO prefill (batch 1, 64
            heads, T=65536, P=64, N=128, R=4, chunk 128) followed by 256 decode
            steps from its final state.

Launch: python bench.py [--gpus N --steps K --warmup W] [--impl reference];
for N > 1 under torch.distributed.run, one rank per GPU, each rank an
independent replica of the workload (the (batch, head) sequences are
independent: no collective on the data path), timing max-reduced over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
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

import numpy as np  # noqa: E402
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


def prefill_prep_bytes(w: synth.Workload) -> int:
    """As prefill_bytes, plus the per-token decay generator (4 B per (token, head)) and dt_bias."""
    return prefill_bytes(w) + 4 * w.batch * w.seqlen * w.heads


def prefill_tc_flops(w: synth.Workload) -> float:
    """Tensor-core FLOPs of the chunked form per call: causal half of the (QR)^2 score
    square times N and P, plus chunk state (N x P x QR) and inter output (QR x N x P)."""
    Q, R, N, P = w.chunk, w.rank, w.dstate, w.headdim
    nchunk_tok = w.batch * w.heads * w.seqlen / Q
    qr = Q * R
    causal = qr * (qr + R) / 2.0
    per_chunk = 2 * causal * N + 2 * causal * P + 2 * N * P * qr + 2 * qr * N * P
    return per_chunk * nchunk_tok


# fp32 CUDA-core peak: 148 SMs x 128 FP32 lanes x 2 FLOPs per FMA x the maximum SM clock
FP32_ALU_TFLOPS = 148 * 128 * 2 * 2032e6 / 1e12


def bwd_flops(w: synth.Workload) -> float:
    """FLOPs of one evaluation of the recurrence plus its adjoint, per state element and token:
    forward v_t (2R), alpha h + beta v_{t-1} (3), rotation (3), + gamma v_t (2); adjoint gbar (2R + 2),
    dv (3), r (2), dphi (2), ubar (3), dalpha / dbeta / dgamma dots (6), dC, dB, dX (6R).
    The checkpoint recomputation the kernels add is not counted."""
    R = w.rank
    per_elem = (8 + 2 * R) + (18 + 8 * R)
    return float(per_elem) * w.dstate * w.headdim * w.batch * w.seqlen * w.heads


def bwd_bytes(w: synth.Workload) -> int:
    """x, B, C, dy, dt, lambda, omega read once; dx, dB, dC, ddt, dlambda, domega written once (fp32)."""
    e = io_bytes(w.io)
    R, P, N = w.rank, w.headdim, w.dstate
    per_ht = (2 * R * P + 2 * R * N) * e + 8 + (N // 2) * 4 + (R * P + 2 * R * N) * 4 + 8 + (N // 2) * 4
    return per_ht * w.batch * w.seqlen * w.heads + 8 * w.heads


def decode_bytes(b: int, H: int, P: int, N: int, R: int, io: str = "bf16") -> int:
    """State read + write (fp32), inputs and cache read, cache and y written."""
    e = io_bytes(io)
    per = 8 * N * P + (R * P + 2 * R * N) * e + (N // 2) * 4 + 8 + 2 * R * (N + P) * e + R * P * e
    return b * H * per + H * 4


def profiled_traffic(kernel_source: str, profile: str):
    """DRAM bytes per call (dram__bytes_read.sum + dram__bytes_write.sum summed over the call's
    launches of the kernel; one launch when the call has one) that an ncu capture recorded in
    ``profile`` (a summary under profiles/), or None when the kernel source has changed since:
    the summary names the source file's sha256 at capture time."""
    import hashlib
    try:
        src = open(os.path.join(ROOT, kernel_source), "rb").read()
        text = open(os.path.join(ROOT, "profiles", profile)).read()
    except OSError:
        return None
    digest = hashlib.sha256(src).hexdigest()
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.lstrip("-* ").split(":", 1)[0].strip() in ("source sha256", "traffic per call bytes"):
            k, v = line.lstrip("-* ").split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source sha256") != digest:
        return None
    try:
        return int(fields["traffic per call bytes"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
class ClockSampler:
    """Samples SM clocks and clock-event (throttle) reasons with nvidia-smi while
    the timed work runs (read only; changes no setting)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        self.idx = device_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.error = None

    def __enter__(self):
        import subprocess
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as exc:
            self.error = str(exc)
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if self.error or not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"no clock samples ({self.error})"]}
        samples = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                samples.append((float(f[0]), float(f[1]), float(f[2]), int(f[3], 16), f[4:8]))
            except Exception:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed clock samples"]}
        loaded = [x for x in samples if x[2] > 250.0] or samples     # under load: power above idle
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for x in loaded for n, v in zip(names, x[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(x[0] for x in loaded), "sm_max_mhz": max(x[1] for x in samples),
                "reasons": reasons, "samples": len(samples), "samples_under_load": len(loaded),
                "power_w_max": max(x[2] for x in samples)}


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
def _time_calls(call, stream, steps, warmup, dist, device):
    """W untimed calls, then K timed calls between a barrier and a synchronize on both
    sides: (total seconds max over ranks, per-call event ms list)."""
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
    return max_over_ranks(dist, total_ms, device) / 1e3, per


def prefill_leg(binding, w, d, args, stream, dist, device, local, pk, ws, rank, steps=None, cpu=True):
    """One prefill workload, device resident: Mtok/s, the roofline of the call (algorithmic bytes over
    its event-timed duration; DRAM traffic per launch of the dominant kernel from the committed ncu
    summary while the kernel source is unchanged), launches, clocks and the oracle on the host cores.
    Returns (entry, (y, final_state))."""
    steps = steps or args.steps
    path, launches = binding.m3_scan_fwd_plan(w.batch, w.seqlen, w.heads, w.headdim, w.dstate, w.rank, w.chunk,
                                              binding.io_code(d["x"].dtype))
    with ClockSampler(local) as clk:
        sec, per_ms, out = time_prefill(binding, w, d, stream, steps, args.warmup, dist, device)
    tokens = w.batch * w.seqlen * ws
    avg_call_ms = sum(per_ms) / len(per_ms)
    nbytes = prefill_bytes(w)
    achieved = nbytes / (avg_call_ms * 1e-3) / 1e9
    tflops = prefill_tc_flops(w) / (avg_call_ms * 1e-3) / 1e12
    src = "state_space_sequence_04_b300/csrc/" + ("scan_tc.cu" if path == 1 else "scan_simt.cu")
    ent = {
        "value": tokens * steps / sec / 1e6, "unit": "Mtok/s", "steps": steps,
        "ms_per_step": sec / steps * 1e3,
        "dtype": "bf16" if path == 1 else "f32",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "heads": w.heads,
                   "headdim": w.headdim, "dstate": w.dstate, "rank": w.rank, "chunk": w.chunk, "io": w.io,
                   "l2": (f"inputs larger than L2 ({nbytes / 1e9:.2f} GB per step), no flush" if nbytes > 126e6
                          else f"inputs ({nbytes / 1e6:.2f} MB) fit in L2: a tiny check, not a bandwidth figure")},
        "gpu_launches": launches * steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"],
                     # the committed ncu summary of this workload's dominant kernel (only for the named sizes)
                     "traffic": (profiled_traffic(src, f"{src.rsplit('/', 1)[1][:-3]}_{w.name}.md")
                                 if synth.WORKLOADS.get(w.name) == w else None),
                     "traffic_scope": "ncu DRAM read + write bytes per call, over all its launches",
                     "kernel": "m3_scan_fwd (" + ("tensor-core" if path == 1 else "CUDA-core") +
                               f" path, {launches} launches per call)",
                     "algorithmic_bytes_per_call": nbytes, "peak_source": pk["source"],
                     "tc_tflops": tflops, "tc_frac_of_bf16_peak": tflops / pk["bf16_tflops"]},
    }
    ent["clocks"] = clk.summary()
    if cpu and rank == 0 and ws == 1:
        v, threads, sample, el = cpu_baseline_run(w, d)
        ent["cpu_baseline"] = {"value": v, "unit": "Mtok/s", "cores": threads, "kind": "oracle",
                               "sample": sample, "seconds": el}
    return ent, out


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

    sec, per = _time_calls(call, stream, steps, warmup, dist, device)
    return sec, per, (y, fin)


PREP_KEYS = ("x", "B", "C", "dt_raw", "A", "u", "omega")


def time_prefill_prep(binding, w, dp, stream, steps, warmup, dist, device, bc=None, z=None):
    """The same over m3_scan_fwd_prep (pre-activations, one decay generator per token; ``bc``:
    the B / C normalisation and channel biases, device tensors)."""
    y = torch.empty_like(dp["x"])
    fin = torch.empty((w.batch, w.heads, w.dstate, w.headdim), dtype=torch.float32, device=device)
    ws = binding.alloc_workspace_prep(dp["x"].shape, w.dstate, w.rank, w.chunk, dp["x"].dtype, device)
    args = [dp[k] for k in PREP_KEYS]
    params = binding.prep_params(dp["dt_bias"], bc, z)

    def call():
        st = binding.m3_scan_fwd_prep(*args, w.rank, w.chunk, y, fin, ws, params, stream)
        if st != 0:
            raise binding.M3Error(st, "m3_scan_fwd_prep")

    return _time_calls(call, stream, steps, warmup, dist, device)


def time_backward(binding, w, d, stream, steps, warmup, dist, device, seed=0):
    """m3_scan_bwd on the prefill workload's inputs with a random dy (io dtype); device resident."""
    gen = torch.Generator(device=device).manual_seed(1000 + seed)
    dy = torch.randn(d["x"].shape, generator=gen, device=device).to(d["x"].dtype)
    f = dict(dtype=torch.float32, device=device)
    grads = {"dx": torch.empty(d["x"].shape, **f), "dB": torch.empty(d["B"].shape, **f),
             "dC": torch.empty(d["C"].shape, **f), "ddt": torch.empty(d["dt"].shape, **f),
             "dA": torch.empty(d["A"].shape, **f), "dlam": torch.empty(d["lam"].shape, **f),
             "domega": torch.empty(d["omega"].shape, **f)}
    nbytes = binding.m3_scan_bwd_workspace_size(w.batch, w.seqlen, w.heads, w.headdim, w.dstate, w.rank,
                                                binding.io_code(d["x"].dtype))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    args = [d[k] for k in KEYS]

    def call():
        st = binding.m3_scan_bwd(*args, w.rank, dy, None, grads, ws, stream)
        if st != 0:
            raise binding.M3Error(st, "m3_scan_bwd")

    sec, per = _time_calls(call, stream, steps, warmup, dist, device)
    del grads, ws, dy
    return sec, per


def time_backward_prep(binding, w, stream, steps, warmup, dist, device, seed=0, gate=False):
    """m3_scan_bwd_prep on the workload's pre-activation inputs (dt_bias set) with a random dy; ``gate``:
    through the output gate as well (its z drawn like the forward leg's)."""
    dp = synth.make_prep_inputs(w, seed=seed, device=device)
    z = synth.make_gate(tuple(dp["x"].shape), io=w.io, seed=seed, device=device) if gate else None
    gen = torch.Generator(device=device).manual_seed(2000 + seed)
    dy = torch.randn(dp["x"].shape, generator=gen, device=device).to(dp["x"].dtype)
    f = dict(dtype=torch.float32, device=device)
    grads = {"dx": torch.empty(dp["x"].shape, **f), "dB": torch.empty(dp["B"].shape, **f),
             "dC": torch.empty(dp["C"].shape, **f), "ddt_raw": torch.empty(dp["dt_raw"].shape, **f),
             "dA": torch.empty(dp["A"].shape, **f), "du": torch.empty(dp["u"].shape, **f),
             "domega": torch.empty(dp["omega"].shape, **f), "ddt_bias": torch.empty((w.heads,), **f),
             "dz": torch.empty(dp["x"].shape, **f) if gate else None}
    nbytes = binding.m3_scan_bwd_prep_workspace_size(w.batch, w.seqlen, w.heads, w.headdim, w.dstate, w.rank,
                                                     binding.io_code(dp["x"].dtype))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    params = binding.prep_params(dp["dt_bias"], None, z)
    args = [dp[k] for k in ("x", "B", "C", "dt_raw", "A", "u", "omega")]

    def call():
        st = binding.m3_scan_bwd_prep(*args, w.rank, dy, None, grads, ws, params, stream)
        if st != 0:
            raise binding.M3Error(st, "m3_scan_bwd_prep")

    sec, per = _time_calls(call, stream, steps, warmup, dist, device)
    del grads, ws, dy, dp, z
    return sec, per


def time_prefill_e2e(binding, w, host, stream, steps, warmup, dist, device, copy_streams=4):
    """End to end through the C ABI: every step copies its inputs from pinned host
    buffers to the device, runs m3_scan_fwd and copies y and the final state back to
    pinned host buffers, all inside the timed region.  Steps are pipelined over two
    device input/output buffer sets: the inputs of step k+1 are copied (split over
    ``copy_streams`` streams so that several copy engines share them) while step k
    computes and its results are copied out.  The region ends when the last step's
    results are on the host."""
    sets = []
    for _ in range(2):
        dev = {k: torch.empty_like(host[k], device=device) for k in KEYS}
        y = torch.empty_like(dev["x"])
        fin = torch.empty((w.batch, w.heads, w.dstate, w.headdim), dtype=torch.float32, device=device)
        sets.append((dev, y, fin))
    y_h = [torch.empty_like(sets[0][1], device="cpu").pin_memory() for _ in range(2)]
    fin_h = [torch.empty_like(sets[0][2], device="cpu").pin_memory() for _ in range(2)]
    ws = binding.alloc_workspace(sets[0][0]["x"].shape, w.dstate, w.rank, w.chunk, sets[0][0]["x"].dtype, device)
    h2d = sum(host[k].numel() * host[k].element_size() for k in KEYS)
    d2h = sets[0][1].numel() * sets[0][1].element_size() + sets[0][2].numel() * sets[0][2].element_size()
    cps = [torch.cuda.Stream(device=device) for _ in range(copy_streams)]
    outs = torch.cuda.Stream(device=device)
    # the big tensors first, spread over the copy streams (largest remaining to the least loaded)
    order = sorted(KEYS, key=lambda k: -host[k].numel() * host[k].element_size())

    computed = [None, None]   # per set: its last compute (its inputs are free after it)
    copied_out = [None, None]  # per set: its last results copied to the host

    def step(j):
        dev, y, fin = sets[j & 1]
        load = [0] * len(cps)
        done = []
        for k in order:
            i = load.index(min(load))
            cs = cps[i]
            if computed[j & 1] is not None:
                cs.wait_event(computed[j & 1])   # step j-2 has read this set's inputs
            with torch.cuda.stream(cs):
                dev[k].copy_(host[k], non_blocking=True)
            load[i] += host[k].numel() * host[k].element_size()
            ev = torch.cuda.Event()
            ev.record(cs)
            done.append(ev)
        for ev in done:
            stream.wait_event(ev)
        if copied_out[j & 1] is not None:
            stream.wait_event(copied_out[j & 1])  # step j-2's results have left this set
        st = binding.m3_scan_fwd(*[dev[k] for k in KEYS], w.rank, w.chunk, y, fin, ws, stream)
        if st != 0:
            raise binding.M3Error(st, "m3_scan_fwd")
        ev = torch.cuda.Event()
        ev.record(stream)
        computed[j & 1] = ev
        outs.wait_event(ev)
        with torch.cuda.stream(outs):
            y_h[j & 1].copy_(y, non_blocking=True)
            fin_h[j & 1].copy_(fin, non_blocking=True)
        ev2 = torch.cuda.Event()
        ev2.record(outs)
        copied_out[j & 1] = ev2

    for j in range(warmup):
        step(j)
    torch.cuda.synchronize()
    barrier(dist)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s_ in cps + [outs]:
        s_.wait_stream(stream)               # nothing of the region starts before t0
    for j in range(steps):
        step(j)
    stream.wait_stream(outs)
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
    torch.cuda.synchronize()          # inputs were drawn on the default stream
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
    eager = t0.elapsed_time(t1) / 1e3
    # the same carried steps replayed from a CUDA graph of `ring` calls (no host launch cost)
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(ring):
                call(i)
        torch.cuda.synchronize()
        reps = max(1, steps // ring)
        with torch.cuda.stream(stream):      # replay on the stream the events are recorded on
            g.replay()
            torch.cuda.synchronize()
            t0.record(stream)
            for _ in range(reps):
                g.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        graph = t0.elapsed_time(t1) / 1e3 / (reps * ring) * steps
    except Exception as exc:  # report, do not hide
        graph = f"graph capture failed: {exc}"
    ok = bool(torch.isfinite(state).all())
    return eager, graph, ok


def decode_after_prefill(binding, w, d, y_fin, stream, device, pk, steps=256):
    """``steps`` carried decode calls continuing the prefill (its final state and delayed-write cache),
    per-step inputs of the workload's distributions; steps/s and the HBM roofline of a step."""
    _, fin = y_fin
    H, P, N, R = w.heads, w.headdim, w.dstate, w.rank
    state = fin.clone()
    cache = binding.cache_from_prefill(d["B"], d["x"])
    ins = synth.make_decode_steps(w.batch, H, P, N, R, steps, io=w.io, seed=7, device=device, dt_mu=w.dt_mu,
                                  dt_sd=w.dt_sd, lam_uniform=w.lam_uniform, A=d["A"])
    y_t = torch.empty((w.batch, H, R, P), dtype=d["x"].dtype, device=device)
    per = [[ins[k][i] for k in ("x", "B", "C", "dt", "lam", "omega")] for i in range(steps)]
    torch.cuda.synchronize()

    def run(lo, hi):
        for i in range(lo, hi):
            a = per[i]
            st = binding.m3_decode_step(state, a[0], a[1], cache, a[2], a[3], d["A"], a[4], a[5], y_t, R, stream)
            if st != 0:
                raise binding.M3Error(st, "m3_decode_step")

    # the 256 carried steps are captured once in a CUDA graph (as a serving loop would replay them) from a
    # copy of the starting state and cache, then replayed from the prefill's own state and cache
    state0, cache0 = state.clone(), cache.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run(0, steps)
    torch.cuda.synchronize()
    state.copy_(state0)
    cache.copy_(cache0)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    sec = t0.elapsed_time(t1) / 1e3
    nbytes = decode_bytes(w.batch, H, P, N, R, w.io)
    per_step = sec / steps
    return {"steps": steps, "unit": "steps/s", "steps_per_s": 1.0 / per_step, "us_per_step": per_step * 1e6,
            "bytes_per_step": nbytes, "achieved_gbs": nbytes / per_step / 1e9, "launch": "CUDA graph of the steps",
            "note": "batch 1: the 2.1 MB state stays in L2 between steps; launch-bound, not an HBM figure",
            "finite": bool(torch.isfinite(state).all()), "gpu_launches": steps}


def decode_cpu_baseline(b=64, R=1, target_s=10.0, max_steps=1024):
    """The float64 oracle's decode step (OpenMP over (batch, head)) at batch b, rank R, H=64, P=64, N=128
    on this host's cores: carried steps until ``target_s`` seconds or ``max_steps`` steps."""
    import oracle
    H, P, N = 64, 64, 128
    state = synth.make_decode_state(b, H, N, P, seed=0)
    ins = synth.make_decode_steps(b, H, P, N, R, 4, io="bf16", seed=1)
    h = oracle.f64(state)
    prev = np.zeros((b, H, R * (N + P)))
    el, n = 0.0, 0
    while el < target_s and n < max_steps:
        i = n % 4
        t0 = time.perf_counter()
        _, h, prev = oracle.decode_step(h, ins["x"][i], ins["B"][i], prev, ins["C"][i], ins["dt"][i], ins["A"],
                                        ins["lam"][i], ins["omega"][i])
        el += time.perf_counter() - t0
        n += 1
    return {"value": n / el, "unit": "steps/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} carried steps at batch {b}, R={R}, 64 heads, P=64, N=128, float64", "seconds": el}


def decode_sweep(binding, args, stream, device, pk):
    dec = {}
    ranks = synth.DECODE_RANKS if args.decode_rank is None else (args.decode_rank,)
    batches = synth.DECODE_BATCHES if args.decode_batch is None else (args.decode_batch,)
    for R in ranks:
        for b in batches:
            esec, gsec, ok = time_decode(binding, b, R, stream, device, steps=args.decode_steps)
            nbytes = decode_bytes(b, 64, 64, 128, R)
            ent = {"bytes_per_step": nbytes, "finite": ok}
            for tag, sec in (("eager", esec), ("graph", gsec)):
                if not isinstance(sec, float):
                    ent[tag] = sec
                    continue
                per_step = sec / args.decode_steps
                gbs = nbytes / per_step / 1e9
                ent[tag] = {"steps_per_s": 1.0 / per_step, "us_per_step": per_step * 1e6,
                            "tokens_per_s": b / per_step, "achieved_gbs": gbs,
                            "frac_of_measured_hbm": gbs / pk["hbm_gbs"], "frac_of_8tbs": gbs / 8000.0}
            dec[f"b{b}_R{R}"] = ent
    return {"unit": "steps/s", "steps": args.decode_steps, "heads": 64, "headdim": 64, "dstate": 128,
            "sweep": dec}


# ---------------------------------------------------------------------------
def _oracle_sample(inp, w, n):
    """The first n (batch, head) sequences of the workload, stacked as heads of one
    batch-1 problem (float64 numpy), in the oracle's argument order."""
    import numpy as np
    import oracle
    pairs = [(b, h) for b in range(w.batch) for h in range(w.heads)][:n]
    cols = []
    for i, key in enumerate(KEYS):
        if key == "A":
            cols.append(np.array([float(inp["A"][h]) for _, h in pairs]))
        else:
            cols.append(np.concatenate([oracle.f64(inp[key][b:b + 1, :, h:h + 1]) for b, h in pairs], axis=2))
    return cols


def cpu_baseline_run(w, inp, target_s: float = 10.0, max_s: float = 30.0):
    """Time the float64 oracle on a bounded sample of the workload: whole sequences
    (one (batch, head) of T tokens each), doubling the sample from one per thread
    until one run takes >= target_s or the whole workload is covered.
    ``inp`` are the benchmark's own inputs (on any device); the sampled sequences
    are copied to the host.  Returns (Mtok/s, threads, sample description, seconds)."""
    import oracle
    threads = oracle.num_threads()
    total = w.batch * w.heads
    n = max(1, min(total, threads))
    while True:
        a = _oracle_sample(inp, w, n)
        t0 = time.perf_counter()
        oracle.scan(*a)
        el = time.perf_counter() - t0
        if el >= target_s or n >= total or el * 2 > max_s:
            break
        n = min(total, n * 2)
    runs = 1
    while el < target_s and el * (runs + 1) / runs <= max_s:   # whole workload is quick: repeat it
        t0 = time.perf_counter()
        oracle.scan(*a)
        el += time.perf_counter() - t0
        runs += 1
    tokens = n * w.seqlen / w.heads * runs   # token-equivalents (a token covers all heads)
    sample = f"{n} of {total} (batch, head) sequences x {w.seqlen} tokens, float64, {runs} run(s)"
    return tokens / el / 1e6, threads, sample, el


def run_reference(args):
    """--impl reference: the float64 oracle timed as it stands on the host cores."""
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = synth.WORKLOADS[args.workload]
    threads = oracle.num_threads()
    inp = synth.make_inputs(w, seed=0, batch=1)      # batch row 0 on the host
    n = max(1, min(w.heads, threads))
    a = _oracle_sample(inp, w, n)
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


def backward_leg(binding, w, d, args, stream, dist, device, local, ws, rank):
    """The backward pass (training) on the prefill inputs: three launches per call (the adjoint
    kernel over (batch*head, pair block), the dX and the per-token scalar finishing kernels)."""
    bsteps = max(3, args.steps // 4)
    with ClockSampler(local) as bclk:
        bsec, bper = time_backward(binding, w, d, stream, bsteps, args.warmup, dist, device, seed=rank)
    bms = sum(bper) / len(bper)
    fl, by = bwd_flops(w), bwd_bytes(w)
    pk = peaks()
    out = {
        "value": w.batch * w.seqlen * ws * bsteps / bsec / 1e6, "unit": "Mtok/s", "steps": bsteps,
        "ms_per_step": bsec / bsteps * 1e3, "entry": "m3_scan_bwd", "gpu_launches": 3 * bsteps,
        "config": {"batch": w.batch, "seqlen": w.seqlen, "heads": w.heads, "headdim": w.headdim,
                   "dstate": w.dstate, "rank": w.rank, "io": w.io},
        "roofline": {"bound": "alu", "achieved": fl / (bms * 1e-3) / 1e12, "peak": FP32_ALU_TFLOPS,
                     "unit": "TFLOP/s", "frac": fl / (bms * 1e-3) / 1e12 / FP32_ALU_TFLOPS,
                     "peak_source": "148 SMs x 128 FP32 lanes x 2 x 2032 MHz", "flops_per_call": fl},
        "algorithmic_bytes_per_call": by, "hbm_frac": by / (bms * 1e-3) / 1e9 / pk["hbm_gbs"],
        "clocks": bclk.summary()}
    # the same through m3_scan_bwd_prep (pre-activations with dt_bias, A per token): one more launch
    # (Delta, lambda) and the chain rule through softplus / sigmoid in the scalar finishing kernel
    psec, pper = time_backward_prep(binding, w, stream, bsteps, args.warmup, dist, device, seed=rank)
    pms = sum(pper) / len(pper)
    out["prep"] = {"value": w.batch * w.seqlen * ws * bsteps / psec / 1e6, "unit": "Mtok/s",
                   "ms_per_step": psec / bsteps * 1e3, "entry": "m3_scan_bwd_prep", "gpu_launches": 4 * bsteps,
                   "roofline_frac": fl / (pms * 1e-3) / 1e12 / FP32_ALU_TFLOPS}
    # and through the output gate: one ungated forward launch for y_pre, z staged with dy, one dz launch
    gsec, gper = time_backward_prep(binding, w, stream, bsteps, args.warmup, dist, device, seed=rank, gate=True)
    path, flaunch = binding.m3_scan_fwd_plan(w.batch, w.seqlen, w.heads, w.headdim, w.dstate, w.rank, 64,
                                             binding.io_code(d["x"].dtype))
    out["prep"]["with_gate"] = {"value": w.batch * w.seqlen * ws * bsteps / gsec / 1e6, "unit": "Mtok/s",
                                "ms_per_step": gsec / bsteps * 1e3,
                                # Delta/lambda, the ungated forward, the adjoint, dz, the two finishing kernels
                                "gpu_launches": (5 + flaunch) * bsteps}
    return out


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
    ap.add_argument("--no-prep", action="store_true", help="skip the pre-activation prefill measurement")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward-pass measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the tiny, MIMO and long-context prefill workloads")
    ap.add_argument("--workload", default=synth.SISO_1P5B.name, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mode", choices=["all", "decode", "bwd"], default="all",
                    help="decode: only the decode sweep (restricted by --decode-batch/--decode-rank); "
                         "bwd: only the backward pass (sizes overridable by --bwd-batch/--bwd-seqlen)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (a smaller case of the same shape, e.g. for a profiler)")
    ap.add_argument("--seqlen", type=int, default=None, help="override the workload's sequence length")
    ap.add_argument("--bwd-batch", type=int, default=None)
    ap.add_argument("--bwd-seqlen", type=int, default=None)
    ap.add_argument("--decode-batch", type=int, default=None)
    ap.add_argument("--decode-rank", type=int, default=None)
    ap.add_argument("--decode-steps", type=int, default=synth.DECODE_STEPS)
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
    if args.batch or args.seqlen:
        w = dataclasses.replace(w, batch=args.batch or w.batch, seqlen=args.seqlen or w.seqlen)
    stream = torch.cuda.Stream(device=device)

    if args.mode == "decode":
        line = {"metric": METRIC, "mode": "decode",
                "decode": decode_sweep(binding, args, stream, device, pk)}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0

    if args.mode == "bwd":
        wb = dataclasses.replace(w, batch=args.bwd_batch or w.batch, seqlen=args.bwd_seqlen or w.seqlen)
        db = synth.make_inputs(wb, seed=rank, device=device)
        line = {"metric": METRIC, "mode": "bwd", "workload": w.name,
                "backward": backward_leg(binding, wb, db, args, stream, dist, device, local, ws, rank)}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0

    # every rank draws its own replica of the workload (seeded by rank)
    d = synth.make_inputs(w, seed=rank, device=device)
    torch.cuda.synchronize()
    head, _ = prefill_leg(binding, w, d, args, stream, dist, device, local, pk, ws, rank,
                          cpu=not args.no_cpu_baseline)
    tokens = w.batch * w.seqlen * ws                  # per step, all ranks
    path, launches = binding.m3_scan_fwd_plan(w.batch, w.seqlen, w.heads, w.headdim, w.dstate, w.rank, w.chunk,
                                              binding.io_code(d["x"].dtype))
    line = {
        "metric": METRIC, "value": head["value"], "unit": "Mtok/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
        "config": dict(head["config"], parallelism=f"replicas x{ws} (independent (batch, head) sequences, "
                                                   "no collective)"),
        "gpu_launches": head["gpu_launches"], "roofline": head["roofline"], "clocks": head["clocks"],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]

    if not args.no_prep:
        # the same workload through m3_scan_fwd_prep: Delta, lambda from pre-activations and one
        # decay generator per token, derived inside the kernels
        dp = {k: v for k, v in synth.make_prep_inputs(w, seed=rank, device=device).items()
              if k in PREP_KEYS or k == "dt_bias"}
        psec, pper = time_prefill_prep(binding, w, dp, stream, args.steps, args.warmup, dist, device)
        pms = sum(pper) / len(pper)
        pbytes = prefill_prep_bytes(w)
        line["prefill_prep"] = {
            "value": tokens * args.steps / psec / 1e6, "unit": "Mtok/s", "ms_per_step": psec / args.steps * 1e3,
            "entry": "m3_scan_fwd_prep", "algorithmic_bytes_per_call": pbytes,
            "roofline": {"bound": "hbm", "achieved": pbytes / (pms * 1e-3) / 1e9, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": pbytes / (pms * 1e-3) / 1e9 / pk["hbm_gbs"]},
            # the CUDA-core path derives Delta and lambda in one extra elementwise launch
            "gpu_launches": (launches + (1 if path == 0 else 0)) * args.steps}
        # and with the B / C RMS normalisation, gains and head-specific channel biases
        bc = {k: (v.to(device) if hasattr(v, "shape") else v)
              for k, v in synth.make_bc_params(w.heads, w.rank, w.dstate).items()}
        bsec, bper = time_prefill_prep(binding, w, dp, stream, args.steps, args.warmup, dist, device, bc=bc)
        bms = sum(bper) / len(bper)
        line["prefill_prep"]["with_bc_norm"] = {
            "value": tokens * args.steps / bsec / 1e6, "unit": "Mtok/s", "ms_per_step": bsec / args.steps * 1e3,
            "roofline_frac": pbytes / (bms * 1e-3) / 1e9 / pk["hbm_gbs"]}
        # and with the output gate as well (the SSM + rotary + gate fusion level); z is read once
        z = synth.make_gate(tuple(dp["x"].shape), io=w.io, seed=rank, device=device)
        gsec, gper = time_prefill_prep(binding, w, dp, stream, args.steps, args.warmup, dist, device, bc=bc, z=z)
        gms = sum(gper) / len(gper)
        gbytes = pbytes + z.numel() * z.element_size()
        line["prefill_prep"]["with_bc_norm_and_gate"] = {
            "value": tokens * args.steps / gsec / 1e6, "unit": "Mtok/s", "ms_per_step": gsec / args.steps * 1e3,
            "algorithmic_bytes_per_call": gbytes, "roofline_frac": gbytes / (gms * 1e-3) / 1e9 / pk["hbm_gbs"]}
        del dp, bc, z

    if not args.no_bwd:
        line["backward"] = backward_leg(binding, w, d, args, stream, dist, device, local, ws, rank)

    if not args.no_e2e:
        host = {k: d[k].to("cpu").pin_memory() for k in KEYS}
        esec, h2d, d2h = time_prefill_e2e(binding, w, host, stream, max(3, args.steps // 4), 3, dist, device)
        line["e2e"] = {"value": tokens / (esec / max(3, args.steps // 4)) / 1e6, "unit": "Mtok/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        del host

    if not args.no_decode and rank == 0:
        line["decode"] = decode_sweep(binding, args, stream, device, pk)
        if not args.no_cpu_baseline and ws == 1:
            line["decode"]["cpu_baseline"] = decode_cpu_baseline()

    if not args.no_workloads:
        # the other prefill workloads, each a complete leg (every rank its own replica)
        del d
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for wn in (synth.TINY, synth.MIMO_R4, synth.LONG_MIMO):
            if wn.name == w.name:
                continue
            dn = synth.make_inputs(wn, seed=rank, device=device)
            torch.cuda.synchronize()
            ent, out = prefill_leg(binding, wn, dn, args, stream, dist, device, local, pk, ws, rank,
                                   cpu=not args.no_cpu_baseline)
            if wn is synth.LONG_MIMO and rank == 0:
                ent["decode_after"] = decode_after_prefill(binding, wn, dn, out, stream, device, pk)
            line["workloads"][wn.name] = ent
            del dn, out
            torch.cuda.empty_cache()

    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
