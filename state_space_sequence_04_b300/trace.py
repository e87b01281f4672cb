"""Phase trace of the tensor-core prefill kernel (a diagnostic, not part of the product path).

Builds libm3_trace.so -- the library compiled with -DM3_TRACE, in which the
prefill kernel records clock64 at the phase boundaries of the first chunks of
each CTA, and the start and end clocks and the SM of every CTA -- runs one
m3_scan_fwd call on a workload after warm-up calls, and prints the spread of
CTA durations by how many CTAs their SM ran, and, for the CTAs that share
their SM with another (those set the call's time), the median cycles each
phase of each warp group takes and the chunk period, plus the tensor-pipe rate
inside two of the chunk's MMA batches measured in place: the chunk-state GEMM
H += B''^T X (issue by thread 0 right after the group barrier, completion seen
by a consumer thread spinning on its commit barrier) and the intra-chunk
output GEMM Y = SL X (likewise).  A batch's rate is its executed FLOPs over
its issue-to-completion cycles, against the SM's share of the measured dense
bf16 peak at the traced clock.

    python -m state_space_sequence_04_b300.trace [--workload NAME] [--json PATH]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from state_space_sequence_04_b300 import binding, build, synth  # noqa: E402

CTAS, CHUNKS, SLOTS = 512, 32, 32        # kTraceCtas, kTraceChunks, kTraceSlots of the kernel
CLK_CTAS, CLK_SLOTS = 4096, 6            # kClkCtas, kClkSlots: per CTA (t0 ns, clk0, t1 ns, clk1, SM id, -)
SMS = 148
KEYS = ("x", "B", "C", "dt", "A", "lam", "omega")
# slot names: consumer thread 0 (0-9, in the time order below), observers (11, 12), rotate thread 128 (16-24)
# (the state step runs at the top of a chunk with R >= 2 (slots 8 -> 9), at the end with R = 1 (14 -> 15))
CONSUMER = [(0, "top"), (8, "stage ready (rot_done)"), (9, "state step, R >= 2"), (1, "barrier"),
            (2, "H+= and Yi issued"), (3, "S and H+= waited"), (4, "mask + barrier"), (5, "Y issued (+ next S)"),
            (6, "Y waited"), (7, "output stored"), (14, "R = 1: Hb written, next coefficients waited"),
            (15, "R = 1: H scaled")]
ROTATE = ["top", "dt/lambda boxes", "coefficients + angle partial sums", "C/B landed", "rotation (C~, B'')",
          "barrier + next boxes issued", "-", "-", "barrier"]


def peak_bf16_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1800.0, "fallback"


PREP_KEYS = ("x", "B", "C", "dt_raw", "A", "u", "omega")
ENTRIES = ("plain", "prep", "prep_bc", "prep_bc_gate")


def run(wname: str, entry: str = "plain"):
    lib_path = build.build(trace=True)
    binding.LIB_PATH = lib_path
    lib = binding.load()
    lib.m3_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.m3_trace_read.restype = ctypes.c_int
    n = CTAS * CHUNKS * SLOTS + CLK_CTAS * CLK_SLOTS
    w = synth.WORKLOADS[wname]
    if entry == "plain":
        d = synth.make_inputs(w, seed=0, device="cuda")
        args = [d[k] for k in KEYS]
    else:   # m3_scan_fwd_prep: pre-activations, optionally the B / C normalisation and the gate
        d = synth.make_prep_inputs(w, seed=0, device="cuda")
        args = [d[k] for k in PREP_KEYS]
        bc = None if entry == "prep" else {k: (v.to("cuda") if hasattr(v, "shape") else v)
                                           for k, v in synth.make_bc_params(w.heads, w.rank, w.dstate).items()}
        z = synth.make_gate(tuple(d["x"].shape), io=w.io, seed=0, device="cuda") if entry == "prep_bc_gate" else None
        params = binding.prep_params(d["dt_bias"], bc, z)
    path, launches = binding.m3_scan_fwd_plan(w.batch, w.seqlen, w.heads, w.headdim, w.dstate, w.rank, w.chunk,
                                              binding.io_code(d["x"].dtype))
    if path != 1:
        raise SystemExit(f"{wname} does not take the tensor-core path")
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.batch, w.heads, w.dstate, w.headdim), dtype=torch.float32, device="cuda")
    if entry == "plain":
        ws = binding.alloc_workspace(d["x"].shape, w.dstate, w.rank, w.chunk, d["x"].dtype, "cuda")

        def call():
            binding._check(binding.m3_scan_fwd(*args, w.rank, w.chunk, y, fin, ws), "m3_scan_fwd")
    else:
        ws = binding.alloc_workspace_prep(d["x"].shape, w.dstate, w.rank, w.chunk, d["x"].dtype, "cuda")

        def call():
            binding._check(binding.m3_scan_fwd_prep(*args, w.rank, w.chunk, y, fin, ws, params), "m3_scan_fwd_prep")
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    binding._check(lib.m3_trace_read(None, n), "m3_trace_read")
    call()
    torch.cuda.synchronize()
    buf = (ctypes.c_longlong * n)()
    binding._check(lib.m3_trace_read(ctypes.addressof(buf), n), "m3_trace_read")
    tr = list(buf)
    clk = tr[CTAS * CHUNKS * SLOTS:]
    cta = [clk[k * CLK_SLOTS:(k + 1) * CLK_SLOTS] for k in range(CLK_CTAS)]
    ran_idx = [k for k, c in enumerate(cta) if c[2] > c[0] > 0]
    ran = [cta[k] for k in ran_idx]
    # cycles per ns from the CTAs' (globaltimer, clock64) pairs
    ghz = statistics.median((c[3] - c[1]) / (c[2] - c[0]) for c in ran[:CTAS])
    # CTA durations of the last launch of the call, by how many of its CTAs shared the SM
    t0 = min(c[0] for c in ran)
    per_sm = {}
    for c in ran:
        per_sm.setdefault(c[4], []).append(c)
    spread = {}
    for k in sorted({len(v) for v in per_sm.values()}):
        d = [(c[2] - c[0]) / 1e3 for v in per_sm.values() if len(v) == k for c in v]
        e = [(c[2] - t0) / 1e3 for v in per_sm.values() if len(v) == k for c in v]
        spread[f"{k}_per_sm"] = {"sms": sum(1 for v in per_sm.values() if len(v) == k), "ctas": len(d),
                                 "duration_us_min_med_max": [min(d), statistics.median(d), max(d)],
                                 "end_us_max": max(e)}
    pair_gap = [abs((v[0][2] - v[0][0]) - (v[1][2] - v[1][0])) / 1e3 for v in per_sm.values() if len(v) == 2]
    # the phases are taken from CTAs that share their SM with another: those set the call's time
    load = {k: len(per_sm[cta[k][4]]) for k in ran_idx}
    most = max(load.values())
    traced = [k for k in ran_idx if k < CTAS and load[k] == most]

    def at(cta, i, slot):
        return tr[(cta * CHUNKS + i) * SLOTS + slot]

    # the last launch of the call (the full pass) is the one traced last: its values overwrite the state pass's
    QR, P, N = 64, w.headdim, w.dstate   # every chunk runs as 64-row sub-chunks (64 / R tokens)
    MM = 64
    out = {"workload": wname, "entry": entry, "launches_per_call": launches, "sm_ghz_traced": ghz, "consumer": {}, "rotate": {},
           "ctas": {"count": len(ran), "span_us": (max(c[2] for c in ran) - t0) / 1e3, "by_sm_load": spread,
                    "pair_duration_gap_us_median": statistics.median(pair_gap) if pair_gap else None}}
    out["ctas"]["phases_from"] = f"{len(traced)} CTAs on SMs running {most} CTAs, first {CHUNKS} chunks each"
    # every CTA of the launch: (start us, duration us, SM), by block index
    out["ctas"]["per_cta"] = [[(cta[k][0] - t0) / 1e3, (cta[k][2] - cta[k][0]) / 1e3, cta[k][4]] for k in ran_idx]
    nchunk = {}
    for c in traced:
        k = 0
        while k < CHUNKS and at(c, k, 0) != 0 and at(c, k, 9) != 0:
            k += 1
        nchunk[c] = k
    use = [(c, i) for c in traced for i in range(1, nchunk[c] - 1)]
    if not use:
        raise SystemExit("no traced chunks")
    for j in range(1, len(CONSUMER)):
        (a, _), (b, name) = CONSUMER[j - 1], CONSUMER[j]
        dts = [at(c, i, b) - at(c, i, a) for c, i in use if at(c, i, b) and at(c, i, a)]
        out["consumer"][name] = statistics.median(dts) if dts else None
    for j in range(1, len(ROTATE)):
        dts = [at(c, i, 16 + j) - at(c, i, 16 + j - 1) for c, i in use]
        out["rotate"][ROTATE[j]] = statistics.median(dts)
    # inside the rotate group's coefficient phase (slots 16+1 -> 16+9 .. 16+13 -> 16+2)
    sub = [(1, 9, "box values read + log-decay warp scan"), (9, 10, "coefficient-block release + barrier"),
           (10, 11, "coefficients written"), (11, 12, "angle partial sums written"), (12, 13, "barrier"),
           (13, 2, "mask factors + angle prefix")]
    out["rotate_coefficient_phase"] = {name: statistics.median(at(c, i, 16 + b) - at(c, i, 16 + a) for c, i in use)
                                       for a, b, name in sub}
    out["chunk_period_cycles"] = statistics.median(at(c, i + 1, 0) - at(c, i, 0) for c, i in use)
    out["chunk_period_us"] = out["chunk_period_cycles"] / ghz / 1e3
    out["rotate_busy_cycles"] = statistics.median(at(c, i, 24) - at(c, i, 16) for c, i in use)
    out["scores_issued_early"] = sum(at(c, i, 10) for c, i in use) / len(use)
    pk, src = peak_bf16_tflops()
    per_cycle = pk * 1e12 / SMS / (ghz * 1e9)          # FLOP per cycle of one SM at the traced clock
    # chunks whose scores went out early: thread 0 issued only H+= (and Yi) after the barrier
    hplus = [at(c, i, 12) - at(c, i, 1) for c, i in use if at(c, i - 1, 10) == 1 and at(c, i, 12)]
    yb = [at(c, i, 11) - at(c, i, 4) for c, i in use if at(c, i, 11)]
    f_h = 2.0 * N * P * QR                              # executed: M = N state rows, N = P, K = QR
    f_y = 2.0 * MM * P * QR                             # executed: M = MM rows, N = P, K = QR
    out["gemm_phase"] = {
        "peak_bf16_tflops": pk, "peak_source": src, "sm_flop_per_cycle": per_cycle,
        "chunk_state": {"shape_MxNxK": [N, P, QR], "cycles": statistics.median(hplus) if hplus else None,
                        "frac_of_sm_peak": f_h / statistics.median(hplus) / per_cycle if hplus else None},
        "output_SLX": {"shape_MxNxK": [MM, P, QR], "cycles": statistics.median(yb) if yb else None,
                       "frac_of_sm_peak": f_y / statistics.median(yb) / per_cycle if yb else None},
        "note": "issue-to-completion in place, the SM's tensor pipe shared by its CTAs",
    }
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=synth.SISO_1P5B.name, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--entry", default="plain", choices=ENTRIES,
                    help="m3_scan_fwd, or m3_scan_fwd_prep alone / with the B/C normalisation / and the gate")
    ap.add_argument("--json", default=None)
    a = ap.parse_args()
    out = run(a.workload, a.entry)
    print(json.dumps(out, indent=1))
    if a.json:
        with open(a.json, "w") as f:
            json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
