"""Parity at the full workload sizes, in the launch configuration the benchmark
times.  The GPU computes every (batch, head); the float64 oracle recomputes a
few sampled (batch, head) sequences in full and they are compared element by
element (y and final state), with the tolerances max|err|/max|ref| <= 2e-2
(bf16 inputs, fp32 accumulation) and <= 1e-4 (fp32 inputs)."""
import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_04_b300 import binding, synth

from parity_util import TOL, KEYS, assert_close, need_gpu, oracle_sampled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _check_prefill(w, samples, seed=0):
    inp = synth.make_inputs(w, seed=seed, device="cuda")
    y, fin = binding.scan_fwd(*[inp[k] for k in KEYS], w.rank, w.chunk)
    torch.cuda.synchronize()
    ref = oracle_sampled(inp, samples)
    for b, h in samples:
        yr, hr, _ = ref[(b, h)]
        assert_close(y[b:b + 1, :, h:h + 1], yr, TOL[w.io], f"{w.name} y (b={b},h={h})")
        assert_close(fin[b:b + 1, h:h + 1], hr, TOL[w.io], f"{w.name} final (b={b},h={h})")
    assert torch.isfinite(y.float()).all()
    return inp, y, fin, ref


def test_tiny_fp32_full():
    w = synth.TINY
    inp = synth.make_inputs(w, seed=0)
    d = {k: inp[k].cuda() for k in KEYS}
    y, fin = binding.scan_fwd(*[d[k] for k in KEYS], w.rank, w.chunk)
    torch.cuda.synchronize()
    yr, hr, _ = oracle.scan(*[inp[k] for k in KEYS])
    assert_close(y, yr, TOL["fp32"], "y")
    assert_close(fin, hr, TOL["fp32"], "final")


def test_siso_prefill_1p5b_width():
    w = synth.SISO_1P5B
    _check_prefill(w, [(0, 0), (3, 63), (1, 17), (2, 40)])


def test_mimo_prefill_r4():
    w = synth.MIMO_R4
    _check_prefill(w, [(0, 0), (1, 31), (0, 13)])


def _decode_run(state, A, b, H, P, N, R, steps, samples, seed, io="bf16", dt_mu=-3.0, dt_sd=1.0,
                lam_uniform=False, cache=None, block=64):
    """Run ``steps`` carried decode calls; return the sampled y per step and their inputs (CPU)."""
    dev = state.device
    iot = synth.io_torch_dtype(io)
    if cache is None:
        cache = binding.new_decode_cache(b, H, N, P, R, iot, dev)
    ys = {s: [] for s in samples}
    ins_s = {s: {k: [] for k in ("x", "B", "C", "dt", "lam", "omega")} for s in samples}
    y_t = torch.empty((b, H, R, P), dtype=iot, device=dev)
    for s0 in range(0, steps, block):
        nb = min(block, steps - s0)
        ins = synth.make_decode_steps(b, H, P, N, R, nb, io=io, seed=seed + s0, device=dev, dt_mu=dt_mu,
                                      dt_sd=dt_sd, lam_uniform=lam_uniform, A=A)
        for t in range(nb):
            a = [ins[k][t] for k in ("x", "B", "C", "dt", "lam", "omega")]
            binding.decode_step(state, a[0], a[1], cache, a[2], a[3], A, a[4], a[5], R, y_t=y_t)
            for (bb, hh) in samples:
                ys[(bb, hh)].append(y_t[bb, hh].float().cpu())
        for (bb, hh) in samples:
            for k in ins_s[(bb, hh)]:
                ins_s[(bb, hh)][k].append(ins[k][:, bb, hh].cpu())
    torch.cuda.synchronize()
    return ys, ins_s, cache


def _decode_oracle(h0, prev0, A_h, ins):
    """Sequential oracle over the sampled sequence's steps (one (b, h))."""
    x = torch.cat(ins["x"])[None, :, None]       # [1, S, 1, R, P]
    B = torch.cat(ins["B"])[None, :, None]
    C = torch.cat(ins["C"])[None, :, None]
    dt = torch.cat(ins["dt"])[None, :, None]
    lam = torch.cat(ins["lam"])[None, :, None]
    om = torch.cat(ins["omega"])[None, :, None]
    return oracle.scan(x, B, C, dt, A_h, lam, om, h0=h0, prev=prev0)


@pytest.mark.parametrize("R", [1, 4])
@pytest.mark.parametrize("b", [1, 8, 64, 256])
def test_decode_sweep(b, R):
    H, P, N, steps = 64, 64, 128, synth.DECODE_STEPS
    state = synth.make_decode_state(b, H, N, P, seed=0, device="cuda")
    h0 = state.clone()
    A = synth.make_decode_steps(1, H, P, N, R, 1, seed=99, device="cuda")["A"]
    samples = sorted({(0, 0), (b - 1, H - 1), (b // 2, 17)})
    ys, ins, _ = _decode_run(state, A, b, H, P, N, R, steps, samples, seed=1000 * R + b)
    for (bb, hh) in samples:
        yr, hr, _ = _decode_oracle(h0[bb:bb + 1, hh:hh + 1], None, A[hh:hh + 1], ins[(bb, hh)])
        got = torch.stack(ys[(bb, hh)])          # [S, R, P]
        assert_close(got, yr[0, :, 0], TOL["bf16"], f"decode y b={b} R={R} ({bb},{hh})")
        assert_close(state[bb, hh], hr[0, 0], TOL["bf16"], f"decode state b={b} R={R} ({bb},{hh})")


def test_long_context_mimo_prefill_then_decode():
    w = synth.LONG_MIMO
    samples = [(0, 0), (0, 37), (0, 63)]
    inp, y, fin, ref = _check_prefill(w, samples)
    # 256 decode steps from the prefill's final state and delayed-write cache
    H, P, N, R = w.heads, w.headdim, w.dstate, w.rank
    cache = binding.cache_from_prefill(inp["B"], inp["x"])
    state = fin.clone()
    h_start = fin.clone()
    cache0 = cache.clone()
    ys, ins, _ = _decode_run(state, inp["A"], 1, H, P, N, R, 256, samples, seed=7, dt_mu=w.dt_mu,
                             dt_sd=w.dt_sd, lam_uniform=True, cache=cache)
    for (bb, hh) in samples:
        # the oracle continues from its own prefill state for this sequence
        _, hr_pre, prev_pre = ref[(bb, hh)]
        assert np.array_equal(prev_pre[0, 0], oracle.f64(cache0[bb, hh]))
        yr, hr, _ = _decode_oracle(hr_pre, prev_pre, inp["A"][hh:hh + 1], ins[(bb, hh)])
        got = torch.stack(ys[(bb, hh)])
        assert_close(got, yr[0, :, 0], TOL["bf16"], f"long decode y ({bb},{hh})")
        assert_close(state[bb, hh], hr[0, 0], TOL["bf16"], f"long decode state ({bb},{hh})")
    del h_start
