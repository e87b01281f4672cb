"""GPU-vs-oracle parity of the three entry points on small and ragged shapes.

Every call goes through the C ABI (libm3.so via ctypes); the float64 oracle
reads the very same (bf16- or fp32-rounded) input values.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import forms
from state_space_sequence_04_b300 import binding, synth

from parity_util import TOL, KEYS, assert_close, need_gpu, oracle_full, slice_bh, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


# ---------------------------------------------------------------------------
# m3_state_passing
@pytest.mark.parametrize("b,H,nc,N,P", [(2, 3, 5, 16, 8), (1, 2, 64, 128, 64), (3, 1, 1, 2, 4), (1, 1, 0, 8, 8)])
@pytest.mark.parametrize("with_init", [False, True])
def test_state_passing(b, H, nc, N, P, with_init):
    sp = synth.make_state_passing_inputs(b, H, max(nc, 1), N, P, seed=nc + N)
    U = sp["chunk_states"][:, :, :nc].contiguous()
    ld = sp["chunk_logdecay"][:, :, :nc].contiguous()
    ang = sp["chunk_angle"][:, :, :nc].contiguous()
    h0 = sp["init_state"] if with_init else None
    ref_carries, ref_fin = forms.state_passing(U, ld, ang, h0)
    Ud = U.cuda()
    fin = binding.state_passing(Ud, ld.cuda(), ang.cuda(), None if h0 is None else h0.cuda())
    torch.cuda.synchronize()
    assert_close(fin, ref_fin, TOL["fp32"], "final")
    if nc:
        assert_close(Ud, ref_carries, TOL["fp32"], "carries")


# ---------------------------------------------------------------------------
# m3_decode_step
@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("b,H,P,N,R", [(3, 2, 16, 16, 1), (2, 3, 64, 128, 1), (2, 2, 64, 64, 4), (1, 2, 32, 8, 2),
                                       (2, 1, 16, 32, 8)])
def test_decode_steps(io, b, H, P, N, R):
    steps = 12
    st = synth.make_decode_state(b, H, N, P, seed=1)
    ins = synth.make_decode_steps(b, H, P, N, R, steps, io=io, seed=2)
    state = st.cuda()
    cache = binding.new_decode_cache(b, H, N, P, R, synth.io_torch_dtype(io), "cuda")
    # a nonzero delayed write for the first step as well
    cache.copy_(torch.randn(cache.shape, generator=torch.Generator().manual_seed(3)).to(cache.dtype))
    h_ref = oracle.f64(st)
    prev_ref = oracle.f64(cache)
    A = ins["A"].cuda()
    for t in range(steps):
        args = [ins[k][t].cuda().contiguous() for k in ("x", "B", "C", "dt", "lam", "omega")]
        x_t, B_t, C_t, dt_t, lam_t, om_t = args
        y = binding.decode_step(state, x_t, B_t, cache, C_t, dt_t, A, lam_t, om_t, R)
        yr, h_ref, prev_ref = oracle.decode_step(h_ref, ins["x"][t], ins["B"][t], prev_ref, ins["C"][t],
                                                 ins["dt"][t], ins["A"], ins["lam"][t], ins["omega"][t])
        torch.cuda.synchronize()
        assert_close(y, yr, TOL[io], f"y step {t}")
    assert_close(state, h_ref, TOL[io], "state")
    assert np.array_equal(oracle.f64(cache), prev_ref), "delayed-write cache"


# ---------------------------------------------------------------------------
# m3_scan_fwd on small shapes: ragged tails, every rank, both dtypes
CASES = [
    # Bt, H, T, P, N, R, Q
    (1, 2, 256, 16, 16, 1, 64),      # the tiny fp32 workload's shape
    (2, 3, 1, 16, 16, 1, 64),
    (1, 2, 63, 32, 64, 1, 64),
    (1, 2, 64, 64, 128, 1, 64),
    (1, 1, 65, 64, 128, 1, 64),
    (2, 2, 1000, 64, 128, 1, 64),
    (1, 2, 200, 64, 64, 4, 64),
    (1, 2, 131, 64, 128, 4, 128),
    (1, 3, 77, 32, 32, 2, 16),
    (1, 1, 50, 16, 16, 8, 32),
    (1, 2, 300, 128, 64, 1, 256),
]


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("Bt,H,T,P,N,R,Q", CASES)
def test_scan_small(io, Bt, H, T, P, N, R, Q):
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, io)
    inp = synth.make_inputs(w, seed=T + N + R)
    d = to_dev(inp)
    y, fin = binding.scan_fwd(*[d[k] for k in KEYS], R, Q)
    torch.cuda.synchronize()
    yr, hr, _ = oracle_full(inp)
    assert_close(y, yr, TOL[io], "y")
    assert_close(fin, hr, TOL[io], "final_state")


# shapes the tensor-core path takes (bf16, P = 64, H % 4 == 0).  Few (batch, head)
# sequences against many chunks make it cut each sequence into segments (state
# pass, segment scan, full pass: 3 launches); every chunk runs as sub-chunks of
# 64/R tokens (64-row tiles), and with R >= 2 the state pass takes chunks of
# 128/R tokens (segments of an even number of sub-chunks).
TC_CASES = [
    # Bt, H, T, P, N, R, Q
    (1, 4, 1, 64, 128, 1, 64),
    (1, 4, 63, 64, 128, 1, 64),
    (2, 4, 65, 64, 128, 1, 64),
    (1, 8, 300, 64, 128, 1, 64),
    (2, 4, 1000, 64, 128, 1, 128),
    (1, 4, 200, 64, 128, 2, 64),
    (1, 4, 129, 64, 128, 2, 64),
    (1, 4, 6400, 64, 128, 1, 64),     # segments of two chunks
    (1, 4, 150, 64, 64, 1, 64),
    (1, 4, 200, 64, 64, 4, 64),       # MIMO, N = 64: sub-chunks of 16 tokens
    (2, 4, 333, 64, 128, 4, 128),     # MIMO, N = 128: sub-chunks of 16 tokens
    (1, 4, 100, 64, 128, 4, 64),
    (1, 4, 257, 64, 64, 2, 128),      # R = 2, N = 64: sub-chunks of 32 tokens
    (1, 4, 9001, 64, 128, 4, 64),     # segments of 8 sub-chunks (4 state-pass chunks), ragged end
    (1, 4, 5000, 64, 64, 2, 64),      # R = 2: segments of 4 sub-chunks (2 state-pass chunks)
    (1, 4, 9000, 64, 64, 1, 64),      # N = 64, R = 1: segments of 2 chunks, ragged end
]


@pytest.mark.parametrize("Bt,H,T,P,N,R,Q", TC_CASES)
def test_scan_tensor_core_path(Bt, H, T, P, N, R, Q):
    path, launches = binding.m3_scan_fwd_plan(Bt, T, H, P, N, R, Q, binding.M3_DTYPE_BF16)
    assert path == 1 and launches in (1, 3)
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, "bf16")
    inp = synth.make_inputs(w, seed=T + R + Q)
    d = to_dev(inp)
    ws = binding.alloc_workspace(d["x"].shape, N, R, Q, d["x"].dtype, "cuda")
    y, fin = binding.scan_fwd(*[d[k] for k in KEYS], R, Q, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "device-side wait gave up"
    yr, hr, _ = oracle_full(inp)
    assert_close(y, yr, TOL["bf16"], "y")
    assert_close(fin, hr, TOL["bf16"], "final_state")


@pytest.mark.parametrize("Bt,H,T,P,N,R,Q", [(1, 4, 300, 64, 128, 1, 64), (1, 4, 200, 64, 64, 4, 64),
                                            (1, 4, 150, 64, 128, 4, 128), (1, 4, 180, 64, 128, 2, 64)])
def test_scan_tensor_core_extreme_decay(Bt, H, T, P, N, R, Q):
    """Decays far beyond fp32's range inside one chunk: every 7th token has Delta = 8 and head 0
    has A = -16 (a log-decay of -128 for one token), so the tensor-core kernel's decay-to-chunk-end
    factor of earlier tokens hits its 2^-100 clamp and the mask's factors reach 2^100."""
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, "bf16")
    inp = synth.make_inputs(w, seed=T + 5 * R)
    inp["dt"][:, ::7] = 8.0
    inp["A"][0] = -16.0
    d = to_dev(inp)
    path, _ = binding.m3_scan_fwd_plan(Bt, T, H, P, N, R, Q, binding.M3_DTYPE_BF16)
    assert path == 1
    y, fin = binding.scan_fwd(*[d[k] for k in KEYS], R, Q)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all() and torch.isfinite(fin).all()
    yr, hr, _ = oracle_full(inp)
    assert_close(y, yr, TOL["bf16"], "y")
    assert_close(fin, hr, TOL["bf16"], "final_state")


def test_scan_chunk_independence():
    """Different chunk lengths give the same result up to rounding (section 3.3)."""
    w = synth.Workload("case", 1, 2, 300, 64, 64, 2, 64, "fp32")
    d = to_dev(synth.make_inputs(w, seed=4))
    outs = [binding.scan_fwd(*[d[k] for k in KEYS], 2, Q) for Q in (16, 32, 64, 128, 256)]
    torch.cuda.synchronize()
    for y, f in outs[1:]:
        assert_close(y, outs[0][0], TOL["fp32"], "y vs chunk 16")
        assert_close(f, outs[0][1], TOL["fp32"], "final vs chunk 16")


def test_scan_zero_length():
    w = synth.Workload("case", 2, 2, 4, 16, 16, 1, 64, "bf16")
    d = to_dev(synth.make_inputs(w, seed=0))
    x = d["x"][:, :0].contiguous()
    B = d["B"][:, :0].contiguous()
    C = d["C"][:, :0].contiguous()
    y, fin = binding.scan_fwd(x, B, C, d["dt"][:, :0].contiguous(), d["A"], d["lam"][:, :0].contiguous(),
                              d["omega"][:, :0].contiguous(), 1, 64)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert float(fin.abs().max()) == 0.0


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_prefill_then_decode_continuation(io):
    """prefill(T0) then decode steps T0..T-1 equals the oracle's prefill(T)."""
    Bt, H, T, P, N, R, Q, T0 = 2, 2, 150, 32, 64, 2, 64, 130
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, io)
    inp = synth.make_inputs(w, seed=11)
    d = to_dev(inp)
    pre = {k: (d[k][:, :T0].contiguous() if k != "A" else d[k]) for k in KEYS}
    _, state = binding.scan_fwd(*[pre[k] for k in KEYS], R, Q)
    cache = binding.cache_from_prefill(pre["B"], pre["x"])
    yr, hr, _ = oracle_full(inp)
    for t in range(T0, T):
        sl = [d[k][:, t].contiguous() for k in ("x", "B", "C", "dt", "lam", "omega")]
        x_t, B_t, C_t, dt_t, lam_t, om_t = sl
        y = binding.decode_step(state, x_t, B_t, cache, C_t, dt_t, d["A"], lam_t, om_t, R)
        torch.cuda.synchronize()
        assert_close(y, yr[:, t], TOL[io], f"decode y at t={t}")
    assert_close(state, hr, TOL[io], "state after decode")


def test_status_codes_from_device_calls():
    """Bad calls made with real device tensors fail with a status and launch nothing."""
    w = synth.Workload("case", 1, 2, 64, 16, 16, 1, 64, "fp32")
    d = to_dev(synth.make_inputs(w, seed=0))
    y = torch.empty_like(d["x"])
    st = binding.m3_scan_fwd(*[d[k] for k in KEYS], 1, 64, y, None, None)
    assert st == binding.M3_ERR_WORKSPACE
    st = binding.m3_scan_fwd(*[d[k] for k in KEYS], 1, 40, y, None, None)
    assert st == binding.M3_ERR_UNSUPPORTED
    with pytest.raises(binding.M3Error):
        binding.scan_fwd(*[d[k] for k in KEYS], 3, 64)
