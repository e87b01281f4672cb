"""GPU-vs-oracle parity of the pre-activation entry points (m3_scan_fwd_prep,
m3_decode_step_prep): Delta = softplus(dt_raw + dt_bias), lambda = sigmoid(u)
and one decay generator A_t per token, derived inside the kernels.

Every call goes through the C ABI; the float64 oracle (``oracle.scan_prep``)
reads the same rounded input values and applies softplus / sigmoid in float64.
"""
import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_04_b300 import binding, synth

from parity_util import TOL, assert_close, need_gpu

pytestmark = pytest.mark.gpu

PKEYS = ("x", "B", "C", "dt_raw", "dt_bias", "A", "u", "omega")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _dev(inp):
    return {k: inp[k].cuda().contiguous() for k in PKEYS}


def _bc_f64(bc):
    return None if bc is None else {k: (oracle.f64(v) if hasattr(v, "shape") else v) for k, v in bc.items()}


def _bc_dev(bc):
    return None if bc is None else {k: (v.cuda().contiguous() if hasattr(v, "shape") else v) for k, v in bc.items()}


def _oracle(inp, bias=True, bc=None, z=None):
    return oracle.scan_prep(inp["x"], inp["B"], inp["C"], inp["dt_raw"], inp["dt_bias"] if bias else None, inp["A"],
                            inp["u"], inp["omega"], bc=_bc_f64(bc), z=None if z is None else oracle.f64(z))


def _oracle_sampled(inp, samples, bc=None):
    """Oracle on sampled (batch, head) sequences stacked as heads of a batch-1 problem."""
    f = oracle.f64
    cols = {k: [] for k in PKEYS}
    for b, h in samples:
        for k in PKEYS:
            cols[k].append(f(inp[k][h:h + 1]) if k == "dt_bias" else f(inp[k][b:b + 1, :, h:h + 1]))
    st = {k: np.concatenate(cols[k], axis=0 if k == "dt_bias" else 2) for k in PKEYS}
    bcs = None
    if bc is not None:   # the biases of the sampled heads, stacked like the heads
        bcs = _bc_f64(bc)
        for k in ("B_bias", "C_bias"):
            if bcs.get(k) is not None:
                bcs[k] = np.concatenate([bcs[k][h:h + 1] for _, h in samples], axis=0)
    y, hT, _ = oracle.scan_prep(st["x"], st["B"], st["C"], st["dt_raw"], st["dt_bias"], st["A"], st["u"], st["omega"],
                                bc=bcs)
    return {s: (y[:, :, i:i + 1], hT[:, i:i + 1]) for i, s in enumerate(samples)}


def _run(inp, R, Q, bias=True, bc=None, z=None):
    d = _dev(inp)
    Bt, T, H, _, P = d["x"].shape
    N = d["B"].shape[-1]
    ws = binding.alloc_workspace_prep(d["x"].shape, N, R, Q, d["x"].dtype, "cuda")
    y, fin = binding.scan_fwd_prep(d["x"], d["B"], d["C"], d["dt_raw"], d["A"], d["u"], d["omega"], R, Q,
                                   dt_bias=d["dt_bias"] if bias else None, bc=_bc_dev(bc),
                                   z=None if z is None else z.cuda().contiguous(), workspace=ws)
    torch.cuda.synchronize()
    return y, fin, ws


# ---------------------------------------------------------------------------
# tensor-core path (bf16, P = 64, H % 4 == 0): ragged tails, segments, MIMO sub-chunks
TC_CASES = [
    # Bt, H, T, P, N, R, Q
    (1, 4, 1, 64, 128, 1, 64),
    (2, 4, 65, 64, 128, 1, 64),
    (1, 8, 300, 64, 128, 1, 64),
    (2, 4, 1000, 64, 128, 1, 128),
    (1, 4, 200, 64, 128, 2, 64),
    (1, 4, 6400, 64, 128, 1, 64),     # segments: state pass, segment scan, full pass
    (1, 4, 150, 64, 64, 1, 64),
    (1, 4, 200, 64, 64, 4, 64),       # MIMO, N = 64: sub-chunks of 16 tokens
    (2, 4, 333, 64, 128, 4, 128),     # MIMO, N = 128: sub-chunks of 32 tokens
]


def _bc_case(kind, H, R, N):
    """None, or the B / C options: "norm" (RMS norm, gains, biases) or "bias" (biases only)."""
    if kind is None:
        return None
    bc = synth.make_bc_params(H, R, N, seed=H + R + N)
    if kind == "bias":
        bc = {"B_bias": bc["B_bias"], "C_bias": bc["C_bias"]}
    return bc


@pytest.mark.parametrize("bc_kind", [None, "norm"])
@pytest.mark.parametrize("Bt,H,T,P,N,R,Q", TC_CASES)
def test_scan_prep_tensor_core(Bt, H, T, P, N, R, Q, bc_kind):
    path, _ = binding.m3_scan_fwd_plan(Bt, T, H, P, N, R, Q, binding.M3_DTYPE_BF16)
    assert path == 1
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, "bf16")
    inp = synth.make_prep_inputs(w, seed=T + R + Q)
    bc = _bc_case(bc_kind, H, R, N)
    y, fin, ws = _run(inp, R, Q, bc=bc)
    assert int(ws[:4].view(torch.int32).item()) == 0, "device-side wait gave up"
    yr, hr, _ = _oracle(inp, bc=bc)
    assert_close(y, yr, TOL["bf16"], "y")
    assert_close(fin, hr, TOL["bf16"], "final_state")


@pytest.mark.parametrize("Bt,H,T,P,N,R,Q", [(1, 8, 300, 64, 128, 1, 64), (1, 4, 200, 64, 64, 4, 64)])
def test_scan_prep_tensor_core_bias_only(Bt, H, T, P, N, R, Q):
    """B / C channel biases without the normalisation."""
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, "bf16")
    inp = synth.make_prep_inputs(w, seed=3)
    bc = _bc_case("bias", H, R, N)
    y, fin, _ = _run(inp, R, Q, bc=bc)
    yr, hr, _ = _oracle(inp, bc=bc)
    assert_close(y, yr, TOL["bf16"], "y")
    assert_close(fin, hr, TOL["bf16"], "final_state")


# output gate y * silu(z): 64-row tiles (SISO, MIMO sub-chunks) and 128-row tiles, with and
# without the B / C normalisation, on both prefill paths
@pytest.mark.parametrize("with_bc", [False, True])
@pytest.mark.parametrize("io,Bt,H,T,P,N,R,Q", [
    ("bf16", 1, 8, 300, 64, 128, 1, 64),
    ("bf16", 1, 4, 200, 64, 64, 4, 64),
    ("bf16", 2, 4, 333, 64, 128, 1, 128),
    ("bf16", 1, 4, 129, 64, 128, 2, 64),
    ("fp32", 1, 2, 256, 16, 16, 1, 64),
    ("fp32", 2, 3, 77, 32, 64, 2, 64),
])
def test_scan_prep_gate(io, Bt, H, T, P, N, R, Q, with_bc):
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, io)
    inp = synth.make_prep_inputs(w, seed=T + N)
    z = synth.make_gate(tuple(inp["x"].shape), io=io, seed=T)
    bc = _bc_case("norm", H, R, N) if with_bc else None
    y, fin, _ = _run(inp, R, Q, bc=bc, z=z)
    yr, hr, _ = _oracle(inp, bc=bc, z=z)
    assert_close(y, yr, TOL[io], "gated y")
    assert_close(fin, hr, TOL[io], "final_state (the gate leaves the state alone)")


# ---------------------------------------------------------------------------
# CUDA-core path: fp32 io (and a bf16 shape outside the tensor-core tiles)
@pytest.mark.parametrize("io,Bt,H,T,P,N,R,Q", [
    ("fp32", 1, 2, 256, 16, 16, 1, 64),    # the tiny fp32 workload's shape
    ("fp32", 2, 3, 77, 32, 64, 2, 64),
    ("fp32", 1, 2, 130, 64, 128, 4, 64),
    ("bf16", 1, 3, 90, 32, 64, 1, 64),
])
@pytest.mark.parametrize("bc_kind", [None, "norm", "bias"])
def test_scan_prep_cuda_cores(io, Bt, H, T, P, N, R, Q, bc_kind):
    path, _ = binding.m3_scan_fwd_plan(Bt, T, H, P, N, R, Q, binding.io_code(synth.io_torch_dtype(io)))
    assert path == 0
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, io)
    inp = synth.make_prep_inputs(w, seed=T + P)
    bc = _bc_case(bc_kind, H, R, N)
    y, fin, _ = _run(inp, R, Q, bc=bc)
    yr, hr, _ = _oracle(inp, bc=bc)
    assert_close(y, yr, TOL[io], "y")
    assert_close(fin, hr, TOL[io], "final_state")


@pytest.mark.parametrize("io,P", [("bf16", 64), ("fp32", 16)])
def test_scan_prep_without_bias(io, P):
    w = synth.Workload("case", 1, 4, 140, P, 64 if io == "bf16" else 16, 1, 64, io)
    inp = synth.make_prep_inputs(w, seed=5)
    y, fin, _ = _run(inp, 1, 64, bias=False)
    yr, hr, _ = _oracle(inp, bias=False)
    assert_close(y, yr, TOL[io], "y")
    assert_close(fin, hr, TOL[io], "final_state")


def test_scan_prep_extreme_preactivations():
    """Very large / very negative pre-activations: Delta -> dt_raw (softplus's linear
    branch) or -> 0, lambda -> 1 or 0, on the tensor-core path."""
    w = synth.Workload("case", 1, 4, 200, 64, 128, 1, 64, "bf16")
    inp = synth.make_prep_inputs(w, seed=8)
    g = torch.Generator().manual_seed(4)
    pick = torch.rand(inp["u"].shape, generator=g)
    inp["u"] = torch.where(pick < 0.3, torch.full_like(inp["u"], 40.0),
                           torch.where(pick > 0.7, torch.full_like(inp["u"], -40.0), inp["u"]))
    pick = torch.rand(inp["dt_raw"].shape, generator=g)
    inp["dt_raw"] = torch.where(pick < 0.05, torch.full_like(inp["dt_raw"], 1.5),
                                torch.where(pick > 0.8, torch.full_like(inp["dt_raw"], -30.0), inp["dt_raw"]))
    y, fin, _ = _run(inp, 1, 64)
    yr, hr, _ = _oracle(inp)
    assert_close(y, yr, TOL["bf16"], "y")
    assert_close(fin, hr, TOL["bf16"], "final_state")


# ---------------------------------------------------------------------------
# full-size workloads in the benchmark's launch configuration, checked on sampled sequences
@pytest.mark.parametrize("bc_kind", [None, "norm"])
@pytest.mark.parametrize("wl,samples", [
    (synth.SISO_1P5B, [(0, 0), (1, 37), (2, 63), (3, 12)]),
    (synth.MIMO_R4, [(0, 0), (1, 31), (0, 17)]),
])
def test_scan_prep_full_workload_sampled(wl, samples, bc_kind):
    inp = synth.make_prep_inputs(wl, seed=0)
    bc = _bc_case(bc_kind, wl.heads, wl.rank, wl.dstate)
    y, fin, ws = _run(inp, wl.rank, wl.chunk, bc=bc)
    assert int(ws[:4].view(torch.int32).item()) == 0, "device-side wait gave up"
    ref = _oracle_sampled(inp, samples, bc=bc)
    for (b, h), (yr, hr) in ref.items():
        assert_close(y[b:b + 1, :, h:h + 1], yr, TOL["bf16"], f"y (b={b}, h={h})")
        assert_close(fin[b:b + 1, h:h + 1], hr, TOL["bf16"], f"final_state (b={b}, h={h})")


# ---------------------------------------------------------------------------
# m3_decode_step_prep
@pytest.mark.parametrize("bc_kind", [None, "norm", "norm+gate"])
@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("b,H,P,N,R", [(3, 2, 16, 16, 1), (2, 3, 64, 128, 1), (2, 2, 64, 128, 4), (2, 1, 16, 32, 8),
                                       (64, 4, 64, 128, 1), (2, 1, 4, 2, 1)])
def test_decode_prep_steps(io, b, H, P, N, R, bc_kind):
    steps = 10
    st = synth.make_decode_state(b, H, N, P, seed=1)
    ins = synth.make_decode_prep_steps(b, H, P, N, R, steps, io=io, seed=2)
    gate = bc_kind == "norm+gate"
    bc = _bc_case("norm" if gate else bc_kind, H, R, N)
    bcd, bcf = _bc_dev(bc), _bc_f64(bc)
    zs = synth.make_gate((steps, b, H, R, P), io=io, seed=5) if gate else None
    state = st.cuda()
    cache = binding.new_decode_cache(b, H, N, P, R, synth.io_torch_dtype(io), "cuda")
    cache.copy_(torch.randn(cache.shape, generator=torch.Generator().manual_seed(3)).to(cache.dtype))
    h_ref, prev_ref = oracle.f64(st), oracle.f64(cache)
    bias = ins["dt_bias"].cuda()
    for t in range(steps):
        x_t, B_t, C_t, dr_t, A_t, u_t, om_t = [ins[k][t].cuda().contiguous()
                                               for k in ("x", "B", "C", "dt_raw", "A", "u", "omega")]
        z_t = None if zs is None else zs[t].cuda().contiguous()
        y = binding.decode_step_prep(state, x_t, B_t, cache, C_t, dr_t, A_t, u_t, om_t, R, dt_bias=bias, bc=bcd,
                                     z_t=z_t)
        yr, h_ref, prev_ref = oracle.decode_step_prep(h_ref, ins["x"][t], ins["B"][t], prev_ref, ins["C"][t],
                                                      ins["dt_raw"][t], ins["dt_bias"], ins["A"][t], ins["u"][t],
                                                      ins["omega"][t], bc=bcf,
                                                      z_t=None if zs is None else oracle.f64(zs[t]))
        torch.cuda.synchronize()
        assert_close(y, yr, TOL[io], f"y step {t}")
    assert_close(state, h_ref, TOL[io], "state")
    assert np.array_equal(oracle.f64(cache), prev_ref), "delayed-write cache (raw B, X)"
    assert binding.m3_device_status(clear=True) == binding.M3_OK


@pytest.mark.parametrize("bc_kind", [None, "norm"])
@pytest.mark.parametrize("io,P,N,R", [("fp32", 32, 64, 2), ("bf16", 64, 128, 1), ("bf16", 64, 64, 4)])
def test_prefill_prep_then_decode_prep(io, P, N, R, bc_kind):
    """scan_fwd_prep over T0 tokens, then decode_step_prep over the rest, equals the
    oracle's prefill over all T tokens."""
    Bt, H, T, Q, T0 = 2, 4, 150, 64, 131
    w = synth.Workload("case", Bt, H, T, P, N, R, Q, io)
    inp = synth.make_prep_inputs(w, seed=11)
    bc = _bc_case(bc_kind, H, R, N)
    bcd = _bc_dev(bc)
    d = _dev(inp)
    pre = {k: (d[k][:, :T0].contiguous() if k != "dt_bias" else d[k]) for k in PKEYS}
    _, state = binding.scan_fwd_prep(pre["x"], pre["B"], pre["C"], pre["dt_raw"], pre["A"], pre["u"], pre["omega"],
                                     R, Q, dt_bias=pre["dt_bias"], bc=bcd)
    cache = binding.cache_from_prefill(pre["B"], pre["x"])
    yr, hr, _ = _oracle(inp, bc=bc)
    for t in range(T0, T):
        x_t, B_t, C_t, dr_t, A_t, u_t, om_t = [d[k][:, t].contiguous()
                                               for k in ("x", "B", "C", "dt_raw", "A", "u", "omega")]
        y = binding.decode_step_prep(state, x_t, B_t, cache, C_t, dr_t, A_t, u_t, om_t, R, dt_bias=d["dt_bias"],
                                     bc=bcd)
        torch.cuda.synchronize()
        assert_close(y, yr[:, t], TOL[io], f"decode y at t={t}")
    assert_close(state, hr, TOL[io], "state after decode")


def test_prep_entry_points_reject_bad_arguments():
    w = synth.Workload("case", 1, 4, 64, 64, 128, 1, 64, "bf16")
    d = _dev(synth.make_prep_inputs(w, seed=1))
    y = torch.empty_like(d["x"])
    ws = binding.alloc_workspace_prep(d["x"].shape, 128, 1, 64, d["x"].dtype, "cuda")
    args = [d[k] for k in ("x", "B", "C", "dt_raw", "A", "u", "omega")]
    params = binding.prep_params(d["dt_bias"])
    assert binding.m3_scan_fwd_prep(*args, 1, 64, y, None, ws, params) == binding.M3_OK
    assert binding.m3_scan_fwd_prep(*args, 1, 64, y, None, ws, None) == binding.M3_OK   # NULL params: all off
    bad = list(args)
    bad[4] = None   # A (per token) is required
    assert binding.m3_scan_fwd_prep(*bad, 1, 64, y, None, ws, params) == binding.M3_ERR_INVALID_ARG
    assert binding.m3_scan_fwd_prep(*args, 1, 64, y, None, ws[:16], params) == binding.M3_ERR_WORKSPACE
    neg = binding.prep_params(d["dt_bias"], {"norm": True, "eps": -1.0})
    assert binding.m3_scan_fwd_prep(*args, 1, 64, y, None, ws, neg) == binding.M3_ERR_INVALID_ARG
    mis = binding.PrepParams(d["dt_bias"].data_ptr() + 4, 0, 0.0, None, None, None, None)   # misaligned
    assert binding.m3_scan_fwd_prep(*args, 1, 64, y, None, ws, mis) == binding.M3_ERR_INVALID_ARG
    torch.cuda.synchronize()
