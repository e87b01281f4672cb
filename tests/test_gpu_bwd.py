"""GPU-vs-oracle parity of the backward pass (m3_scan_bwd).

Small problems: every gradient element against central differences of the
float64 oracle (``oracle.grad.grad_fd``).  Larger problems: the loss is linear
in x, in B and in C, so along a random step d the loss changes by exactly
<grad, d> (two oracle evaluations); along dt, lambda, omega and A the
directional derivative by central differences.  Tolerances: the kernel
computes in fp32 (and reads bf16 inputs as given), the references are
float64; errors are measured relative to the largest reference value.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import grad
from state_space_sequence_04_b300 import binding, synth

from parity_util import KEYS, need_gpu, slice_bh

pytestmark = pytest.mark.gpu

TOL_BWD = {"fp32": 2e-4, "bf16": 2e-3}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _run(inp, R, dy, dfin=None):
    d = {k: inp[k].cuda().contiguous() for k in KEYS}
    g = binding.scan_bwd(*[d[k] for k in KEYS], R, dy.cuda().contiguous(),
                         None if dfin is None else dfin.cuda().contiguous())
    torch.cuda.synchronize()
    return {k: v.cpu().double().numpy() for k, v in g.items()}


def _ref_inputs(inp):
    return {"x": oracle.f64(inp["x"]), "B": oracle.f64(inp["B"]), "C": oracle.f64(inp["C"]), "dt": oracle.f64(inp["dt"]),
            "A": oracle.f64(inp["A"]), "lam": oracle.f64(inp["lam"]), "omega": oracle.f64(inp["omega"])}


NAMES = {"x": "dx", "B": "dB", "C": "dC", "dt": "ddt", "A": "dA", "lam": "dlam", "omega": "domega"}


# chunks of Q = 16 (R <= 2), 8 (R = 4), 4 (R = 8) tokens; pair blocks of 128 / (P / 4) pairs
@pytest.mark.parametrize("io,Bt,H,T,P,N,R", [
    ("fp32", 1, 2, 9, 4, 4, 1),      # one ragged chunk
    ("fp32", 2, 1, 7, 8, 6, 2),
    ("fp32", 1, 2, 6, 4, 8, 4),
    ("bf16", 1, 2, 8, 4, 4, 2),
    ("fp32", 1, 2, 37, 4, 4, 1),     # three chunks, ragged tail
    ("fp32", 1, 1, 19, 8, 6, 4),     # three chunks of 8
    ("fp32", 1, 1, 11, 4, 4, 8),     # three chunks of 4
    ("fp32", 1, 1, 20, 32, 40, 1),   # two pair blocks (16 + 4 pairs), two chunks
    ("fp32", 1, 1, 12, 128, 8, 1),   # 32 column lanes per pair
])
@pytest.mark.parametrize("with_final", [False, True])
def test_bwd_small_every_element(io, Bt, H, T, P, N, R, with_final):
    w = synth.Workload("case", Bt, H, T, P, N, R, 64, io)
    inp = synth.make_inputs(w, seed=T + N + R)
    gen = torch.Generator().manual_seed(3)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfin = torch.randn((Bt, H, N, P), generator=gen) if with_final else None
    got = _run(inp, R, dy, dfin)
    ref = grad.grad_fd(_ref_inputs(inp), oracle.f64(dy), None if dfin is None else oracle.f64(dfin))
    for k, name in NAMES.items():
        err = oracle.rel_err(got[name], ref[k])
        assert err < TOL_BWD[io], f"{name}: {err:.2e}"


@pytest.mark.parametrize("io,Bt,H,T,P,N,R", [
    ("fp32", 1, 2, 150, 64, 128, 1),
    ("bf16", 2, 2, 200, 64, 64, 4),
    ("fp32", 1, 4, 96, 32, 64, 2),
    ("fp32", 1, 2, 64, 64, 32, 2),    # P = 64 with eight pairs per block: the compile-time-shape kernels
    ("bf16", 1, 1, 40, 64, 16, 8),
])
def test_bwd_larger_directional(io, Bt, H, T, P, N, R):
    w = synth.Workload("case", Bt, H, T, P, N, R, 64, io)
    inp = synth.make_inputs(w, seed=7)
    gen = torch.Generator().manual_seed(5)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfin = torch.randn((Bt, H, N, P), generator=gen)
    got = _run(inp, R, dy, dfin)
    ref = _ref_inputs(inp)
    dy64, df64 = oracle.f64(dy), oracle.f64(dfin)
    rng = np.random.default_rng(9)
    l0 = grad.loss(ref, dy64, df64)
    for k in ("x", "B", "C"):   # exact: the loss is linear in each of them
        d = rng.standard_normal(ref[k].shape)
        moved = dict(ref)
        moved[k] = ref[k] + d
        exact = grad.loss(moved, dy64, df64) - l0
        kern = float(np.sum(got[NAMES[k]] * d))
        assert abs(kern - exact) <= TOL_BWD[io] * max(1.0, abs(exact)), (k, kern, exact)
    for k in ("dt", "lam", "omega", "A"):
        d = rng.standard_normal(ref[k].shape)
        if k == "lam":   # stay inside [0, 1]
            d = d * np.minimum(ref[k], 1.0 - ref[k])
        if k == "dt":
            d = d * ref[k]
        num = grad.directional(ref, k, d, dy64, df64, eps=1e-6)
        kern = float(np.sum(got[NAMES[k]] * d))
        assert abs(kern - num) <= TOL_BWD[io] * max(1.0, abs(num)), (k, kern, num)


def _directional_checks(got, ref, dy64, df64, tol, rng):
    l0 = grad.loss(ref, dy64, df64)
    for k in ("x", "B", "C"):   # exact: the loss is linear in each of them
        d = rng.standard_normal(ref[k].shape)
        moved = dict(ref)
        moved[k] = ref[k] + d
        exact = grad.loss(moved, dy64, df64) - l0
        kern = float(np.sum(got[NAMES[k]] * d))
        assert abs(kern - exact) <= tol * max(1.0, abs(exact)), (k, kern, exact)
    for k in ("dt", "lam", "omega"):
        d = rng.standard_normal(ref[k].shape) * (ref[k] if k == "dt" else 1.0)
        num = grad.directional(ref, k, d, dy64, df64, eps=1e-6)
        kern = float(np.sum(got[NAMES[k]] * d))
        assert abs(kern - num) <= tol * max(1.0, abs(num)), (k, kern, num)


def test_bwd_full_size_sampled():
    """Batch 4, 4096 tokens, 64 heads, P = 64, N = 128, SISO, bf16 (the prefill workload's size):
    each (batch, head) is an independent problem, so the gradients of two sampled ones are
    checked against the oracle run on that slice alone (dA, summed over the batch, excepted)."""
    Bt, T, H, P, N, R = 4, 4096, 64, 64, 128, 1
    w = synth.Workload("case", Bt, H, T, P, N, R, 64, "bf16")
    inp = synth.make_inputs(w, seed=11)
    gen = torch.Generator().manual_seed(12)
    dy = torch.randn(inp["x"].shape, generator=gen).to(torch.bfloat16)
    dfin = torch.randn((Bt, H, N, P), generator=gen)
    got = _run(inp, R, dy, dfin)
    rng = np.random.default_rng(13)
    for b, h in ((0, 5), (3, 62)):
        ref = dict(zip(grad.INPUTS, slice_bh(inp, b, h)))
        sl = {NAMES[k]: (got[NAMES[k]][b:b + 1, :, h:h + 1] if k != "A" else got["dA"][h:h + 1])
              for k in grad.INPUTS}
        _directional_checks(sl, ref, oracle.f64(dy[b:b + 1, :, h:h + 1]), oracle.f64(dfin[b:b + 1, h:h + 1]),
                            TOL_BWD["bf16"], rng)


def test_bwd_rejects_unsupported_and_bad_arguments():
    assert binding.m3_scan_bwd_workspace_size(1, 8, 2, 12, 16, 1, 1) == 0          # P = 12: not a power of two / 4
    w = synth.Workload("case", 1, 2, 8, 4, 4, 1, 64, "fp32")
    d = {k: v.cuda() for k, v in synth.make_inputs(w, seed=1).items() if k in KEYS}
    dy = torch.zeros_like(d["x"])
    f = dict(dtype=torch.float32, device="cuda")
    grads = {"dx": torch.empty(d["x"].shape, **f), "dB": torch.empty(d["B"].shape, **f),
             "dC": torch.empty(d["C"].shape, **f), "ddt": torch.empty(d["dt"].shape, **f),
             "dA": torch.empty(d["A"].shape, **f), "dlam": torch.empty(d["lam"].shape, **f),
             "domega": torch.empty(d["omega"].shape, **f)}
    ws = torch.empty(binding.m3_scan_bwd_workspace_size(1, 8, 2, 4, 4, 1, 1), dtype=torch.uint8, device="cuda")
    args = [d[k] for k in KEYS]
    assert binding.m3_scan_bwd(*args, 1, dy, None, grads, ws) == binding.M3_OK
    assert binding.m3_scan_bwd(*args, 1, dy, None, grads, ws[:64]) == binding.M3_ERR_WORKSPACE
    grads2 = dict(grads)
    grads2["dB"] = None
    assert binding.m3_scan_bwd(*args, 1, dy, None, grads2, ws) == binding.M3_ERR_INVALID_ARG
    torch.cuda.synchronize()


# ---- m3_scan_bwd_prep: pre-activations (Delta = softplus(dt_raw + dt_bias), lambda = sigmoid(u), A per token)
PREP_NAMES = {"x": "dx", "B": "dB", "C": "dC", "dt_raw": "ddt_raw", "dt_bias": "ddt_bias", "A": "dA",
              "u": "du", "omega": "domega"}
PREP_DEV = ("x", "B", "C", "dt_raw", "dt_bias", "A", "u", "omega")


def _run_prep(inp, R, dy, dfin=None):
    d = {k: inp[k].cuda().contiguous() for k in PREP_DEV}
    g = binding.scan_bwd_prep(d["x"], d["B"], d["C"], d["dt_raw"], d["A"], d["u"], d["omega"], R,
                              dy.cuda().contiguous(), None if dfin is None else dfin.cuda().contiguous(),
                              dt_bias=d["dt_bias"])
    torch.cuda.synchronize()
    return {k: v.cpu().double().numpy() for k, v in g.items() if v is not None}


@pytest.mark.parametrize("io,Bt,H,T,P,N,R", [
    ("fp32", 1, 2, 21, 4, 4, 1),    # three chunks of 8, ragged tail
    ("fp32", 2, 1, 13, 8, 6, 4),    # chunks of 4
    ("bf16", 1, 2, 18, 4, 4, 2),
])
def test_bwd_prep_small_every_element(io, Bt, H, T, P, N, R):
    w = synth.Workload("case", Bt, H, T, P, N, R, 64, io)
    inp = synth.make_prep_inputs(w, seed=T + R)
    gen = torch.Generator().manual_seed(31)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfin = torch.randn((Bt, H, N, P), generator=gen)
    got = _run_prep(inp, R, dy, dfin)
    ref = grad.grad_fd({k: oracle.f64(inp[k]) for k in grad.PREP_INPUTS}, oracle.f64(dy), oracle.f64(dfin),
                       prep=True)
    for k, name in PREP_NAMES.items():
        err = oracle.rel_err(got[name], ref[k])
        assert err < TOL_BWD[io], f"{name}: {err:.2e}"


@pytest.mark.parametrize("io,Bt,H,T,P,N,R", [
    ("fp32", 1, 2, 150, 64, 128, 1),
    ("bf16", 2, 2, 100, 64, 64, 4),
])
def test_bwd_prep_larger_directional(io, Bt, H, T, P, N, R):
    w = synth.Workload("case", Bt, H, T, P, N, R, 64, io)
    inp = synth.make_prep_inputs(w, seed=41)
    gen = torch.Generator().manual_seed(42)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfin = torch.randn((Bt, H, N, P), generator=gen)
    got = _run_prep(inp, R, dy, dfin)
    ref = {k: oracle.f64(inp[k]) for k in grad.PREP_INPUTS}
    dy64, df64 = oracle.f64(dy), oracle.f64(dfin)
    rng = np.random.default_rng(43)
    for k in grad.PREP_INPUTS:
        d = rng.standard_normal(ref[k].shape)
        num = grad.directional(ref, k, d, dy64, df64, eps=1e-6, prep=True)
        kern = float(np.sum(got[PREP_NAMES[k]] * d))
        assert abs(kern - num) <= TOL_BWD[io] * max(1.0, abs(num)), (k, kern, num)


def test_bwd_prep_gate_outside_forward_shapes_and_bad_arguments():
    """The gate's backward needs the forward entry, which takes no P = 4; the B/C normalisation needs no
    forward and runs."""
    w = synth.Workload("case", 1, 2, 8, 4, 4, 1, 64, "fp32")
    d = {k: v.cuda() for k, v in synth.make_prep_inputs(w, seed=1).items() if k in PREP_DEV}
    dy = torch.zeros_like(d["x"])
    f = dict(dtype=torch.float32, device="cuda")
    grads = {"dx": torch.empty(d["x"].shape, **f), "dB": torch.empty(d["B"].shape, **f),
             "dC": torch.empty(d["C"].shape, **f), "ddt_raw": torch.empty(d["dt_raw"].shape, **f),
             "dA": torch.empty(d["A"].shape, **f), "du": torch.empty(d["u"].shape, **f),
             "domega": torch.empty(d["omega"].shape, **f), "ddt_bias": torch.empty((2,), **f)}
    ws = torch.empty(binding.m3_scan_bwd_prep_workspace_size(1, 8, 2, 4, 4, 1, 1), dtype=torch.uint8, device="cuda")
    args = [d[k] for k in ("x", "B", "C", "dt_raw", "A", "u", "omega")]
    ok = binding.prep_params(d["dt_bias"], None, None)
    assert binding.m3_scan_bwd_prep(*args, 1, dy, None, grads, ws, ok) == binding.M3_OK
    bc = binding.prep_params(d["dt_bias"], {"norm": True, "eps": 1e-5}, None)
    assert binding.m3_scan_bwd_prep(*args, 1, dy, None, grads, ws, bc) == binding.M3_OK
    gate = binding.prep_params(d["dt_bias"], None, torch.zeros_like(d["x"]))
    grads["dz"] = torch.empty(d["x"].shape, **f)
    assert binding.m3_scan_bwd_prep(*args, 1, dy, None, grads, ws, gate) == binding.M3_ERR_UNSUPPORTED
    assert binding.m3_scan_bwd_prep(*args, 1, dy, None, grads, ws[:64], ok) == binding.M3_ERR_WORKSPACE
    torch.cuda.synchronize()


@pytest.mark.parametrize("Bt,T", [(1, 0), (0, 5)])
def test_bwd_empty_inputs(Bt, T):
    """No tokens or no sequences: both entries succeed, dA (summed over nothing) and ddt_bias are 0,
    and the final-state seed alone has nothing to flow into."""
    w = synth.Workload("case", Bt, 2, T, 8, 8, 1, 64, "fp32")
    inp = synth.make_inputs(w, seed=0)
    g = binding.scan_bwd(*[inp[k].cuda() for k in KEYS], 1, torch.zeros(inp["x"].shape, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(g["dA"]).item() == 0 and g["dx"].numel() == 0
    pi = {k: v.cuda() for k, v in synth.make_prep_inputs(w, seed=0).items() if k in PREP_DEV}
    gp = binding.scan_bwd_prep(pi["x"], pi["B"], pi["C"], pi["dt_raw"], pi["A"], pi["u"], pi["omega"], 1,
                               torch.zeros(pi["x"].shape, device="cuda"), dt_bias=pi["dt_bias"])
    torch.cuda.synchronize()
    assert torch.count_nonzero(gp["ddt_bias"]).item() == 0 and gp["dA"].numel() == 0


# ---- through the output gate y = y_pre silu(z) (dz from the forward entry's ungated output)
TOL_DZ = {"fp32": 2e-4, "bf16": 1e-2}   # bf16: y_pre as the forward writes it, rounded to bf16


def _run_gate(inp, z, R, dy, dfin):
    d = {k: inp[k].cuda().contiguous() for k in PREP_DEV}
    g = binding.scan_bwd_prep(d["x"], d["B"], d["C"], d["dt_raw"], d["A"], d["u"], d["omega"], R,
                              dy.cuda().contiguous(), dfin.cuda().contiguous(), dt_bias=d["dt_bias"],
                              z=z.cuda().contiguous())
    torch.cuda.synchronize()
    return {k: v.cpu().double().numpy() for k, v in g.items()}


def test_bwd_gate_small_every_element():
    """fp32, P = 16 (the forward's CUDA-core path), three chunks: every gradient, dz included."""
    w = synth.Workload("case", 1, 2, 21, 16, 8, 1, 64, "fp32")
    inp = synth.make_prep_inputs(w, seed=51)
    z = synth.make_gate(tuple(inp["x"].shape), io="fp32", seed=52)
    gen = torch.Generator().manual_seed(53)
    dy = torch.randn(inp["x"].shape, generator=gen)
    dfin = torch.randn((1, 2, 8, 16), generator=gen)
    got = _run_gate(inp, z, 1, dy, dfin)
    ref_in = {k: oracle.f64(inp[k]) for k in grad.PREP_INPUTS}
    ref_in["z"] = oracle.f64(z)
    ref = grad.grad_fd(ref_in, oracle.f64(dy), oracle.f64(dfin), prep=True)
    for k, name in list(PREP_NAMES.items()) + [("z", "dz")]:
        err = oracle.rel_err(got[name], ref[k])
        assert err < TOL_BWD["fp32"], f"{name}: {err:.2e}"


@pytest.mark.parametrize("io,Bt,H,T,P,N,R", [
    ("bf16", 1, 2, 130, 64, 64, 1),    # the forward's tensor-core path
    ("fp32", 2, 1, 70, 32, 32, 2),
])
def test_bwd_gate_larger_directional(io, Bt, H, T, P, N, R):
    w = synth.Workload("case", Bt, H, T, P, N, R, 64, io)
    inp = synth.make_prep_inputs(w, seed=61)
    z = synth.make_gate(tuple(inp["x"].shape), io=io, seed=62)
    gen = torch.Generator().manual_seed(63)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfin = torch.randn((Bt, H, N, P), generator=gen)
    got = _run_gate(inp, z, R, dy, dfin)
    ref = {k: oracle.f64(inp[k]) for k in grad.PREP_INPUTS}
    ref["z"] = oracle.f64(z)
    dy64, df64 = oracle.f64(dy), oracle.f64(dfin)
    rng = np.random.default_rng(64)
    for k in grad.PREP_INPUTS + ("z",):
        d = rng.standard_normal(ref[k].shape)
        num = grad.directional(ref, k, d, dy64, df64, eps=1e-6, prep=True)
        kern = float(np.sum(got[PREP_NAMES.get(k, "dz")] * d))
        tol = TOL_DZ[io] if k == "z" else TOL_BWD[io]
        assert abs(kern - num) <= tol * max(1.0, abs(num)), (k, kern, num)


# ---- through the B / C normalisation (rows v -> v r gain + bias), alone and with the gate
BC_KEYS = ("B_gain", "C_gain", "B_bias", "C_bias")


def _bc_case(w, seed):
    inp = synth.make_prep_inputs(w, seed=seed)
    bc = synth.make_bc_params(w.heads, w.rank, w.dstate, seed=seed + 1)
    return inp, bc


def _run_bc(inp, bc, R, dy, dfin, z=None):
    d = {k: inp[k].cuda().contiguous() for k in PREP_DEV}
    bcd = {k: (v.cuda() if hasattr(v, "cuda") else v) for k, v in bc.items()}
    g = binding.scan_bwd_prep(d["x"], d["B"], d["C"], d["dt_raw"], d["A"], d["u"], d["omega"], R,
                              dy.cuda().contiguous(), dfin.cuda().contiguous(), dt_bias=d["dt_bias"], bc=bcd,
                              z=None if z is None else z.cuda().contiguous())
    torch.cuda.synchronize()
    return {k: v.cpu().double().numpy() for k, v in g.items() if v is not None}


def _bc_ref(inp, bc, z=None):
    ref = {k: oracle.f64(inp[k]) for k in grad.PREP_INPUTS}
    ref.update({k: oracle.f64(bc[k]) for k in BC_KEYS})
    ref["bc_norm"], ref["bc_eps"] = bool(bc["norm"]), float(bc["eps"])
    if z is not None:
        ref["z"] = oracle.f64(z)
    return ref


def test_bwd_bc_small_every_element():
    """fp32, three chunks, R = 2: every gradient, the gains' and the biases' included."""
    w = synth.Workload("case", 1, 2, 19, 4, 8, 2, 64, "fp32")
    inp, bc = _bc_case(w, 71)
    gen = torch.Generator().manual_seed(72)
    dy = torch.randn(inp["x"].shape, generator=gen)
    dfin = torch.randn((1, 2, 8, 4), generator=gen)
    got = _run_bc(inp, bc, 2, dy, dfin)
    ref = grad.grad_fd(_bc_ref(inp, bc), oracle.f64(dy), oracle.f64(dfin), prep=True)
    names = dict(PREP_NAMES, **{k: "d" + k for k in BC_KEYS})
    for k, name in names.items():
        err = oracle.rel_err(got[name], ref[k])
        assert err < TOL_BWD["fp32"], f"{name}: {err:.2e}"


@pytest.mark.parametrize("io,gate", [("bf16", False), ("fp32", True), ("bf16", True)])
def test_bwd_bc_bf16_and_gate_every_element(io, gate):
    """The B / C normalisation's backward with bf16 io and together with the output gate (the adjoint in
    fp32 on fp32 copies): every gradient against the oracle's, dz and the gains' and biases' included."""
    # P = 16: the gate's y_pre comes from the forward entry, whose CUDA-core path takes P >= 16
    w = synth.Workload("case", 1, 2, 19, 16, 8, 2, 64, io)
    inp, bc = _bc_case(w, 91)
    z = synth.make_gate(tuple(inp["x"].shape), io=io, seed=92) if gate else None
    gen = torch.Generator().manual_seed(93)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfin = torch.randn((1, 2, 8, 16), generator=gen)
    got = _run_bc(inp, bc, 2, dy, dfin, z=z)
    ref = grad.grad_fd(_bc_ref(inp, bc, z), oracle.f64(dy), oracle.f64(dfin), prep=True)
    names = dict(PREP_NAMES, **{k: "d" + k for k in BC_KEYS})
    if gate:
        names["z"] = "dz"
    for k, name in names.items():
        tol = TOL_DZ[io] if k == "z" else TOL_BWD[io]
        err = oracle.rel_err(got[name], ref[k])
        assert err < tol, f"{name}: {err:.2e}"


@pytest.mark.parametrize("io,gate", [("bf16", False), ("bf16", True)])
def test_bwd_bc_bf16_larger_directional(io, gate):
    """bf16, the forward's tensor-core shape (P = 64, N = 128), B / C normalisation alone and with the gate:
    inner products of the gradients with random directions against the oracle's derivatives."""
    Bt, H, T, P, N, R = 1, 4, 90, 64, 128, 1
    w = synth.Workload("case", Bt, H, T, P, N, R, 64, io)
    inp, bc = _bc_case(w, 95)
    z = synth.make_gate(tuple(inp["x"].shape), io=io, seed=96) if gate else None
    gen = torch.Generator().manual_seed(97)
    dy = torch.randn(inp["x"].shape, generator=gen).to(inp["x"].dtype)
    dfin = torch.randn((Bt, H, N, P), generator=gen)
    got = _run_bc(inp, bc, R, dy, dfin, z=z)
    ref = _bc_ref(inp, bc, z)
    dy64, df64 = oracle.f64(dy), oracle.f64(dfin)
    rng = np.random.default_rng(98)
    keys = grad.PREP_INPUTS + BC_KEYS + (("z",) if gate else ())
    for k in keys:
        d = rng.standard_normal(ref[k].shape)
        num = grad.directional(ref, k, d, dy64, df64, eps=1e-6, prep=True)
        kern = float(np.sum(got[PREP_NAMES.get(k, "dz" if k == "z" else "d" + k)] * d))
        tol = TOL_DZ[io] if k == "z" else TOL_BWD[io]
        assert abs(kern - num) <= tol * max(1.0, abs(num)), (k, kern, num)
