"""Pins of the oracle's per-token path: A_t per token, Delta and lambda from
their pre-activations.

The time-varying discretizations of "Mamba-3: Improved Sequence Modeling using
State Space Principles" take a decay generator per token, exp(Delta_t A_t)
(thelatestinai.com/papers/2603.15569, Table 1), and the default lambda
parameterisation of the appendix ablation table is lambda_t = sigmoid(u_t);
Delta_t = softplus(dt_raw_t + dt_bias_h) is the Mamba family's
parameterisation (the pages leave it open).  B and C may also be
RMS-normalised over N and shifted by per-head channel biases before the
rotation (section 3.4).  Each test compares the oracle with something other
than itself: the independent numpy evaluations of ``oracle.forms`` (which take
the decay generator per token), hand-derived closed forms, identities of
softplus and sigmoid, invariances of the normalisation and the linearity of the
readout in C; planted mistakes in the normalisation fail these pins.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import forms
from state_space_sequence_04_b300 import synth


def _prep_inputs(Bt=2, H=3, T=29, P=5, N=6, R=2, seed=0, **kw):
    w = synth.Workload("small_prep", Bt, H, T, P, N, R, 8, "fp32", **kw)
    inp = synth.make_prep_inputs(w, seed=seed)
    f = oracle.f64
    d, lam = oracle.prep(inp["dt_raw"], inp["dt_bias"], inp["u"])
    return {"x": f(inp["x"]), "B": f(inp["B"]), "C": f(inp["C"]), "dt": d, "A": f(inp["A"]), "lam": lam,
            "omega": f(inp["omega"]), "raw": inp}


def _args(inp):
    return [inp[k] for k in ("x", "B", "C", "dt", "A", "lam", "omega")]


# ---------------------------------------------------------------------------
# softplus and sigmoid against closed forms and identities
def test_softplus_sigmoid_identities():
    z = np.linspace(-30.0, 30.0, 241)
    sp, sg = oracle.softplus(z), oracle.sigmoid(z)
    assert abs(oracle.softplus(0.0) - math.log(2.0)) < 1e-16
    assert abs(oracle.sigmoid(0.0) - 0.5) == 0.0
    assert abs(oracle.sigmoid(math.log(3.0)) - 0.75) < 1e-15            # 1 / (1 + 1/3)
    assert abs(oracle.softplus(math.log(math.e - 1.0)) - 1.0) < 1e-15   # log(1 + e - 1) = 1
    assert np.max(np.abs(sp - oracle.softplus(-z) - z)) < 1e-13          # softplus(z) - softplus(-z) = z
    assert np.max(np.abs(sg + oracle.sigmoid(-z) - 1.0)) < 1e-15         # sigma(u) + sigma(-u) = 1
    eps = 1e-6                                                           # softplus' = sigmoid
    dsp = (oracle.softplus(z + eps) - oracle.softplus(z - eps)) / (2 * eps)
    assert np.max(np.abs(dsp - sg)) < 1e-8
    assert np.all(sp > 0) and np.all((sg > 0) & (sg < 1))
    # no overflow far out: softplus(z) -> z, sigmoid -> 0 / 1
    assert oracle.softplus(800.0) == 800.0 and oracle.sigmoid(-800.0) == 0.0 and oracle.sigmoid(800.0) == 1.0


def test_prep_is_softplus_of_biased_raw_and_sigmoid():
    inp = _prep_inputs(T=7)
    raw = inp["raw"]
    dr, bias, u = (oracle.f64(raw[k]) for k in ("dt_raw", "dt_bias", "u"))
    d, lam = oracle.prep(dr, bias, u)
    for b, t, h in [(0, 0, 0), (1, 6, 2), (0, 3, 1)]:
        z = dr[b, t, h] + bias[h]
        assert abs(d[b, t, h] - math.log1p(math.exp(z))) < 1e-15
        assert abs(lam[b, t, h] - 1.0 / (1.0 + math.exp(-u[b, t, h]))) < 1e-15
    d0, _ = oracle.prep(dr, None, u)
    assert abs(d0[1, 2, 0] - math.log1p(math.exp(dr[1, 2, 0]))) < 1e-15


# ---------------------------------------------------------------------------
# per-token decay generator: the oracle against the independent evaluations
def test_mamba2_reduction_per_token_A():
    inp = _prep_inputs(R=1, T=50)
    inp["lam"] = np.ones_like(inp["lam"])
    inp["omega"] = np.zeros_like(inp["omega"])
    y, _, _ = oracle.scan(*_args(inp))
    ref = forms.mamba2_euler(inp["x"], inp["B"], inp["C"], inp["dt"], inp["A"])
    assert oracle.rel_err(y, ref) < 1e-13


@pytest.mark.parametrize("T,R", [(17, 1), (33, 3)])
def test_matrix_form_per_token_A(T, R):
    inp = _prep_inputs(T=T, R=R, seed=T)
    y, _, _ = oracle.scan(*_args(inp))
    assert oracle.rel_err(forms.matrix_form(*_args(inp)), y) < 1e-12


@pytest.mark.parametrize("R", [1, 2])
def test_complex_and_rotating_frame_per_token_A(R):
    inp = _prep_inputs(T=31, R=R, seed=5 + R)
    y, _, _ = oracle.scan(*_args(inp))
    assert oracle.rel_err(forms.complex_form(*_args(inp)), y) < 1e-12
    assert oracle.rel_err(forms.rotating_frame(*_args(inp)), y) < 1e-12


@pytest.mark.parametrize("Q", [1, 5, 16, 64])
def test_chunked_per_token_A(Q):
    inp = _prep_inputs(T=70, R=2, seed=11)
    y, hT, _ = oracle.scan(*_args(inp))
    yc, fc = forms.chunked(*_args(inp), Q)
    assert oracle.rel_err(yc, y) < 1e-12
    assert oracle.rel_err(fc, hT) < 1e-12


def test_closed_form_two_steps_per_token_A():
    """One real pair, rank 1, B = (1, 0), C = (0, 1), x0 then x1; the second
    step decays with its own A_1: h_1 = R(p1)((al1 g0 + be1) x0 e1) + g1 x1 e1,
    al1 = exp(d1 A_1), be1 = (1 - l1) d1 al1."""
    d0, d1, a0, a1, l0, l1, p0, p1, x0, x1 = 0.4, 0.7, -0.3, -2.1, 0.35, 0.6, 0.3, 1.1, 1.7, -0.6
    x = np.array([x0, x1]).reshape(1, 2, 1, 1, 1)
    B = np.zeros((1, 2, 1, 1, 2))
    B[..., 0] = 1.0
    C = np.zeros((1, 2, 1, 1, 2))
    C[..., 1] = 1.0
    dt = np.array([d0, d1]).reshape(1, 2, 1)
    A = np.array([a0, a1]).reshape(1, 2, 1)
    lam = np.array([l0, l1]).reshape(1, 2, 1)
    om = np.array([p0 / d0, p1 / d1]).reshape(1, 2, 1, 1)
    y, h, _ = oracle.scan(x, B, C, dt, A, lam, om)
    al1 = math.exp(d1 * a1)
    be1 = (1 - l1) * d1 * al1
    g0, g1 = l0 * d0, l1 * d1
    amp = (al1 * g0 + be1) * x0
    assert abs(y[0, 1, 0, 0, 0] - amp * math.sin(p1)) < 1e-14
    assert abs(h[0, 0, 0, 0] - (amp * math.cos(p1) + g1 * x1)) < 1e-14
    # the first token's generator does not enter the second step's decay
    A2 = A.copy()
    A2[0, 0, 0] = -7.0
    y2, _, _ = oracle.scan(x, B, C, dt, A2, lam, om)
    assert abs(y2[0, 1, 0, 0, 0] - y[0, 1, 0, 0, 0]) < 1e-15


def test_per_head_A_is_constant_per_token_A():
    inp = _prep_inputs(T=23, seed=3)
    Ah = -np.exp(np.linspace(0.0, math.log(16.0), 3))
    a = _args(inp)
    a[4] = Ah
    y1, h1, _ = oracle.scan(*a)
    a[4] = np.broadcast_to(Ah, inp["dt"].shape).copy()
    y2, h2, _ = oracle.scan(*a)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)


def test_scan_prep_equals_scan_on_prepared_values():
    inp = _prep_inputs(T=19, seed=4)
    raw = inp["raw"]
    y, h, _ = oracle.scan_prep(raw["x"], raw["B"], raw["C"], raw["dt_raw"], raw["dt_bias"], raw["A"],
                               raw["u"], raw["omega"])
    dr, bias, u = (oracle.f64(raw[k]) for k in ("dt_raw", "dt_bias", "u"))
    d = np.vectorize(lambda z: math.log1p(math.exp(z)))(dr + bias)
    lam = np.vectorize(lambda v: 1.0 / (1.0 + math.exp(-v)))(u)
    y2, h2, _ = oracle.scan(inp["x"], inp["B"], inp["C"], d, inp["A"], lam, inp["omega"])
    assert oracle.rel_err(y, y2) < 1e-14 and oracle.rel_err(h, h2) < 1e-14


def test_continuation_prefill_then_decode_prep():
    """Prefill of T0 tokens, then single-token steps on pre-activations, equals
    the prefill of all tokens."""
    inp = _prep_inputs(R=2, T=40, seed=9)
    raw = {k: oracle.f64(v) for k, v in inp["raw"].items() if hasattr(v, "shape")}
    keys = ("x", "B", "C", "dt_raw", "A", "u", "omega")
    yfull, hfull, _ = oracle.scan_prep(*[raw[k] for k in keys[:4]], raw["dt_bias"], raw["A"], raw["u"], raw["omega"])
    T0 = 29
    pre = {k: raw[k][:, :T0] for k in keys}
    _, h, prev = oracle.scan_prep(pre["x"], pre["B"], pre["C"], pre["dt_raw"], raw["dt_bias"], pre["A"], pre["u"],
                                  pre["omega"])
    for t in range(T0, 40):
        yt, h, prev = oracle.decode_step_prep(h, raw["x"][:, t], raw["B"][:, t], prev, raw["C"][:, t],
                                              raw["dt_raw"][:, t], raw["dt_bias"], raw["A"][:, t], raw["u"][:, t],
                                              raw["omega"][:, t])
        assert oracle.rel_err(yt, yfull[:, t]) < 1e-13
    assert oracle.rel_err(h, hfull) < 1e-13


def test_large_u_removes_delayed_write():
    """u -> +inf gives lambda = 1: no dependence on x_{t-1} through the delayed write
    (the lambda = 1 case of the exponential-trapezoidal rule, section 2.2)."""
    inp = _prep_inputs(T=12, R=1, seed=6)
    raw = inp["raw"]
    u = np.full(oracle.f64(raw["u"]).shape, 60.0)
    y, _, _ = oracle.scan_prep(raw["x"], raw["B"], raw["C"], raw["dt_raw"], raw["dt_bias"], raw["A"], u, raw["omega"])
    ref = forms.complex_form(inp["x"], inp["B"], inp["C"], inp["dt"], inp["A"], np.ones_like(inp["lam"]), inp["omega"])
    assert oracle.rel_err(y, ref) < 1e-12


# ---------------------------------------------------------------------------
# B / C normalisation and head-specific channel biases (section 3.4), applied
# to every (token, rank) row over the state dimension N before the rotation
def test_bc_prep_closed_form():
    v = np.array([3.0, 4.0]).reshape(1, 1, 1, 1, 2)        # one row, N = 2
    out = oracle.bc_prep(v, norm=True, eps=0.0, gain=np.array([2.0, 0.5]), bias=np.array([1.0, -1.0]).reshape(1, 1, 2))
    r = math.sqrt((9.0 + 16.0) / 2.0)
    assert abs(out[0, 0, 0, 0, 0] - (2.0 * 3.0 / r + 1.0)) < 1e-15
    assert abs(out[0, 0, 0, 0, 1] - (0.5 * 4.0 / r - 1.0)) < 1e-15
    # eps enters the mean square; without the norm only the bias is added
    out = oracle.bc_prep(v, norm=True, eps=0.5)
    assert abs(out[0, 0, 0, 0, 0] - 3.0 / math.sqrt(12.5 + 0.5)) < 1e-15
    out = oracle.bc_prep(v, norm=False, bias=np.array([1.0, -1.0]).reshape(1, 1, 2))
    assert np.array_equal(out.ravel(), [4.0, 3.0])


def test_bc_norm_rows_have_unit_rms():
    inp = _prep_inputs(T=9, R=3, N=8, seed=2)
    Bn = oracle.bc_prep(inp["B"], norm=True, eps=0.0)
    assert np.max(np.abs(np.mean(Bn * Bn, axis=-1) - 1.0)) < 1e-14


def _scan_bc(inp, B, C, bc):
    raw = inp["raw"]
    return oracle.scan_prep(inp["x"], B, C, raw["dt_raw"], raw["dt_bias"], raw["A"], raw["u"], raw["omega"], bc=bc)


def test_bc_norm_scale_invariance():
    """With the norm on (eps = 0, no bias) rescaling each row of B and C changes nothing."""
    inp = _prep_inputs(T=21, R=2, seed=12)
    bc = {"norm": True, "eps": 0.0}
    y1, h1, _ = _scan_bc(inp, inp["B"], inp["C"], bc)
    sB = np.exp(np.random.default_rng(0).standard_normal(inp["B"].shape[:-1]))[..., None]
    y2, h2, _ = _scan_bc(inp, inp["B"] * sB, inp["C"] * 0.2, bc)
    assert oracle.rel_err(y2, y1) < 1e-12 and oracle.rel_err(h2, h1) < 1e-12


def test_bc_bias_enters_the_readout_linearly():
    """y_t = h_t^T C_t is linear in C_t: a C bias b adds exactly the output of C = b."""
    inp = _prep_inputs(T=17, R=2, seed=13)
    Bt, T, H, R, N = inp["C"].shape
    b = 0.3 * np.random.default_rng(1).standard_normal((H, R, N))
    y_b, _, _ = _scan_bc(inp, inp["B"], inp["C"], {"C_bias": b})
    y_0, _, _ = _scan_bc(inp, inp["B"], inp["C"], None)
    y_only, _, _ = _scan_bc(inp, inp["B"], np.zeros_like(inp["C"]), {"C_bias": b})
    assert oracle.rel_err(y_b, y_0 + y_only) < 1e-12


def test_bc_gain_scales_the_readout():
    inp = _prep_inputs(T=15, R=1, seed=14)
    N = inp["C"].shape[-1]
    y1, _, _ = _scan_bc(inp, inp["B"], inp["C"], {"norm": True, "eps": 1e-5})
    y2, _, _ = _scan_bc(inp, inp["B"], inp["C"], {"norm": True, "eps": 1e-5, "C_gain": np.full(N, 2.5)})
    assert oracle.rel_err(y2, 2.5 * y1) < 1e-13


def test_continuation_with_bc():
    """Prefill then decode with the B / C normalisation and biases; the cache holds raw B, X."""
    inp = _prep_inputs(R=2, T=36, N=6, seed=15)
    raw = {k: oracle.f64(v) for k, v in inp["raw"].items() if hasattr(v, "shape")}
    bcp = synth.make_bc_params(3, 2, 6, seed=3)
    bc = {k: (oracle.f64(v) if hasattr(v, "shape") else v) for k, v in bcp.items()}
    yfull, hfull, _ = oracle.scan_prep(raw["x"], raw["B"], raw["C"], raw["dt_raw"], raw["dt_bias"], raw["A"],
                                       raw["u"], raw["omega"], bc=bc)
    T0 = 27
    _, h, prev = oracle.scan_prep(raw["x"][:, :T0], raw["B"][:, :T0], raw["C"][:, :T0], raw["dt_raw"][:, :T0],
                                  raw["dt_bias"], raw["A"][:, :T0], raw["u"][:, :T0], raw["omega"][:, :T0], bc=bc)
    assert np.array_equal(prev[..., :2 * 6].reshape(raw["B"][:, T0 - 1].shape), raw["B"][:, T0 - 1])
    for t in range(T0, 36):
        yt, h, prev = oracle.decode_step_prep(h, raw["x"][:, t], raw["B"][:, t], prev, raw["C"][:, t],
                                              raw["dt_raw"][:, t], raw["dt_bias"], raw["A"][:, t], raw["u"][:, t],
                                              raw["omega"][:, t], bc=bc)
        assert oracle.rel_err(yt, yfull[:, t]) < 1e-13
    assert oracle.rel_err(h, hfull) < 1e-13


BC_PINS = [test_bc_prep_closed_form, test_bc_norm_rows_have_unit_rms, test_bc_norm_scale_invariance,
           test_bc_bias_enters_the_readout_linearly, test_bc_gain_scales_the_readout]


def _mut_axis(V, norm=False, eps=0.0, gain=None, bias=None):
    V = oracle.f64(V)
    if norm:
        V = V / np.sqrt(np.mean(V * V, axis=-2, keepdims=True) + eps)   # over the ranks, not N
        if gain is not None:
            V = V * oracle.f64(gain)
    return V if bias is None else V + oracle.f64(bias)


def _mut_bias_first(V, norm=False, eps=0.0, gain=None, bias=None):
    V = oracle.f64(V)
    if bias is not None:
        V = V + oracle.f64(bias)
    if norm:
        V = V / np.sqrt(np.mean(V * V, axis=-1, keepdims=True) + eps)
        if gain is not None:
            V = V * oracle.f64(gain)
    return V


def _mut_gain_after_bias(V, norm=False, eps=0.0, gain=None, bias=None):
    V = oracle.f64(V)
    if norm:
        V = V / np.sqrt(np.mean(V * V, axis=-1, keepdims=True) + eps)
    if bias is not None:
        V = V + oracle.f64(bias)
    if norm and gain is not None:
        V = V * oracle.f64(gain)
    return V


def _mut_no_eps(V, norm=False, eps=0.0, gain=None, bias=None):
    V = oracle.f64(V)
    if norm:
        V = V / np.sqrt(np.mean(V * V, axis=-1, keepdims=True))
        if gain is not None:
            V = V * oracle.f64(gain)
    return V if bias is None else V + oracle.f64(bias)


@pytest.mark.parametrize("mutant", [_mut_axis, _mut_bias_first, _mut_gain_after_bias, _mut_no_eps])
def test_bc_mutants_fail_a_pin(mutant, monkeypatch):
    monkeypatch.setattr(oracle, "bc_prep", mutant)
    failed = 0
    for pin in BC_PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0


# ---------------------------------------------------------------------------
# output gate y * silu(z)
def test_silu_closed_forms():
    z = np.linspace(-20.0, 20.0, 81)
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert np.max(np.abs(oracle.silu(z) - oracle.silu(-z) - z)) < 1e-13      # silu(z) - silu(-z) = z
    assert np.max(np.abs(oracle.silu(z) - z * oracle.sigmoid(z))) == 0.0
    assert abs(oracle.silu(-800.0)) == 0.0 and oracle.silu(800.0) == 800.0


def test_gate_multiplies_each_output_element():
    """The gate acts elementwise on y and leaves the state alone: with z = 0 the output
    vanishes, with a positive constant z = c it is y * silu(c)."""
    inp = _prep_inputs(T=13, R=2, seed=16)
    raw = inp["raw"]
    args = [raw[k] for k in ("x", "B", "C", "dt_raw", "dt_bias", "A", "u", "omega")]
    y, h, _ = oracle.scan_prep(*args)
    y0, h0, _ = oracle.scan_prep(*args, z=np.zeros(y.shape))
    assert np.max(np.abs(y0)) == 0.0 and np.array_equal(h0, h)
    yc, _, _ = oracle.scan_prep(*args, z=np.full(y.shape, 0.7))
    assert oracle.rel_err(yc, y * (0.7 / (1.0 + math.exp(-0.7)))) < 1e-14
    zz = np.random.default_rng(2).standard_normal(y.shape)
    yz, _, _ = oracle.scan_prep(*args, z=zz)
    assert oracle.rel_err(yz, y * zz / (1.0 + np.exp(-zz))) < 1e-14
