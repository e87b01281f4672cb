"""Pins of the finite-difference gradients of the oracle (backward-pass reference).

The finite differences are pinned against exact results that do not come from
differencing: the output is linear in x, in B and in C (for fixed other
inputs), so along those inputs the loss changes exactly by the inner product
of the gradient with the step; along C the gradient has the closed form
dL/dC_t[r, n] = sum_p h_t[n, p] dy_t[r, p] (the readout Y_t = h_t^T C_t of
section 3.3); along x it is M^T dy for the linear map M that the independent
masked-score evaluation of ``forms.matrix_form`` materialises; and along the
scalar parameters of one real pair over two steps it is the derivative of a
hand-written closed form of the exponential-trapezoidal step (Eq. 6).
"""
import math

import numpy as np
import pytest

import oracle
from oracle import forms, grad
from state_space_sequence_04_b300 import synth


def _inp(Bt=1, H=2, T=9, P=3, N=4, R=2, seed=0):
    w = synth.Workload("g", Bt, H, T, P, N, R, 8, "fp32")
    d = synth.make_inputs(w, seed=seed)
    return {k: oracle.f64(d[k]) for k in grad.INPUTS}


def _dy(inp, seed=1):
    return np.random.default_rng(seed).standard_normal(inp["x"].shape)


def test_grad_x_equals_transposed_matrix_form():
    inp = _inp(T=7, seed=3)
    dy = _dy(inp)
    g = grad.grad_fd(inp, dy, keys=("x",))["x"]
    # M x via the independent masked-score form: column i = M e_i
    x = inp["x"]
    M = np.zeros((dy.size, x.size))
    args = [inp[k] for k in grad.INPUTS]
    for i in range(x.size):
        e = np.zeros(x.size)
        e[i] = 1.0
        args[0] = e.reshape(x.shape)
        M[:, i] = forms.matrix_form(*args).reshape(-1)
    ref = (M.T @ dy.reshape(-1)).reshape(x.shape)
    assert np.max(np.abs(g - ref)) < 1e-8 * max(1.0, np.max(np.abs(ref)))


def test_grad_C_closed_form():
    inp = _inp(T=6, seed=4)
    dy = _dy(inp, seed=2)
    g = grad.grad_fd(inp, dy, keys=("C",))["C"]
    Bt, T, H, R, P = inp["x"].shape
    ref = np.zeros_like(inp["C"])
    for t in range(T):
        pre = [a[:, :t + 1] if a.ndim >= 3 else a for a in (inp[k] for k in grad.INPUTS)]
        _, h_t, _ = oracle.scan(*pre)                      # [Bt,H,N,P]
        ref[:, t] = np.einsum("bhnp,bhrp->bhrn", h_t, dy[:, t])
    assert np.max(np.abs(g - ref)) < 1e-8


@pytest.mark.parametrize("key", ["x", "B", "C"])
def test_linear_inputs_exact_inner_product(key):
    """L is linear in x, in B and in C: L(v + d) - L(v) = <dL/dv, d> exactly (and with
    a final-state seed as well)."""
    inp = _inp(T=8, seed=5)
    dy = _dy(inp, seed=6)
    dfin = np.random.default_rng(7).standard_normal((1, 2, 4, 3))
    g = grad.grad_fd(inp, dy, dfin, keys=(key,))[key]
    d = np.random.default_rng(8).standard_normal(inp[key].shape)
    l0 = grad.loss(inp, dy, dfin)
    moved = dict(inp)
    moved[key] = inp[key] + d
    assert abs(grad.loss(moved, dy, dfin) - l0 - float(np.sum(g * d))) < 1e-7


def test_two_steps_scalar_parameters_closed_form():
    """One real pair, rank 1, B = (1, 0), C = (0, 1), x0 then x1, only dy_1 = 1:
    y_1 = sin(phi_1) (alpha_1 gamma_0 + beta_1) x_0 with alpha_1 = exp(d1 a),
    beta_1 = (1 - l1) d1 alpha_1, gamma_0 = l0 d0, phi_1 = d1 w1."""
    d0, d1, a, l0, l1, w0, w1, x0, x1 = 0.4, 0.7, -0.9, 0.35, 0.6, 0.75, 1.6, 1.7, -0.6
    inp = {"x": np.array([x0, x1]).reshape(1, 2, 1, 1, 1),
           "B": np.tile(np.array([1.0, 0.0]), (1, 2, 1, 1, 1)),
           "C": np.tile(np.array([0.0, 1.0]), (1, 2, 1, 1, 1)),
           "dt": np.array([d0, d1]).reshape(1, 2, 1), "A": np.array([a]),
           "lam": np.array([l0, l1]).reshape(1, 2, 1), "omega": np.array([w0, w1]).reshape(1, 2, 1, 1)}
    dy = np.zeros((1, 2, 1, 1, 1))
    dy[0, 1] = 1.0
    g = grad.grad_fd(inp, dy, keys=("dt", "A", "lam", "omega"))
    al1 = math.exp(d1 * a)
    be1 = (1 - l1) * d1 * al1
    g0 = l0 * d0
    amp = al1 * g0 + be1
    s1, c1 = math.sin(d1 * w1), math.cos(d1 * w1)
    # derivatives of y_1 = sin(d1 w1) (al1 l0 d0 + (1 - l1) d1 al1) x0
    d_d1 = c1 * w1 * amp * x0 + s1 * (a * al1 * g0 + (1 - l1) * (al1 + d1 * a * al1)) * x0
    d_d0 = s1 * al1 * l0 * x0
    d_a = s1 * (d1 * al1 * g0 + (1 - l1) * d1 * d1 * al1) * x0
    d_l1 = s1 * (-d1 * al1) * x0
    d_l0 = s1 * al1 * d0 * x0
    d_w1 = c1 * d1 * amp * x0
    assert abs(g["dt"][0, 1, 0] - d_d1) < 1e-8 and abs(g["dt"][0, 0, 0] - d_d0) < 1e-8
    assert abs(g["A"][0] - d_a) < 1e-8
    assert abs(g["lam"][0, 1, 0] - d_l1) < 1e-8 and abs(g["lam"][0, 0, 0] - d_l0) < 1e-8
    assert abs(g["omega"][0, 1, 0, 0] - d_w1) < 1e-8 and abs(g["omega"][0, 0, 0, 0]) < 1e-8


def test_directional_matches_full_gradient():
    inp = _inp(T=7, seed=9)
    dy = _dy(inp, seed=10)
    g = grad.grad_fd(inp, dy, keys=("dt", "lam", "omega"))
    rng = np.random.default_rng(11)
    for k in ("dt", "lam", "omega"):
        v = rng.standard_normal(inp[k].shape)
        assert abs(grad.directional(inp, k, v, dy) - float(np.sum(g[k] * v))) < 1e-7


# ---- pre-activation inputs (Delta = softplus(dt_raw + dt_bias), lambda = sigmoid(u), A per token)
def _prep_inp(T=7, seed=21):
    w = synth.Workload("gp", 1, 2, T, 3, 4, 2, 8, "fp32")
    d = synth.make_prep_inputs(w, seed=seed)
    return {k: oracle.f64(d[k]) for k in grad.PREP_INPUTS}


def _plain_of(pi):
    """The plain inputs the pre-activations stand for (Delta, lambda evaluated, A per token)."""
    d, lam = oracle.prep(pi["dt_raw"], pi["dt_bias"], pi["u"])
    return {"x": pi["x"], "B": pi["B"], "C": pi["C"], "dt": d, "A": pi["A"], "lam": lam, "omega": pi["omega"]}


def test_prep_chain_rule_through_softplus_and_sigmoid():
    """dL/d dt_raw = dL/dDelta * sigmoid(z) (softplus' = sigmoid) and dL/du = dL/dlambda * lambda (1 - lambda),
    with dL/dDelta, dL/dlambda the (separately pinned) gradients of the plain recurrence at the same point;
    dL/d dt_bias[h] sums dL/d dt_raw over batch and tokens; the per-token dA equals the plain one."""
    pi = _prep_inp()
    dy = _dy(pi, seed=22)
    gp = grad.grad_fd(pi, dy, keys=("dt_raw", "dt_bias", "A", "u"), prep=True)
    pl = _plain_of(pi)
    g = grad.grad_fd(pl, dy, keys=("dt", "lam", "A"))
    z = pi["dt_raw"] + pi["dt_bias"]
    assert np.max(np.abs(gp["dt_raw"] - g["dt"] * oracle.sigmoid(z))) < 1e-7
    lam = pl["lam"]
    assert np.max(np.abs(gp["u"] - g["lam"] * lam * (1.0 - lam))) < 1e-7
    assert np.max(np.abs(gp["dt_bias"] - gp["dt_raw"].sum(axis=(0, 1)))) < 1e-7
    assert np.max(np.abs(gp["A"] - g["A"])) < 1e-7


def test_per_token_A_gradient_sums_to_the_per_head_one():
    """With A_t = A_h for every token, the per-token gradients summed over batch and tokens are the
    gradient with respect to the per-head generator."""
    inp = _inp(T=8, seed=23)
    dy = _dy(inp, seed=24)
    g_head = grad.grad_fd(inp, dy, keys=("A",))["A"]
    tok = dict(inp)
    tok["A"] = np.broadcast_to(inp["A"], inp["dt"].shape).copy()
    g_tok = grad.grad_fd(tok, dy, keys=("A",))["A"]
    assert np.max(np.abs(g_tok.sum(axis=(0, 1)) - g_head)) < 1e-7


def test_gate_gradients_closed_form_and_reduction():
    """Output gate y = y_pre * silu(z): dL/dz = dy * y_pre * silu'(z) with y_pre the ungated output and
    silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z))); every other gradient equals the ungated one for the
    seed dy * silu(z) (the loss is linear in dy)."""
    pi = _prep_inp(T=6, seed=25)
    rng = np.random.default_rng(26)
    z = rng.standard_normal(pi["x"].shape)
    dy = _dy(pi, seed=27)
    gated = dict(pi)
    gated["z"] = z
    g = grad.grad_fd(gated, dy, prep=True)
    y_pre, _, _ = oracle.scan_prep(*[pi[k] for k in grad.PREP_INPUTS])
    s = oracle.sigmoid(z)
    assert np.max(np.abs(g["z"] - dy * y_pre * s * (1.0 + z * (1.0 - s)))) < 1e-7
    g0 = grad.grad_fd(pi, dy * oracle.silu(z), prep=True)
    for k in grad.PREP_INPUTS:
        assert np.max(np.abs(g[k] - g0[k])) < 1e-7, k


# ---- through the B / C normalisation (section 3.4): rows v -> v r gain + bias, r = (mean(v^2) + eps)^(-1/2)
def _bc_inp(T=6, seed=29, eps=1e-5):
    pi = _prep_inp(T=T, seed=seed)
    bc = synth.make_bc_params(2, 2, 4, seed=seed + 1)
    pi.update({k: oracle.f64(bc[k]) for k in grad.BC_INPUTS})
    pi["bc_norm"], pi["bc_eps"] = True, eps
    return pi


def test_bc_gradients_against_the_normalised_rows():
    """With dn = dL/d(normalised B) from the plain recurrence run on the normalised rows: dB_bias sums dn
    over batch and tokens, dB_gain sums dn v r over every row, and dB = r (gain dn) - v r^3 / N
    sum(gain dn v) (the Jacobian of v -> v r gain, written out); the same for C."""
    pi = _bc_inp()
    dy = _dy(pi, seed=30)
    g = grad.grad_fd(pi, dy, prep=True)
    d, lam = oracle.prep(pi["dt_raw"], pi["dt_bias"], pi["u"])
    Bn = oracle.bc_prep(pi["B"], True, pi["bc_eps"], pi["B_gain"], pi["B_bias"])
    Cn = oracle.bc_prep(pi["C"], True, pi["bc_eps"], pi["C_gain"], pi["C_bias"])
    plain = {"x": pi["x"], "B": Bn, "C": Cn, "dt": d, "A": pi["A"], "lam": lam, "omega": pi["omega"]}
    gp = grad.grad_fd(plain, dy, keys=("B", "C"))
    N = pi["B"].shape[-1]
    for V, key in (("B", "B"), ("C", "C")):
        v, dn, gain = pi[V], gp[key], pi[V + "_gain"]
        r = 1.0 / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + pi["bc_eps"])
        assert np.max(np.abs(g[V + "_bias"] - dn.sum(axis=(0, 1)))) < 1e-6
        assert np.max(np.abs(g[V + "_gain"] - (dn * v * r).sum(axis=(0, 1, 2, 3)))) < 1e-6
        gd = gain * dn
        dv = r * gd - v * r ** 3 / N * np.sum(gd * v, axis=-1, keepdims=True)
        assert np.max(np.abs(g[V] - dv)) < 1e-6


def test_bc_normalisation_is_scale_invariant():
    """With eps = 0 the normalised rows do not change when a row is scaled, so every raw row's gradient is
    orthogonal to the row."""
    pi = _bc_inp(eps=0.0)
    g = grad.grad_fd(pi, _dy(pi, seed=31), prep=True, keys=("B", "C"))
    for V in ("B", "C"):
        assert np.max(np.abs(np.sum(g[V] * pi[V], axis=-1))) < 1e-7


@pytest.mark.parametrize("T,P,N,R,seed", [(9, 3, 4, 2, 41), (7, 4, 6, 1, 42), (5, 2, 8, 3, 43)])
@pytest.mark.parametrize("with_final", [False, True])
def test_adjoint_equals_finite_differences(T, P, N, R, seed, with_final):
    """The step-by-step adjoint and the central differences of the recurrence agree to rounding."""
    w = synth.Workload("g", 1, 2, T, P, N, R, 8, "fp32")
    d = synth.make_inputs(w, seed=seed)
    inp = {k: oracle.f64(d[k]) for k in grad.INPUTS}
    dy = _dy(inp, seed=seed + 1)
    dfin = np.random.default_rng(seed + 2).standard_normal((1, 2, N, P)) if with_final else None
    a = grad.adjoint(inp, dy, dfin)
    g = grad.grad_fd(inp, dy, dfin)
    for k in grad.INPUTS:
        assert np.max(np.abs(a[k] - g[k])) < 1e-6 * max(1.0, np.max(np.abs(g[k]))), k
