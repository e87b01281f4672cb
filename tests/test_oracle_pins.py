"""Pins of the float64 oracle against what the pages and mathematics fix.

Sources are the pages on "Mamba-3: Improved Sequence Modeling using State Space
Principles" (abhik.ai/papers/mamba3 sections 2.2, 3.1-3.4, Propositions 1-4,
Eqs. 6, 7, 11-14 and panels 1-5; thelatestinai.com/papers/2603.15569 Tables 1-2).
Each test compares the sequential C oracle with something other than itself:
an independent evaluation of the same recurrence, a hand-derived closed form,
a construction printed on a page, or an invariant.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import forms
from state_space_sequence_04_b300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _args(inp):
    return [inp[k] for k in ("x", "B", "C", "dt", "A", "lam", "omega")]


def _small(Bt=2, H=3, T=29, P=5, N=6, R=2, seed=0, io="fp32", **kw):
    w = synth.Workload("small", Bt, H, T, P, N, R, 8, io, **kw)
    return synth.make_inputs(w, seed=seed)


def _f(a):
    return oracle.f64(a)


# ---------------------------------------------------------------------------
# Check 1: lambda = 1, omega = 0, R = 1 is Mamba-2's exponential-Euler update
# (page 2 Table 1 "Exponential-Euler" row; page 4 section 2.2 and panel 1).
def test_mamba2_reduction():
    inp = _small(R=1, T=50)
    inp["lam"] = torch.ones_like(inp["lam"])
    inp["omega"] = torch.zeros_like(inp["omega"])
    y, _, _ = oracle.scan(*_args(inp))
    ref = forms.mamba2_euler(inp["x"], inp["B"], inp["C"], inp["dt"], inp["A"])
    assert oracle.rel_err(y, ref) < 1e-13


# ---------------------------------------------------------------------------
# Check 2: decay x two-band mask matrix form (page 4 sections 3.1.2-3.1.3,
# Eq. 7; page 2 Figure 1), materialised for T <= 64, equals the scan.
@pytest.mark.parametrize("T,R", [(1, 1), (17, 1), (64, 1), (33, 3), (64, 4)])
def test_matrix_form_equals_scan(T, R):
    inp = _small(T=T, R=R, seed=T + R)
    y, _, _ = oracle.scan(*_args(inp))
    ym = forms.matrix_form(*_args(inp))
    assert oracle.rel_err(ym, y) < 1e-12


def test_two_band_constant_coefficients_match_closed_form():
    # page 4 panel 2: L_ts = gamma alpha^(t-s) + [s<t] beta alpha^(t-s-1)
    T, d, a, lam = 12, 0.37, -1.3, 0.3
    L = forms.two_band_matrix(np.full(T, d), a, np.full(T, lam))
    Lc = forms.two_band_closed_form(T, d, a, lam)
    assert np.max(np.abs(L - Lc)) < 1e-15
    # and the scan itself, with one real pair, B = C = (1, 0), no rotation and
    # constant coefficients, is y = L x (the page's scalar setting).
    Bt, H, P, N, R = 1, 1, 1, 2, 1
    rng = np.random.default_rng(3)
    x = rng.standard_normal((Bt, T, H, R, P))
    B = np.zeros((Bt, T, H, R, N)); B[..., 0] = 1.0
    C = B.copy()
    dt = np.full((Bt, T, H), d)
    lamv = np.full((Bt, T, H), lam)
    om = np.zeros((Bt, T, H, N // 2))
    y, _, _ = oracle.scan(x, B, C, dt, np.array([a]), lamv, om)
    assert np.max(np.abs(y[0, :, 0, 0, 0] - Lc @ x[0, :, 0, 0, 0])) < 1e-14


# ---------------------------------------------------------------------------
# Check 3: complex-diagonal state (Proposition 2, incl. the conjugated C
# readout) and the rotating-frame form (Propositions 3-4, Eq. 11).
@pytest.mark.parametrize("R", [1, 2, 4])
def test_complex_and_rotating_frame_equal_scan(R):
    inp = _small(R=R, T=41, seed=10 + R)
    y, _, _ = oracle.scan(*_args(inp))
    assert oracle.rel_err(forms.complex_form(*_args(inp)), y) < 1e-12
    assert oracle.rel_err(forms.rotating_frame(*_args(inp)), y) < 1e-12


def test_delayed_write_keeps_its_own_phase():
    """Rotating the delayed write with the current phase (the mistake Eq. 11
    warns about) must NOT reproduce the scan; the correct frame does."""
    inp = _small(R=1, T=20, seed=5)
    x, B, C, dt, A, lam, om = (_f(v) for v in _args(inp))
    y, _, _ = oracle.scan(x, B, C, dt, A, lam, om)
    alpha, beta, gamma = forms.coefficients(dt, A, lam)
    Phi = np.cumsum(dt[..., None] * om, axis=1)
    Bt, T, H, R, P = x.shape
    N = B.shape[-1]
    hs = np.zeros((Bt, H, N, P))
    raw_prev = np.zeros((Bt, H, R, N)); x_prev = np.zeros((Bt, H, R, P))
    wrong = np.zeros_like(y)
    for t in range(T):
        rot = lambda v: forms.rotate_pairs(v, -Phi[:, t, :, None, :])
        v = np.einsum("bhrn,bhrp->bhnp", rot(B[:, t]), x[:, t])
        vprev_wrong = np.einsum("bhrn,bhrp->bhnp", rot(raw_prev), x_prev)
        hs = (alpha[:, t, :, None, None] * hs + beta[:, t, :, None, None] * vprev_wrong
              + gamma[:, t, :, None, None] * v)
        wrong[:, t] = np.einsum("bhnp,bhrn->bhrp", hs, rot(C[:, t]))
        raw_prev, x_prev = B[:, t], x[:, t]
    assert oracle.rel_err(wrong, y) > 1e-3


# ---------------------------------------------------------------------------
# Check 4: chunked evaluation (section 3.3) equals sequential for every chunk
# length, including lengths that do not divide T.
def test_chunked_equals_sequential_every_chunk():
    inp = _small(Bt=1, H=1, T=67, P=3, N=4, R=2, seed=7)
    y, hT, _ = oracle.scan(*_args(inp))
    for Q in range(1, 68):
        yq, fq = forms.chunked(*_args(inp), Q)
        assert oracle.rel_err(yq, y) < 1e-12, Q
        assert oracle.rel_err(fq, hT) < 1e-12, Q


@pytest.mark.parametrize("Q", [16, 64, 100, 256])
def test_chunked_equals_sequential_T256(Q):
    inp = _small(Bt=1, H=2, T=256, P=4, N=8, R=1, seed=8)
    y, hT, _ = oracle.scan(*_args(inp))
    yq, fq = forms.chunked(*_args(inp), Q)
    assert oracle.rel_err(yq, y) < 1e-12
    assert oracle.rel_err(fq, hT) < 1e-12


# ---------------------------------------------------------------------------
# Hand-derived closed forms for T <= 3 with one real pair (N = 2), P = R = 1.
# They fix the rotation direction, which coefficient multiplies which write,
# and that the delayed write is rotated with the state (page 4 panel 3).
def _one_pair(xs, bs, cs, ds, a, lams, phis):
    T = len(xs)
    x = np.array(xs, float).reshape(1, T, 1, 1, 1)
    B = np.array(bs, float).reshape(1, T, 1, 1, 2)
    C = np.array(cs, float).reshape(1, T, 1, 1, 2)
    dt = np.array(ds, float).reshape(1, T, 1)
    lam = np.array(lams, float).reshape(1, T, 1)
    om = (np.array(phis, float) / np.array(ds, float)).reshape(1, T, 1, 1)
    y, hT, _ = oracle.scan(x, B, C, dt, np.array([a]), lam, om)
    return y[0, :, 0, 0, 0], hT[0, 0, :, 0]


def test_closed_form_two_steps():
    d0, d1, a, l0, l1, p0, p1, x0, x1 = 0.4, 0.7, -0.9, 0.35, 0.6, 0.3, 1.1, 1.7, -0.6
    al1 = math.exp(d1 * a)
    be1 = (1 - l1) * d1 * al1
    g0, g1 = l0 * d0, l1 * d1
    # B = (1, 0) at both steps; read the second coordinate with C = (0, 1)
    y, h = _one_pair([x0, x1], [(1, 0), (1, 0)], [(0, 1), (0, 1)], [d0, d1], a, [l0, l1], [p0, p1])
    # h_0 = g0 x0 (1, 0) (the initial zero state's rotation is irrelevant)
    assert abs(y[0] - 0.0) < 1e-15
    # h_1 = R(p1)((al1 g0 + be1) x0 (1,0)) + g1 x1 (1, 0)
    amp = (al1 * g0 + be1) * x0
    assert abs(y[1] - amp * math.sin(p1)) < 1e-14
    assert abs(h[0] - (amp * math.cos(p1) + g1 * x1)) < 1e-14
    assert abs(h[1] - amp * math.sin(p1)) < 1e-14


def test_closed_form_three_steps_delayed_term_rotation():
    # Only the t=0 write is nonzero and lambda_0 = 1, lambda_1 = 0.25,
    # lambda_2 = 0.5.  h_2 = R(p2)(al2 R(p1)(al1 g0 + be1) x0 e1) + ... the
    # delayed write of t=1 is zero because x_1 = 0.
    d, a, p0, p1, p2, x0 = 0.5, -0.4, 0.2, -0.7, 0.45, 2.0
    ls = [1.0, 0.25, 0.5]
    al = math.exp(d * a)
    be1 = (1 - ls[1]) * d * al
    g0 = ls[0] * d
    y, h = _one_pair([x0, 0.0, 0.0], [(1, 0)] * 3, [(1, 0)] * 3, [d] * 3, a, ls, [p0, p1, p2])
    amp = al * (al * g0 + be1) * x0
    ang = p1 + p2
    assert abs(h[0] - amp * math.cos(ang)) < 1e-14
    assert abs(h[1] - amp * math.sin(ang)) < 1e-14
    assert abs(y[2] - amp * math.cos(ang)) < 1e-14


# ---------------------------------------------------------------------------
# Parity construction (page 4, "Decay remembers magnitude; rotation can
# remember state"): start at (1, 0), rotate by pi on a one.
def test_parity_construction_golden():
    path = os.path.join(HERE, "golden", "parity_construction.txt")
    cases = []
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        bits, *signs = line.split()
        cases.append((bits, [int(s) for s in signs]))
    assert len(cases) >= 5
    for bits, signs in cases:
        T = len(bits) + 1
        xs = [1.0] + [0.0] * len(bits)               # the initial write (1, 0)
        phis = [0.0] + [math.pi * int(b) for b in bits]
        y, _ = _one_pair(xs, [(1, 0)] * T, [(1, 0)] * T, [1.0] * T, 0.0, [1.0] * T, phis)
        assert abs(y[0] - 1.0) < 1e-15
        got = [int(np.sign(v)) for v in y[1:]]
        assert got == signs, bits
        assert np.allclose(np.abs(y[1:]), 1.0, atol=1e-12)


def test_rotation_preserves_norm_without_decay():
    # A = 0 and lambda = 1, a write at t = 0 only: each step is a pure rotation
    rng = np.random.default_rng(1)
    T, N, P = 30, 6, 3
    x = np.zeros((1, T, 1, 1, P)); x[0, 0, 0, 0] = rng.standard_normal(P)
    B = rng.standard_normal((1, T, 1, 1, N)); C = rng.standard_normal((1, T, 1, 1, N))
    dt = np.abs(rng.standard_normal((1, T, 1))) + 0.1
    om = rng.uniform(-math.pi, math.pi, (1, T, 1, N // 2))
    lam = np.ones((1, T, 1))
    norms = []
    for k in range(1, T + 1):
        _, hT, _ = oracle.scan(x[:, :k], B[:, :k], C[:, :k], dt[:, :k], np.zeros(1), lam[:, :k], om[:, :k])
        norms.append(np.linalg.norm(hT))
    assert np.allclose(norms, norms[0], rtol=1e-13)
    assert norms[0] > 0


# ---------------------------------------------------------------------------
# MIMO write B X^T (page 4 section 3.3, Eqs. 12-14, panel 4).
@pytest.mark.parametrize("R", [1, 3])
def test_single_token_mimo_write_and_readout(R):
    rng = np.random.default_rng(R)
    N, P, H = 6, 4, 2
    x = rng.standard_normal((1, 1, H, R, P))
    B = rng.standard_normal((1, 1, H, R, N)); C = rng.standard_normal((1, 1, H, R, N))
    dt = np.array([[[0.3, 0.8]]]); lam = np.array([[[0.6, 0.2]]])
    A = np.array([-1.0, -2.0])
    om = rng.uniform(-3, 3, (1, 1, H, N // 2))
    y, hT, prevT = oracle.scan(x, B, C, dt, A, lam, om)
    for h in range(H):
        g = lam[0, 0, h] * dt[0, 0, h]
        W = np.zeros((N, P))
        for n in range(N):
            for p in range(P):
                W[n, p] = sum(B[0, 0, h, r, n] * x[0, 0, h, r, p] for r in range(R))
        if R == 1:
            assert np.allclose(W, np.outer(B[0, 0, h, 0], x[0, 0, h, 0]), rtol=0, atol=1e-15)
        assert np.allclose(hT[0, h], g * W, rtol=0, atol=1e-14)
        for r in range(R):
            for p in range(P):
                ref = sum(g * W[n, p] * C[0, 0, h, r, n] for n in range(N))
                assert abs(y[0, 0, h, r, p] - ref) < 1e-13
        assert np.allclose(prevT[0, h], np.concatenate([B[0, 0, h].ravel(), x[0, 0, h].ravel()]))


# ---------------------------------------------------------------------------
def test_lambda_one_ignores_delayed_write():
    """lambda_t = 1 gives beta_t = 0 (page 4 panel 1): the carried delayed
    write then has no effect; with lambda_0 < 1 it does."""
    inp = _small(R=2, T=6, seed=4)
    args = _args(inp)
    Bt, H, R, P, N = 2, 3, 2, 5, 6
    prev = np.random.default_rng(0).standard_normal((Bt, H, R * (N + P)))
    lam1 = torch.ones_like(inp["lam"])
    a1 = args[:5] + [lam1, args[6]]
    y0, _, _ = oracle.scan(*a1)
    y1, _, _ = oracle.scan(*a1, prev=prev)
    assert np.max(np.abs(y0 - y1)) == 0.0
    y2, _, _ = oracle.scan(*args)
    y3, _, _ = oracle.scan(*args, prev=prev)
    assert np.max(np.abs(y2 - y3)) > 1e-6


def test_linearity_and_zero_input():
    inp = _small(R=2, T=25, seed=6)
    x, B, C, dt, A, lam, om = (_f(v) for v in _args(inp))
    x2 = np.random.default_rng(2).standard_normal(x.shape)
    y1, _, _ = oracle.scan(x, B, C, dt, A, lam, om)
    y2, _, _ = oracle.scan(x2, B, C, dt, A, lam, om)
    y12, _, _ = oracle.scan(2.0 * x + x2, B, C, dt, A, lam, om)
    assert oracle.rel_err(y12, 2.0 * y1 + y2) < 1e-13
    y0, h0, _ = oracle.scan(np.zeros_like(x), B, C, dt, A, lam, om)
    assert np.max(np.abs(y0)) == 0.0 and np.max(np.abs(h0)) == 0.0


def test_continuation_prefill_then_decode():
    """Prefill of T tokens, then k single-token steps from the carried state
    and delayed-write cache, equals prefill of T + k tokens."""
    inp = _small(R=2, T=40, seed=9)
    args = [_f(v) for v in _args(inp)]
    T0 = 31
    yfull, hfull, _ = oracle.scan(*args)
    pre = [a[:, :T0] if a.ndim >= 3 else a for a in args]
    _, h, prev = oracle.scan(*pre)
    x, B, C, dt, A, lam, om = args
    for t in range(T0, 40):
        yt, h, prev = oracle.decode_step(h, x[:, t], B[:, t], prev, C[:, t], dt[:, t], A, lam[:, t], om[:, t])
        assert oracle.rel_err(yt, yfull[:, t]) < 1e-13
    assert oracle.rel_err(h, hfull) < 1e-13


def test_state_passing_closed_form():
    """H_c = sum_k exp(sum_{m=k+1..c} l_m) R(sum_{m=k+1..c} Theta_m) U_k
    + exp(sum_{m<=c} l_m) R(sum_{m<=c} Theta_m) H_init."""
    sp = synth.make_state_passing_inputs(1, 2, 5, 4, 3, seed=3)
    U, ld, ang, h0 = (_f(sp[k]) for k in ("chunk_states", "chunk_logdecay", "chunk_angle", "init_state"))
    carries, fin = forms.state_passing(U, ld, ang, h0)
    nc = U.shape[2]

    def rot_rows(Hm, th):  # rotate state rows (2j, 2j+1)
        return forms.rotate_pairs(Hm.swapaxes(-1, -2), th[..., None, :]).swapaxes(-1, -2)

    for c in range(nc + 1):
        ref = np.exp(ld[:, :, :c].sum(-1))[..., None, None] * rot_rows(h0, ang[:, :, :c].sum(2))
        for k in range(c):
            ref = ref + np.exp(ld[:, :, k + 1:c].sum(-1))[..., None, None] * rot_rows(U[:, :, k], ang[:, :, k + 1:c].sum(2))
        got = carries[:, :, c] if c < nc else fin
        assert np.max(np.abs(got - ref)) < 1e-12


def test_preconditions_rejected():
    inp = _small(T=4)
    args = [_f(v) for v in _args(inp)]
    bad_dt = [a.copy() for a in args]; bad_dt[3][0, 1, 0] = -0.1
    bad_A = [a.copy() for a in args]; bad_A[4][0] = 0.5
    bad_l = [a.copy() for a in args]; bad_l[5][0, 2, 1] = 1.5
    for bad in (bad_dt, bad_A, bad_l):
        with pytest.raises(ValueError):
            oracle.scan(*bad)


def test_arithmetic_intensity_model():
    # Table 2 / panel 5; at R = 1 the numerator is the SISO count 5NP - P
    for N, P in ((64, 64), (128, 64), (16, 16)):
        assert forms.arithmetic_intensity(N, P, 1) == (5 * N * P - P) / (2 * (1 + 2 * N + P + N * P))
    # intensity grows with R at fixed N, P
    vals = [forms.arithmetic_intensity(128, 64, r) for r in (1, 2, 4, 8)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
