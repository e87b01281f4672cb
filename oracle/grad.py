"""Gradients of the float64 oracle by finite differences (backward pass reference).

TEST INFRASTRUCTURE ONLY (see the package docstring).

For a loss L = sum(y * dy) + sum(h_{T-1} * d_final) (the adjoint seeds of a
backward pass: dy = dL/dy, d_final = dL/d final_state), the gradient of L with
respect to every input of the sequential recurrence of ``oracle.scan`` --
x, B, C, dt, A, lambda, omega -- by central differences of that recurrence in
float64.  The recurrence is the one of "Mamba-3: Improved Sequence Modeling
using State Space Principles" (Proposition 1 / Eq. 6 with the rotation of
Propositions 2-4); its backward pass for training is the last of the chunked
algorithm's uses listed in section 3.3.

``grad_fd`` perturbs every element (small problems only); ``directional`` gives
the derivative of L along one direction per input, for larger problems.  With
``prep=True`` the loss runs ``oracle.scan_prep`` on pre-activations instead
(Delta = softplus(dt_raw + dt_bias), lambda = sigmoid(u), A per token; the
time-varying discretisations of the page's Table 1), over PREP_INPUTS, with a
"z" entry in the inputs through the output gate y * silu(z) as well, and with
"bc_norm" / "bc_eps" entries through the B / C normalisation of ``bc_prep``
(section 3.4), whose present "B_gain", "C_gain", "B_bias", "C_bias" entries are
then inputs too.
"""
from __future__ import annotations

import numpy as np

from . import f64, scan, scan_prep

INPUTS = ("x", "B", "C", "dt", "A", "lam", "omega")
PREP_INPUTS = ("x", "B", "C", "dt_raw", "dt_bias", "A", "u", "omega")


BC_INPUTS = ("B_gain", "C_gain", "B_bias", "C_bias")


def _names(inp: dict, prep: bool):
    if not prep:
        return INPUTS
    extra = ("z",) if inp.get("z") is not None else ()
    if "bc_norm" in inp:
        extra += tuple(k for k in BC_INPUTS if inp.get(k) is not None)
    return PREP_INPUTS + extra


def _bc_of(inp: dict):
    if "bc_norm" not in inp:
        return None
    bc = {"norm": bool(inp["bc_norm"]), "eps": float(inp.get("bc_eps", 0.0))}
    bc.update({k: inp.get(k) for k in BC_INPUTS})
    return bc


def loss(inp: dict, dy, d_final=None, prep: bool = False) -> float:
    if prep:
        y, hT, _ = scan_prep(*[inp[k] for k in PREP_INPUTS], bc=_bc_of(inp), z=inp.get("z"))
    else:
        y, hT, _ = scan(*[inp[k] for k in INPUTS])
    val = float(np.sum(y * f64(dy)))
    if d_final is not None:
        val += float(np.sum(hT * f64(d_final)))
    return val


def grad_fd(inp: dict, dy, d_final=None, eps: float = 1e-6, keys=None, prep: bool = False) -> dict:
    """dL/d(input) for every element of the listed inputs, central differences with step eps."""
    names = _names(inp, prep)
    keys = names if keys is None else keys
    base = dict(inp)   # settings (bc_norm, bc_eps) as given, inputs as float64 copies
    base.update({k: f64(inp[k]).copy() for k in names})
    out = {}
    for k in keys:
        g = np.zeros_like(base[k])
        flat = base[k].reshape(-1)
        gf = g.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            lp = loss(base, dy, d_final, prep)
            flat[i] = keep - eps
            lm = loss(base, dy, d_final, prep)
            flat[i] = keep
            gf[i] = (lp - lm) / (2.0 * eps)
        out[k] = g
    return out


def directional(inp: dict, key: str, v, dy, d_final=None, eps: float = 1e-6, prep: bool = False) -> float:
    """d/ds L(input[key] + s v) at s = 0, central differences with step eps."""
    base = dict(inp)
    base.update({k: f64(inp[k]).copy() for k in _names(inp, prep)})
    v = f64(v)
    keep = base[key].copy()
    base[key] = keep + eps * v
    lp = loss(base, dy, d_final, prep)
    base[key] = keep - eps * v
    lm = loss(base, dy, d_final, prep)
    return (lp - lm) / (2.0 * eps)


def adjoint(inp: dict, dy, d_final=None) -> dict:
    """The same gradients as ``grad_fd`` for the plain inputs, from the adjoint of the recurrence
    written out step by step (float64, no finite differences).  With u_t = alpha_t h_{t-1} +
    beta_t v_{t-1}, h_t = R(phi_t) u_t + gamma_t v_t, v_t = B_t^T X_t and y_t = h_t^T C_t, going
    backwards from gbar_{T-1} = d_final:
      gbar_t = C_t dy_t^T + alpha_{t+1} ubar_{t+1},  ubar_t = R(phi_t)^T gbar_t,
      dv_t = gamma_t gbar_t + beta_{t+1} ubar_{t+1},
    and dalpha_t = <ubar_t, h_{t-1}>, dbeta_t = <ubar_t, v_{t-1}>, dgamma_t = <gbar_t, v_t>,
    dphi_t = sum_p (gbar[2j+1] r[2j] - gbar[2j] r[2j+1]) with r = R(phi_t) u_t; then the chain rule
    through alpha = exp(Delta A), beta = (1 - lambda) Delta alpha, gamma = lambda Delta, phi = Delta omega."""
    x, B, C, dt, A, lam, om = (f64(inp[k]) for k in INPUTS)
    dy = f64(dy)
    Bt, T, H, R, P = x.shape
    N = B.shape[-1]
    out = {k: np.zeros_like(f64(inp[k])) for k in INPUTS}

    def rot(phi, u, sign=1.0):
        c, s = np.cos(phi)[:, None], sign * np.sin(phi)[:, None]
        o = np.empty_like(u)
        o[0::2] = c * u[0::2] - s * u[1::2]
        o[1::2] = s * u[0::2] + c * u[1::2]
        return o

    for b in range(Bt):
        for h in range(H):
            V = [B[b, t, h].T @ x[b, t, h] for t in range(T)]       # v_t, N x P
            hs, st = [], np.zeros((N, P))
            for t in range(T):                                      # the forward states
                al = np.exp(dt[b, t, h] * A[h])
                be = (1.0 - lam[b, t, h]) * dt[b, t, h] * al
                u = al * st + (be * V[t - 1] if t > 0 else 0.0)
                st = rot(dt[b, t, h] * om[b, t, h], u) + lam[b, t, h] * dt[b, t, h] * V[t]
                hs.append(st)
            ub = np.zeros((N, P))
            al_n = be_n = 0.0
            for t in range(T - 1, -1, -1):
                d, l = dt[b, t, h], lam[b, t, h]
                al = np.exp(d * A[h])
                be, ga, phi = (1.0 - l) * d * al, l * d, d * om[b, t, h]
                g = C[b, t, h].T @ dy[b, t, h] + al_n * ub
                if t == T - 1 and d_final is not None:
                    g = g + f64(d_final)[b, h]
                dv = ga * g + be_n * ub
                r = hs[t] - ga * V[t]
                dphi = (g[1::2] * r[0::2] - g[0::2] * r[1::2]).sum(axis=1)
                un = rot(phi, g, sign=-1.0)
                hp = hs[t - 1] if t > 0 else np.zeros((N, P))
                vp = V[t - 1] if t > 0 else np.zeros((N, P))
                da, db, dg = float(np.sum(un * hp)), float(np.sum(un * vp)), float(np.sum(g * V[t]))
                out["C"][b, t, h] = (hs[t] @ dy[b, t, h].T).T
                out["B"][b, t, h] = (dv @ x[b, t, h].T).T
                out["x"][b, t, h] = B[b, t, h] @ dv
                out["omega"][b, t, h] = d * dphi
                dal = da + db * (1.0 - l) * d
                out["dt"][b, t, h] = dal * A[h] * al + db * (1.0 - l) * al + dg * l + float(np.sum(om[b, t, h] * dphi))
                out["lam"][b, t, h] = -d * al * db + d * dg
                out["A"][h] += dal * d * al
                ub, al_n, be_n = un, al, be
    return out
