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
the derivative of L along one direction per input, for larger problems.
"""
from __future__ import annotations

import numpy as np

from . import f64, scan

INPUTS = ("x", "B", "C", "dt", "A", "lam", "omega")


def loss(inp: dict, dy, d_final=None) -> float:
    y, hT, _ = scan(*[inp[k] for k in INPUTS])
    val = float(np.sum(y * f64(dy)))
    if d_final is not None:
        val += float(np.sum(hT * f64(d_final)))
    return val


def grad_fd(inp: dict, dy, d_final=None, eps: float = 1e-6, keys=INPUTS) -> dict:
    """dL/d(input) for every element of the listed inputs, central differences with step eps."""
    base = {k: f64(inp[k]).copy() for k in INPUTS}
    out = {}
    for k in keys:
        g = np.zeros_like(base[k])
        flat = base[k].reshape(-1)
        gf = g.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            lp = loss(base, dy, d_final)
            flat[i] = keep - eps
            lm = loss(base, dy, d_final)
            flat[i] = keep
            gf[i] = (lp - lm) / (2.0 * eps)
        out[k] = g
    return out


def directional(inp: dict, key: str, v, dy, d_final=None, eps: float = 1e-6) -> float:
    """d/ds L(input[key] + s v) at s = 0, central differences with step eps."""
    base = {k: f64(inp[k]).copy() for k in INPUTS}
    v = f64(v)
    keep = base[key].copy()
    base[key] = keep + eps * v
    lp = loss(base, dy, d_final)
    base[key] = keep - eps * v
    lm = loss(base, dy, d_final)
    return (lp - lm) / (2.0 * eps)
