"""Float64 CPU oracle of the Mamba-3 SSM layer recurrence.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library (``state_space_sequence_04_b300``) and never imports it.

Two parts:

* ``m3_oracle.c`` (built to ``liboracle.so`` with gcc, float64, OpenMP over
  independent (batch, head) sequences): the sequential recurrence in the
  physical frame, one token at a time.  ``scan`` below wraps it; a decode step
  is ``scan`` with T = 1 and a carried state.
* ``forms.py`` (numpy, float64): the other evaluations of the same recurrence
  that the tests use to pin the sequential oracle (Mamba-2 reduction, decay x
  two-band mask matrix form, complex-diagonal state, rotating-frame form,
  chunked evaluation with state passing), and the state-passing recurrence.

Layouts are those of ``synth.py``: x [Bt,T,H,R,P], B/C [Bt,T,H,R,N],
dt/lam [Bt,T,H], A [H] (or [Bt,T,H]: one A_t per token), omega [Bt,T,H,N/2],
y [Bt,T,H,R,P], states [Bt,H,N,P], delayed-write cache [Bt,H,R*N+R*P].

``prep`` / ``scan_prep`` / ``decode_step_prep`` take the pre-activations of
the per-token parameters instead: Delta_t = softplus(dt_raw_t + dt_bias_h),
lambda_t = sigmoid(u_t) (the default lambda parameterisation of the appendix
ablation table), A_t given per token; optionally B and C are RMS-normalised
over N, then shifted by per-head channel biases, before the rotation
(``bc_prep``; the BC normalisation and biases of section 3.4); and the
output may be gated, y * silu(z) (the SSM+Gate fusion of Tables 11-12; the
pages give no gate formula, this is the Mamba family's).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m3_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``m3_oracle.c`` to ``liboracle.so`` (gcc -O2 -fopenmp, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.m3o_scan.argtypes = [dp] * 7 + [i64] * 6 + [dp] * 5
        lib.m3o_scan.restype = ctypes.c_int
        lib.m3o_scan_tok.argtypes = [dp] * 7 + [i64] * 6 + [dp] * 5
        lib.m3o_scan_tok.restype = ctypes.c_int
        lib.m3o_num_threads.argtypes = []
        lib.m3o_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().m3o_num_threads())


def f64(a) -> np.ndarray:
    """Contiguous float64 numpy copy of a numpy array or (CPU or CUDA) torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def scan(x, B, C, dt, A, lam, omega, h0=None, prev=None):
    """Sequential recurrence (float64) over all tokens.

    Returns (y [Bt,T,H,R,P], hT [Bt,H,N,P], prevT [Bt,H,R*(N+P)]).
    ``h0`` / ``prev`` are the carried state and delayed-write factors (zero if None).
    ``A`` is [H] (one decay generator per head) or [Bt,T,H] (one per token).
    """
    x, B, C, dt, A, lam, omega = (f64(v) for v in (x, B, C, dt, A, lam, omega))
    Bt, T, H, R, P = x.shape
    N = B.shape[-1]
    if B.shape != (Bt, T, H, R, N) or C.shape != B.shape:
        raise ValueError("B, C must be [Bt,T,H,R,N]")
    if dt.shape != (Bt, T, H) or lam.shape != (Bt, T, H) or A.shape not in ((H,), (Bt, T, H)):
        raise ValueError("dt, lam must be [Bt,T,H]; A must be [H] or [Bt,T,H]")
    if omega.shape != (Bt, T, H, N // 2):
        raise ValueError("omega must be [Bt,T,H,N/2]")
    h0 = None if h0 is None else f64(h0).reshape(Bt, H, N, P)
    prev = None if prev is None else f64(prev).reshape(Bt, H, R * (N + P))
    y = np.zeros((Bt, T, H, R, P))
    hT = np.zeros((Bt, H, N, P))
    prevT = np.zeros((Bt, H, R * (N + P)))
    fn = _load().m3o_scan if A.shape == (H,) else _load().m3o_scan_tok
    st = fn(_ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A), _ptr(lam), _ptr(omega),
            Bt, T, H, P, N, R, _ptr(h0), _ptr(prev), _ptr(y), _ptr(hT), _ptr(prevT))
    if st != 0:
        raise ValueError(f"oracle rejected its inputs (code {st}): shapes, or a precondition "
                         "Delta >= 0, A <= 0, lambda in [0, 1], finite values")
    return y, hT, prevT


def decode_step(state, x_t, B_t, prev, C_t, dt_t, A, lam_t, omega_t):
    """One decode token: the sequential step from a carried state.

    state [b,H,N,P]; x_t [b,H,R,P]; B_t, C_t [b,H,R,N]; prev [b,H,R*(N+P)];
    dt_t, lam_t [b,H]; A [H]; omega_t [b,H,N/2].
    Returns (y_t [b,H,R,P], new state, new prev).
    """
    xt = f64(x_t)[:, None]
    y, hT, prevT = scan(xt, f64(B_t)[:, None], f64(C_t)[:, None], f64(dt_t)[:, None], A,
                        f64(lam_t)[:, None], f64(omega_t)[:, None], h0=state, prev=prev)
    return y[:, 0], hT, prevT


def softplus(z):
    """log(1 + e^z) in float64 (numpy's logaddexp(0, z))."""
    return np.logaddexp(0.0, f64(z))


def sigmoid(u):
    """1 / (1 + e^-u) in float64, evaluated without overflow for either sign of u."""
    u = f64(u)
    e = np.exp(-np.abs(u))
    return np.where(u >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def prep(dt_raw, dt_bias, u):
    """Per-token parameters from their pre-activations (float64):
    Delta = softplus(dt_raw + dt_bias[h]) (dt_bias None = 0), lambda = sigmoid(u)."""
    z = f64(dt_raw)
    if dt_bias is not None:
        z = z + f64(dt_bias)
    return softplus(z), sigmoid(u)


def silu(z):
    """z * sigmoid(z) in float64."""
    z = f64(z)
    return z * sigmoid(z)


def bc_prep(V, norm: bool = False, eps: float = 0.0, gain=None, bias=None):
    """B or C before the rotation (float64): every (token, rank) row v of V [..., H, R, N]
    becomes v / sqrt(mean(v^2) + eps) * gain when ``norm`` (gain [N], None = 1), then
    the head-specific channel bias [H, R, N] is added (None = 0)."""
    V = f64(V)
    if norm:
        V = V / np.sqrt(np.mean(V * V, axis=-1, keepdims=True) + eps)
        if gain is not None:
            V = V * f64(gain)
    if bias is not None:
        V = V + f64(bias)
    return V


def _bc(B, C, bc):
    bc = bc or {}
    norm, eps = bool(bc.get("norm", False)), float(bc.get("eps", 0.0))
    return (bc_prep(B, norm, eps, bc.get("B_gain"), bc.get("B_bias")),
            bc_prep(C, norm, eps, bc.get("C_gain"), bc.get("C_bias")))


def scan_prep(x, B, C, dt_raw, dt_bias, A_tok, u, omega, h0=None, prev=None, bc=None, z=None):
    """``scan`` on pre-activations: Delta, lambda from ``prep``, A_tok [Bt,T,H] per token;
    ``bc`` (dict: norm, eps, B_gain, C_gain, B_bias, C_bias) normalises and biases B and C
    with ``bc_prep`` first.  ``prev`` holds the raw (unnormalised) B_{t-1}, X_{t-1}.
    ``z`` (y's shape): the output gate, y <- y * silu(z)."""
    d, lam = prep(dt_raw, dt_bias, u)
    Bn, Cn = _bc(B, C, bc)
    if prev is not None and bc:
        prev = _prev_bc(prev, f64(B).shape[-3:], f64(x).shape[-1], bc)
    y, hT, prevT = scan(x, Bn, Cn, d, A_tok, lam, omega, h0=h0, prev=prev)
    if bc:   # hand back the raw factors of the last token, as the kernels keep them
        prevT = _prev_raw(f64(B)[:, -1], f64(x)[:, -1])
    if z is not None:
        y = y * silu(z)
    return y, hT, prevT


def _prev_bc(prev, hrn, P, bc):
    """The delayed-write cache [b,H,R*N+R*P] with its B_{t-1} part normalised and biased."""
    prev = f64(prev).copy()
    H, R, N = hrn
    b = prev.shape[0]
    Bp = prev[:, :, :R * N].reshape(b, H, R, N)
    Bn, _ = _bc(Bp, Bp, bc)
    prev[:, :, :R * N] = Bn.reshape(b, H, R * N)
    return prev


def _prev_raw(B_last, x_last):
    b, H = B_last.shape[:2]
    return np.concatenate([B_last.reshape(b, H, -1), x_last.reshape(b, H, -1)], axis=-1)


def decode_step_prep(state, x_t, B_t, prev, C_t, dt_raw_t, dt_bias, A_t, u_t, omega_t, bc=None, z_t=None):
    """One decode token on pre-activations: dt_raw_t, A_t, u_t [b,H]; dt_bias [H] or None;
    ``prev`` and the returned cache hold the raw B_{t-1}, X_{t-1}; ``z_t`` [b,H,R,P]: the
    output gate."""
    d, lam = prep(dt_raw_t, dt_bias, u_t)
    Bt, Ct = f64(B_t), f64(C_t)
    Bn, Cn = _bc(Bt, Ct, bc)
    if prev is not None and bc:
        prev = _prev_bc(prev, Bt.shape[-3:], f64(x_t).shape[-1], bc)
    xt = f64(x_t)[:, None]
    y, hT, prevT = scan(xt, Bn[:, None], Cn[:, None], d[:, None], f64(A_t)[:, None],
                        lam[:, None], f64(omega_t)[:, None], h0=state, prev=prev)
    if bc:
        prevT = _prev_raw(Bt, f64(x_t))
    yt = y[:, 0] if z_t is None else y[:, 0] * silu(z_t)
    return yt, hT, prevT


def rel_err(got, ref) -> float:
    """max |got - ref| / max |ref| (the parity metric)."""
    got = f64(got)
    ref = f64(ref)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


from . import forms  # noqa: E402,F401
