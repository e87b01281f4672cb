"""Thin ctypes binding of libm3.so (the C ABI declared in include/m3.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  Tensors are torch CUDA tensors (torch provides the
device memory and the stream); the functions named ``m3_*`` mirror the C entry
points one to one.  ``scan_fwd`` / ``decode_step`` / ``state_passing`` are
conveniences that allocate outputs and workspace with torch and then call the
same entry points.

There is no fallback: if libm3.so is missing or cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libm3.so")

M3_OK = 0
M3_ERR_INVALID_ARG = -1
M3_ERR_UNSUPPORTED = -2
M3_ERR_WORKSPACE = -3
M3_ERR_CUDA = -4
M3_ERR_TIMEOUT = -5
M3_DTYPE_BF16 = 0
M3_DTYPE_F32 = 1
M3_TEST_LAUNCH_FAILURE = 1
M3_TEST_PREFILL_TIMEOUT = 2

class PrepParams(ctypes.Structure):
    """m3_prep_params: pre-SSM options of the _prep entry points (device pointers or NULL)."""
    _fields_ = [("dt_bias", ctypes.c_void_p), ("bc_norm", ctypes.c_int), ("bc_eps", ctypes.c_float),
                ("B_gain", ctypes.c_void_p), ("C_gain", ctypes.c_void_p), ("B_bias", ctypes.c_void_p),
                ("C_bias", ctypes.c_void_p), ("z", ctypes.c_void_p)]


# Every symbol include/m3.h declares, with its ctypes signature.
_vp, _fp = ctypes.c_void_p, ctypes.c_void_p
_i64, _int, _sz = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "m3_status_string": ([_int], ctypes.c_char_p),
    "m3_version": ([], _int),
    "m3_scan_fwd_workspace_size": ([_i64, _i64, _i64, _i64, _i64, _int, _int, _int], _sz),
    "m3_scan_fwd_plan": ([_i64, _i64, _i64, _i64, _i64, _int, _int, _int, ctypes.POINTER(_int),
                          ctypes.POINTER(_int)], _int),
    "m3_scan_fwd": ([_vp, _vp, _vp, _fp, _fp, _fp, _fp, _int, _int, _vp, _fp,
                     _i64, _i64, _i64, _i64, _i64, _int, _vp, _sz, _vp], _int),
    "m3_scan_fwd_noalloc": ([_vp, _vp, _vp, _fp, _fp, _fp, _fp, _int, _int, _vp, _fp,
                             _i64, _i64, _i64, _i64, _i64, _int, _vp], _int),
    "m3_decode_step": ([_fp, _vp, _vp, _vp, _vp, _fp, _fp, _fp, _fp, _vp,
                        _i64, _i64, _i64, _i64, _int, _int, _vp], _int),
    "m3_device_status": ([_int], _int),
    "m3_test_inject": ([_int, _int], _int),
    "m3_scan_bwd_workspace_size": ([_i64, _i64, _i64, _i64, _i64, _int, _int], _sz),
    "m3_scan_bwd": ([_vp, _vp, _vp, _fp, _fp, _fp, _fp, _int, _vp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp,
                     _i64, _i64, _i64, _i64, _i64, _int, _vp, _sz, _vp], _int),
    "m3_scan_fwd_prep_workspace_size": ([_i64, _i64, _i64, _i64, _i64, _int, _int, _int], _sz),
    "m3_scan_fwd_prep": ([_vp, _vp, _vp, _fp, _fp, _fp, _fp, _int, _int, _vp, _fp,
                          _i64, _i64, _i64, _i64, _i64, _int, ctypes.POINTER(PrepParams), _vp, _sz, _vp], _int),
    "m3_decode_step_prep": ([_fp, _vp, _vp, _vp, _vp, _fp, _fp, _fp, _fp, _vp,
                             _i64, _i64, _i64, _i64, _int, _int, ctypes.POINTER(PrepParams), _vp], _int),
    "m3_state_passing": ([_fp, _fp, _fp, _fp, _fp, _i64, _i64, _i64, _i64, _i64, _vp], _int),
    "m3_scan_bwd_prep_workspace_size": ([_i64, _i64, _i64, _i64, _i64, _int, _int], _sz),
    "m3_scan_bwd_prep": ([_vp, _vp, _vp, _fp, _fp, _fp, _fp, _int, _vp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp,
                          _fp, _fp, _fp, _fp, _fp, _i64, _i64, _i64, _i64, _i64, _int, ctypes.POINTER(PrepParams),
                          _vp, _sz, _vp], _int),
}

_lib = None


class M3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {m3_status_string(status)} ({status})")


def load():
    """Load libm3.so (raises if it is missing: there is no CPU fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libm3.so not built at {LIB_PATH}; run state_space_sequence_04_b300/build.py")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (argt, rest) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argt
            fn.restype = rest
        _lib = lib
    return _lib


def m3_status_string(status: int) -> str:
    return load().m3_status_string(int(status)).decode()


def m3_version() -> int:
    return int(load().m3_version())


def io_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return M3_DTYPE_BF16
    if dtype == torch.float32:
        return M3_DTYPE_F32
    raise TypeError(f"io dtype must be bfloat16 or float32, got {dtype}")


def _ptr(t: Optional[torch.Tensor], dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libm3 takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libm3 takes contiguous tensors")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(st: int, where: str):
    if st != M3_OK:
        raise M3Error(st, where)


# ---------------------------------------------------------------------------
# One-to-one wrappers of the C entry points.
def m3_scan_fwd_workspace_size(batch, seqlen, nheads, headdim, dstate, R, chunk, io) -> int:
    return int(load().m3_scan_fwd_workspace_size(batch, seqlen, nheads, headdim, dstate, R, chunk, io))


def m3_scan_fwd_plan(batch, seqlen, nheads, headdim, dstate, R, chunk, io):
    """(path, launches) of m3_scan_fwd for these sizes: path 0 = CUDA cores, 1 = tensor cores."""
    path, launches = _int(0), _int(0)
    _check(int(load().m3_scan_fwd_plan(batch, seqlen, nheads, headdim, dstate, R, chunk, io,
                                       ctypes.byref(path), ctypes.byref(launches))), "m3_scan_fwd_plan")
    return path.value, launches.value


def m3_scan_fwd(x, B, C, dt, A, lam, omega, R: int, chunk: int, y, final_state, workspace,
                stream=None) -> int:
    """Call m3_scan_fwd; returns the status code (does not raise)."""
    Bt, T, H, R_, P = x.shape
    N = B.shape[-1]
    io = io_code(x.dtype)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return int(load().m3_scan_fwd(
        _ptr(x, x.dtype), _ptr(B, x.dtype), _ptr(C, x.dtype), _ptr(dt, torch.float32),
        _ptr(A, torch.float32), _ptr(lam, torch.float32), _ptr(omega, torch.float32), int(R), int(chunk),
        _ptr(y, x.dtype), _ptr(final_state, torch.float32), Bt, T, H, P, N, io, _ptr(workspace), ws_bytes,
        _stream(stream)))


def m3_scan_fwd_noalloc(x, B, C, dt, A, lam, omega, R: int, chunk: int, y, final_state, stream=None) -> int:
    """Call m3_scan_fwd_noalloc: m3_scan_fwd without a workspace (the library's
    fixed scratch array instead); returns the status code (does not raise)."""
    Bt, T, H, R_, P = x.shape
    N = B.shape[-1]
    io = io_code(x.dtype)
    return int(load().m3_scan_fwd_noalloc(
        _ptr(x, x.dtype), _ptr(B, x.dtype), _ptr(C, x.dtype), _ptr(dt, torch.float32),
        _ptr(A, torch.float32), _ptr(lam, torch.float32), _ptr(omega, torch.float32), int(R), int(chunk),
        _ptr(y, x.dtype), _ptr(final_state, torch.float32), Bt, T, H, P, N, io, _stream(stream)))


def m3_decode_step(state, x_t, B_t, cache, C_t, dt_t, A, lam_t, omega_t, y_t, R: int, stream=None) -> int:
    """Call m3_decode_step; returns the status code (does not raise)."""
    b, H, R_, P = x_t.shape
    N = B_t.shape[-1]
    io = io_code(x_t.dtype)
    return int(load().m3_decode_step(
        _ptr(state, torch.float32), _ptr(x_t, x_t.dtype), _ptr(B_t, x_t.dtype), _ptr(cache, x_t.dtype),
        _ptr(C_t, x_t.dtype), _ptr(dt_t, torch.float32), _ptr(A, torch.float32), _ptr(lam_t, torch.float32),
        _ptr(omega_t, torch.float32), _ptr(y_t, x_t.dtype), b, H, P, N, int(R), io, _stream(stream)))


def m3_scan_fwd_prep_workspace_size(batch, seqlen, nheads, headdim, dstate, R, chunk, io) -> int:
    return int(load().m3_scan_fwd_prep_workspace_size(batch, seqlen, nheads, headdim, dstate, R, chunk, io))


def prep_params(dt_bias=None, bc=None, z=None):
    """PrepParams from device tensors: dt_bias [H]; bc = dict(norm, eps, B_gain, C_gain,
    B_bias, C_bias), tensors [N] / [H, R, N] or absent; z: the output gate's input (y's shape)."""
    bc = bc or {}
    return PrepParams(_ptr(dt_bias, torch.float32), 1 if bc.get("norm") else 0, float(bc.get("eps", 0.0)),
                      _ptr(bc.get("B_gain"), torch.float32), _ptr(bc.get("C_gain"), torch.float32),
                      _ptr(bc.get("B_bias"), torch.float32), _ptr(bc.get("C_bias"), torch.float32), _ptr(z))


def m3_scan_fwd_prep(x, B, C, dt_raw, A, u, omega, R: int, chunk: int, y, final_state, workspace, params=None,
                     stream=None) -> int:
    """Call m3_scan_fwd_prep (pre-activations, A per token; ``params``: PrepParams or None);
    returns the status code."""
    Bt, T, H, R_, P = x.shape
    N = B.shape[-1]
    io = io_code(x.dtype)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return int(load().m3_scan_fwd_prep(
        _ptr(x, x.dtype), _ptr(B, x.dtype), _ptr(C, x.dtype), _ptr(dt_raw, torch.float32), _ptr(A, torch.float32),
        _ptr(u, torch.float32), _ptr(omega, torch.float32), int(R), int(chunk), _ptr(y, x.dtype),
        _ptr(final_state, torch.float32), Bt, T, H, P, N, io, None if params is None else ctypes.byref(params),
        _ptr(workspace), ws_bytes, _stream(stream)))


def m3_decode_step_prep(state, x_t, B_t, cache, C_t, dt_raw_t, A_t, u_t, omega_t, y_t, R: int, params=None,
                        stream=None) -> int:
    """Call m3_decode_step_prep (pre-activations, A per (batch, head)); returns the status code."""
    b, H, R_, P = x_t.shape
    N = B_t.shape[-1]
    io = io_code(x_t.dtype)
    return int(load().m3_decode_step_prep(
        _ptr(state, torch.float32), _ptr(x_t, x_t.dtype), _ptr(B_t, x_t.dtype), _ptr(cache, x_t.dtype),
        _ptr(C_t, x_t.dtype), _ptr(dt_raw_t, torch.float32), _ptr(A_t, torch.float32), _ptr(u_t, torch.float32),
        _ptr(omega_t, torch.float32), _ptr(y_t, x_t.dtype), b, H, P, N, int(R), io,
        None if params is None else ctypes.byref(params), _stream(stream)))


def m3_scan_bwd_workspace_size(batch, seqlen, nheads, headdim, dstate, R, io) -> int:
    return int(load().m3_scan_bwd_workspace_size(batch, seqlen, nheads, headdim, dstate, R, io))


def m3_scan_bwd(x, B, C, dt, A, lam, omega, R: int, dy, d_final, grads: dict, workspace, stream=None) -> int:
    """Call m3_scan_bwd; ``grads`` holds the fp32 outputs dx, dB, dC, ddt, dA, dlam, domega.
    Returns the status code."""
    Bt, T, H, R_, P = x.shape
    N = B.shape[-1]
    io = io_code(x.dtype)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    f = torch.float32
    return int(load().m3_scan_bwd(
        _ptr(x, x.dtype), _ptr(B, x.dtype), _ptr(C, x.dtype), _ptr(dt, f), _ptr(A, f), _ptr(lam, f), _ptr(omega, f),
        int(R), _ptr(dy, x.dtype), _ptr(d_final, f), _ptr(grads["dx"], f), _ptr(grads["dB"], f), _ptr(grads["dC"], f),
        _ptr(grads["ddt"], f), _ptr(grads["dA"], f), _ptr(grads["dlam"], f), _ptr(grads["domega"], f),
        Bt, T, H, P, N, io, _ptr(workspace), ws_bytes, _stream(stream)))


def scan_bwd(x, B, C, dt, A, lam, omega, R: int, dy, d_final=None, workspace=None, stream=None) -> dict:
    """Backward pass of scan_fwd: fp32 gradients dx, dB, dC, ddt, dA, dlam, domega."""
    Bt, T, H, _, P = x.shape
    N = B.shape[-1]
    f = dict(dtype=torch.float32, device=x.device)
    grads = {"dx": torch.empty(x.shape, **f), "dB": torch.empty(B.shape, **f), "dC": torch.empty(C.shape, **f),
             "ddt": torch.empty(dt.shape, **f), "dA": torch.empty(A.shape, **f), "dlam": torch.empty(lam.shape, **f),
             "domega": torch.empty(omega.shape, **f)}
    if workspace is None:
        nbytes = m3_scan_bwd_workspace_size(Bt, T, H, P, N, R, io_code(x.dtype))
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    _check(m3_scan_bwd(x, B, C, dt, A, lam, omega, R, dy, d_final, grads, workspace, stream), "m3_scan_bwd")
    return grads


def m3_scan_bwd_prep_workspace_size(batch, seqlen, nheads, headdim, dstate, R, io) -> int:
    return int(load().m3_scan_bwd_prep_workspace_size(batch, seqlen, nheads, headdim, dstate, R, io))


def m3_scan_bwd_prep(x, B, C, dt_raw, A, u, omega, R: int, dy, d_final, grads: dict, workspace, params=None,
                     stream=None) -> int:
    """Call m3_scan_bwd_prep; ``grads`` holds the fp32 outputs dx, dB, dC, ddt_raw, dA, du, domega and
    (optional, may be None) ddt_bias, dz, dB_gain, dC_gain, dB_bias, dC_bias.  Returns the status code."""
    Bt, T, H, R_, P = x.shape
    N = B.shape[-1]
    io = io_code(x.dtype)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    f = torch.float32
    return int(load().m3_scan_bwd_prep(
        _ptr(x, x.dtype), _ptr(B, x.dtype), _ptr(C, x.dtype), _ptr(dt_raw, f), _ptr(A, f), _ptr(u, f), _ptr(omega, f),
        int(R), _ptr(dy, x.dtype), _ptr(d_final, f), _ptr(grads["dx"], f), _ptr(grads["dB"], f), _ptr(grads["dC"], f),
        _ptr(grads["ddt_raw"], f), _ptr(grads["dA"], f), _ptr(grads["du"], f), _ptr(grads["domega"], f),
        _ptr(grads.get("ddt_bias"), f), _ptr(grads.get("dz"), f), _ptr(grads.get("dB_gain"), f),
        _ptr(grads.get("dC_gain"), f), _ptr(grads.get("dB_bias"), f), _ptr(grads.get("dC_bias"), f), Bt, T, H, P, N, io,
        None if params is None else ctypes.byref(params),
        _ptr(workspace), ws_bytes, _stream(stream)))


def scan_bwd_prep(x, B, C, dt_raw, A, u, omega, R: int, dy, d_final=None, dt_bias=None, z=None, bc=None,
                  workspace=None, stream=None) -> dict:
    """Backward pass of scan_fwd_prep: fp32 gradients dx, dB, dC, ddt_raw, dA (per token), du, domega, with
    ``dt_bias`` ddt_bias, with the output gate's ``z`` dz, and with ``bc`` (as scan_fwd_prep's) the gradients
    of its present gains and biases (dB_gain, dC_gain, dB_bias, dC_bias)."""
    Bt, T, H, _, P = x.shape
    N = B.shape[-1]
    f = dict(dtype=torch.float32, device=x.device)
    grads = {"dx": torch.empty(x.shape, **f), "dB": torch.empty(B.shape, **f), "dC": torch.empty(C.shape, **f),
             "ddt_raw": torch.empty(dt_raw.shape, **f), "dA": torch.empty(A.shape, **f),
             "du": torch.empty(u.shape, **f), "domega": torch.empty(omega.shape, **f),
             "ddt_bias": None if dt_bias is None else torch.empty((H,), **f),
             "dz": None if z is None else torch.empty(x.shape, **f)}
    for k in ("B_gain", "C_gain", "B_bias", "C_bias"):
        if bc is not None and bc.get(k) is not None:
            grads["d" + k] = torch.empty(bc[k].shape, **f)
    if workspace is None:
        nbytes = m3_scan_bwd_prep_workspace_size(Bt, T, H, P, N, R, io_code(x.dtype))
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    params = None if dt_bias is None and z is None and bc is None else prep_params(dt_bias, bc, z)
    _check(m3_scan_bwd_prep(x, B, C, dt_raw, A, u, omega, R, dy, d_final, grads, workspace, params, stream),
           "m3_scan_bwd_prep")
    return grads


def m3_device_status(clear: bool = False) -> int:
    """Device-side error words of the calls without a workspace (the decode kernels, sticky; the most
    recent m3_scan_fwd_noalloc call): M3_OK or M3_ERR_TIMEOUT.  Synchronises the current device."""
    return int(load().m3_device_status(1 if clear else 0))


def m3_test_inject(what: int, count: int) -> int:
    """Arm a test failure (M3_TEST_LAUNCH_FAILURE, M3_TEST_PREFILL_TIMEOUT; 0 disarms)."""
    return int(load().m3_test_inject(int(what), int(count)))


def m3_state_passing(chunk_states, chunk_logdecay, chunk_angle, init_state, final_state, stream=None) -> int:
    """Call m3_state_passing; returns the status code (does not raise)."""
    b, H, nc, N, P = chunk_states.shape
    return int(load().m3_state_passing(
        _ptr(chunk_states, torch.float32), _ptr(chunk_logdecay, torch.float32), _ptr(chunk_angle, torch.float32),
        _ptr(init_state, torch.float32), _ptr(final_state, torch.float32), b, H, nc, N, P, _stream(stream)))


# ---------------------------------------------------------------------------
# Conveniences: allocate with torch, call the entry point, raise on error.
def alloc_workspace(x_shape, N: int, R: int, chunk: int, dtype: torch.dtype, device) -> Optional[torch.Tensor]:
    Bt, T, H, _, P = x_shape
    nbytes = m3_scan_fwd_workspace_size(Bt, T, H, P, N, R, chunk, io_code(dtype))
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def alloc_workspace_prep(x_shape, N: int, R: int, chunk: int, dtype: torch.dtype, device) -> Optional[torch.Tensor]:
    Bt, T, H, _, P = x_shape
    nbytes = m3_scan_fwd_prep_workspace_size(Bt, T, H, P, N, R, chunk, io_code(dtype))
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def scan_fwd_prep(x, B, C, dt_raw, A, u, omega, R: int, chunk: int, dt_bias=None, bc=None, z=None,
                  want_final: bool = True, workspace=None, stream=None):
    """Prefill on pre-activations (Delta = softplus(dt_raw + dt_bias), lambda = sigmoid(u), A per
    token; ``bc``: B / C normalisation and biases, see prep_params); returns (y, final_state or None)."""
    Bt, T, H, _, P = x.shape
    N = B.shape[-1]
    y = torch.empty_like(x)
    fin = torch.empty((Bt, H, N, P), dtype=torch.float32, device=x.device) if want_final else None
    if workspace is None:
        workspace = alloc_workspace_prep(x.shape, N, R, chunk, x.dtype, x.device)
    params = prep_params(dt_bias, bc, z)
    _check(m3_scan_fwd_prep(x, B, C, dt_raw, A, u, omega, R, chunk, y, fin, workspace, params, stream),
           "m3_scan_fwd_prep")
    return y, fin


def decode_step_prep(state, x_t, B_t, cache, C_t, dt_raw_t, A_t, u_t, omega_t, R: int, dt_bias=None, bc=None,
                     z_t=None, y_t=None, stream=None):
    """One decode token on pre-activations, in place on ``state`` and ``cache`` (raw B, X); returns y_t."""
    if y_t is None:
        y_t = torch.empty_like(x_t)
    params = prep_params(dt_bias, bc, z_t)
    _check(m3_decode_step_prep(state, x_t, B_t, cache, C_t, dt_raw_t, A_t, u_t, omega_t, y_t, R, params, stream),
           "m3_decode_step_prep")
    return y_t


def scan_fwd(x, B, C, dt, A, lam, omega, R: int, chunk: int, want_final: bool = True, workspace=None,
             stream=None):
    """Prefill; returns (y, final_state or None)."""
    Bt, T, H, _, P = x.shape
    N = B.shape[-1]
    y = torch.empty_like(x)
    fin = torch.empty((Bt, H, N, P), dtype=torch.float32, device=x.device) if want_final else None
    if workspace is None:
        workspace = alloc_workspace(x.shape, N, R, chunk, x.dtype, x.device)
    _check(m3_scan_fwd(x, B, C, dt, A, lam, omega, R, chunk, y, fin, workspace, stream), "m3_scan_fwd")
    return y, fin


def decode_step(state, x_t, B_t, cache, C_t, dt_t, A, lam_t, omega_t, R: int, y_t=None, stream=None):
    """One decode token in place on ``state`` and ``cache``; returns y_t."""
    if y_t is None:
        y_t = torch.empty_like(x_t)
    _check(m3_decode_step(state, x_t, B_t, cache, C_t, dt_t, A, lam_t, omega_t, y_t, R, stream), "m3_decode_step")
    return y_t


def state_passing(chunk_states, chunk_logdecay, chunk_angle, init_state=None, want_final: bool = True,
                  stream=None):
    """In-place state passing; returns final_state (or None)."""
    b, H, nc, N, P = chunk_states.shape
    fin = torch.empty((b, H, N, P), dtype=torch.float32, device=chunk_states.device) if want_final else None
    _check(m3_state_passing(chunk_states, chunk_logdecay, chunk_angle, init_state, fin, stream), "m3_state_passing")
    return fin


def new_decode_cache(batch: int, heads: int, dstate: int, headdim: int, R: int, dtype, device) -> torch.Tensor:
    """Zeroed delayed-write cache [b, H, R*N + R*P] (a sequence's first token)."""
    return torch.zeros((batch, heads, R * (dstate + headdim)), dtype=dtype, device=device)


def cache_from_prefill(B: torch.Tensor, x: torch.Tensor) -> torch.Tensor:
    """Delayed-write cache after a prefill: B[:, T-1] then x[:, T-1], flattened per (b, h)."""
    Bl = B[:, -1]                       # [b, H, R, N]
    Xl = x[:, -1]                       # [b, H, R, P]
    b, H = Bl.shape[:2]
    return torch.cat([Bl.reshape(b, H, -1), Xl.reshape(b, H, -1)], dim=-1).contiguous()
