"""Shared helpers of the GPU parity tests (oracle on sampled (batch, head) pairs)."""
import os

import numpy as np
import pytest
import torch

import oracle

# Tolerances on max|err| / max|ref|: bf16 inputs with fp32 accumulation, and fp32 inputs.
TOL = {"bf16": 2e-2, "fp32": 1e-4}

KEYS = ("x", "B", "C", "dt", "A", "lam", "omega")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from state_space_sequence_04_b300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    binding.load()


def to_dev(inp, device="cuda"):
    out = dict(inp)
    for k in KEYS:
        out[k] = inp[k].to(device).contiguous()
    return out


def slice_bh(inp, b, h):
    """The inputs of one (batch, head) as a batch-1, head-1 problem (CPU float64)."""
    return [oracle.f64(inp["x"][b:b + 1, :, h:h + 1]), oracle.f64(inp["B"][b:b + 1, :, h:h + 1]),
            oracle.f64(inp["C"][b:b + 1, :, h:h + 1]), oracle.f64(inp["dt"][b:b + 1, :, h:h + 1]),
            oracle.f64(inp["A"][h:h + 1]), oracle.f64(inp["lam"][b:b + 1, :, h:h + 1]),
            oracle.f64(inp["omega"][b:b + 1, :, h:h + 1])]


def oracle_sampled(inp, samples):
    """Oracle on the sampled (batch, head) sequences, stacked as heads of one
    batch-1 problem so that they run in parallel.  Returns per sample
    (y [1,T,1,R,P], final state [1,1,N,P], delayed-write cache [1,1,R*(N+P)])."""
    parts = [slice_bh(inp, b, h) for b, h in samples]
    stacked = []
    for i in range(7):
        if i == 4:   # A [1] per sample
            stacked.append(np.concatenate([p[i] for p in parts]))
        else:        # concatenate along the head axis (2)
            stacked.append(np.concatenate([p[i] for p in parts], axis=2))
    y, hT, prevT = oracle.scan(*stacked)
    return {s: (y[:, :, i:i + 1], hT[:, i:i + 1], prevT[:, i:i + 1]) for i, s in enumerate(samples)}


def oracle_full(inp):
    return oracle.scan(*[inp[k] for k in KEYS])


# Every comparison's achieved error, for the margin report at the end of the run (conftest.py).
MARGINS = []


def assert_close(got, ref, tol, what):
    err = oracle.rel_err(got, ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    MARGINS.append((test, what, float(err), float(tol)))
    assert err <= tol, f"{what}: max|err|/max|ref| = {err:.3e} > {tol:.0e}"
    return err
