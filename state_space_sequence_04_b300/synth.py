"""Seeded synthetic inputs for the Mamba-3 SSM layer recurrence.

This module only draws random tensors.  It holds none of the layer's
arithmetic: it is shared by the tests, the benchmark and the float64 oracle so
that every side reads identical values.

Layouts (row-major, time-major; ``R`` is the MIMO rank):

    x      [Bt, T, H, R, P]   io dtype (bf16 or fp32)
    B, C   [Bt, T, H, R, N]   io dtype
    dt     [Bt, T, H]         fp32   (Delta_t, already positive)
    A      [H]                fp32   (per-head decay generator, negative)
    lam    [Bt, T, H]         fp32   (lambda_t in [0, 1])
    omega  [Bt, T, H, N/2]    fp32   (rotation frequency per state pair)

Distributions follow the workloads of "Mamba-3: Improved Sequence Modeling
using State Space Principles": x ~ N(0,1); B, C ~ N(0, 1/N);
dt = softplus(N(mu, sd)); A = -exp(U(0, ln 16)) per head;
lambda = sigmoid(N(0,1)) (or U(0,1) for the long-context workload);
omega ~ U(-pi, pi) per state pair per step.

Draw order is fixed: x, B, C, dt, A, lambda, omega.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and distribution recipe of one synthetic workload."""

    name: str
    batch: int
    heads: int
    seqlen: int
    headdim: int          # P
    dstate: int           # N (even)
    rank: int = 1         # R
    chunk: int = 64       # Q, tokens per chunk
    io: str = "bf16"      # dtype of x, B, C, y
    dt_mu: float = -3.0
    dt_sd: float = 1.0
    lam_uniform: bool = False

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


# The named workloads.  Sizes are the ones the method's paper-style workloads
# use: a tiny fp32 check, SISO prefill at ~1.5B layer width, MIMO prefill,
# and long-context MIMO prefill.
TINY = Workload("tiny_fp32_b1_h2_T256_P16_N16_R1_Q64", 1, 2, 256, 16, 16, 1, 64, "fp32")
SISO_1P5B = Workload("siso_prefill_b4_h64_T4096_P64_N128_R1_Q64", 4, 64, 4096, 64, 128, 1, 64, "bf16")
MIMO_R4 = Workload("mimo_prefill_b2_h32_T8192_P64_N64_R4_Q64", 2, 32, 8192, 64, 64, 4, 64, "bf16")
LONG_MIMO = Workload("long_mimo_prefill_b1_h64_T65536_P64_N128_R4_Q128", 1, 64, 65536, 64, 128, 4, 128,
                     "bf16", dt_mu=-4.0, dt_sd=1.5, lam_uniform=True)

WORKLOADS = {w.name: w for w in (TINY, SISO_1P5B, MIMO_R4, LONG_MIMO)}

# Decode sweep: batch sizes and ranks at H=64, P=64, N=128, 1024 carried steps.
DECODE_BATCHES = (1, 8, 64, 256)
DECODE_RANKS = (1, 4)
DECODE_STEPS = 1024


def io_torch_dtype(io: str) -> torch.dtype:
    if io == "bf16":
        return torch.bfloat16
    if io == "fp32":
        return torch.float32
    raise ValueError(f"unknown io dtype {io!r}")


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_inputs(w: Workload, seed: int = 0, device="cpu", seqlen: Optional[int] = None,
                batch: Optional[int] = None) -> dict:
    """Draw one workload's prefill inputs.

    ``seqlen``/``batch`` override the workload's sizes (used to build small
    cases with the same distributions).  Returns a dict of tensors on
    ``device``; x, B, C are in the io dtype, the rest fp32.
    """
    Bt = w.batch if batch is None else batch
    T = w.seqlen if seqlen is None else seqlen
    H, P, N, R = w.heads, w.headdim, w.dstate, w.rank
    if N % 2:
        raise ValueError("N must be even")
    g = _gen(seed, device)
    io = io_torch_dtype(w.io)
    f32 = torch.float32
    x = torch.randn((Bt, T, H, R, P), generator=g, device=device, dtype=f32)
    B = torch.randn((Bt, T, H, R, N), generator=g, device=device, dtype=f32) * (1.0 / math.sqrt(N))
    C = torch.randn((Bt, T, H, R, N), generator=g, device=device, dtype=f32) * (1.0 / math.sqrt(N))
    dt = torch.nn.functional.softplus(
        torch.randn((Bt, T, H), generator=g, device=device, dtype=f32) * w.dt_sd + w.dt_mu)
    A = -torch.exp(torch.rand((H,), generator=g, device=device, dtype=f32) * math.log(16.0))
    if w.lam_uniform:
        lam = torch.rand((Bt, T, H), generator=g, device=device, dtype=f32)
    else:
        lam = torch.sigmoid(torch.randn((Bt, T, H), generator=g, device=device, dtype=f32))
    omega = (torch.rand((Bt, T, H, N // 2), generator=g, device=device, dtype=f32) * 2.0 - 1.0) * math.pi
    return {
        "x": x.to(io), "B": B.to(io), "C": C.to(io), "dt": dt, "A": A, "lam": lam, "omega": omega,
        "R": R, "chunk": w.chunk, "io": w.io,
    }


def make_prep_inputs(w: Workload, seed: int = 0, device="cpu", seqlen: Optional[int] = None,
                     batch: Optional[int] = None) -> dict:
    """Prefill inputs in pre-activation form, for the entry points that derive
    Delta and lambda inside the kernels and take one decay generator per token.

    Draw order: x, B, C, dt_raw, dt_bias, A (per token), u, omega.
      dt_raw [Bt,T,H] ~ N(dt_mu, dt_sd)      (Delta = softplus(dt_raw + dt_bias))
      dt_bias [H]     ~ U(-0.5, 0.5)
      A [Bt,T,H]      = -exp(U(0, ln 16))    (one decay generator per token)
      u [Bt,T,H]      ~ N(0, 1), or logit(U(0,1)) for lam_uniform workloads (lambda = sigmoid(u))
    x, B, C, omega as in ``make_inputs``.
    """
    Bt = w.batch if batch is None else batch
    T = w.seqlen if seqlen is None else seqlen
    H, P, N, R = w.heads, w.headdim, w.dstate, w.rank
    if N % 2:
        raise ValueError("N must be even")
    g = _gen(seed, device)
    io = io_torch_dtype(w.io)
    f32 = torch.float32
    x = torch.randn((Bt, T, H, R, P), generator=g, device=device, dtype=f32)
    B = torch.randn((Bt, T, H, R, N), generator=g, device=device, dtype=f32) * (1.0 / math.sqrt(N))
    C = torch.randn((Bt, T, H, R, N), generator=g, device=device, dtype=f32) * (1.0 / math.sqrt(N))
    dt_raw = torch.randn((Bt, T, H), generator=g, device=device, dtype=f32) * w.dt_sd + w.dt_mu
    dt_bias = torch.rand((H,), generator=g, device=device, dtype=f32) - 0.5
    A = -torch.exp(torch.rand((Bt, T, H), generator=g, device=device, dtype=f32) * math.log(16.0))
    if w.lam_uniform:
        p = torch.rand((Bt, T, H), generator=g, device=device, dtype=f32).clamp(1e-6, 1 - 1e-6)
        u = torch.log(p) - torch.log1p(-p)
    else:
        u = torch.randn((Bt, T, H), generator=g, device=device, dtype=f32)
    omega = (torch.rand((Bt, T, H, N // 2), generator=g, device=device, dtype=f32) * 2.0 - 1.0) * math.pi
    return {
        "x": x.to(io), "B": B.to(io), "C": C.to(io), "dt_raw": dt_raw, "dt_bias": dt_bias, "A": A, "u": u,
        "omega": omega, "R": R, "chunk": w.chunk, "io": w.io,
    }


def make_bc_params(heads: int, rank: int, dstate: int, seed: int = 7, device="cpu") -> dict:
    """Parameters of the B / C normalisation and channel biases.

    Draw order: B_gain, C_gain [N] ~ 1 + 0.1 N(0,1); B_bias, C_bias [H, R, N] ~ 0.1 N(0,1).
    eps = 1e-5.
    """
    g = _gen(seed, device)
    f32 = torch.float32
    N = dstate
    B_gain = 1.0 + 0.1 * torch.randn((N,), generator=g, device=device, dtype=f32)
    C_gain = 1.0 + 0.1 * torch.randn((N,), generator=g, device=device, dtype=f32)
    B_bias = 0.1 * torch.randn((heads, rank, N), generator=g, device=device, dtype=f32)
    C_bias = 0.1 * torch.randn((heads, rank, N), generator=g, device=device, dtype=f32)
    return {"norm": True, "eps": 1e-5, "B_gain": B_gain, "C_gain": C_gain, "B_bias": B_bias, "C_bias": C_bias}


def make_gate(shape, io: str = "bf16", seed: int = 9, device="cpu") -> torch.Tensor:
    """The output gate's input z (y's shape) ~ N(0, 1.5^2), in the io dtype."""
    g = _gen(seed, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 1.5).to(io_torch_dtype(io))


def make_decode_state(batch: int, heads: int, dstate: int, headdim: int, seed: int = 0,
                      device="cpu") -> torch.Tensor:
    """fp32 state [b, H, N, P] ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn((batch, heads, dstate, headdim), generator=g, device=device, dtype=torch.float32)


def make_decode_steps(batch: int, heads: int, headdim: int, dstate: int, rank: int, steps: int,
                      io: str = "bf16", seed: int = 1, device="cpu", dt_mu: float = -3.0,
                      dt_sd: float = 1.0, lam_uniform: bool = False, A: Optional[torch.Tensor] = None) -> dict:
    """Per-step decode inputs for ``steps`` consecutive tokens, stacked on dim 0.

    x [S, b, H, R, P], B/C [S, b, H, R, N] (io dtype), dt/lam [S, b, H],
    omega [S, b, H, N/2] (fp32) and A [H] (fp32, drawn unless given).
    """
    g = _gen(seed, device)
    iot = io_torch_dtype(io)
    f32 = torch.float32
    S, b, H, P, N, R = steps, batch, heads, headdim, dstate, rank
    x = torch.randn((S, b, H, R, P), generator=g, device=device, dtype=f32)
    Bm = torch.randn((S, b, H, R, N), generator=g, device=device, dtype=f32) * (1.0 / math.sqrt(N))
    Cm = torch.randn((S, b, H, R, N), generator=g, device=device, dtype=f32) * (1.0 / math.sqrt(N))
    dt = torch.nn.functional.softplus(torch.randn((S, b, H), generator=g, device=device, dtype=f32) * dt_sd + dt_mu)
    if A is None:
        A = -torch.exp(torch.rand((H,), generator=g, device=device, dtype=f32) * math.log(16.0))
    if lam_uniform:
        lam = torch.rand((S, b, H), generator=g, device=device, dtype=f32)
    else:
        lam = torch.sigmoid(torch.randn((S, b, H), generator=g, device=device, dtype=f32))
    omega = (torch.rand((S, b, H, N // 2), generator=g, device=device, dtype=f32) * 2.0 - 1.0) * math.pi
    return {"x": x.to(iot), "B": Bm.to(iot), "C": Cm.to(iot), "dt": dt, "A": A, "lam": lam,
            "omega": omega, "R": R, "io": io}


def make_decode_prep_steps(batch: int, heads: int, headdim: int, dstate: int, rank: int, steps: int,
                           io: str = "bf16", seed: int = 1, device="cpu", dt_mu: float = -3.0,
                           dt_sd: float = 1.0) -> dict:
    """Per-step decode inputs in pre-activation form, stacked on dim 0.

    Draw order: x, B, C, dt_raw, dt_bias, A, u, omega.  x [S, b, H, R, P], B/C
    [S, b, H, R, N] (io dtype); dt_raw ~ N(dt_mu, dt_sd), A = -exp(U(0, ln 16))
    and u ~ N(0, 1), each [S, b, H]; dt_bias [H] ~ U(-0.5, 0.5); omega [S, b, H, N/2].
    """
    g = _gen(seed, device)
    iot = io_torch_dtype(io)
    f32 = torch.float32
    S, b, H, P, N, R = steps, batch, heads, headdim, dstate, rank
    x = torch.randn((S, b, H, R, P), generator=g, device=device, dtype=f32)
    Bm = torch.randn((S, b, H, R, N), generator=g, device=device, dtype=f32) * (1.0 / math.sqrt(N))
    Cm = torch.randn((S, b, H, R, N), generator=g, device=device, dtype=f32) * (1.0 / math.sqrt(N))
    dt_raw = torch.randn((S, b, H), generator=g, device=device, dtype=f32) * dt_sd + dt_mu
    dt_bias = torch.rand((H,), generator=g, device=device, dtype=f32) - 0.5
    A = -torch.exp(torch.rand((S, b, H), generator=g, device=device, dtype=f32) * math.log(16.0))
    u = torch.randn((S, b, H), generator=g, device=device, dtype=f32)
    omega = (torch.rand((S, b, H, N // 2), generator=g, device=device, dtype=f32) * 2.0 - 1.0) * math.pi
    return {"x": x.to(iot), "B": Bm.to(iot), "C": Cm.to(iot), "dt_raw": dt_raw, "dt_bias": dt_bias, "A": A,
            "u": u, "omega": omega, "R": R, "io": io}


def make_state_passing_inputs(batch: int, heads: int, nchunks: int, dstate: int, headdim: int,
                              seed: int = 2, device="cpu") -> dict:
    """Inputs of the inter-chunk state-passing scan.

    chunk_states [b, H, nc, N, P] ~ N(0,1); chunk_logdecay [b, H, nc] = -softplus(N(1, 1))
    (sums of Delta*A over a chunk are negative); chunk_angle [b, H, nc, N/2] ~ U(-pi, pi);
    init_state [b, H, N, P] ~ N(0, 1).
    """
    g = _gen(seed, device)
    f32 = torch.float32
    U = torch.randn((batch, heads, nchunks, dstate, headdim), generator=g, device=device, dtype=f32)
    ld = -torch.nn.functional.softplus(torch.randn((batch, heads, nchunks), generator=g, device=device, dtype=f32) + 1.0)
    ang = (torch.rand((batch, heads, nchunks, dstate // 2), generator=g, device=device, dtype=f32) * 2 - 1) * math.pi
    h0 = torch.randn((batch, heads, dstate, headdim), generator=g, device=device, dtype=f32)
    return {"chunk_states": U, "chunk_logdecay": ld, "chunk_angle": ang, "init_state": h0}
