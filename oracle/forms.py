"""Other float64 evaluations of the Mamba-3 recurrence, used to pin the oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Each function evaluates the same recurrence a different way, as derived on
abhik.ai/papers/mamba3 ("Mamba-3: Improved Sequence Modeling using State Space
Principles"), so that a mistake in any one of them shows up as a disagreement:

* ``mamba2_euler``      -- section 2.2: the lambda = 1, zero-rotation, rank-1
                            special case, h = exp(Delta A) h + Delta B x^T.
* ``matrix_form``       -- sections 3.1.2-3.1.3, Eq. 7 and panel 2: the
                            decay x lower two-band mask applied to the
                            rotated C B^T scores, materialised for small T.
* ``two_band_closed_form`` -- panel 2: the constant-coefficient closed form
                            L_ts = gamma alpha^(t-s) + [s<t] beta alpha^(t-s-1).
* ``complex_form``      -- Proposition 2: a diagonal complex state of size N/2
                            with transition alpha e^{i phi}, readout through
                            the conjugate of the complex C projection.
* ``rotating_frame``    -- Propositions 3-4, Eq. 11, panel 3: rotations moved
                            onto B and C by the cumulative phase, scalar
                            transition, the delayed write keeping its own phase.
* ``chunked``           -- section 3.3 (chunked algorithm): chunk-local
                            phases and log-decays, intra-chunk masked scores,
                            per-chunk state, inter-chunk state passing.
* ``state_passing``     -- the inter-chunk recurrence
                            H_c = exp(l_c) R(Theta_c) H_{c-1} + U_c.
* ``arithmetic_intensity`` -- Table 2 / panel 5 model of FLOPs per byte.

Rotation convention everywhere: R(theta)(a, b) = (a cos - b sin, a sin + b cos),
state pair j = components (2j, 2j+1), phi_{t,j} = Delta_t omega_{t,j}.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def _unpack(x, B, C, dt, A, lam, omega):
    return tuple(_f64(v) for v in (x, B, C, dt, A, lam, omega))


def a_per_token(A, dt):
    """The decay generator of every (batch, token, head): A [H] repeats over tokens;
    A [Bt,T,H] (the per-token A_t of Table 1) is taken as given."""
    A, dt = _f64(A), _f64(dt)
    return np.broadcast_to(A, dt.shape) if A.ndim == 1 else A


def rotate_pairs(v: np.ndarray, theta: np.ndarray) -> np.ndarray:
    """Rotate consecutive pairs (2j, 2j+1) of the last axis of ``v`` by ``theta[..., j]``."""
    a = v[..., 0::2]
    b = v[..., 1::2]
    c, s = np.cos(theta), np.sin(theta)
    out = np.empty(v.shape, dtype=np.float64)
    out[..., 0::2] = c * a - s * b
    out[..., 1::2] = s * a + c * b
    return out


def coefficients(dt, A, lam):
    """alpha, beta, gamma of the exponential-trapezoidal rule (Proposition 1, Eq. 6).

    dt, lam [..., T, H]; A [H] broadcast over the last axis, or A of dt's shape.
    """
    alpha = np.exp(dt * A)
    beta = (1.0 - lam) * dt * alpha
    gamma = lam * dt
    return alpha, beta, gamma


# ---------------------------------------------------------------------------
def mamba2_euler(x, B, C, dt, A):
    """Mamba-2 exponential-Euler recurrence (rank 1, no rotation, lambda = 1).

    h_t = exp(Delta_t A) h_{t-1} + Delta_t B_t x_t^T ; y_t = h_t^T C_t.
    x [Bt,T,H,1,P], B/C [Bt,T,H,1,N]; returns y [Bt,T,H,1,P].
    """
    x, B, C, dt, A = (_f64(v) for v in (x, B, C, dt, A))
    Bt, T, H, R, P = x.shape
    assert R == 1
    N = B.shape[-1]
    At = a_per_token(A, dt)
    y = np.zeros_like(x)
    h = np.zeros((Bt, H, N, P))
    for t in range(T):
        decay = np.exp(dt[:, t] * At[:, t])              # [Bt,H]
        write = B[:, t, :, 0, :, None] * x[:, t, :, 0, None, :]   # [Bt,H,N,P]
        h = decay[..., None, None] * h + dt[:, t][..., None, None] * write
        y[:, t, :, 0, :] = np.einsum("bhnp,bhn->bhp", h, C[:, t, :, 0, :])
    return y


# ---------------------------------------------------------------------------
def decay_matrix(dt, A):
    """D[t, s] = prod_{k=s+1..t} alpha_k for s <= t (1 on the diagonal), 0 above.

    dt [T] for one head; A scalar or [T] (per token).  Built as an explicit product, not from
    differences of cumulative sums, so it is exact for small T.
    """
    T = dt.shape[0]
    alpha = np.exp(dt * A)
    D = np.zeros((T, T))
    for t in range(T):
        D[t, t] = 1.0
        for s in range(t - 1, -1, -1):
            D[t, s] = D[t, s + 1] * alpha[s + 1]
    return D


def two_band_matrix(dt, A, lam):
    """L = decay x lower two-band operator for one head (Eq. 7 form).

    L[t, s] = D[t, s] gamma_s + [s < t] D[t, s+1] beta_{s+1}.
    """
    T = dt.shape[0]
    D = decay_matrix(dt, A)
    _, beta, gamma = coefficients(dt, A, lam)
    L = np.zeros((T, T))
    for t in range(T):
        for s in range(t + 1):
            L[t, s] = D[t, s] * gamma[s]
            if s < t:
                L[t, s] += D[t, s + 1] * beta[s + 1]
    return L


def two_band_closed_form(T: int, delta: float, a: float, weight: float) -> np.ndarray:
    """Constant-coefficient closed form of the causal operator (panel 2)."""
    alpha = np.exp(delta * a)
    beta = (1.0 - weight) * delta * alpha
    gamma = weight * delta
    L = np.zeros((T, T))
    for t in range(T):
        for s in range(t + 1):
            L[t, s] = gamma * alpha ** (t - s) + (beta * alpha ** (t - s - 1) if s < t else 0.0)
    return L


def matrix_form(x, B, C, dt, A, lam, omega):
    """Materialised masked-score evaluation (zero initial state), small T.

    For each (batch, head): Phi_t = sum_{i<=t} phi_i (global, inclusive),
    B~_t = R(-Phi_t) B_t, C~_t = R(-Phi_t) C_t per rank, and
    Y[(t,r), p] = sum_{s,r'} L[t,s] (C~_t[r] . B~_s[r']) X_s[r', p].
    """
    x, B, C, dt, A, lam, omega = _unpack(x, B, C, dt, A, lam, omega)
    Bt, T, H, R, P = x.shape
    At = a_per_token(A, dt)
    y = np.zeros_like(x)
    for b in range(Bt):
        for h in range(H):
            phi = dt[b, :, h, None] * omega[b, :, h, :]          # [T, N/2]
            Phi = np.cumsum(phi, axis=0)
            Bm = rotate_pairs(B[b, :, h], -Phi[:, None, :])     # [T, R, N]
            Cm = rotate_pairs(C[b, :, h], -Phi[:, None, :])
            L = two_band_matrix(dt[b, :, h], At[b, :, h], lam[b, :, h])  # [T, T]
            S = np.einsum("trn,sqn->trsq", Cm, Bm)               # [T,R,T,R]
            M = S * L[:, None, :, None]
            y[b, :, h] = np.einsum("trsq,sqp->trp", M, x[b, :, h])
    return y


# ---------------------------------------------------------------------------
def complex_form(x, B, C, dt, A, lam, omega):
    """Diagonal complex state (Proposition 2), zero initial state.

    z_{t,j} = alpha_t e^{i phi_{t,j}} z_{t-1,j} + beta_t e^{i phi_{t,j}} u_{t-1,j} + gamma_t u_{t,j}
    u_{t,j}[p] = sum_r (B_t[r,2j] + i B_t[r,2j+1]) X_t[r,p]
    y_t[r,p]  = sum_j Re( conj(C_t[r,2j] + i C_t[r,2j+1]) z_{t,j}[p] )
    """
    x, B, C, dt, A, lam, omega = _unpack(x, B, C, dt, A, lam, omega)
    Bt, T, H, R, P = x.shape
    N = B.shape[-1]
    Bc = B[..., 0::2] + 1j * B[..., 1::2]                     # [Bt,T,H,R,N/2]
    Cc = C[..., 0::2] + 1j * C[..., 1::2]
    alpha, beta, gamma = coefficients(dt, A, lam)              # [Bt,T,H]
    z = np.zeros((Bt, H, N // 2, P), dtype=np.complex128)
    u_prev = np.zeros_like(z)
    y = np.zeros_like(x)
    for t in range(T):
        rot = np.exp(1j * dt[:, t, :, None] * omega[:, t])     # [Bt,H,N/2]
        u = np.einsum("bhrj,bhrp->bhjp", Bc[:, t], x[:, t])
        z = (alpha[:, t, :, None, None] * rot[..., None] * z
             + beta[:, t, :, None, None] * rot[..., None] * u_prev
             + gamma[:, t, :, None, None] * u)
        y[:, t] = np.real(np.einsum("bhrj,bhjp->bhrp", np.conj(Cc[:, t]), z))
        u_prev = u
    return y


# ---------------------------------------------------------------------------
def rotating_frame(x, B, C, dt, A, lam, omega):
    """Rotations moved to B and C by the cumulative phase (Props 3-4, Eq. 11).

    Phi_t = sum_{i<=t} phi_i ;  v~_t = R(-Phi_t) B_t X_t^T ;
    h~_t = alpha_t h~_{t-1} + beta_t v~_{t-1} + gamma_t v~_t  (v~_{t-1} keeps Phi_{t-1}) ;
    y_t  = h~_t^T R(-Phi_t) C_t.
    """
    x, B, C, dt, A, lam, omega = _unpack(x, B, C, dt, A, lam, omega)
    Bt, T, H, R, P = x.shape
    N = B.shape[-1]
    alpha, beta, gamma = coefficients(dt, A, lam)
    Phi = np.cumsum(dt[..., None] * omega, axis=1)             # [Bt,T,H,N/2]
    hs = np.zeros((Bt, H, N, P))
    v_prev = np.zeros_like(hs)
    y = np.zeros_like(x)
    for t in range(T):
        Bm = rotate_pairs(B[:, t], -Phi[:, t, :, None, :])      # [Bt,H,R,N]
        Cm = rotate_pairs(C[:, t], -Phi[:, t, :, None, :])
        v = np.einsum("bhrn,bhrp->bhnp", Bm, x[:, t])
        hs = (alpha[:, t, :, None, None] * hs + beta[:, t, :, None, None] * v_prev
              + gamma[:, t, :, None, None] * v)
        y[:, t] = np.einsum("bhnp,bhrn->bhrp", hs, Cm)
        v_prev = v
    return y


# ---------------------------------------------------------------------------
def state_passing(U, logdecay, angle, init=None):
    """Inter-chunk recurrence H_c = exp(l_c) R(Theta_c) H_{c-1} + U_c.

    U [b,H,nc,N,P]; logdecay [b,H,nc]; angle [b,H,nc,N/2]; init [b,H,N,P] or None (zero).
    Returns (carries [b,H,nc,N,P] with carries[:,:,c] = H_{c-1}, final = H_{nc-1}).
    The rotation acts on state rows (2j, 2j+1).
    """
    U, logdecay, angle = _f64(U), _f64(logdecay), _f64(angle)
    b, H, nc, N, P = U.shape
    Hc = np.zeros((b, H, N, P)) if init is None else _f64(init).copy()
    carries = np.zeros_like(U)
    for c in range(nc):
        carries[:, :, c] = Hc
        th = angle[:, :, c]                                     # [b,H,N/2]
        cs, sn = np.cos(th)[..., None], np.sin(th)[..., None]
        h0, h1 = Hc[:, :, 0::2, :], Hc[:, :, 1::2, :]
        rot = np.empty_like(Hc)
        rot[:, :, 0::2, :] = cs * h0 - sn * h1
        rot[:, :, 1::2, :] = sn * h0 + cs * h1
        Hc = np.exp(logdecay[:, :, c])[..., None, None] * rot + U[:, :, c]
    return carries, Hc


def chunked(x, B, C, dt, A, lam, omega, Q: int):
    """Chunked evaluation (zero initial state) with chunk length Q tokens.

    Per chunk c = tokens [c0, c1):
      l_t = Delta_t A_t ; cum_t = sum_{k=c0..t} l_k ; Psi_t = sum_{k=c0..t} phi_k ; Theta_c = Psi_{c1-1}
      gamma_t = lambda_t Delta_t ; w_s = gamma_s + (1 - lambda_{s+1}) Delta_{s+1}
        (for s = c1-1 the next token's lambda, Delta; 0 past the end of the sequence)
      B~_s = R(-Psi_s) B_s ; C~_t = R(-Psi_t) C_t
      intra:  Y_t += sum_{s<=t} exp(cum_t - cum_s) (gamma_t if s == t else w_s) (C~_t . B~_s) X_s
      inter:  Y_t += exp(cum_t) C~_t^T H_{c-1}
      chunk state: U_c = R(Theta_c) sum_s exp(cum_{c1-1} - cum_s) w_s B~_s X_s^T
      state passing: H_c = exp(cum_{c1-1}) R(Theta_c) H_{c-1} + U_c,  H_{-1} = 0.
    H is the physical-frame state plus the pending delayed write of the chunk's
    last token; for the final chunk it is the true final state h_{T-1}.
    Returns (y, final_state).
    """
    x, B, C, dt, A, lam, omega = _unpack(x, B, C, dt, A, lam, omega)
    Bt, T, H, R, P = x.shape
    N = B.shape[-1]
    At = a_per_token(A, dt)
    nc = (T + Q - 1) // Q
    y = np.zeros_like(x)
    finals = np.zeros((Bt, H, N, P))
    for b in range(Bt):
        for h in range(H):
            Ucs = np.zeros((1, 1, nc, N, P))
            lds = np.zeros((1, 1, nc))
            angs = np.zeros((1, 1, nc, N // 2))
            per_chunk = []
            for c in range(nc):
                c0, c1 = c * Q, min(T, (c + 1) * Q)
                d = dt[b, c0:c1, h]
                lm = lam[b, c0:c1, h]
                ell = d * At[b, c0:c1, h]
                cum = np.cumsum(ell)
                Psi = np.cumsum(d[:, None] * omega[b, c0:c1, h, :], axis=0)  # [q, N/2]
                gam = lm * d
                nxt_d = np.append(d[1:], dt[b, c1, h] if c1 < T else 0.0)
                nxt_l = np.append(lm[1:], lam[b, c1, h] if c1 < T else 1.0)
                w = gam + (1.0 - nxt_l) * nxt_d
                Bm = rotate_pairs(B[b, c0:c1, h], -Psi[:, None, :])   # [q,R,N]
                Cm = rotate_pairs(C[b, c0:c1, h], -Psi[:, None, :])
                X = x[b, c0:c1, h]                                     # [q,R,P]
                q = c1 - c0
                Lloc = np.zeros((q, q))
                for t in range(q):
                    for s in range(t + 1):
                        Lloc[t, s] = np.exp(cum[t] - cum[s]) * (gam[t] if s == t else w[s])
                S = np.einsum("trn,sqn->trsq", Cm, Bm)
                y[b, c0:c1, h] = np.einsum("trsq,sqp->trp", S * Lloc[:, None, :, None], X)
                wt = np.exp(cum[-1] - cum) * w                         # [q]
                U = np.einsum("s,srn,srp->np", wt, Bm, X)
                U = rotate_pairs(U.T, Psi[-1][None, :]).T              # rotate rows by Theta_c
                Ucs[0, 0, c] = U
                lds[0, 0, c] = cum[-1]
                angs[0, 0, c] = Psi[-1]
                per_chunk.append((c0, c1, cum, Cm))
            carries, fin = state_passing(Ucs, lds, angs)
            for c, (c0, c1, cum, Cm) in enumerate(per_chunk):
                Hprev = carries[0, 0, c]
                y[b, c0:c1, h] += np.exp(cum)[:, None, None] * np.einsum("trn,np->trp", Cm, Hprev)
            finals[b, h] = fin[0, 0]
    return y, finals


# ---------------------------------------------------------------------------
def arithmetic_intensity(N: int, P: int, R: int) -> float:
    """Table 2 model (2-byte values): (4NPR + NP - PR) / (2 (1 + 2NR + PR + NP))."""
    flops = 4 * N * P * R + N * P - P * R
    nbytes = 2 * (1 + 2 * N * R + P * R + N * P)
    return flops / nbytes
