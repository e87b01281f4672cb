/*
 * Float64 CPU oracle of the Mamba-3 SSM layer recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header or constant with the CUDA library.
 *
 * It is the plain sequential definition, evaluated one token at a time in the
 * physical (unrotated) frame, following "Mamba-3: Improved Sequence Modeling
 * using State Space Principles" as presented on abhik.ai/papers/mamba3:
 *
 *   - exponential-trapezoidal rule (Proposition 1, Eq. 6 and panel 1):
 *       alpha_t = exp(Delta_t A),  beta_t = (1 - lambda_t) Delta_t alpha_t,
 *       gamma_t = lambda_t Delta_t,
 *       h_t = alpha_t h_{t-1} + beta_t v_{t-1} + gamma_t v_t,
 *     with h_{-1} = v_{-1} = 0 unless a carried state is supplied;
 *   - complex state as real pairs with data-dependent rotation (Propositions
 *     2-4, panel 3): in the physical frame the retained state and the delayed
 *     write are both rotated by the current angle phi_t before the current
 *     write is added; state pair j is rows (2j, 2j+1) and phi_{t,j} =
 *     Delta_t * omega_{t,j}; R(phi) maps (a, b) to
 *     (a cos phi - b sin phi, a sin phi + b cos phi);
 *   - MIMO rank R (section 3.3, Eqs. 12-14, panel 4): the write is
 *     v_t = B_t X_t^T (N x P, B_t is N x R and X_t is P x R) and the readout
 *     is Y_t = h_t^T C_t (P x R).
 *
 * Layouts: x [Bt,T,H,R,P], B and C [Bt,T,H,R,N], dt and lam [Bt,T,H], A [H]
 * (m3o_scan) or [Bt,T,H] (m3o_scan_tok: the per-token A_t of Table 1),
 * omega [Bt,T,H,N/2], y [Bt,T,H,R,P], states [Bt,H,N,P], the delayed-write
 * cache [Bt,H,R*N + R*P] = (B_{t-1} as [R,N], then X_{t-1} as [R,P]).
 *
 * Build: gcc -O2 -fopenmp -fPIC -shared (no -ffast-math).  Independent
 * (batch, head) sequences run on separate OpenMP threads; the arithmetic of
 * each sequence is in the order written here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define M3O_OK 0
#define M3O_BAD_SHAPE -1
#define M3O_BAD_PARAM -2
#define M3O_NO_MEMORY -3

/* Precondition of the coefficient helper on the page (panel 1):
 * finite values, Delta >= 0, A <= 0, lambda in [0, 1]. */
static int params_ok(double d, double a, double l) {
    if (!isfinite(d) || !isfinite(a) || !isfinite(l)) return 0;
    if (d < 0.0 || a > 0.0 || l < 0.0 || l > 1.0) return 0;
    return 1;
}

int m3o_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One (batch, head) sequence.  h: [N*P] in/out; bprev [R*N], xprev [R*P]
 * in/out (the factors of v_{t-1}).  Scratch v, vp: [N*P].  The decay
 * generator of token t is a_seq[t * a_stride] (a_stride 0: one A per head). */
static int scan_one(const double* x, const double* B, const double* C, const double* dt,
                    const double* a_seq, int64_t a_stride, const double* lam, const double* omega,
                    int64_t T, int64_t H, int64_t P, int64_t N, int64_t R,
                    double* h, double* bprev, double* xprev, double* v, double* vp,
                    double* y) {
    const int64_t tokstride_x = H * R * P;    /* x, y: next token of this head */
    const int64_t tokstride_b = H * R * N;    /* B, C */
    const int64_t tokstride_s = H;            /* dt, lam */
    const int64_t tokstride_w = H * (N / 2);  /* omega */
    for (int64_t t = 0; t < T; ++t) {
        const double* xt = x + t * tokstride_x;
        const double* bt = B + t * tokstride_b;
        const double* ct = C + t * tokstride_b;
        const double* wt = omega + t * tokstride_w;
        const double d = dt[t * tokstride_s];
        const double l = lam[t * tokstride_s];
        const double a = a_seq[t * a_stride];
        if (!params_ok(d, a, l)) return M3O_BAD_PARAM;
        const double alpha = exp(d * a);
        const double beta = (1.0 - l) * d * alpha;
        const double gamma = l * d;

        /* delayed write v_{t-1} = B_{t-1} X_{t-1}^T and current write v_t = B_t X_t^T */
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t p = 0; p < P; ++p) {
                double sp = 0.0, sc = 0.0;
                for (int64_t r = 0; r < R; ++r) {
                    sp += bprev[r * N + n] * xprev[r * P + p];
                    sc += bt[r * N + n] * xt[r * P + p];
                }
                vp[n * P + p] = sp;
                v[n * P + p] = sc;
            }
        }
        /* h <- R(phi_t) (alpha h + beta v_{t-1}) + gamma v_t, pair by pair */
        for (int64_t j = 0; j < N / 2; ++j) {
            const double phi = d * wt[j];
            const double cs = cos(phi), sn = sin(phi);
            double* h0 = h + (2 * j) * P;
            double* h1 = h + (2 * j + 1) * P;
            const double* vp0 = vp + (2 * j) * P;
            const double* vp1 = vp + (2 * j + 1) * P;
            const double* v0 = v + (2 * j) * P;
            const double* v1 = v + (2 * j + 1) * P;
            for (int64_t p = 0; p < P; ++p) {
                const double u0 = alpha * h0[p] + beta * vp0[p];
                const double u1 = alpha * h1[p] + beta * vp1[p];
                h0[p] = cs * u0 - sn * u1 + gamma * v0[p];
                h1[p] = sn * u0 + cs * u1 + gamma * v1[p];
            }
        }
        /* Y_t = h_t^T C_t : y[r][p] = sum_n h[n][p] C_t[r][n] */
        double* yt = y + t * tokstride_x;
        for (int64_t r = 0; r < R; ++r) {
            for (int64_t p = 0; p < P; ++p) {
                double s = 0.0;
                for (int64_t n = 0; n < N; ++n) s += h[n * P + p] * ct[r * N + n];
                yt[r * P + p] = s;
            }
        }
        /* the current write becomes the next step's delayed write */
        memcpy(bprev, bt, sizeof(double) * (size_t)(R * N));
        memcpy(xprev, xt, sizeof(double) * (size_t)(R * P));
    }
    return M3O_OK;
}

static int scan_all(const double* x, const double* B, const double* C, const double* dt,
                    const double* A, int per_token, const double* lam, const double* omega,
                    int64_t Bt, int64_t T, int64_t H, int64_t P, int64_t N, int64_t R,
                    const double* h0, const double* prev, double* y, double* hT, double* prevT) {
    if (Bt < 0 || T < 0 || H < 1 || P < 1 || N < 2 || (N % 2) != 0 || R < 1) return M3O_BAD_SHAPE;
    const int64_t NP = N * P;
    const int64_t KV = R * (N + P);
    int status = M3O_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < Bt * H; ++bh) {
        const int64_t b = bh / H, hh = bh % H;
        double* work = (double*)malloc(sizeof(double) * (size_t)(3 * NP + KV));
        if (!work) {
#pragma omp atomic write
            status = M3O_NO_MEMORY;
            continue;
        }
        double* h = work;
        double* v = work + NP;
        double* vp = work + 2 * NP;
        double* bprev = work + 3 * NP;
        double* xprev = bprev + R * N;
        if (h0) memcpy(h, h0 + bh * NP, sizeof(double) * (size_t)NP);
        else memset(h, 0, sizeof(double) * (size_t)NP);
        if (prev) memcpy(bprev, prev + bh * KV, sizeof(double) * (size_t)KV);
        else memset(bprev, 0, sizeof(double) * (size_t)KV);
        const int64_t base_x = (b * T * H + hh) * R * P;
        const int64_t base_b = (b * T * H + hh) * R * N;
        const int64_t base_s = b * T * H + hh;
        const int64_t base_w = (b * T * H + hh) * (N / 2);
        const double* a_seq = per_token ? A + base_s : A + hh;
        int st = scan_one(x + base_x, B + base_b, C + base_b, dt + base_s, a_seq, per_token ? H : 0,
                          lam + base_s, omega + base_w, T, H, P, N, R, h, bprev, xprev, v, vp, y + base_x);
        if (st != M3O_OK) {
#pragma omp atomic write
            status = st;
        }
        if (hT) memcpy(hT + bh * NP, h, sizeof(double) * (size_t)NP);
        if (prevT) memcpy(prevT + bh * KV, bprev, sizeof(double) * (size_t)KV);
        free(work);
    }
    return status;
}

/*
 * Sequential scan over T tokens for every (batch, head), one A per head.
 *   h0    nullable: initial state [Bt,H,N,P] (zero if NULL)
 *   prev  nullable: initial delayed-write factors [Bt,H,R*(N+P)] (zero if NULL)
 *   y     out [Bt,T,H,R,P]
 *   hT    nullable out: state after the last token [Bt,H,N,P]
 *   prevT nullable out: delayed-write factors after the last token
 * A decode step is this function with T = 1 and the carried h0 / prev.
 * Returns 0, or a negative code for bad shapes or violated preconditions.
 */
int m3o_scan(const double* x, const double* B, const double* C, const double* dt,
             const double* A, const double* lam, const double* omega,
             int64_t Bt, int64_t T, int64_t H, int64_t P, int64_t N, int64_t R,
             const double* h0, const double* prev, double* y, double* hT, double* prevT) {
    return scan_all(x, B, C, dt, A, 0, lam, omega, Bt, T, H, P, N, R, h0, prev, y, hT, prevT);
}

/* The same with a decay generator per token: A_tok [Bt,T,H] (the A_t of the
 * time-varying discretizations, Table 1). */
int m3o_scan_tok(const double* x, const double* B, const double* C, const double* dt,
                 const double* A_tok, const double* lam, const double* omega,
                 int64_t Bt, int64_t T, int64_t H, int64_t P, int64_t N, int64_t R,
                 const double* h0, const double* prev, double* y, double* hT, double* prevT) {
    return scan_all(x, B, C, dt, A_tok, 1, lam, omega, Bt, T, H, P, N, R, h0, prev, y, hT, prevT);
}
