// Backward pass of the Mamba-3 SSM layer recurrence (training): the gradients
// of a loss L with respect to x, B, C, dt, A, lambda, omega, given the adjoint
// seeds dy = dL/dy and (optionally) dL/d final_state.
//
// Forward recurrence ("Mamba-3: Improved Sequence Modeling using State Space
// Principles", Proposition 1 / Eq. 6, rotation of Propositions 2-4, MIMO
// readout of section 3.3), per (batch, head), physical frame:
//   alpha_t = exp(Delta_t A), beta_t = (1 - lambda_t) Delta_t alpha_t, gamma_t = lambda_t Delta_t,
//   phi_{t,j} = Delta_t omega_{t,j},  v_t = B_t^T X_t (N x P),
//   u_t = alpha_t h_{t-1} + beta_t v_{t-1},  h_t = R(phi_t) u_t + gamma_t v_t,  y_t = h_t^T C_t.
// Adjoint, backwards in time (gbar_t = dL/dh_t, ubar_t = dL/du_t):
//   gbar_t = C_t dy_t^T + alpha_{t+1} ubar_{t+1} (+ dL/dh_{T-1} at the end),
//   ubar_t = R(phi_t)^T gbar_t,  dv_t = gamma_t gbar_t + beta_{t+1} ubar_{t+1},
//   dC_t = h_t dy_t (over p),  dB_t = dv_t X_t (over p),  dX_t = B_t dv_t (over n),
//   dalpha_t = <ubar_t, h_{t-1}>, dbeta_t = <ubar_t, v_{t-1}>, dgamma_t = <gbar_t, v_t>,
//   dphi_{t,j} = sum_p (gbar[2j+1] r[2j] - gbar[2j] r[2j+1]),  r = h_t - gamma_t v_t = R(phi_t) u_t,
// and the chain rule through alpha, beta, gamma, phi to Delta, lambda, A, omega.
//
// Work split: CTA (batch*head, pair block) owns the state rows (2j, 2j+1) of
// PB consecutive pairs j and every column p; thread (pair, c4) holds columns
// 4 c4 .. 4 c4 + 3 of one pair.  Pairs evolve independently (the rotation acts
// within a pair, the decay is a scalar), so only the sums over n (dX and the
// per-token scalars dalpha, dbeta, dgamma, sum_j omega_j dphi_j) cross CTAs:
// each pair block writes partial sums per token, and a finishing kernel adds
// them and applies the chain rule for Delta, lambda and A.
//
// Checkpointing: a forward sweep stores the state entering every chunk of Q
// tokens; the reverse sweep then, chunk by chunk from the last, recomputes the
// chunk's Q states from its checkpoint into shared memory and runs the adjoint
// over the chunk.  Both sweeps receive a chunk's inputs by cp.async into one
// half of a double buffer while the previous chunk is processed, and convert
// them to fp32 working copies.  Arithmetic is fp32, two lanes per instruction
// (f32x2), each lane rounded as the scalar instruction rounds it.
#include <cuda_bf16.h>

#include "m3_common.cuh"

namespace m3 {
namespace {

constexpr int kBwdThreads = 128;

template <int V>
struct Log2 {
    static constexpr int v = V <= 1 ? 0 : 1 + Log2<V / 2>::v;
};
template <>
struct Log2<1> {
    static constexpr int v = 0;
};

template <int R>
struct kLg {
    static constexpr int v = R == 1 ? 0 : (R == 2 ? 1 : (R == 4 ? 2 : 3));
};

// tokens per chunk: the staged inputs and dX partials grow with R
template <int R>
struct BwdChunk {
    static constexpr int Q = R <= 2 ? 8 : 4;
};

__host__ __device__ constexpr int round4(int v) { return (v + 3) & ~3; }

// Shared-memory sections (offsets in floats, each on a 16-byte boundary):
//   sB   [Q+1][PB][R] float2   B rows (2j, 2j+1), slot q <-> token t0 - 1 + q
//   sX   [Q+1][R][P]           X, same slots
//   sC   [Q][PB][R] float2     C rows, slot q <-> token t0 + q
//   sDy  [Q][R][P]             dy
//   sCS  [Q][PB] float2        (cos, sin) of phi_{t,j}
//   sW   [Q][PB]               omega_{t,j}
//   sABG [Q] float4            (alpha, beta, gamma, Delta)
//   sDx  [Q][warps][R][P]      dX partial sums of each warp
//   sScal[Q][PB][4]            per-pair (dalpha, dbeta, dgamma, omega dphi) partials
//   sS   [Q][2][threads] float4 the chunk's recomputed states
//   raw  [2] copy buffers: the loaded inputs of a chunk as stored in global memory (io dtype for B, X,
//        C, dy; fp32 for omega, Delta, lambda), element for element in the order of sB .. sL; the next
//        chunk's copies land in one while the current chunk is converted from the other
struct BwdLayout {
    int PB, lgPB, lgP, threads, nPB;
    int oB, oX, oC, oDy, oCS, oW, oABG, oDx, oScal, oS, oRaw, total;
    int rX, rC, rDy, rW, rDt, rL, rA, rawBytes;   // byte offsets within a copy buffer, and its size
    int unitXY;                               // bytes per copy of an X / dy row (16 or 4)
};

__host__ __device__ constexpr int round16(int v) { return (v + 15) & ~15; }

BwdLayout bwd_layout(int P, int N, int R, int Q, int e, bool gate = false) {
    BwdLayout L{};
    const int P4 = P / 4, NP2 = N / 2;
    int PB = kBwdThreads / P4;   // a power of two, the smallest one >= N/2 if that is smaller
    if (PB < 1) PB = 1;
    while (PB > 1 && PB / 2 >= NP2) PB /= 2;
    L.PB = PB;
    L.lgPB = 0;
    while ((1 << L.lgPB) < PB) ++L.lgPB;
    L.lgP = 0;
    while ((1 << L.lgP) < P) ++L.lgP;
    L.threads = (PB * P4 + 31) / 32 * 32;   // whole warps; threads past PB * P4 idle
    L.nPB = (NP2 + PB - 1) / PB;
    int o = 0;
    L.oB = o;
    o += round4((Q + 1) * PB * R * 2);
    L.oX = o;
    o += round4((Q + 1) * R * P);
    L.oC = o;
    o += round4(Q * PB * R * 2);
    L.oDy = o;
    o += round4(Q * R * P);
    L.oCS = o;
    o += round4(Q * PB * 2);
    L.oW = o;
    o += round4(Q * PB);
    L.oABG = o;
    o += Q * 4;
    L.oDx = o;
    o += Q * (L.threads / 32) * R * P;
    L.oScal = o;
    o += Q * PB * 4;
    L.oS = o;
    o += Q * 2 * L.threads * 4;
    int rb = round16((Q + 1) * PB * R * 2 * e);
    L.rX = rb;
    rb += round16((Q + 1) * R * P * e);
    L.rC = rb;
    rb += round16(Q * PB * R * 2 * e);
    L.rDy = rb;
    rb += round16(Q * R * P * e);
    L.rW = rb;
    rb += round16(Q * PB * 4);
    L.rDt = rb;
    rb += round16(Q * 4);
    L.rL = rb;
    rb += round16(Q * 4);
    L.rA = rb;
    rb += round16(Q * 4);
    if (gate) rb += round16(Q * R * P * e);   // the output gate's z rows, at rA + round16(4 Q)
    L.rawBytes = rb;
    L.unitXY = (R * P * e) % 16 == 0 ? 16 : 4;
    L.oRaw = o;
    o += 2 * (rb / 4);
    L.total = o;
    return L;
}

__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
// asynchronous global -> shared copies of 4, 8 or 16 bytes; ok == false writes zeros and reads nothing
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool ok) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src, bool ok) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 8 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int NPEND>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(NPEND) : "memory"); }

// Two-wide fp32 arithmetic (fma / mul / add .f32x2): one instruction for two lanes, each lane
// rounded exactly as the scalar instruction would round it.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
#define M3_BWD_OP2(name, op)                                                                                    \
    __device__ __forceinline__ float2 name(float2 a, float2 b) {                                               \
        float2 d;                                                                                              \
        asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n " op                  \
            " rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"                                                          \
            : "=f"(d.x), "=f"(d.y)                                                                             \
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                                         \
        return d;                                                                                              \
    }
M3_BWD_OP2(fmul2, "mul.rn.f32x2")
M3_BWD_OP2(fadd2, "add.rn.f32x2")
#undef M3_BWD_OP2

__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 join4(float2 l, float2 h) { return make_float4(l.x, l.y, h.x, h.y); }

__device__ __forceinline__ float4 fma4b(float a, float4 x, float4 y) {   // a x + y
    const float2 aa = make_float2(a, a);
    return join4(ffma2(aa, lo2(x), lo2(y)), ffma2(aa, hi2(x), hi2(y)));
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) { return join4(fadd2(lo2(a), lo2(b)), fadd2(hi2(a), hi2(b))); }
__device__ __forceinline__ float4 mul4(float a, float4 x) {
    const float2 aa = make_float2(a, a);
    return join4(fmul2(aa, lo2(x)), fmul2(aa, hi2(x)));
}
__device__ __forceinline__ float dot4(float4 a, float4 b) {
    const float2 p = ffma2(hi2(a), hi2(b), fmul2(lo2(a), lo2(b)));
    return p.x + p.y;
}
__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }

// Options of the pre-activation entry: EXT = 1, the per-token decay generators A_t; EXT = 3, A_t and the
// output gate's input z (io dtype, y's layout).  The plain entry (EXT = 0) takes an empty parameter, so
// that the plain kernels' parameter block and code are those of a kernel without the options.
template <int EXT>
struct BwdExt {};
template <>
struct BwdExt<1> {
    const float* __restrict__ a;
};
template <>
struct BwdExt<3> {
    const float* __restrict__ a;
    const void* __restrict__ z;
};

// P4T: P / 4 as a compile-time constant (with PB = kBwdThreads / P4T pairs per block and kBwdThreads
// threads), or 0 for shapes taken at run time; EXT: the options of BwdExt
template <typename IO, int R, int P4T, int EXT>
__global__ void __launch_bounds__(kBwdThreads, 4) scan_bwd_kernel(
    const IO* __restrict__ x, const IO* __restrict__ B, const IO* __restrict__ C, const float* __restrict__ dt,
    const float* __restrict__ A, const float* __restrict__ lam, const float* __restrict__ omega,
    const IO* __restrict__ dy, const float* __restrict__ dfin, float* __restrict__ dB, float* __restrict__ dC,
    float* __restrict__ domega, float* __restrict__ ckpt, float* __restrict__ part_dx, float* __restrict__ part_s,
    int64_t T, int H, int P, int N, const BwdLayout L, const BwdExt<EXT> ext) {
    constexpr int Q = BwdChunk<R>::Q;
    constexpr bool TOKA = (EXT & 1) != 0, GATE = (EXT & 2) != 0;
    extern __shared__ __align__(16) float sm[];
    // the pair blocks of one (batch, head) are neighbours in launch order, so they run together and
    // share their X, dy, Delta, lambda reads in L2
    const int64_t bh = blockIdx.x / L.nPB;
    const int pb = (int)(blockIdx.x % L.nPB);
    const int64_t b = bh / H;
    const int h = (int)(bh % H);
    const int P4 = P4T ? P4T : P >> 2, NP2 = N >> 1, PP = 4 * P4;   // PP = P
    const int PB = P4T ? kBwdThreads / P4T : L.PB, nt = P4T ? kBwdThreads : (int)blockDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int c4 = tid % P4, gl = tid / P4;
    const int j = pb * PB + gl;
    const bool on = gl < PB && j < NP2;
    const int gc = gl < PB ? gl : 0;   // shared-memory slot of this thread's pair (idle threads read slot 0)
    const int64_t nC = (T + Q - 1) / Q;
    const int64_t BTH = (int64_t)gridDim.x / L.nPB * T;   // batch * T * H

    float* sB = sm + L.oB;
    float* sX = sm + L.oX;
    float* sC = sm + L.oC;
    float* sDy = sm + L.oDy;
    float* sCS = sm + L.oCS;
    float* sW = sm + L.oW;
    float* sABG = sm + L.oABG;
    float* sDx = sm + L.oDx;
    float* sScal = sm + L.oScal;
    float4* sS4 = reinterpret_cast<float4*>(sm + L.oS);
    const float2* sB2 = reinterpret_cast<const float2*>(sB);
    const float4* sX4 = reinterpret_cast<const float4*>(sX);
    const float2* sC2 = reinterpret_cast<const float2*>(sC);
    const float4* sDy4 = reinterpret_cast<const float4*>(sDy);
    const float2* sCS2 = reinterpret_cast<const float2*>(sCS);
    const float4* sABG4 = reinterpret_cast<const float4*>(sABG);

    float a_h = 0.f;   // one decay generator per head, or A_t per token (staged with the chunk)
    if constexpr (!TOKA) a_h = A[h];
    auto tok = [&](int64_t t) { return (b * T + t) * H + h; };   // (batch, token, head) index

    // Copies of the inputs of tokens t0 - 1 .. t0 + Q - 1 into copy buffer `buf` (zeros outside [0, T)
    // and for pairs past N/2), asynchronous, as one commit group.
    const int lgPB = P4T ? Log2<kBwdThreads / (P4T ? P4T : 1)>::v : L.lgPB;
    const int lgRP = (P4T ? Log2<4 * P4T>::v : L.lgP) + kLg<R>::v;
    const int n1 = (Q + 1) * PB * R * 2, n2 = (Q + 1) * R * PP, n3 = Q * PB * R * 2, n4 = Q * R * PP;
    char* const raw = reinterpret_cast<char*>(sm + L.oRaw);
    constexpr int E = (int)sizeof(IO);
    const int unit = P4T ? ((R * 4 * P4T * E) % 16 == 0 ? 16 : 4) : L.unitXY;
    const int rZoff = L.rA + round16(Q * 4);   // the gate's z rows in a copy buffer
    const int upr = R * P4 * 4 * E / unit;   // copies per X / dy row (a power of two)
    int lgUpr = 0;
    while ((1 << lgUpr) < upr) ++lgUpr;
    // fwd: the forward sweep's copies only (no C, no dy)
    auto issue = [&](int64_t t0, int buf, bool fwd) {
        char* rb = raw + buf * L.rawBytes;
        const int npB = (Q + 1) * PB * R, npC = fwd ? 0 : Q * PB * R;   // (row pair, rank) copies of B, then C
        for (int i = tid; i < npB + npC; i += nt) {
            const bool isB = i < npB;
            const int k = isB ? i : i - npB;
            const int r = k & (R - 1), pl = (k >> kLg<R>::v) & (PB - 1), q = k >> (kLg<R>::v + lgPB);
            const int64_t t = isB ? t0 - 1 + q : t0 + q;
            const int jp = pb * PB + pl;
            const bool ok = t >= 0 && t < T && jp < NP2;
            const IO* src = (isB ? B : C) + (ok ? (tok(t) * R + r) * N + 2 * jp : 0);
            char* dst = rb + (isB ? 0 : L.rC) + k * 2 * E;
            if (E == 2)
                cp_async4(dst, src, ok);
            else
                cp_async8(dst, src, ok);
        }
        if constexpr (GATE) {   // X rows (from t0 - 1), then dy rows, then z rows
            const int nrows = fwd ? Q + 1 : 3 * Q + 1;
            for (int i = tid; i < nrows * upr; i += nt) {
                const int row = i >> lgUpr, u = i & (upr - 1);
                const int sec = row <= Q ? 0 : (row <= 2 * Q ? 1 : 2);
                const int q = sec == 0 ? row : (sec == 1 ? row - (Q + 1) : row - (2 * Q + 1));
                const int64_t t = sec == 0 ? t0 - 1 + q : t0 + q;
                const bool ok = t >= 0 && t < T;
                const void* base = sec == 0 ? (const void*)x : sec == 1 ? (const void*)dy : ext.z;
                const char* src = reinterpret_cast<const char*>(base) + (ok ? tok(t) * R * PP * E + u * unit : 0);
                char* dst = rb + (sec == 0 ? L.rX : sec == 1 ? L.rDy : rZoff) + q * R * PP * E + u * unit;
                if (unit == 16)
                    cp_async16(dst, src, ok);
                else
                    cp_async4(dst, src, ok);
            }
        } else {   // X rows (from t0 - 1), then dy rows
            for (int i = tid; i < (fwd ? Q + 1 : 2 * Q + 1) * upr; i += nt) {
                const int row = i >> lgUpr, u = i & (upr - 1);
                const bool isX = row <= Q;
                const int q = isX ? row : row - (Q + 1);
                const int64_t t = isX ? t0 - 1 + q : t0 + q;
                const bool ok = t >= 0 && t < T;
                const char* src =
                    reinterpret_cast<const char*>(isX ? x : dy) + (ok ? tok(t) * R * PP * E + u * unit : 0);
                char* dst = rb + (isX ? L.rX : L.rDy) + q * R * PP * E + u * unit;
                if (unit == 16)
                    cp_async16(dst, src, ok);
                else
                    cp_async4(dst, src, ok);
            }
        }
        constexpr int nscal = TOKA ? 3 * Q : 2 * Q;
        for (int i = tid; i < Q * PB + nscal; i += nt) {   // omega, then Delta, lambda (and A_t)
            const float* src;
            char* dst;
            bool ok;
            if (i < Q * PB) {
                const int q = i >> lgPB, jp = pb * PB + (i & (PB - 1));
                ok = t0 + q < T && jp < NP2;
                src = omega + (ok ? tok(t0 + q) * NP2 + jp : 0);
                dst = rb + L.rW + 4 * i;
            } else {
                const int k = i - Q * PB, sec = k / Q, q = k - sec * Q;
                ok = t0 + q < T;
                const float* base = sec == 0 ? dt : lam;
                if constexpr (TOKA) base = sec == 2 ? ext.a : base;
                src = base + (ok ? tok(t0 + q) : 0);
                dst = rb + (sec == 0 ? L.rDt : sec == 1 ? L.rL : L.rA) + 4 * q;
            }
            cp_async4(dst, src, ok);
        }
        cp_async_commit();
    };
    // The copied inputs of buffer `buf` in fp32 working form, with the angles and decays they give.
    auto convert = [&](int buf, bool fwd) {
        const char* rb = raw + buf * L.rawBytes;
        const IO* rB = reinterpret_cast<const IO*>(rb);
        const IO* rX = reinterpret_cast<const IO*>(rb + L.rX);
        const IO* rC = reinterpret_cast<const IO*>(rb + L.rC);
        const IO* rDy = reinterpret_cast<const IO*>(rb + L.rDy);
        const float* rW = reinterpret_cast<const float*>(rb + L.rW);
        const float* rDt = reinterpret_cast<const float*>(rb + L.rDt);
        const float* rL = reinterpret_cast<const float*>(rb + L.rL);
        const float* rA = reinterpret_cast<const float*>(rb + L.rA);
        for (int i = tid; i < n1; i += nt) sB[i] = ld_io(rB, i);
        for (int i = tid; i < n2; i += nt) sX[i] = ld_io(rX, i);
        if (!fwd) {
            for (int i = tid; i < n3; i += nt) sC[i] = ld_io(rC, i);
            if constexpr (GATE) {   // the gated output's seed reaches the recurrence as dy silu(z)
                const IO* rZ = reinterpret_cast<const IO*>(rb + rZoff);
                for (int i = tid; i < n4; i += nt) sDy[i] = ld_io(rDy, i) * silu_f(ld_io(rZ, i));
            } else {
                for (int i = tid; i < n4; i += nt) sDy[i] = ld_io(rDy, i);
            }
        }
        for (int i = tid; i < Q * PB; i += nt) {
            const float w = rW[i];
            float sn, cs;
            sincosf(rDt[i >> lgPB] * w, &sn, &cs);
            sW[i] = w;
            sCS[2 * i] = cs;
            sCS[2 * i + 1] = sn;
        }
        for (int q = tid; q < Q; q += nt) {
            const float d = rDt[q], l = rL[q];
            float a = a_h;
            if constexpr (TOKA) a = rA[q];
            const float al = expf(d * a);
            sABG[4 * q] = al;
            sABG[4 * q + 1] = (1.f - l) * d * al;
            sABG[4 * q + 2] = l * d;
            sABG[4 * q + 3] = d;
        }
    };
    // v[rows 2j, 2j+1][cols of c4] of slot s of the B/X buffers: sum_r B[r, 2j / 2j+1] X[r, cols]
    auto outer = [&](int s, float4& v0, float4& v1) {
        v0 = zero4();
        v1 = v0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float2 bb = sB2[(s * PB + gc) * R + r];
            const float4 xx = sX4[(s * R + r) * P4 + c4];
            v0 = fma4b(bb.x, xx, v0);
            v1 = fma4b(bb.y, xx, v1);
        }
    };
    // one step of the recurrence for token slot q of the staged chunk; (vp0, vp1) = v of slot q on entry,
    // of slot q + 1 on return
    auto step = [&](int q, float4& s0, float4& s1, float4& vp0, float4& vp1) {
        float4 v0, v1;
        outer(q + 1, v0, v1);
        const float4 abg = sABG4[q];
        const float4 u0 = fma4b(abg.x, s0, mul4(abg.y, vp0));
        const float4 u1 = fma4b(abg.x, s1, mul4(abg.y, vp1));
        const float2 cs = sCS2[q * PB + gc];
        // R(phi) u: rows (c u0 - s u1, s u0 + c u1), then + gamma v
        s0 = fma4b(abg.z, v0, fma4b(-cs.y, u1, mul4(cs.x, u0)));
        s1 = fma4b(abg.z, v1, fma4b(cs.y, u0, mul4(cs.x, u1)));
        vp0 = v0;
        vp1 = v1;
    };
    float4* ck4 = reinterpret_cast<float4*>(ckpt) + bh * nC * (int64_t)N * P4;
    auto ckrow = [&](int64_t c, int n) { return ck4 + (c * N + n) * P4 + c4; };

    // ---------------- forward sweep: the state entering chunks 1 .. nC-1 ----------------
    {
        float4 h0 = zero4(), h1 = zero4();
        int buf = 0;
        if (nC > 1) issue(0, 0, true);
        for (int64_t c = 0; c + 1 < nC; ++c) {
            if (c + 2 < nC)
                issue((c + 1) * Q, buf ^ 1, true);   // the next chunk's copies overlap this chunk's work
            else
                cp_async_commit();
            cp_async_wait<1>();
            __syncthreads();   // every thread's copies of this chunk have landed
            convert(buf, true);
            __syncthreads();
            buf ^= 1;
            float4 vp0, vp1;
            outer(0, vp0, vp1);
#pragma unroll
            for (int q = 0; q < Q; ++q) step(q, h0, h1, vp0, vp1);
            if (on) {
                *ckrow(c + 1, 2 * j) = h0;
                *ckrow(c + 1, 2 * j + 1) = h1;
            }
            __syncthreads();   // the working inputs are replaced next
        }
        cp_async_wait<0>();
    }

    // ---------------- reverse sweep: the adjoint, chunk by chunk ----------------
    float4 ub0 = zero4(), ub1 = zero4();   // ubar_{t+1}
    float alpha_n = 0.f, beta_n = 0.f;     // alpha_{t+1}, beta_{t+1}
    int buf = 0;
    issue((nC - 1) * Q, 0, false);
    for (int64_t c = nC - 1; c >= 0; --c) {
        const int64_t t0 = c * Q;
        const int qn = (int)((T - t0) < Q ? (T - t0) : Q);
        if (c > 0)
            issue((c - 1) * Q, buf ^ 1, false);
        else
            cp_async_commit();
        float4 hc0 = zero4(), hc1 = zero4();   // h_{t0-1}
        if (c > 0 && on) {
            hc0 = *ckrow(c, 2 * j);
            hc1 = *ckrow(c, 2 * j + 1);
        }
        cp_async_wait<1>();
        __syncthreads();
        convert(buf, false);
        __syncthreads();
        buf ^= 1;
        {
            float4 s0 = hc0, s1 = hc1, vp0, vp1;
            outer(0, vp0, vp1);
            for (int q = 0; q < qn; ++q) {   // each thread reads back only its own slots
                step(q, s0, s1, vp0, vp1);
                sS4[(2 * q) * nt + tid] = s0;
                sS4[(2 * q + 1) * nt + tid] = s1;
            }
        }
        // this chunk's outputs of pair j: token t0 + q at q H R N (dC, dB) and q H N/2 (domega)
        float* const dCc = dC + tok(t0) * R * N + 2 * j;
        float* const dBc = dB + tok(t0) * R * N + 2 * j;
        float* const domc = domega + tok(t0) * NP2 + j;
        float4 v0, v1;   // v of token t0 + q, carried down from the step after
        outer(qn, v0, v1);
#pragma unroll 2
        for (int q = qn - 1; q >= 0; --q) {
            const int64_t t = t0 + q;
            const float4 ht0 = sS4[(2 * q) * nt + tid], ht1 = sS4[(2 * q + 1) * nt + tid];
            const float4 hp0 = q > 0 ? sS4[(2 * q - 2) * nt + tid] : hc0;
            const float4 hp1 = q > 0 ? sS4[(2 * q - 1) * nt + tid] : hc1;
            float4 vp0, vp1;
            outer(q, vp0, vp1);
            const float4 abg = sABG4[q];
            const float gamma = abg.z, d = abg.w;
            // gbar_t = C_t dy_t^T + alpha_{t+1} ubar_{t+1} (+ the final-state seed)
            float4 g0 = mul4(alpha_n, ub0), g1 = mul4(alpha_n, ub1);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 cc = sC2[(q * PB + gc) * R + r];
                const float4 dyr = sDy4[(q * R + r) * P4 + c4];
                g0 = fma4b(cc.x, dyr, g0);
                g1 = fma4b(cc.y, dyr, g1);
            }
            if (t == T - 1 && dfin != nullptr && on) {
                const float4* df4 = reinterpret_cast<const float4*>(dfin + bh * (int64_t)N * PP);
                g0 = add4(g0, df4[(2 * j) * P4 + c4]);
                g1 = add4(g1, df4[(2 * j + 1) * P4 + c4]);
            }
            if (!on) g0 = g1 = zero4();
            const float4 dv0 = fma4b(gamma, g0, mul4(beta_n, ub0));
            const float4 dv1 = fma4b(gamma, g1, mul4(beta_n, ub1));
            const float4 r0 = fma4b(-gamma, v0, ht0), r1 = fma4b(-gamma, v1, ht1);   // R(phi_t) u_t
            const float2 cs = sCS2[q * PB + gc];
            // ubar_t = R(phi_t)^T gbar_t
            const float4 un0 = fma4b(cs.y, g1, mul4(cs.x, g0));
            const float4 un1 = fma4b(-cs.y, g0, mul4(cs.x, g1));
            // sums over this pair's columns: dphi, dalpha, dbeta, dgamma, then dC_t and dB_t per rank
            float red[4 + 4 * R];
            red[0] = dot4(g1, r0) - dot4(g0, r1);
            red[1] = dot4(un0, hp0) + dot4(un1, hp1);
            red[2] = dot4(un0, vp0) + dot4(un1, vp1);
            red[3] = dot4(g0, v0) + dot4(g1, v1);
            float4 dXp[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float4 dyr = sDy4[(q * R + r) * P4 + c4];
                const float4 xr = sX4[((q + 1) * R + r) * P4 + c4];
                red[4 + 4 * r] = dot4(ht0, dyr);   // dC_t[r, n] = sum_p h_t[n, p] dy_t[r, p]
                red[5 + 4 * r] = dot4(ht1, dyr);
                red[6 + 4 * r] = dot4(dv0, xr);    // dB_t[r, n] = sum_p dv_t[n, p] X_t[r, p]
                red[7 + 4 * r] = dot4(dv1, xr);
                const float2 bb = sB2[((q + 1) * PB + gc) * R + r];
                dXp[r] = fma4b(bb.x, dv0, mul4(bb.y, dv1));   // dX_t[r, p] partial over this pair
            }
            ub0 = un0;
            ub1 = un1;
            alpha_n = abg.x;
            beta_n = abg.y;
            for (int o = 1; o < P4; o <<= 1) {
#pragma unroll
                for (int i = 0; i < 4 + 4 * R; ++i) red[i] += __shfl_xor_sync(0xffffffffu, red[i], o);
            }
            if (on && c4 == 0) {
                const int oq = q * H * R * N;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    *reinterpret_cast<float2*>(dCc + oq + r * N) = make_float2(red[4 + 4 * r], red[5 + 4 * r]);
                    *reinterpret_cast<float2*>(dBc + oq + r * N) = make_float2(red[6 + 4 * r], red[7 + 4 * r]);
                }
                domc[q * H * NP2] = d * red[0];
                float* sc = sScal + (q * PB + gl) * 4;
                sc[0] = red[1];
                sc[1] = red[2];
                sc[2] = red[3];
                sc[3] = sW[q * PB + gl] * red[0];
            }
            // dX over the pairs of this warp; the warps' partials are summed at the end of the chunk
            for (int o = P4; o < 32; o <<= 1) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    dXp[r].x += __shfl_xor_sync(0xffffffffu, dXp[r].x, o);
                    dXp[r].y += __shfl_xor_sync(0xffffffffu, dXp[r].y, o);
                    dXp[r].z += __shfl_xor_sync(0xffffffffu, dXp[r].z, o);
                    dXp[r].w += __shfl_xor_sync(0xffffffffu, dXp[r].w, o);
                }
            }
            if (lane < P4) {
                float4* dst = reinterpret_cast<float4*>(sDx) + ((q * nw + warp) * R) * P4 + c4;
#pragma unroll
                for (int r = 0; r < R; ++r) dst[r * P4] = dXp[r];
            }
            v0 = vp0;
            v1 = vp1;
        }
        __syncthreads();
        // this pair block's partial sums of the chunk's tokens
        float* pdx = part_dx + ((int64_t)pb * BTH + tok(t0)) * R * PP;   // token t0 + q at q H R P
        for (int i = tid; i < qn * R * PP; i += nt) {
            const int q = i >> lgRP, rp = i & (R * PP - 1);
            float sx = 0.f;
            for (int w = 0; w < nw; ++w) sx += sDx[(q * nw + w) * R * PP + rp];
            pdx[q * H * R * PP + rp] = sx;
        }
        const int pbn = (NP2 - pb * PB) < PB ? (NP2 - pb * PB) : PB;   // pairs of this block
        for (int i = tid; i < qn * 4; i += nt) {
            const int q = i >> 2, k = i & 3;
            float s = 0.f;
            for (int pl = 0; pl < pbn; ++pl) s += sScal[(q * PB + pl) * 4 + k];
            part_s[((int64_t)pb * BTH + tok(t0) + q * H) * 4 + k] = s;
        }
        // the next chunk's convert() writes none of sDx, sScal, sS; the barriers before it order the reads above
    }
}

// dX = the sum of the pair blocks' partials
__global__ void bwd_finish_dx(const float4* __restrict__ part, float4* __restrict__ dx, int64_t n4, int nPB) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 s = part[i];
        for (int k = 1; k < nPB; ++k) s = add4(s, part[k * n4 + i]);
        dx[i] = s;
    }
}

// per token: (dalpha, dbeta, dgamma, sum_j omega_j dphi_j) summed over the pair blocks, then the chain
// rule through alpha = exp(Delta A), beta = (1 - lambda) Delta alpha, gamma = lambda Delta, phi = Delta omega
__global__ void bwd_finish_scalars(const float4* __restrict__ part_s, const float* __restrict__ dt,
                                   const float* __restrict__ lam, const float* __restrict__ A,
                                   float* __restrict__ ddt, float* __restrict__ dlam, float* __restrict__ dA,
                                   int64_t batch, int64_t T, int H, int nPB) {
    __shared__ float red[32];
    const int h = blockIdx.x;
    const float a = A[h];
    const int64_t BTH = batch * T * H;
    float acc = 0.f;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        for (int64_t t = threadIdx.x; t < T; t += blockDim.x) {
            const int64_t tk = (b * T + t) * H + h;
            float4 s = part_s[tk];
            for (int k = 1; k < nPB; ++k) s = add4(s, part_s[k * BTH + tk]);
            const float d = dt[tk], l = lam[tk], al = expf(d * a);
            const float dalpha = s.x + s.y * (1.f - l) * d;   // through alpha and through beta's alpha
            ddt[tk] = dalpha * a * al + s.y * (1.f - l) * al + s.z * l + s.w;
            dlam[tk] = -d * al * s.y + d * s.z;
            acc += dalpha * d * al;
        }
    }
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
        atomicAdd(&dA[h], s);
    }
}

// The same on pre-activations: Delta = softplus(z), z = dt_raw + dt_bias[h], lambda = sigmoid(u), and A_t
// per token; then dz = dDelta sigmoid(z) (softplus' = sigmoid) gives ddt_raw and, summed over batch and
// tokens, ddt_bias; du = dlambda lambda (1 - lambda); dA_t per token.
__global__ void bwd_finish_scalars_prep(const float4* __restrict__ part_s, const float* __restrict__ dt_eff,
                                        const float* __restrict__ lam_eff, const float* __restrict__ A_tok,
                                        const float* __restrict__ dt_raw, const float* __restrict__ dt_bias,
                                        float* __restrict__ ddt_raw, float* __restrict__ du, float* __restrict__ dA_tok,
                                        float* __restrict__ ddt_bias, int64_t batch, int64_t T, int H, int nPB) {
    __shared__ float red[32];
    const int h = blockIdx.x;
    const float bias = dt_bias != nullptr ? dt_bias[h] : 0.f;
    const int64_t BTH = batch * T * H;
    float acc = 0.f;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        for (int64_t t = threadIdx.x; t < T; t += blockDim.x) {
            const int64_t tk = (b * T + t) * H + h;
            float4 s = part_s[tk];
            for (int k = 1; k < nPB; ++k) s = add4(s, part_s[k * BTH + tk]);
            const float d = dt_eff[tk], l = lam_eff[tk], a = A_tok[tk], al = expf(d * a);
            const float dalpha = s.x + s.y * (1.f - l) * d;
            const float ddelta = dalpha * a * al + s.y * (1.f - l) * al + s.z * l + s.w;
            const float dl = -d * al * s.y + d * s.z;
            const float dz = ddelta * sigmoid_f(dt_raw[tk] + bias);
            ddt_raw[tk] = dz;
            du[tk] = dl * l * (1.f - l);
            dA_tok[tk] = dalpha * d * al;
            acc += dz;
        }
    }
    if (ddt_bias == nullptr) return;
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
        atomicAdd(&ddt_bias[h], s);
    }
}

// dz = dy y_pre silu'(z), silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z))), for the gated output
// y = y_pre silu(z); y_pre is the ungated forward output
template <typename IO>
__global__ void bwd_gate_dz(const IO* __restrict__ dy, const IO* __restrict__ z, const IO* __restrict__ y_pre,
                            float* __restrict__ dz, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float zz = ld_io(z, i), sg = sigmoid_f(zz);
        dz[i] = ld_io(dy, i) * ld_io(y_pre, i) * sg * (1.f + zz * (1.f - sg));
    }
}

// B / C normalisation of every (token, rank) row ("Mamba-3", section 3.4): Vn = V r gain + bias with
// r = rsqrt(mean(V^2) + eps) (the forward entry's formula; r = 1 and no gain without the norm), r kept for
// the rows' backward.  One warp per row; rows are (batch, token, head, rank) major, HR = H * R.  The rows
// are written in OT (fp32 where the adjoint runs on fp32 copies of bf16 inputs).
template <typename IO, typename OT>
__global__ void __launch_bounds__(256) bc_rows_forward(const IO* __restrict__ V, const float* __restrict__ gain,
                                                       const float* __restrict__ bias, int norm, float eps,
                                                       OT* __restrict__ Vn, float* __restrict__ rinv, int64_t rows,
                                                       int HR, int N) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; row < rows; row += nwarps) {
        float ss = 0.f;
        for (int n = lane; n < N; n += 32) {
            const float a = ld_io(V, row * N + n);
            ss = fmaf(a, a, ss);
        }
        ss = warp_sum(ss);
        const float r = norm ? rsqrtf(ss / N + eps) : 1.f;
        const float* bb = bias != nullptr ? bias + (row % HR) * N : nullptr;
        for (int n = lane; n < N; n += 32) {
            float a = ld_io(V, row * N + n);
            if (norm) {
                a *= r;
                if (gain != nullptr) a *= gain[n];
            }
            if (bb != nullptr) a += bb[n];
            st_io(Vn, row * N + n, a);
        }
        if (lane == 0) rinv[row] = r;
    }
}

// The rows' backward: dV holds dL/dVn on entry and dL/dV on return,
//   dV = r (gain dVn) - V r^3 / N sum_n(gain dVn V)   (with the norm; dV = dVn without it);
// dgain [N] += sum over every row of dVn V r, dbias [H, R, N] += sum over (batch, token) of dVn.
// Block (h*R + rank, token block): 8 warps, one row at a time each; per-lane partial sums, then shared-memory
// and one global atomic add per channel and block.
template <typename IO>
__global__ void __launch_bounds__(256) bc_rows_backward(const IO* __restrict__ V, const float* __restrict__ gain,
                                                        const float* __restrict__ rinv, int norm,
                                                        float* __restrict__ dV, float* __restrict__ dgain,
                                                        float* __restrict__ dbias, int64_t BT, int HR, int N) {
    __shared__ float sg[256], sb[256];
    const int hr = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int n = threadIdx.x; n < N; n += blockDim.x) sg[n] = sb[n] = 0.f;
    __syncthreads();
    float ag[8], ab[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) ag[k] = ab[k] = 0.f;
    for (int64_t bt = (int64_t)blockIdx.y * 8 + warp; bt < BT; bt += (int64_t)gridDim.y * 8) {
        const int64_t row = bt * HR + hr;
        const float r = rinv[row];
        float gd[8], vv[8], s = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int n = lane + 32 * k;
            gd[k] = vv[k] = 0.f;
            if (n < N) {
                const float dn = dV[row * N + n], v = ld_io(V, row * N + n);
                gd[k] = (norm && gain != nullptr ? gain[n] : 1.f) * dn;   // the gain acts only with the norm
                vv[k] = v;
                s = fmaf(gd[k], v, s);
                ab[k] += dn;
                ag[k] = fmaf(dn * v, r, ag[k]);
            }
        }
        s = warp_sum(s);
        const float c = r * r * r * s / N;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int n = lane + 32 * k;
            if (n < N) dV[row * N + n] = norm ? fmaf(r, gd[k], -vv[k] * c) : gd[k];
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int n = lane + 32 * k;
        if (n < N) {
            atomicAdd(&sg[n], ag[k]);
            atomicAdd(&sb[n], ab[k]);
        }
    }
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        if (dgain != nullptr && norm) atomicAdd(&dgain[n], sg[n]);
        if (dbias != nullptr) atomicAdd(&dbias[hr * N + n], sb[n]);
    }
}

// fp32 copies for the adjoint of the promoted path: dst = src, and the seed dst = dy silu(z) (z null: dy)
template <typename IO>
__global__ void to_f32(const IO* __restrict__ src, float* __restrict__ dst, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = ld_io(src, i);
}
template <typename IO>
__global__ void gate_seed_f32(const IO* __restrict__ dy, const IO* __restrict__ z, float* __restrict__ dst,
                              int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = z != nullptr ? ld_io(dy, i) * silu_f(ld_io(z, i)) : ld_io(dy, i);
}

// B / C normalisation arguments of m3_scan_bwd_prep (on == false: none)
struct BwdBc {
    bool on;
    int norm;
    float eps;
    const float *B_gain, *C_gain, *B_bias, *C_bias;
    float *dB_gain, *dC_gain, *dB_bias, *dC_bias;
};

// pre-activation inputs of m3_scan_bwd_prep (on == false: the plain entry); z != nullptr: the output gate
struct BwdPrep {
    bool on;
    const float *dt_raw, *dt_bias, *u, *A_tok;
    float* ddt_bias;
    const void *z, *y_pre;
    float* dz;
    BwdBc bc;
};

int bwd_chunk(int R) { return R <= 2 ? 8 : 4; }

struct BwdWs {
    size_t ckpt, part_dx, part_s, dt_eff, lam_eff, bn, cn, rb, rc, total;   // byte offsets; the whole size
};

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

BwdWs bwd_ws(const ScanDims& d) {
    const int Q = bwd_chunk(d.R);
    const BwdLayout L = bwd_layout((int)d.headdim, (int)d.dstate, d.R, Q, d.io == M3_DTYPE_BF16 ? 2 : 4);
    const size_t bh = (size_t)(d.batch * d.nheads), BTH = bh * (size_t)d.seqlen;
    const size_t nC = (size_t)((d.seqlen + Q - 1) / Q);
    BwdWs w{};
    w.ckpt = 0;
    w.part_dx = round256(sizeof(float) * bh * nC * (size_t)(d.dstate * d.headdim));
    w.part_s = w.part_dx + round256(sizeof(float) * (size_t)L.nPB * BTH * (size_t)(d.R * d.headdim));
    w.dt_eff = w.part_s + round256(sizeof(float) * (size_t)L.nPB * BTH * 4);
    w.lam_eff = w.dt_eff + round256(sizeof(float) * BTH);   // Delta and lambda of the pre-activation entry
    w.total = w.dt_eff;
    return w;
}

// the pre-activation entry's sections: Delta, lambda, then the normalised B and C rows (io dtype) and
// their inverse RMS (fp32) for the B / C normalisation
BwdWs bwd_ws_prep(const ScanDims& d) {
    BwdWs w = bwd_ws(d);
    const size_t bth = (size_t)(d.batch * d.nheads) * (size_t)d.seqlen, rows = bth * (size_t)d.R;
    const size_t e = d.io == M3_DTYPE_BF16 ? 2 : 4;
    w.bn = w.lam_eff + round256(sizeof(float) * bth);
    w.cn = w.bn + round256(e * rows * (size_t)d.dstate);
    w.rb = w.cn + round256(e * rows * (size_t)d.dstate);
    w.rc = w.rb + round256(sizeof(float) * rows);
    w.total = w.rc + round256(sizeof(float) * rows);
    return w;
}

// The promoted path of the B / C normalisation's backward (bf16 io, or together with the output gate):
// the adjoint's fp32 run uses the fp32 layout up to its Delta / lambda sections (inner), then come the
// normalised B and C rows in fp32 and their inverse RMS, fp32 copies of x and of the seed dy silu(z).
struct BwdWsUp {
    size_t inner, bn, cn, rb, rc, xf, dyf, total;
};

BwdWsUp bwd_ws_promoted(const ScanDims& d) {
    ScanDims f = d;
    f.io = M3_DTYPE_F32;
    const BwdWs wi = bwd_ws_prep(f);
    const size_t rows = (size_t)(d.batch * d.nheads) * (size_t)d.seqlen * (size_t)d.R;
    BwdWsUp w{};
    w.inner = wi.bn;
    w.bn = wi.bn;
    w.cn = w.bn + round256(sizeof(float) * rows * (size_t)d.dstate);
    w.rb = w.cn + round256(sizeof(float) * rows * (size_t)d.dstate);
    w.rc = w.rb + round256(sizeof(float) * rows);
    w.xf = w.rc + round256(sizeof(float) * rows);
    w.dyf = w.xf + round256(sizeof(float) * rows * (size_t)d.headdim);
    w.total = w.dyf + round256(sizeof(float) * rows * (size_t)d.headdim);
    return w;
}

size_t bwd_ws_prep_total(const ScanDims& d) {
    const size_t a = bwd_ws_prep(d).total, b = bwd_ws_promoted(d).total;
    return a > b ? a : b;
}

template <typename IO>
cudaError_t launch_bwd_io(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                          const float* A, const float* lambda, const float* omega, const void* dy,
                          const float* d_final, float* dx, float* dB, float* dC, float* ddt, float* dA,
                          float* dlambda, float* domega, void* workspace, cudaStream_t stream, const BwdPrep& pp);

// The B / C normalisation's backward for bf16 io or with the output gate: the adjoint runs in its fp32
// instantiation on fp32 copies -- x, the seed dy silu(z), and the normalised rows written in fp32 -- so
// that nothing the recurrence sees is rounded to bf16 beyond the inputs themselves; then the gate's dz
// from the ungated output and the rows' backward on the raw rows, as in the direct path.
template <typename IO>
cudaError_t launch_bwd_promoted(const ScanDims& d, const void* x, const void* B, const void* C, const float* omega,
                                const void* dy, const float* d_final, float* dx, float* dB, float* dC, float* ddt,
                                float* dA, float* dlambda, float* domega, void* workspace, cudaStream_t stream,
                                const BwdPrep& pp) {
    cudaError_t e = cudaSuccess;
    float* zs[] = {pp.bc.dB_gain, pp.bc.dC_gain};
    for (float* q : zs)
        if (q != nullptr && e == cudaSuccess) e = cudaMemsetAsync(q, 0, sizeof(float) * (size_t)d.dstate, stream);
    float* zb[] = {pp.bc.dB_bias, pp.bc.dC_bias};
    for (float* q : zb)
        if (q != nullptr && e == cudaSuccess)
            e = cudaMemsetAsync(q, 0, sizeof(float) * (size_t)(d.nheads * d.R * d.dstate), stream);
    if (e != cudaSuccess) return e;
    const BwdWsUp w = bwd_ws_promoted(d);
    char* ws = static_cast<char*>(workspace);
    const int64_t bh = d.batch * d.nheads, rows = bh * d.seqlen * d.R, nx = rows * d.headdim;
    const int HR = (int)(d.nheads * d.R);
    float* Bn = reinterpret_cast<float*>(ws + w.bn);
    float* Cn = reinterpret_cast<float*>(ws + w.cn);
    float* rb = reinterpret_cast<float*>(ws + w.rb);
    float* rc = reinterpret_cast<float*>(ws + w.rc);
    float* xf = reinterpret_cast<float*>(ws + w.xf);
    float* dyf = reinterpret_cast<float*>(ws + w.dyf);
    if (bh > 0 && d.seqlen > 0) {
        const unsigned rbk = (unsigned)((rows + 7) / 8 < 148 * 16 ? (rows + 7) / 8 : 148 * 16);
        bc_rows_forward<IO, float><<<rbk, 256, 0, stream>>>((const IO*)B, pp.bc.B_gain, pp.bc.B_bias, pp.bc.norm,
                                                            pp.bc.eps, Bn, rb, rows, HR, (int)d.dstate);
        bc_rows_forward<IO, float><<<rbk, 256, 0, stream>>>((const IO*)C, pp.bc.C_gain, pp.bc.C_bias, pp.bc.norm,
                                                            pp.bc.eps, Cn, rc, rows, HR, (int)d.dstate);
        const unsigned eb = (unsigned)((nx + 255) / 256 < 148 * 16 ? (nx + 255) / 256 : 148 * 16);
        to_f32<IO><<<eb, 256, 0, stream>>>((const IO*)x, xf, nx);
        gate_seed_f32<IO><<<eb, 256, 0, stream>>>((const IO*)dy, (const IO*)pp.z, dyf, nx);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    ScanDims f = d;
    f.io = M3_DTYPE_F32;
    BwdPrep p2 = pp;
    p2.z = nullptr;
    p2.y_pre = nullptr;
    p2.dz = nullptr;
    p2.bc.on = false;
    e = launch_bwd_io<float>(f, xf, Bn, Cn, nullptr, nullptr, nullptr, omega, dyf, d_final, dx, dB, dC, ddt, dA,
                             dlambda, domega, workspace, stream, p2);
    if (e != cudaSuccess || bh == 0 || d.seqlen == 0) return e;
    if (pp.z != nullptr) {
        const unsigned gb = (unsigned)((nx + 255) / 256 < 148 * 16 ? (nx + 255) / 256 : 148 * 16);
        bwd_gate_dz<IO><<<gb, 256, 0, stream>>>((const IO*)dy, (const IO*)pp.z, (const IO*)pp.y_pre, pp.dz, nx);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int64_t BT = d.batch * d.seqlen;
    const dim3 g2((unsigned)HR, (unsigned)((BT + 7) / 8 < 1024 ? (BT + 7) / 8 : 1024));
    bc_rows_backward<IO><<<g2, 256, 0, stream>>>((const IO*)B, pp.bc.B_gain, rb, pp.bc.norm, dB, pp.bc.dB_gain,
                                                 pp.bc.dB_bias, BT, HR, (int)d.dstate);
    bc_rows_backward<IO><<<g2, 256, 0, stream>>>((const IO*)C, pp.bc.C_gain, rc, pp.bc.norm, dC, pp.bc.dC_gain,
                                                 pp.bc.dC_bias, BT, HR, (int)d.dstate);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_bwd_io(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                          const float* A, const float* lambda, const float* omega, const void* dy,
                          const float* d_final, float* dx, float* dB, float* dC, float* ddt, float* dA,
                          float* dlambda, float* domega, void* workspace, cudaStream_t stream, const BwdPrep& pp) {
    if (pp.on && pp.bc.on && (sizeof(IO) == 2 || pp.z != nullptr))
        return launch_bwd_promoted<IO>(d, x, B, C, omega, dy, d_final, dx, dB, dC, ddt, dA, dlambda, domega,
                                       workspace, stream, pp);
    const int Q = bwd_chunk(d.R);
    const bool gate = pp.on && pp.z != nullptr;
    const BwdLayout L = bwd_layout((int)d.headdim, (int)d.dstate, d.R, Q, (int)sizeof(IO), gate);
    const int64_t bh = d.batch * d.nheads;
    cudaError_t e = cudaSuccess;
    if (!pp.on)
        e = cudaMemsetAsync(dA, 0, sizeof(float) * (size_t)d.nheads, stream);
    else if (pp.ddt_bias != nullptr)
        e = cudaMemsetAsync(pp.ddt_bias, 0, sizeof(float) * (size_t)d.nheads, stream);
    if (e == cudaSuccess && pp.bc.on) {
        float* zs[] = {pp.bc.dB_gain, pp.bc.dC_gain};
        for (float* q : zs)
            if (q != nullptr && e == cudaSuccess) e = cudaMemsetAsync(q, 0, sizeof(float) * (size_t)d.dstate, stream);
        float* zb[] = {pp.bc.dB_bias, pp.bc.dC_bias};
        for (float* q : zb)
            if (q != nullptr && e == cudaSuccess)
                e = cudaMemsetAsync(q, 0, sizeof(float) * (size_t)(d.nheads * d.R * d.dstate), stream);
    }
    if (e != cudaSuccess || bh == 0 || d.seqlen == 0) return e;
    const BwdWs w = pp.on ? bwd_ws_prep(d) : bwd_ws(d);
    char* ws = static_cast<char*>(workspace);
    const void *B_raw = B, *C_raw = C;
    const int64_t rows = bh * d.seqlen * d.R;
    const int HR = (int)(d.nheads * d.R);
    if (pp.bc.on) {   // the normalised rows the recurrence sees
        void* Bn = ws + w.bn;
        void* Cn = ws + w.cn;
        const unsigned rbk = (unsigned)((rows + 7) / 8 < 148 * 16 ? (rows + 7) / 8 : 148 * 16);
        bc_rows_forward<IO, IO><<<rbk, 256, 0, stream>>>((const IO*)B, pp.bc.B_gain, pp.bc.B_bias, pp.bc.norm,
                                                         pp.bc.eps, (IO*)Bn, reinterpret_cast<float*>(ws + w.rb),
                                                         rows, HR, (int)d.dstate);
        bc_rows_forward<IO, IO><<<rbk, 256, 0, stream>>>((const IO*)C, pp.bc.C_gain, pp.bc.C_bias, pp.bc.norm,
                                                         pp.bc.eps, (IO*)Cn, reinterpret_cast<float*>(ws + w.rc),
                                                         rows, HR, (int)d.dstate);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        B = Bn;
        C = Cn;
    }
    if (pp.on) {   // Delta and lambda from their pre-activations, as the forward entry derives them
        float* dt_eff = reinterpret_cast<float*>(ws + w.dt_eff);
        float* lam_eff = reinterpret_cast<float*>(ws + w.lam_eff);
        if ((e = launch_prep_params(pp.dt_raw, pp.dt_bias, pp.u, dt_eff, lam_eff, bh * d.seqlen, (int)d.nheads,
                                    stream)) != cudaSuccess)
            return e;
        dt = dt_eff;
        lambda = lam_eff;
    }
    float* ckpt = reinterpret_cast<float*>(ws + w.ckpt);
    float* part_dx = reinterpret_cast<float*>(ws + w.part_dx);
    float* part_s = reinterpret_cast<float*>(ws + w.part_s);
    const size_t smem = sizeof(float) * (size_t)L.total;
    const unsigned grid = (unsigned)(bh * L.nPB);   // (batch*head, pair block), pair block fastest
    const bool p64 = d.headdim == 64 && L.PB == kBwdThreads / 16;   // the compile-time P = 64 kernels
#define M3_BWD_LAUNCH(RR, P4C, EX, EXTV)                                                                        \
    {                                                                                                             \
        auto k = scan_bwd_kernel<IO, RR, P4C, EX>;                                                                \
        if (smem > 48 * 1024 &&                                                                                   \
            (e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) \
            return e;                                                                                             \
        k<<<grid, L.threads, smem, stream>>>((const IO*)x, (const IO*)B, (const IO*)C, dt, A, lambda, omega,      \
                                             (const IO*)dy, d_final, dB, dC, domega, ckpt, part_dx, part_s,       \
                                             d.seqlen, (int)d.nheads, (int)d.headdim, (int)d.dstate, L, EXTV);    \
    }
#define M3_BWD_CASE(RR)                                                                                           \
    case RR:                                                                                                      \
        if (gate) {                                                                                               \
            const BwdExt<3> ex{pp.A_tok, pp.z};                                                                   \
            if (p64)                                                                                              \
                M3_BWD_LAUNCH(RR, 16, 3, ex)                                                                      \
            else                                                                                                  \
                M3_BWD_LAUNCH(RR, 0, 3, ex)                                                                       \
        } else if (pp.on) {                                                                                       \
            const BwdExt<1> ex{pp.A_tok};                                                                         \
            if (p64)                                                                                              \
                M3_BWD_LAUNCH(RR, 16, 1, ex)                                                                      \
            else                                                                                                  \
                M3_BWD_LAUNCH(RR, 0, 1, ex)                                                                       \
        } else {                                                                                                  \
            const BwdExt<0> ex{};                                                                                 \
            if (p64)                                                                                              \
                M3_BWD_LAUNCH(RR, 16, 0, ex)                                                                      \
            else                                                                                                  \
                M3_BWD_LAUNCH(RR, 0, 0, ex)                                                                       \
        }                                                                                                         \
        break;
    switch (d.R) {
        M3_BWD_CASE(1)
        M3_BWD_CASE(2)
        M3_BWD_CASE(4)
        M3_BWD_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef M3_BWD_CASE
#undef M3_BWD_LAUNCH
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (gate) {
        const int64_t n = bh * d.seqlen * d.R * d.headdim;
        const unsigned gb = (unsigned)((n + 255) / 256 < 148 * 16 ? (n + 255) / 256 : 148 * 16);
        bwd_gate_dz<IO><<<gb, 256, 0, stream>>>((const IO*)dy, (const IO*)pp.z, (const IO*)pp.y_pre, pp.dz, n);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int64_t n4 = bh * d.seqlen * d.R * d.headdim / 4;
    int64_t nb = (n4 + 255) / 256;
    if (nb > 148 * 16) nb = 148 * 16;
    bwd_finish_dx<<<(unsigned)nb, 256, 0, stream>>>(reinterpret_cast<const float4*>(part_dx),
                                                    reinterpret_cast<float4*>(dx), n4, L.nPB);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const unsigned gy = (unsigned)(d.batch < 65535 ? d.batch : 65535);
    if (pp.on)
        bwd_finish_scalars_prep<<<dim3((unsigned)d.nheads, gy), 256, 0, stream>>>(
            reinterpret_cast<const float4*>(part_s), dt, lambda, pp.A_tok, pp.dt_raw, pp.dt_bias, ddt, dlambda, dA,
            pp.ddt_bias, d.batch, d.seqlen, (int)d.nheads, L.nPB);
    else
        bwd_finish_scalars<<<dim3((unsigned)d.nheads, gy), 256, 0, stream>>>(
            reinterpret_cast<const float4*>(part_s), dt, lambda, A, ddt, dlambda, dA, d.batch, d.seqlen,
            (int)d.nheads, L.nPB);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (pp.bc.on) {   // from the normalised rows' gradients to the raw rows', the gains' and the biases'
        const int64_t BT = d.batch * d.seqlen;
        const dim3 g2((unsigned)HR, (unsigned)((BT + 7) / 8 < 1024 ? (BT + 7) / 8 : 1024));
        bc_rows_backward<IO><<<g2, 256, 0, stream>>>((const IO*)B_raw, pp.bc.B_gain,
                                                     reinterpret_cast<const float*>(ws + w.rb), pp.bc.norm, dB,
                                                     pp.bc.dB_gain, pp.bc.dB_bias, BT, HR, (int)d.dstate);
        bc_rows_backward<IO><<<g2, 256, 0, stream>>>((const IO*)C_raw, pp.bc.C_gain,
                                                     reinterpret_cast<const float*>(ws + w.rc), pp.bc.norm, dC,
                                                     pp.bc.dC_gain, pp.bc.dC_bias, BT, HR, (int)d.dstate);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

bool bwd_supported(const ScanDims& d) {
    if (!(d.R == 1 || d.R == 2 || d.R == 4 || d.R == 8)) return false;
    if (d.headdim < 4 || d.headdim % 4 || d.headdim > 128) return false;
    const int P4 = (int)(d.headdim / 4);
    if (P4 & (P4 - 1)) return false;   // a pair's column lanes are an aligned power-of-two group
    if (d.dstate < 2 || d.dstate % 2 || d.dstate > 256) return false;
    const BwdLayout L =
        bwd_layout((int)d.headdim, (int)d.dstate, d.R, bwd_chunk(d.R), d.io == M3_DTYPE_BF16 ? 2 : 4);
    if ((int64_t)L.nPB * d.batch * d.nheads > (int64_t)INT32_MAX) return false;   // one-dimensional grid
    return sizeof(float) * (size_t)L.total <= 200 * 1024;
}

size_t bwd_workspace_size(const ScanDims& d) { return bwd_ws(d).total; }

size_t bwd_prep_workspace_size(const ScanDims& d) { return bwd_ws_prep_total(d); }

bool bwd_bc_supported(const ScanDims& d) {
    ScanDims f = d;
    f.io = M3_DTYPE_F32;   // the promoted path runs the fp32 adjoint
    return bwd_supported(d) && bwd_supported(f);
}

bool bwd_gate_supported(const ScanDims& d) {
    if (!bwd_supported(d)) return false;
    const BwdLayout L =
        bwd_layout((int)d.headdim, (int)d.dstate, d.R, bwd_chunk(d.R), d.io == M3_DTYPE_BF16 ? 2 : 4, true);
    return sizeof(float) * (size_t)L.total <= 200 * 1024;
}

cudaError_t launch_scan_bwd(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                            const float* A, const float* lambda, const float* omega, const void* dy,
                            const float* d_final, float* dx, float* dB, float* dC, float* ddt, float* dA,
                            float* dlambda, float* domega, void* workspace, cudaStream_t stream) {
    const BwdPrep pp{false, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, BwdBc{}};
    if (d.io == M3_DTYPE_BF16)
        return launch_bwd_io<__nv_bfloat16>(d, x, B, C, dt, A, lambda, omega, dy, d_final, dx, dB, dC, ddt, dA,
                                            dlambda, domega, workspace, stream, pp);
    return launch_bwd_io<float>(d, x, B, C, dt, A, lambda, omega, dy, d_final, dx, dB, dC, ddt, dA, dlambda,
                                domega, workspace, stream, pp);
}

cudaError_t launch_scan_bwd_prep(const ScanDims& d, const void* x, const void* B, const void* C,
                                 const float* dt_raw, const float* dt_bias, const float* A_tok, const float* u,
                                 const float* omega, const void* dy, const float* d_final, float* dx, float* dB,
                                 float* dC, float* ddt_raw, float* dA_tok, float* du, float* domega,
                                 float* ddt_bias, const void* z, const void* y_pre, float* dz, const BwdBcArgs& bca,
                                 void* workspace, cudaStream_t stream) {
    const BwdBc bc{bca.on, bca.norm, bca.eps, bca.B_gain, bca.C_gain, bca.B_bias, bca.C_bias,
                   bca.dB_gain, bca.dC_gain, bca.dB_bias, bca.dC_bias};
    const BwdPrep pp{true, dt_raw, dt_bias, u, A_tok, ddt_bias, z, y_pre, dz, bc};
    if (d.io == M3_DTYPE_BF16)
        return launch_bwd_io<__nv_bfloat16>(d, x, B, C, nullptr, nullptr, nullptr, omega, dy, d_final, dx, dB, dC,
                                            ddt_raw, dA_tok, du, domega, workspace, stream, pp);
    return launch_bwd_io<float>(d, x, B, C, nullptr, nullptr, nullptr, omega, dy, d_final, dx, dB, dC, ddt_raw,
                                dA_tok, du, domega, workspace, stream, pp);
}

}  // namespace m3
