// Fused single-token decode step of the Mamba-3 recurrence.
//
// Per (batch, head) the fp32 N x P state is read once and written once
// (float4, coalesced); everything else a step touches is a few hundred bytes,
// so the kernel is bound by HBM bandwidth on the state (single-token mode of
// "Mamba-3: Improved Sequence Modeling using State Space Principles",
// section 3.3 / Table 6: MIMO rank R adds R-fold arithmetic per state load).
//
//   h <- R(phi_t) (alpha_t h + beta_t B_{t-1} X_{t-1}^T) + gamma_t B_t X_t^T
//   y_t = h^T C_t
//
// One CTA owns one (batch, head).  Thread (g, c4) handles state pairs
// j = g, g + G, ... (rows 2j, 2j+1) for float4 column c4; the readout's sum
// over N is a per-thread partial followed by a shared-memory reduction over
// the G pair groups.
#include "m3_common.cuh"

namespace m3 {
namespace {

constexpr int kMaxUnits = 4;   // state pairs per thread

template <typename IO, int R>
__global__ void __launch_bounds__(512) decode_kernel(
    float* __restrict__ state, const IO* __restrict__ x_t, const IO* __restrict__ B_t,
    IO* __restrict__ cache, const IO* __restrict__ C_t, const float* __restrict__ dt_t,
    const float* __restrict__ A, const float* __restrict__ lam_t, const float* __restrict__ omega_t,
    IO* __restrict__ y_t, int H, int P, int N, int G) {
    extern __shared__ float sm[];
    const int64_t bh = blockIdx.x;
    const int h = (int)(bh % H);
    const int P4 = P >> 2, NP2 = N >> 1;
    const int tid = threadIdx.x, nt = blockDim.x;

    float* sB = sm;              // [R][N]  B_t
    float* sC = sB + R * N;      // [R][N]  C_t
    float* sBp = sC + R * N;     // [R][N]  B_{t-1}
    float* sX = sBp + R * N;     // [R][P]  X_t
    float* sXp = sX + R * P;     // [R][P]  X_{t-1}
    float* sCos = sXp + R * P;   // [N/2]
    float* sSin = sCos + NP2;    // [N/2]
    float* sRed = sSin + NP2;    // [nt][R*4]

    const float d = dt_t[bh], l = lam_t[bh], a = A[h];
    const float alpha = expf(d * a);
    const float beta = (1.0f - l) * d * alpha;
    const float gamma = l * d;

    const IO* xb = x_t + bh * R * P;
    const IO* Bb = B_t + bh * R * N;
    const IO* Cb = C_t + bh * R * N;
    IO* cb = cache + bh * (int64_t)R * (N + P);

    // Issue the state loads first: they are the bytes that matter.
    const int c4 = tid % P4, g = tid / P4;
    float4* st4 = reinterpret_cast<float4*>(state + bh * (int64_t)N * P);
    float4 h0[kMaxUnits], h1[kMaxUnits];
#pragma unroll
    for (int k = 0; k < kMaxUnits; ++k) {
        const int j = g + k * G;
        if (j < NP2) {
            h0[k] = st4[(2 * j) * P4 + c4];
            h1[k] = st4[(2 * j + 1) * P4 + c4];
        }
    }

    for (int i = tid; i < R * N; i += nt) {
        sB[i] = ld_io(Bb, i);
        sC[i] = ld_io(Cb, i);
        sBp[i] = ld_io(cb, i);
    }
    for (int i = tid; i < R * P; i += nt) {
        sX[i] = ld_io(xb, i);
        sXp[i] = ld_io(cb, R * N + i);
    }
    for (int j = tid; j < NP2; j += nt) {
        float sn, cs;
        sincosf(d * omega_t[bh * NP2 + j], &sn, &cs);
        sCos[j] = cs;
        sSin[j] = sn;
    }
    __syncthreads();
    // The old cache is in shared memory now: replace it with this token's factors.
    for (int i = tid; i < R * N; i += nt) cb[i] = Bb[i];
    for (int i = tid; i < R * P; i += nt) cb[R * N + i] = xb[i];

    float acc[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][e] = 0.0f;

#pragma unroll
    for (int k = 0; k < kMaxUnits; ++k) {
        const int j = g + k * G;
        if (j < NP2) {
            const float cs = sCos[j], sn = sSin[j];
            float o0[4], o1[4];
            const float a0v[4] = {h0[k].x, h0[k].y, h0[k].z, h0[k].w};
            const float a1v[4] = {h1[k].x, h1[k].y, h1[k].z, h1[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int p = c4 * 4 + e;
                float vp0 = 0.f, vp1 = 0.f, v0 = 0.f, v1 = 0.f;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float xp = sXp[r * P + p], xc = sX[r * P + p];
                    vp0 = fmaf(sBp[r * N + 2 * j], xp, vp0);
                    vp1 = fmaf(sBp[r * N + 2 * j + 1], xp, vp1);
                    v0 = fmaf(sB[r * N + 2 * j], xc, v0);
                    v1 = fmaf(sB[r * N + 2 * j + 1], xc, v1);
                }
                const float u0 = fmaf(alpha, a0v[e], beta * vp0);
                const float u1 = fmaf(alpha, a1v[e], beta * vp1);
                float n0, n1;
                rot2(cs, sn, u0, u1, n0, n1);
                o0[e] = fmaf(gamma, v0, n0);
                o1[e] = fmaf(gamma, v1, n1);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    acc[r][e] = fmaf(o0[e], sC[r * N + 2 * j], fmaf(o1[e], sC[r * N + 2 * j + 1], acc[r][e]));
            }
            st4[(2 * j) * P4 + c4] = make_float4(o0[0], o0[1], o0[2], o0[3]);
            st4[(2 * j + 1) * P4 + c4] = make_float4(o1[0], o1[1], o1[2], o1[3]);
        }
    }

    // Readout: sum the G pair-group partials of each (r, p).
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) sRed[tid * (R * 4) + r * 4 + e] = acc[r][e];
    __syncthreads();
    IO* yb = y_t + bh * R * P;
    for (int o = tid; o < R * P; o += nt) {
        const int r = o / P, p = o % P;
        const int cc = p >> 2, e = p & 3;
        float s = 0.f;
        for (int gg = 0; gg < G; ++gg) s += sRed[(gg * P4 + cc) * (R * 4) + r * 4 + e];
        st_io(yb, o, s);
    }
}

struct DecodeShape {
    int G, threads;
    size_t smem;
};

DecodeShape decode_shape(int64_t P, int64_t N, int R) {
    DecodeShape s{};
    const int P4 = (int)(P / 4), NP2 = (int)(N / 2);
    int G = (NP2 + kMaxUnits - 1) / kMaxUnits;
    const int want = 256 / P4 > 0 ? 256 / P4 : 1;
    if (G < want) G = want < NP2 ? want : NP2;
    s.G = G;
    s.threads = G * P4;
    s.smem = sizeof(float) * (size_t)(3 * R * N + 2 * R * P + N + (size_t)s.threads * R * 4);
    return s;
}

template <typename IO, int R>
cudaError_t launch_t(float* state, const void* x_t, const void* B_t, void* cache, const void* C_t,
                     const float* dt_t, const float* A, const float* lambda_t, const float* omega_t, void* y_t,
                     int64_t batch, int64_t nheads, int64_t P, int64_t N, cudaStream_t stream) {
    const DecodeShape s = decode_shape(P, N, R);
    auto kern = decode_kernel<IO, R>;
    if (s.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.smem);
        if (e != cudaSuccess) return e;
    }
    const int64_t blocks = batch * nheads;
    kern<<<(unsigned)blocks, s.threads, s.smem, stream>>>(
        state, (const IO*)x_t, (const IO*)B_t, (IO*)cache, (const IO*)C_t, dt_t, A, lambda_t, omega_t, (IO*)y_t,
        (int)nheads, (int)P, (int)N, s.G);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_io(int R, float* state, const void* x_t, const void* B_t, void* cache, const void* C_t,
                      const float* dt_t, const float* A, const float* lambda_t, const float* omega_t, void* y_t,
                      int64_t batch, int64_t nheads, int64_t P, int64_t N, cudaStream_t stream) {
#define M3_DEC_CASE(RR) \
    case RR: return launch_t<IO, RR>(state, x_t, B_t, cache, C_t, dt_t, A, lambda_t, omega_t, y_t, batch, nheads, P, N, stream);
    switch (R) {
        M3_DEC_CASE(1)
        M3_DEC_CASE(2)
        M3_DEC_CASE(4)
        M3_DEC_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef M3_DEC_CASE
}

}  // namespace

bool decode_supported(int64_t headdim, int64_t dstate, int R) {
    if (!(R == 1 || R == 2 || R == 4 || R == 8)) return false;
    if (headdim % 4 || headdim < 4 || headdim > 256) return false;
    if (dstate % 2 || dstate < 2 || dstate > 256) return false;
    const DecodeShape s = decode_shape(headdim, dstate, R);
    if (s.threads > 512) return false;
    if ((int64_t)s.G * kMaxUnits < dstate / 2) return false;
    return s.smem <= 200 * 1024;
}

cudaError_t launch_decode(float* state, const void* x_t, const void* B_t, void* cache, const void* C_t,
                          const float* dt_t, const float* A, const float* lambda_t, const float* omega_t,
                          void* y_t, int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate, int R,
                          int io, cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    if (io == M3_DTYPE_BF16)
        return launch_io<__nv_bfloat16>(R, state, x_t, B_t, cache, C_t, dt_t, A, lambda_t, omega_t, y_t, batch,
                                        nheads, headdim, dstate, stream);
    return launch_io<float>(R, state, x_t, B_t, cache, C_t, dt_t, A, lambda_t, omega_t, y_t, batch, nheads,
                            headdim, dstate, stream);
}

}  // namespace m3
