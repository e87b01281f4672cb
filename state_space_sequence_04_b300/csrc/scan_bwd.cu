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
// One CTA per (batch, head) sequence, CUDA cores, fp32 arithmetic: a forward
// pass stores every state h_t to the workspace, then the adjoint runs from
// the last token to the first, reading h_t and h_{t-1} back.  Thread layout
// of the decode kernel: thread (g, c4) holds state rows (2j, 2j+1) of pairs
// j = g, g + G, ... and columns 4 c4 .. 4 c4 + 3; sums over p combine the P/4
// lanes of a pair group with shuffles, sums over n go through shared memory.
#include <cuda_bf16.h>

#include "m3_common.cuh"

namespace m3 {
namespace {

constexpr int kBwdMaxK = 8;   // state pairs per thread

__device__ __forceinline__ float4 fma4b(float a, float4 x, float4 y) {
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ float4 sub4(float4 a, float4 b) { return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }
__device__ __forceinline__ float4 mul4(float a, float4 x) { return make_float4(a * x.x, a * x.y, a * x.z, a * x.w); }
__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }

struct BwdShape {
    int G, threads;
    size_t smem;
};

__host__ __device__ constexpr int round4(int v) { return (v + 3) & ~3; }

// Shared-memory sections, each starting on a 16-byte boundary (floats):
// B/X ping-pong [2][RN + R*P], C pairs [RN], dy [R*P], (cos, sin) [N/2] pairs,
// dX partials [warps][R*P], block partials [warps][4]; RN = R*N rounded up to 4.
BwdShape bwd_shape(int64_t P, int64_t N, int R) {
    BwdShape s{};
    const int P4 = (int)(P / 4), NP2 = (int)(N / 2);
    int G = 256 / P4;
    if (G > NP2) G = NP2;
    if (G < 1) G = 1;
    s.G = G;
    s.threads = (G * P4 + 31) / 32 * 32;   // whole warps; threads past G * P4 idle
    const int nw = s.threads / 32, RN = round4(R * (int)N), RP = R * (int)P;
    s.smem = sizeof(float) * (size_t)(2 * (RN + RP) + RN + RP + round4((int)N) + nw * RP + nw * 4);
    return s;
}

template <typename IO, int R>
__global__ void __launch_bounds__(256, 1) scan_bwd_kernel(
    const IO* __restrict__ x, const IO* __restrict__ B, const IO* __restrict__ C, const float* __restrict__ dt,
    const float* __restrict__ A, const float* __restrict__ lam, const float* __restrict__ omega,
    const IO* __restrict__ dy, const float* __restrict__ dfin, float* __restrict__ dx, float* __restrict__ dB,
    float* __restrict__ dC, float* __restrict__ ddt, float* __restrict__ dA, float* __restrict__ dlam,
    float* __restrict__ domega, float* __restrict__ S, int64_t T, int H, int P, int N, int G) {
    extern __shared__ __align__(16) float sm[];
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / H;
    const int h = (int)(bh % H);
    const int P4 = P >> 2, NP2 = N >> 1;
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = (nt + 31) >> 5;
    const int c4 = tid % P4, g = tid / P4;
    const bool gv = g < G;   // holds state pairs (threads past G * P4 only join reductions)
    const int RN = round4(R * N);

    float* sBX[2] = {sm, sm + (RN + R * P)};   // B rows as pairs [N/2][R] float2, then X [R*P] at RN
    float* sCp = sm + 2 * (RN + R * P);        // C pairs [N/2][R]
    float* sDy = sCp + RN;                     // [R*P]
    float2* sCS = reinterpret_cast<float2*>(sDy + R * P);   // [N/2] (cos, sin) of phi_t
    float* sRed = reinterpret_cast<float*>(sCS) + round4(N);  // [warps][R*P]
    float* sBlk = sRed + nw * R * P;                        // [warps][4]

    const float a_h = A[h];
    auto tok = [&](int64_t t) { return (b * T + t) * H + h; };   // (batch, token, head) index
    auto stage_bx = [&](int64_t t, float* dst) {   // B_t (pairs) and X_t of this head; zeros for t < 0
        for (int i = tid; i < R * N; i += nt) {
            const int r = i / N, n = i % N;
            dst[((n >> 1) * R + r) * 2 + (n & 1)] = t >= 0 ? ld_io(B, tok(t) * R * N + i) : 0.f;
        }
        for (int i = tid; i < R * P; i += nt) dst[RN + i] = t >= 0 ? ld_io(x, tok(t) * R * P + i) : 0.f;
    };
    // v[rows 2j, 2j+1][cols of c4] = sum_r B[r, 2j / 2j+1] X[r, cols] from a staged buffer
    auto outer = [&](const float* buf, int j, float4& v0, float4& v1) {
        const float2* b2 = reinterpret_cast<const float2*>(buf);
        const float4* x4 = reinterpret_cast<const float4*>(buf + RN);
        v0 = make_float4(0.f, 0.f, 0.f, 0.f);
        v1 = v0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float2 bb = b2[j * R + r];
            const float4 xx = x4[r * P4 + c4];
            v0 = fma4b(bb.x, xx, v0);
            v1 = fma4b(bb.y, xx, v1);
        }
    };
    float4* S4 = reinterpret_cast<float4*>(S + bh * T * (int64_t)N * P);
    auto srow = [&](int64_t t, int n) { return S4 + (t * N + n) * P4 + c4; };

    // ------------------------------ forward: every h_t ------------------------------
    float4 h0[kBwdMaxK], h1[kBwdMaxK];
#pragma unroll
    for (int k = 0; k < kBwdMaxK; ++k) h0[k] = h1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    stage_bx(-1, sBX[1]);
    for (int64_t t = 0; t < T; ++t) {
        float* cur = sBX[t & 1];
        const float* prv = sBX[(t + 1) & 1];
        stage_bx(t, cur);
        const float d = dt[tok(t)], l = lam[tok(t)];
        for (int j = tid; j < NP2; j += nt) {
            float sn, cs;
            sincosf(d * omega[tok(t) * NP2 + j], &sn, &cs);
            sCS[j] = make_float2(cs, sn);
        }
        __syncthreads();
        const float alpha = expf(d * a_h), beta = (1.f - l) * d * alpha, gamma = l * d;
#pragma unroll
        for (int k = 0; k < kBwdMaxK; ++k) {
            const int j = g + k * G;
            if (gv && j < NP2) {
                float4 vp0, vp1, v0, v1;
                outer(prv, j, vp0, vp1);
                outer(cur, j, v0, v1);
                const float4 u0 = fma4b(alpha, h0[k], mul4(beta, vp0));
                const float4 u1 = fma4b(alpha, h1[k], mul4(beta, vp1));
                const float2 cs = sCS[j];
                float4 o0, o1;
                rot2(cs.x, cs.y, u0.x, u1.x, o0.x, o1.x);
                rot2(cs.x, cs.y, u0.y, u1.y, o0.y, o1.y);
                rot2(cs.x, cs.y, u0.z, u1.z, o0.z, o1.z);
                rot2(cs.x, cs.y, u0.w, u1.w, o0.w, o1.w);
                h0[k] = fma4b(gamma, v0, o0);
                h1[k] = fma4b(gamma, v1, o1);
                *srow(t, 2 * j) = h0[k];
                *srow(t, 2 * j + 1) = h1[k];
            }
        }
        __syncthreads();   // the buffers and (cos, sin) are restaged next
    }

    // ------------------------------ backward: the adjoint ------------------------------
    float4 ub0[kBwdMaxK], ub1[kBwdMaxK];   // ubar_{t+1}
#pragma unroll
    for (int k = 0; k < kBwdMaxK; ++k) ub0[k] = ub1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float alpha_n = 0.f, beta_n = 0.f;     // alpha_{t+1}, beta_{t+1}
    float dA_acc = 0.f;
    // the buffers: B_t, X_t in sBX[t & 1] and B_{t-1}, X_{t-1} in the other one
    stage_bx(T - 1, sBX[(T - 1) & 1]);
    for (int64_t t = T - 1; t >= 0; --t) {
        float* cur = sBX[t & 1];
        float* prv = sBX[(t + 1) & 1];
        stage_bx(t - 1, prv);
        for (int i = tid; i < R * N; i += nt) {
            const int r = i / N, n = i % N;
            sCp[((n >> 1) * R + r) * 2 + (n & 1)] = ld_io(C, tok(t) * R * N + i);
        }
        for (int i = tid; i < R * P; i += nt) sDy[i] = ld_io(dy, tok(t) * R * P + i);
        const float d = dt[tok(t)], l = lam[tok(t)];
        for (int j = tid; j < NP2; j += nt) {
            float sn, cs;
            sincosf(d * omega[tok(t) * NP2 + j], &sn, &cs);
            sCS[j] = make_float2(cs, sn);
        }
        __syncthreads();
        const float alpha = expf(d * a_h), beta = (1.f - l) * d * alpha, gamma = l * d;
        const float2* c2 = reinterpret_cast<const float2*>(sCp);
        const float2* b2 = reinterpret_cast<const float2*>(cur);
        const float4* x4 = reinterpret_cast<const float4*>(cur + RN);
        const float4* dy4 = reinterpret_cast<const float4*>(sDy);
        float p_alpha = 0.f, p_beta = 0.f, p_gamma = 0.f, p_omega = 0.f;
        float4 dXp[R];
#pragma unroll
        for (int r = 0; r < R; ++r) dXp[r] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kBwdMaxK; ++k) {
            if (k * G >= NP2) break;   // uniform over the block
            const int j = g + k * G;
            const bool on = gv && j < NP2;
            const int jj = on ? j : 0;
            float4 ht0 = make_float4(0.f, 0.f, 0.f, 0.f), ht1 = ht0, hp0 = ht0, hp1 = ht0;
            if (on) {
                ht0 = *srow(t, 2 * j);
                ht1 = *srow(t, 2 * j + 1);
                if (t > 0) {
                    hp0 = *srow(t - 1, 2 * j);
                    hp1 = *srow(t - 1, 2 * j + 1);
                }
            }
            float4 v0, v1, vp0, vp1;
            outer(cur, jj, v0, v1);
            outer(prv, jj, vp0, vp1);
            // gbar_t = C_t dy_t^T + alpha_{t+1} ubar_{t+1} (+ the final-state seed)
            float4 g0 = mul4(alpha_n, ub0[k]), g1 = mul4(alpha_n, ub1[k]);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 cc = c2[jj * R + r];
                g0 = fma4b(cc.x, dy4[r * P4 + c4], g0);
                g1 = fma4b(cc.y, dy4[r * P4 + c4], g1);
            }
            if (t == T - 1 && dfin != nullptr && on) {
                const float4* df4 = reinterpret_cast<const float4*>(dfin + bh * (int64_t)N * P);
                g0 = add4(g0, df4[(2 * j) * P4 + c4]);
                g1 = add4(g1, df4[(2 * j + 1) * P4 + c4]);
            }
            if (!on) g0 = g1 = make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 dv0 = fma4b(gamma, g0, mul4(beta_n, ub0[k]));
            const float4 dv1 = fma4b(gamma, g1, mul4(beta_n, ub1[k]));
            const float4 r0 = sub4(ht0, mul4(gamma, v0)), r1 = sub4(ht1, mul4(gamma, v1));
            // dphi_j partial over this thread's columns, then over the pair group's lanes
            float dphi = dot4(g1, r0) - dot4(g0, r1);
            const float2 cs = sCS[jj];
            // ubar_t = R(phi)^T gbar_t
            const float4 un0 = add4(mul4(cs.x, g0), mul4(cs.y, g1));
            const float4 un1 = sub4(mul4(cs.x, g1), mul4(cs.y, g0));
            p_alpha += dot4(un0, hp0) + dot4(un1, hp1);
            p_beta += dot4(un0, vp0) + dot4(un1, vp1);
            p_gamma += dot4(g0, v0) + dot4(g1, v1);
            ub0[k] = un0;
            ub1[k] = un1;
            // dC_t[r, n] = sum_p h_t[n, p] dy_t[r, p];  dB_t[r, n] = sum_p dv_t[n, p] X_t[r, p]
            float pc[2 * R], pb[2 * R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float4 dyr = dy4[r * P4 + c4], xr = x4[r * P4 + c4];
                pc[2 * r] = dot4(ht0, dyr);
                pc[2 * r + 1] = dot4(ht1, dyr);
                pb[2 * r] = dot4(dv0, xr);
                pb[2 * r + 1] = dot4(dv1, xr);
                // dX_t[r, p] = sum_n dv_t[n, p] B_t[r, n]
                const float2 bb = b2[jj * R + r];
                dXp[r] = fma4b(bb.x, dv0, fma4b(bb.y, dv1, dXp[r]));
            }
            for (int o = 1; o < P4; o <<= 1) {
                dphi += __shfl_xor_sync(0xffffffffu, dphi, o);
#pragma unroll
                for (int i = 0; i < 2 * R; ++i) {
                    pc[i] += __shfl_xor_sync(0xffffffffu, pc[i], o);
                    pb[i] += __shfl_xor_sync(0xffffffffu, pb[i], o);
                }
            }
            if (on && c4 == 0) {
                const int64_t tb = tok(t);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    dC[(tb * R + r) * N + 2 * j] = pc[2 * r];
                    dC[(tb * R + r) * N + 2 * j + 1] = pc[2 * r + 1];
                    dB[(tb * R + r) * N + 2 * j] = pb[2 * r];
                    dB[(tb * R + r) * N + 2 * j + 1] = pb[2 * r + 1];
                }
                const float w = omega[tb * NP2 + j];
                domega[tb * NP2 + j] = d * dphi;
                p_omega += w * dphi;
            }
        }
        // dX over the pair groups: lanes of one warp first, then the warps through shared memory
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
            float4* red4 = reinterpret_cast<float4*>(sRed) + warp * (R * P4);
#pragma unroll
            for (int r = 0; r < R; ++r) red4[r * P4 + c4] = dXp[r];
        }
        p_alpha = warp_sum(p_alpha);
        p_beta = warp_sum(p_beta);
        p_gamma = warp_sum(p_gamma);
        p_omega = warp_sum(p_omega);
        if (lane == 0) {
            sBlk[warp * 4 + 0] = p_alpha;
            sBlk[warp * 4 + 1] = p_beta;
            sBlk[warp * 4 + 2] = p_gamma;
            sBlk[warp * 4 + 3] = p_omega;
        }
        __syncthreads();
        for (int i = tid; i < R * P; i += nt) {
            float s = 0.f;
            for (int w = 0; w < nw; ++w) s += sRed[w * R * P + i];
            dx[tok(t) * R * P + i] = s;
        }
        if (tid == 0) {
            float da = 0.f, db = 0.f, dg = 0.f, dw = 0.f;
            for (int w = 0; w < nw; ++w) {
                da += sBlk[w * 4 + 0];
                db += sBlk[w * 4 + 1];
                dg += sBlk[w * 4 + 2];
                dw += sBlk[w * 4 + 3];
            }
            // alpha = e^{d a}, beta = (1 - l) d alpha, gamma = l d, phi = d omega
            const float dalpha = da + db * (1.f - l) * d;          // through alpha and beta's alpha
            ddt[tok(t)] = dalpha * a_h * alpha + db * (1.f - l) * alpha + dg * l + dw;
            dlam[tok(t)] = -d * alpha * db + d * dg;
            dA_acc += dalpha * d * alpha;
        }
        alpha_n = alpha;
        beta_n = beta;
        __syncthreads();   // every buffer is restaged next
    }
    if (tid == 0) atomicAdd(&dA[h], dA_acc);
}

template <typename IO>
cudaError_t launch_bwd_io(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                          const float* A, const float* lambda, const float* omega, const void* dy,
                          const float* d_final, float* dx, float* dB, float* dC, float* ddt, float* dA,
                          float* dlambda, float* domega, void* workspace, cudaStream_t stream) {
    const BwdShape s = bwd_shape(d.headdim, d.dstate, d.R);
    const int64_t bh = d.batch * d.nheads;
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * (size_t)d.nheads, stream);
    if (e != cudaSuccess || bh == 0 || d.seqlen == 0) return e;
#define M3_BWD_CASE(RR)                                                                                            \
    case RR: {                                                                                                     \
        auto k = scan_bwd_kernel<IO, RR>;                                                                          \
        if (s.smem > 48 * 1024 &&                                                                                  \
            (e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.smem)) != cudaSuccess) \
            return e;                                                                                              \
        k<<<(unsigned)bh, s.threads, s.smem, stream>>>((const IO*)x, (const IO*)B, (const IO*)C, dt, A, lambda,    \
                                                      omega, (const IO*)dy, d_final, dx, dB, dC, ddt, dA, dlambda, \
                                                      domega, static_cast<float*>(workspace), d.seqlen,           \
                                                      (int)d.nheads, (int)d.headdim, (int)d.dstate, s.G);          \
        return cudaGetLastError();                                                                                 \
    }
    switch (d.R) {
        M3_BWD_CASE(1)
        M3_BWD_CASE(2)
        M3_BWD_CASE(4)
        M3_BWD_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef M3_BWD_CASE
}

}  // namespace

bool bwd_supported(const ScanDims& d) {
    if (!(d.R == 1 || d.R == 2 || d.R == 4 || d.R == 8)) return false;
    if (d.headdim < 4 || d.headdim % 4 || d.headdim > 128) return false;
    const int P4 = (int)(d.headdim / 4);
    if (P4 & (P4 - 1)) return false;                       // the pair-group lanes are a power of two
    if (d.dstate < 2 || d.dstate % 2 || d.dstate > 256) return false;
    const BwdShape s = bwd_shape(d.headdim, d.dstate, d.R);
    if ((d.dstate / 2 + s.G - 1) / s.G > kBwdMaxK) return false;
    return s.smem <= 200 * 1024;
}

size_t bwd_workspace_size(const ScanDims& d) {
    return sizeof(float) * (size_t)(d.batch * d.nheads) * (size_t)d.seqlen * (size_t)(d.dstate * d.headdim);
}

cudaError_t launch_scan_bwd(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                            const float* A, const float* lambda, const float* omega, const void* dy,
                            const float* d_final, float* dx, float* dB, float* dC, float* ddt, float* dA,
                            float* dlambda, float* domega, void* workspace, cudaStream_t stream) {
    if (d.io == M3_DTYPE_BF16)
        return launch_bwd_io<__nv_bfloat16>(d, x, B, C, dt, A, lambda, omega, dy, d_final, dx, dB, dC, ddt, dA,
                                            dlambda, domega, workspace, stream);
    return launch_bwd_io<float>(d, x, B, C, dt, A, lambda, omega, dy, d_final, dx, dB, dC, ddt, dA, dlambda,
                                domega, workspace, stream);
}

}  // namespace m3
