// Chunked Mamba-3 prefill on CUDA cores (fp32 arithmetic), for any size the
// ABI accepts and for both io dtypes.  It is the exact-fp32 mode and the
// fallback where the tensor-core path does not apply.
//
// The chunked algorithm ("Mamba-3: Improved Sequence Modeling using State
// Space Principles", section 3.3, with the decay x two-band mask of section
// 3.1.3 / Eq. 7 and the rotary equivalence of Propositions 3-4) for chunk c =
// tokens [c0, c0+q):
//
//   l_t = dt_t A, cum_t = sum_{k=c0..t} l_k,  Psi_t = sum_{k=c0..t} dt_k omega_k,
//   gamma_t = lambda_t dt_t,  w_s = gamma_s + (1 - lambda_{s+1}) dt_{s+1},
//   B~_s = R(-Psi_s) B_s,  C~_t = R(-Psi_t) C_t,
//   y_t = sum_{s<=t} exp(cum_t - cum_s) (s==t ? gamma_t : w_s) (C~_t . B~_s) X_s
//         + exp(cum_t) C~_t^T H_{c-1},
//   U_c = sum_s exp(cum_end - cum_s) w_s R(Theta_c - Psi_s) B_s X_s^T,
//   H_c = exp(cum_end) R(Theta_c) H_{c-1} + U_c.
//
// H is the physical-frame state plus the pending delayed write of the chunk's
// last token (whose w uses the next chunk's first lambda, dt; 0 past the end),
// so the trapezoidal term that crosses a chunk boundary is carried exactly.
//
// Three launches: chunk states U_c (kernel A), the state-passing scan (in
// place, giving H_{c-1}), chunk outputs (kernel C).
#include <algorithm>

#include "m3_common.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxAcc = 64;     // N*P <= 256 * 64
constexpr int kRowTile = 64;    // rows (token, rank) per output tile
constexpr int kPad = 4;

// Inclusive prefix sum over a 256-thread block.  sWarp: 8 floats of smem.
__device__ __forceinline__ float block_scan256(float v, float* sWarp) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_inclusive_sum(v);
    if (lane == 31) sWarp[w] = v;
    __syncthreads();
    float off = 0.f;
    for (int i = 0; i < w; ++i) off += sWarp[i];
    __syncthreads();
    return v + off;
}

// ---------------------------------------------------------------------------
// B or C of the pre-activation entry points: RMS normalisation of each
// (token, rank) row over N (inverse RMS precomputed per row in `inv`), gain [N],
// head-specific channel bias [H, R, N].  on = 0: the values as given.
struct BcArgs {
    int on, norm;
    const float* inv;
    const float* gain;
    const float* bias;
};

// Element n of the row starting at `base` (= row * N); hr = h * R + r.
template <typename IO>
__device__ __forceinline__ float ld_bc(const IO* p, int64_t base, int n, int N, int hr, const BcArgs& a) {
    float v = ld_io(p, base + n);
    if (a.on) {
        if (a.norm) v *= a.inv[base / N] * (a.gain != nullptr ? a.gain[n] : 1.f);
        if (a.bias != nullptr) v += a.bias[(int64_t)hr * N + n];
    }
    return v;
}

// ---------------------------------------------------------------------------
// Kernel A: U_c, l_c = cum_end, Theta_c for every (batch*head, chunk).
template <typename IO, int R>
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(
    const IO* __restrict__ x, const IO* __restrict__ B, const float* __restrict__ dt,
    const float* __restrict__ A, const float* __restrict__ lam, const float* __restrict__ omega,
    float* __restrict__ U, float* __restrict__ ld_out, float* __restrict__ ang_out,
    int64_t T, int H, int P, int N, int Q, int nc, int a_tok, const BcArgs bcB) {
    extern __shared__ float sm[];
    constexpr int KB = 32 / R > 0 ? 32 / R : 1;   // tokens per staging block
    const int64_t bh = blockIdx.x;
    const int c = blockIdx.y;
    const int64_t b = bh / H;
    const int h = (int)(bh % H);
    const int64_t c0 = (int64_t)c * Q;
    const int q = (int)min((int64_t)Q, T - c0);
    const int tid = threadIdx.x;
    const int NP2 = N / 2;

    float* sWt = sm;                 // [Q]
    float* sWarp = sWt + Q;          // [8]
    float* sCe = sWarp + 8;          // [1] cum_end
    float* sAng = sCe + 4;           // [N/2] running suffix angle
    float* sBr = sAng + NP2;         // [KB*R][N]
    float* sX = sBr + KB * R * N;    // [KB*R][P]

    const float a_head = a_tok ? 0.f : A[h];
    float ell = 0.f, gam = 0.f, wnext = 0.f;
    if (tid < q) {
        const int64_t idx = (b * T + c0 + tid) * H + h;
        const float d = dt[idx], l = lam[idx];
        ell = d * (a_tok ? A[idx] : a_head);
        gam = l * d;
        if (c0 + tid + 1 < T) {
            const int64_t in = idx + H;
            wnext = (1.f - lam[in]) * dt[in];
        }
    }
    const float cum = block_scan256(ell, sWarp);
    if (tid == q - 1) sCe[0] = cum;
    for (int j = tid; j < NP2; j += kThreads) sAng[j] = 0.f;
    __syncthreads();
    const float cend = sCe[0];
    if (tid < q) sWt[tid] = expf(cend - cum) * (gam + wnext);
    if (tid == 0) ld_out[bh * nc + c] = cend;
    __syncthreads();

    const int NPel = N * P;
    float acc[kMaxAcc];
#pragma unroll
    for (int i = 0; i < kMaxAcc; ++i) acc[i] = 0.f;

    const int nblk = (q + KB - 1) / KB;
    for (int blk = nblk - 1; blk >= 0; --blk) {
        const int s0 = blk * KB;
        const int kb = min(KB, q - s0);
        // rotate B_s by the remaining angle Theta_c - Psi_s and scale by its weight
        for (int j = tid; j < NP2; j += kThreads) {
            float run = sAng[j];
            for (int sl = kb - 1; sl >= 0; --sl) {
                const int s = s0 + sl;
                const int64_t tok = b * T + c0 + s;
                float sn, cs;
                sincosf(run, &sn, &cs);
                const float wt = sWt[s];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int64_t base = ((tok * H + h) * R + r) * N;
                    float o0, o1;
                    rot2(cs, sn, ld_bc(B, base, 2 * j, N, h * R + r, bcB), ld_bc(B, base, 2 * j + 1, N, h * R + r, bcB),
                         o0, o1);
                    sBr[(sl * R + r) * N + 2 * j] = wt * o0;
                    sBr[(sl * R + r) * N + 2 * j + 1] = wt * o1;
                }
                run += dt[tok * H + h] * omega[(tok * H + h) * NP2 + j];
            }
            sAng[j] = run;
        }
        for (int i = tid; i < kb * R * P; i += kThreads) {
            const int row = i / P, p = i % P;
            const int sl = row / R, r = row % R;
            const int64_t tok = b * T + c0 + s0 + sl;
            sX[i] = ld_io(x, ((tok * H + h) * R + r) * P + p);
        }
        __syncthreads();
        const int K = kb * R;
#pragma unroll
        for (int i = 0; i < kMaxAcc; ++i) {
            const int e = tid + i * kThreads;
            if (e < NPel) {
                const int n = e / P, p = e % P;
                float s = acc[i];
                for (int k = 0; k < K; ++k) s = fmaf(sBr[k * N + n], sX[k * P + p], s);
                acc[i] = s;
            }
        }
        __syncthreads();
    }
    float* Uc = U + (bh * nc + c) * (int64_t)NPel;
#pragma unroll
    for (int i = 0; i < kMaxAcc; ++i) {
        const int e = tid + i * kThreads;
        if (e < NPel) Uc[e] = acc[i];
    }
    for (int j = tid; j < NP2; j += kThreads) ang_out[(bh * nc + c) * NP2 + j] = sAng[j];
}

// ---------------------------------------------------------------------------
// Kernel C: outputs of one 64-row tile (TT = 64/R tokens) of one chunk.
template <typename IO, int R>
__global__ void __launch_bounds__(kThreads) chunk_scan_kernel(
    const IO* __restrict__ x, const IO* __restrict__ B, const IO* __restrict__ C,
    const float* __restrict__ dt, const float* __restrict__ A, const float* __restrict__ lam,
    const float* __restrict__ omega, const float* __restrict__ Hc, IO* __restrict__ y,
    int64_t T, int H, int P, int N, int Q, int nc, int a_tok, const BcArgs bcB, const BcArgs bcC,
    const IO* __restrict__ gate) {
    extern __shared__ float sm[];
    constexpr int RT = kRowTile;
    constexpr int TT = RT / R;
    constexpr int LD = RT + kPad;
    const int64_t bh = blockIdx.x;
    const int c = blockIdx.y;
    const int rt = blockIdx.z;
    const int64_t b = bh / H;
    const int h = (int)(bh % H);
    const int64_t c0 = (int64_t)c * Q;
    const int q = (int)min((int64_t)Q, T - c0);
    const int ta = rt * TT;
    if (ta >= q) return;
    const int tid = threadIdx.x;
    const int NP2 = N / 2;
    const int tlast = min(q, ta + TT);   // tokens needed: [0, tlast)

    float* sCum = sm;                    // [Q]
    float* sGam = sCum + Q;              // [Q]
    float* sW = sGam + Q;                // [Q]
    float* sWarp = sW + Q;               // [8]
    float* sPsi = sWarp + 8;             // [Q][N/2]
    float* sCt = sPsi + Q * NP2;         // [N][LD]  C~ of the row tile, transposed
    float* sBt = sCt + N * LD;           // [N][LD]  B~ of a column tile, transposed / H slices
    float* sX = sBt + N * LD;            // [RT][P]
    float* sS = sX + RT * P;             // [RT][RT+1]

    const float a_head = a_tok ? 0.f : A[h];
    float ell = 0.f, gam = 0.f, wsh = 0.f;
    if (tid < q) {
        const int64_t idx = (b * T + c0 + tid) * H + h;
        const float d = dt[idx], l = lam[idx];
        ell = d * (a_tok ? A[idx] : a_head);
        gam = l * d;
        wsh = gam;
        if (tid + 1 < q) wsh += (1.f - lam[idx + H]) * dt[idx + H];
    }
    const float cum = block_scan256(ell, sWarp);
    if (tid < q) {
        sCum[tid] = cum;
        sGam[tid] = gam;
        sW[tid] = wsh;
    }
    // chunk-local inclusive angle prefix, one thread per pair
    for (int j = tid; j < NP2; j += kThreads) {
        float run = 0.f;
        for (int t = 0; t < tlast; ++t) {
            const int64_t tok = b * T + c0 + t;
            run += dt[tok * H + h] * omega[(tok * H + h) * NP2 + j];
            sPsi[t * NP2 + j] = run;
        }
    }
    __syncthreads();

    // C~ rows of this tile: row = tl*R + r
    for (int i = tid; i < TT * R * NP2; i += kThreads) {
        const int j = i % NP2, row = i / NP2;
        const int tl = row / R, r = row % R;
        const int t = ta + tl;
        float o0 = 0.f, o1 = 0.f;
        if (t < q) {
            const int64_t base = (((b * T + c0 + t) * H + h) * R + r) * N;
            float sn, cs;
            sincosf(-sPsi[t * NP2 + j], &sn, &cs);
            rot2(cs, sn, ld_bc(C, base, 2 * j, N, h * R + r, bcC), ld_bc(C, base, 2 * j + 1, N, h * R + r, bcC), o0, o1);
        }
        sCt[(2 * j) * LD + row] = o0;
        sCt[(2 * j + 1) * LD + row] = o1;
    }

    // Output accumulator: thread (rg, cg) owns rows rg*RPT .. +RPT-1, cols 4cg .. 4cg+3.
    const int CG = P / 4;
    const int RG = kThreads / CG;
    const int RPT = RT / RG;             // P/16 rows per thread (1..8)
    const int cg = tid % CG, rg = tid / CG;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;

    // inter-chunk term: exp(cum_t) C~_t^T H_{c-1}, H streamed in row slices
    {
        const float* Hp = Hc + (bh * nc + c) * (int64_t)N * P;
        int NS = (N * LD) / P;
        if (NS > N) NS = N;
        for (int n0 = 0; n0 < N; n0 += NS) {
            const int ns = min(NS, N - n0);
            __syncthreads();
            for (int i = tid; i < ns * P; i += kThreads) sBt[i] = Hp[(int64_t)n0 * P + i];
            __syncthreads();
            for (int n = 0; n < ns; ++n) {
                const float4 hv = *reinterpret_cast<const float4*>(&sBt[n * P + 4 * cg]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i < RPT) {
                        const float cv = sCt[(n0 + n) * LD + rg * RPT + i];
                        acc[i][0] = fmaf(cv, hv.x, acc[i][0]);
                        acc[i][1] = fmaf(cv, hv.y, acc[i][1]);
                        acc[i][2] = fmaf(cv, hv.z, acc[i][2]);
                        acc[i][3] = fmaf(cv, hv.w, acc[i][3]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < RPT) {
                const int t = ta + (rg * RPT + i) / R;
                const float e = t < q ? expf(sCum[t]) : 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[i][k] *= e;
            }
        }
    }

    // intra-chunk term over column tiles st = 0 .. rt
    const int ti = tid / 16, tj = tid % 16;   // 4x4 block of the 64x64 score tile
    for (int st = 0; st <= rt; ++st) {
        const int sa = st * TT;
        __syncthreads();
        for (int i = tid; i < TT * R * NP2; i += kThreads) {
            const int j = i % NP2, col = i / NP2;
            const int sl = col / R, r = col % R;
            const int s = sa + sl;
            float o0 = 0.f, o1 = 0.f;
            if (s < q) {
                const int64_t base = (((b * T + c0 + s) * H + h) * R + r) * N;
                float sn, cs;
                sincosf(-sPsi[s * NP2 + j], &sn, &cs);
                rot2(cs, sn, ld_bc(B, base, 2 * j, N, h * R + r, bcB), ld_bc(B, base, 2 * j + 1, N, h * R + r, bcB),
                     o0, o1);
            }
            sBt[(2 * j) * LD + col] = o0;
            sBt[(2 * j + 1) * LD + col] = o1;
        }
        for (int i = tid; i < RT * P; i += kThreads) {
            const int col = i / P, p = i % P;
            const int sl = col / R, r = col % R;
            const int s = sa + sl;
            sX[i] = s < q ? ld_io(x, (((b * T + c0 + s) * H + h) * R + r) * P + p) : 0.f;
        }
        __syncthreads();
        // S = C~ B~^T on the 64x64 tile, then the mask
        float sc[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) sc[u][v] = 0.f;
        for (int n = 0; n < N; ++n) {
            const float4 cv = *reinterpret_cast<const float4*>(&sCt[n * LD + 4 * ti]);
            const float4 bv = *reinterpret_cast<const float4*>(&sBt[n * LD + 4 * tj]);
            const float cc[4] = {cv.x, cv.y, cv.z, cv.w};
            const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) sc[u][v] = fmaf(cc[u], bb[v], sc[u][v]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int row = 4 * ti + u;
            const int t = ta + row / R;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int col = 4 * tj + v;
                const int s = sa + col / R;
                float m = 0.f;
                if (t < q && s <= t) m = (s == t) ? sGam[t] : expf(sCum[t] - sCum[s]) * sW[s];
                sS[row * (RT + 1) + col] = m * sc[u][v];
            }
        }
        __syncthreads();
        for (int k = 0; k < RT; ++k) {
            const float4 xv = *reinterpret_cast<const float4*>(&sX[k * P + 4 * cg]);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < RPT) {
                    const float sv = sS[(rg * RPT + i) * (RT + 1) + k];
                    acc[i][0] = fmaf(sv, xv.x, acc[i][0]);
                    acc[i][1] = fmaf(sv, xv.y, acc[i][1]);
                    acc[i][2] = fmaf(sv, xv.z, acc[i][2]);
                    acc[i][3] = fmaf(sv, xv.w, acc[i][3]);
                }
            }
        }
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < RPT) {
            const int row = rg * RPT + i;
            const int t = ta + row / R, r = row % R;
            if (t < q) {
                const int64_t base = (((b * T + c0 + t) * H + h) * R + r) * P + 4 * cg;
#pragma unroll
                for (int e = 0; e < 4; ++e)   // output gate y * silu(z) when given
                    st_io(y, base + e, gate != nullptr ? acc[i][e] * silu_f(ld_io(gate, base + e)) : acc[i][e]);
            }
        }
    }
}

size_t smem_a(const ScanDims& d) {
    const int KB = 32 / d.R > 0 ? 32 / d.R : 1;
    return sizeof(float) * (size_t)(d.chunk + 8 + 4 + d.dstate / 2 + KB * d.R * (d.dstate + d.headdim));
}

size_t smem_c(const ScanDims& d) {
    const int64_t LD = kRowTile + kPad;
    return sizeof(float) * (size_t)(3 * d.chunk + 8 + d.chunk * (d.dstate / 2) + 2 * d.dstate * LD +
                                    kRowTile * d.headdim + kRowTile * (kRowTile + 1));
}

template <typename IO, int R>
cudaError_t launch_rt(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                      const float* A, const float* lambda, const float* omega, void* y, float* final_state,
                      void* workspace, int a_tok, const BcArgs& bcB, const BcArgs& bcC, const void* gate,
                      cudaStream_t stream) {
    const int64_t bh = d.batch * d.nheads;
    const int64_t nc = d.nchunks();
    const int64_t NP = d.dstate * d.headdim;
    float* U = static_cast<float*>(workspace);
    float* ld = U + bh * nc * NP;
    float* ang = ld + bh * nc;
    cudaError_t e;
    if (bh > 0 && nc > 0) {
        const size_t sa = smem_a(d);
        auto ka = chunk_state_kernel<IO, R>;
        if ((e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sa)) != cudaSuccess) return e;
        ka<<<dim3((unsigned)bh, (unsigned)nc), kThreads, sa, stream>>>(
            (const IO*)x, (const IO*)B, dt, A, lambda, omega, U, ld, ang, d.seqlen, (int)d.nheads, (int)d.headdim,
            (int)d.dstate, d.chunk, (int)nc, a_tok, bcB);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = launch_state_passing(U, ld, ang, nullptr, final_state, d.batch, d.nheads, nc, d.dstate, d.headdim,
                                  stream)) != cudaSuccess)
        return e;
    if (bh > 0 && nc > 0) {
        const size_t sc = smem_c(d);
        auto kc = chunk_scan_kernel<IO, R>;
        if ((e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc)) != cudaSuccess) return e;
        const int TT = kRowTile / R;
        const unsigned tiles = (unsigned)((d.chunk + TT - 1) / TT);
        kc<<<dim3((unsigned)bh, (unsigned)nc, tiles), kThreads, sc, stream>>>(
            (const IO*)x, (const IO*)B, (const IO*)C, dt, A, lambda, omega, U, (IO*)y, d.seqlen, (int)d.nheads,
            (int)d.headdim, (int)d.dstate, d.chunk, (int)nc, a_tok, bcB, bcC, (const IO*)gate);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename IO>
cudaError_t launch_io(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                      const float* A, const float* lambda, const float* omega, void* y, float* final_state,
                      void* workspace, int a_tok, const BcArgs& bcB, const BcArgs& bcC, const void* gate,
                      cudaStream_t stream) {
#define M3_SIMT_CASE(RR) \
    case RR: return launch_rt<IO, RR>(d, x, B, C, dt, A, lambda, omega, y, final_state, workspace, a_tok, bcB, bcC, \
                                      gate, stream);
    switch (d.R) {
        M3_SIMT_CASE(1)
        M3_SIMT_CASE(2)
        M3_SIMT_CASE(4)
        M3_SIMT_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef M3_SIMT_CASE
}

// Inverse RMS of every (token, rank) row of V over its N channels: 1 / sqrt(mean(v^2) + eps).
template <typename IO>
__global__ void __launch_bounds__(256) row_inv_rms_kernel(const IO* __restrict__ V, float* __restrict__ inv,
                                                          int64_t rows, int N, float eps) {
    for (int64_t row = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; row < rows;
         row += (int64_t)gridDim.x * blockDim.x) {
        float ss = 0.f;
        for (int n = 0; n < N; ++n) {
            const float v = ld_io(V, row * N + n);
            ss = fmaf(v, v, ss);
        }
        inv[row] = rsqrtf(ss / N + eps);
    }
}

// Delta = softplus(dt_raw + dt_bias[h]) and lambda = sigmoid(u) of every (batch, token, head).
__global__ void __launch_bounds__(256) prep_kernel(const float* __restrict__ dt_raw, const float* __restrict__ dt_bias,
                                                   const float* __restrict__ u, float* __restrict__ dt_out,
                                                   float* __restrict__ lam_out, int64_t n, int H) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float bias = dt_bias != nullptr ? dt_bias[i % H] : 0.f;
        dt_out[i] = softplus_f(dt_raw[i] + bias);
        lam_out[i] = sigmoid_f(u[i]);
    }
}

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

cudaError_t launch_prep_params(const float* dt_raw, const float* dt_bias, const float* u, float* dt_out,
                               float* lam_out, int64_t n, int H, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 148 * 16);
    prep_kernel<<<blocks, 256, 0, stream>>>(dt_raw, dt_bias, u, dt_out, lam_out, n, H);
    return cudaGetLastError();
}

bool simt_supported(const ScanDims& d) {
    if (!(d.R == 1 || d.R == 2 || d.R == 4 || d.R == 8)) return false;
    if (!(d.headdim == 16 || d.headdim == 32 || d.headdim == 64 || d.headdim == 128)) return false;
    if (d.dstate < 2 || d.dstate % 2 || d.dstate > 256) return false;
    if (d.dstate * d.headdim > kThreads * kMaxAcc) return false;
    if (d.chunk < 16 || d.chunk > 256 || d.chunk % 16) return false;
    return smem_a(d) <= 220 * 1024 && smem_c(d) <= 220 * 1024;
}

size_t simt_workspace_size(const ScanDims& d, bool prep) {
    const int64_t bh = d.batch * d.nheads;
    const int64_t nc = d.nchunks();
    const size_t base = sizeof(float) * (size_t)(bh * nc * (d.dstate * d.headdim + 1 + d.dstate / 2));
    if (!prep) return base;
    // Delta, lambda per (batch, token, head); inverse RMS of B and C per (batch, token, head, rank)
    const size_t n = (size_t)(d.batch * d.seqlen * d.nheads);
    return al256(base) + 2 * al256(n * sizeof(float)) + 2 * al256(n * (size_t)d.R * sizeof(float));
}

cudaError_t launch_scan_simt(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                             const float* A, const float* lambda, const float* omega, void* y,
                             float* final_state, void* workspace, const Prep& prep, cudaStream_t stream) {
    BcArgs bcB{}, bcC{};
    if (prep.on) {
        // Delta, lambda of every token (and the inverse RMS of every B / C row) into the tail of
        // the workspace, then the same kernels with one decay generator per token
        const int64_t n = d.batch * d.seqlen * d.nheads, rows = n * d.R;
        uint8_t* tail = static_cast<uint8_t*>(workspace) + al256(simt_workspace_size(d, false));
        float* dt_eff = reinterpret_cast<float*>(tail);
        float* lam_eff = reinterpret_cast<float*>(tail + al256((size_t)n * sizeof(float)));
        float* invB = reinterpret_cast<float*>(tail + 2 * al256((size_t)n * sizeof(float)));
        float* invC = reinterpret_cast<float*>(tail + 2 * al256((size_t)n * sizeof(float)) +
                                               al256((size_t)rows * sizeof(float)));
        cudaError_t e;
        if (n > 0) {
            const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 148 * 16);
            prep_kernel<<<blocks, 256, 0, stream>>>(dt, prep.dt_bias, lambda, dt_eff, lam_eff, n, (int)d.nheads);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            if (prep.bc_norm) {
                const unsigned rb = (unsigned)std::min<int64_t>((rows + 255) / 256, 148 * 16);
                if (d.io == M3_DTYPE_BF16) {
                    row_inv_rms_kernel<<<rb, 256, 0, stream>>>((const __nv_bfloat16*)B, invB, rows, (int)d.dstate, prep.bc_eps);
                    row_inv_rms_kernel<<<rb, 256, 0, stream>>>((const __nv_bfloat16*)C, invC, rows, (int)d.dstate, prep.bc_eps);
                } else {
                    row_inv_rms_kernel<<<rb, 256, 0, stream>>>((const float*)B, invB, rows, (int)d.dstate, prep.bc_eps);
                    row_inv_rms_kernel<<<rb, 256, 0, stream>>>((const float*)C, invC, rows, (int)d.dstate, prep.bc_eps);
                }
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
            }
        }
        dt = dt_eff;
        lambda = lam_eff;
        if (prep.bc()) {
            const int norm = prep.bc_norm ? 1 : 0;
            bcB = BcArgs{1, norm, invB, prep.B_gain, prep.B_bias};
            bcC = BcArgs{1, norm, invC, prep.C_gain, prep.C_bias};
        }
    }
    const int a_tok = prep.on ? 1 : 0;
    if (d.io == M3_DTYPE_BF16)
        return launch_io<__nv_bfloat16>(d, x, B, C, dt, A, lambda, omega, y, final_state, workspace, a_tok, bcB, bcC,
                                        prep.on ? prep.z : nullptr, stream);
    return launch_io<float>(d, x, B, C, dt, A, lambda, omega, y, final_state, workspace, a_tok, bcB, bcC,
                            prep.on ? prep.z : nullptr, stream);
}

}  // namespace m3
