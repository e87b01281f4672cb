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
// One CTA (at most 256 threads) owns one (batch, head).  Thread (g, c4)
// handles state pairs j = g, g + G, ... (rows 2j, 2j+1) for float4 column c4,
// in slabs of four pairs whose loads are issued together (the first slab
// before anything else).  B_t, B_{t-1}, C_t are staged in shared
// memory pair-major ([j][r] float2) and X_t, X_{t-1} row-major, so that a
// pair costs a handful of vector shared-memory loads for its 24R
// multiply-adds.  The readout's sum over N is a warp-shuffle reduction over
// the pair groups of a warp followed by a shared-memory sum over warps.
//
// Two kernels share that arithmetic:
//   decode_stream_kernel  persistent CTAs (two per SM) walk the (batch, head)
//                         units; each unit's state and step inputs are
//                         brought into shared memory by bulk asynchronous
//                         copies (cp.async.bulk, mbarrier completion) two or
//                         three units ahead, so HBM reads overlap the
//                         arithmetic of earlier units.  Used when every per-unit block is a
//                         multiple of 16 bytes (N % 8 == 0 and the io rows
//                         16-byte sized).
//   decode_kernel         one CTA per unit, state loaded straight into
//                         registers; any other supported shape.
#include "m3_common.cuh"
#include "tc_ptx.cuh"

namespace m3 {
namespace {

constexpr int kMaxUnits = 4;   // state pairs per thread

__device__ __forceinline__ float4 fma4(float a, float4 x, float4 y) {
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

#ifndef M3_DECODE_OCC_R4
#define M3_DECODE_OCC_R4 2
#endif
template <int R>
struct DecodeOcc {   // resident CTAs per SM the register budget is sized for (256-thread CTAs)
    static constexpr int value = R == 1 ? 4 : (R == 2 ? 3 : (R == 4 ? M3_DECODE_OCC_R4 : 2));
};

// The pre-activation options as a kernel parameter: the Prep descriptor for the
// *_prep entry point, an empty struct for the plain kernels (whose parameter
// block, and so their code, then stays as it is).
template <bool ON>
struct DecodeExt {
    Prep p;
};
template <>
struct DecodeExt<false> {};

// Delta, lambda and A of unit bh = batch * H + h: as given (A per head), or from the
// pre-activations of the *_prep entry points (A per unit).
template <bool PREP>
__device__ __forceinline__ void unit_params(const float* dt_t, const float* lam_t, const float* A,
                                            const DecodeExt<PREP>& ext, int64_t bh, int H, float& d, float& l,
                                            float& a) {
    if constexpr (PREP) {
        d = softplus_f(dt_t[bh] + (ext.p.dt_bias != nullptr ? ext.p.dt_bias[bh % H] : 0.f));
        l = sigmoid_f(lam_t[bh]);
        a = A[bh];
    } else {
        d = dt_t[bh];
        l = lam_t[bh];
        a = A[bh % H];
    }
}

// The B / C normalisation and channel biases of the pre-activation entry point,
// in place on the staged rows (float pairs laid out [N/2][R]) of B_t, C_t and
// the cached B_{t-1}: v / sqrt(mean(v^2) + eps) * gain + bias[h, r, :].
// Block-wide; the caller synchronises before and after.
__device__ void bc_rows(float* sB2f, float* sC2f, float* sBp2f, int R, int N, int h, const Prep& p) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int rows = 3 * R;   // B_t, C_t, B_{t-1}
    auto row_ptrs = [&](int row, float*& base, const float*& g, const float*& bb, int& r) {
        const int k = row / R;
        r = row % R;
        base = k == 0 ? sB2f : (k == 1 ? sC2f : sBp2f);
        g = k == 1 ? p.C_gain : p.B_gain;
        bb = k == 1 ? p.C_bias : p.B_bias;
    };
    auto at = [&](float* base, int r, int n) { return base + ((n >> 1) * R + r) * 2 + (n & 1); };
    auto apply = [&](float* base, const float* g, const float* bb, int r, int n0, int step, float sc) {
        for (int n = n0; n < N; n += step) {
            float* q = at(base, r, n);
            float v = *q;
            if (p.bc_norm) v *= sc * (g != nullptr ? g[n] : 1.f);
            if (bb != nullptr) v += bb[((int64_t)h * R + r) * N + n];
            *q = v;
        }
    };
    if ((nt & 31) == 0) {   // one warp per row
        const int warp = tid >> 5, lane = tid & 31, nw = nt >> 5;
        for (int row = warp; row < rows; row += nw) {
            float* base;
            const float *g, *bb;
            int r;
            row_ptrs(row, base, g, bb, r);
            float sc = 1.f;
            if (p.bc_norm) {
                float ss = 0.f;
                for (int n = lane; n < N; n += 32) {
                    const float v = *at(base, r, n);
                    ss = fmaf(v, v, ss);
                }
                sc = rsqrtf(warp_sum(ss) / N + p.bc_eps);
            }
            apply(base, g, bb, r, lane, 32, sc);
        }
    } else {                // small blocks: one thread per row
        for (int row = tid; row < rows; row += nt) {
            float* base;
            const float *g, *bb;
            int r;
            row_ptrs(row, base, g, bb, r);
            float sc = 1.f;
            if (p.bc_norm) {
                float ss = 0.f;
                for (int n = 0; n < N; ++n) {
                    const float v = *at(base, r, n);
                    ss = fmaf(v, v, ss);
                }
                sc = rsqrtf(ss / N + p.bc_eps);
            }
            apply(base, g, bb, r, 0, 1, sc);
        }
    }
}

template <typename IO, int R, bool PREP>
__global__ void __launch_bounds__(256, DecodeOcc<R>::value) decode_kernel(
    float* __restrict__ state, const IO* __restrict__ x_t, const IO* __restrict__ B_t,
    IO* __restrict__ cache, const IO* __restrict__ C_t, const float* __restrict__ dt_t,
    const float* __restrict__ A, const float* __restrict__ lam_t, const float* __restrict__ omega_t,
    IO* __restrict__ y_t, int H, int P, int N, int G, const DecodeExt<PREP> ext) {
    extern __shared__ __align__(16) float sm[];
    const int64_t bh = blockIdx.x;
    const int P4 = P >> 2, NP2 = N >> 1;
    const int tid = threadIdx.x, nt = blockDim.x;

    float2* sB2 = reinterpret_cast<float2*>(sm);     // [N/2][R]  B_t pairs
    float2* sBp2 = sB2 + NP2 * R;                    // [N/2][R]  B_{t-1} pairs
    float2* sC2 = sBp2 + NP2 * R;                    // [N/2][R]  C_t pairs
    float2* sCS = sC2 + NP2 * R;                     // [N/2]     (cos, sin) of phi_t
    float* sX = reinterpret_cast<float*>(sCS + NP2); // [R][P]    X_t
    float* sXp = sX + R * P;                         // [R][P]    X_{t-1}
    float* sRed = sXp + R * P;                       // [rows][R*P] readout partials

    // Issue the first slab of state loads before anything else: they are the
    // bytes that matter.  Slab s covers pairs j = g + (s*kMaxUnits + k)*G.
    const int c4 = tid % P4, g = tid / P4;
    float4* st4 = reinterpret_cast<float4*>(state + bh * (int64_t)N * P);
    float4 h0[kMaxUnits], h1[kMaxUnits];
    auto load_slab = [&](int s0) {
#pragma unroll
        for (int k = 0; k < kMaxUnits; ++k) {
            const int j = g + (s0 + k) * G;
            if (j < NP2) {
                h0[k] = st4[(2 * j) * P4 + c4];
                h1[k] = st4[(2 * j + 1) * P4 + c4];
            }
        }
    };
    load_slab(0);

    float d, l, a;
    unit_params<PREP>(dt_t, lam_t, A, ext, bh, H, d, l, a);
    const float alpha = expf(d * a);
    const float beta = (1.0f - l) * d * alpha;
    const float gamma = l * d;

    const IO* xb = x_t + bh * R * P;
    const IO* Bb = B_t + bh * R * N;
    const IO* Cb = C_t + bh * R * N;
    IO* cb = cache + bh * (int64_t)R * (N + P);

    float* sB2f = reinterpret_cast<float*>(sB2);
    float* sBp2f = reinterpret_cast<float*>(sBp2);
    float* sC2f = reinterpret_cast<float*>(sC2);
    for (int i = tid; i < R * N; i += nt) {
        const int r = i / N, n = i % N;
        const int o = ((n >> 1) * R + r) * 2 + (n & 1);
        sB2f[o] = ld_io(Bb, i);
        sC2f[o] = ld_io(Cb, i);
        sBp2f[o] = ld_io(cb, i);
    }
    for (int i = tid; i < R * P; i += nt) {
        sX[i] = ld_io(xb, i);
        sXp[i] = ld_io(cb, R * N + i);
    }
    for (int j = tid; j < NP2; j += nt) {
        float sn, cs;
        sincosf(d * omega_t[bh * NP2 + j], &sn, &cs);
        sCS[j] = make_float2(cs, sn);
    }
    __syncthreads();
    if constexpr (PREP) {
        if (ext.p.bc()) {
            bc_rows(sB2f, sC2f, sBp2f, R, N, (int)(bh % H), ext.p);
            __syncthreads();
        }
    }
    // The old cache is in shared memory now: replace it with this token's factors.
    for (int i = tid; i < R * N; i += nt) cb[i] = Bb[i];
    for (int i = tid; i < R * P; i += nt) cb[R * N + i] = xb[i];

    const float4* sX4 = reinterpret_cast<const float4*>(sX);
    const float4* sXp4 = reinterpret_cast<const float4*>(sXp);
    float4 acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);

    const int slabs = (NP2 + G * kMaxUnits - 1) / (G * kMaxUnits);
    for (int sl = 0; sl < slabs; ++sl) {
        if (sl > 0) load_slab(sl * kMaxUnits);
#pragma unroll
        for (int k = 0; k < kMaxUnits; ++k) {
            const int j = g + (sl * kMaxUnits + k) * G;
            if (j < NP2) {
                const float2 cs = sCS[j];
                // u = alpha h + beta v_{t-1}, v_{t-1} = B_{t-1} X_{t-1}^T (rows 2j, 2j+1)
                float4 w0 = make_float4(0.f, 0.f, 0.f, 0.f), w1 = w0;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float2 bp = sBp2[j * R + r];
                    const float4 xp = sXp4[r * P4 + c4];
                    w0 = fma4(bp.x, xp, w0);
                    w1 = fma4(bp.y, xp, w1);
                }
                const float4 u0 = fma4(alpha, h0[k], make_float4(beta * w0.x, beta * w0.y, beta * w0.z, beta * w0.w));
                const float4 u1 = fma4(alpha, h1[k], make_float4(beta * w1.x, beta * w1.y, beta * w1.z, beta * w1.w));
                // h' = R(phi) u + gamma v_t, v_t = B_t X_t^T
                float4 o0, o1;
                rot2(cs.x, cs.y, u0.x, u1.x, o0.x, o1.x);
                rot2(cs.x, cs.y, u0.y, u1.y, o0.y, o1.y);
                rot2(cs.x, cs.y, u0.z, u1.z, o0.z, o1.z);
                rot2(cs.x, cs.y, u0.w, u1.w, o0.w, o1.w);
                float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float2 bc = sB2[j * R + r];
                    const float4 xc = sX4[r * P4 + c4];
                    v0 = fma4(bc.x, xc, v0);
                    v1 = fma4(bc.y, xc, v1);
                }
                o0 = fma4(gamma, v0, o0);
                o1 = fma4(gamma, v1, o1);
                st4[(2 * j) * P4 + c4] = o0;
                st4[(2 * j + 1) * P4 + c4] = o1;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float2 cc = sC2[j * R + r];
                    acc[r] = fma4(cc.x, o0, fma4(cc.y, o1, acc[r]));
                }
            }
        }
    }

    // Readout: sum the G pair-group partials of each (r, p).  Pair groups that
    // share a full warp (P4 a power of two below 32) are combined with shuffles
    // first.
    int gpw = 1;
    if (P4 < 32 && (P4 & (P4 - 1)) == 0 && nt % 32 == 0) {
        gpw = 32 / P4;
        for (int o = P4; o < 32; o <<= 1) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                acc[r].x += __shfl_xor_sync(0xffffffffu, acc[r].x, o);
                acc[r].y += __shfl_xor_sync(0xffffffffu, acc[r].y, o);
                acc[r].z += __shfl_xor_sync(0xffffffffu, acc[r].z, o);
                acc[r].w += __shfl_xor_sync(0xffffffffu, acc[r].w, o);
            }
        }
    }
    const int rows = (G + gpw - 1) / gpw;
    if (g % gpw == 0) {
        float4* red4 = reinterpret_cast<float4*>(sRed) + (g / gpw) * (R * P4);
#pragma unroll
        for (int r = 0; r < R; ++r) red4[r * P4 + c4] = acc[r];
    }
    __syncthreads();
    IO* yb = y_t + bh * R * P;
    const IO* zb = nullptr;
    if constexpr (PREP) zb = ext.p.z != nullptr ? static_cast<const IO*>(ext.p.z) + bh * R * P : nullptr;
    for (int o = tid; o < R * P; o += nt) {
        float s = 0.f;
        for (int gg = 0; gg < rows; ++gg) s += sRed[gg * (R * P) + o];
        st_io(yb, o, zb != nullptr ? s * silu_f(ld_io(zb, o)) : s);   // output gate
    }
}

// ---------------------------------------------------------------------------
// Streaming variant.  Per-unit slot in shared memory (16-byte aligned pieces):
//   state [N*P] fp32 | B_t [R*N] | C_t [R*N] | x_t [R*P] | cache [R*(N+P)] (io) | omega [N/2] fp32
constexpr int kMaxSlots = 3;   // units in flight per CTA (3, or 2 when 3 do not fit)
constexpr uint64_t kStreamWaitNs = 2000000000ull;   // 2 s per wait, then give up

// Sticky error word of the decode kernels (they have no workspace): set to
// M3_ERR_TIMEOUT when a bounded wait gives up; read by m3_device_status.
__device__ int g_decode_status = 0;

__host__ __device__ inline int round16(int v) { return (v + 15) & ~15; }

struct StreamLayout {
    int st, b, c, x, ca, om, slot, tx;
};

__host__ __device__ inline StreamLayout stream_layout(int N, int P, int R, int es) {
    StreamLayout L;
    L.st = 0;
    L.b = L.st + N * P * 4;
    L.c = L.b + round16(R * N * es);
    L.x = L.c + round16(R * N * es);
    L.ca = L.x + round16(R * P * es);
    L.om = L.ca + round16(R * (N + P) * es);
    L.slot = (L.om + round16((N / 2) * 4) + 127) & ~127;
    L.tx = N * P * 4 + 2 * R * N * es + R * P * es + R * (N + P) * es + (N / 2) * 4;
    return L;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            tc::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}

template <typename IO, int R, bool PREP>
__global__ void __launch_bounds__(256, 2) decode_stream_kernel(
    float* __restrict__ state, const IO* __restrict__ x_t, const IO* __restrict__ B_t,
    IO* __restrict__ cache, const IO* __restrict__ C_t, const float* __restrict__ dt_t,
    const float* __restrict__ A, const float* __restrict__ lam_t, const float* __restrict__ omega_t,
    IO* __restrict__ y_t, int H, int P, int N, int G, int64_t units, int nslots, const DecodeExt<PREP> ext) {
    extern __shared__ __align__(128) uint8_t smraw[];
    const int P4 = P >> 2, NP2 = N >> 1;
    const int tid = threadIdx.x, nt = blockDim.x;
    const StreamLayout L = stream_layout(N, P, R, (int)sizeof(IO));

    uint8_t* slots = smraw;
    float2* sB2 = reinterpret_cast<float2*>(smraw + nslots * L.slot);
    float2* sBp2 = sB2 + NP2 * R;
    float2* sC2 = sBp2 + NP2 * R;
    float2* sCS = sC2 + NP2 * R;
    float* sX = reinterpret_cast<float*>(sCS + NP2);
    float* sXp = sX + R * P;
    float* sRed = sXp + R * P;
    const int gpw = (P4 < 32 && (P4 & (P4 - 1)) == 0 && nt % 32 == 0) ? 32 / P4 : 1;
    const int rows = (G + gpw - 1) / gpw;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRed + rows * R * P + 2);   // 8-byte aligned
    int* sFail = reinterpret_cast<int*>(bars + kMaxSlots);

    const int64_t first = blockIdx.x, step = gridDim.x;
    auto issue = [&](int64_t u, int slot) {
        uint8_t* sl = slots + slot * L.slot;
        uint64_t* bar = &bars[slot];
        tc::mbar_arrive_expect_tx(bar, (uint32_t)L.tx);
        const int es = (int)sizeof(IO);
        bulk_g2s(sl + L.st, state + u * (int64_t)N * P, (uint32_t)(N * P * 4), bar);
        bulk_g2s(sl + L.b, B_t + u * R * N, (uint32_t)(R * N * es), bar);
        bulk_g2s(sl + L.c, C_t + u * R * N, (uint32_t)(R * N * es), bar);
        bulk_g2s(sl + L.x, x_t + u * R * P, (uint32_t)(R * P * es), bar);
        bulk_g2s(sl + L.ca, cache + u * (int64_t)R * (N + P), (uint32_t)(R * (N + P) * es), bar);
        bulk_g2s(sl + L.om, omega_t + u * NP2, (uint32_t)(NP2 * 4), bar);
    };
    if (tid == 0) {
        for (int s = 0; s < nslots; ++s) tc::mbar_init(&bars[s], 1);
        *sFail = 0;
        tc::fence_mbar_init();
        for (int s = 0; s < nslots; ++s) {
            const int64_t u = first + s * step;
            if (u < units) issue(u, s);
        }
    }
    __syncthreads();

    const int c4 = tid % P4, g = tid / P4;
    // scalars of the first unit; later units' are prefetched one unit ahead
    float d_n = 0.f, l_n = 0.f, a_n = 0.f;
    if (first < units) unit_params<PREP>(dt_t, lam_t, A, ext, first, H, d_n, l_n, a_n);
    int it = 0;
    for (int64_t u = first; u < units; u += step, ++it) {
        const int slot = it % nslots;
        const uint32_t parity = (uint32_t)((it / nslots) & 1);
        const float d = d_n, l = l_n, a = a_n;
        const int64_t un = u + step;
        if (un < units) unit_params<PREP>(dt_t, lam_t, A, ext, un, H, d_n, l_n, a_n);
        if (!tc::mbar_wait(&bars[slot], parity, kStreamWaitNs)) *sFail = 1;
        __syncthreads();
        if (*sFail) break;
        const uint8_t* sl = slots + slot * L.slot;
        const IO* sBt = reinterpret_cast<const IO*>(sl + L.b);
        const IO* sCt = reinterpret_cast<const IO*>(sl + L.c);
        const IO* sXt = reinterpret_cast<const IO*>(sl + L.x);
        const IO* sCa = reinterpret_cast<const IO*>(sl + L.ca);
        const float* sOm = reinterpret_cast<const float*>(sl + L.om);
        const float4* sSt4 = reinterpret_cast<const float4*>(sl + L.st);

        const float alpha = expf(d * a);
        const float beta = (1.0f - l) * d * alpha;
        const float gamma = l * d;

        float* sB2f = reinterpret_cast<float*>(sB2);
        float* sBp2f = reinterpret_cast<float*>(sBp2);
        float* sC2f = reinterpret_cast<float*>(sC2);
        for (int i = tid; i < R * N; i += nt) {
            const int r = i / N, n = i % N;
            const int o = ((n >> 1) * R + r) * 2 + (n & 1);
            sB2f[o] = ld_io(sBt, i);
            sC2f[o] = ld_io(sCt, i);
            sBp2f[o] = ld_io(sCa, i);
        }
        for (int i = tid; i < R * P; i += nt) {
            sX[i] = ld_io(sXt, i);
            sXp[i] = ld_io(sCa, R * N + i);
        }
        for (int j = tid; j < NP2; j += nt) {
            float sn, cs;
            sincosf(d * sOm[j], &sn, &cs);
            sCS[j] = make_float2(cs, sn);
        }
        __syncthreads();
        if constexpr (PREP) {
            if (ext.p.bc()) {
                bc_rows(sB2f, sC2f, sBp2f, R, N, (int)(u % H), ext.p);
                __syncthreads();
            }
        }
        // new delayed-write cache: this token's B_t then X_t (raw io values)
        IO* cb = cache + u * (int64_t)R * (N + P);
        for (int i = tid; i < R * N; i += nt) cb[i] = sBt[i];
        for (int i = tid; i < R * P; i += nt) cb[R * N + i] = sXt[i];

        const float4* sX4 = reinterpret_cast<const float4*>(sX);
        const float4* sXp4 = reinterpret_cast<const float4*>(sXp);
        float4* st4 = reinterpret_cast<float4*>(state + u * (int64_t)N * P);
        float4 acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = g; j < NP2; j += G) {
            const float4 h0 = sSt4[(2 * j) * P4 + c4], h1 = sSt4[(2 * j + 1) * P4 + c4];
            const float2 cs = sCS[j];
            float4 w0 = make_float4(0.f, 0.f, 0.f, 0.f), w1 = w0;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 bp = sBp2[j * R + r];
                const float4 xp = sXp4[r * P4 + c4];
                w0 = fma4(bp.x, xp, w0);
                w1 = fma4(bp.y, xp, w1);
            }
            const float4 u0 = fma4(alpha, h0, make_float4(beta * w0.x, beta * w0.y, beta * w0.z, beta * w0.w));
            const float4 u1 = fma4(alpha, h1, make_float4(beta * w1.x, beta * w1.y, beta * w1.z, beta * w1.w));
            float4 o0, o1;
            rot2(cs.x, cs.y, u0.x, u1.x, o0.x, o1.x);
            rot2(cs.x, cs.y, u0.y, u1.y, o0.y, o1.y);
            rot2(cs.x, cs.y, u0.z, u1.z, o0.z, o1.z);
            rot2(cs.x, cs.y, u0.w, u1.w, o0.w, o1.w);
            float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 bc = sB2[j * R + r];
                const float4 xc = sX4[r * P4 + c4];
                v0 = fma4(bc.x, xc, v0);
                v1 = fma4(bc.y, xc, v1);
            }
            o0 = fma4(gamma, v0, o0);
            o1 = fma4(gamma, v1, o1);
            st4[(2 * j) * P4 + c4] = o0;
            st4[(2 * j + 1) * P4 + c4] = o1;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 cc = sC2[j * R + r];
                acc[r] = fma4(cc.x, o0, fma4(cc.y, o1, acc[r]));
            }
        }
        if (gpw > 1) {
            for (int o = P4; o < 32; o <<= 1) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    acc[r].x += __shfl_xor_sync(0xffffffffu, acc[r].x, o);
                    acc[r].y += __shfl_xor_sync(0xffffffffu, acc[r].y, o);
                    acc[r].z += __shfl_xor_sync(0xffffffffu, acc[r].z, o);
                    acc[r].w += __shfl_xor_sync(0xffffffffu, acc[r].w, o);
                }
            }
        }
        if (g % gpw == 0) {
            float4* red4 = reinterpret_cast<float4*>(sRed) + (g / gpw) * (R * P4);
#pragma unroll
            for (int r = 0; r < R; ++r) red4[r * P4 + c4] = acc[r];
        }
        __syncthreads();   // readout partials written; every read of this slot done
        if (tid == 0) {
            const int64_t u3 = u + (int64_t)nslots * step;
            if (u3 < units) issue(u3, slot);
        }
        IO* yb = y_t + u * R * P;
        const IO* zb = nullptr;
        if constexpr (PREP) zb = ext.p.z != nullptr ? static_cast<const IO*>(ext.p.z) + u * R * P : nullptr;
        for (int o = tid; o < R * P; o += nt) {
            float s = 0.f;
            for (int gg = 0; gg < rows; ++gg) s += sRed[gg * (R * P) + o];
            st_io(yb, o, zb != nullptr ? s * silu_f(ld_io(zb, o)) : s);   // output gate
        }
        __syncthreads();   // sRed and the staged operands are free for the next unit
    }
    if (*sFail && tid == 0) {
        atomicExch(&g_decode_status, (int)M3_ERR_TIMEOUT);
        // let the copies still in flight land before the CTA's shared memory goes away (bounded)
        int it2 = it;
        for (int64_t u = first + (int64_t)it * step; u < units && it2 < it + nslots; u += step, ++it2)
            (void)tc::mbar_wait(&bars[it2 % nslots], (uint32_t)((it2 / nslots) & 1), kStreamWaitNs);
    }
}

bool stream_ok(int64_t P, int64_t N, int R, int es) {
    if (N % 8) return false;
    if ((R * N * es) % 16 || (R * P * es) % 16 || (R * (N + P) * es) % 16) return false;
    return true;
}

size_t stream_smem(int64_t P, int64_t N, int R, int es, int G, int nslots) {
    const StreamLayout L = stream_layout((int)N, (int)P, R, es);
    const int P4 = (int)(P / 4);
    const int gpw = (P4 < 32 && (P4 & (P4 - 1)) == 0 && (G * P4) % 32 == 0) ? 32 / P4 : 1;
    const int rows = (G + gpw - 1) / gpw;
    const size_t fixed = sizeof(float) * (size_t)(3 * R * N + N + 2 * R * P + (size_t)rows * R * P + 2);
    return (size_t)nslots * L.slot + fixed + 8 * kMaxSlots + 16;
}

int device_sms() {
    static int sms[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    if (sms[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        sms[dev] = v;
    }
    return sms[dev];
}

struct DecodeShape {
    int G, threads;
    size_t smem;
};

DecodeShape decode_shape(int64_t P, int64_t N, int R) {
    DecodeShape s{};
    const int P4 = (int)(P / 4), NP2 = (int)(N / 2);
    int G = 256 / P4;
    if (G > NP2) G = NP2;
    if (G < 1) G = 1;
    s.G = G;
    s.threads = G * P4;
    const int gpw = P4 < 32 ? 32 / P4 : 1;
    const int rows = (G + gpw - 1) / gpw;
    s.smem = sizeof(float) * (size_t)(3 * R * N + N + 2 * R * P + (size_t)rows * R * P);
    return s;
}

template <typename IO, int R, bool PREP>
cudaError_t launch_p(float* state, const void* x_t, const void* B_t, void* cache, const void* C_t,
                     const float* dt_t, const float* A, const float* lambda_t, const float* omega_t, void* y_t,
                     int64_t batch, int64_t nheads, int64_t P, int64_t N, const DecodeExt<PREP>& ext,
                     cudaStream_t stream) {
    const DecodeShape s = decode_shape(P, N, R);
    const int64_t units = batch * nheads;
    const int es = (int)sizeof(IO);
    if (stream_ok(P, N, R, es)) {
        // two CTAs per SM: at most ~110 KB of shared memory each
        int nslots = kMaxSlots;
        size_t smem = stream_smem(P, N, R, es, s.G, nslots);
        if (smem > 110 * 1024) smem = stream_smem(P, N, R, es, s.G, nslots = 2);
        if (smem <= 110 * 1024) {
            auto kern = decode_stream_kernel<IO, R, PREP>;
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            int64_t grid = 2 * (int64_t)device_sms();
            if (grid > units) grid = units;
            kern<<<(unsigned)grid, s.threads, smem, stream>>>(
                state, (const IO*)x_t, (const IO*)B_t, (IO*)cache, (const IO*)C_t, dt_t, A, lambda_t, omega_t,
                (IO*)y_t, (int)nheads, (int)P, (int)N, s.G, units, nslots, ext);
            return cudaGetLastError();
        }
    }
    auto kern = decode_kernel<IO, R, PREP>;
    if (s.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s.smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<(unsigned)units, s.threads, s.smem, stream>>>(
        state, (const IO*)x_t, (const IO*)B_t, (IO*)cache, (const IO*)C_t, dt_t, A, lambda_t, omega_t, (IO*)y_t,
        (int)nheads, (int)P, (int)N, s.G, ext);
    return cudaGetLastError();
}

template <typename IO, int R>
cudaError_t launch_t(float* state, const void* x_t, const void* B_t, void* cache, const void* C_t,
                     const float* dt_t, const float* A, const float* lambda_t, const float* omega_t, void* y_t,
                     int64_t batch, int64_t nheads, int64_t P, int64_t N, const Prep& prep, cudaStream_t stream) {
    if (prep.on)
        return launch_p<IO, R, true>(state, x_t, B_t, cache, C_t, dt_t, A, lambda_t, omega_t, y_t, batch, nheads, P,
                                     N, DecodeExt<true>{prep}, stream);
    return launch_p<IO, R, false>(state, x_t, B_t, cache, C_t, dt_t, A, lambda_t, omega_t, y_t, batch, nheads, P, N,
                                  DecodeExt<false>{}, stream);
}

template <typename IO>
cudaError_t launch_io(int R, float* state, const void* x_t, const void* B_t, void* cache, const void* C_t,
                      const float* dt_t, const float* A, const float* lambda_t, const float* omega_t, void* y_t,
                      int64_t batch, int64_t nheads, int64_t P, int64_t N, const Prep& prep, cudaStream_t stream) {
#define M3_DEC_CASE(RR) \
    case RR: return launch_t<IO, RR>(state, x_t, B_t, cache, C_t, dt_t, A, lambda_t, omega_t, y_t, batch, nheads, P, N, prep, stream);
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
    if (s.threads > 256) return false;
    return s.smem <= 200 * 1024;
}

cudaError_t launch_decode(float* state, const void* x_t, const void* B_t, void* cache, const void* C_t,
                          const float* dt_t, const float* A, const float* lambda_t, const float* omega_t,
                          void* y_t, int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate, int R,
                          int io, const Prep& prep, cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    if (io == M3_DTYPE_BF16)
        return launch_io<__nv_bfloat16>(R, state, x_t, B_t, cache, C_t, dt_t, A, lambda_t, omega_t, y_t, batch,
                                        nheads, headdim, dstate, prep, stream);
    return launch_io<float>(R, state, x_t, B_t, cache, C_t, dt_t, A, lambda_t, omega_t, y_t, batch, nheads,
                            headdim, dstate, prep, stream);
}

int decode_device_status(int clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(int)) != cudaSuccess) return M3_ERR_CUDA;
    if (clear && v != 0) {
        const int z = 0;
        if (cudaMemcpyToSymbol(g_decode_status, &z, sizeof(int)) != cudaSuccess) return M3_ERR_CUDA;
    }
    return v;
}

}  // namespace m3
