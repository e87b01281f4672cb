// Tensor-core chunked prefill (bf16 io) for sm_103a: tcgen05 MMAs with TMEM
// accumulators, operands staged by TMA in 128-byte-swizzled shared memory.
//
// The chunked algorithm of "Mamba-3: Improved Sequence Modeling using State
// Space Principles" (section 3.3; decay x two-band mask of section 3.1.3 /
// Eq. 7; rotary form of Propositions 3-4), fused into one kernel: one CTA owns
// one (batch, head) sequence and walks its chunks in order, carrying the
// fp32 N x P state in TMEM, so no chunk state ever goes to HBM.  Per chunk
// c = tokens [c0, c0+Q) (rows ordered (token, rank), QR = Q*R <= 128):
//
//   coefficients   l_t = dt_t A, cum_t = sum_{k<=t} l_k (chunk-local),
//                  gamma_t = lambda_t dt_t, w_s = gamma_s + (1-lambda_{s+1}) dt_{s+1}
//   rotation       Psi_t = sum_{k<=t} dt_k omega_k (chunk-local),
//                  B~ = R(-Psi) B, C~ = R(-Psi) C, in place in shared memory
//   MMA1           S = C~ B~^T                                (TMEM, fp32)
//   mask           SL_ts = S_ts exp(cum_t - cum_s) (t == s ? gamma_t : w_s), s <= t
//   MMA2, MMA4     Y = SL X + (exp(cum_t) C~) H_{c-1}          (TMEM, fp32)
//   MMA3           U = (exp(cum_end - cum_s) w_s B~)^T X        (TMEM, fp32)
//   state          H_c = R(Theta_c) (exp(cum_end) H_{c-1} + U),  Theta_c = Psi_end
//                  (U is in the chunk's rotating frame; the rotation commutes
//                  with the scalar decay, so one rotation serves both terms)
//
// H is the physical-frame state plus the pending delayed write of the
// chunk's last token (its w uses the next token's lambda, dt; zero past the
// end), so H after the last chunk is the true final state h_{T-1}.
//
// MMA operand layouts (all 128-byte swizzled, bf16):
//   C~, C~'  A, K-major  (rows (t,r), K = n)     B~  B, K-major (rows (s,r), K = n)
//   SL       A, K-major  (rows (t,r), K = (s,r')) X   B, MN-major (K = (s,r'), N = p)
//   Hb       B, MN-major (K = n, N = p)          B^  A, MN-major (M = n, K = (s,r'))
// When QR = 64 the MMAs still run with M = 128; rows 64..127 read the next
// 8 KB of shared memory (always inside this CTA's allocation) and their
// results are never read.
#include <cuda.h>

#include "m3_common.cuh"
#include "tc_ptx.cuh"

namespace m3 {
namespace {

using namespace tc;

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait, then give up with M3_ERR_TIMEOUT

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

template <int NS, int R, int Q>
struct Cfg {
    static constexpr int P = 64;                 // head dim (one 128-byte swizzle panel of bf16)
    static constexpr int QR = Q * R;             // rows of the chunk
    static constexpr int NPAN = NS / 64;         // 64-wide panels of B / C
    static constexpr int kThreads = 128;
    static_assert(QR == 64 || QR == 128, "chunk rows must be 64 or 128");
    static_assert(NS == 64 || NS == 128, "state size must be 64 or 128");
    static_assert(Q <= 128, "chunk too long");

    static constexpr int X_BYTES = QR * 128;
    static constexpr int BC_BYTES = NPAN * QR * 128;
    static constexpr int SC_BYTES = 16 * (Q + 1);          // dt / lambda box {4 heads, Q+1 tokens}
    static constexpr int OFF_C = 0;
    static constexpr int OFF_B = OFF_C + BC_BYTES;
    static constexpr int OFF_X = OFF_B + BC_BYTES;
    static constexpr int OFF_DT = OFF_X + X_BYTES;
    static constexpr int OFF_LAM = OFF_DT + align_up(SC_BYTES, 128);
    static constexpr int STAGE = align_up(OFF_LAM + align_up(SC_BYTES, 128), 1024);
    static constexpr int TX_BYTES = X_BYTES + 2 * BC_BYTES + 2 * SC_BYTES;

    static constexpr int OFF_SL = 2 * STAGE;
    static constexpr int SL_BYTES = (QR / 64) * QR * 128;
    static constexpr int OFF_HB = OFF_SL + SL_BYTES;
    static constexpr int HB_BYTES = NS * 128;
    static constexpr int OFF_SMALL = OFF_HB + HB_BYTES;
    // small arrays (floats): cum[Q], gam[Q], w[Q], warp sums[4], theta[NS/2]
    static constexpr int TG = kThreads / (NS / 8);          // token groups of the rotation phase
    static constexpr int TPG = Q / TG;                      // tokens per group
    static_assert(Q % TG == 0, "tokens must split evenly over token groups");
    // the rotation phase's partial angle sums [TG][NS/2] live in the SL buffer (free at that point)
    static_assert(TG * (NS / 2) * 4 <= SL_BYTES, "partial angle sums must fit in the SL buffer");
    static constexpr int SMALL_FLOATS = 3 * Q + 4 + NS / 2;
    static constexpr int OFF_BAR = align_up(OFF_SMALL + 4 * SMALL_FLOATS, 16);
    static constexpr int SMEM = OFF_BAR + 64 + 1024;        // barriers, tmem slot, alignment slack

    // TMEM columns
    static constexpr int T_S = 0;
    static constexpr int T_Y = QR;
    static constexpr int T_U = QR + P;
    static constexpr int T_H = QR + 2 * P;
    static constexpr int TMEM_COLS = (QR + 3 * P) <= 256 ? 256 : 512;
};

struct TcArgs {
    const float* A;
    const float* omega;
    __nv_bfloat16* y;
    float* final_state;
    int* status;
    int T, H, nc;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}

template <int NS, int R, int Q>
__global__ void __launch_bounds__(128, 2) scan_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                         const __grid_constant__ CUtensorMap tm_B,
                                                         const __grid_constant__ CUtensorMap tm_C,
                                                         const __grid_constant__ CUtensorMap tm_dt,
                                                         const __grid_constant__ CUtensorMap tm_lam, TcArgs args) {
    using K = Cfg<NS, R, Q>;
    constexpr int P = K::P, QR = K::QR, NP2 = NS / 2, NG = NS / 8, TG = K::TG, TPG = K::TPG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sCum = reinterpret_cast<float*>(sm + K::OFF_SMALL);
    float* sGam = sCum + Q;
    float* sW = sGam + Q;
    float* sWarp = sW + Q;
    float* sTheta = sWarp + 4;           // [NS/2]
    float* sPart = reinterpret_cast<float*>(sm + K::OFF_SL);   // [TG][NS/2], before SL is written
    uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + K::OFF_BAR);   // [2]
    uint64_t* bar_mma = bar_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
    int* sFail = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int b = bh / args.H, h = bh % args.H;
    const int T = args.T, nc = args.nc;
    const float a = args.A[h];

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(bar_mma, 1);
        *sFail = 0;
        fence_mbar_init();
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_C);
        prefetch_tensormap(&tm_dt);
        prefetch_tensormap(&tm_lam);
    }
    __syncthreads();
    if (warp == 0) {
        tmem_alloc(tmem_slot, K::TMEM_COLS);
        tmem_relinquish();
    }

    auto issue_loads = [&](int c, int s) {
        uint8_t* st = sm + s * K::STAGE;
        const int c0 = c * Q;
        mbar_arrive_expect_tx(&bar_full[s], K::TX_BYTES);
#pragma unroll
        for (int p = 0; p < K::NPAN; ++p) {
            tma_load_5d(st + K::OFF_C + p * QR * 128, &tm_C, &bar_full[s], 64 * p, 0, h, c0, b);
            tma_load_5d(st + K::OFF_B + p * QR * 128, &tm_B, &bar_full[s], 64 * p, 0, h, c0, b);
        }
        tma_load_5d(st + K::OFF_X, &tm_x, &bar_full[s], 0, 0, h, c0, b);
        tma_load_3d(st + K::OFF_DT, &tm_dt, &bar_full[s], h & ~3, c0, b);
        tma_load_3d(st + K::OFF_LAM, &tm_lam, &bar_full[s], h & ~3, c0, b);
    };
    // chunk whose loads are in flight into each stage (-1: none), for the bounded drain on failure
    int inflight[2] = {-1, -1};
    if (tid == 0) {
        if (nc > 0) issue_loads(0, 0);
        if (nc > 1) issue_loads(1, 1);
    }
    if (nc > 0) inflight[0] = 0;
    if (nc > 1) inflight[1] = 1;

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);

    // H_{-1} = 0
    if (tid < NS) {
        float z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
        for (int cc = 0; cc < P; cc += 16) tmem_st16(tlane + K::T_H + cc, z);
        tmem_st_wait();
    }

    // rotation-phase mapping: pair group jg (4 pairs = 16 bytes of a row), token group tg
    const int jg = tid % NG, tg = tid / NG;
    const int pan = jg / 8, cib = (jg % 8) * 16;     // panel and byte-in-row of my 16-byte piece
    const float* om_base = args.omega + ((int64_t)b * T * args.H + h) * NP2 + 4 * jg;
    const int64_t om_tok = (int64_t)args.H * NP2;
    float4 om[TPG];
    auto load_omega = [&](int c) {
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
            const int t = c * Q + tg * TPG + i;
            om[i] = t < T ? *reinterpret_cast<const float4*>(om_base + t * om_tok) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    if (nc > 0) load_omega(0);

    uint32_t mma_phase = 0;
    bool failed = false;
    for (int c = 0; c < nc; ++c) {
        const int s = c & 1;
        uint8_t* st = sm + s * K::STAGE;
        const float* sDt = reinterpret_cast<const float*>(st + K::OFF_DT);
        const float* sLam = reinterpret_cast<const float*>(st + K::OFF_LAM);
        if (!mbar_wait(&bar_full[s], (c >> 1) & 1, kWaitLimitNs)) *sFail = 1;
        __syncthreads();
        if (*sFail) { failed = true; break; }
        inflight[s] = -1;

        // ---- coefficients and chunk-local log-decay prefix
        const int hq = h & 3;
        {
            float ell = 0.f, gam = 0.f, wv = 0.f;
            if (tid < Q) {
                const float d = sDt[tid * 4 + hq], l = sLam[tid * 4 + hq];
                const float dn = sDt[(tid + 1) * 4 + hq], ln = sLam[(tid + 1) * 4 + hq];
                ell = d * a;
                gam = l * d;
                wv = gam + (1.f - ln) * dn;
            }
            float v = warp_inclusive_sum(ell);
            if (lane == 31) sWarp[warp] = v;
            __syncthreads();
            float off = 0.f;
            for (int i = 0; i < warp; ++i) off += sWarp[i];
            if (tid < Q) {
                sCum[tid] = v + off;
                sGam[tid] = gam;
                sW[tid] = wv;
            }
        }
        // ---- rotation angles: partial sums per token group
        float dtk[TPG];
        {
            float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < TPG; ++i) {
                const float d = sDt[(tg * TPG + i) * 4 + hq];
                dtk[i] = d;
                part.x = fmaf(d, om[i].x, part.x);
                part.y = fmaf(d, om[i].y, part.y);
                part.z = fmaf(d, om[i].z, part.z);
                part.w = fmaf(d, om[i].w, part.w);
            }
            *reinterpret_cast<float4*>(&sPart[tg * NP2 + 4 * jg]) = part;
        }
        __syncthreads();
        {
            float4 psi = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int g = 0; g < tg; ++g) {
                const float4 p4 = *reinterpret_cast<const float4*>(&sPart[g * NP2 + 4 * jg]);
                psi.x += p4.x; psi.y += p4.y; psi.z += p4.z; psi.w += p4.w;
            }
#pragma unroll
            for (int i = 0; i < TPG; ++i) {
                const int t = tg * TPG + i;
                psi.x = fmaf(dtk[i], om[i].x, psi.x);
                psi.y = fmaf(dtk[i], om[i].y, psi.y);
                psi.z = fmaf(dtk[i], om[i].z, psi.z);
                psi.w = fmaf(dtk[i], om[i].w, psi.w);
                float cs[4], sn[4];
                __sincosf(-psi.x, &sn[0], &cs[0]);
                __sincosf(-psi.y, &sn[1], &cs[1]);
                __sincosf(-psi.z, &sn[2], &cs[2]);
                __sincosf(-psi.w, &sn[3], &cs[3]);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int row = t * R + r;
                    const uint32_t off = pan * QR * 128 + sw128_offset(row, cib);
#pragma unroll
                    for (int m = 0; m < 2; ++m) {   // m = 0: C, m = 1: B
                        uint4* p = reinterpret_cast<uint4*>(st + (m == 0 ? K::OFF_C : K::OFF_B) + off);
                        uint4 v = *p;
                        uint32_t wv4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_bf16(wv4[e]);
                            float o0, o1;
                            rot2(cs[e], sn[e], f.x, f.y, o0, o1);
                            wv4[e] = pack_bf16(o0, o1);
                        }
                        *p = make_uint4(wv4[0], wv4[1], wv4[2], wv4[3]);
                    }
                }
            }
            if (tg == TG - 1) *reinterpret_cast<float4*>(&sTheta[4 * jg]) = psi;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- MMA1: S = C~ B~^T
        if (tid == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, QR, false, false);
            const uint32_t aC = smem_u32(st + K::OFF_C), aB = smem_u32(st + K::OFF_B);
#pragma unroll
            for (int kk = 0; kk < NS / 16; ++kk) {
                const uint32_t koff = (kk >> 2) * QR * 128 + (kk & 3) * 32;
                mma_bf16_ss(tmem + K::T_S, smem_desc(aC + koff, 16, 1024, kSwizzle128B),
                            smem_desc(aB + koff, 16, 1024, kSwizzle128B), idesc, kk > 0);
            }
            mma_commit(bar_mma);
        }
        // overlap: next chunk's omega, and H_{c-1} -> bf16 operand
        if (c + 1 < nc) load_omega(c + 1);
        if (tid < NS) {
            uint8_t* hb = sm + K::OFF_HB;
#pragma unroll
            for (int cc = 0; cc < P; cc += 16) {
                float v[16];
                tmem_ld16(tlane + K::T_H + cc, v);
                tmem_ld_wait();
#pragma unroll
                for (int q8 = 0; q8 < 2; ++q8) {
                    uint4 pk = make_uint4(pack_bf16(v[q8 * 8 + 0], v[q8 * 8 + 1]), pack_bf16(v[q8 * 8 + 2], v[q8 * 8 + 3]),
                                          pack_bf16(v[q8 * 8 + 4], v[q8 * 8 + 5]), pack_bf16(v[q8 * 8 + 6], v[q8 * 8 + 7]));
                    *reinterpret_cast<uint4*>(hb + sw128_offset(tid, (cc + q8 * 8) * 2)) = pk;
                }
            }
        }
        if (!mbar_wait(bar_mma, mma_phase, kWaitLimitNs)) *sFail = 1;
        mma_phase ^= 1;
        tc_fence_after();

        // ---- mask: SL = S o L (bf16, K-major rows (t,r))
        if (tid < QR) {
            const int t = tid / R;
            const float ct = sCum[t], gt = sGam[t];
            uint8_t* sl = sm + K::OFF_SL;
#pragma unroll
            for (int cc = 0; cc < QR; cc += 16) {
                float v[16];
                tmem_ld16(tlane + K::T_S + cc, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int sidx = (cc + i) / R;
                    float m = 0.f;
                    if (sidx < t) m = __expf(ct - sCum[sidx]) * sW[sidx];
                    else if (sidx == t) m = gt;
                    v[i] *= m;
                }
#pragma unroll
                for (int q8 = 0; q8 < 2; ++q8) {
                    const int col = cc + q8 * 8;
                    uint4 pk = make_uint4(pack_bf16(v[q8 * 8 + 0], v[q8 * 8 + 1]), pack_bf16(v[q8 * 8 + 2], v[q8 * 8 + 3]),
                                          pack_bf16(v[q8 * 8 + 4], v[q8 * 8 + 5]), pack_bf16(v[q8 * 8 + 6], v[q8 * 8 + 7]));
                    *reinterpret_cast<uint4*>(sl + (col / 64) * QR * 128 + sw128_offset(tid, (col % 64) * 2)) = pk;
                }
            }
        }
        // ---- scale in place: C~' = exp(cum_t) C~ ; B^ = exp(cum_end - cum_s) w_s B~
        {
            const float cend = sCum[Q - 1];
#pragma unroll
            for (int i = 0; i < TPG; ++i) {
                const int t = tg * TPG + i;
                const float fc = __expf(sCum[t]);
                const float fb = __expf(cend - sCum[t]) * sW[t];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t off = pan * QR * 128 + sw128_offset(t * R + r, cib);
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const float f = m == 0 ? fc : fb;
                        uint4* p = reinterpret_cast<uint4*>(st + (m == 0 ? K::OFF_C : K::OFF_B) + off);
                        uint4 v = *p;
                        uint32_t wv4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 g = unpack_bf16(wv4[e]);
                            wv4[e] = pack_bf16(g.x * f, g.y * f);
                        }
                        *p = make_uint4(wv4[0], wv4[1], wv4[2], wv4[3]);
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*sFail) { failed = true; break; }

        // ---- MMA2 + MMA4 -> Y ; MMA3 -> U
        if (tid == 0) {
            const uint32_t aSL = smem_u32(sm + K::OFF_SL), aX = smem_u32(st + K::OFF_X);
            const uint32_t aC = smem_u32(st + K::OFF_C), aHb = smem_u32(sm + K::OFF_HB);
            const uint32_t aB = smem_u32(st + K::OFF_B);
            constexpr uint32_t id_y = idesc_bf16_f32(128, P, false, true);
            constexpr uint32_t id_u = idesc_bf16_f32(128, P, true, true);
#pragma unroll
            for (int kk = 0; kk < QR / 16; ++kk) {   // Y = SL X
                const uint32_t koff = (kk >> 2) * QR * 128 + (kk & 3) * 32;
                mma_bf16_ss(tmem + K::T_Y, smem_desc(aSL + koff, 16, 1024, kSwizzle128B),
                            smem_desc(aX + kk * 2048, 16, 1024, kSwizzle128B), id_y, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < NS / 16; ++kk) {   // Y += C~' Hb
                const uint32_t koff = (kk >> 2) * QR * 128 + (kk & 3) * 32;
                mma_bf16_ss(tmem + K::T_Y, smem_desc(aC + koff, 16, 1024, kSwizzle128B),
                            smem_desc(aHb + kk * 2048, 16, 1024, kSwizzle128B), id_y, 1);
            }
            // U = B^^T X : A is MN-major over n (NS rows; panels QR*128 bytes apart)
            // (NS = 64: the second panel reads the next QR*128 bytes, results unused)
            constexpr uint32_t lbo_u = QR * 128;
#pragma unroll
            for (int kk = 0; kk < QR / 16; ++kk) {
                mma_bf16_ss(tmem + K::T_U, smem_desc(aB + kk * 2048, lbo_u, 1024, kSwizzle128B),
                            smem_desc(aX + kk * 2048, 16, 1024, kSwizzle128B), id_u, kk > 0);
            }
            mma_commit(bar_mma);
        }
        if (!mbar_wait(bar_mma, mma_phase, kWaitLimitNs)) *sFail = 1;
        mma_phase ^= 1;
        tc_fence_after();
        __syncthreads();
        if (*sFail) { failed = true; break; }
        // the stage is free again: prefetch chunk c+2 into it
        if (tid == 0 && c + 2 < nc) issue_loads(c + 2, s);
        if (c + 2 < nc) inflight[s] = c + 2;

        // ---- state update H_c = R(Theta) (exp(cum_end) H_{c-1} + U)   (thread = state row n)
        if (tid < NS) {
            const float e = __expf(sCum[Q - 1]);
            float sn, cs;
            sincosf(sTheta[tid >> 1], &sn, &cs);
            const bool odd = tid & 1;
#pragma unroll
            for (int cc = 0; cc < P; cc += 16) {
                float hv[16], uv[16];
                tmem_ld16(tlane + K::T_H + cc, hv);
                tmem_ld16(tlane + K::T_U + cc, uv);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float pre = fmaf(e, hv[i], uv[i]);
                    const float other = __shfl_xor_sync(0xffffffffu, pre, 1);
                    // even row 2j: cos*v_2j - sin*v_2j+1 ; odd row 2j+1: sin*v_2j + cos*v_2j+1
                    hv[i] = odd ? fmaf(sn, other, cs * pre) : fmaf(-sn, other, cs * pre);
                }
                tmem_st16(tlane + K::T_H + cc, hv);
            }
            tmem_st_wait();
        }
        // ---- outputs y rows (t, r)
        if (tid < QR) {
            const int t = tid / R, r = tid % R;
            const int tok = c * Q + t;
            __nv_bfloat16* yrow = args.y + ((((int64_t)b * T + tok) * args.H + h) * R + r) * P;
#pragma unroll
            for (int cc = 0; cc < P; cc += 16) {
                float v[16];
                tmem_ld16(tlane + K::T_Y + cc, v);
                tmem_ld_wait();
                if (tok < T) {
                    uint4 p0 = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                                          pack_bf16(v[6], v[7]));
                    uint4 p1 = make_uint4(pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]), pack_bf16(v[12], v[13]),
                                          pack_bf16(v[14], v[15]));
                    *reinterpret_cast<uint4*>(yrow + cc) = p0;
                    *reinterpret_cast<uint4*>(yrow + cc + 8) = p1;
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (!failed) {
        if (args.final_state != nullptr && tid < NS) {
            float* fs = args.final_state + ((int64_t)bh * NS + tid) * P;
#pragma unroll
            for (int cc = 0; cc < P; cc += 16) {
                float v[16];
                tmem_ld16(tlane + K::T_H + cc, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4*>(fs + cc + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
        }
    } else {
        if (tid == 0) {
            atomicExch(args.status, (int)M3_ERR_TIMEOUT);
            // drain the loads still in flight (bounded) before the shared memory goes away
            for (int s2 = 0; s2 < 2; ++s2)
                if (inflight[s2] >= 0) (void)mbar_wait(&bar_full[s2], (inflight[s2] >> 1) & 1, kWaitLimitNs);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, K::TMEM_COLS);
}

// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const cuuint64_t* dims,
              const cuuint64_t* strides_bytes, const cuuint32_t* box, CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;   // no driver entry point: the launch reports an error
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides_bytes, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NS, int R, int Q>
cudaError_t launch_cfg(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                       const float* A, const float* lambda, const float* omega, void* y, float* final_state,
                       void* workspace, cudaStream_t stream) {
    using K = Cfg<NS, R, Q>;
    const cuuint64_t Bt = d.batch, T = d.seqlen, H = d.nheads, P = d.headdim, N = d.dstate;
    CUtensorMap mx, mB, mC, mdt, mlam;
    {
        cuuint64_t dims[5] = {P, (cuuint64_t)R, H, T, Bt};
        cuuint64_t str[4] = {P * 2, R * P * 2, H * R * P * 2, T * H * R * P * 2};
        cuuint32_t box[5] = {64, (cuuint32_t)R, 1, (cuuint32_t)Q, 1};
        if (!make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, x, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[5] = {N, (cuuint64_t)R, H, T, Bt};
        cuuint64_t str[4] = {N * 2, R * N * 2, H * R * N * 2, T * H * R * N * 2};
        cuuint32_t box[5] = {64, (cuuint32_t)R, 1, (cuuint32_t)Q, 1};
        if (!make_map(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        if (!make_map(&mC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, C, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[3] = {H, T, Bt};
        cuuint64_t str[2] = {H * 4, T * H * 4};
        cuuint32_t box[3] = {4, (cuuint32_t)(Q + 1), 1};
        if (!make_map(&mdt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dt, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        if (!make_map(&mlam, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, lambda, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    TcArgs args;
    args.A = A;
    args.omega = omega;
    args.y = static_cast<__nv_bfloat16*>(y);
    args.final_state = final_state;
    args.status = static_cast<int*>(workspace);
    args.T = (int)d.seqlen;
    args.H = (int)d.nheads;
    args.nc = (int)d.nchunks();
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
    auto kern = scan_tc_kernel<NS, R, Q>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(d.batch * d.nheads), K::kThreads, K::SMEM, stream>>>(mx, mB, mC, mdt, mlam, args);
    return cudaGetLastError();
}

typedef cudaError_t (*LaunchFn)(const ScanDims&, const void*, const void*, const void*, const float*, const float*,
                                const float*, const float*, void*, float*, void*, cudaStream_t);

LaunchFn pick(const ScanDims& d) {
    if (d.headdim != 64 || d.io != M3_DTYPE_BF16) return nullptr;
    if (d.nheads % 4) return nullptr;
    if (d.dstate == 128) {
        if (d.R == 1 && d.chunk == 64) return launch_cfg<128, 1, 64>;
        if (d.R == 1 && d.chunk == 128) return launch_cfg<128, 1, 128>;
        if (d.R == 2 && d.chunk == 64) return launch_cfg<128, 2, 64>;
    }
    return nullptr;
}

}  // namespace

size_t tc_workspace_size(const ScanDims&) { return 256; }
bool tc_supported(const ScanDims& d) { return d.seqlen > 0 && pick(d) != nullptr; }
int tc_launch_count(const ScanDims&) { return 1; }
cudaError_t launch_scan_tc(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                           const float* A, const float* lambda, const float* omega, void* y, float* final_state,
                           void* workspace, cudaStream_t stream) {
    LaunchFn f = pick(d);
    if (!f) return cudaErrorNotSupported;
    return f(d, x, B, C, dt, A, lambda, omega, y, final_state, workspace, stream);
}

}  // namespace m3
