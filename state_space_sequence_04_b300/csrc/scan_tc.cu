// Tensor-core chunked prefill (bf16 io) for sm_103a: tcgen05 MMAs with TMEM
// accumulators, operands staged by TMA in 128-byte-swizzled shared memory.
//
// The chunked algorithm of "Mamba-3: Improved Sequence Modeling using State
// Space Principles" (section 3.3; decay x two-band mask of section 3.1.3 /
// Eq. 7; rotary form of Propositions 3-4), fused into one kernel: one CTA owns
// one (batch, head) sequence, or one segment of it, and walks its chunks in
// order, carrying the fp32 N x P state in TMEM, so no chunk state ever goes to
// HBM.  Per chunk c = tokens [c0, c0+Q) (rows ordered (token, rank), QR = Q*R):
//
//   coefficients   l_t = dt_t A, cum_t = sum_{k<=t} l_k (chunk-local),
//                  gamma_t = lambda_t dt_t, w_s = gamma_s + (1-lambda_{s+1}) dt_{s+1},
//                  rho_t = gamma_t / w_t (0 when w_t = 0; w_t >= gamma_t >= 0),
//                  g_s = log2 of exp(cum_end - cum_s), clamped at -100
//   rotation       Phi_t = the angle sum_k dt_k omega_k since the segment start (mod 2 pi),
//                  C~ = R(-Phi) C,  B'' = 2^g w R(-Phi) B   (in place in shared memory)
//   batch 1        H += B''^T X                       (chunk state onto the carry)
//                  Yi = C~ Hb_{c-1}                   (inter-chunk readout)
//   scores         S  = C~ B''^T
//   mask           SL_ts = S_ts 2^(cum2_t - cum2_s - g_s) for s < t, S_tt rho_t 2^-g_t, 0 for s > t
//                  (cum2 = cum log2 e; bf16, written over the B'' tile, which the MMAs have consumed)
//   batch 2        Y  = SL X
//   output         y_t = Y_t + exp(cum_t) Yi_t
//   state          Hb_c = bf16(H),  H <- exp(cum_end(c+1)) H
//
// The carry stays in the segment's rotating frame (B and C carry the phase since
// the segment start), where the transition between chunks is the scalar decay
// alone; the segment's final state is rotated back by R(Phi_end).  The decay
// to the chunk end rides on B'' (2^g), so the chunk-state MMA reads the raw X
// tile, and the mask divides it out again (every mask factor <= 2^100).  w_s
// takes the next token's lambda and dt (zero past the end), so the carry after
// a chunk already holds the delayed half of its last token's trapezoid, and
// after the last chunk it is the final state h_{T-1}.
//
// Warp roles (256 threads): warps 0-3 "consumer" (mask, state, output; thread
// 0 issues every MMA, thread 96 the C, B and X loads and the TMA store of each
// chunk's output tile), warps 4-7 "rotate" (coefficients, angles, rotation, the
// dt/lambda loads), which run one chunk ahead of the consumer on the other
// shared-memory stage.
// Every wait is bounded: on timeout the kernel records M3_ERR_TIMEOUT in the
// status word, drains its copies and MMAs and exits.
//
// Kernel modes (template bitmask PM) for the pre-activation entry point: bit 0
// takes Delta and lambda as pre-activations and one decay generator per token,
// bit 1 RMS-normalises and biases B and C in the rotation, bit 2 gates the
// output; mode 0 is the plain kernel.  FULL = false is the state pass of a
// segmented call: the rotated, scaled B and the chunk-state MMA only.
//
// MMA operand layouts (all 128-byte swizzled, bf16):
//   C~   A, K-major  (rows (t,r), K = n)     B''  B, K-major (rows (s,r), K = n)
//   SL   A, K-major  (rows (t,r), K = (s,r')) X   B, MN-major (K = (s,r'), N = p)
//   Hb   B, MN-major (K = n, N = p)          B''^T A, MN-major (M = n, K = (s,r'))
// When QR = 64 the score, inter-readout and output MMAs run with M = 64: row r
// of those accumulators sits in TMEM lane 32 (r / 16) + r % 16, and every
// consumer thread takes half a row (16-lane loads, two column halves), so all
// four consumer warps share the mask and the output.  With QR = 128 they run
// with M = 128 (row r in lane r).  The chunk-state MMA has M = N (state rows
// n): with N = 64 the carry takes the M = 64 layout too, its rows spread over
// the four consumer warps' lane quadrants.
#include <cuda.h>

#include "m3_common.cuh"
#include "tc_ptx.cuh"

namespace m3 {
namespace {

using namespace tc;

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait, then give up with M3_ERR_TIMEOUT
constexpr float kLog2e = 1.4426950408889634f;

#ifdef M3_TRACE
// Phase trace of a diagnostic build (compiled with -DM3_TRACE; the product build has none of it):
// clock64 at the phase boundaries of the first kTraceChunks chunks of each of the first kTraceCtas CTAs.
// Per (CTA, chunk): slots 0-15 the consumer group (thread 0; slots 11-12 thread 32), 16-31 the
// rotate group (thread 128).  g_m3_trace_clk holds, for each of the first kClkCtas CTAs of a launch,
// (globaltimer, clock64) at its start and its end and its SM's id: cycles into time, and the spread
// of CTA durations by SM.
constexpr int kTraceCtas = 512, kTraceChunks = 32, kTraceSlots = 32, kClkCtas = 4096, kClkSlots = 6;
__device__ long long g_m3_trace[kTraceCtas * kTraceChunks * kTraceSlots];
__device__ long long g_m3_trace_clk[kClkCtas * kClkSlots];
#define M3_TRACE_BY(thread, i, slot)                                                                    \
    do {                                                                                                \
        if (blockIdx.x < kTraceCtas && (i) < kTraceChunks && threadIdx.x == (thread))                   \
            g_m3_trace[((int)blockIdx.x * kTraceChunks + (i)) * kTraceSlots + (slot)] = clock64();     \
    } while (0)
#else
#define M3_TRACE_BY(thread, i, slot) \
    do {                             \
    } while (0)
#endif
#define M3_TRACE_C(i, slot) M3_TRACE_BY(0, i, slot)
#define M3_TRACE_R(i, slot) M3_TRACE_BY(128, i, 16 + (slot))

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// FULL = false is the state pass's layout: no C tile, no bf16 copy of the carry, only the carry in TMEM.
template <int NS, int R, int Q, bool FULL = true>
struct Cfg {
    static constexpr int P = 64;                 // head dim (one 128-byte swizzle panel of bf16)
    static constexpr int QR = Q * R;             // rows of the chunk
    static constexpr int NPAN = NS / 64;         // 64-wide panels of B / C
    static constexpr int kThreads = 256;
    static_assert(QR == 64 || QR == 128, "chunk rows must be 64 or 128");
    static_assert(NS == 64 || NS == 128, "state size must be 64 or 128");
    static_assert(Q <= 128, "chunk too long");
    // rows of the score / inter / output accumulators: M = 64 puts row r in TMEM lane
    // 32 (r / 16) + r % 16 (16 lanes of each warp's quadrant), M = 128 in lane r
    static constexpr bool M64 = QR == 64;
    static constexpr int MM = M64 ? 64 : 128;

    static constexpr int X_BYTES = QR * 128;
    static constexpr int BC_BYTES = NPAN * QR * 128;
    static constexpr int SL_BYTES = QR * QR * 2;
    static_assert(!FULL || SL_BYTES <= BC_BYTES, "the masked scores are written over the chunk's B tile");
    // one stage: C | B | X, or B | X in the state pass
    static constexpr int STG_B = FULL ? BC_BYTES : 0, STG_X = STG_B + BC_BYTES;
    static constexpr int STG_TILE = STG_X + X_BYTES;
    static constexpr int BOX_BYTES = 16 * (Q + 1);                // dt / lambda box {4 heads, Q+1 tokens}
    static constexpr int BOX_STRIDE = align_up(BOX_BYTES, 128);
    // rotate-phase mapping: pair group jg (4 pairs = 16 bytes of a row), token group tg
    static constexpr int NG = NS / 8;
    static constexpr int TG = 128 / NG;
    static constexpr int TPG = Q / TG;
    static_assert(Q % TG == 0, "tokens must split evenly over token groups");
    static constexpr int PART_BYTES = TG * (NS / 2) * 4;          // partial angle sums [TG][NS/2]
    // the partial sums go over the stage's two boxes once their values are in registers
    static constexpr bool PART_IN_BOX = PART_BYTES <= 2 * BOX_STRIDE;
    // coefficient block of a stage (floats): cum*log2e[Q], rho[Q], exp(cum)[Q], b[Q],
    // f = exp(cum_end - cum)[Q], Theta[NS/2] (the phase of each pair at the chunk's last token since
    // the segment start, mod 2 pi), exp(cum_end), cum_end
    static constexpr int CO_CUM2 = 0, CO_RHO = Q, CO_ECUM = 2 * Q, CO_BNEG = 3 * Q, CO_CG = 4 * Q, CO_THETA = 5 * Q,
                         CO_EEND = 5 * Q + NS / 2, CO_CEND = 5 * Q + NS / 2 + 1;
    static constexpr int CO_BYTES = align_up((5 * Q + NS / 2 + 2) * 4, 16);

    static constexpr int OFF_HB = 2 * STG_TILE;
    // the full pass's output tile y (QR rows x P, bf16, 128-byte swizzle), written by the consumer
    // threads and stored by one TMA store
    static constexpr int OFF_OUT = OFF_HB + (FULL ? NS * 128 : 0);
    static constexpr int OFF_BOX = OFF_OUT + (FULL ? QR * 128 : 0);   // [stage][dt | lambda]
    static constexpr int OFF_PART = OFF_BOX + 4 * BOX_STRIDE;     // only when not in the boxes
    static constexpr int OFF_CO = OFF_PART + (PART_IN_BOX ? 0 : align_up(PART_BYTES, 16));
    static constexpr int OFF_RPRIV = OFF_CO + 2 * CO_BYTES;       // w[Q], warp sums[4]
    static constexpr int OFF_BAR = align_up(OFF_RPRIV + (Q + 4) * 4, 16);
    static constexpr int SMEM = OFF_BAR + 192 + 1024;             // barriers / flags, alignment slack
    // two CTAs per SM when both fit (228 KB per SM, 1 KB reserved per CTA)
    static constexpr int MIN_BLOCKS = 2 * (SMEM + 1024) <= 233472 ? 2 : 1;
    static constexpr int TX_BOX = 2 * BOX_BYTES;

    // TMEM columns (the state pass holds the carry alone)
    static constexpr int T_S = 0;
    static constexpr int T_YI = QR;
    static constexpr int T_Y = QR + P;
    static constexpr int T_H = FULL ? QR + 2 * P : 0;
    static constexpr int TMEM_COLS = !FULL ? P : (QR + 3 * P) <= 256 ? 256 : 512;
    static_assert(SMEM <= 232448, "shared memory over the 227 KB per-CTA limit");
    static_assert(FULL ? !M64 || MIN_BLOCKS == 2 : MIN_BLOCKS == 2, "64-row tiles and the state pass are laid out for two CTAs per SM");
};

struct TcArgs {
    const float* A;          // [H], or [Bt,T,H] (one per token) in the pre-activation variant
    const float* dt_bias;    // pre-activation variant: [H] or null
    const float* omega;
    __nv_bfloat16* y;
    float* final_state;
    int* status;
    int T, H, nc;
    // sequence segments: this launch covers segments 0 .. nseg-1 of S of L chunks each
    int L, nseg, S;
    const float* h_in;       // [bh][S-1][N][P]: state entering segment k (k <= S-2), or null
    const float* h_in_last;  // [bh][N][P]: state entering segment S-1, or null
    float* seg_U;            // state pass: [bh][S-1][N][P] carry at the segment's end from a zero start
    float* seg_ld;           // state pass: [bh][S-1] summed log-decay of the segment
    float* seg_th;           // state pass: [bh][S-1][N/2] summed rotation angle of the segment
};

// Arguments of the pre-activation variants' B / C normalisation and output gate
// (a separate kernel parameter, an empty struct for the plain kernel so that its
// parameter block stays as it is): per-channel gains [N] (null = 1), channel
// biases [H, R, N] (null = 0), RMS normalisation on / off and its eps, the gate
// input z (y's layout, bf16).
template <int PM>
struct ExtArgs {
    const float* B_gain;
    const float* C_gain;
    const float* B_bias;
    const float* C_bias;
    int bc_norm;
    float bc_eps;
    const __nv_bfloat16* z;
};
template <>
struct ExtArgs<0> {};
// The failure-path test mode (kTestHook): every CTA's consumer group gives up at its local chunk
// fail_chunk by waiting, with a short limit, on a barrier that nothing completes.
constexpr int kTestHook = 8;
template <>
struct ExtArgs<kTestHook> {
    int fail_chunk;
};

// Word i (two bf16) of a run of 16-byte pieces.
__device__ __forceinline__ uint32_t word_at(const uint4* a, int i) {
    const uint4 v = a[i >> 2];
    return (i & 3) == 0 ? v.x : (i & 3) == 1 ? v.y : (i & 3) == 2 ? v.z : v.w;
}

// Shared control block (after the barriers).  Two TMA groups per stage, each
// issued as soon as its previous contents are dead: the dt / lambda boxes
// (once the rotate group has read them), and C, B and X together (once the
// chunk's output MMAs are complete).
struct Ctl {
    uint64_t fbox[2], fcbx[2];   // TMA groups landed: the dt / lambda boxes; C, B and X
    uint64_t bc_done[2];     // rotate group rotated the stage's C and B (count 128)
    uint64_t rot_done[2];    // rotate group finished the stage (count 128)
    uint64_t coef_ready[2];  // coefficient block of the stage written (count 128)
    uint64_t coef_free[2];   // consumer done reading the stage's coefficient block (count 128)
    uint64_t bH;             // chunk state onto the carry H complete (one per chunk)
    uint64_t bY;             // output Y (and the inter readout Yi issued before it) complete (one per chunk)
    uint64_t never;          // completed by nothing: the failure-path test mode waits on it
    uint64_t drain;          // on failure: one commit covering every MMA issued, waited before TMEM is freed
    uint32_t tmem;
    int fail_c, fail_r;      // per-group failure flags
    // copies issued and waited for, modulo 2^16 (only their difference, at most 2, and
    // their parity matter: they drive the bounded drain on failure)
    uint16_t box_issued[2], box_waited[2], cbx_issued[2], cbx_waited[2];
};
static_assert(sizeof(Ctl) <= 192, "control block must fit its reserved space");

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void group_bar(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

// Bounded wait on an mbarrier phase.  Gives up (setting *mine) on timeout or
// when either group has already failed.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* mine,
                                             volatile int* other, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*mine || *other || globaltimer_ns() - t0 > limit_ns) {
                *mine = 1;
                return false;
            }
        }
    }
}

// An angle reduced modulo 2 pi to [-pi, pi]: x - k 2pi with k = rint(x / 2pi), the product k 2pi
// taken in two parts (2pi = 6.28125 + 1.9353071795864769e-3; the first part has few enough bits
// that k times it is exact for |k| < 2^15), after Cody and Waite's argument reduction.
__device__ __forceinline__ float reduce_2pi(float x) {
    const float k = rintf(x * 0.15915494309189535f);
    return fmaf(-k, 1.9353071795864769e-3f, fmaf(-k, 6.28125f, x));
}
__device__ __forceinline__ float4 reduce_2pi(float4 v) {
    return make_float4(reduce_2pi(v.x), reduce_2pi(v.y), reduce_2pi(v.z), reduce_2pi(v.w));
}

// Rotate the 4 pairs of one 16-byte piece by (c[k], s[k]) (angle -Psi), optionally
// scaled, in place; fp32 arithmetic on packed pairs of pairs.
__device__ __forceinline__ uint4 rotate4(uint4 v, const float2 (&c01)[2], const float2 (&s01)[2]) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float2 a = make_float2(bf_lo(w[2 * h]), bf_lo(w[2 * h + 1]));
        const float2 b = make_float2(bf_hi(w[2 * h]), bf_hi(w[2 * h + 1]));
        // a' = c a - s b ; b' = s a + c b
        const float2 na = __ffma2_rn(c01[h], a, __fmul2_rn(make_float2(-s01[h].x, -s01[h].y), b));
        const float2 nb = __ffma2_rn(s01[h], a, __fmul2_rn(c01[h], b));
        w[2 * h] = pack_bf16(na.x, nb.x);
        w[2 * h + 1] = pack_bf16(na.y, nb.y);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The B / C normalisation of the pre-activation variant fused with the rotation.
// sumsq8: the sum of squares of the 8 channels of a 16-byte piece (4 pairs) of a
// row; the row's total comes from the NG lanes holding it (lanes differing in
// their low log2(NG) bits).  bc_rotate4: the piece's channels become
// v * sc * g + bias (sc = 1 / sqrt(mean(v^2) + eps)) or, without the norm,
// v + bias, then its pairs are rotated as in rotate4.
__device__ __forceinline__ float sumsq8(uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        ss = fmaf(bf_lo(w[q]), bf_lo(w[q]), ss);
        ss = fmaf(bf_hi(w[q]), bf_hi(w[q]), ss);
    }
    return ss;
}

__device__ __forceinline__ uint4 bc_rotate4(uint4 v, const float2 (&c01)[2], const float2 (&s01)[2],
                                            const float (&g)[8], const float (&bb)[8], bool norm, float sc) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float e[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        e[2 * q] = bf_lo(w[q]);
        e[2 * q + 1] = bf_hi(w[q]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = norm ? fmaf(e[i] * sc, g[i], bb[i]) : e[i] + bb[i];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float2 a = make_float2(e[4 * h], e[4 * h + 2]);
        const float2 b = make_float2(e[4 * h + 1], e[4 * h + 3]);
        const float2 na = __ffma2_rn(c01[h], a, __fmul2_rn(make_float2(-s01[h].x, -s01[h].y), b));
        const float2 nb = __ffma2_rn(s01[h], a, __fmul2_rn(c01[h], b));
        w[2 * h] = pack_bf16(na.x, nb.x);
        w[2 * h + 1] = pack_bf16(na.y, nb.y);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Per-thread registers of the B / C normalisation (gains of this thread's 8
// channels; with one rank, its head's biases); empty when the variant is off.
template <bool ON>
struct BcRegs {
    float gB[8], gC[8], bB1[8], bC1[8];
};
template <>
struct BcRegs<false> {};

// 8 consecutive floats from p (16-byte aligned), or `fill` when p is null.
__device__ __forceinline__ void load8(const float* p, float fill, float (&o)[8]) {
    if (p == nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = fill;
        return;
    }
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// Mask one 16-column block of a score row held in v[0..15]: columns cb..cb+15
// (tokens cb/R ..), row token t.  The scores were taken with B'' = f' B' (f'_s =
// 2^g_s, the decay from token s to the chunk's end, clamped at 2^-100), so the
// mask also divides by f'_s.  Blocks strictly below the diagonal use the
// factorised factor 2^(cum2_t - cum2_e) 2^(cum2_e - cum2_s - g_s), e = the
// block's last token (the first factor <= 1, the second, b_s, <= 2^100); the
// diagonal block uses 2^(cum2_t - (cum2_s + g_s)) directly (cg = cum2 + g) and
// rho_t 2^-g_t on the diagonal; blocks above are zero.  The per-token factors
// come in as 16-byte loads.  With R >= 2 a block holds 16 / R tokens, each on R
// columns: one exponential per token, and the diagonal block selects instead of
// branching per column (the lanes of a warp hold different rows t).  With R = 1
// the diagonal block's exponentials stay predicated per column: measured, the
// select form is slower there (SISO 62.9 against 64.8 Mtok/s) and faster with
// R = 4 (long-context MIMO 15.3 against 15.1).
template <int R>
__device__ __forceinline__ void mask_block(float* v, int cb, int t, float ct, float rt, const float* cum2,
                                           const float* bneg, const float* cg) {
    if constexpr (R == 1) {
        const int s_lo = cb, s_hi = cb + 15;
        if (s_lo > t) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        } else if (s_hi < t) {
            const float a = ex2_approx(ct - cum2[s_hi]);
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const float4 q = *reinterpret_cast<const float4*>(bneg + cb + i);
                const float2 r0 = __fmul2_rn(make_float2(v[i], v[i + 1]), __fmul2_rn(a2, make_float2(q.x, q.y)));
                const float2 r1 = __fmul2_rn(make_float2(v[i + 2], v[i + 3]), __fmul2_rn(a2, make_float2(q.z, q.w)));
                v[i] = r0.x;
                v[i + 1] = r0.y;
                v[i + 2] = r1.x;
                v[i + 3] = r1.y;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const float4 q = *reinterpret_cast<const float4*>(cg + cb + i);
                const float g4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int sidx = cb + i + k;
                    float m = 0.f;
                    if (sidx < t) m = ex2_approx(ct - g4[k]);
                    else if (sidx == t) m = rt;
                    v[i + k] *= m;
                }
            }
        }
    } else {
        constexpr int NSB = 16 / R;   // tokens of the block
        static_assert(16 % R == 0 && NSB % 4 == 0, "a block holds a multiple of 4 tokens");
        const int s0 = cb / R, s_hi = s0 + NSB - 1;   // cb is a multiple of 16: s0 of NSB (16-byte aligned)
        if (s0 > t) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        } else if (s_hi < t) {
            const float a = ex2_approx(ct - cum2[s_hi]);
#pragma unroll
            for (int j = 0; j < NSB; j += 4) {
                const float4 q = *reinterpret_cast<const float4*>(bneg + s0 + j);
                const float b[4] = {a * q.x, a * q.y, a * q.z, a * q.w};
#pragma unroll
                for (int k = 0; k < 4 * R; ++k) v[j * R + k] *= b[k / R];
            }
        } else {
#pragma unroll
            for (int j = 0; j < NSB; j += 4) {
                const float4 q = *reinterpret_cast<const float4*>(cg + s0 + j);
                const float e[4] = {ct - q.x, ct - q.y, ct - q.z, ct - q.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int sj = s0 + j + k;
                    const float x = ex2_approx(e[k]);   // +inf above the diagonal is selected away
                    const float m = sj < t ? x : (sj == t ? rt : 0.f);
#pragma unroll
                    for (int r = 0; r < R; ++r) v[(j + k) * R + r] *= m;
                }
            }
        }
    }
}

// FULL = true: the whole chunked prefill of its segment (outputs y; the last
// segment writes the final state).  FULL = false: the state pass of the
// segmented prefill -- only the carry (rotated, scaled B, scaled X and the
// chunk-state MMA), whose value at the segment's end from a zero start, summed
// log-decay and summed angles go to the workspace for the segment scan.
// PM (bitmask) & 1, the pre-activation variant: the dt and lambda inputs are
// pre-activations (Delta = softplus(dt + dt_bias[h]), lambda = sigmoid(u), applied
// to the staged boxes in shared memory) and A holds one decay generator per
// token.  PM & 2 adds the B / C normalisation and channel biases, fused with the
// rotation; PM & 4 the output gate y * silu(z) in the epilogue.  PM == kTestHook
// is the plain kernel with a simulated timeout (the failure-path test).
template <int NS, int R, int Q, bool FULL, int PM>
__global__ void __launch_bounds__(256, (Cfg<NS, R, Q, FULL>::MIN_BLOCKS)) scan_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                         const __grid_constant__ CUtensorMap tm_B,
                                                         const __grid_constant__ CUtensorMap tm_C,
                                                         const __grid_constant__ CUtensorMap tm_dt,
                                                         const __grid_constant__ CUtensorMap tm_lam,
                                                         const __grid_constant__ CUtensorMap tm_y, TcArgs args,
                                                         const ExtArgs<PM> ext) {
    using K = Cfg<NS, R, Q, FULL>;
    constexpr bool HOOK = PM == kTestHook;
    constexpr bool PREP = !HOOK && (PM & 1) != 0, BC = !HOOK && (PM & 2) != 0, GATE = !HOOK && (PM & 4) != 0;
    constexpr int P = K::P, QR = K::QR, NP2 = NS / 2, NG = K::NG, TG = K::TG, TPG = K::TPG;
    constexpr int TX_CB = FULL ? 2 * K::BC_BYTES : K::BC_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(sm + K::OFF_BAR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef M3_TRACE
    if (tid == 0 && blockIdx.x < kClkCtas) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        g_m3_trace_clk[blockIdx.x * kClkSlots + 0] = (long long)globaltimer_ns();
        g_m3_trace_clk[blockIdx.x * kClkSlots + 1] = clock64();
        g_m3_trace_clk[blockIdx.x * kClkSlots + 4] = smid;
    }
#endif
    const int bh = blockIdx.x / args.nseg, seg = blockIdx.x % args.nseg;
    const int b = bh / args.H, h = bh % args.H, hq = h & 3;
    const int T = args.T;
    const int c_begin = seg * args.L;
    const int nl = min(args.nc, c_begin + args.L) - c_begin;   // chunks of this segment (>= 1)

    auto tile_c = [&](int s) { return sm + s * K::STG_TILE; };   // full pass only
    auto tile_b = [&](int s) { return sm + s * K::STG_TILE + K::STG_B; };
    auto tile_x = [&](int s) { return sm + s * K::STG_TILE + K::STG_X; };
    auto box_dt = [&](int s) { return reinterpret_cast<float*>(sm + K::OFF_BOX + (2 * s) * K::BOX_STRIDE); };
    auto box_lam = [&](int s) { return reinterpret_cast<float*>(sm + K::OFF_BOX + (2 * s + 1) * K::BOX_STRIDE); };
    auto coef = [&](int s) { return reinterpret_cast<float*>(sm + K::OFF_CO + s * K::CO_BYTES); };
    uint8_t* hb = sm + K::OFF_HB;
    uint8_t* out_tile = sm + K::OFF_OUT;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&ctl->fbox[s], 1);
            mbar_init(&ctl->fcbx[s], 1);
            mbar_init(&ctl->bc_done[s], 128);
            mbar_init(&ctl->rot_done[s], 128);
            mbar_init(&ctl->coef_ready[s], 128);
            mbar_init(&ctl->coef_free[s], 128);
            ctl->box_issued[s] = ctl->box_waited[s] = 0;
            ctl->cbx_issued[s] = ctl->cbx_waited[s] = 0;
        }
        mbar_init(&ctl->bH, 1);
        mbar_init(&ctl->bY, 1);
        mbar_init(&ctl->never, 1);
        mbar_init(&ctl->drain, 1);
        ctl->fail_c = 0;
        ctl->fail_r = 0;
        fence_mbar_init();
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_B);
        if (FULL) prefetch_tensormap(&tm_C);
        if (FULL) prefetch_tensormap(&tm_y);
        prefetch_tensormap(&tm_dt);
        prefetch_tensormap(&tm_lam);
    }
    __syncthreads();

    // the two TMA groups of local chunk i into stage s (single issuing thread each)
    auto load_box = [&](int i, int s) {
        const int c0 = (c_begin + i) * Q;
        mbar_arrive_expect_tx(&ctl->fbox[s], K::TX_BOX);
        tma_load_3d(box_dt(s), &tm_dt, &ctl->fbox[s], h & ~3, c0, b);
        tma_load_3d(box_lam(s), &tm_lam, &ctl->fbox[s], h & ~3, c0, b);
        ctl->box_issued[s] += 1;
    };
    // C, B and X on one barrier: the rotate group waits for them once, and its rot_done then tells the
    // consumer's MMAs that X has landed as well
    auto load_cbx = [&](int i, int s) {
        const int c0 = (c_begin + i) * Q;
        mbar_arrive_expect_tx(&ctl->fcbx[s], TX_CB + K::X_BYTES);
#pragma unroll
        for (int p = 0; p < K::NPAN; ++p) {
            if (FULL) tma_load_5d(tile_c(s) + p * QR * 128, &tm_C, &ctl->fcbx[s], 64 * p, 0, h, c0, b);
            tma_load_5d(tile_b(s) + p * QR * 128, &tm_B, &ctl->fcbx[s], 64 * p, 0, h, c0, b);
        }
        tma_load_5d(tile_x(s), &tm_x, &ctl->fcbx[s], 0, 0, h, c0, b);
        ctl->cbx_issued[s] += 1;
    };

    if (warp == 0) {
        tmem_alloc(&ctl->tmem, K::TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2 && i < nl; ++i) {
            load_box(i, i);
            load_cbx(i, i);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    volatile int* fail_c = &ctl->fail_c;
    volatile int* fail_r = &ctl->fail_r;

    if (warp < 4) {
        // =============================== consumer ===============================
        const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
        // the state entering the segment: zero, or from the segment scan
        const float* hin = nullptr;
        if (FULL && seg > 0)
            hin = seg < args.S - 1 ? args.h_in + ((int64_t)bh * (args.S - 1) + seg) * NS * P
                                   : args.h_in_last + (int64_t)bh * NS * P;
        // Carry rows and columns of a thread.  The chunk-state MMA runs at M = NS: with NS = 128 thread =
        // row n, all P columns (lane n); with NS = 64 row n sits in lane 32 (n / 16) + n % 16 (lanes 0-15
        // of each warp's quadrant) and two threads share it, 32 columns each.  Every consumer thread
        // takes part either way.
        constexpr bool H64 = NS == 64;
        static_assert(NS == 64 || NS == 128, "carry layouts for NS = 64 and 128");
        const int hrow = H64 ? warp * 16 + (lane & 15) : tid;
        const int hc0 = H64 ? 32 * (lane >> 4) : 0;
        constexpr int HCOLS = H64 ? 32 : P;
        auto h_ld = [&](int cc, float (&v)[32]) {
            if constexpr (H64) tmem_ld16x2_sync(tlane + K::T_H, v);
            else tmem_ld32_sync(tlane + K::T_H + cc, v);
        };
        auto h_st = [&](int cc, const float (&v)[32]) {
            if constexpr (H64) tmem_st16x2(tlane + K::T_H, v);
            else tmem_st32(tlane + K::T_H + cc, v);
        };
        // the carry entering the segment: H_in, or zero (its bf16 copy and the first chunk's decay come
        // from a state step, below)
        {
#pragma unroll
            for (int cc = 0; cc < HCOLS; cc += 32) {
                float v[32];
                if (hin != nullptr) {
#pragma unroll
                    for (int i4 = 0; i4 < 32; i4 += 4) {
                        const float4 q = *reinterpret_cast<const float4*>(hin + (int64_t)hrow * P + hc0 + cc + i4);
                        v[i4] = q.x; v[i4 + 1] = q.y; v[i4 + 2] = q.z; v[i4 + 3] = q.w;
                    }
                } else {
#pragma unroll
                    for (int i4 = 0; i4 < 32; ++i4) v[i4] = 0.f;
                }
                h_st(cc, v);
            }
            tmem_st_wait();
        }
        // ---- the state step: Hb <- bf16(H) (read by the next inter readout Yi), H <- e H with e the decay
        //      of the chunk about to run (the carry rows and columns of each thread, above; the TMEM
        //      loads are warp-collective).  The carry lives in the segment's rotating frame (B and C are
        //      rotated by the phase since the segment start), where the transition is the scalar decay
        //      alone (Propositions 3-4).
        auto hb_write = [&](int cc, const float (&hv)[32]) {   // Hb <- bf16(H), 32 columns
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                const uint4 pk = make_uint4(pack_bf16(hv[q8 * 8 + 0], hv[q8 * 8 + 1]),
                                            pack_bf16(hv[q8 * 8 + 2], hv[q8 * 8 + 3]),
                                            pack_bf16(hv[q8 * 8 + 4], hv[q8 * 8 + 5]),
                                            pack_bf16(hv[q8 * 8 + 6], hv[q8 * 8 + 7]));
                *reinterpret_cast<uint4*>(hb + sw128_offset(hrow, (hc0 + cc + q8 * 8) * 2)) = pk;
            }
        };
        auto h_scale_st = [&](int cc, float (&hv)[32], float e) {   // H <- e H, 32 columns
            const float2 e2 = make_float2(e, e);
#pragma unroll
            for (int i2 = 0; i2 < 32; i2 += 2) {
                const float2 sc = __fmul2_rn(e2, make_float2(hv[i2], hv[i2 + 1]));
                hv[i2] = sc.x;
                hv[i2 + 1] = sc.y;
            }
            h_st(cc, hv);
        };
        auto state_step = [&](float e) {
#pragma unroll
            for (int cc = 0; cc < HCOLS; cc += 32) {
                float hv[32];
                h_ld(cc, hv);
                if (FULL) hb_write(cc, hv);
                h_scale_st(cc, hv, e);
            }
            tmem_st_wait();
            if (FULL) fence_proxy_async_smem();
        };
        // Where it runs.  With R >= 2, at the top of each chunk once rot_done is in (which implies the
        // chunk's coefficient block), so the consumer -- the critical path of these configurations --
        // waits one barrier less per chunk.  With R = 1, at the end of the previous chunk (after waiting
        // for the next chunk's coefficients), where it overlaps the rotate group's longer 64-token
        // rotation.  Measured both ways: SISO 61.0 / 57.6 Mtok/s, MIMO 30.5 / 31.7, long context
        // 13.4 / 13.7 (end / top).
        constexpr bool STEP_AT_TOP = R >= 2;
        if (!STEP_AT_TOP) {   // chunk 0's step: Hb_{-1} = bf16(H_in), H = e^{cum_end} H_in
            float e0 = 1.f;
            if (hin != nullptr) {
                (void)wait_bounded(&ctl->coef_ready[0], 0, fail_c, fail_r);
                e0 = coef(0)[K::CO_EEND];
            }
            tc_fence_after();
            state_step(e0);
        }
        tc_fence_before();
        group_bar(1);
        // the next C, B and X loads and the output stores go out from warp 3: warp 0 issues every MMA
        // and is the last to reach the output
        constexpr int kCbxThread = 96;
        // y of local chunk j from the output tile (every consumer thread wrote and fenced its rows
        // before the barrier this follows)
        auto store_y = [&](int j) {
            tma_store_5d(&tm_y, out_tile, 0, 0, h, (c_begin + j) * Q, b);
            bulk_commit_group();
        };
        float ld_sum = 0.f;   // state pass: summed log-decay (thread 0)
        // S = C~ B''^T of the chunk in stage s (thread 0, which issues every MMA).  No commit of its own:
        // the chunk-state commit that follows it on the same thread completes only after it
        auto issue_scores = [&](int s) {
            const uint64_t dC = smem_desc(smem_u32(tile_c(s)), 16, 1024, kSwizzle128B);
            const uint64_t dB = smem_desc(smem_u32(tile_b(s)), 16, 1024, kSwizzle128B);
            constexpr uint32_t id_s = idesc_bf16_f32(K::MM, QR, false, false);
#pragma unroll
            for (int kk = 0; kk < NS / 16; ++kk) {
                const uint32_t ko = ((kk >> 2) * QR * 128 + (kk & 3) * 32) >> 4;
                mma_bf16_ss(tmem + K::T_S, dC + ko, dB + ko, id_s, kk > 0);
            }
        };
        // the scores of local chunk s_next are the next ones to issue (thread 0): each chunk's go
        // out as soon as its rotation is done and the previous chunk's mask has read the S columns
        int s_next = 0;
        if (FULL && tid == 0 && wait_bounded(&ctl->bc_done[0], 0, fail_c, fail_r)) {
            tc_fence_after();
            issue_scores(0);
            s_next = 1;
        }

        for (int i = 0; i < nl; ++i) {
            const int c = c_begin + i, s = i & 1;
            const float* co = coef(s);
            M3_TRACE_C(i, 0);
            // ---- once the rotate group has finished this stage:
            //      H += B''^T X (the chunk state onto the carry), then Yi = C~ Hb_{c-1}
            (void)wait_bounded(&ctl->rot_done[s], (i >> 1) & 1, fail_c, fail_r);
            if constexpr (HOOK) {
                if (FULL && i == ext.fail_chunk) (void)wait_bounded(&ctl->never, 0, fail_c, fail_r, 50000ull);
            }
            M3_TRACE_C(i, 8);
            if constexpr (STEP_AT_TOP) {   // into this chunk: its decay; H+= and Yi of the last are complete
                tc_fence_after();
                state_step(co[K::CO_EEND]);
            }
            M3_TRACE_C(i, 9);
            tc_fence_before();
            group_bar(1);
            if (*fail_c) break;
            if (FULL && tid == kCbxThread && i > 0) store_y(i - 1);
            M3_TRACE_C(i, 1);
            // output gate: this thread's z values of the chunk, loaded now so that their latency
            // hides behind the MMAs and the mask (zero past the end of the sequence)
            constexpr int NZ = GATE && FULL ? (K::M64 ? 4 : 8) : 1;
            uint4 zg[NZ];
            if constexpr (GATE && FULL) {
                const bool mine = K::M64 || warp * 32 < QR;
                const int row = K::M64 ? warp * 16 + (lane & 15) : tid, t = row / R, r = row % R;
                const int tok = c * Q + t;
                const __nv_bfloat16* zrow = ext.z + ((((int64_t)b * T + tok) * args.H + h) * R + r) * P +
                                            (K::M64 ? 32 * (lane >> 4) : 0);
#pragma unroll
                for (int k = 0; k < NZ; ++k)
                    zg[k] = mine && tok < T ? __ldg(reinterpret_cast<const uint4*>(zrow) + k) : make_uint4(0u, 0u, 0u, 0u);
            }
            if (tid == 0) {
                tc_fence_after();
                if (FULL && s_next == i) {   // not issued early: the rotation was not done in time
                    issue_scores(s);
                    s_next = i + 1;
                }
                // the chunk's X (read by the chunk state here and by the output later) has landed:
                // the rotate group waited for it (with C and B) before arriving on rot_done
                // descriptors of the operand bases; a byte offset o moves the start address field by o >> 4
                const uint64_t dBt = smem_desc(smem_u32(tile_b(s)), QR * 128, 1024, kSwizzle128B);
                const uint64_t dX = smem_desc(smem_u32(tile_x(s)), 16, 1024, kSwizzle128B);
                constexpr uint32_t id_u = idesc_bf16_f32(NS, P, true, true);
                // A is MN-major over n (M = NS rows; panels QR*128 bytes apart)
#pragma unroll
                for (int kk = 0; kk < QR / 16; ++kk)
                    mma_bf16_ss(tmem + K::T_H, dBt + kk * (2048 >> 4), dX + kk * (2048 >> 4), id_u, 1);
                mma_commit(&ctl->bH);
                if (FULL) {   // Yi = C~ Hb_{c-1}: tracked by the output's commit
                    const uint64_t dC = smem_desc(smem_u32(tile_c(s)), 16, 1024, kSwizzle128B);
                    const uint64_t dHb = smem_desc(smem_u32(hb), 16, 1024, kSwizzle128B);
                    constexpr uint32_t id_y = idesc_bf16_f32(K::MM, P, false, true);
#pragma unroll
                    for (int kk = 0; kk < NS / 16; ++kk) {
                        const uint32_t ko = ((kk >> 2) * QR * 128 + (kk & 3) * 32) >> 4;
                        mma_bf16_ss(tmem + K::T_YI, dC + ko, dHb + kk * (2048 >> 4), id_y, kk > 0);
                    }
                }
                M3_TRACE_C(i, 2);
            }
            (void)wait_bounded(&ctl->bH, i & 1, fail_c, fail_r);
            M3_TRACE_BY(32, i, 12);
            M3_TRACE_C(i, 3);
            tc_fence_after();

            float ecum_t = 0.f;
            if constexpr (FULL) {
                uint8_t* sl = tile_b(s);
                // ---- mask: SL = S o L (bf16, K-major rows (t,r)) over the chunk's B' tile, which
                //      the scores and the chunk-state MMA have consumed
                if constexpr (K::M64) {
                    // thread = (row, half): row 16 warp + lane % 16, columns [32 half, 32 half + 32)
                    const int row = warp * 16 + (lane & 15), half = lane >> 4, t = row / R;
                    const float* cum2 = co + K::CO_CUM2;
                    const float ct = cum2[t], rt = co[K::CO_RHO + t];
                    ecum_t = co[K::CO_ECUM + t];
                    float v[32];
                    tmem_ld16x2_sync(tlane + K::T_S, v);
                    mask_block<R>(v, 32 * half, t, ct, rt, cum2, co + K::CO_BNEG, co + K::CO_CG);
                    mask_block<R>(v + 16, 32 * half + 16, t, ct, rt, cum2, co + K::CO_BNEG, co + K::CO_CG);
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        const int col = 32 * half + q8 * 8;
                        *reinterpret_cast<uint4*>(sl + sw128_offset(row, col * 2)) =
                            make_uint4(pack_bf16(v[q8 * 8 + 0], v[q8 * 8 + 1]), pack_bf16(v[q8 * 8 + 2], v[q8 * 8 + 3]),
                                       pack_bf16(v[q8 * 8 + 4], v[q8 * 8 + 5]), pack_bf16(v[q8 * 8 + 6], v[q8 * 8 + 7]));
                    }
                    fence_proxy_async_smem();
                } else if (warp * 32 < QR) {
                    const int row = tid, t = row / R;
                    const float* cum2 = co + K::CO_CUM2;
                    const float ct = cum2[t], rt = co[K::CO_RHO + t];
                    ecum_t = co[K::CO_ECUM + t];
                    const int tmax = (warp * 32 + 31) / R;   // last token of this warp's rows
#pragma unroll
                    for (int c32 = 0; c32 < QR; c32 += 32) {
                        float v[32];
                        if (c32 / R <= tmax) {   // warp-uniform
                            tmem_ld32_sync(tlane + K::T_S + c32, v);
                        } else {
#pragma unroll
                            for (int i4 = 0; i4 < 32; ++i4) v[i4] = 0.f;
                        }
                        mask_block<R>(v, c32, t, ct, rt, cum2, co + K::CO_BNEG, co + K::CO_CG);
                        mask_block<R>(v + 16, c32 + 16, t, ct, rt, cum2, co + K::CO_BNEG, co + K::CO_CG);
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            const int col = c32 + q8 * 8;
                            *reinterpret_cast<uint4*>(sl + (col / 64) * QR * 128 + sw128_offset(row, (col % 64) * 2)) =
                                make_uint4(pack_bf16(v[q8 * 8 + 0], v[q8 * 8 + 1]), pack_bf16(v[q8 * 8 + 2], v[q8 * 8 + 3]),
                                           pack_bf16(v[q8 * 8 + 4], v[q8 * 8 + 5]), pack_bf16(v[q8 * 8 + 6], v[q8 * 8 + 7]));
                        }
                    }
                    fence_proxy_async_smem();
                }
                // the previous chunk's output store has read the output tile: it may be rewritten
                if (tid == kCbxThread && i > 0) bulk_wait_read_all();
                tc_fence_before();
                group_bar(1);
                M3_TRACE_C(i, 4);
                if (tid == 0) {   // Y = SL X, then the next chunk's scores if its rotation is done
                    tc_fence_after();
                    const uint64_t dSL = smem_desc(smem_u32(sl), 16, 1024, kSwizzle128B);
                    const uint64_t dX = smem_desc(smem_u32(tile_x(s)), 16, 1024, kSwizzle128B);
                    constexpr uint32_t id_y = idesc_bf16_f32(K::MM, P, false, true);
#pragma unroll
                    for (int kk = 0; kk < QR / 16; ++kk) {
                        const uint32_t ko = ((kk >> 2) * QR * 128 + (kk & 3) * 32) >> 4;
                        mma_bf16_ss(tmem + K::T_Y, dSL + ko, dX + kk * (2048 >> 4), id_y, kk > 0);
                    }
                    mma_commit(&ctl->bY);
                    if (i + 1 < nl && !*fail_c && mbar_test_wait(&ctl->bc_done[s ^ 1], ((i + 1) >> 1) & 1)) {
                        tc_fence_after();
                        issue_scores(s ^ 1);
                        s_next = i + 2;
                    }
                    M3_TRACE_C(i, 5);
#ifdef M3_TRACE
                    if (blockIdx.x < kTraceCtas && i < kTraceChunks)
                        g_m3_trace[((int)blockIdx.x * kTraceChunks + i) * kTraceSlots + 10] = s_next == i + 2;
#endif
                }
                // ---- output rows (t, r) once Yi and Y are done; C, B, X of chunk i+2 may then come in
                (void)wait_bounded(&ctl->bY, i & 1, fail_c, fail_r);
                M3_TRACE_BY(32, i, 11);
                M3_TRACE_C(i, 6);
                tc_fence_after();
                if (tid == kCbxThread && i + 2 < nl && !*fail_c) {
                    load_cbx(i + 2, s);
                }
                // into the output tile (row (t, r) = t R + r, as x's tile; rows past the sequence's end
                // are not stored)
                if constexpr (K::M64) {
                    const int row = warp * 16 + (lane & 15), half = lane >> 4;
                    const float2 e2 = make_float2(ecum_t, ecum_t);
                    float yv[32], iv[32];
                    tmem_ld16x2x2_sync(tlane + K::T_Y, tlane + K::T_YI, yv, iv);
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        float2 o = __ffma2_rn(e2, make_float2(iv[2 * q], iv[2 * q + 1]),
                                              make_float2(yv[2 * q], yv[2 * q + 1]));
                        if constexpr (GATE) {   // y * silu(z)
                            const uint32_t zw = word_at(zg, q);
                            o = make_float2(o.x * silu_f(bf_lo(zw)), o.y * silu_f(bf_hi(zw)));
                        }
                        pk[q] = pack_bf16(o.x, o.y);
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<uint4*>(out_tile + sw128_offset(row, (32 * half + 8 * q4) * 2)) =
                            make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    fence_proxy_async_smem();
                } else if (warp * 32 < QR) {
                    const int row = tid;
                    const float2 e2 = make_float2(ecum_t, ecum_t);
#pragma unroll
                    for (int cc = 0; cc < P; cc += 32) {
                        float yv[32], iv[32];
                        tmem_ld32x2_sync(tlane + K::T_Y + cc, tlane + K::T_YI + cc, yv, iv);
                        uint32_t pk[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            float2 o = __ffma2_rn(e2, make_float2(iv[2 * q], iv[2 * q + 1]),
                                                  make_float2(yv[2 * q], yv[2 * q + 1]));
                            if constexpr (GATE) {   // y * silu(z)
                                const uint32_t zw = word_at(zg, cc / 2 + q);
                                o = make_float2(o.x * silu_f(bf_lo(zw)), o.y * silu_f(bf_hi(zw)));
                            }
                            pk[q] = pack_bf16(o.x, o.y);
                        }
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            *reinterpret_cast<uint4*>(out_tile + sw128_offset(row, (cc + 8 * q4) * 2)) =
                                make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    }
                    fence_proxy_async_smem();
                }
                M3_TRACE_C(i, 7);
            } else {
                // B'' and X are consumed: the next loads may come in
                if (tid == kCbxThread && i + 2 < nl && !*fail_c) {
                    load_cbx(i + 2, s);
                }
                if (tid == 0) ld_sum += co[K::CO_CEND];
            }

            if constexpr (!STEP_AT_TOP) {   // into the next chunk: its decay (none after the last)
                // Hb = bf16(H) needs no decay: it goes out before the wait for the next chunk's
                // coefficients, and the last 32 columns stay in registers for the scaling
                tc_fence_after();
                float hv[32];
#pragma unroll
                for (int cc = 0; cc < HCOLS; cc += 32) {
                    h_ld(cc, hv);
                    if (FULL) hb_write(cc, hv);
                }
                float e_next = 1.f;
                if (i + 1 < nl) {
                    const int s1 = (i + 1) & 1;
                    (void)wait_bounded(&ctl->coef_ready[s1], ((i + 1) >> 1) & 1, fail_c, fail_r);
                    e_next = coef(s1)[K::CO_EEND];
                }
                M3_TRACE_C(i, 14);
                h_scale_st(HCOLS - 32, hv, e_next);
#pragma unroll
                for (int cc = 0; cc < HCOLS - 32; cc += 32) {
                    float hv2[32];
                    h_ld(cc, hv2);
                    h_scale_st(cc, hv2, e_next);
                }
                tmem_st_wait();
                if (FULL) fence_proxy_async_smem();
            }
            // every read of this stage's coefficient block is done (the output took exp(cum_t)
            // in a register): the rotate group may fill it for chunk i+2.  (The next chunk's barrier,
            // after its rot_done wait, orders the state step's writes before its MMAs.)
            mbar_arrive(&ctl->coef_free[s]);
            M3_TRACE_C(i, 15);
        }
        if constexpr (FULL) {   // the last chunk's outputs (the loop ends, or breaks, uniformly)
            group_bar(1);
            if (tid == kCbxThread) {
                if (!*fail_c && nl > 0) store_y(nl - 1);
                bulk_wait_all();   // the output tile stays until the stores have read it
            }
        }
        // the carry after the segment's last chunk (no decay after it), rotated from the segment's frame
        // to the physical frame by the segment's phase Theta (the last chunk's phase, mod 2 pi)
        const float* co_last = coef((nl - 1) & 1);
        float* dst = nullptr;
        if (FULL) {
            if (seg == args.nseg - 1) dst = args.final_state;
            if (dst != nullptr) dst += (int64_t)bh * NS * P;
        } else {
            dst = args.seg_U + ((int64_t)bh * (args.S - 1) + seg) * NS * P;
            if (!*fail_c && !*fail_r) {
                if (tid == 0) args.seg_ld[(int64_t)bh * (args.S - 1) + seg] = ld_sum;
                if (tid < NP2) args.seg_th[((int64_t)bh * (args.S - 1) + seg) * NP2 + tid] = co_last[K::CO_THETA + tid];
            }
        }
        if (!*fail_c && !*fail_r && dst != nullptr) {
            tc_fence_after();
            float sn, cs;
            sincosf(co_last[K::CO_THETA + (hrow >> 1)], &sn, &cs);
            // even row 2j: cos*v_2j - sin*v_2j+1 ; odd row 2j+1: sin*v_2j + cos*v_2j+1 (row 2j+1 is in the
            // next lane, the same columns, with either carry layout)
            const float2 c2 = make_float2(cs, cs);
            const float2 s2 = (hrow & 1) ? make_float2(sn, sn) : make_float2(-sn, -sn);
            float* fs = dst + (int64_t)hrow * P + hc0;
#pragma unroll
            for (int cc = 0; cc < HCOLS; cc += 32) {
                float v[32];
                h_ld(cc, v);
#pragma unroll
                for (int i2 = 0; i2 < 32; i2 += 2) {
                    const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, v[i2], 1),
                                                 __shfl_xor_sync(0xffffffffu, v[i2 + 1], 1));
                    const float2 r = __ffma2_rn(c2, make_float2(v[i2], v[i2 + 1]), __fmul2_rn(s2, o));
                    v[i2] = r.x;
                    v[i2 + 1] = r.y;
                }
#pragma unroll
                for (int i4 = 0; i4 < 32; i4 += 4)
                    *reinterpret_cast<float4*>(fs + cc + i4) = make_float4(v[i4], v[i4 + 1], v[i4 + 2], v[i4 + 3]);
            }
        }
    } else {
        // =============================== rotate ===============================
        const int rt = tid - 128, rw = rt >> 5;
        float* sW = reinterpret_cast<float*>(sm + K::OFF_RPRIV);
        float* sWarpR = sW + Q;
        const int jg = rt % NG, tg = rt / NG;
        const int pan = jg / 8, cib = (jg % 8) * 16;     // panel and byte-in-row of my 16-byte piece
        const float* om_base = args.omega + ((int64_t)b * T * args.H + h) * NP2 + 4 * jg;
        const int64_t om_tok = (int64_t)args.H * NP2;
        float4 om[TPG];
        auto load_omega = [&](int c) {
#pragma unroll
            for (int k = 0; k < TPG; ++k) {
                const int t = c * Q + tg * TPG + k;
                om[k] = t < T ? *reinterpret_cast<const float4*>(om_base + t * om_tok) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        load_omega(c_begin);
        // phase of this thread's 4 pairs at the end of the previous chunk, since the segment start (mod 2 pi)
        float4 phi0 = make_float4(0.f, 0.f, 0.f, 0.f);
        const float a = PREP ? 0.f : args.A[h];
        // pre-activation variant: this thread's token's decay generator, one chunk ahead
        float a_nx = 0.f;
        const float bias = PREP && args.dt_bias != nullptr ? args.dt_bias[h] : 0.f;
        auto load_a = [&](int c) {
            const int t = c * Q + rt;
            return rt < Q && t < T ? args.A[((int64_t)b * T + t) * args.H + h] : 0.f;
        };
        if (PREP) a_nx = load_a(c_begin);
        // B / C normalisation: this thread's 8 channels' gains, and with one rank its head's biases
        BcRegs<BC> bcr;
        if constexpr (BC) {
            load8(ext.B_gain ? ext.B_gain + 8 * jg : nullptr, 1.f, bcr.gB);
            load8(FULL && ext.C_gain ? ext.C_gain + 8 * jg : nullptr, 1.f, bcr.gC);
            load8(R == 1 && ext.B_bias ? ext.B_bias + (int64_t)h * NS + 8 * jg : nullptr, 0.f, bcr.bB1);
            load8(R == 1 && FULL && ext.C_bias ? ext.C_bias + (int64_t)h * NS + 8 * jg : nullptr, 0.f, bcr.bC1);
        }
        for (int i = 0; i < nl; ++i) {
            const int c = c_begin + i, s = i & 1;
            M3_TRACE_R(i, 0);
            // every thread waits for the boxes itself; a failure is acted on at the next group barrier
            const bool got_box = wait_bounded(&ctl->fbox[s], (i >> 1) & 1, fail_r, fail_c);
            if (rt == 0 && got_box) ctl->box_waited[s] += 1;
            float a_t = a;
            if constexpr (PREP) {
                // Delta and lambda of this head's Q+1 staged tokens, in place (0 past the end)
                for (int k = rt; k <= Q; k += 128) {
                    const bool in = (int64_t)c * Q + k < T;
                    float* pd = box_dt(s) + k * 4 + hq;
                    float* pl = box_lam(s) + k * 4 + hq;
                    *pd = in ? softplus_f(*pd + bias) : 0.f;
                    *pl = in ? sigmoid_f(*pl) : 0.f;
                }
                a_t = a_nx;
                group_bar(2);
            }
            M3_TRACE_R(i, 1);
            const float* sDt = box_dt(s);
            const float* sLam = box_lam(s);
            float* co = coef(s);
            float* sPart = K::PART_IN_BOX ? box_dt(s) : reinterpret_cast<float*>(sm + K::OFF_PART);

            // ---- every value the chunk needs from the boxes, into registers
            float d = 0.f, l = 0.f, dn = 0.f, ln = 0.f;
            if (rt < Q) {
                d = sDt[rt * 4 + hq];
                l = sLam[rt * 4 + hq];
                dn = sDt[(rt + 1) * 4 + hq];
                ln = sLam[(rt + 1) * 4 + hq];
            }
            float dtk[TPG];
#pragma unroll
            for (int k = 0; k < TPG; ++k) dtk[k] = sDt[(tg * TPG + k) * 4 + hq];
            // ---- coefficients and chunk-local log-decay prefix
            const float ell = d * a_t, gam = l * d, wv = gam + (1.f - ln) * dn;
            float cum = warp_inclusive_sum(ell);
            M3_TRACE_R(i, 9);
            if (lane == 31) sWarpR[rw] = cum;
            // the consumer is done with chunk i-2's coefficients in this stage
            if (i >= 2) (void)wait_bounded(&ctl->coef_free[s], ((i - 2) >> 1) & 1, fail_r, fail_c);
            group_bar(2);   // every box value is read (the boxes may now hold partial sums)
            if (*fail_r) break;   // set only inside this group's waits, all before the barrier
            M3_TRACE_R(i, 10);
            float off = 0.f, cend = 0.f;
            for (int k = 0; k < 4; ++k) {
                const float v = sWarpR[k];
                if (k < rw) off += v;
                cend += v;
            }
            cum += off;
            if (rt < Q) {
                // g = log2 of the decay from this token to the chunk's end, clamped at -100: B is
                // scaled by it here (B'' = 2^g w R(-Psi) B, the chunk state's weight), and the mask
                // divides the scores by it again (every mask factor stays <= 2^100)
                const float g = fmaxf((cend - cum) * kLog2e, -100.f);
                if (FULL) {
                    co[K::CO_CUM2 + rt] = cum * kLog2e;
                    co[K::CO_CG + rt] = fmaf(cum, kLog2e, g);
                    co[K::CO_RHO + rt] = (wv > 0.f ? __fdividef(gam, wv) : 0.f) * ex2_approx(-g);
                    co[K::CO_ECUM + rt] = __expf(cum);
                }
                sW[rt] = wv * ex2_approx(g);
            }
            if (rt == 0) {
                co[K::CO_EEND] = __expf(cend);
                co[K::CO_CEND] = cend;
            }
            M3_TRACE_R(i, 11);
            // ---- rotation angles: partial sums per token group
            {
                float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < TPG; ++k) {
                    part.x = fmaf(dtk[k], om[k].x, part.x);
                    part.y = fmaf(dtk[k], om[k].y, part.y);
                    part.z = fmaf(dtk[k], om[k].z, part.z);
                    part.w = fmaf(dtk[k], om[k].w, part.w);
                }
                *reinterpret_cast<float4*>(&sPart[tg * NP2 + 4 * jg]) = part;
            }
            M3_TRACE_R(i, 12);
            group_bar(2);   // coefficient block and partial sums written
            M3_TRACE_R(i, 13);
            if (FULL && rt < Q) {   // b_s of the mask: 2^(cum2[last token of s's 16-column block] - cum2[s])
                const int e_tok = ((rt * R) / 16 * 16 + 15) / R;
                co[K::CO_BNEG + rt] = ex2_approx(co[K::CO_CUM2 + e_tok] - co[K::CO_CG + rt]);
            }
            // exclusive prefix of the token groups' partial sums: every load issued together
            float4 psi = phi0;
            {
                float4 p4[TG - 1];
#pragma unroll
                for (int g = 0; g < TG - 1; ++g)
                    p4[g] = g < tg ? *reinterpret_cast<const float4*>(&sPart[g * NP2 + 4 * jg])
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int g = 0; g < TG - 1; ++g) {
                    psi.x += p4[g].x; psi.y += p4[g].y; psi.z += p4[g].z; psi.w += p4[g].w;
                }
            }
            // ---- rotate C and B in place once they have landed.  C and B of chunk i+2
            //      are issued only after batch 1 of chunk i, so waiting for them here keeps
            //      this group at most one chunk ahead of the consumer: every barrier the
            //      consumer waits on is then at most one phase ahead.
            M3_TRACE_R(i, 2);
            const bool got_cb = wait_bounded(&ctl->fcbx[s], (i >> 1) & 1, fail_r, fail_c);
            M3_TRACE_R(i, 3);
            if (rt == 0 && got_cb) ctl->cbx_waited[s] += 1;
            // the consumer may use this chunk's coefficients (exp(cum_end), f) now
            mbar_arrive(&ctl->coef_ready[s]);
            {
                uint8_t* tC = tile_c(s);
                uint8_t* tB = tile_b(s);
                // tokens per batch of the plain rotation: the loads of a batch's 8 row pieces go out
                // together, ahead of their stores (the compiler cannot tell the in-place stores from
                // the next pieces' loads)
                constexpr int TB = BC || R >= 2 ? 1 : 2;
                static_assert(TPG % TB == 0, "token batches must divide the token group");
#pragma unroll
                for (int k0 = 0; k0 < TPG; k0 += TB) {
                uint4 vc[TB * R], vb[TB * R];
                float wb[TB];
                if constexpr (!BC) {
#pragma unroll
                    for (int kb = 0; kb < TB; ++kb) {
                        const int t = tg * TPG + k0 + kb;
                        wb[kb] = sW[t];
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t off2 = pan * QR * 128 + sw128_offset(t * R + r, cib);
                            if (FULL) vc[kb * R + r] = *reinterpret_cast<const uint4*>(tC + off2);
                            vb[kb * R + r] = *reinterpret_cast<const uint4*>(tB + off2);
                        }
                    }
                }
#pragma unroll
                for (int kb = 0; kb < TB; ++kb) {
                    const int k = k0 + kb;
                    const int t = tg * TPG + k;
                    psi.x = fmaf(dtk[k], om[k].x, psi.x);
                    psi.y = fmaf(dtk[k], om[k].y, psi.y);
                    psi.z = fmaf(dtk[k], om[k].z, psi.z);
                    psi.w = fmaf(dtk[k], om[k].w, psi.w);
                    float cs[4], sn[4];
                    __sincosf(-psi.x, &sn[0], &cs[0]);
                    __sincosf(-psi.y, &sn[1], &cs[1]);
                    __sincosf(-psi.z, &sn[2], &cs[2]);
                    __sincosf(-psi.w, &sn[3], &cs[3]);
                    const float wt = BC ? sW[t] : wb[kb];
                    const float2 c01[2] = {make_float2(cs[0], cs[1]), make_float2(cs[2], cs[3])};
                    const float2 s01[2] = {make_float2(sn[0], sn[1]), make_float2(sn[2], sn[3])};
                    const float2 w2 = make_float2(wt, wt);
                    const float2 cw01[2] = {__fmul2_rn(w2, c01[0]), __fmul2_rn(w2, c01[1])};
                    const float2 sw01[2] = {__fmul2_rn(w2, s01[0]), __fmul2_rn(w2, s01[1])};
                    if constexpr (BC) {
                        // every row of this token (C and B of each rank) into registers first, their
                        // sums of squares reduced together (independent shuffle chains), then each
                        // row normalised, biased, rotated (B' also scaled by w) and stored
                        constexpr int NR = FULL ? 2 * R : R;
                        uint4 vr[NR];
                        float ss[NR];
                        const bool bc_norm = ext.bc_norm != 0;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t off2 = pan * QR * 128 + sw128_offset(t * R + r, cib);
                            if (FULL) vr[2 * r] = *reinterpret_cast<const uint4*>(tC + off2);
                            vr[FULL ? 2 * r + 1 : r] = *reinterpret_cast<const uint4*>(tB + off2);
                        }
                        if (bc_norm) {
#pragma unroll
                            for (int i = 0; i < NR; ++i) ss[i] = sumsq8(vr[i]);
#pragma unroll
                            for (int o = 1; o < NG; o <<= 1) {
#pragma unroll
                                for (int i = 0; i < NR; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
                            }
#pragma unroll
                            for (int i = 0; i < NR; ++i) ss[i] = rsqrtf(fmaf(ss[i], 1.f / NS, ext.bc_eps));
                        }
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t off2 = pan * QR * 128 + sw128_offset(t * R + r, cib);
                            float bbB[8], bbC[8];
                            if (R == 1) {
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    bbB[q] = bcr.bB1[q];
                                    bbC[q] = bcr.bC1[q];
                                }
                            } else {
                                load8(ext.B_bias ? ext.B_bias + ((int64_t)h * R + r) * NS + 8 * jg : nullptr, 0.f, bbB);
                                if (FULL)
                                    load8(ext.C_bias ? ext.C_bias + ((int64_t)h * R + r) * NS + 8 * jg : nullptr, 0.f,
                                          bbC);
                            }
                            if (FULL)
                                *reinterpret_cast<uint4*>(tC + off2) =
                                    bc_rotate4(vr[2 * r], c01, s01, bcr.gC, bbC, bc_norm, bc_norm ? ss[2 * r] : 1.f);
                            const int ib = FULL ? 2 * r + 1 : r;
                            *reinterpret_cast<uint4*>(tB + off2) =
                                bc_rotate4(vr[ib], cw01, sw01, bcr.gB, bbB, bc_norm, bc_norm ? ss[ib] : 1.f);
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t off2 = pan * QR * 128 + sw128_offset(t * R + r, cib);
                            if (FULL) *reinterpret_cast<uint4*>(tC + off2) = rotate4(vc[kb * R + r], c01, s01);
                            *reinterpret_cast<uint4*>(tB + off2) = rotate4(vb[kb * R + r], cw01, sw01);
                        }
                    }
                }
                }
                // the phase at the chunk's last token: the next chunk starts from it
                if (tg == TG - 1) *reinterpret_cast<float4*>(&co[K::CO_THETA + 4 * jg]) = reduce_2pi(psi);
            }
            // C~ and B' are in place: the consumer may issue this chunk's scores
            fence_proxy_async_smem();
            mbar_arrive(&ctl->bc_done[s]);
            M3_TRACE_R(i, 4);
            if (i + 1 < nl) {
                load_omega(c + 1);
                if (PREP) a_nx = load_a(c + 1);
            }
            if constexpr (K::PART_IN_BOX) group_bar(2);   // partial sums read: the box may take chunk i+2
            M3_TRACE_R(i, 5);
            M3_TRACE_R(i, 6);
            M3_TRACE_R(i, 7);
            mbar_arrive(&ctl->rot_done[s]);
            group_bar(2);   // sW is reused by the next chunk; the chunk-end phase Theta is written
            M3_TRACE_R(i, 8);
            if (*fail_r) break;
            phi0 = *reinterpret_cast<const float4*>(&co[K::CO_THETA + 4 * jg]);
            // the boxes' values and (without PART_IN_BOX) nothing else of the stage's boxes is still read
            if (rt == 0 && i + 2 < nl) load_box(i + 2, s);
        }
    }

    // ------------------------------- teardown -------------------------------
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && (ctl->fail_c || ctl->fail_r)) {
        atomicExch(args.status, (int)M3_ERR_TIMEOUT);
        // let copies and MMAs still in flight finish (bounded) before the shared
        // memory and TMEM go away
        auto drain = [&](uint64_t* bar, uint16_t waited, uint16_t issued) {
            const uint16_t n = (uint16_t)(issued - waited);
            for (uint16_t j = 0; j < n && j < 4; ++j) (void)mbar_wait(bar, (uint32_t)((waited + j) & 1), kWaitLimitNs);
        };
        for (int s = 0; s < 2; ++s) {
            drain(&ctl->fbox[s], ctl->box_waited[s], ctl->box_issued[s]);
            drain(&ctl->fcbx[s], ctl->cbx_waited[s], ctl->cbx_issued[s]);
        }
        // thread 0 issued every MMA: a commit arrives once all of them are complete
        mma_commit(&ctl->drain);
        (void)mbar_wait(&ctl->drain, 0, kWaitLimitNs);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, K::TMEM_COLS);
#ifdef M3_TRACE
    if (tid == 0 && blockIdx.x < kClkCtas) {
        g_m3_trace_clk[blockIdx.x * kClkSlots + 2] = (long long)globaltimer_ns();
        g_m3_trace_clk[blockIdx.x * kClkSlots + 3] = clock64();
    }
#endif
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

// Sequence segments: with fewer (batch, head) sequences than CTA slots on the
// GPU, each sequence is cut into S segments of L chunks so that the machine
// fills up; a state pass gives every segment's carry from a zero start, the
// segment scan (m3_state_passing's kernel) turns those into the state entering
// each segment, and the full pass starts each segment from it.  The state pass
// has no scores or outputs, so its tiles can be longer at two CTAs per SM: with
// R >= 2 it takes chunks of 128 / R tokens (128 rows), twice the full pass's,
// and segments hold an even number of the full pass's chunks.
constexpr int kPlanSMs = 148;   // SMs of the B300 the plan is sized for (fixed: the workspace size must not depend on the device)

template <int R, int Q>
constexpr int state_pass_q() { return R >= 2 && 2 * Q * R <= 128 ? 2 * Q : Q; }

struct SegPlan {
    int S, L, nc;
};

template <int NS, int R, int Q>
SegPlan seg_plan(const ScanDims& d) {
    using K = Cfg<NS, R, Q>;
    constexpr int F = state_pass_q<R, Q>() / Q;
    SegPlan p;
    p.nc = (int)((d.seqlen + Q - 1) / Q);
    const int64_t seqs = d.batch * d.nheads, slots = (int64_t)kPlanSMs * K::MIN_BLOCKS;
    int64_t S = seqs >= slots ? 1 : slots / seqs;
    if (S > p.nc) S = p.nc;
    if (S < 1) S = 1;
    p.L = (int)((p.nc + S - 1) / S);
    if (S > 1) p.L = (p.L + F - 1) / F * F;   // whole state-pass chunks per segment
    p.S = (p.nc + p.L - 1) / p.L;   // no empty segment
    return p;
}

struct SegWs {
    size_t status, U, ld, th, last, total;
};

inline size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

template <int NS, int R, int Q>
SegWs seg_ws(const ScanDims& d) {
    const SegPlan p = seg_plan<NS, R, Q>(d);
    const size_t seqs = (size_t)(d.batch * d.nheads), P = (size_t)d.headdim, S1 = (size_t)(p.S - 1);
    SegWs w;
    w.status = 0;
    w.U = 256;
    w.ld = w.U + (p.S > 1 ? al256(S1 * seqs * NS * P * 4) : 0);
    w.th = w.ld + (p.S > 1 ? al256(S1 * seqs * 4) : 0);
    w.last = w.th + (p.S > 1 ? al256(S1 * seqs * (NS / 2) * 4) : 0);
    w.total = w.last + (p.S > 1 ? al256(seqs * NS * P * 4) : 0);
    return w;
}

// The five tensor maps of chunks of QT tokens: x, B, C (boxes of QT tokens x R ranks x 64
// channels, 128-byte swizzle) and dt, lambda (boxes of 4 heads x QT+1 tokens).
struct Maps {
    CUtensorMap x, B, C, dt, lam;
};

template <int R>
bool make_maps(Maps& m, const ScanDims& d, int QT, const void* x, const void* B, const void* C, const float* dt,
               const float* lambda) {
    const cuuint64_t Bt = d.batch, T = d.seqlen, H = d.nheads, P = d.headdim, N = d.dstate;
    {
        cuuint64_t dims[5] = {P, (cuuint64_t)R, H, T, Bt};
        cuuint64_t str[4] = {P * 2, R * P * 2, H * R * P * 2, T * H * R * P * 2};
        cuuint32_t box[5] = {64, (cuuint32_t)R, 1, (cuuint32_t)QT, 1};
        if (!make_map(&m.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, x, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
    }
    {
        cuuint64_t dims[5] = {N, (cuuint64_t)R, H, T, Bt};
        cuuint64_t str[4] = {N * 2, R * N * 2, H * R * N * 2, T * H * R * N * 2};
        cuuint32_t box[5] = {64, (cuuint32_t)R, 1, (cuuint32_t)QT, 1};
        if (!make_map(&m.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
        if (!make_map(&m.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, C, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
    }
    {
        cuuint64_t dims[3] = {H, T, Bt};
        cuuint64_t str[2] = {H * 4, T * H * 4};
        cuuint32_t box[3] = {4, (cuuint32_t)(QT + 1), 1};
        if (!make_map(&m.dt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dt, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
        if (!make_map(&m.lam, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, lambda, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
    }
    return true;
}

template <int NS, int R, int Q, int PM>
cudaError_t launch_cfg(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                       const float* A, const float* lambda, const float* omega, void* y, float* final_state,
                       void* workspace, const Prep& prep, cudaStream_t stream) {
    using K = Cfg<NS, R, Q>;
    constexpr int QS = state_pass_q<R, Q>();
    using KS = Cfg<NS, R, QS, false>;
    const cuuint64_t P = d.headdim;
    Maps mf;
    if (!make_maps<R>(mf, d, Q, x, B, C, dt, lambda)) return cudaErrorInvalidValue;
    CUtensorMap my;   // y as x: tiles of Q tokens x R ranks x 64 channels, 128-byte swizzle
    {
        const cuuint64_t Bt = d.batch, T = d.seqlen, H = d.nheads;
        cuuint64_t dims[5] = {P, (cuuint64_t)R, H, T, Bt};
        cuuint64_t str[4] = {P * 2, R * P * 2, H * R * P * 2, T * H * R * P * 2};
        cuuint32_t box[5] = {64, (cuuint32_t)R, 1, (cuuint32_t)Q, 1};
        if (!make_map(&my, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, y, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const SegPlan pl = seg_plan<NS, R, Q>(d);
    const SegWs ws = seg_ws<NS, R, Q>(d);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    const int64_t seqs = d.batch * d.nheads;
    TcArgs args{};
    args.A = A;
    args.dt_bias = prep.dt_bias;
    ExtArgs<PM> ext{};
    if constexpr (PM == kTestHook)
        ext.fail_chunk = prep.test_timeout_at - 1;
    else if constexpr (PM != 0)
        ext = ExtArgs<PM>{prep.B_gain, prep.C_gain, prep.B_bias, prep.C_bias, prep.bc_norm ? 1 : 0, prep.bc_eps,
                          static_cast<const __nv_bfloat16*>(prep.z)};
    args.omega = omega;
    args.y = static_cast<__nv_bfloat16*>(y);
    args.final_state = final_state;
    args.status = reinterpret_cast<int*>(wsb + ws.status);
    args.T = (int)d.seqlen;
    args.H = (int)d.nheads;
    args.nc = pl.nc;
    args.L = pl.L;
    args.S = pl.S;
    cudaError_t e = cudaMemsetAsync(args.status, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
    if (pl.S > 1) {
        float* segU = reinterpret_cast<float*>(wsb + ws.U);
        float* segLD = reinterpret_cast<float*>(wsb + ws.ld);
        float* segTH = reinterpret_cast<float*>(wsb + ws.th);
        float* last = reinterpret_cast<float*>(wsb + ws.last);
        Maps ms;
        if (QS == Q) ms = mf;
        else if (!make_maps<R>(ms, d, QS, x, B, C, dt, lambda)) return cudaErrorInvalidValue;
        TcArgs a1 = args;
        // the same segments in the state pass's chunks (segments 0 .. S-2 hold L whole chunks of Q tokens)
        a1.nc = (int)((d.seqlen + QS - 1) / QS);
        a1.L = pl.L * Q / QS;
        a1.nseg = pl.S - 1;
        a1.seg_U = segU;
        a1.seg_ld = segLD;
        a1.seg_th = segTH;
        auto k1 = scan_tc_kernel<NS, R, QS, false, PM>;
        e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, KS::SMEM);
        if (e != cudaSuccess) return e;
        k1<<<(unsigned)(seqs * a1.nseg), KS::kThreads, KS::SMEM, stream>>>(ms.x, ms.B, ms.C, ms.dt, ms.lam, ms.x, a1,
                                                                           ext);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // segment carries -> the state entering each segment (in place), and into the last one
        e = launch_state_passing(segU, segLD, segTH, nullptr, last, 1, seqs, pl.S - 1, NS, (int64_t)P, stream);
        if (e != cudaSuccess) return e;
        args.h_in = segU;
        args.h_in_last = last;
    }
    args.nseg = pl.S;
    auto kern = scan_tc_kernel<NS, R, Q, true, PM>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(seqs * pl.S), K::kThreads, K::SMEM, stream>>>(mf.x, mf.B, mf.C, mf.dt, mf.lam, my, args, ext);
    return cudaGetLastError();
}

template <int NS, int R, int Q>
size_t ws_cfg(const ScanDims& d) { return seg_ws<NS, R, Q>(d).total; }
template <int NS, int R, int Q>
int launches_cfg(const ScanDims& d) { return seg_plan<NS, R, Q>(d).S > 1 ? 3 : 1; }

typedef cudaError_t (*LaunchFn)(const ScanDims&, const void*, const void*, const void*, const float*, const float*,
                                const float*, const float*, void*, float*, void*, const Prep&, cudaStream_t);
struct TcImpl {
    // by kernel mode: 0 = dt, lambda, A[H] as given; bit 0 = pre-activations, A per token;
    // bit 1 = B / C normalisation; bit 2 = output gate (modes 0, 1, 3, 5, 7)
    LaunchFn launch[8];
    size_t (*workspace)(const ScanDims&);
    int (*launches)(const ScanDims&);
    LaunchFn hook;   // the plain kernel with the failure-path test's simulated timeout (one shape only)
};

template <int NS, int R, int Q>
TcImpl impl() {
    return TcImpl{{launch_cfg<NS, R, Q, 0>, launch_cfg<NS, R, Q, 1>, nullptr, launch_cfg<NS, R, Q, 3>, nullptr,
                   launch_cfg<NS, R, Q, 5>, nullptr, launch_cfg<NS, R, Q, 7>},
                  ws_cfg<NS, R, Q>, launches_cfg<NS, R, Q>, nullptr};
}

// Tile configuration for (N, R, chunk).  Every chunk runs as sub-chunks of 64 / R tokens -- 64-row
// tiles, the MIMO chunk-length reduction of section 3.3 taken to one tile shape -- so that two CTAs
// fit on an SM (measured faster than 128-row tiles at one CTA per SM for every workload here); the
// state passes between sub-chunks exactly as between chunks, and the result differs only in rounding.
bool pick(const ScanDims& d, TcImpl* out) {
    if (d.headdim != 64 || d.io != M3_DTYPE_BF16) return false;
    if (d.nheads % 4) return false;
    if (d.chunk != 64 && d.chunk != 128) return false;
    const int N = (int)d.dstate, R = d.R;
    TcImpl f{};
    if (N == 128 && R == 1) {
        f = impl<128, 1, 64>();
        f.hook = launch_cfg<128, 1, 64, kTestHook>;
    } else if (N == 128 && R == 2) f = impl<128, 2, 32>();
    else if (N == 128 && R == 4) f = impl<128, 4, 16>();
    else if (N == 64 && R == 1) f = impl<64, 1, 64>();
    else if (N == 64 && R == 2) f = impl<64, 2, 32>();
    else if (N == 64 && R == 4) f = impl<64, 4, 16>();
    else return false;
    if (out) *out = f;
    return true;
}

}  // namespace

size_t tc_workspace_size(const ScanDims& d) {
    TcImpl f;
    return pick(d, &f) ? f.workspace(d) : 0;
}
bool tc_supported(const ScanDims& d) { return d.seqlen > 0 && pick(d, nullptr); }
int tc_launch_count(const ScanDims& d) {
    TcImpl f;
    return pick(d, &f) ? f.launches(d) : 0;
}
cudaError_t launch_scan_tc(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                           const float* A, const float* lambda, const float* omega, void* y, float* final_state,
                           void* workspace, const Prep& prep, cudaStream_t stream) {
    TcImpl f;
    if (!pick(d, &f)) return cudaErrorNotSupported;
    const int mode = !prep.on ? 0 : 1 | (prep.bc() ? 2 : 0) | (prep.z != nullptr ? 4 : 0);
    if (mode == 0 && prep.test_timeout_at > 0 && f.hook != nullptr)
        return f.hook(d, x, B, C, dt, A, lambda, omega, y, final_state, workspace, prep, stream);
    return f.launch[mode](d, x, B, C, dt, A, lambda, omega, y, final_state, workspace, prep, stream);
}

}  // namespace m3

#ifdef M3_TRACE
// Diagnostic build only: copy out (or clear, dst = NULL) the phase trace; n = number of int64 entries of
// the trace (kTraceCtas * kTraceChunks * kTraceSlots) followed by the per-CTA clocks (kClkCtas * kClkSlots).
extern "C" __attribute__((visibility("default"))) int m3_trace_read(long long* dst, int n) {
    using namespace m3;
    constexpr int nt = kTraceCtas * kTraceChunks * kTraceSlots, nc = kClkCtas * kClkSlots;
    if (n != nt + nc) return M3_ERR_INVALID_ARG;
    if (dst == nullptr) {
        void *pt = nullptr, *pc = nullptr;
        if (cudaGetSymbolAddress(&pt, g_m3_trace) != cudaSuccess) return M3_ERR_CUDA;
        if (cudaGetSymbolAddress(&pc, g_m3_trace_clk) != cudaSuccess) return M3_ERR_CUDA;
        if (cudaMemset(pt, 0, sizeof(long long) * nt) != cudaSuccess) return M3_ERR_CUDA;
        if (cudaMemset(pc, 0, sizeof(long long) * nc) != cudaSuccess) return M3_ERR_CUDA;
        return cudaDeviceSynchronize() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
    }
    if (cudaMemcpyFromSymbol(dst, g_m3_trace, sizeof(long long) * nt) != cudaSuccess) return M3_ERR_CUDA;
    if (cudaMemcpyFromSymbol(dst + nt, g_m3_trace_clk, sizeof(long long) * nc) != cudaSuccess) return M3_ERR_CUDA;
    return M3_OK;
}
#endif
