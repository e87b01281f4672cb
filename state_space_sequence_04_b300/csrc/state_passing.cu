// Inter-chunk state passing of the chunked Mamba-3 prefill:
//
//   H_c = exp(l_c) R(Theta_c) H_{c-1} + U_c,   H_{-1} = init (or 0)
//
// (the chunked algorithm of "Mamba-3: Improved Sequence Modeling using State
// Space Principles", section 3.3, with the rotation of Propositions 3-4 acting
// on state rows (2j, 2j+1)).  The recurrence is elementwise over the N x P
// state, so each thread carries one pair of rows x one float4 of columns in
// fp32 registers through all chunks, streaming U_c in and H_{c-1} out in place
// with the next chunk's load issued before the current store.
#include "m3_common.cuh"

namespace m3 {
namespace {

__global__ void __launch_bounds__(256) state_passing_kernel(
    float* __restrict__ S, const float* __restrict__ ld, const float* __restrict__ ang,
    const float* __restrict__ init, float* __restrict__ fin, int nc, int N, int P) {
    const int64_t bh = blockIdx.x;
    const int P4 = P >> 2, NP2 = N >> 1;
    const int u = blockIdx.y * blockDim.x + threadIdx.x;
    if (u >= NP2 * P4) return;
    const int j = u / P4, c4 = u % P4;
    const int64_t NP4 = (int64_t)N * P4;
    const int64_t r0 = (int64_t)(2 * j) * P4 + c4, r1 = (int64_t)(2 * j + 1) * P4 + c4;

    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    if (init) {
        const float4* i4 = reinterpret_cast<const float4*>(init) + bh * NP4;
        a0 = i4[r0];
        a1 = i4[r1];
    }
    float4* S4 = reinterpret_cast<float4*>(S) + bh * nc * NP4;
    const float* ldb = ld + bh * nc;
    const float* angb = ang + bh * nc * NP2 + j;

    float4 u0 = make_float4(0.f, 0.f, 0.f, 0.f), u1 = u0;
    if (nc > 0) {
        u0 = S4[r0];
        u1 = S4[r1];
    }
    for (int c = 0; c < nc; ++c) {
        float4 n0 = u0, n1 = u1;
        if (c + 1 < nc) {
            n0 = S4[(c + 1) * NP4 + r0];
            n1 = S4[(c + 1) * NP4 + r1];
        }
        S4[c * NP4 + r0] = a0;   // the state entering chunk c
        S4[c * NP4 + r1] = a1;
        const float e = expf(ldb[c]);
        float sn, cs;
        sincosf(angb[(int64_t)c * NP2], &sn, &cs);
        float4 b0, b1;
        rot2(cs, sn, a0.x, a1.x, b0.x, b1.x);
        rot2(cs, sn, a0.y, a1.y, b0.y, b1.y);
        rot2(cs, sn, a0.z, a1.z, b0.z, b1.z);
        rot2(cs, sn, a0.w, a1.w, b0.w, b1.w);
        a0 = make_float4(fmaf(e, b0.x, u0.x), fmaf(e, b0.y, u0.y), fmaf(e, b0.z, u0.z), fmaf(e, b0.w, u0.w));
        a1 = make_float4(fmaf(e, b1.x, u1.x), fmaf(e, b1.y, u1.y), fmaf(e, b1.z, u1.z), fmaf(e, b1.w, u1.w));
        u0 = n0;
        u1 = n1;
    }
    if (fin) {
        float4* f4 = reinterpret_cast<float4*>(fin) + bh * NP4;
        f4[r0] = a0;
        f4[r1] = a1;
    }
}

}  // namespace

cudaError_t launch_state_passing(float* chunk_states, const float* chunk_logdecay, const float* chunk_angle,
                                 const float* init_state, float* final_state, int64_t batch, int64_t nheads,
                                 int64_t nchunks, int64_t dstate, int64_t headdim, cudaStream_t stream) {
    const int64_t bh = batch * nheads;
    if (bh == 0) return cudaSuccess;
    if (nchunks == 0 && final_state == nullptr) return cudaSuccess;
    const int64_t units = (dstate / 2) * (headdim / 4);
    const int threads = 256;
    dim3 grid((unsigned)bh, (unsigned)((units + threads - 1) / threads));
    state_passing_kernel<<<grid, threads, 0, stream>>>(chunk_states, chunk_logdecay, chunk_angle, init_state,
                                                       final_state, (int)nchunks, (int)dstate, (int)headdim);
    return cudaGetLastError();
}

}  // namespace m3
