// Shared device helpers of libm3 (kernels and host launchers only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/m3.h"

namespace m3 {

// ---- io element access ----------------------------------------------------
__device__ __forceinline__ float ld_io(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_io(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_io(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_io(__nv_bfloat16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// Rotate the pair (a, b) counter-clockwise by the angle whose cosine and sine are c, s.
__device__ __forceinline__ void rot2(float c, float s, float a, float b, float& oa, float& ob) {
    oa = c * a - s * b;
    ob = s * a + c * b;
}

// Inclusive prefix sum over a warp.
__device__ __forceinline__ float warp_inclusive_sum(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Per-token parameters from their pre-activations (the *_prep entry points):
// Delta = softplus(z) = log(1 + e^z), evaluated as max(z, 0) + log1p(e^-|z|);
// lambda = sigmoid(u) = 1 / (1 + e^-u) (0 for very negative u, 1 for very positive u).
__device__ __forceinline__ float softplus_f(float z) { return fmaxf(z, 0.f) + log1pf(__expf(-fabsf(z))); }
__device__ __forceinline__ float sigmoid_f(float u) { return 1.f / (1.f + __expf(-u)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace m3

// ---- host-side launchers shared between translation units ----------------
namespace m3 {

// How the per-token parameters arrive.  on = false: dt = Delta, lambda as given,
// A one value per head [H].  on = true (the *_prep entry points): dt holds the
// pre-activation of Delta (Delta = softplus(dt + dt_bias[h]), dt_bias nullable),
// lambda holds u (lambda = sigmoid(u)), and A holds one value per token with
// dt's layout.
// With on, B and C may also be RMS-normalised per (token, rank) row over N
// (bc_norm, bc_eps, gains [N]) and shifted by channel biases [H, R, N], and the
// output gated by z.
struct Prep {
    bool on;
    const float* dt_bias;
    bool bc_norm;
    float bc_eps;
    const float* B_gain;
    const float* C_gain;
    const float* B_bias;
    const float* C_bias;
    const void* z;   // output gate input (y's layout, io dtype): y <- y * silu(z); null = off
    // failure-path test (m3_test_inject): k + 1 makes the tensor-core prefill's consumer groups give up at
    // their local chunk k (plain mode, the one shape that has the test kernel); 0 = off
    int test_timeout_at;
    __host__ __device__ bool bc() const { return on && (bc_norm || B_bias != nullptr || C_bias != nullptr); }
};

// silu(z) = z / (1 + e^-z), the output gate.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.f + __expf(-z)); }

struct ScanDims {
    int64_t batch, seqlen, nheads, headdim, dstate;
    int R, chunk, io;
    int64_t nchunks() const { return (seqlen + chunk - 1) / chunk; }
};

cudaError_t launch_decode(float* state, const void* x_t, const void* B_t, void* cache, const void* C_t,
                          const float* dt_t, const float* A, const float* lambda_t, const float* omega_t,
                          void* y_t, int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate, int R,
                          int io, const Prep& prep, cudaStream_t stream);
bool decode_supported(int64_t headdim, int64_t dstate, int R);
int decode_device_status(int clear);
// the status word of the last m3_scan_fwd_noalloc call on the current device (M3_OK when it has none)
int noalloc_device_status(int clear);

cudaError_t launch_state_passing(float* chunk_states, const float* chunk_logdecay, const float* chunk_angle,
                                 const float* init_state, float* final_state, int64_t batch, int64_t nheads,
                                 int64_t nchunks, int64_t dstate, int64_t headdim, cudaStream_t stream);

// Generic CUDA-core chunked prefill (any supported size; fp32 or bf16 io).
// With prep.on the workspace also holds Delta and lambda of every token.
size_t simt_workspace_size(const ScanDims& d, bool prep);
bool simt_supported(const ScanDims& d);
cudaError_t launch_scan_simt(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                             const float* A, const float* lambda, const float* omega, void* y,
                             float* final_state, void* workspace, const Prep& prep, cudaStream_t stream);

// Backward pass (CUDA cores, fp32): workspace holds every forward state.
bool bwd_supported(const ScanDims& d);
size_t bwd_workspace_size(const ScanDims& d);
cudaError_t launch_scan_bwd(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                            const float* A, const float* lambda, const float* omega, const void* dy,
                            const float* d_final, float* dx, float* dB, float* dC, float* ddt, float* dA,
                            float* dlambda, float* domega, void* workspace, cudaStream_t stream);
size_t bwd_prep_workspace_size(const ScanDims& d);
// the B / C normalisation of m3_scan_bwd_prep: settings, parameters and their gradients (nullable)
struct BwdBcArgs {
    bool on;
    int norm;
    float eps;
    const float *B_gain, *C_gain, *B_bias, *C_bias;
    float *dB_gain, *dC_gain, *dB_bias, *dC_bias;
};
// m3_scan_bwd on pre-activations (Delta = softplus(dt_raw + dt_bias), lambda = sigmoid(u), A_t per token);
// z != nullptr: through the output gate y = y_pre silu(z), y_pre the ungated output (io dtype), dz out;
// bc.on: through the B / C normalisation
cudaError_t launch_scan_bwd_prep(const ScanDims& d, const void* x, const void* B, const void* C,
                                 const float* dt_raw, const float* dt_bias, const float* A_tok, const float* u,
                                 const float* omega, const void* dy, const float* d_final, float* dx, float* dB,
                                 float* dC, float* ddt_raw, float* dA_tok, float* du, float* domega,
                                 float* ddt_bias, const void* z, const void* y_pre, float* dz, const BwdBcArgs& bc,
                                 void* workspace, cudaStream_t stream);
// the backward through the output gate (z) fits the shared-memory budget
bool bwd_gate_supported(const ScanDims& d);
// the B / C normalisation's backward (its fp32 adjoint run) fits it
bool bwd_bc_supported(const ScanDims& d);
// Delta = softplus(dt_raw + dt_bias[h]) and lambda = sigmoid(u) of n (batch, token, head) entries
cudaError_t launch_prep_params(const float* dt_raw, const float* dt_bias, const float* u, float* dt_out,
                               float* lam_out, int64_t n, int H, cudaStream_t stream);

}  // namespace m3
