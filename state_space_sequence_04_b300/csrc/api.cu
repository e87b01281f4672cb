// C ABI of libm3: host-side validation, then launches on the caller's stream.
// Every entry point checks its arguments before touching the GPU and returns
// an m3_status; nothing is launched when a check fails.
#include <stdint.h>

#include <atomic>

#include "m3_common.cuh"

namespace m3 {

// Prefill paths other than the CUDA-core one register here (tensor-core path).
size_t tc_workspace_size(const ScanDims& d);
int tc_launch_count(const ScanDims& d);
bool tc_supported(const ScanDims& d);
cudaError_t launch_scan_tc(const ScanDims& d, const void* x, const void* B, const void* C, const float* dt,
                           const float* A, const float* lambda, const float* omega, void* y, float* final_state,
                           void* workspace, const Prep& prep, cudaStream_t stream);

}  // namespace m3

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
bool ok_nullable(const void* p) { return p == nullptr || aligned16(p); }
bool ok_io(int io) { return io == M3_DTYPE_BF16 || io == M3_DTYPE_F32; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? M3_OK : M3_ERR_CUDA; }

// Failure injection of m3_test_inject: launch failures made on the host (the next n launching calls
// return M3_ERR_CUDA after their checks), and the tensor-core prefill's simulated timeout.
std::atomic<int> g_inject_launch{0};
std::atomic<int> g_inject_timeout{0};   // k + 1: give up at local chunk k; 0 = off

// True (and one armed failure used up) when this launching call is to fail.
bool injected_launch_failure() {
    int v = g_inject_launch.load();
    while (v > 0)
        if (g_inject_launch.compare_exchange_weak(v, v - 1)) return true;
    return false;
}

// Which prefill implementation runs for these sizes: 1 = tensor cores, 0 = CUDA cores.
int pick_path(const m3::ScanDims& d) { return (d.io == M3_DTYPE_BF16 && m3::tc_supported(d)) ? 1 : 0; }

int validate_scan_sizes(const m3::ScanDims& d) {
    if (!ok_io(d.io)) return M3_ERR_INVALID_ARG;
    if (d.batch < 0 || d.seqlen < 0 || d.nheads < 1 || d.headdim < 1 || d.dstate < 2) return M3_ERR_INVALID_ARG;
    if (d.dstate % 2) return M3_ERR_INVALID_ARG;
    if (d.R < 1 || d.chunk < 1) return M3_ERR_INVALID_ARG;
    if (d.batch * d.nheads > (int64_t)INT32_MAX || d.seqlen > (int64_t)INT32_MAX) return M3_ERR_UNSUPPORTED;
    if (!m3::simt_supported(d) && !(d.io == M3_DTYPE_BF16 && m3::tc_supported(d))) return M3_ERR_UNSUPPORTED;
    return M3_OK;
}

size_t scan_workspace(const m3::ScanDims& d, bool prep) {
    return pick_path(d) == 1 ? m3::tc_workspace_size(d) : m3::simt_workspace_size(d, prep);
}

// The pre-SSM options of a _prep call (NULL params: all off); false for
// misaligned pointers or a negative / non-finite bc_eps.
bool prep_from(const m3_prep_params* p, m3::Prep* out) {
    m3::Prep q{};
    q.on = true;
    if (p != nullptr) {
        if (!ok_nullable(p->dt_bias) || !ok_nullable(p->B_gain) || !ok_nullable(p->C_gain) ||
            !ok_nullable(p->B_bias) || !ok_nullable(p->C_bias) || !ok_nullable(p->z))
            return false;
        if (!(p->bc_eps >= 0.f) || p->bc_eps > 3.0e38f) return false;
        q.dt_bias = p->dt_bias;
        q.bc_norm = p->bc_norm != 0;
        q.bc_eps = p->bc_eps;
        q.B_gain = p->B_gain;
        q.C_gain = p->C_gain;
        q.B_bias = p->B_bias;
        q.C_bias = p->C_bias;
        q.z = p->z;
    }
    *out = q;
    return true;
}

int scan_impl(const void* x, const void* B, const void* C, const float* dt, const float* A, const float* lambda,
              const float* omega, int R, int chunk, void* y, float* final_state, int64_t batch, int64_t seqlen,
              int64_t nheads, int64_t headdim, int64_t dstate, int io_dtype, void* workspace,
              size_t workspace_bytes, void* stream, const m3::Prep& prep) {
    const m3::ScanDims d{batch, seqlen, nheads, headdim, dstate, R, chunk, io_dtype};
    int st = validate_scan_sizes(d);
    if (st != M3_OK) return st;
    if (!ok_nullable(final_state) || !ok_nullable(prep.dt_bias)) return M3_ERR_INVALID_ARG;
    if (!prep.on && !ok_ptr(A)) return M3_ERR_INVALID_ARG;
    const bool any_tokens = batch > 0 && seqlen > 0;
    if (any_tokens) {
        if (!ok_ptr(x) || !ok_ptr(B) || !ok_ptr(C) || !ok_ptr(dt) || !ok_ptr(lambda) || !ok_ptr(omega) || !ok_ptr(y))
            return M3_ERR_INVALID_ARG;
        if (prep.on && !ok_ptr(A)) return M3_ERR_INVALID_ARG;
    }
    const size_t need = scan_workspace(d, prep.on);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return M3_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (batch == 0) return M3_OK;
    if (injected_launch_failure()) return M3_ERR_CUDA;
    if (pick_path(d) == 1) {
        m3::Prep p = prep;
        if (!prep.on && d.dstate == 128 && d.R == 1 && d.chunk == 64) p.test_timeout_at = g_inject_timeout.exchange(0);
        return cuda_status(m3::launch_scan_tc(d, x, B, C, dt, A, lambda, omega, y, final_state, workspace, p, s));
    }
    return cuda_status(m3::launch_scan_simt(d, x, B, C, dt, A, lambda, omega, y, final_state, workspace, prep, s));
}

int decode_impl(float* state, const void* x_t, const void* B_t, void* B_prev_x_prev, const void* C_t,
                const float* dt_t, const float* A, const float* lambda_t, const float* omega_t, void* y_t,
                int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate, int R, int io_dtype, void* stream,
                const m3::Prep& prep) {
    if (!ok_io(io_dtype)) return M3_ERR_INVALID_ARG;
    if (batch < 0 || nheads < 1 || headdim < 1 || dstate < 2 || dstate % 2 || R < 1) return M3_ERR_INVALID_ARG;
    if (!m3::decode_supported(headdim, dstate, R)) return M3_ERR_UNSUPPORTED;
    if (batch * nheads > (int64_t)INT32_MAX) return M3_ERR_UNSUPPORTED;
    if (!ok_nullable(prep.dt_bias)) return M3_ERR_INVALID_ARG;
    if (!prep.on && !ok_ptr(A)) return M3_ERR_INVALID_ARG;
    if (batch == 0) return M3_OK;
    if (!ok_ptr(state) || !ok_ptr(x_t) || !ok_ptr(B_t) || !ok_ptr(B_prev_x_prev) || !ok_ptr(C_t) || !ok_ptr(dt_t) ||
        !ok_ptr(lambda_t) || !ok_ptr(omega_t) || !ok_ptr(y_t) || !ok_ptr(A))
        return M3_ERR_INVALID_ARG;
    if (injected_launch_failure()) return M3_ERR_CUDA;
    return cuda_status(m3::launch_decode(state, x_t, B_t, B_prev_x_prev, C_t, dt_t, A, lambda_t, omega_t, y_t, batch,
                                         nheads, headdim, dstate, R, io_dtype, prep,
                                         static_cast<cudaStream_t>(stream)));
}

// The backward on pre-activations: m3_scan_bwd's sections, Delta and lambda; then, for the output gate,
// the ungated forward output y_pre (io dtype) and the forward entry's own workspace (chunk 64).
struct BwdPrepWs {
    size_t y_pre, fwd, total;
    bool gate;   // the forward supports the shape, so the gate's backward can run
};

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

BwdPrepWs bwd_prep_ws(const m3::ScanDims& d) {
    BwdPrepWs w{};
    w.y_pre = al256(m3::bwd_prep_workspace_size(d));
    w.total = w.y_pre;
    const m3::ScanDims f{d.batch, d.seqlen, d.nheads, d.headdim, d.dstate, d.R, 64, d.io};
    w.gate = validate_scan_sizes(f) == M3_OK && m3::bwd_gate_supported(d);
    if (w.gate) {
        const size_t e = d.io == M3_DTYPE_BF16 ? 2 : 4;
        w.fwd = w.y_pre + al256(e * (size_t)(d.batch * d.seqlen * d.nheads) * (size_t)(d.R * d.headdim));
        w.total = w.fwd + al256(scan_workspace(f, true));
    }
    return w;
}

}  // namespace

extern "C" {

const char* m3_status_string(int status) {
    switch (status) {
        case M3_OK: return "M3_OK";
        case M3_ERR_INVALID_ARG: return "M3_ERR_INVALID_ARG: null or misaligned pointer, or an invalid size or dtype";
        case M3_ERR_UNSUPPORTED: return "M3_ERR_UNSUPPORTED: valid arguments outside the sizes the kernels implement";
        case M3_ERR_WORKSPACE: return "M3_ERR_WORKSPACE: workspace missing or smaller than m3_scan_fwd_workspace_size";
        case M3_ERR_CUDA: return "M3_ERR_CUDA: a CUDA call or kernel launch failed";
        case M3_ERR_TIMEOUT: return "M3_ERR_TIMEOUT: a bounded device-side wait gave up";
        default: return "unknown m3 status";
    }
}

int m3_version(void) { return 100; }

int m3_test_inject(int what, int count) {
    if (count < 0) return M3_ERR_INVALID_ARG;
    switch (what) {
        case 0: g_inject_launch.store(0); g_inject_timeout.store(0); return 0;
        case M3_TEST_LAUNCH_FAILURE: return g_inject_launch.exchange(count);
        case M3_TEST_PREFILL_TIMEOUT: {
            const int prev = g_inject_timeout.exchange(count + 1);
            return prev > 0 ? prev - 1 : -1;
        }
        default: return M3_ERR_INVALID_ARG;
    }
}

size_t m3_scan_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                                  int R, int chunk, int io_dtype) {
    const m3::ScanDims d{batch, seqlen, nheads, headdim, dstate, R, chunk, io_dtype};
    if (validate_scan_sizes(d) != M3_OK) return 0;
    return scan_workspace(d, false);
}

size_t m3_scan_fwd_prep_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                       int64_t dstate, int R, int chunk, int io_dtype) {
    const m3::ScanDims d{batch, seqlen, nheads, headdim, dstate, R, chunk, io_dtype};
    if (validate_scan_sizes(d) != M3_OK) return 0;
    return scan_workspace(d, true);
}

int m3_scan_fwd_plan(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate, int R,
                     int chunk, int io_dtype, int* path, int* launches) {
    const m3::ScanDims d{batch, seqlen, nheads, headdim, dstate, R, chunk, io_dtype};
    const int st = validate_scan_sizes(d);
    if (st != M3_OK) return st;
    const int p = pick_path(d);
    int n = 0;
    if (batch > 0) n = p == 1 ? m3::tc_launch_count(d) : (batch * nheads > 0 && seqlen > 0 ? 3 : 1);
    if (path) *path = p;
    if (launches) *launches = n;
    return M3_OK;
}

int m3_scan_fwd(const void* x, const void* B, const void* C, const float* dt, const float* A, const float* lambda,
                const float* omega, int R, int chunk, void* y, float* final_state, int64_t batch, int64_t seqlen,
                int64_t nheads, int64_t headdim, int64_t dstate, int io_dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
    return scan_impl(x, B, C, dt, A, lambda, omega, R, chunk, y, final_state, batch, seqlen, nheads, headdim, dstate,
                     io_dtype, workspace, workspace_bytes, stream, m3::Prep{});
}

int m3_scan_fwd_prep(const void* x, const void* B, const void* C, const float* dt_raw, const float* A,
                     const float* u, const float* omega, int R, int chunk, void* y, float* final_state,
                     int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate, int io_dtype,
                     const m3_prep_params* params, void* workspace, size_t workspace_bytes, void* stream) {
    m3::Prep prep;
    if (!prep_from(params, &prep)) return M3_ERR_INVALID_ARG;
    return scan_impl(x, B, C, dt_raw, A, u, omega, R, chunk, y, final_state, batch, seqlen, nheads, headdim, dstate,
                     io_dtype, workspace, workspace_bytes, stream, prep);
}

int m3_decode_step(float* state, const void* x_t, const void* B_t, void* B_prev_x_prev, const void* C_t,
                   const float* dt_t, const float* A, const float* lambda_t, const float* omega_t, void* y_t,
                   int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate, int R, int io_dtype,
                   void* stream) {
    return decode_impl(state, x_t, B_t, B_prev_x_prev, C_t, dt_t, A, lambda_t, omega_t, y_t, batch, nheads, headdim,
                       dstate, R, io_dtype, stream, m3::Prep{});
}

int m3_decode_step_prep(float* state, const void* x_t, const void* B_t, void* B_prev_x_prev, const void* C_t,
                        const float* dt_raw_t, const float* A_t, const float* u_t, const float* omega_t, void* y_t,
                        int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate, int R, int io_dtype,
                        const m3_prep_params* params, void* stream) {
    m3::Prep prep;
    if (!prep_from(params, &prep)) return M3_ERR_INVALID_ARG;
    return decode_impl(state, x_t, B_t, B_prev_x_prev, C_t, dt_raw_t, A_t, u_t, omega_t, y_t, batch, nheads, headdim,
                       dstate, R, io_dtype, stream, prep);
}

int m3_device_status(int clear) {
    // the words are written by kernels on the caller's streams, which may be non-blocking
    if (cudaDeviceSynchronize() != cudaSuccess) return M3_ERR_CUDA;
    const int dec = m3::decode_device_status(clear);
    if (dec == M3_ERR_CUDA) return dec;
    const int na = m3::noalloc_device_status(clear);
    if (na == M3_ERR_CUDA || na == M3_ERR_UNSUPPORTED) return na;
    return dec != M3_OK ? dec : na;
}

size_t m3_scan_bwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                                  int R, int io_dtype) {
    const m3::ScanDims d{batch, seqlen, nheads, headdim, dstate, R, 64, io_dtype};
    if (!ok_io(io_dtype) || batch < 0 || seqlen < 0 || nheads < 1 || !m3::bwd_supported(d)) return 0;
    return m3::bwd_workspace_size(d);
}

int m3_scan_bwd(const void* x, const void* B, const void* C, const float* dt, const float* A, const float* lambda,
                const float* omega, int R, const void* dy, const float* d_final, float* dx, float* dB, float* dC,
                float* ddt, float* dA, float* dlambda, float* domega, int64_t batch, int64_t seqlen,
                int64_t nheads, int64_t headdim, int64_t dstate, int io_dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
    const m3::ScanDims d{batch, seqlen, nheads, headdim, dstate, R, 64, io_dtype};
    if (!ok_io(io_dtype)) return M3_ERR_INVALID_ARG;
    if (batch < 0 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 2 || dstate % 2 || R < 1)
        return M3_ERR_INVALID_ARG;
    if (batch * nheads > (int64_t)INT32_MAX || seqlen > (int64_t)INT32_MAX) return M3_ERR_UNSUPPORTED;
    if (!m3::bwd_supported(d)) return M3_ERR_UNSUPPORTED;
    if (!ok_ptr(A) || !ok_ptr(dA) || !ok_nullable(d_final)) return M3_ERR_INVALID_ARG;
    if (batch > 0 && seqlen > 0) {
        const void* ptrs[] = {x, B, C, dt, lambda, omega, dy, dx, dB, dC, ddt, dlambda, domega};
        for (const void* q : ptrs)
            if (!ok_ptr(q)) return M3_ERR_INVALID_ARG;
        const size_t need = m3::bwd_workspace_size(d);
        if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return M3_ERR_WORKSPACE;
    }
    if (batch > 0 && injected_launch_failure()) return M3_ERR_CUDA;
    return cuda_status(m3::launch_scan_bwd(d, x, B, C, dt, A, lambda, omega, dy, d_final, dx, dB, dC, ddt, dA,
                                           dlambda, domega, workspace, static_cast<cudaStream_t>(stream)));
}

size_t m3_scan_bwd_prep_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                       int64_t dstate, int R, int io_dtype) {
    const m3::ScanDims d{batch, seqlen, nheads, headdim, dstate, R, 64, io_dtype};
    if (!ok_io(io_dtype) || batch < 0 || seqlen < 0 || nheads < 1 || !m3::bwd_supported(d)) return 0;
    return bwd_prep_ws(d).total;
}

int m3_scan_bwd_prep(const void* x, const void* B, const void* C, const float* dt_raw, const float* A,
                     const float* u, const float* omega, int R, const void* dy, const float* d_final, float* dx,
                     float* dB, float* dC, float* ddt_raw, float* dA, float* du, float* domega, float* ddt_bias,
                     float* dz, float* dB_gain, float* dC_gain, float* dB_bias, float* dC_bias, int64_t batch,
                     int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate, int io_dtype,
                     const m3_prep_params* params, void* workspace, size_t workspace_bytes, void* stream) {
    const m3::ScanDims d{batch, seqlen, nheads, headdim, dstate, R, 64, io_dtype};
    if (!ok_io(io_dtype)) return M3_ERR_INVALID_ARG;
    if (batch < 0 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 2 || dstate % 2 || R < 1)
        return M3_ERR_INVALID_ARG;
    const float* dt_bias = params != nullptr ? params->dt_bias : nullptr;
    const void* z = params != nullptr ? params->z : nullptr;
    if (!ok_nullable(dt_bias) || !ok_nullable(ddt_bias) || !ok_nullable(d_final) || !ok_nullable(z))
        return M3_ERR_INVALID_ARG;
    m3::Prep fp{};
    if (params != nullptr && !prep_from(params, &fp)) return M3_ERR_INVALID_ARG;
    const float* gouts[] = {dB_gain, dC_gain, dB_bias, dC_bias};
    for (const float* q : gouts)
        if (!ok_nullable(q)) return M3_ERR_INVALID_ARG;
    const m3::BwdBcArgs bca{params != nullptr && fp.bc(), fp.bc_norm ? 1 : 0, fp.bc_eps, fp.B_gain, fp.C_gain,
                            fp.B_bias, fp.C_bias, dB_gain, dC_gain, dB_bias, dC_bias};
    if (batch * nheads > (int64_t)INT32_MAX || seqlen > (int64_t)INT32_MAX) return M3_ERR_UNSUPPORTED;
    if (!m3::bwd_supported(d)) return M3_ERR_UNSUPPORTED;
    if (bca.on && !m3::bwd_bc_supported(d)) return M3_ERR_UNSUPPORTED;
    const BwdPrepWs w = bwd_prep_ws(d);
    if (z != nullptr && !w.gate) return M3_ERR_UNSUPPORTED;
    const bool any_tokens = batch > 0 && seqlen > 0;
    if (any_tokens) {
        const void* ptrs[] = {x, B, C, dt_raw, A, u, omega, dy, dx, dB, dC, ddt_raw, dA, du, domega};
        for (const void* q : ptrs)
            if (!ok_ptr(q)) return M3_ERR_INVALID_ARG;
        if (z != nullptr && !ok_ptr(dz)) return M3_ERR_INVALID_ARG;
        if (workspace == nullptr || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return M3_ERR_WORKSPACE;
    }
    if (batch > 0 && injected_launch_failure()) return M3_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    void* y_pre = nullptr;
    if (z != nullptr && any_tokens) {   // the ungated forward output, by the forward entry itself
        m3::Prep ug = fp;
        ug.z = nullptr;
        y_pre = ws + w.y_pre;
        const int st = scan_impl(x, B, C, dt_raw, A, u, omega, R, 64, y_pre, nullptr, batch, seqlen, nheads, headdim,
                                 dstate, io_dtype, ws + w.fwd, w.total - w.fwd, stream, ug);
        if (st != M3_OK) return st;
    }
    return cuda_status(m3::launch_scan_bwd_prep(d, x, B, C, dt_raw, dt_bias, A, u, omega, dy, d_final, dx, dB, dC,
                                                ddt_raw, dA, du, domega, ddt_bias, z, y_pre, dz, bca, workspace,
                                                static_cast<cudaStream_t>(stream)));
}

int m3_state_passing(float* chunk_states, const float* chunk_logdecay, const float* chunk_angle,
                     const float* init_state, float* final_state, int64_t batch, int64_t nheads, int64_t nchunks,
                     int64_t dstate, int64_t headdim, void* stream) {
    if (batch < 0 || nheads < 1 || nchunks < 0) return M3_ERR_INVALID_ARG;
    if (dstate < 2 || dstate % 2 || headdim < 4 || headdim % 4) return M3_ERR_INVALID_ARG;
    if (dstate > 256 || headdim > 256) return M3_ERR_UNSUPPORTED;
    if (batch * nheads > (int64_t)INT32_MAX || nchunks > (int64_t)INT32_MAX) return M3_ERR_UNSUPPORTED;
    if (!ok_nullable(init_state) || !ok_nullable(final_state)) return M3_ERR_INVALID_ARG;
    if (batch > 0 && nchunks > 0) {
        if (!ok_ptr(chunk_states) || !ok_ptr(chunk_logdecay) || !ok_ptr(chunk_angle)) return M3_ERR_INVALID_ARG;
    }
    if (batch == 0) return M3_OK;
    if (injected_launch_failure()) return M3_ERR_CUDA;
    return cuda_status(m3::launch_state_passing(chunk_states, chunk_logdecay, chunk_angle, init_state, final_state,
                                                batch, nheads, nchunks, dstate, headdim,
                                                static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
