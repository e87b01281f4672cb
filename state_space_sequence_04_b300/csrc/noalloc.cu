// m3_scan_fwd_noalloc: the chunked prefill for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain device scratch: an application that owns
// every device allocation and hands the library only its inputs and outputs,
// a serving loop that forbids allocation once it is running (allocation can
// stall or fail under fragmentation), or a plugin host that offers no
// allocator callback.  m3_scan_fwd needs a caller-provided workspace; this
// entry point instead uses a fixed scratch array that is part of the
// library's own device image and stays reserved on every GPU that loads the
// library until the process exits.
//
// It calls no cudaMalloc / cudaFree and no allocating library routine.  On
// the first call on each device (with that device current) it looks up the
// array's device address once with cudaGetSymbolAddress: in host code the
// array's name is only a host-side stand-in, never a device address, so it
// must not be handed to a kernel directly.  Make that first call on a device
// before any stream capture.
#include <mutex>

#include "m3_common.cuh"

// The scratch array.  All calls on a device share it and it keeps the last
// call's contents.  The prefill clears the part that must start at zero (its
// status word) on every call and writes the rest before reading it.
static __device__ __align__(256) unsigned char g_m3_noalloc_scratch[M3_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return M3_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return M3_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_m3_noalloc_scratch) != cudaSuccess || p == nullptr) return M3_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return M3_OK;
}

}  // namespace

extern "C" int m3_scan_fwd_noalloc(const void* x, const void* B, const void* C, const float* dt, const float* A,
                                   const float* lambda, const float* omega, int R, int chunk, void* y,
                                   float* final_state, int64_t batch, int64_t seqlen, int64_t nheads,
                                   int64_t headdim, int64_t dstate, int io_dtype, void* stream) {
    // 0 means "no scratch needed" or "sizes m3_scan_fwd rejects"; in both
    // cases m3_scan_fwd below answers without touching the scratch array.
    const size_t need = m3_scan_fwd_workspace_size(batch, seqlen, nheads, headdim, dstate, R, chunk, io_dtype);
    if (need > (size_t)M3_NOALLOC_SCRATCH_BYTES) return M3_ERR_WORKSPACE;
    void* ws = nullptr;
    if (need > 0) {
        const int st = scratch_for_current_device(&ws);
        if (st != M3_OK) return st;
    }
    return m3_scan_fwd(x, B, C, dt, A, lambda, omega, R, chunk, y, final_state, batch, seqlen, nheads, headdim,
                       dstate, io_dtype, ws, need > 0 ? (size_t)M3_NOALLOC_SCRATCH_BYTES : 0, stream);
}
