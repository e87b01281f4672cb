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
// before any stream capture.  The address is cached per device together with
// the unique id of the context it was looked up in; when the device's context
// is torn down and re-created (cudaDeviceReset) the next call sees a new
// context id and looks the address up again.
#include <cuda.h>

#include <mutex>

#include "m3_common.cuh"

// The scratch array.  All calls on a device share it and it keeps the last
// call's contents.  The prefill clears the part that must start at zero (its
// status word) on every call and writes the rest before reading it.
static __device__ __align__(256) unsigned char g_m3_noalloc_scratch[M3_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 128;

struct DevScratch {
    void* addr;                  // device address of the array in the context below
    unsigned long long ctx_id;   // unique id of that context (0 = not looked up yet)
    int last_path;               // path of the last call on this device: 1 = tensor cores, 0 = CUDA cores, -1 = none
};

std::mutex g_mu;
DevScratch g_dev[kMaxDevices] = {};
bool g_dev_init = false;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the current context (driver entry points, so the library needs no link to libcuda);
// 0 when there is none yet or it cannot be read.
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked = false;
    if (!looked) {
        looked = true;
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    }
    if (get_cur == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array on the current device, looked up once per device and context.
// Caller holds g_mu.
int scratch_for_current_device(int dev, void** out) {
    DevScratch& s = g_dev[dev];
    const unsigned long long id = current_ctx_id();
    if (s.addr == nullptr || id == 0 || id != s.ctx_id) {
        void* p = nullptr;
        // also creates the device's primary context if the caller has not yet
        if (cudaGetSymbolAddress(&p, g_m3_noalloc_scratch) != cudaSuccess || p == nullptr) return M3_ERR_CUDA;
        s.addr = p;
        s.ctx_id = current_ctx_id();
    }
    *out = s.addr;
    return M3_OK;
}

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return M3_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return M3_ERR_UNSUPPORTED;
    if (!g_dev_init) {
        for (int i = 0; i < kMaxDevices; ++i) g_dev[i] = DevScratch{nullptr, 0ull, -1};
        g_dev_init = true;
    }
    return M3_OK;
}

}  // namespace

namespace m3 {

// The tensor-core prefill records M3_ERR_TIMEOUT in the first word of its workspace; for the noalloc
// entry that is the scratch array, which the caller cannot read, so m3_device_status reads it here
// (the last call's word, when that call took the tensor-core path; the CUDA-core kernels have no
// waits and keep chunk states there).  clear != 0 resets it.
int noalloc_device_status(int clear) {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = -1;
    const int st = current_device(&dev);
    if (st != M3_OK) return st;
    if (g_dev[dev].last_path != 1 || g_dev[dev].addr == nullptr) return M3_OK;
    if (g_dev[dev].ctx_id != current_ctx_id()) return M3_OK;   // the context (and the array's contents) is gone
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_m3_noalloc_scratch, sizeof(int)) != cudaSuccess) return M3_ERR_CUDA;
    if (clear && v != 0) {
        const int z = 0;
        if (cudaMemcpyToSymbol(g_m3_noalloc_scratch, &z, sizeof(int)) != cudaSuccess) return M3_ERR_CUDA;
    }
    return v;
}

}  // namespace m3

extern "C" int m3_scan_fwd_noalloc(const void* x, const void* B, const void* C, const float* dt, const float* A,
                                   const float* lambda, const float* omega, int R, int chunk, void* y,
                                   float* final_state, int64_t batch, int64_t seqlen, int64_t nheads,
                                   int64_t headdim, int64_t dstate, int io_dtype, void* stream) {
    // 0 means "no scratch needed" or "sizes m3_scan_fwd rejects"; in both
    // cases m3_scan_fwd below answers without touching the scratch array.
    const size_t need = m3_scan_fwd_workspace_size(batch, seqlen, nheads, headdim, dstate, R, chunk, io_dtype);
    if (need > (size_t)M3_NOALLOC_SCRATCH_BYTES) return M3_ERR_WORKSPACE;
    void* ws = nullptr;
    int path = 0, dev = -1;
    if (need > 0) {
        int launches = 0;
        int st = m3_scan_fwd_plan(batch, seqlen, nheads, headdim, dstate, R, chunk, io_dtype, &path, &launches);
        if (st != M3_OK) return st;
        std::lock_guard<std::mutex> lock(g_mu);
        st = current_device(&dev);
        if (st != M3_OK) return st;
        st = scratch_for_current_device(dev, &ws);
        if (st != M3_OK) return st;
    }
    const int st = m3_scan_fwd(x, B, C, dt, A, lambda, omega, R, chunk, y, final_state, batch, seqlen, nheads,
                               headdim, dstate, io_dtype, ws, need > 0 ? (size_t)M3_NOALLOC_SCRATCH_BYTES : 0, stream);
    if (st == M3_OK && need > 0) {   // what m3_device_status finds in the scratch array's first word
        std::lock_guard<std::mutex> lock(g_mu);
        g_dev[dev].last_path = path;
    }
    return st;
}
