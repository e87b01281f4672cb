// Tensor-core (tcgen05 / TMEM / TMA) chunked prefill for bf16 io.
#include "m3_common.cuh"

namespace m3 {

size_t tc_workspace_size(const ScanDims&) { return 0; }
bool tc_supported(const ScanDims&) { return false; }
int tc_launch_count(const ScanDims&) { return 0; }
cudaError_t launch_scan_tc(const ScanDims&, const void*, const void*, const void*, const float*, const float*,
                           const float*, const float*, void*, float*, void*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace m3
