// iso_backward_noalloc: the backward of the fit for callers that cannot allocate
// device memory.  Some hosts hand a library only the buffers of the call: a
// plugin whose host owns every device allocation, a pre-sized embedded
// pipeline with a fixed memory budget, or a loop that cannot afford the
// device-wide synchronisation that cudaMalloc and cudaFree may cause.  For them
// this entry point takes no workspace: the scratch that long rows need (one
// record per tile of 8,192 elements) lives in a fixed array in the library's
// device memory instead.
#include <mutex>

#include "../../include/iso.h"
#include "iso_internal.h"

namespace {

// 2 MiB: enough for 21,845 tiles of 8,192 elements, i.e. rows * ceil(n / 8192)
// <= 21,845 (about 1.8e8 elements).  Every GPU that loads the library keeps it
// until the process exits.
constexpr size_t kScratchBytes = size_t(2) << 20;
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's name
// is only a host-side stand-in for it, so its address is asked of the runtime
// once per device, with that device current.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" iso_status iso_backward_noalloc(const float* grad, const uint8_t* blocks,
                                           const float* w, int64_t rows, int64_t n, float* out,
                                           void* stream) {
    if (rows >= 0 && n >= 0 && (rows == 0 || n == 0)) return ISO_OK;   // empty: nothing to do
    if (!grad || !blocks || !out || rows < 1 || n < 1 || n > 2147483647LL ||
        rows > (int64_t(1) << 40) / n)
        return ISO_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t need = iso_backward_workspace_bytes(rows, n, w != nullptr);
    if (need == 0)   // whole rows: no scratch at all
        return iso_backward(grad, blocks, w, rows, n, out, nullptr, 0, stream);
    if (need > kScratchBytes) return ISO_ERR_WORKSPACE;
    void* ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) return ISO_ERR_CUDA;
    isodev::prof_start(st);
    return isodev::long_backward<float>(grad, blocks, w, rows, n, out, nullptr, nullptr, nullptr, ws,
                                 kScratchBytes, st) == cudaSuccess
               ? ISO_OK
               : ISO_ERR_CUDA;
}
