// C ABI of libiso (declared in include/iso.h): argument checks and dispatch by
// row length to the whole-row kernels or the long-row path.
#include "../../include/iso.h"
#include "iso_internal.h"

namespace {

constexpr int64_t kMaxN = 2147483647LL;
constexpr int64_t kMaxElems = 1LL << 40;

bool shape_ok(int64_t rows, int64_t n) {
    return rows >= 1 && n >= 1 && n <= kMaxN && rows <= kMaxElems / n;
}

iso_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ISO_OK : ISO_ERR_CUDA; }

}  // namespace

extern "C" {

int iso_version(void) { return 100; }

const char* iso_status_string(int status) {
    switch (status) {
        case ISO_OK: return "ok";
        case ISO_ERR_INVALID_ARG: return "invalid argument";
        case ISO_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case ISO_ERR_CUDA: return "CUDA error";
        case ISO_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

size_t iso_fit_workspace_bytes(int64_t rows, int64_t n, int weighted) {
    if (!shape_ok(rows, n)) return 0;
    if (n <= isodev::kRowMax) return 0;
    return isodev::long_fit_workspace(rows, n, weighted != 0);
}

iso_status iso_fit(const float* y, const float* w, int64_t rows, int64_t n, int increasing,
                   float* out, uint8_t* blocks, void* workspace, size_t workspace_bytes,
                   uint32_t* row_status, void* stream) {
    if (!y || !out || !shape_ok(rows, n) || (increasing != 0 && increasing != 1))
        return ISO_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n <= isodev::kRowMax)
        return from_cuda(isodev::rows_fit(y, w, rows, (int)n, increasing, out, blocks,
                                          row_status, st));
    const size_t need = isodev::long_fit_workspace(rows, n, w != nullptr);
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return ISO_ERR_WORKSPACE;
    return from_cuda(isodev::long_fit(y, w, rows, n, increasing, out, blocks, workspace,
                                      workspace_bytes, row_status, st));
}

size_t iso_backward_workspace_bytes(int64_t rows, int64_t n, int weighted) {
    if (!shape_ok(rows, n)) return 0;
    if (n <= isodev::kRowMax) return 0;
    return isodev::long_backward_workspace(rows, n, weighted != 0);
}

iso_status iso_backward(const float* grad, const uint8_t* blocks, const float* w, int64_t rows,
                        int64_t n, float* out, void* workspace, size_t workspace_bytes,
                        void* stream) {
    if (!grad || !blocks || !out || !shape_ok(rows, n)) return ISO_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n <= isodev::kRowMax)
        return from_cuda(isodev::rows_backward(grad, blocks, w, rows, (int)n, out, st));
    const size_t need = isodev::long_backward_workspace(rows, n, w != nullptr);
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return ISO_ERR_WORKSPACE;
    return from_cuda(isodev::long_backward(grad, blocks, w, rows, n, out, workspace,
                                           workspace_bytes, st));
}

}  // extern "C"
