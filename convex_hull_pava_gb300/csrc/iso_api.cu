// C ABI of libiso (declared in include/iso.h): argument checks and dispatch by
// row length to the whole-row kernels or the long-row path.
#include "../../include/iso.h"
#include "iso_internal.h"

namespace isodev {

namespace {
constexpr int kProfMax = 16;
struct Profile {
    bool on = false;
    bool created = false;
    cudaEvent_t ev[kProfMax + 1];
    const char* name[kProfMax];
    int count = 0;      // kernels marked in the current call
    bool started = false;
} g_prof;
}  // namespace

void prof_start(cudaStream_t stream) {
    if (!g_prof.on) return;
    g_prof.count = 0;
    g_prof.started = cudaEventRecord(g_prof.ev[0], stream) == cudaSuccess;
}

void prof_mark(cudaStream_t stream, const char* name) {
    if (!g_prof.on || !g_prof.started || g_prof.count >= kProfMax) return;
    if (cudaEventRecord(g_prof.ev[g_prof.count + 1], stream) == cudaSuccess)
        g_prof.name[g_prof.count++] = name;
}

namespace {
constexpr int kStatDevices = 64;
constexpr int kStatCount = 8;
int g_bridge_mode = 0;
unsigned long long* g_bridge_stats[kStatDevices];
}  // namespace

int device_sms() {
    static int sms[kStatDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStatDevices) return 1;
    if (sms[dev] <= 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
        sms[dev] = n;
    }
    return sms[dev];
}

BridgeDebug bridge_debug() {
    BridgeDebug d{nullptr, ISO_BRIDGE_MAX_PASSES};
    if (g_bridge_mode == 0) return d;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStatDevices) return d;
    d.stats = g_bridge_stats[dev];
    if (d.stats && g_bridge_mode == 2) d.max_passes = 0;
    return d;
}

iso_status bridge_stats_mode(int mode) {
    if (mode < 0 || mode > 2) return ISO_ERR_INVALID_ARG;
    if (mode == 0) { g_bridge_mode = 0; return ISO_OK; }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ISO_ERR_CUDA;
    if (dev < 0 || dev >= kStatDevices) return ISO_ERR_INVALID_ARG;
    if (!g_bridge_stats[dev] &&
        cudaMalloc(&g_bridge_stats[dev], kStatCount * sizeof(unsigned long long)) != cudaSuccess) {
        g_bridge_stats[dev] = nullptr;
        return ISO_ERR_CUDA;
    }
    if (cudaMemset(g_bridge_stats[dev], 0, kStatCount * sizeof(unsigned long long)) != cudaSuccess)
        return ISO_ERR_CUDA;
    g_bridge_mode = mode;
    return ISO_OK;
}

iso_status bridge_stats_read(uint64_t* out) {
    if (!out) return ISO_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ISO_ERR_CUDA;
    if (dev < 0 || dev >= kStatDevices || !g_bridge_stats[dev]) return ISO_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return ISO_ERR_CUDA;
    unsigned long long v[kStatCount];
    if (cudaMemcpy(v, g_bridge_stats[dev], sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return ISO_ERR_CUDA;
    for (int i = 0; i < kStatCount; ++i) out[i] = (uint64_t)v[i];
    return ISO_OK;
}

}  // namespace isodev

namespace {

constexpr int64_t kMaxN = 2147483647LL;
constexpr int64_t kMaxElems = 1LL << 40;

bool shape_ok(int64_t rows, int64_t n) {
    return rows >= 1 && n >= 1 && n <= kMaxN && rows <= kMaxElems / n;
}

iso_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ISO_OK : ISO_ERR_CUDA; }

// An empty batch (no rows, or rows of no elements): nothing to do, whatever
// the pointers.
bool empty_call(int64_t rows, int64_t n) { return rows >= 0 && n >= 0 && (rows == 0 || n == 0); }

// Typed implementations of the entry points: IO is the I/O type (float or
// double); the arithmetic inside is the same fixed point for both.
template <class IO>
iso_status fit_impl(const IO* y, const IO* w, int64_t rows, int64_t n, int increasing, IO* out,
                    uint8_t* blocks, void* workspace, size_t workspace_bytes,
                    uint32_t* row_status, void* stream) {
    if (empty_call(rows, n) && (increasing == 0 || increasing == 1)) return ISO_OK;
    if (!y || !out || !shape_ok(rows, n) || (increasing != 0 && increasing != 1))
        return ISO_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    isodev::prof_start(st);
    if (n <= isodev::kRowMax)
        return from_cuda(isodev::rows_fit<IO>(y, w, rows, (int)n, increasing, out, blocks,
                                              row_status, st));
    const size_t need = isodev::long_fit_workspace(rows, n, w != nullptr);
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return ISO_ERR_WORKSPACE;
    return from_cuda(isodev::long_fit<IO>(y, w, rows, n, increasing, out, blocks, workspace,
                                          workspace_bytes, row_status, st));
}

bool ragged_ok(int64_t segments, int64_t total, int64_t max_len) {
    return segments >= 1 && segments <= kMaxN && total >= 0 && total <= kMaxElems &&
           max_len <= kMaxN;
}
int64_t ragged_max_len(int64_t total, int64_t max_len) {
    return max_len <= 0 || max_len > total ? total : max_len;
}

template <class IO>
iso_status ragged_impl(const IO* y, const IO* w, const int64_t* offsets, int64_t segments,
                       int64_t total, int64_t max_len, int increasing, IO* out, uint8_t* blocks,
                       void* workspace, size_t workspace_bytes, uint32_t* row_status,
                       void* stream) {
    if (segments == 0 && total >= 0 && (increasing == 0 || increasing == 1)) return ISO_OK;
    // with no elements every segment is empty (or rejected): y and out are not read
    if ((total > 0 && (!y || !out)) || !offsets || !ragged_ok(segments, total, max_len) ||
        (increasing != 0 && increasing != 1))
        return ISO_ERR_INVALID_ARG;
    const int64_t ml = ragged_max_len(total, max_len);
    if (ml > kMaxN) return ISO_ERR_INVALID_ARG;
    const size_t need = isodev::ragged_workspace(segments, total, ml, w != nullptr);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ISO_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    isodev::prof_start(st);
    return from_cuda(isodev::ragged_fit<IO>(y, w, offsets, segments, total, ml, increasing, out,
                                            blocks, workspace, row_status, st));
}

template <class IO>
iso_status control_impl(const IO* y, const IO* w, int64_t rows, int64_t n, int increasing,
                        IO* out, uint8_t* blocks, void* workspace, size_t workspace_bytes,
                        uint32_t* row_status, void* stream) {
    if (empty_call(rows, n) && (increasing == 0 || increasing == 1)) return ISO_OK;
    if (!y || !out || !shape_ok(rows, n) || n > (1LL << 30) || (increasing != 0 && increasing != 1))
        return ISO_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    isodev::prof_start(st);
    if (n <= isodev::kRowMax)
        return from_cuda(isodev::rows_fit<IO>(y, w, rows, (int)n, increasing, out, blocks,
                                              row_status, st));
    const size_t need = isodev::long_control_workspace(rows, n, w != nullptr);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ISO_ERR_WORKSPACE;
    return from_cuda(isodev::long_fit_control<IO>(y, w, rows, n, increasing, out, blocks,
                                                  workspace, row_status, st));
}

// Both gradients (out_dy and/or out_dw; y and fit needed only for out_dw).
template <class IO>
iso_status backward_impl(const IO* grad, const uint8_t* blocks, const IO* w, const IO* y,
                         const IO* fit, int64_t rows, int64_t n, IO* out_dy, IO* out_dw,
                         void* workspace, size_t workspace_bytes, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    isodev::prof_start(st);
    if (n <= isodev::kRowMax)
        return from_cuda(isodev::rows_backward<IO>(grad, blocks, w, rows, (int)n, out_dy, y, fit,
                                                   out_dw, st));
    const size_t need = isodev::long_backward_workspace(rows, n, w != nullptr);
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return ISO_ERR_WORKSPACE;
    return from_cuda(isodev::long_backward<IO>(grad, blocks, w, rows, n, out_dy, y, fit, out_dw,
                                               workspace, workspace_bytes, st));
}

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
    return fit_impl<float>(y, w, rows, n, increasing, out, blocks, workspace, workspace_bytes,
                           row_status, stream);
}

iso_status iso_fit_f64(const double* y, const double* w, int64_t rows, int64_t n, int increasing,
                       double* out, uint8_t* blocks, void* workspace, size_t workspace_bytes,
                       uint32_t* row_status, void* stream) {
    return fit_impl<double>(y, w, rows, n, increasing, out, blocks, workspace, workspace_bytes,
                            row_status, stream);
}

size_t iso_fit_ragged_workspace_bytes(int64_t segments, int64_t total, int64_t max_len,
                                      int weighted) {
    if (!ragged_ok(segments, total, max_len)) return 0;
    return isodev::ragged_workspace(segments, total, ragged_max_len(total, max_len), weighted != 0);
}

iso_status iso_fit_ragged(const float* y, const float* w, const int64_t* offsets,
                          int64_t segments, int64_t total, int64_t max_len, int increasing,
                          float* out, uint8_t* blocks, void* workspace, size_t workspace_bytes,
                          uint32_t* row_status, void* stream) {
    return ragged_impl<float>(y, w, offsets, segments, total, max_len, increasing, out, blocks,
                              workspace, workspace_bytes, row_status, stream);
}

iso_status iso_fit_ragged_f64(const double* y, const double* w, const int64_t* offsets,
                              int64_t segments, int64_t total, int64_t max_len, int increasing,
                              double* out, uint8_t* blocks, void* workspace,
                              size_t workspace_bytes, uint32_t* row_status, void* stream) {
    return ragged_impl<double>(y, w, offsets, segments, total, max_len, increasing, out, blocks,
                               workspace, workspace_bytes, row_status, stream);
}

size_t iso_fit_copy_control_workspace_bytes(int64_t rows, int64_t n, int weighted) {
    if (!shape_ok(rows, n) || n > (1LL << 30)) return 0;
    if (n <= isodev::kRowMax) return 0;
    return isodev::long_control_workspace(rows, n, weighted != 0);
}

iso_status iso_fit_copy_control(const float* y, const float* w, int64_t rows, int64_t n,
                                int increasing, float* out, uint8_t* blocks, void* workspace,
                                size_t workspace_bytes, uint32_t* row_status, void* stream) {
    return control_impl<float>(y, w, rows, n, increasing, out, blocks, workspace,
                               workspace_bytes, row_status, stream);
}

size_t iso_backward_workspace_bytes(int64_t rows, int64_t n, int weighted) {
    if (!shape_ok(rows, n)) return 0;
    if (n <= isodev::kRowMax) return 0;
    return isodev::long_backward_workspace(rows, n, weighted != 0);
}

iso_status iso_backward(const float* grad, const uint8_t* blocks, const float* w, int64_t rows,
                        int64_t n, float* out, void* workspace, size_t workspace_bytes,
                        void* stream) {
    if (empty_call(rows, n)) return ISO_OK;
    if (!grad || !blocks || !out || !shape_ok(rows, n)) return ISO_ERR_INVALID_ARG;
    return backward_impl<float>(grad, blocks, w, nullptr, nullptr, rows, n, out, nullptr,
                                workspace, workspace_bytes, stream);
}

iso_status iso_backward_f64(const double* grad, const uint8_t* blocks, const double* w,
                            int64_t rows, int64_t n, double* out, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if (empty_call(rows, n)) return ISO_OK;
    if (!grad || !blocks || !out || !shape_ok(rows, n)) return ISO_ERR_INVALID_ARG;
    return backward_impl<double>(grad, blocks, w, nullptr, nullptr, rows, n, out, nullptr,
                                 workspace, workspace_bytes, stream);
}

iso_status iso_backward_w(const float* grad, const uint8_t* blocks, const float* w, const float* y,
                          const float* fit, int64_t rows, int64_t n, float* out_dy, float* out_dw,
                          void* workspace, size_t workspace_bytes, void* stream) {
    if (empty_call(rows, n)) return ISO_OK;
    if (!grad || !blocks || !y || !fit || !out_dw || !shape_ok(rows, n)) return ISO_ERR_INVALID_ARG;
    return backward_impl<float>(grad, blocks, w, y, fit, rows, n, out_dy, out_dw, workspace,
                                workspace_bytes, stream);
}

iso_status iso_backward_w_f64(const double* grad, const uint8_t* blocks, const double* w,
                              const double* y, const double* fit, int64_t rows, int64_t n,
                              double* out_dy, double* out_dw, void* workspace,
                              size_t workspace_bytes, void* stream) {
    if (empty_call(rows, n)) return ISO_OK;
    if (!grad || !blocks || !y || !fit || !out_dw || !shape_ok(rows, n)) return ISO_ERR_INVALID_ARG;
    return backward_impl<double>(grad, blocks, w, y, fit, rows, n, out_dy, out_dw, workspace,
                                 workspace_bytes, stream);
}

int iso_profile_enable(int on) {
    auto& P = isodev::g_prof;
    if (on && !P.created) {
        for (int i = 0; i <= isodev::kProfMax; ++i)
            if (cudaEventCreate(&P.ev[i]) != cudaSuccess) return ISO_ERR_CUDA;
        P.created = true;
    }
    P.on = on != 0;
    P.count = 0;
    P.started = false;
    return ISO_OK;
}

int iso_profile_read(float* ms, const char** names, int max_kernels) {
    auto& P = isodev::g_prof;
    if (!P.created || !P.started) return ISO_ERR_INVALID_ARG;
    const int k = P.count < max_kernels ? P.count : max_kernels;
    if (k > 0 && cudaEventSynchronize(P.ev[P.count]) != cudaSuccess) return ISO_ERR_CUDA;
    for (int i = 0; i < k; ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, P.ev[i], P.ev[i + 1]) != cudaSuccess) return ISO_ERR_CUDA;
        if (ms) ms[i] = t;
        if (names) names[i] = P.name[i];
    }
    return k;
}

iso_status iso_bridge_stats_mode(int mode) { return isodev::bridge_stats_mode(mode); }

iso_status iso_bridge_stats_read(uint64_t* out) { return isodev::bridge_stats_read(out); }

}  // extern "C"
