// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/iso.h"

namespace isodev {

// Optional per-kernel timing (see iso_profile_enable): marks the start of an
// API call, and the end of each kernel it launches.
void prof_start(cudaStream_t stream);
void prof_mark(cudaStream_t stream, const char* name);

// The bridge-search counters of the current device (nullptr unless counting is
// on) and the passes a segment-list search takes before its nested bisection.
struct BridgeDebug {
    unsigned long long* stats;
    int max_passes;
};
BridgeDebug bridge_debug();

// The current device's SM count (queried once per device; 1 if unknown).
int device_sms();
iso_status bridge_stats_mode(int mode);
iso_status bridge_stats_read(uint64_t* out);

// Longest row handled by the whole-row kernels (one CTA of 256 lanes x 32).
constexpr int kRowMax = 8192;

// IO: float or double (the I/O type; the arithmetic is the same fixed point).
template <class IO>
cudaError_t rows_fit(const IO* y, const IO* w, int64_t rows, int n, int increasing, IO* out,
                     uint8_t* blocks, uint32_t* row_status, cudaStream_t stream);

// Backward: out (may be null) gets d/dy; dw, when not null, gets d/dw from the
// forward's input y and fit.
template <class IO>
cudaError_t rows_backward(const IO* grad, const uint8_t* blocks, const IO* w, int64_t rows, int n,
                          IO* out, const IO* y, const IO* fit, IO* dw, cudaStream_t stream);

// Long rows (n > kRowMax): chunk hulls, segment-list merge tree, expansion.
size_t long_fit_workspace(int64_t rows, int64_t n, bool weighted);
template <class IO>
cudaError_t long_fit(const IO* y, const IO* w, int64_t rows, int64_t n, int increasing, IO* out,
                     uint8_t* blocks, void* ws, size_t ws_bytes, uint32_t* row_status,
                     cudaStream_t stream);

// Ragged batches (iso_ragged.cu): segments laid end to end, offsets on the
// device.  The segments of each lane class L (n <= 32 L) and the long ones
// are listed on the device; `count` is the list's length (device), `cap` its
// capacity.  A grid of at most kRaggedCtas CTAs walks a class's list.
constexpr int64_t kRaggedCtas = 152 * 16;
size_t ragged_workspace(int64_t segments, int64_t total, int64_t max_len, bool weighted);
template <class IO>
cudaError_t ragged_fit(const IO* y, const IO* w, const int64_t* off, int64_t segments,
                       int64_t total, int64_t max_len, int increasing, IO* out, uint8_t* blocks,
                       void* ws, uint32_t* row_status, cudaStream_t stream);
template <class IO>
cudaError_t rows_fit_ragged(const IO* y, const IO* w, const int64_t* off, const int32_t* list,
                            const unsigned long long* count, int64_t cap, int L, int increasing,
                            IO* out, uint8_t* blocks, uint32_t* row_status, cudaStream_t stream);
size_t long_ragged_workspace(int64_t rows_max, int64_t total, bool weighted);
template <class IO>
cudaError_t long_fit_ragged(const IO* y, const IO* w, const int64_t* off,
                            const int32_t* long_id, const unsigned long long* nlong,
                            int64_t rows_max, int64_t total, int increasing, IO* out,
                            uint8_t* blocks, void* ws, uint32_t* row_status, cudaStream_t stream);

// The materialised-copy control of the merge levels (measurement only): the
// same fit as long_fit, with every merged hull copied into a flat array.
size_t long_control_workspace(int64_t rows, int64_t n, bool weighted);
template <class IO>
cudaError_t long_fit_control(const IO* y, const IO* w, int64_t rows, int64_t n, int increasing,
                             IO* out, uint8_t* blocks, void* ws, uint32_t* row_status,
                             cudaStream_t stream);

size_t long_backward_workspace(int64_t rows, int64_t n, bool weighted);
template <class IO>
cudaError_t long_backward(const IO* grad, const uint8_t* blocks, const IO* w, int64_t rows,
                          int64_t n, IO* out, const IO* y, const IO* fit, IO* dw, void* ws,
                          size_t ws_bytes, cudaStream_t stream);

}  // namespace isodev
