// Whole-row kernels, float64 I/O (the templates are in iso_rows.cuh).
#include "iso_rows.cuh"

namespace isodev {

template cudaError_t rows_fit<double>(const double*, const double*, int64_t, int, int, double*,
                                      uint8_t*, uint32_t*, cudaStream_t);
template cudaError_t rows_fit_ragged<double>(const double*, const double*, const int64_t*,
                                             const int32_t*, const unsigned long long*, int64_t,
                                             int, int, double*, uint8_t*, uint32_t*,
                                             cudaStream_t);

}  // namespace isodev
