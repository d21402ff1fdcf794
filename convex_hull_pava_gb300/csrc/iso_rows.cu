// Whole-row kernels, float32 I/O (the templates are in iso_rows.cuh).
#include "iso_rows.cuh"

namespace isodev {

template cudaError_t rows_fit<float>(const float*, const float*, int64_t, int, int, float*,
                                     uint8_t*, uint32_t*, cudaStream_t);
template cudaError_t rows_fit_ragged<float>(const float*, const float*, const int64_t*,
                                            const int32_t*, const unsigned long long*, int64_t,
                                            int, int, float*, uint8_t*, uint32_t*, cudaStream_t);

}  // namespace isodev
