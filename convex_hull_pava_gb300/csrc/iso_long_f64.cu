// Long rows, float64 I/O (the templates are in iso_long.cuh; root-edge slopes
// in double).
#define ISO_LONG_F64_IO
#include "iso_long.cuh"

namespace isodev {

#define ISO_LONG_INSTANTIATE(IO)                                                                 \
    template cudaError_t long_fit<IO>(const IO*, const IO*, int64_t, int64_t, int, IO*, uint8_t*, \
                                      void*, size_t, uint32_t*, cudaStream_t);                   \
    template cudaError_t long_fit_ragged<IO>(const IO*, const IO*, const int64_t*,               \
                                             const int32_t*, const unsigned long long*, int64_t, \
                                             int64_t, int, IO*, uint8_t*, void*, uint32_t*,      \
                                             cudaStream_t);                                      \
    template cudaError_t long_fit_control<IO>(const IO*, const IO*, int64_t, int64_t, int, IO*,  \
                                              uint8_t*, void*, uint32_t*, cudaStream_t);
ISO_LONG_INSTANTIATE(double)
#undef ISO_LONG_INSTANTIATE

}  // namespace isodev
