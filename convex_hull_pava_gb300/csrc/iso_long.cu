// Long rows, float32 I/O, and the workspace sizes (the templates are in
// iso_long.cuh).
#include "iso_long.cuh"

namespace isodev {

size_t long_fit_workspace(int64_t rows, int64_t n, bool weighted) {
    const int64_t C = weighted ? LongCfg<true>::C : LongCfg<false>::C;
    const int64_t M = rows * ((n + C - 1) / C);
    return weighted ? carve<true>(nullptr, rows, M, nullptr) : carve<false>(nullptr, rows, M, nullptr);
}

size_t long_ragged_workspace(int64_t rows_max, int64_t total, bool weighted) {
    return weighted ? carve_ragged<true>(nullptr, rows_max, total, nullptr, nullptr)
                    : carve_ragged<false>(nullptr, rows_max, total, nullptr, nullptr);
}

size_t long_control_workspace(int64_t rows, int64_t n, bool weighted) {
    const int64_t C = weighted ? LongCfg<true>::C : LongCfg<false>::C;
    const int64_t M = rows * ((n + C - 1) / C);
    return weighted ? carve<true>(nullptr, rows, M, nullptr) + carve_ctl<true>(nullptr, rows, M, nullptr)
                    : carve<false>(nullptr, rows, M, nullptr) + carve_ctl<false>(nullptr, rows, M, nullptr);
}

#define ISO_LONG_INSTANTIATE(IO)                                                                 \
    template cudaError_t long_fit<IO>(const IO*, const IO*, int64_t, int64_t, int, IO*, uint8_t*, \
                                      void*, size_t, uint32_t*, cudaStream_t);                   \
    template cudaError_t long_fit_ragged<IO>(const IO*, const IO*, const int64_t*,               \
                                             const int32_t*, const unsigned long long*, int64_t, \
                                             int64_t, int, IO*, uint8_t*, void*, uint32_t*,      \
                                             cudaStream_t);                                      \
    template cudaError_t long_fit_control<IO>(const IO*, const IO*, int64_t, int64_t, int, IO*,  \
                                              uint8_t*, void*, uint32_t*, cudaStream_t);
ISO_LONG_INSTANTIATE(float)
#undef ISO_LONG_INSTANTIATE

}  // namespace isodev
