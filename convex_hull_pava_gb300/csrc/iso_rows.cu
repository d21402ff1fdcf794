// Whole-row kernels: every row fits in one tile of L lanes (n <= 32 * L), so
// its hull is finished inside the CTA and the fit is written directly.  Rows
// of up to 1,024 elements take one warp (or a fraction of one: L = 1..32
// lanes, several rows per warp, the paper's Section 3.5); rows of up to 8,192
// elements take one CTA of up to 256 threads (Section 6, "Blocks and memory").
#include "iso_internal.h"
#include "iso_tile.cuh"

namespace isodev {

// Fit of whole rows: CTA of NT threads, R = NT / L rows of L lanes each.
template <int NT, bool WEIGHTED>
__global__ void __launch_bounds__(NT)
rows_fit_kernel(const float* __restrict__ y, const float* __restrict__ w, int64_t rows, int n,
                int L, int increasing, float* __restrict__ out, uint8_t* __restrict__ blocks,
                uint32_t* __restrict__ row_status) {
    extern __shared__ __align__(128) unsigned char smem[];
    using SM = TileSmem<NT, WEIGHTED>;
    const int R = NT / L;
    const int tile = threadIdx.x / L;
    const int64_t row = (int64_t)blockIdx.x * R + tile;
    const bool live = row < rows;
    const float* yr = y + (live ? row : 0) * (int64_t)n;
    const float* wr = WEIGHTED ? w + (live ? row : 0) * (int64_t)n : nullptr;
    const bool neg = !increasing;

    TileHull H;
    tile_hull_phase<NT, WEIGHTED>(yr, wr, n, live, neg, L, smem, H);

    float* stage = reinterpret_cast<float*>(smem + SM::oStage);
    uint8_t* bst = smem + SM::oBst;
    const Tile& T = H.T;
    const int lane = H.lane, gl = H.gl, e = H.e;
    const bool work = live && H.bad == 0;

    // ---- emit the fit: each element gets the slope of the hull edge above it
    // (eq. (3)); an element whose point is a vertex starts a block. ----
    if (work && e > 0) {
        const int p0 = lane << 5;
        const uint32_t mask = T.mask[lane];
        int a = (mask & 1u) ? p0 : tile_pred(T, p0, 0);
        int k = 0;
        while (k < e) {
            const int b = tile_succ(T, p0 + k, L, n);
            const int kend = min(b - p0, e);
            float slope;
            if (b == a + 1) {
                slope = stage[spos(gl, k)];            // one-element block: its own value
            } else {
                slope = tile_slope<WEIGHTED>(T, a, b, H.qs, H.qw);
            }
            if (neg) slope = -slope;
            for (int j = k; j < kend; ++j) {
                stage[spos(gl, j)] = slope;
                bst[(gl << 5) + j] = (uint8_t)(p0 + j == a);
            }
            k = kend;
            a = b;
        }
    }
    __syncthreads();

    // ---- coalesced write-out ----
    if (live) {
        const int lane_in = threadIdx.x - H.tile * L;
        float* orow = out + row * (int64_t)n;
        uint8_t* brow = blocks ? blocks + row * (int64_t)n : nullptr;
        const float qnan = __int_as_float(0x7fffffff);
        for (int i = lane_in; i < n; i += L) {
            const int g = H.tile * L + (i >> 5);
            if (work) {
                orow[i] = stage[spos(g, i & 31)];
                if (brow) brow[i] = bst[(g << 5) + (i & 31)];
            } else {
                orow[i] = qnan;
                if (brow) brow[i] = 0;
            }
        }
        if (row_status && lane_in == 0) row_status[row] = H.bad;
    }
}

template <int NT, bool WEIGHTED>
static cudaError_t launch_rows_fit(const float* y, const float* w, int64_t rows, int n, int L,
                                   int increasing, float* out, uint8_t* blocks,
                                   uint32_t* row_status, cudaStream_t stream) {
    using SM = TileSmem<NT, WEIGHTED>;
    auto kern = rows_fit_kernel<NT, WEIGHTED>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           SM::kBytes);
    if (err != cudaSuccess) return err;
    const int R = NT / L;
    const int64_t grid = (rows + R - 1) / R;
    kern<<<(unsigned)grid, NT, SM::kBytes, stream>>>(y, w, rows, n, L, increasing, out, blocks,
                                                    row_status);
    prof_mark(stream, "rows_fit");
    return cudaGetLastError();
}

// n <= 8192.  Lanes per row: the smallest power of two L with 32 L >= n.
cudaError_t rows_fit(const float* y, const float* w, int64_t rows, int n, int increasing,
                     float* out, uint8_t* blocks, uint32_t* row_status, cudaStream_t stream) {
    int L = 1;
    while (32 * L < n) L <<= 1;
    const bool weighted = w != nullptr;
    if (L <= 32) {
        // several rows per CTA of 128 threads
        return weighted ? launch_rows_fit<128, true>(y, w, rows, n, L, increasing, out, blocks,
                                                     row_status, stream)
                        : launch_rows_fit<128, false>(y, w, rows, n, L, increasing, out, blocks,
                                                      row_status, stream);
    }
    if (L <= 64)
        return weighted ? launch_rows_fit<64, true>(y, w, rows, n, L, increasing, out, blocks,
                                                    row_status, stream)
                        : launch_rows_fit<64, false>(y, w, rows, n, L, increasing, out, blocks,
                                                     row_status, stream);
    if (L <= 128)
        return weighted ? launch_rows_fit<128, true>(y, w, rows, n, L, increasing, out, blocks,
                                                     row_status, stream)
                        : launch_rows_fit<128, false>(y, w, rows, n, L, increasing, out, blocks,
                                                      row_status, stream);
    return weighted ? launch_rows_fit<256, true>(y, w, rows, n, L, increasing, out, blocks,
                                                 row_status, stream)
                    : launch_rows_fit<256, false>(y, w, rows, n, L, increasing, out, blocks,
                                                  row_status, stream);
}

}  // namespace isodev
