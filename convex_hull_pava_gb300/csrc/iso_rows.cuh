// Whole-row kernels (templates; iso_rows.cu and iso_rows_f64.cu instantiate
// them for float and double I/O).  Every row fits in one tile of L lanes (n <= 32 * L), so
// its hull is finished inside the CTA and the fit is written directly.  Rows
// of up to 1,024 elements take one warp (or a fraction of one: L = 1..32
// lanes, several rows per warp, the paper's Section 3.5); rows of up to 8,192
// elements take one CTA of up to 256 threads (Section 6, "Blocks and memory").
#pragma once

#include "iso_internal.h"
#include "iso_tile.cuh"

#include <algorithm>

namespace isodev {

// Fit of the rows of one CTA of NT threads: R = NT / L tiles of L lanes, each
// thread's tile a row of n <= 32 L elements at yr (wr), its fit written to
// orow and its block flags to brow (may be null), its status to *status (may
// be null).  A tile that is not live reads and writes nothing.  `mark0`: a
// rejected row still flags its first element as a block start (ragged
// batches, where each segment's first element must start a block).  Every
// thread of the CTA calls it.
template <int NT, int RMAX, bool WEIGHTED, class IO>
__device__ __forceinline__ void fit_row_tiles(const IO* __restrict__ yr,
                                              const IO* __restrict__ wr, int n, bool live,
                                              int L, bool neg, IO* __restrict__ orow,
                                              uint8_t* __restrict__ brow, uint32_t* status,
                                              bool mark0, unsigned char* smem) {
    using SM = TileSmem<NT, WEIGHTED, true, RMAX, IO>;
    TileHull H;
    tile_hull_phase<NT, WEIGHTED, true, RMAX, IO>(yr, wr, n, live, neg, L, smem, H);

    if constexpr (RMAX == 1) {
        if (H.oneblock && live && H.bad == 0 && n > 1) {
            // the row is one block: every element is fitted by its mean, the
            // slope from the first point to the end (as the vertex's slope
            // below), written with 16-byte stores; one block start, element 0
            __shared__ IO s_mean;
            if (threadIdx.x == 0)
                s_mean = ratio_t<IO>(H.T.LS[L], WEIGHTED ? H.T.LW[L] : (int64_t)n, H.qs - H.qw);
            __syncthreads();
            const IO v = neg ? -s_mean : s_mean;
            const int lane = H.lane;
            if ((reinterpret_cast<uintptr_t>(orow) & 15u) == 0) {
                using V = typename IoT<IO>::V;
                constexpr int P = IoT<IO>::kPerV;
                V vv;
                IO* pv = reinterpret_cast<IO*>(&vv);
#pragma unroll
                for (int u = 0; u < P; ++u) pv[u] = v;
                const int nv = n / P;
                for (int i = lane; i < nv; i += L) reinterpret_cast<V*>(orow)[i] = vv;
                for (int i = nv * P + lane; i < n; i += L) orow[i] = v;
            } else {
                for (int i = lane; i < n; i += L) orow[i] = v;
            }
            if (brow) {
                if ((reinterpret_cast<uintptr_t>(brow) & 3u) == 0) {
                    const int n4 = n >> 2;
                    for (int i = lane; i < n4; i += L) reinterpret_cast<uint32_t*>(brow)[i] = i == 0 ? 1u : 0u;
                    for (int i = (n4 << 2) + lane; i < n; i += L) brow[i] = i == 0 ? 1 : 0;
                } else {
                    for (int i = lane; i < n; i += L) brow[i] = i == 0 ? 1 : 0;
                }
            }
            if (status && lane == 0) *status = 0;
            return;
        }
    }

    const Tile& T = H.T;
    const int lane = H.lane, gl = H.gl, e = H.e;
    const bool work = live && H.bad == 0;
    const uint32_t mask = work ? T.mask[lane] : 0u;
    int64_t* Sx = reinterpret_cast<int64_t*>(smem + SM::oSx);
    const int64_t* myS = Sx + gl * kRow;            // tile-relative sums at the lane's points
    const int64_t* myW = reinterpret_cast<const int64_t*>(smem + SM::oWx) + gl * kRow;
    IO* mySlope = reinterpret_cast<IO*>(Sx + gl * kRow);

    // ---- 1. every vertex: the slope of the hull edge leaving it (eq. (3)).  A
    // one-element block is fitted by its own value, read again from y.  A lane
    // writes its vertices' slopes over its own row of sums (slot k for the
    // vertex at bit k, which covers only sums at or before point k, not read
    // again once that vertex's slope is known); the sums at the vertex after
    // its last one, in a later lane's row or at the tile's end, are read
    // before any lane writes. ----
    const int bl = mask ? tile_succ(T, (lane << 5) + 31 - __clz(mask), L, n) : 0;
    const int64_t Sbl = mask ? tile_S<WEIGHTED>(T, bl) : 0;
    const int64_t Wbl = mask ? tile_W<WEIGHTED>(T, bl) : 0;
    __syncthreads();
    {
        uint32_t m = mask;
        while (m) {
            const int k = __ffs(m) - 1;
            m &= m - 1u;
            const int k2 = m ? __ffs(m) - 1 : -1;         // this lane's next vertex
            const int v = (lane << 5) + k;
            const int b = k2 >= 0 ? (lane << 5) + k2 : bl;
            IO sl;
            if (b == v + 1) {
                const IO yv = __ldg(yr + v);
                sl = neg ? -yv : yv;
            } else {
                const int64_t Sb = k2 >= 0 ? myS[k2] : Sbl;
                const int64_t Wb = k2 >= 0 ? (WEIGHTED ? myW[k2] : (int64_t)b) : Wbl;
                const int64_t Wv = WEIGHTED ? myW[k] : (int64_t)v;
                sl = ratio_t<IO>(Sb - myS[k], Wb - Wv, H.qs - H.qw);
            }
            mySlope[k] = sl;
        }
    }
    __syncthreads();
    // ---- 2. every element: the slope of the edge leaving the last vertex at or
    // before it ----
    IO o[32];
    {
        IO carry = IO(0);
        if (work && e > 0 && !(mask & 1u)) {
            const int cv = tile_pred(T, lane << 5, 0);
            carry = reinterpret_cast<const IO*>(Sx + (H.tile * L + (cv >> 5)) * kRow)[cv & 31];
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const uint32_t upto = k == 31 ? mask : (mask & ((2u << k) - 1u));
            const IO v = upto ? mySlope[31 - __clz(upto)] : carry;
            o[k] = neg ? -v : v;
        }
    }
    __syncthreads();   // Sx is dead: stage the output in Sx
    IO* ost = reinterpret_cast<IO*>(smem + SM::oSx);
    stage_out<IO>(ost, gl, o);
    __syncthreads();

    // ---- coalesced write-out of the fit and of the block-start bytes ----
    if (live) {
        const int g0 = H.tile * L;
        write_row<IO>(orow, ost, g0, n, lane, L, work);
        if (brow) {
            const uint32_t* ma = T.mask;
            if ((reinterpret_cast<uintptr_t>(brow) & 3u) == 0) {
                const int n4 = n >> 2;
                for (int i = lane; i < n4; i += L) {
                    const int e4 = i << 2;
                    const uint32_t bits = work ? (ma[e4 >> 5] >> (e4 & 31)) & 0xfu : 0u;
                    const uint32_t word = (bits & 1u) | ((bits & 2u) << 7) | ((bits & 4u) << 14) |
                                          ((bits & 8u) << 21);
                    reinterpret_cast<uint32_t*>(brow)[i] = word;
                }
                for (int i = (n4 << 2) + lane; i < n; i += L)
                    brow[i] = work ? (uint8_t)((ma[i >> 5] >> (i & 31)) & 1u) : 0;
            } else {
                for (int i = lane; i < n; i += L)
                    brow[i] = work ? (uint8_t)((ma[i >> 5] >> (i & 31)) & 1u) : 0;
            }
            if (mark0 && !work && lane == 0) brow[0] = 1;   // lane 0 wrote element 0 above
        }
        if (status && lane == 0) *status = H.bad;
    }
}

// CTAs per SM that a kernel's shared memory allows (228 KB per SM, 1 KB of it
// reserved per CTA, at most 2,048 threads): the float32 kernels' registers are
// held to that occupancy, so they never limit it further; the float64 ones,
// whose 32 staged values take twice the registers, get 128 per thread.
template <int NT, int RMAX, bool WEIGHTED, class IO>
constexpr int rows_min_blocks() {
    constexpr int by_smem = (228 * 1024) / (TileSmem<NT, WEIGHTED, true, RMAX, IO>::kBytes + 1024);
    constexpr int by_threads = sizeof(IO) == 4 ? 2048 / NT : 512 / NT;
    constexpr int b = by_smem < by_threads ? by_smem : by_threads;
    return b < 1 ? 1 : b;
}

// Fit of whole rows: CTA of NT threads, R = NT / L rows of L lanes each.
template <int NT, int RMAX, bool WEIGHTED, class IO>
__global__ void __launch_bounds__(NT, rows_min_blocks<NT, RMAX, WEIGHTED, IO>())
rows_fit_kernel(const IO* __restrict__ y, const IO* __restrict__ w, int64_t rows, int n,
                int L, int increasing, IO* __restrict__ out, uint8_t* __restrict__ blocks,
                uint32_t* __restrict__ row_status) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int R = NT / L;
    const int64_t row = (int64_t)blockIdx.x * R + threadIdx.x / L;
    const bool live = row < rows;
    const int64_t e0 = (live ? row : 0) * (int64_t)n;
    fit_row_tiles<NT, RMAX, WEIGHTED, IO>(y + e0, WEIGHTED ? w + e0 : nullptr, n, live, L,
                                          !increasing, out + e0, blocks ? blocks + e0 : nullptr,
                                          row_status ? row_status + (live ? row : 0) : nullptr,
                                          false, smem);
}

// Fit of the segments of one lane class of a ragged batch: list[0 .. count)
// holds segment indices s, each of n = off[s+1] - off[s] <= 32 L elements at
// element off[s].  Persistent: each CTA takes R segments at a time.
template <int NT, int RMAX, bool WEIGHTED, class IO>
__global__ void __launch_bounds__(NT)
rows_fit_ragged_kernel(const IO* __restrict__ y, const IO* __restrict__ w,
                       const int64_t* __restrict__ off, const int32_t* __restrict__ list,
                       const unsigned long long* __restrict__ count, int64_t cap, int L,
                       int increasing, IO* __restrict__ out, uint8_t* __restrict__ blocks,
                       uint32_t* __restrict__ row_status) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int R = NT / L;
    const int tile = threadIdx.x / L;
    const int64_t cnt = (int64_t)min((unsigned long long)cap, *count);
    for (int64_t b = (int64_t)blockIdx.x * R; b < cnt; b += (int64_t)gridDim.x * R) {
        const int64_t i = b + tile;
        const bool live = i < cnt;
        int64_t e0 = 0;
        int n = 0, s = 0;
        if (live) {
            s = list[i];
            e0 = off[s];
            n = (int)(off[s + 1] - e0);
        }
        fit_row_tiles<NT, RMAX, WEIGHTED, IO>(y + e0, WEIGHTED ? w + e0 : nullptr, n, live, L,
                                              !increasing, out + e0,
                                              blocks ? blocks + e0 : nullptr,
                                              row_status ? row_status + s : nullptr, true, smem);
        __syncthreads();   // shared memory is reused by the next segments
    }
}

template <int NT, int RMAX, bool WEIGHTED, class IO>
static cudaError_t launch_rows_fit(const IO* y, const IO* w, int64_t rows, int n, int L,
                                   int increasing, IO* out, uint8_t* blocks,
                                   uint32_t* row_status, cudaStream_t stream) {
    using SM = TileSmem<NT, WEIGHTED, true, RMAX, IO>;
    auto kern = rows_fit_kernel<NT, RMAX, WEIGHTED, IO>;
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
// RMAX bounds the rows of a CTA (its per-row arrays in shared memory): 128
// for L <= 16, 4 for L = 32, 1 for rows of a CTA of their own.
template <class IO>
cudaError_t rows_fit(const IO* y, const IO* w, int64_t rows, int n, int increasing, IO* out,
                     uint8_t* blocks, uint32_t* row_status, cudaStream_t stream) {
    int L = 1;
    while (32 * L < n) L <<= 1;
    const bool weighted = w != nullptr;
#define ISO_ROWS_LAUNCH(NT_, RMAX_)                                                             \
    return weighted ? launch_rows_fit<NT_, RMAX_, true, IO>(y, w, rows, n, L, increasing, out,  \
                                                            blocks, row_status, stream)         \
                    : launch_rows_fit<NT_, RMAX_, false, IO>(y, w, rows, n, L, increasing, out, \
                                                             blocks, row_status, stream)
    if (L <= 16) { ISO_ROWS_LAUNCH(128, 128); }   // several rows per CTA of 128 threads
    if (L <= 32) { ISO_ROWS_LAUNCH(128, 4); }
    if (L <= 64) { ISO_ROWS_LAUNCH(64, 1); }      // one row per CTA
    if (L <= 128) { ISO_ROWS_LAUNCH(128, 1); }
    ISO_ROWS_LAUNCH(256, 1);
#undef ISO_ROWS_LAUNCH
}

template <int NT, int RMAX, bool WEIGHTED, class IO>
static cudaError_t launch_rows_ragged(const IO* y, const IO* w, const int64_t* off,
                                      const int32_t* list, const unsigned long long* count,
                                      int64_t cap, int L, int increasing, IO* out,
                                      uint8_t* blocks, uint32_t* row_status, cudaStream_t stream) {
    using SM = TileSmem<NT, WEIGHTED, true, RMAX, IO>;
    auto kern = rows_fit_ragged_kernel<NT, RMAX, WEIGHTED, IO>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           SM::kBytes);
    if (err != cudaSuccess) return err;
    const int R = NT / L;
    const int64_t grid = std::min<int64_t>((cap + R - 1) / R, kRaggedCtas);
    kern<<<(unsigned)grid, NT, SM::kBytes, stream>>>(y, w, off, list, count, cap, L, increasing,
                                                    out, blocks, row_status);
    prof_mark(stream, "rows_ragged");
    return cudaGetLastError();
}

template <class IO>
cudaError_t rows_fit_ragged(const IO* y, const IO* w, const int64_t* off, const int32_t* list,
                            const unsigned long long* count, int64_t cap, int L, int increasing,
                            IO* out, uint8_t* blocks, uint32_t* row_status, cudaStream_t stream) {
    const bool weighted = w != nullptr;
#define ISO_RAGGED_LAUNCH(NT_, RMAX_)                                                           \
    return weighted ? launch_rows_ragged<NT_, RMAX_, true, IO>(y, w, off, list, count, cap, L,  \
                                                               increasing, out, blocks,         \
                                                               row_status, stream)              \
                    : launch_rows_ragged<NT_, RMAX_, false, IO>(y, w, off, list, count, cap, L, \
                                                                increasing, out, blocks,        \
                                                                row_status, stream)
    if (L <= 16) { ISO_RAGGED_LAUNCH(128, 128); }
    if (L <= 32) { ISO_RAGGED_LAUNCH(128, 4); }
    if (L <= 64) { ISO_RAGGED_LAUNCH(64, 1); }
    if (L <= 128) { ISO_RAGGED_LAUNCH(128, 1); }
    ISO_RAGGED_LAUNCH(256, 1);
#undef ISO_RAGGED_LAUNCH
}

}  // namespace isodev
