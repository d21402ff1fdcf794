// Backward of the fit (the paper's Section 6, "Gradient"): the fit is the
// weighted block mean, so its vector-Jacobian product is block averaging,
// d/dy_i = w_i * G / W with G, W the sums of grad and w over element i's block.
// Blocks are given by the block-start bytes of the forward pass.
//
// Sums are exact: grad and w are rounded to a fixed-point grid of 2^-31 of the
// tile's largest magnitude and summed as integers, so the result does not
// depend on the order of the additions.  A row that is one tile is finished in
// one kernel; a longer row takes three steps (tile sums, a pass over the
// tiles' boundary sums, and the fill of blocks that cross tiles), as in the
// paper, without atomics.
#include "iso_internal.h"
#include "iso_tile.cuh"

namespace isodev {

namespace {

// Shared memory of a backward tile of NT lanes: grad and w staging, the
// block-prefix sums of both, masks of block starts and scan scratch.
template <int NT>
struct BwdSmem {
    static constexpr int oStage = 0;                              // grad (later the output)
    static constexpr int oStageW = oStage + NT * 128;             // w
    static constexpr int oSx = oStageW + NT * 128;                // block prefix of grad
    static constexpr int oWx = oSx + NT * kRow * 8;               // block prefix of w
    static constexpr int oMask = oWx + NT * kRow * 8;
    static constexpr int oSumm = oMask + NT * 4;
    static constexpr int oInfo = oSumm + ((NT + 63) / 64) * 8;
    static constexpr int oScan = oInfo + NT * 16;
    static constexpr int oLS = oScan + (NT / 16 + 2) * 8;         // per-lane inclusive carries
    static constexpr int oLW = oLS + NT * 8;
    static constexpr int oBridge = oLW + NT * 8;                  // scan flags
    static constexpr int kBytes = ((oBridge + NT * 4 + 127) / 128) * 128;
};

// Block sums of one tile: on return, stage holds, for every element whose
// block both starts and ends inside the tile, its output value; `Px`/`Qx` hold
// the block-prefix sums (fixed point) of grad and w, restarting at each block
// start and at the tile's first element.  Tail/head information is returned
// for the long-row path.
struct BwdTile {
    int first_start;   // first block start in the tile, or -1
    int last_start;    // last block start in the tile, or -1
    int qg, qw;        // quantum exponents of grad and w
    bool nan;          // a non-finite grad or an invalid weight in the tile
};

template <int NT, bool WEIGHTED>
__device__ __forceinline__ void bwd_tile_phase(const float* __restrict__ gr,
                                               const uint8_t* __restrict__ br,
                                               const float* __restrict__ wr, int nt, bool live,
                                               bool first_is_start, int L, unsigned char* smem,
                                               BwdTile& B) {
    using SM = BwdSmem<NT>;
    float* stage = reinterpret_cast<float*>(smem + SM::oStage);
    int64_t* Px = reinterpret_cast<int64_t*>(smem + SM::oSx);
    int64_t* Qx = reinterpret_cast<int64_t*>(smem + SM::oWx);
    float* stagew = reinterpret_cast<float*>(smem + SM::oStageW);
    uint32_t* maska = reinterpret_cast<uint32_t*>(smem + SM::oMask);
    uint32_t* summ = reinterpret_cast<uint32_t*>(smem + SM::oSumm);
    int* info = reinterpret_cast<int*>(smem + SM::oInfo);
    int64_t* scan = reinterpret_cast<int64_t*>(smem + SM::oScan);
    int64_t* incl = reinterpret_cast<int64_t*>(smem + SM::oLS);
    int64_t* inclw = reinterpret_cast<int64_t*>(smem + SM::oLW);
    int* scanf = reinterpret_cast<int*>(smem + SM::oBridge);

    const int tid = threadIdx.x;
    const int tile = tid / L;
    const int lane = tid - tile * L;
    const int gl = tid;

    for (int i = lane; i < 4; i += L) info[tile * 4 + i] = 0;
    __syncthreads();
    int gmax = 0, ewmax = 0;
    uint32_t bad = 0;
    uint32_t starts = 0;
    const int e = live ? min(max(nt - (lane << 5), 0), 32) : 0;
    if (live) {
        stage_tile<false>(gr, nt, lane, L, tile * L, false, stage, gmax, bad);
        if constexpr (WEIGHTED) stage_tile<true>(wr, nt, lane, L, tile * L, false, stagew, ewmax, bad);
        // the lane's 32 block-start bytes, as a bit mask
        const uint8_t* bl = br + (lane << 5);
        if (e == 32 && (reinterpret_cast<uintptr_t>(bl) & 15u) == 0) {
            const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(bl));
            const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(bl) + 1);
            const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                // high bit of each byte set iff the byte is non-zero
                const uint32_t h = ((wd[q] & 0x7f7f7f7fu) + 0x7f7f7f7fu) | wd[q];
                const uint32_t b4 = (((h >> 7) & 0x01010101u) * 0x01020408u) >> 24;
                starts |= (b4 & 0xfu) << (4 * q);
            }
        } else {
            uint8_t v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = k < e ? __ldg(bl + k) : (uint8_t)0;
#pragma unroll
            for (int k = 0; k < 32; ++k) starts |= (v[k] != 0 ? 1u : 0u) << k;
        }
        if (lane == 0 && first_is_start) starts |= 1u;
    }
    maska[gl] = starts;
    gmax = tile_warp_max(gmax, L);
    if (WEIGHTED) ewmax = tile_warp_max(ewmax, L);
    const int bad_or = tile_warp_or((int)bad, L);
    const int seg = L < 32 ? L : 32;
    if (live && ((tid & 31) & (seg - 1)) == 0) {
        atomicMax(&info[tile * 4 + 0], gmax);
        if (WEIGHTED) atomicMax(&info[tile * 4 + 1], ewmax);
        if (bad_or) atomicOr(&info[tile * 4 + 2], 1);
    }
    __syncthreads();
    gmax = max(info[tile * 4 + 0], 1);
    ewmax = max(info[tile * 4 + 1], 1);
    B.nan = info[tile * 4 + 2] != 0;
    B.qg = qexp_unit(gmax);
    B.qw = WEIGHTED ? qexp_unit(ewmax) : 0;
    {
        const uint32_t bal = __ballot_sync(kFull, starts != 0u);
        if ((tid & 31) == 0) summ[tid >> 5] = bal;
    }

    // one pass over the lane's staged values: fixed-point grad and w, and the
    // sums after the lane's last block start (or the lane totals)
    const float4* st4 = reinterpret_cast<const float4*>(stage);
    const float4* sw4 = reinterpret_cast<const float4*>(stagew);
    auto lane_values = [&](int q, float (&vv)[4], float (&ww)[4]) {
        const int unit = (gl << 3) | ((q ^ gl) & 7);
        const float4 v = st4[unit];
        vv[0] = v.x; vv[1] = v.y; vv[2] = v.z; vv[3] = v.w;
        ww[0] = ww[1] = ww[2] = ww[3] = 1.0f;
        if constexpr (WEIGHTED) {
            const float4 t = sw4[unit];
            ww[0] = t.x; ww[1] = t.y; ww[2] = t.z; ww[3] = t.w;
        }
    };
    int64_t sg = 0, sw = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float vv[4], ww[4];
        lane_values(q, vv, ww);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = 4 * q + j;
            if ((starts >> k) & 1u) { sg = 0; sw = 0; }
            if (k < e) {
                sg += quant(vv[j], gmax);
                sw += WEIGHTED ? quant(ww[j], ewmax) : 1;
            }
        }
    }
    int64_t cg, cw;
    {
        int64_t vg = sg, vw = sw;
        int fl = starts ? 1 : 0;
        const int wl = tid & 31;
        const int seg = L < 32 ? L : 32;
        const int lseg = wl & (seg - 1);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int64_t og = __shfl_up_sync(kFull, vg, d);
            int64_t ow = __shfl_up_sync(kFull, vw, d);
            int of = __shfl_up_sync(kFull, fl, d);
            if (d < seg && lseg >= d) {
                if (!fl) { vg += og; vw += ow; }
                fl |= of;
            }
        }
        if (L > 32) {
            const int warp = tid >> 5;
            if (wl == 31) { scan[warp] = vg; scanf[warp] = fl; scan[NT / 32 + warp] = vw; }
            __syncthreads();
            const int w0 = warp - (lane >> 5);
            int64_t ag = 0, aw = 0;
            for (int q = w0; q < warp; ++q) {
                if (scanf[q]) { ag = scan[q]; aw = scan[NT / 32 + q]; }
                else { ag += scan[q]; aw += scan[NT / 32 + q]; }
            }
            if (!fl) { vg += ag; vw += aw; }
        }
        incl[gl] = vg;
        inclw[gl] = vw;
        __syncthreads();
        cg = lane ? incl[gl - 1] : 0;
        cw = lane ? inclw[gl - 1] : 0;
    }
    {
        int64_t pg = cg, pw = cw;
        int64_t* myP = Px + gl * kRow;
        int64_t* myQ = Qx + gl * kRow;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float vv[4], ww[4];
            lane_values(q, vv, ww);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = 4 * q + j;
                if ((starts >> k) & 1u) { pg = 0; pw = 0; }
                if (k < e) {
                    pg += quant(vv[j], gmax);
                    pw += WEIGHTED ? quant(ww[j], ewmax) : 1;
                }
                myP[k] = pg;
                myQ[k] = pw;
            }
        }
    }
    __syncthreads();

    Tile T;
    T.Sx = Px; T.Wx = Qx; T.LS = nullptr; T.LW = nullptr;
    T.mask = maska + tile * L; T.summ = summ; T.sbase = tile * L; T.L = L; T.nt = nt;
    {
        // first / last block start of the tile (scan of the starts masks)
        const int fl = next_nonempty(T, 0, L);
        const int ll = prev_nonempty(T, 0, L);
        B.first_start = fl < 0 ? -1 : (fl << 5) + __ffs(T.mask[fl]) - 1;
        B.last_start = ll < 0 ? -1 : (ll << 5) + 31 - __clz(T.mask[ll]);
    }

    // each element inside the tile's complete blocks: the block sums are the
    // prefixes at the block's last element, one before the next start
    const int p0 = lane << 5;
    const int qd = B.qg - B.qw;
    int cur_last = -1;
    float ratio = 0.0f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        if (k < e) {
            if (p0 + k > cur_last) {
                const int nxt = tile_succ(T, p0 + k, L, nt);
                cur_last = nxt - 1;
                const int gll = tile * L + (cur_last >> 5);
                const int64_t G = Px[gll * kRow + (cur_last & 31)];
                const int64_t Wb = Qx[gll * kRow + (cur_last & 31)];
                ratio = ldexpf(i64_to_f32(G) / i64_to_f32(Wb), qd);
                if (B.nan) ratio = __int_as_float(0x7fffffff);
            }
            stage[spos(gl, k)] = WEIGHTED ? stagew[spos(gl, k)] * ratio : ratio;
        }
    }
    __syncthreads();
}

template <int NT, bool WEIGHTED>
__global__ void __launch_bounds__(NT)
rows_backward_kernel(const float* __restrict__ grad, const uint8_t* __restrict__ blocks,
                     const float* __restrict__ w, int64_t rows, int n, int L,
                     float* __restrict__ out) {
    extern __shared__ __align__(128) unsigned char smem[];
    using SM = BwdSmem<NT>;
    const int R = NT / L;
    const int tile = threadIdx.x / L;
    const int lane = threadIdx.x - tile * L;
    const int64_t row = (int64_t)blockIdx.x * R + tile;
    const bool live = row < rows;
    const int64_t off = (live ? row : 0) * (int64_t)n;
    BwdTile B;
    bwd_tile_phase<NT, WEIGHTED>(grad + off, blocks + off, WEIGHTED ? w + off : nullptr, n, live,
                                 true, L, smem, B);
    const float* stage = reinterpret_cast<const float*>(smem + SM::oStage);
    if (live) {
        float* orow = out + off;
        for (int i = lane; i < n; i += L) orow[i] = stage[spos(tile * L + (i >> 5), i & 31)];
    }
}

// ---- long rows: tiles of 8,192 elements (256 lanes) ----
constexpr int kBT = 8192;
constexpr int kBNT = 256;

struct BwdRec {
    int32_t fs, ls;      // first / last block start in the tile (-1: none)
    int32_t nan, pad;
    double hG, hW;       // sums of the head part (elements before fs, or the whole tile)
    double tG, tW;       // sums of the tail part (elements from ls to the tile's end)
};

struct BwdTot {
    double headG, headW;   // totals of the block holding the tile's first element
    double tailG, tailW;   // totals of the block holding the tile's last element
    int32_t nan, pad0, pad1, pad2;
};

template <bool WEIGHTED>
__global__ void __launch_bounds__(kBNT)
long_bwd_tiles_kernel(const float* __restrict__ grad, const uint8_t* __restrict__ blocks,
                      const float* __restrict__ w, int64_t n, int64_t m, float* __restrict__ out,
                      BwdRec* __restrict__ rec) {
    extern __shared__ __align__(128) unsigned char smem[];
    using SM = BwdSmem<kBNT>;
    const int64_t c = blockIdx.x;
    const int64_t row = c / m;
    const int64_t j = c - row * m;
    const int64_t e0 = j * kBT;
    const int nt = (int)imin64(kBT, n - e0);
    const int64_t off = row * n + e0;
    BwdTile B;
    bwd_tile_phase<kBNT, WEIGHTED>(grad + off, blocks + off, WEIGHTED ? w + off : nullptr, nt,
                                   true, j == 0, kBNT, smem, B);
    const float* stage = reinterpret_cast<const float*>(smem + SM::oStage);
    const int64_t* Px = reinterpret_cast<const int64_t*>(smem + SM::oSx);
    const int64_t* Qx = reinterpret_cast<const int64_t*>(smem + SM::oWx);
    // elements of complete blocks: from the first start to one before the last start
    const int lo = B.first_start < 0 ? nt : B.first_start;
    const int hi = B.last_start < 0 ? nt : B.last_start;
    float* o = out + off;
    for (int i = lo + threadIdx.x; i < hi; i += kBNT) o[i] = stage[spos(i >> 5, i & 31)];
    if (threadIdx.x == 0) {
        BwdRec r;
        r.fs = B.first_start;
        r.ls = B.last_start;
        r.nan = B.nan ? 1 : 0;
        r.pad = 0;
        const double sg = ldexp(1.0, B.qg), sw = ldexp(1.0, B.qw);
        const int hl = (B.first_start < 0 ? nt : B.first_start) - 1;   // last element of the head
        if (hl >= 0) {
            r.hG = (double)Px[(hl >> 5) * kRow + (hl & 31)] * sg;
            r.hW = (double)Qx[(hl >> 5) * kRow + (hl & 31)] * sw;
        } else {
            r.hG = 0.0; r.hW = 0.0;
        }
        if (B.last_start >= 0) {
            const int tl = nt - 1;
            r.tG = (double)Px[(tl >> 5) * kRow + (tl & 31)] * sg;
            r.tW = (double)Qx[(tl >> 5) * kRow + (tl & 31)] * sw;
        } else {
            r.tG = 0.0; r.tW = 0.0;
        }
        rec[c] = r;
    }
}

// Totals of the blocks that cross tile boundaries: one thread per row walks the
// tiles backwards (continuations into later tiles) and forwards (the open block
// entering each tile).
__global__ void long_bwd_totals_kernel(int64_t rows, int64_t m, const BwdRec* __restrict__ rec,
                                       BwdTot* __restrict__ tot) {
    const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= rows) return;
    const BwdRec* rr = rec + row * m;
    BwdTot* tt = tot + row * m;
    int rownan = 0;
    for (int64_t t = 0; t < m; ++t) rownan |= rr[t].nan;
    // backwards: cont = sums of the later tiles' heads, until a tile with a start
    double contG = 0.0, contW = 0.0;
    for (int64_t t = m - 1; t >= 0; --t) {
        const BwdRec r = rr[t];
        if (r.ls >= 0) {
            tt[t].tailG = r.tG + contG;
            tt[t].tailW = r.tW + contW;
            contG = r.hG; contW = r.hW;
        } else {
            contG += r.hG; contW += r.hW;
        }
        tt[t].nan = rownan;
    }
    // forwards: the block entering tile t is the tail block of the last tile before
    // it with a start
    double openG = 0.0, openW = 0.0;
    for (int64_t t = 0; t < m; ++t) {
        tt[t].headG = openG;
        tt[t].headW = openW;
        if (rr[t].ls >= 0) { openG = tt[t].tailG; openW = tt[t].tailW; }
    }
}

template <bool WEIGHTED>
__global__ void __launch_bounds__(kBNT)
long_bwd_fill_kernel(const float* __restrict__ w, int64_t n, int64_t m,
                     const BwdRec* __restrict__ rec, const BwdTot* __restrict__ tot,
                     float* __restrict__ out) {
    const int64_t c = blockIdx.x;
    const int64_t row = c / m;
    const int64_t j = c - row * m;
    const int64_t e0 = j * kBT;
    const int nt = (int)imin64(kBT, n - e0);
    const BwdRec r = rec[c];
    const BwdTot t = tot[c];
    const int64_t off = row * n + e0;
    float* o = out + off;
    const float* wr = WEIGHTED ? w + off : nullptr;
    const float qnan = __int_as_float(0x7fffffff);
    const float rh = t.nan ? qnan : (float)(t.headG / t.headW);
    const float rt = t.nan ? qnan : (float)(t.tailG / t.tailW);
    const int hend = r.fs < 0 ? nt : r.fs;
    for (int i = threadIdx.x; i < hend; i += kBNT) o[i] = WEIGHTED ? __ldg(wr + i) * rh : rh;
    if (r.ls >= 0)
        for (int i = r.ls + threadIdx.x; i < nt; i += kBNT) o[i] = WEIGHTED ? __ldg(wr + i) * rt : rt;
    if (t.nan)
        for (int i = hend + threadIdx.x; i < (r.ls >= 0 ? r.ls : nt); i += kBNT) o[i] = qnan;
}

__host__ __device__ inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

template <int NT, bool WEIGHTED>
cudaError_t launch_rows_bwd(const float* grad, const uint8_t* blocks, const float* w,
                            int64_t rows, int n, int L, float* out, cudaStream_t stream) {
    using SM = BwdSmem<NT>;
    auto kern = rows_backward_kernel<NT, WEIGHTED>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           SM::kBytes);
    if (err != cudaSuccess) return err;
    const int R = NT / L;
    const int64_t grid = (rows + R - 1) / R;
    kern<<<(unsigned)grid, NT, SM::kBytes, stream>>>(grad, blocks, w, rows, n, L, out);
    prof_mark(stream, "rows_backward");
    return cudaGetLastError();
}

template <bool WEIGHTED>
cudaError_t long_bwd_t(const float* grad, const uint8_t* blocks, const float* w, int64_t rows,
                       int64_t n, float* out, void* ws, cudaStream_t stream) {
    using SM = BwdSmem<kBNT>;
    const int64_t m = (n + kBT - 1) / kBT;
    const int64_t M = rows * m;
    BwdRec* rec = static_cast<BwdRec*>(ws);
    BwdTot* tot = reinterpret_cast<BwdTot*>(static_cast<char*>(ws) + a256(sizeof(BwdRec) * M));
    auto k1 = long_bwd_tiles_kernel<WEIGHTED>;
    cudaError_t err = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           SM::kBytes);
    if (err != cudaSuccess) return err;
    k1<<<(unsigned)M, kBNT, SM::kBytes, stream>>>(grad, blocks, w, n, m, out, rec);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "bwd_tiles");
    long_bwd_totals_kernel<<<(unsigned)((rows + 63) / 64), 64, 0, stream>>>(rows, m, rec, tot);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "bwd_totals");
    long_bwd_fill_kernel<WEIGHTED><<<(unsigned)M, kBNT, 0, stream>>>(w, n, m, rec, tot, out);
    prof_mark(stream, "bwd_fill");
    return cudaGetLastError();
}

}  // namespace

cudaError_t rows_backward(const float* grad, const uint8_t* blocks, const float* w, int64_t rows,
                          int n, float* out, cudaStream_t stream) {
    int L = 1;
    while (32 * L < n) L <<= 1;
    const bool weighted = w != nullptr;
    if (L <= 32)
        return weighted ? launch_rows_bwd<128, true>(grad, blocks, w, rows, n, L, out, stream)
                        : launch_rows_bwd<128, false>(grad, blocks, w, rows, n, L, out, stream);
    if (L <= 64)
        return weighted ? launch_rows_bwd<64, true>(grad, blocks, w, rows, n, L, out, stream)
                        : launch_rows_bwd<64, false>(grad, blocks, w, rows, n, L, out, stream);
    if (L <= 128)
        return weighted ? launch_rows_bwd<128, true>(grad, blocks, w, rows, n, L, out, stream)
                        : launch_rows_bwd<128, false>(grad, blocks, w, rows, n, L, out, stream);
    return weighted ? launch_rows_bwd<256, true>(grad, blocks, w, rows, n, L, out, stream)
                    : launch_rows_bwd<256, false>(grad, blocks, w, rows, n, L, out, stream);
}

size_t long_backward_workspace(int64_t rows, int64_t n, bool weighted) {
    (void)weighted;
    const int64_t M = rows * ((n + kBT - 1) / kBT);
    return a256(sizeof(BwdRec) * M) + a256(sizeof(BwdTot) * M);
}

cudaError_t long_backward(const float* grad, const uint8_t* blocks, const float* w, int64_t rows,
                          int64_t n, float* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
    (void)ws_bytes;
    return w ? long_bwd_t<true>(grad, blocks, w, rows, n, out, ws, stream)
             : long_bwd_t<false>(grad, blocks, w, rows, n, out, ws, stream);
}

}  // namespace isodev
