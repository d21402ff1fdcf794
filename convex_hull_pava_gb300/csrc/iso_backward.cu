// Backward of the fit (the paper's Section 6, "Gradient"): the fit is the
// weighted block mean, so its vector-Jacobian product is block averaging,
// d/dy_i = w_i * G / W with G, W the sums of grad and w over element i's block.
// Blocks are given by the block-start bytes of the forward pass.
//
// Sums are exact: grad and w are rounded to a fixed-point grid of 2^-50 of the
// tile's largest magnitude and summed as integers, so the result does not
// depend on the order of the additions.  The I/O type IO is float or double.  A row that is one tile is finished in
// one kernel; a longer row takes three steps (tile sums, a pass over the
// tiles' boundary sums, and the fill of blocks that cross tiles), as in the
// paper, without atomics.
#include "iso_internal.h"
#include "iso_tile.cuh"

namespace isodev {

namespace {

// Shared memory of a backward CTA of NT lanes: grad (and w) staging, which
// later holds each run's ratio and then the output, and the lanes' carries of
// the two segmented scans.
template <int NT, bool WEIGHTED, class IO = float>
struct BwdSmem {
    static constexpr int kRowB = 32 * (int)sizeof(IO);                // one lane's 32 values
    static constexpr int oStage = 0;                                  // grad, ratios, output
    static constexpr int oStageW = oStage + NT * kRowB;               // w
    static constexpr int oCarry = oStageW + (WEIGHTED ? NT * kRowB : 0);   // [4][NT] int64
    static constexpr int oWarp = oCarry + 4 * NT * 8;                 // [4][NT/32] int64 + flags
    static constexpr int oWarpF = oWarp + 4 * (NT / 32) * 8;          // [2][NT/32] int
    static constexpr int oInfo = oWarpF + 2 * (NT / 32) * 4;          // per tile: 8 int64
    static constexpr int kBytes = ((oInfo + NT * 8 * 8 + 127) / 128) * 128;
};

// Result of a backward tile.  hG/hW: sums (fixed point) of the elements before
// the tile's first block start (the whole tile if it has none); tG/tW: sums
// from its last block start to its end.
struct BwdTile {
    int first_start;   // first block start in the tile, or -1
    int last_start;    // last block start in the tile, or -1
    int qg, qw;        // quantum exponents of grad and w
    bool nan;          // a non-finite grad or an invalid weight in the tile
    int64_t hG, hW, tG, tW;
};

// Per-tile info: ints 0..4 (exponent maxima, status, first and last start),
// then 64-bit slots for the tile's head and tail sums.
enum { kBInfoG = 0, kBInfoW = 1, kBInfoBad = 2, kBInfoFs = 3, kBInfoLs = 4 };
enum { kSlotTW = 4, kSlotHG = 5, kSlotHW = 6, kSlotTG = 7 };

// Optional weight gradient: d/dw_i = (y_i - z_i) G / W (the paper's Section 6,
// "Gradient"), from the fit z of the forward pass.
template <class IO>
struct WGrad {
    const IO* y;      // the forward pass's input, [rows, n]
    const IO* fit;    // its output z, [rows, n]
    IO* dw;           // nullptr: not wanted
};

// Component j of a 16-byte vector of the I/O type.
__device__ __forceinline__ float vcomp(const float4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
__device__ __forceinline__ double vcomp(const double2& v, int j) { return j == 0 ? v.x : v.y; }

// One tile of L lanes (32 elements each): every element gets w_i G / W of its
// block, where the block's sums come from the lane's own run sums and, for
// runs that cross lanes, from a forward segmented scan (the part before the
// lane) and a backward one (the part after it) over the lanes' sums.  Each
// run's ratio is written at the run's last element and spread back over the
// run by a reverse pass.  Runs that cross the tile's edges get only the
// tile's part; the long-row path completes them.  All threads of the CTA call
// it.  On return, stage holds the output of the tile's elements and, for
// weighted tiles, the w staging holds each element's ratio G / W.
template <int NT, bool WEIGHTED, class IO>
__device__ __forceinline__ void bwd_tile_phase(const IO* __restrict__ gr,
                                               const uint8_t* __restrict__ br,
                                               const IO* __restrict__ wr, int nt, bool live,
                                               bool first_is_start, int L, unsigned char* smem,
                                               BwdTile& B) {
    using SM = BwdSmem<NT, WEIGHTED, IO>;
    IO* stage = reinterpret_cast<IO*>(smem + SM::oStage);
    IO* stagew = reinterpret_cast<IO*>(smem + SM::oStageW);
    int64_t* carry = reinterpret_cast<int64_t*>(smem + SM::oCarry);
    int64_t* wsum = reinterpret_cast<int64_t*>(smem + SM::oWarp);
    int* wflag = reinterpret_cast<int*>(smem + SM::oWarpF);
    int64_t* info64 = reinterpret_cast<int64_t*>(smem + SM::oInfo);

    const int tid = threadIdx.x;
    const int tile = tid / L;
    const int lane = tid - tile * L;
    const int gl = tid;
    const int wl = tid & 31, warp = tid >> 5;
    const int seg = L < 32 ? L : 32;
    const int lseg = wl & (seg - 1);
    int* info = reinterpret_cast<int*>(info64 + tile * 8);

    if (lane == 0) {
        info[kBInfoG] = 0; info[kBInfoW] = 0; info[kBInfoBad] = 0;
        info[kBInfoFs] = 0x7fffffff; info[kBInfoLs] = -1;
        info64[tile * 8 + kSlotHG] = 0; info64[tile * 8 + kSlotHW] = 0;
        info64[tile * 8 + kSlotTG] = 0; info64[tile * 8 + kSlotTW] = 0;
    }
    __syncthreads();
    int gmax = 0, ewmax = 0;
    uint32_t bad = 0;
    uint32_t starts = 0;
    const int e = live ? min(max(nt - (lane << 5), 0), 32) : 0;
    if (live) {
        stage_tile<false, IO>(gr, nt, lane, L, tile * L, false, stage, gmax, bad);
        if constexpr (WEIGHTED)
            stage_tile<true, IO>(wr, nt, lane, L, tile * L, false, stagew, ewmax, bad);
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
    gmax = tile_warp_max(gmax, L);
    if (WEIGHTED) ewmax = tile_warp_max(ewmax, L);
    const int bad_or = tile_warp_or((int)bad, L);
    if (live && lseg == 0) {
        atomicMax(&info[kBInfoG], gmax);
        if (WEIGHTED) atomicMax(&info[kBInfoW], ewmax);
        if (bad_or) atomicOr(&info[kBInfoBad], 1);
    }
    if (starts) {
        atomicMin(&info[kBInfoFs], (lane << 5) + __ffs(starts) - 1);
        atomicMax(&info[kBInfoLs], (lane << 5) + 31 - __clz(starts));
    }
    __syncthreads();
    gmax = max(info[kBInfoG], 1);
    ewmax = max(info[kBInfoW], 1);
    B.nan = info[kBInfoBad] != 0;
    B.qg = qexp_unit_t<IO>(gmax);
    B.qw = WEIGHTED ? qexp_unit_t<IO>(ewmax) : 0;
    B.first_start = info[kBInfoFs] == 0x7fffffff ? -1 : info[kBInfoFs];
    B.last_start = info[kBInfoLs];
    const QuantT<IO> qg(gmax), qwt(ewmax);

    using V = typename IoT<IO>::V;
    constexpr int P = IoT<IO>::kPerV;
    const V* stv = reinterpret_cast<const V*>(stage);
    const V* swv = reinterpret_cast<const V*>(stagew);
    auto lane_values = [&](int q, IO (&vv)[P], IO (&ww)[P]) {
        const int unit = sunit_t<IO>(gl, q);
        const V v = stv[unit];
#pragma unroll
        for (int j = 0; j < P; ++j) { vv[j] = vcomp(v, j); ww[j] = IO(1); }
        if constexpr (WEIGHTED) {
            const V t = swv[unit];
#pragma unroll
            for (int j = 0; j < P; ++j) ww[j] = vcomp(t, j);
        }
    };
    const IO qnan = qnan_t<IO>();
    auto ratio = [&](int64_t G, int64_t Wt) -> IO {
        return B.nan ? qnan : ratio_t<IO>(G, Wt, B.qg - B.qw);
    };
    // pass 1: the lane's head (before its first start) and tail (from its
    // last start) sums, a lane without a start having head = tail = its total;
    // the ratio of every run between two starts of the lane is written over the
    // run's last element
    int64_t hg = 0, hw = 0, tg = 0, tw = 0;
    {
        bool seen = false;
#pragma unroll
        for (int q = 0; q < 32 / P; ++q) {
            IO vv[P], ww[P];
            lane_values(q, vv, ww);
#pragma unroll
            for (int j = 0; j < P; ++j) {
                const int k = P * q + j;
                if ((starts >> k) & 1u) {
                    if (seen) stage[spos_t<IO>(gl, k - 1)] = ratio(tg, tw);
                    else { hg = tg; hw = tw; seen = true; }
                    tg = 0; tw = 0;
                }
                if (k < e) {
                    tg += qg(vv[j]);
                    tw += WEIGHTED ? qwt(ww[j]) : 1;
                }
            }
        }
        if (!seen) { hg = tg; hw = tw; }
    }
    const int fl0 = starts ? 1 : 0;
    int64_t* inG = carry;            // forward inclusive
    int64_t* inW = carry + NT;
    int64_t* bkG = carry + 2 * NT;   // backward inclusive
    int64_t* bkW = carry + 3 * NT;
    {
        // forward: I_l = f_l ? tail_l : I_{l-1} + total_l
        int64_t vg = tg, vw = tw;
        int fl = fl0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t og = __shfl_up_sync(kFull, vg, d);
            const int64_t ow = __shfl_up_sync(kFull, vw, d);
            const int of = __shfl_up_sync(kFull, fl, d);
            if (d < seg && lseg >= d) {
                if (!fl) { vg += og; vw += ow; }
                fl |= of;
            }
        }
        // backward: J_l = f_l ? head_l : total_l + J_{l+1}
        int64_t ug = hg, uw = hw;
        int fr = fl0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t og = __shfl_down_sync(kFull, ug, d);
            const int64_t ow = __shfl_down_sync(kFull, uw, d);
            const int of = __shfl_down_sync(kFull, fr, d);
            if (d < seg && lseg + d < seg) {
                if (!fr) { ug += og; uw += ow; }
                fr |= of;
            }
        }
        if (L > 32) {
            const int nw = NT / 32;
            if (wl == 31) { wsum[warp] = vg; wsum[nw + warp] = vw; wflag[warp] = fl; }
            if (wl == 0) { wsum[2 * nw + warp] = ug; wsum[3 * nw + warp] = uw; wflag[nw + warp] = fr; }
            __syncthreads();
            const int w0 = warp - (lane >> 5);            // first warp of this tile
            const int w1 = w0 + (L >> 5);                 // one past its last
            if (!fl) {
                int64_t ag = 0, aw = 0;
                for (int q = warp - 1; q >= w0; --q) {
                    ag += wsum[q]; aw += wsum[nw + q];
                    if (wflag[q]) break;
                }
                vg += ag; vw += aw;
            }
            if (!fr) {
                int64_t ag = 0, aw = 0;
                for (int q = warp + 1; q < w1; ++q) {
                    ag += wsum[2 * nw + q]; aw += wsum[3 * nw + q];
                    if (wflag[nw + q]) break;
                }
                ug += ag; uw += aw;
            }
        }
        inG[gl] = vg; inW[gl] = vw;
        bkG[gl] = ug; bkW[gl] = uw;
    }
    __syncthreads();
    // the part of the lane's first run before the lane, and of its last run after it
    const int64_t cing = lane ? inG[gl - 1] : 0, cinw = lane ? inW[gl - 1] : 0;
    const int64_t coutg = lane + 1 < L ? bkG[gl + 1] : 0, coutw = lane + 1 < L ? bkW[gl + 1] : 0;
    // the tile's head and tail sums, from the lanes that hold its first and last start
    if (B.first_start >= 0 && lane == (B.first_start >> 5)) {
        info64[tile * 8 + kSlotHG] = cing + hg;
        info64[tile * 8 + kSlotHW] = cinw + hw;
    }
    if (B.first_start < 0 && lane == L - 1) {
        info64[tile * 8 + kSlotHG] = inG[gl];
        info64[tile * 8 + kSlotHW] = inW[gl];
    }
    if (B.last_start >= 0 && lane == (B.last_start >> 5)) {
        info64[tile * 8 + kSlotTG] = tg + coutg;
        info64[tile * 8 + kSlotTW] = tw + coutw;
    }
    // the lane's first and last runs, which may reach into other lanes
    if (e > 0) {
        if (starts) {
            const int f = __ffs(starts) - 1;
            if (f > 0) stage[spos_t<IO>(gl, f - 1)] = ratio(cing + hg, cinw + hw);
            stage[spos_t<IO>(gl, e - 1)] = ratio(tg + coutg, tw + coutw);
        } else {
            stage[spos_t<IO>(gl, e - 1)] = ratio(cing + tg + coutg, cinw + tw + coutw);
        }
    }
    // pass 2, backwards: each element takes the ratio of its run (times w)
    {
        IO r = IO(0);
#pragma unroll
        for (int k = 31; k >= 0; --k) {
            if (k < e) {
                const bool last = k == e - 1 || ((starts >> (k + 1)) & 1u);
                const int p = spos_t<IO>(gl, k);
                if (last) r = stage[p];
                if constexpr (WEIGHTED) {
                    stage[p] = stagew[p] * r;
                    stagew[p] = r;          // the ratio G / W, for the weight gradient
                } else {
                    stage[p] = r;
                }
            }
        }
    }
    __syncthreads();
    B.hG = info64[tile * 8 + kSlotHG];
    B.hW = info64[tile * 8 + kSlotHW];
    B.tG = info64[tile * 8 + kSlotTG];
    B.tW = info64[tile * 8 + kSlotTW];
}

// The 256-thread instance (rows of 4,097 to 8,192 elements) is held to the
// registers of three CTAs per SM, which its shared memory allows (measured
// 12% faster than two CTAs at its natural register count).
template <int NT, bool WEIGHTED, class IO>
__global__ void __launch_bounds__(NT, NT == 256 ? 3 : 1)
rows_backward_kernel(const IO* __restrict__ grad, const uint8_t* __restrict__ blocks,
                     const IO* __restrict__ w, int64_t rows, int n, int L,
                     IO* __restrict__ out, WGrad<IO> wg) {
    extern __shared__ __align__(128) unsigned char smem[];
    using SM = BwdSmem<NT, WEIGHTED, IO>;
    const int R = NT / L;
    const int tile = threadIdx.x / L;
    const int lane = threadIdx.x - tile * L;
    const int64_t row = (int64_t)blockIdx.x * R + tile;
    const bool live = row < rows;
    const int64_t off = (live ? row : 0) * (int64_t)n;
    BwdTile B;
    bwd_tile_phase<NT, WEIGHTED, IO>(grad + off, blocks + off, WEIGHTED ? w + off : nullptr, n,
                                     live, true, L, smem, B);
    const IO* stage = reinterpret_cast<const IO*>(smem + SM::oStage);
    const IO* ratio = reinterpret_cast<const IO*>(smem + (WEIGHTED ? SM::oStageW : SM::oStage));
    if (live) {
        if (out) write_row<IO>(out + off, stage, tile * L, n, lane, L, true);   // 16-byte stores
        if (wg.dw) {
            const IO* yrow = wg.y + off;
            const IO* zrow = wg.fit + off;
            IO* drow = wg.dw + off;
            for (int i = lane; i < n; i += L)
                drow[i] = (__ldg(yrow + i) - __ldg(zrow + i)) *
                          ratio[spos_t<IO>(tile * L + (i >> 5), i & 31)];
        }
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

template <bool WEIGHTED, class IO>
__global__ void __launch_bounds__(kBNT, 3)
long_bwd_tiles_kernel(const IO* __restrict__ grad, const uint8_t* __restrict__ blocks,
                      const IO* __restrict__ w, int64_t n, int64_t m, IO* __restrict__ out,
                      WGrad<IO> wg, BwdRec* __restrict__ rec) {
    extern __shared__ __align__(128) unsigned char smem[];
    using SM = BwdSmem<kBNT, WEIGHTED, IO>;
    const int64_t c = blockIdx.x;
    const int64_t row = c / m;
    const int64_t j = c - row * m;
    const int64_t e0 = j * kBT;
    const int nt = (int)imin64(kBT, n - e0);
    const int64_t off = row * n + e0;
    BwdTile B;
    bwd_tile_phase<kBNT, WEIGHTED, IO>(grad + off, blocks + off, WEIGHTED ? w + off : nullptr, nt,
                                       true, j == 0, kBNT, smem, B);
    const IO* stage = reinterpret_cast<const IO*>(smem + SM::oStage);
    // elements of complete blocks: from the first start to one before the last start
    const int lo = B.first_start < 0 ? nt : B.first_start;
    const int hi = B.last_start < 0 ? nt : B.last_start;
    if (out) {
        IO* o = out + off;
        for (int i = lo + threadIdx.x; i < hi; i += kBNT) o[i] = stage[spos_t<IO>(i >> 5, i & 31)];
    }
    if (wg.dw) {
        const IO* ratio = reinterpret_cast<const IO*>(smem + (WEIGHTED ? SM::oStageW : SM::oStage));
        for (int i = lo + threadIdx.x; i < hi; i += kBNT)
            wg.dw[off + i] = (__ldg(wg.y + off + i) - __ldg(wg.fit + off + i)) *
                             ratio[spos_t<IO>(i >> 5, i & 31)];
    }
    if (threadIdx.x == 0) {
        BwdRec r;
        r.fs = B.first_start;
        r.ls = B.last_start;
        r.nan = B.nan ? 1 : 0;
        r.pad = 0;
        const double sg = ldexp(1.0, B.qg), sw = ldexp(1.0, B.qw);
        r.hG = (double)B.hG * sg;
        r.hW = (double)B.hW * sw;
        if (B.last_start >= 0) {
            r.tG = (double)B.tG * sg;
            r.tW = (double)B.tW * sw;
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

template <bool WEIGHTED, class IO>
__global__ void __launch_bounds__(kBNT)
long_bwd_fill_kernel(const IO* __restrict__ w, int64_t n, int64_t m,
                     const BwdRec* __restrict__ rec, const BwdTot* __restrict__ tot,
                     IO* __restrict__ out, WGrad<IO> wg) {
    const int64_t c = blockIdx.x;
    const int64_t row = c / m;
    const int64_t j = c - row * m;
    const int64_t e0 = j * kBT;
    const int nt = (int)imin64(kBT, n - e0);
    const BwdRec r = rec[c];
    const BwdTot t = tot[c];
    const int64_t off = row * n + e0;
    IO* o = out ? out + off : nullptr;
    const IO* wr = WEIGHTED ? w + off : nullptr;
    const IO qnan = qnan_t<IO>();
    const IO rh = t.nan ? qnan : (IO)(t.headG / t.headW);
    const IO rt = t.nan ? qnan : (IO)(t.tailG / t.tailW);
    const int hend = r.fs < 0 ? nt : r.fs;
    const int tbeg = r.ls >= 0 ? r.ls : nt;
    // the head (elements before the tile's first start) and the tail (from its
    // last start) belong to blocks that cross tiles; a bad row is NaN throughout
    auto put = [&](int i, IO rt) {
        if (o) o[i] = WEIGHTED ? __ldg(wr + i) * rt : rt;
        if (wg.dw) wg.dw[off + i] = (__ldg(wg.y + off + i) - __ldg(wg.fit + off + i)) * rt;
    };
    for (int i = threadIdx.x; i < hend; i += kBNT) put(i, rh);
    for (int i = tbeg + threadIdx.x; i < nt; i += kBNT) put(i, rt);
    if (t.nan)
        for (int i = hend + threadIdx.x; i < tbeg; i += kBNT) {
            if (o) o[i] = qnan;
            if (wg.dw) wg.dw[off + i] = qnan;
        }
}

__host__ __device__ inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

template <int NT, bool WEIGHTED, class IO>
cudaError_t launch_rows_bwd(const IO* grad, const uint8_t* blocks, const IO* w, int64_t rows,
                            int n, int L, IO* out, WGrad<IO> wg, cudaStream_t stream) {
    using SM = BwdSmem<NT, WEIGHTED, IO>;
    auto kern = rows_backward_kernel<NT, WEIGHTED, IO>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           SM::kBytes);
    if (err != cudaSuccess) return err;
    const int R = NT / L;
    const int64_t grid = (rows + R - 1) / R;
    kern<<<(unsigned)grid, NT, SM::kBytes, stream>>>(grad, blocks, w, rows, n, L, out, wg);
    prof_mark(stream, "rows_backward");
    return cudaGetLastError();
}

template <bool WEIGHTED, class IO>
cudaError_t long_bwd_t(const IO* grad, const uint8_t* blocks, const IO* w, int64_t rows,
                       int64_t n, IO* out, WGrad<IO> wg, void* ws, cudaStream_t stream) {
    using SM = BwdSmem<kBNT, WEIGHTED, IO>;
    const int64_t m = (n + kBT - 1) / kBT;
    const int64_t M = rows * m;
    BwdRec* rec = static_cast<BwdRec*>(ws);
    BwdTot* tot = reinterpret_cast<BwdTot*>(static_cast<char*>(ws) + a256(sizeof(BwdRec) * M));
    auto k1 = long_bwd_tiles_kernel<WEIGHTED, IO>;
    cudaError_t err = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           SM::kBytes);
    if (err != cudaSuccess) return err;
    k1<<<(unsigned)M, kBNT, SM::kBytes, stream>>>(grad, blocks, w, n, m, out, wg, rec);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "bwd_tiles");
    long_bwd_totals_kernel<<<(unsigned)((rows + 63) / 64), 64, 0, stream>>>(rows, m, rec, tot);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "bwd_totals");
    long_bwd_fill_kernel<WEIGHTED, IO><<<(unsigned)M, kBNT, 0, stream>>>(w, n, m, rec, tot, out, wg);
    prof_mark(stream, "bwd_fill");
    return cudaGetLastError();
}

}  // namespace

template <class IO>
cudaError_t rows_backward(const IO* grad, const uint8_t* blocks, const IO* w, int64_t rows, int n,
                          IO* out, const IO* y, const IO* fit, IO* dw, cudaStream_t stream) {
    int L = 1;
    while (32 * L < n) L <<= 1;
    const WGrad<IO> wg{y, fit, dw};
    const bool weighted = w != nullptr;
#define ISO_BWD_LAUNCH(NT_)                                                                     \
    return weighted                                                                             \
               ? launch_rows_bwd<NT_, true, IO>(grad, blocks, w, rows, n, L, out, wg, stream)  \
               : launch_rows_bwd<NT_, false, IO>(grad, blocks, w, rows, n, L, out, wg, stream)
    if (L <= 32) { ISO_BWD_LAUNCH(128); }
    if (L <= 64) { ISO_BWD_LAUNCH(64); }
    if (L <= 128) { ISO_BWD_LAUNCH(128); }
    ISO_BWD_LAUNCH(256);
#undef ISO_BWD_LAUNCH
}

size_t long_backward_workspace(int64_t rows, int64_t n, bool weighted) {
    (void)weighted;
    const int64_t M = rows * ((n + kBT - 1) / kBT);
    return a256(sizeof(BwdRec) * M) + a256(sizeof(BwdTot) * M);
}

template <class IO>
cudaError_t long_backward(const IO* grad, const uint8_t* blocks, const IO* w, int64_t rows,
                          int64_t n, IO* out, const IO* y, const IO* fit, IO* dw, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
    (void)ws_bytes;
    const WGrad<IO> wg{y, fit, dw};
    return w ? long_bwd_t<true, IO>(grad, blocks, w, rows, n, out, wg, ws, stream)
             : long_bwd_t<false, IO>(grad, blocks, w, rows, n, out, wg, ws, stream);
}

#define ISO_BWD_INSTANTIATE(IO)                                                                  \
    template cudaError_t rows_backward<IO>(const IO*, const uint8_t*, const IO*, int64_t, int,   \
                                           IO*, const IO*, const IO*, IO*, cudaStream_t);        \
    template cudaError_t long_backward<IO>(const IO*, const uint8_t*, const IO*, int64_t,        \
                                           int64_t, IO*, const IO*, const IO*, IO*, void*,       \
                                           size_t, cudaStream_t);
ISO_BWD_INSTANTIATE(float)
ISO_BWD_INSTANTIATE(double)
#undef ISO_BWD_INSTANTIATE

}  // namespace isodev
