// Tile-level machinery shared by the whole-row kernels and the chunk kernel of
// long rows: staging a tile through shared memory, fixed-point cumulative sums,
// lane hulls, and the lane -> warp -> CTA merge rounds (the paper's Sections
// 3.1-3.2 and 3.5).
#pragma once

#include "iso_device.cuh"

namespace isodev {

// Shared-memory position of element k (0..31) of lane row gl in a staging buffer
// of 32-float rows.  16-byte units are XOR-swizzled by the row index so that
// both the coalesced fill (consecutive elements) and the lane reads (one
// float4 per lane, eight consecutive lanes per phase) are free of conflicts.
__device__ __forceinline__ int spos(int gl, int k) {
    return (gl << 5) | ((((k >> 2) ^ gl) & 7) << 2) | (k & 3);
}

// Layout of the dynamic shared memory of a CTA of NT threads holding R = NT/L
// tiles of L lanes.  The w staging is separate from the coordinate arrays (it
// is read while they are written); the block-start byte staging of the
// whole-row kernels reuses it (weighted) once the hull is built.
template <int NT, bool WEIGHTED>
struct TileSmem {
    static constexpr int kStageB = NT * 32 * 4;                 // y (or output) staging
    static constexpr int kStageWB = WEIGHTED ? NT * 32 * 4 : 0; // w staging
    static constexpr int kSxB = NT * kRow * 8;                  // lane-relative S
    static constexpr int kWxB = WEIGHTED ? NT * kRow * 8 : 0;   // lane-relative W
    static constexpr int kLSB = (NT + NT) * 8;                  // lane starts, L+1 per tile <= 2*NT
    static constexpr int kLWB = WEIGHTED ? kLSB : 0;
    static constexpr int kMaskB = NT * 4;
    static constexpr int kSummB = ((NT + 63) / 64) * 8;
    static constexpr int kBridgeB = (NT / 2 > 0 ? NT / 2 : 1) * 8;
    static constexpr int kInfoB = NT * 4 * 4;                   // 4 ints per tile (R <= NT)
    static constexpr int kBstB = WEIGHTED ? 0 : NT * 32;        // block-start byte staging
    static constexpr int kScanB = (NT / 16 + 2) * 8;            // cross-warp scan partials
    static constexpr int oStage = 0;
    static constexpr int oStageW = oStage + kStageB;
    static constexpr int oSx = oStageW + kStageWB;
    static constexpr int oWx = oSx + kSxB;
    static constexpr int oLS = oWx + kWxB;
    static constexpr int oLW = oLS + kLSB;
    static constexpr int oMask = oLW + kLWB;
    static constexpr int oSumm = oMask + kMaskB;
    static constexpr int oBridge = oSumm + kSummB;
    static constexpr int oInfo = oBridge + kBridgeB;
    static constexpr int oScan = oInfo + kInfoB;
    static constexpr int oBstOwn = oScan + kScanB;
    static constexpr int oBst = WEIGHTED ? oStageW : oBstOwn;
    static constexpr int kBytes = ((oBstOwn + kBstB + 127) / 128) * 128;
};

// Per-tile reduction slots in the info area.
enum { kInfoEmax = 0, kInfoPemax = 1, kInfoEwmax = 2, kInfoBad = 3 };

// Inclusive prefix sum of an int64 over the L lanes of each tile of a CTA of NT
// threads (L a power of two).  `tmp` holds NT/32 int64 entries.
template <int NT>
__device__ __forceinline__ int64_t tile_scan_incl(int64_t v, int lane, int L, int64_t* tmp) {
    const int wl = threadIdx.x & 31;
    const int seg = L < 32 ? L : 32;
    const int lseg = wl & (seg - 1);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int64_t o = __shfl_up_sync(kFull, v, d);
        if (d < seg && lseg >= d) v += o;
    }
    if (L > 32) {
        const int warp = threadIdx.x >> 5;
        if (wl == 31) tmp[warp] = v;
        __syncthreads();
        const int wpt = L >> 5;                 // warps per tile
        const int w0 = warp - (lane >> 5);      // first warp of this tile
        int64_t add = 0;
        for (int q = w0; q < warp; ++q) add += tmp[q];
        __syncthreads();
        v += add;
        (void)wpt;
    }
    return v;
}

}  // namespace isodev

namespace isodev {

// Result of the common hull phase, per thread (one lane of one tile).
struct TileHull {
    Tile T;          // view of the tile (coordinates, masks)
    int tile;        // tile index in the CTA
    int lane;        // lane in the tile
    int gl;          // lane index in the CTA's arrays (tile * L + lane)
    int e;           // elements of this lane (0..32)
    int qs, qw;      // quantum exponents of S and W (W: 0 for unit weights)
    uint32_t bad;    // ISO_ROW_BAD_* bits of the tile (0 = valid)
    bool live;       // the tile exists (row index in range)
};

// Common phase of every tile kernel: stage the tile's nt elements (y, and w
// when WEIGHTED) through shared memory, flag non-finite values, choose the
// fixed-point grid, form lane-relative cumulative sums and lane starts, build
// the lane hulls (Section 3.1) and merge them in rounds by walking (Section
// 3.2), up to the hull of the whole tile.  `yr`/`wr` point at the tile's first
// element; `neg` negates y on load (the decreasing fit, Section 2.1).
// All threads of the CTA must call it (it synchronises the CTA).
template <int NT, bool WEIGHTED>
__device__ __forceinline__ void tile_hull_phase(const float* __restrict__ yr,
                                                const float* __restrict__ wr, int nt, bool live,
                                                bool neg, int L, unsigned char* smem,
                                                TileHull& H) {
    using SM = TileSmem<NT, WEIGHTED>;
    float* stage = reinterpret_cast<float*>(smem + SM::oStage);
    int64_t* Sx = reinterpret_cast<int64_t*>(smem + SM::oSx);
    int64_t* Wx = reinterpret_cast<int64_t*>(smem + SM::oWx);
    float* stagew = reinterpret_cast<float*>(smem + SM::oStageW);
    int64_t* LSa = reinterpret_cast<int64_t*>(smem + SM::oLS);
    int64_t* LWa = reinterpret_cast<int64_t*>(smem + SM::oLW);
    uint32_t* maska = reinterpret_cast<uint32_t*>(smem + SM::oMask);
    uint32_t* summ = reinterpret_cast<uint32_t*>(smem + SM::oSumm);
    int2* bridge = reinterpret_cast<int2*>(smem + SM::oBridge);
    int* info = reinterpret_cast<int*>(smem + SM::oInfo);
    int64_t* scan = reinterpret_cast<int64_t*>(smem + SM::oScan);

    const int tid = threadIdx.x;
    const int tile = tid / L;
    const int lane = tid - tile * L;
    const int gl = tid;
    H.tile = tile; H.lane = lane; H.gl = gl; H.live = live;

    for (int i = lane; i < 4; i += L) info[tile * 4 + i] = 0;
    __syncthreads();

    // ---- load (coalesced) into the swizzled staging rows, with validation ----
    int emax = 0, pemax = 0, ewmax = 0;
    uint32_t bad = 0;
    if (live) {
        for (int e = lane; e < nt; e += L) {
            float v = __ldg(yr + e);
            if (neg) v = -v;
            const int pos = spos(tile * L + (e >> 5), e & 31);
            stage[pos] = v;
            int ey = (__float_as_uint(v) >> 23) & 0xff;
            if (ey == 0xff) bad |= 1u;
            else emax = max(emax, ey == 0 ? 1 : ey);
            if constexpr (WEIGHTED) {
                float wv = __ldg(wr + e);
                stagew[pos] = wv;
                int ew = (__float_as_uint(wv) >> 23) & 0xff;
                if (!(wv > 0.0f) || ew == 0xff) bad |= 2u;
                else {
                    int eww = ew == 0 ? 1 : ew;
                    ewmax = max(ewmax, eww);
                    if (ey != 0xff) pemax = max(pemax, eww + (ey == 0 ? 1 : ey));
                }
            }
        }
        if (emax) atomicMax(&info[tile * 4 + kInfoEmax], emax);
        if (WEIGHTED && pemax) atomicMax(&info[tile * 4 + kInfoPemax], pemax);
        if (WEIGHTED && ewmax) atomicMax(&info[tile * 4 + kInfoEwmax], ewmax);
        if (bad) atomicOr(&info[tile * 4 + kInfoBad], (int)bad);
    }
    __syncthreads();
    emax = max(info[tile * 4 + kInfoEmax], 1);
    pemax = max(info[tile * 4 + kInfoPemax], 2);
    ewmax = max(info[tile * 4 + kInfoEwmax], 1);
    H.bad = live ? (uint32_t)info[tile * 4 + kInfoBad] : 0u;
    H.qs = WEIGHTED ? qexp_prod(pemax) : qexp_unit(emax);
    H.qw = WEIGHTED ? qexp_unit(ewmax) : 0;
    const bool work = live && H.bad == 0;

    // ---- lane values, candidates and lane-relative cumulative sums, in one
    // pass over the lane's 32 staged values ----
    const int e = work ? min(max(nt - (lane << 5), 0), 32) : 0;
    H.e = e;
    int64_t* myS = Sx + gl * kRow;
    int64_t* myW = Wx + gl * kRow;
    int64_t s = 0, wsum = 0;
    uint32_t cand = 0;
    {
        const float4* st4 = reinterpret_cast<const float4*>(stage);
        const float4* sw4 = reinterpret_cast<const float4*>(stagew);
        int64_t up = 0, op = 1;   // previous element's value and weight
        myS[0] = 0;
        if constexpr (WEIGHTED) myW[0] = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int unit = (gl << 3) | ((q ^ gl) & 7);
            const float4 v = st4[unit];
            const float vv[4] = {v.x, v.y, v.z, v.w};
            float ww[4] = {1.f, 1.f, 1.f, 1.f};
            if constexpr (WEIGHTED) {
                const float4 wq = sw4[unit];
                ww[0] = wq.x; ww[1] = wq.y; ww[2] = wq.z; ww[3] = wq.w;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = 4 * q + j;
                const bool in = k < e;
                int64_t uk, ok;
                if constexpr (WEIGHTED) {
                    uk = in ? quant_prod(ww[j], vv[j], pemax) : 0;
                    ok = in ? max(quant(ww[j], ewmax), (int64_t)1) : 0;
                    // point k is locally convex: mean of element k-1 < mean of element k
                    if (k > 0 && in && (__int128)up * ok < (__int128)uk * op) cand |= 1u << k;
                } else {
                    uk = in ? quant(vv[j], emax) : 0;
                    ok = in ? 1 : 0;
                    if (k > 0 && in && up < uk) cand |= 1u << k;
                }
                up = uk;
                op = ok > 0 ? ok : 1;
                s += uk;
                myS[k + 1] = s;
                if constexpr (WEIGHTED) {
                    wsum += ok;
                    myW[k + 1] = wsum;
                }
            }
        }
    }
    // lane starts: exclusive scan of lane totals over the tile
    {
        int64_t inc = tile_scan_incl<NT>(s, lane, L, scan);
        LSa[tile * (L + 1) + lane] = inc - s;
        if (lane == L - 1) LSa[tile * (L + 1) + L] = inc;
        if constexpr (WEIGHTED) {
            int64_t incw = tile_scan_incl<NT>(wsum, lane, L, scan);
            LWa[tile * (L + 1) + lane] = incw - wsum;
            if (lane == L - 1) LWa[tile * (L + 1) + L] = incw;
        }
    }

    // ---- lane hulls in bit masks ----
    uint32_t mask = e > 0 ? lane_hull<WEIGHTED>(myS, myW, cand, e) : 0u;
    maska[gl] = mask;
    {
        uint32_t bal = __ballot_sync(kFull, mask != 0u);
        if ((tid & 31) == 0) summ[tid >> 5] = bal;
    }
    __syncthreads();

    Tile& T = H.T;
    T.Sx = Sx + tile * L * kRow;
    T.Wx = Wx + tile * L * kRow;
    T.LS = LSa + tile * (L + 1);
    T.LW = LWa + tile * (L + 1);
    T.mask = maska + tile * L;
    T.summ = summ;
    T.sbase = tile * L;
    T.L = L;
    T.nt = nt;

    // ---- merge rounds: pairs of 2^r lanes, up to the whole tile ----
    for (int r = 0; (1 << r) < L; ++r) {
        const int grp = lane >> (r + 1);
        const int A0 = grp << (r + 1);
        const int B0 = A0 + (1 << r);
        const int Bend = A0 + (2 << r);
        const bool active = work && ((B0 << 5) < nt);
        if (active && lane == A0) {
            int a, b;
            tile_bridge<WEIGHTED>(T, A0, B0, Bend, a, b);
            bridge[tid >> (r + 1)] = make_int2(a, b);
        }
        __syncthreads();
        if (active) {
            int2 ab = bridge[tid >> (r + 1)];
            if (ab.x != ab.y) {
                mask = clear_between(mask, lane, ab.x, ab.y);
                maska[gl] = mask;
            }
        }
        uint32_t bal = __ballot_sync(kFull, mask != 0u);
        if ((tid & 31) == 0) summ[tid >> 5] = bal;
        __syncthreads();
    }
}

// Slope of the edge between tile points a < b, rounded to float32 once from
// the exact integer differences (up to the rounding of the two conversions).
template <bool WEIGHTED>
__device__ __forceinline__ float tile_slope(const Tile& T, int a, int b, int qs, int qw) {
    int64_t dS = tile_S<WEIGHTED>(T, b) - tile_S<WEIGHTED>(T, a);
    int64_t dW = tile_W<WEIGHTED>(T, b) - tile_W<WEIGHTED>(T, a);
    float f = __ll2float_rn(dS) / __ll2float_rn(dW);
    return ldexpf(f, qs - qw);
}

}  // namespace isodev
