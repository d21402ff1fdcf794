// Tile-level machinery shared by the whole-row kernels and the chunk kernel of
// long rows: staging a tile through shared memory, fixed-point cumulative sums,
// lane hulls, and the lane -> warp -> CTA merge rounds (the paper's Sections
// 3.1-3.2 and 3.5).
#pragma once

#include "iso_device.cuh"
#include "iso_qhull.cuh"
#include "iso_filter.cuh"

#include <type_traits>

namespace isodev {

// Shared-memory position of element k (0..31) of lane row gl in a staging buffer
// of 32-float rows.  16-byte units are XOR-swizzled by the row index so that
// both the coalesced fill (consecutive elements) and the lane reads (one
// float4 per lane, eight consecutive lanes per phase) are free of conflicts.
__device__ __forceinline__ int spos(int gl, int k) {
    return (gl << 5) | ((((k >> 2) ^ gl) & 7) << 2) | (k & 3);
}
__device__ __forceinline__ int sunit(int gl, int q) { return (gl << 3) | ((q ^ gl) & 7); }

// The same for rows of 32 elements of the I/O type IO: 16-byte units of
// IoT<IO>::kPerV elements (8 units of float4, or 16 of double2 per row),
// XOR-swizzled by the row index (eight consecutive rows per phase).
template <class IO> __device__ __forceinline__ int spos_t(int gl, int k);
template <> __device__ __forceinline__ int spos_t<float>(int gl, int k) { return spos(gl, k); }
template <> __device__ __forceinline__ int spos_t<double>(int gl, int k) {
    return (gl << 5) | ((((k >> 1) ^ gl) & 15) << 1) | (k & 1);
}
template <class IO> __device__ __forceinline__ int sunit_t(int gl, int q);
template <> __device__ __forceinline__ int sunit_t<float>(int gl, int q) { return sunit(gl, q); }
template <> __device__ __forceinline__ int sunit_t<double>(int gl, int q) {
    return (gl << 4) | ((q ^ gl) & 15);
}

// Layout of the dynamic shared memory of a CTA of NT threads holding R = NT/L
// tiles of L lanes.  The input staging lives inside the lane-relative sums
// array Sx (2 x 128 B per lane fit in its 264 B per lane): it is read into
// registers before Sx is written.  Kernels that write the fit (EMIT) merge the
// lane hulls by walking over vertex masks and later write each vertex's edge
// slope over the lane's row of Sx.  The others (chunks of long rows) compact
// each lane hull into the front of its row, with the points' indices in Px,
// and merge the compact lists.
template <int NT, bool WEIGHTED, bool EMIT, int RMAX = NT, class IO = float>
struct TileSmem {
    // 33 entries per lane row (an odd stride: the lanes' rows start in
    // different banks), points 0..32 of the lane.  Compact lists use the first
    // 32 entries of each row, flat entry i living at i + i/32, so that the
    // lists of neighbouring lanes are contiguous in flat order.
    static constexpr int kSxB = NT * kRow * 8;                  // lane-relative S (+ staging)
    static constexpr int kWxB = WEIGHTED ? NT * kRow * 8 : 0;   // lane-relative W
    static constexpr int kPxB = EMIT ? 0 : ((NT * kRow * 2 + 15) / 16) * 16;   // point indices
    static constexpr int kCntB = EMIT ? 0 : NT * 4;             // entries of each compact list
    static constexpr int kLSB = (NT + RMAX) * 8;                // lane starts, L+1 per tile
    static constexpr int kLWB = WEIGHTED ? kLSB : 0;
    static constexpr int kMaskB = NT * 4;
    static constexpr int kSummB = ((NT + 63) / 64) * 8;
    static constexpr int kBridgeB = (NT / 2 > 0 ? NT / 2 : 1) * 8;
    static constexpr int kInfoB = RMAX * 4 * 4;                 // 4 ints per tile
    static constexpr int kScanB = (NT / 16 + 2) * 8;            // cross-warp scan partials
    static constexpr int oSx = 0;
    static constexpr int oWx = oSx + kSxB;
    static constexpr int oPx = oWx + kWxB;
    static constexpr int oCnt = oPx + kPxB;
    static constexpr int oLS = oCnt + kCntB;
    static constexpr int oLW = oLS + kLSB;
    static constexpr int oMask = oLW + kLWB;
    static constexpr int oSumm = oMask + kMaskB;
    static constexpr int oBridge = oSumm + kSummB;
    static constexpr int oInfo = oBridge + kBridgeB;
    static constexpr int oScan = oInfo + kInfoB;
    static constexpr int kBytes = ((oScan + kScanB + 127) / 128) * 128;
    // staging: y at the start of Sx; w after it for float32 (2 x 128 B per lane
    // <= 264 B), in Wx for float64 (256 B per lane each)
    static constexpr int oStageY = oSx;
    static constexpr int oStageW = sizeof(IO) == 4 ? oSx + NT * 128 : oWx;
};

// Per-tile reduction slots in the info area.
enum { kInfoEmax = 0, kInfoPemax = 1, kInfoEwmax = 2, kInfoBad = 3 };

// Inclusive prefix sum of an int64 over the L lanes of each tile of a CTA of NT
// threads (L a power of two).  `tmp` holds NT/32 int64 entries.  Every thread of
// the CTA must call it.
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
        const int w0 = warp - (lane >> 5);      // first warp of this tile
        int64_t add = 0;
        for (int q = w0; q < warp; ++q) add += tmp[q];
        __syncthreads();
        v += add;
    }
    return v;
}

// Maximum / bitwise or of v over the lanes of a tile that share this warp
// (L < 32: the tile's L lanes; else the whole warp).
__device__ __forceinline__ int tile_warp_max(int v, int L) {
    const int seg = L < 32 ? L : 32;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
        if (d < seg) v = max(v, __shfl_xor_sync(kFull, v, d));
    return v;
}
__device__ __forceinline__ int tile_warp_or(int v, int L) {
    const int seg = L < 32 ? L : 32;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
        if (d < seg) v |= __shfl_xor_sync(kFull, v, d);
    return v;
}

// Coalesced load of a tile's nt floats from `src` into the swizzled staging
// rows of lanes [gl0, gl0 + L), by the tile's L threads.  All loads of a
// thread are issued before any store.  Tracks the largest biased exponent and
// flags non-finite values (and, for weights, values that are not > 0): the
// bit patterns of non-negative floats order like their values, so the largest
// |bits| gives both the exponent and whether an Inf or NaN occurred, and for
// weights the smallest signed bits is > 0 exactly when every weight is.
template <bool IS_W, class IO>
__device__ __forceinline__ void stage_tile(const IO* __restrict__ src, int nt, int lane, int L,
                                           int gl0, bool neg, IO* stage, int& emax,
                                           uint32_t& bad) {
    using UB = typename std::conditional<sizeof(IO) == 4, int32_t, long long>::type;
    constexpr UB kMag = sizeof(IO) == 4 ? (UB)0x7fffffff : (UB)0x7fffffffffffffffll;
    constexpr UB kInf = sizeof(IO) == 4 ? (UB)0x7f800000 : (UB)0x7ff0000000000000ll;
    UB bhi = 0, blo = kMag;
    auto note = [&](IO v) {
        UB b;
        if constexpr (sizeof(IO) == 4) b = __float_as_int(v); else b = __double_as_longlong(v);
        if (IS_W) { bhi = max(bhi, b); blo = min(blo, b); }
        else bhi = max(bhi, b & kMag);
    };
    auto finish = [&]() {
        const int e = sizeof(IO) == 4 ? (int)((bhi >> 23) & 0xff) : (int)((bhi >> 52) & 0x7ff);
        if (IS_W ? (blo <= 0 || bhi >= kInf) : bhi >= kInf) bad |= IS_W ? 2u : 1u;
        else emax = max(emax, e == 0 ? 1 : e);
    };
    const bool aligned = ((reinterpret_cast<uintptr_t>(src) & 15u) == 0);
    if (aligned) {
        if constexpr (sizeof(IO) == 4) {
            const int n4 = nt >> 2;
            const float4* s4 = reinterpret_cast<const float4*>(src);
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = lane + j * L;
                v[j] = i < n4 ? __ldg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float4* st4 = reinterpret_cast<float4*>(stage);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = lane + j * L;
                if (i < n4) {
                    float4 x = v[j];
                    if (neg) { x.x = -x.x; x.y = -x.y; x.z = -x.z; x.w = -x.w; }
                    note(x.x); note(x.y); note(x.z); note(x.w);
                    const int e = i << 2;
                    st4[sunit(gl0 + (e >> 5), (e & 31) >> 2)] = x;
                }
            }
            for (int e = (n4 << 2) + lane; e < nt; e += L) {
                float x = __ldg(src + e);
                if (neg) x = -x;
                note(x);
                stage[spos(gl0 + (e >> 5), e & 31)] = x;
            }
        } else {
            const int n2 = nt >> 1;
            const double2* s2 = reinterpret_cast<const double2*>(src);
            double2 v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = lane + j * L;
                v[j] = i < n2 ? __ldg(s2 + i) : make_double2(0.0, 0.0);
            }
            double2* st2 = reinterpret_cast<double2*>(stage);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = lane + j * L;
                if (i < n2) {
                    double2 x = v[j];
                    if (neg) { x.x = -x.x; x.y = -x.y; }
                    note(x.x); note(x.y);
                    const int e = i << 1;
                    st2[sunit_t<double>(gl0 + (e >> 5), (e & 31) >> 1)] = x;
                }
            }
            for (int e = (n2 << 1) + lane; e < nt; e += L) {
                double x = __ldg(src + e);
                if (neg) x = -x;
                note(x);
                stage[spos_t<double>(gl0 + (e >> 5), e & 31)] = x;
            }
        }
    } else {
        IO v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int e = lane + j * L;
            v[j] = e < nt ? __ldg(src + e) : IO(0);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int e = lane + j * L;
            if (e < nt) {
                const IO x = neg ? -v[j] : v[j];
                note(x);
                stage[spos_t<IO>(gl0 + (e >> 5), e & 31)] = x;
            }
        }
    }
    finish();
}

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
    bool quick;      // the hull came from tile_quickhull (vertex masks only)
    int list;        // chunks: entries of the list whose hull was found (0: none)
    bool all;        // chunks: every point is a hull vertex (the element means increase)
    bool oneblock;   // whole rows of one tile per CTA: the row is one block
};

// Whole rows of kQuickMinLanes to 32 lanes (one warp) whose first half has a
// larger mean than their second half (a trend against the fit's direction, so
// few blocks) take the levels of farthest-point splits (iso_qhull.cuh) instead
// of the lane hulls and merging rounds: a row of one block is finished by one
// level, where the merging rounds walk long bridges.  Rows with the trend
// along the fit keep the merging rounds, which measured faster there (each
// level's lanes evaluate their points one by one, and the warp waits for its
// busiest lane); so do longer rows (merging the warps' hulls by CTA-wide
// levels measured slower) and the chunks of long rows.  A CTA in which more
// than one lane in kQuickDense has over 24 of its 31 inner points locally
// convex (a dense hull) also keeps them.
constexpr int kQuickMinLanes = 4;
constexpr int kQuickDense = 8;

// Common phase of every tile kernel: stage the tile's nt elements (y, and w
// when WEIGHTED) through shared memory, flag non-finite values, choose the
// fixed-point grid, form lane-relative cumulative sums and lane starts, build
// the lane hulls (Section 3.1) and merge them in rounds by walking (Section
// 3.2), up to the hull of the whole tile.  `yr`/`wr` point at the tile's first
// element; `neg` negates y on load (the decreasing fit, Section 2.1).
// All threads of the CTA must call it (it synchronises the CTA).
template <int NT, bool WEIGHTED, bool EMIT, int RMAX = NT, class IO = float>
__device__ __forceinline__ void tile_hull_phase(const IO* __restrict__ yr,
                                                const IO* __restrict__ wr, int nt, bool live,
                                                bool neg, int L, unsigned char* smem,
                                                TileHull& H) {
    using SM = TileSmem<NT, WEIGHTED, EMIT, RMAX, IO>;
    int64_t* Sx = reinterpret_cast<int64_t*>(smem + SM::oSx);
    int64_t* Wx = reinterpret_cast<int64_t*>(smem + SM::oWx);
    IO* stagey = reinterpret_cast<IO*>(smem + SM::oStageY);
    IO* stagew = reinterpret_cast<IO*>(smem + SM::oStageW);
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
    const int seg = L < 32 ? L : 32;
    const bool seg_first = ((tid & 31) & (seg - 1)) == 0;
    H.tile = tile; H.lane = lane; H.gl = gl; H.live = live;

    for (int i = lane; i < 4; i += L) info[tile * 4 + i] = 0;
    __syncthreads();

    // ---- load (coalesced, vectorised) into the swizzled staging rows ----
    int emax = 0, ewmax = 0;
    uint32_t bad = 0;
    if (live) {
        stage_tile<false, IO>(yr, nt, lane, L, tile * L, neg, stagey, emax, bad);
        if constexpr (WEIGHTED)
            stage_tile<true, IO>(wr, nt, lane, L, tile * L, false, stagew, ewmax, bad);
    }
    emax = tile_warp_max(emax, L);
    const int bad_or = tile_warp_or((int)bad, L);
    if (WEIGHTED) ewmax = tile_warp_max(ewmax, L);
    if (live && seg_first) {
        atomicMax(&info[tile * 4 + kInfoEmax], emax);
        if (WEIGHTED) atomicMax(&info[tile * 4 + kInfoEwmax], ewmax);
        if (bad_or) atomicOr(&info[tile * 4 + kInfoBad], bad_or);
    }
    __syncthreads();
    H.bad = live ? (uint32_t)info[tile * 4 + kInfoBad] : 0u;
    const bool work = live && H.bad == 0;
    const int e = work ? min(max(nt - (lane << 5), 0), 32) : 0;
    H.e = e;

    // ---- the lane's values into registers ----
    IO yv[32], wv[WEIGHTED ? 32 : 1];
    if constexpr (sizeof(IO) == 4) {
        const float4* sy4 = reinterpret_cast<const float4*>(stagey);
        const float4* sw4 = reinterpret_cast<const float4*>(stagew);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 v = sy4[sunit(gl, q)];
            yv[4 * q] = v.x; yv[4 * q + 1] = v.y; yv[4 * q + 2] = v.z; yv[4 * q + 3] = v.w;
            if constexpr (WEIGHTED) {
                const float4 x = sw4[sunit(gl, q)];
                wv[4 * q] = x.x; wv[4 * q + 1] = x.y; wv[4 * q + 2] = x.z; wv[4 * q + 3] = x.w;
            }
        }
    } else {
        const double2* sy2 = reinterpret_cast<const double2*>(stagey);
        const double2* sw2 = reinterpret_cast<const double2*>(stagew);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const double2 v = sy2[sunit_t<double>(gl, q)];
            yv[2 * q] = v.x; yv[2 * q + 1] = v.y;
            if constexpr (WEIGHTED) {
                const double2 x = sw2[sunit_t<double>(gl, q)];
                wv[2 * q] = x.x; wv[2 * q + 1] = x.y;
            }
        }
    }
    int pemax = 0;
    if constexpr (WEIGHTED) {
        // the S grid comes from the largest exponent of the products w*y
        int pe = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (k < e) pe = max(pe, bexp(wv[k]) + bexp(yv[k]));
        pe = tile_warp_max(pe, L);
        if (live && seg_first) atomicMax(&info[tile * 4 + kInfoPemax], pe);
    }
    __syncthreads();   // staging read: Sx may now be written
    emax = max(info[tile * 4 + kInfoEmax], 1);
    pemax = max(info[tile * 4 + kInfoPemax], 2);
    ewmax = max(info[tile * 4 + kInfoEwmax], 1);
    H.qs = WEIGHTED ? qexp_prod_t<IO>(pemax) : qexp_unit_t<IO>(emax);
    H.qw = WEIGHTED ? qexp_unit_t<IO>(ewmax) : 0;

    // ---- candidates and lane-relative cumulative sums ----
    int64_t* myS = Sx + gl * kRow;
    int64_t* myW = Wx + gl * kRow;
    int64_t s = 0, wsum = 0;
    uint32_t cand = 0;
    int64_t u_first = 0, o_first = 1, u_last = 0, o_last = 1;   // the lane's first and last elements
    {
        const QuantT<IO> qy(emax), qw(ewmax);
        int64_t up = 0, op = 1;   // previous element's value and weight
        myS[0] = 0;
        if constexpr (WEIGHTED) myW[0] = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const bool in = k < e;
            int64_t uk, ok;
            if constexpr (WEIGHTED) {
                uk = in ? quant_prod(wv[k], yv[k], pemax) : 0;
                ok = in ? max(qw(wv[k]), (int64_t)1) : 0;
                // point k is locally convex: mean of element k-1 < mean of element k
                if (k > 0 && in && (__int128)up * ok < (__int128)uk * op) cand |= 1u << k;
            } else {
                uk = in ? qy(yv[k]) : 0;
                ok = in ? 1 : 0;
                if (k > 0 && in && up < uk) cand |= 1u << k;
            }
            if (k == 0) { u_first = uk; o_first = ok > 0 ? ok : 1; }
            up = uk;
            op = ok > 0 ? ok : 1;
            s += uk;
            myS[k + 1] = s;
            if constexpr (WEIGHTED) {
                wsum += ok;
                myW[k + 1] = wsum;
            }
        }
        u_last = up;
        o_last = op;
    }
    // lane starts: exclusive scan of lane totals over the tile
    {
        const int64_t inc = tile_scan_incl<NT>(s, lane, L, scan);
        LSa[tile * (L + 1) + lane] = inc - s;
        if (lane == L - 1) LSa[tile * (L + 1) + L] = inc;
        if constexpr (WEIGHTED) {
            const int64_t incw = tile_scan_incl<NT>(wsum, lane, L, scan);
            LWa[tile * (L + 1) + lane] = incw - wsum;
            if (lane == L - 1) LWa[tile * (L + 1) + L] = incw;
        }
    }

    const int64_t ls = LSa[tile * (L + 1) + lane];
    const int64_t lw = WEIGHTED ? LWa[tile * (L + 1) + lane] : 0;
    const uint32_t allp = e >= 32 ? 0xffffffffu : ((1u << e) - 1u);

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

    // ---- chunks of long rows (the tile is the CTA): when every point is
    // locally convex (each element's mean below the next one's, across lane
    // boundaries too) the polyline of cumulative sums turns strictly left at
    // every point, so every point is a hull vertex and no hull needs building ----
    H.all = false;
    if constexpr (!EMIT && RMAX == 1) {
        // first without the lanes' first points (one barrier, which also
        // orders the lane starts' writes before their reads below)
        const bool inner = !work || ((cand | 1u) & allp) == allp;
        if (__syncthreads_and(inner) && live && H.bad == 0) {
            // the previous lane's last element: a shuffle inside a warp, shared
            // memory across warps (the bridge area is free until the rounds)
            int64_t pu = __shfl_up_sync(kFull, u_last, 1), po = __shfl_up_sync(kFull, o_last, 1);
            int64_t* xl = reinterpret_cast<int64_t*>(bridge);
            if ((tid & 31) == 31 && tid + 1 < NT) { xl[2 * (tid >> 5)] = u_last; xl[2 * (tid >> 5) + 1] = o_last; }
            __syncthreads();
            if ((tid & 31) == 0 && tid > 0) { pu = xl[2 * ((tid >> 5) - 1)]; po = xl[2 * ((tid >> 5) - 1) + 1]; }
            bool rise;
            if constexpr (WEIGHTED) rise = (__int128)pu * o_first < (__int128)u_first * po;
            else rise = pu < u_first;
            const bool ok = !work || lane == 0 || rise;
            if (__syncthreads_and(ok)) {
                H.all = true;
                return;
            }
        }
    }

    // ---- chunks of long rows (unit weights, float32 input; the tile is the
    // CTA): the candidates filter (iso_filter.cuh); when few survive, their
    // list, whose hull one warp finds by farthest-point levels ----
    H.list = 0;
    if constexpr (!EMIT && !WEIGHTED && sizeof(IO) == 4) {
        static_assert((3 * NT + 3 * (NT / 32)) * 4 <= SM::kPxB &&
                      kListCap * 10 + list_scratch_bytes(NT) <= SM::kPxB, "list area");
        unsigned char* area = smem + SM::oPx;
        if constexpr (RMAX != 1) __syncthreads();            // lane starts written (RMAX 1: above)
        cand = chunk_filter<NT>(yv, e, lane, nt, H.qs, LSa, work ? cand : 0u,
                                reinterpret_cast<float*>(area));
        const int cnt_l = __popc(cand);
        const int64_t inc = tile_scan_incl<NT>(cnt_l, lane, L, scan);
        __shared__ int s_total;
        if (lane == L - 1) s_total = (int)inc;
        __syncthreads();                                     // scratch read, total known
        const int n_list = s_total + 2;
        if (work && n_list <= kListCap) {
            uint16_t* LP = reinterpret_cast<uint16_t*>(area);
            int64_t* LSv = reinterpret_cast<int64_t*>(area + 2 * kListCap);
            int j = 1 + (int)inc - cnt_l;
            uint32_t m = cand;
            while (m) {
                const int k = __ffs(m) - 1;
                m &= m - 1u;
                LP[j] = (uint16_t)((lane << 5) + k);
                LSv[j] = ls + myS[k];
                ++j;
            }
            if (lane == 0) { LP[0] = 0; LSv[0] = 0; LP[n_list - 1] = (uint16_t)nt; LSv[n_list - 1] = LSa[L]; }
            __syncthreads();
            if (n_list <= NT) {
                // a short list: the CTA's pairwise passes
                cta_list_hull<NT>(LP, LSv, n_list, maska, area + 10 * kListCap);
                H.list = n_list;
                return;
            }
            __shared__ int s_ok;
            if (tid < 32) {
                const bool ok = warp_list_hull(LP, LSv, n_list, maska);
                if (tid == 0) s_ok = ok;
            }
            __syncthreads();
            if (s_ok) { H.list = n_list; return; }
        }
    }



    bool rel = false;       // rows hold tile-relative sums
    bool oneblock = false;  // every tile of the CTA is one block
    H.quick = false;
    H.oneblock = false;
    // ---- whole rows of more than one warp: a tile none of whose points (the
    // locally convex ones, and each lane's first) lies strictly below the
    // chord from its first point to its end is one block, its hull that chord;
    // the lane hulls and merging rounds are then skipped (a soft-rank row,
    // whose merging rounds would each walk the whole merged hull).  Rows of
    // one warp or less have the farthest-point levels for that. ----
    if constexpr (EMIT && RMAX == 1) {
        __syncthreads();                                     // lane starts written
        bool below = false;
        uint32_t m = work ? (cand | (lane > 0 ? 1u : 0u)) & allp : 0u;
        if (m) {
            const int64_t Sn = T.LS[L];
            while (m && !below) {
                const int k = __ffs(m) - 1;
                m &= m - 1u;
                const int64_t Sp = ls + myS[k];
                if constexpr (WEIGHTED) {
                    QBest<true> d;
                    below = qdist(lw + myW[k], Sp, T.LW[L], Sn, d);
                } else {
                    QBest<false> d;
                    below = qdist((lane << 5) + k, Sp, nt, Sn, d);
                }
            }
        }
        oneblock = !__syncthreads_or(below);
        H.oneblock = oneblock;
    }
    // ---- few vertices expected: the hull by levels of farthest-point splits,
    // on tile-relative rows ----
    if constexpr (EMIT && RMAX > 1) if (!oneblock && L >= kQuickMinLanes && L <= 32) {
        __syncthreads();   // lane starts written
        // the tile's trend: mean of lanes [0, L/2) against the rest
        bool down = false;
        if (work && lane == 0) {
            const int h = L >> 1;
            const int64_t S1 = T.LS[h], S2 = T.LS[L] - S1;
            const int64_t W1 = WEIGHTED ? T.LW[h] : (int64_t)min(h << 5, nt);
            const int64_t W2 = (WEIGHTED ? T.LW[L] : (int64_t)nt) - W1;
            down = W2 > 0 && (__int128)S1 * W2 > (__int128)S2 * W1;
        }
        const int tiles = __syncthreads_count(work && lane == 0);
        const int downs = __syncthreads_count(down);
        const int dense = __syncthreads_count(work && __popc(cand & allp) > 24);
        const int filled = __syncthreads_count(e > 0);
        if (tiles > 0 && downs == tiles && dense * kQuickDense <= filled) {
#pragma unroll
            for (int k = 0; k <= 32; ++k) myS[k] += ls;
            if constexpr (WEIGHTED) {
#pragma unroll
                for (int k = 0; k <= 32; ++k) myW[k] += lw;
            }
            rel = true;
            H.quick = tile_quickhull<WEIGHTED>(T, summ, lane, L, e, work, cand);
        }
    }
    if (H.quick) return;

    // ---- lane hulls in bit masks ----
    // Each edge's slope is its element's mean, so a lane whose every interior
    // point is locally convex (strictly increasing means) is a strictly convex
    // chain: all its points are vertices and the monotone chain is not needed.
    uint32_t mask = oneblock ? ((work && lane == 0 && nt > 0) ? 1u : 0u)
                             : ((cand | 1u) & allp) == allp ? (e > 0 ? allp : 0u)
                                                            : lane_hull<WEIGHTED>(myS, myW, cand, e);

    if constexpr (EMIT) {
        // ---- rows become tile-relative; the lane hulls are merged in rounds
        // by walking over the vertex masks: pairs of 2^r lanes, up to the
        // whole tile (Section 3.2).  Rounds whose groups lie inside one warp
        // synchronise the warp only. ----
        if (!rel) {
#pragma unroll
            for (int k = 0; k <= 32; ++k) myS[k] += ls;
            if constexpr (WEIGHTED) {
#pragma unroll
                for (int k = 0; k <= 32; ++k) myW[k] += lw;
            }
        }
        maska[gl] = mask;
        {
            const uint32_t bal = __ballot_sync(kFull, mask != 0u);
            if ((tid & 31) == 0) summ[tid >> 5] = bal;
        }
        __syncthreads();
        for (int r = 0; !oneblock && (1 << r) < L; ++r) {
            const int grp = lane >> (r + 1);
            const int A0 = grp << (r + 1);
            const int B0 = A0 + (1 << r);
            const int Bend = A0 + (2 << r);
            const bool active = work && ((B0 << 5) < nt);
            // one slot per group; rounds inside a warp use slots of their own warp
            // only, since warps are not synchronised with each other there
            const int slot = r < 5 ? ((tid >> 5) << 4) + ((tid & 31) >> (r + 1)) : (tid >> (r + 1));
            if (active && lane == A0) {
                int a, b;
                if (r < 5) tile_bridge<WEIGHTED, true>(T, A0, B0, Bend, a, b);
                else tile_bridge<WEIGHTED, false>(T, A0, B0, Bend, a, b);
                bridge[slot] = make_int2(a, b);
            }
            if (r < 5) __syncwarp(); else __syncthreads();
            if (active) {
                const int2 ab = bridge[slot];
                if (ab.x != ab.y) {
                    mask = clear_between(mask, lane, ab.x, ab.y);
                    maska[gl] = mask;
                }
            }
            const uint32_t bal = __ballot_sync(kFull, mask != 0u);
            if ((tid & 31) == 0) summ[tid >> 5] = bal;
            if (r + 1 < 5) __syncwarp(); else __syncthreads();
        }
        __syncthreads();
    } else {
        // ---- each lane hull moves to the front of its row, tile-relative,
        // with its points' indices; the end point of a group of lanes is the
        // next group's first point (lane starts LS, LW) ----
        uint16_t* Px = reinterpret_cast<uint16_t*>(smem + SM::oPx);
        int* cnt = reinterpret_cast<int*>(smem + SM::oCnt);
        uint16_t* myP = Px + gl * kRow;
        int c = 0;
        uint32_t mm = mask;
        const int64_t ls2 = rel ? 0 : ls, lw2 = rel ? 0 : lw;
        while (mm) {
            const int k = __ffs(mm) - 1;
            mm &= mm - 1u;
            myS[c] = myS[k] + ls2;
            if constexpr (WEIGHTED) myW[c] = myW[k] + lw2;
            myP[c] = (uint16_t)((lane << 5) + k);
            ++c;
        }
        cnt[gl] = c;
        __syncwarp();
        // ---- merge rounds over the compact lists: pairs of 2^r lanes.  The
        // group's first lane finds the bridge; the group's lanes in its first
        // warp move the right list's kept tail behind the left list's kept
        // head (the copy the paper's segment lists avoid; here the lists are
        // short and in shared memory, and on a chain convex at the junction
        // the lists are already adjacent). ----
        for (int r = 0; (1 << r) < L; ++r) {
            const bool cross = (2 << r) > 32;
            if (cross) __syncthreads();
            const int A0 = (lane >> (r + 1)) << (r + 1);
            const int B0 = A0 + (1 << r);
            const int T_ = cross ? 32 : (2 << r);
            int dst = 0, src = 0, len = 0;
            if (work && lane == A0 && (B0 << 5) < nt) {
                const int base = tile * L;
                const int eb = min(A0 + (2 << r), L);          // R's end point: lane eb's start
                const int64_t SE = LSa[tile * (L + 1) + eb];
                const int64_t WE = WEIGHTED ? LWa[tile * (L + 1) + eb] : (int64_t)min(eb << 5, nt);
                dst = (base + A0) << 5;                         // flat list starts
                src = (base + B0) << 5;
                compact_merge<WEIGHTED>(Sx, Wx, Px, dst, cnt + base + A0, src, cnt[base + B0],
                                        SE, WE, dst, src, len);
            }
            const int lead = (tid & 31) & ~(T_ - 1);
            dst = __shfl_sync(kFull, dst, lead);
            src = __shfl_sync(kFull, src, lead);
            len = __shfl_sync(kFull, len, lead);
            if (dst == src) len = 0;                           // already in place
            const int tl = (tid & 31) & (T_ - 1);
            int nr = (len + T_ - 1) / T_;
            for (int d = T_; d < 32; d <<= 1) nr = max(nr, __shfl_xor_sync(kFull, nr, d));
            for (int q = 0; q < nr; ++q) {
                const int t = q * T_ + tl;
                int64_t sv = 0, wv = 0;
                uint16_t pv = 0;
                const int fs = src + t, fd = dst + t;           // flat entries
                if (t < len) {
                    sv = Sx[fs + (fs >> 5)];
                    if constexpr (WEIGHTED) wv = Wx[fs + (fs >> 5)];
                    pv = Px[fs + (fs >> 5)];
                }
                __syncwarp();
                if (t < len) {
                    Sx[fd + (fd >> 5)] = sv;
                    if constexpr (WEIGHTED) Wx[fd + (fd >> 5)] = wv;
                    Px[fd + (fd >> 5)] = pv;
                }
                __syncwarp();
            }
        }
        __syncthreads();
    }
}

// Slope of the edge between tile points a < b, rounded to the I/O type from
// the exact integer differences (up to the rounding of the two conversions).
template <bool WEIGHTED, class IO = float>
__device__ __forceinline__ IO tile_slope(const Tile& T, int a, int b, int qs, int qw) {
    const int64_t dS = tile_S<WEIGHTED>(T, b) - tile_S<WEIGHTED>(T, a);
    const int64_t dW = tile_W<WEIGHTED>(T, b) - tile_W<WEIGHTED>(T, a);
    return ratio_t<IO>(dS, dW, qs - qw);
}

// A lane's 32 outputs into its swizzled staging row (16-byte stores).
template <class IO>
__device__ __forceinline__ void stage_out(IO* ost, int gl, const IO (&o)[32]) {
    if constexpr (sizeof(IO) == 4) {
        float4* o4 = reinterpret_cast<float4*>(ost);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            o4[sunit(gl, q)] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    } else {
        double2* o2 = reinterpret_cast<double2*>(ost);
#pragma unroll
        for (int q = 0; q < 16; ++q) o2[sunit_t<double>(gl, q)] = make_double2(o[2 * q], o[2 * q + 1]);
    }
}

// Coalesced write of a tile's n staged outputs (rows g0.. of ost) to orow by
// its L lanes, with 16-byte stores where orow is 16-byte aligned; NaN for a
// rejected row.
template <class IO>
__device__ __forceinline__ void write_row(IO* __restrict__ orow, const IO* ost, int g0, int n,
                                          int lane, int L, bool work) {
    const IO qnan = qnan_t<IO>();
    constexpr int P = IoT<IO>::kPerV;
    using V = typename IoT<IO>::V;
    if ((reinterpret_cast<uintptr_t>(orow) & 15u) == 0) {
        const int nv = n / P;
        const V* sv = reinterpret_cast<const V*>(ost);
        for (int i = lane; i < nv; i += L) {
            const int ev = i * P;
            V v = sv[sunit_t<IO>(g0 + (ev >> 5), (ev & 31) / P)];
            if (!work) {
                if constexpr (sizeof(IO) == 4) v = make_float4(qnan, qnan, qnan, qnan);
                else v = make_double2(qnan, qnan);
            }
            reinterpret_cast<V*>(orow)[i] = v;
        }
        for (int i = nv * P + lane; i < n; i += L)
            orow[i] = work ? ost[spos_t<IO>(g0 + (i >> 5), i & 31)] : qnan;
    } else {
        for (int i = lane; i < n; i += L)
            orow[i] = work ? ost[spos_t<IO>(g0 + (i >> 5), i & 31)] : qnan;
    }
}

}  // namespace isodev
