// Long rows (n > 8,192): the paper's three-level algorithm (Section 3).  Templates;
// iso_long.cu and iso_long_f64.cu instantiate them for float and double I/O.
//
//  1. chunk_hull_kernel: one CTA per chunk builds the chunk's hull (lanes ->
//     warps -> CTA, Sections 3.1-3.2) and writes its vertices once into the
//     chunk's slot, with coordinates relative to the chunk (Section 3.3).
//  2. merge_groups_kernel and merge_top_kernel: the chunk hulls are merged in
//     a tree.  A node is a list of segments (chunk, first vertex, last vertex),
//     at most one per chunk (Definition 4.3, Theorem 4.4); a merge finds the
//     bridge by moving its two ends to their tangent points in turn, a few
//     steps by walking and then by bisection over the list, cuts two segments
//     and moves the right list's descriptors down.  No vertex is ever copied
//     between levels.  The first levels run in one CTA per group of 64 chunks,
//     all groups at once; the rest in one CTA per row.  A CTA reads the hull
//     vertices it needs into shared memory when they fit (noisy rows keep few
//     vertices), else it reads them from the slots in global memory.  The top
//     kernel then finds each chunk's range in the root list and the root
//     vertices before and after it (Section 3.4, Corollary 4.5).
//  3. expand_kernel: one CTA per chunk writes every element's slope and its
//     block-start byte (Section 3.4).
//
// The rows are either a dense [rows, n] batch or the long segments of a ragged
// batch (LongGeo): the kernels find their row's place from the geometry.
#pragma once

#include "../../include/iso.h"
#include "iso_internal.h"
#include "iso_tile.cuh"

#include <algorithm>

namespace isodev {

namespace {

constexpr int kMergeThreads = 512;
constexpr int64_t kRaggedTopCtas = 152;  // one top-merge CTA per SM
constexpr int kMergeSmem = 210 * 1024;    // shared memory of the merge kernel

template <bool WEIGHTED> struct LongCfg;
#ifndef ISO_UNIT_NT
#define ISO_UNIT_NT 128
#endif
template <> struct LongCfg<false> { static constexpr int NT = ISO_UNIT_NT; static constexpr int C = 32 * ISO_UNIT_NT; };
#ifndef ISO_WEIGHTED_NT
#define ISO_WEIGHTED_NT 128
#endif
template <> struct LongCfg<true> { static constexpr int NT = ISO_WEIGHTED_NT; static constexpr int C = 32 * ISO_WEIGHTED_NT; };

typedef __int128 i128;

#ifndef ISO_GROUP
#define ISO_GROUP 64
#endif
constexpr int kGroup = ISO_GROUP;
// Vertices of a group's merged hull kept as a flat array in the workspace for
// the top merge (groups with more take the segment-list route).
constexpr int kGroupFlatCap = 1024;

struct ChunkMeta {
    int32_t h;      // hull vertices (both ends included)
    int32_t bad;    // ISO_ROW_BAD_* bits
    int32_t qs, qw; // quantum exponents of S and W
    int64_t totS, totW;   // chunk totals (chunk quanta)
};

struct ChunkEnds {            // per chunk, from the root list
    int32_t lo, hi;           // rank range of the chunk's root segment, lo > hi if none
    int32_t pt0_vertex;       // 1 if the chunk's first point is a root vertex (closes the previous segment)
    int32_t bad;              // row status bits
    double in_sl;             // slope of the root edge entering the chunk (chunk 0: 0)
    double out_sl;            // slope of the root edge leaving its last root vertex (0 if none)
};                            // (slopes in values: edge_slope, before the cast to the I/O type)

struct LongWs {
    ChunkMeta* meta;   // [M]
    uint16_t* slot_p;  // [M][C+1] vertex point index within the chunk
    int64_t* slot_S;   // [M][C+1]
    int64_t* slot_W;   // [M][C+1] (weighted)
    int4* seg;         // [M] segment lists (global-memory trees)
    int32_t* cnt;      // [M]
    int32_t* segOf;    // [M]
    int32_t* nextSeg;  // [M]
    int32_t* prevSeg;  // [M]
    i128* offS;        // [M] chunk start, row coordinates (row quanta)
    i128* offW;        // [M]
    int32_t* dS;       // [M] shift from chunk to row quantum
    int32_t* dW;       // [M]
    int4* eInfo;       // [M] chunk ends (ChunkEnds), as arrays: (lo, hi, pt0_vertex, bad)
    double* eIn;       // [M] slope of the root edge entering the chunk
    double* eOut;      // [M] slope of the root edge leaving its last root vertex
    int32_t* rowq;     // [rows][4]: qs_row, qw_row, bad
    i128* gfS;         // [G][kGroupFlatCap] each group's merged hull, row coordinates
    void* gfW;         // i128 (weighted) or int64 (unit weights: point index) per vertex
    uint32_t* gfTag;   // chunk << 13 | rank
    int32_t* gfN;      // [G] its vertices, -1 when it is only a segment list
    unsigned long long* bst;   // bridge-search counters (nullptr: not counted)
    int bmax;                  // passes of a segment-list search before its nested bisection
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// A chunk's ends, kept as arrays so that a warp's stores for consecutive
// chunks are contiguous.
__device__ __forceinline__ void store_ends(const LongWs& ws, int64_t c, const ChunkEnds& ce) {
    ws.eInfo[c] = make_int4(ce.lo, ce.hi, ce.pt0_vertex, ce.bad);
    ws.eIn[c] = ce.in_sl;
    ws.eOut[c] = ce.out_sl;
}
__device__ __forceinline__ ChunkEnds load_ends(const LongWs& ws, int64_t c) {
    ChunkEnds ce;
    const int4 e = ws.eInfo[c];
    ce.lo = e.x; ce.hi = e.y; ce.pt0_vertex = e.z; ce.bad = e.w;
    ce.in_sl = ws.eIn[c];
    ce.out_sl = ws.eOut[c];
    return ce;
}

// Workspace of `rows` long rows holding M chunks in all.
template <bool WEIGHTED>
__host__ __device__ inline size_t carve(void* base, int64_t rows, int64_t M, LongWs* ws) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const size_t cap = (size_t)C + 1;
    size_t off = 0;
    char* b = static_cast<char*>(base);
    auto take = [&](size_t bytes) -> void* {
        void* p = b ? (void*)(b + off) : nullptr;
        off += align256(bytes);
        return p;
    };
    LongWs w;
    w.meta = (ChunkMeta*)take(sizeof(ChunkMeta) * M);
    w.slot_p = (uint16_t*)take(sizeof(uint16_t) * cap * M);
    w.slot_S = (int64_t*)take(sizeof(int64_t) * cap * M);
    w.slot_W = WEIGHTED ? (int64_t*)take(sizeof(int64_t) * cap * M) : nullptr;
    w.seg = (int4*)take(sizeof(int4) * M);
    w.cnt = (int32_t*)take(sizeof(int32_t) * M);
    w.segOf = (int32_t*)take(sizeof(int32_t) * M);
    w.nextSeg = (int32_t*)take(sizeof(int32_t) * M);
    w.prevSeg = (int32_t*)take(sizeof(int32_t) * M);
    w.offS = (i128*)take(sizeof(i128) * M);
    w.offW = (i128*)take(sizeof(i128) * M);
    w.dS = (int32_t*)take(sizeof(int32_t) * M);
    w.dW = (int32_t*)take(sizeof(int32_t) * M);
    w.eInfo = (int4*)take(sizeof(int4) * M);
    w.eIn = (double*)take(sizeof(double) * M);
    w.eOut = (double*)take(sizeof(double) * M);
    w.rowq = (int32_t*)take(sizeof(int32_t) * 4 * rows);
    const size_t G = (size_t)(M / kGroup + rows + 1);      // groups of all rows, at most
    w.gfS = (i128*)take(sizeof(i128) * kGroupFlatCap * G);
    w.gfW = take((WEIGHTED ? sizeof(i128) : sizeof(int64_t)) * kGroupFlatCap * G);
    w.gfTag = (uint32_t*)take(sizeof(uint32_t) * kGroupFlatCap * G);
    w.gfN = (int32_t*)take(sizeof(int32_t) * G);
#ifdef __CUDA_ARCH__
    w.bst = nullptr;
    w.bmax = ISO_BRIDGE_MAX_PASSES;
#else
    if (ws) {
        const BridgeDebug bd = bridge_debug();
        w.bst = bd.stats;
        w.bmax = bd.max_passes;
    }
#endif
    if (ws) *ws = w;
    return off;
}

// Where the long rows of a call lie.  A dense batch: row r holds elements
// r*n .. r*n+n-1 and chunks r*m .. r*m+m-1.  A ragged batch (segments of their
// own lengths laid end to end, see iso_ragged.cu): per-row tables that a plan
// kernel writes on the device, and the counts of rows, chunks and groups that
// the grids, sized for the largest possible counts, are checked against.
struct LongGeo {
    int64_t n = 0, m = 0;                 // dense: row length, chunks per row
    const int64_t* e0 = nullptr;          // ragged [rows]: the row's first element (null: dense)
    const int64_t* len = nullptr;         // [rows]: its length (> kRowMax)
    const int64_t* c0 = nullptr;          // [rows]: its first chunk
    const int64_t* g0 = nullptr;          // [rows]: its first group of kGroup chunks
    const int32_t* id = nullptr;          // [rows]: its segment index
    const int32_t* chunk_row = nullptr;   // [chunks]: row of each chunk
    const int32_t* group_row = nullptr;   // [groups]: row of each group
    const int64_t* count = nullptr;       // [3]: rows, chunks, groups
};

struct RowRef { int64_t id, e0, n, m, c0; };

template <int C>
__device__ __forceinline__ RowRef geo_row(const LongGeo& g, int64_t r) {
    if (!g.e0) return RowRef{r, r * g.n, g.n, g.m, r * g.m};
    const int64_t n = g.len[r];
    return RowRef{g.id[r], g.e0[r], n, (n + C - 1) / C, g.c0[r]};
}

// Programmatic dependent launch: a kernel launched with
// cudaLaunchAttributeProgrammaticStreamSerialization may start before the
// previous kernel of the stream has finished; it waits here, before touching
// anything that kernel writes, until that kernel has completed and its memory
// is visible.  A kernel launched without the attribute passes straight on.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the stream's next kernel (launched with the attribute) be scheduled now:
// its CTAs become resident on idle SMs and wait in wait_prior_grid().
__device__ __forceinline__ void launch_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ bool fits64(i128 x) { return (i128)(int64_t)x == x; }

// A double within 3 ulp of a 128-bit integer (exact below 2^53).
__device__ __forceinline__ double i128_to_double(i128 x) {
    if (fits64(x)) return (double)(int64_t)x;
    const bool neg = x < 0;
    const unsigned __int128 u = neg ? (unsigned __int128)0 - (unsigned __int128)x : (unsigned __int128)x;
    const double d = ldexp((double)(uint64_t)(u >> 64), 64) + (double)(uint64_t)u;
    return neg ? -d : d;
}

// The slope of the root edge from (Wa, Sa) to (Wb, Sb) in row coordinates,
// scaled by 2^k from the row's quanta to values (k = qs_row - qw_row): the
// expansion casts it to the I/O type.
__device__ __forceinline__ double edge_slope(i128 Wa, i128 Sa, i128 Wb, i128 Sb, int k);

// Round x / 2^d to nearest (half up); d >= 0.
__device__ __forceinline__ int64_t conv(int64_t x, int d) {
    if (d <= 0) return x;
    if (d >= 63) return 0;
    return (x + (1LL << (d - 1))) >> d;
}

#ifdef ISO_LONG_F64_IO
// float64 I/O: in double.
__device__ __forceinline__ double edge_slope(i128 Wa, i128 Sa, i128 Wb, i128 Sb, int k) {
    const double f = i128_to_double(Sb - Sa) / i128_to_double(Wb - Wa);
    return ldexp(f, k);
}
#else
// A float32 within a few ulp of a 128-bit integer, from 32-bit conversions
// (no 64-bit conversion: those run on the slow FP64 pipe of this part).
__device__ __forceinline__ float i128_to_f32(i128 x) {
    if (fits64(x)) return i64_to_f32((int64_t)x);
    const bool neg = x < 0;
    const unsigned __int128 u = neg ? (unsigned __int128)0 - (unsigned __int128)x : (unsigned __int128)x;
    const uint64_t hi = (uint64_t)(u >> 64), lo = (uint64_t)u;
    const float fh = __fmaf_rn(__uint2float_rn((unsigned)(hi >> 32)), 4294967296.0f, __uint2float_rn((unsigned)hi));
    const float fl = __fmaf_rn(__uint2float_rn((unsigned)(lo >> 32)), 4294967296.0f, __uint2float_rn((unsigned)lo));
    const float f = __fmaf_rn(fh, 0x1p64f, fl);
    return neg ? -f : f;
}
// float32 I/O: in float32, as the slopes inside a chunk are (two rounded
// conversions and one division, scaled exactly): the slope is cast to
// float32 anyway, and the FP64 pipe of one SM would otherwise carry every
// root edge's division.
__device__ __forceinline__ double edge_slope(i128 Wa, i128 Sa, i128 Wb, i128 Sb, int k) {
    return (double)Pow2(k)(i128_to_f32(Sb - Sa) / i128_to_f32(Wb - Wa));
}
#endif

// ---------------------------------------------------------------------------
// 1. chunk hulls
// ---------------------------------------------------------------------------
template <bool WEIGHTED, class IO>
__device__ __forceinline__ void chunk_hull_one(const IO* __restrict__ y,
                                               const IO* __restrict__ w, const LongGeo& geo,
                                               int increasing, const LongWs& ws, int64_t c) {
    constexpr int NT = LongCfg<WEIGHTED>::NT;
    constexpr int C = LongCfg<WEIGHTED>::C;
    extern __shared__ __align__(128) unsigned char smem[];
    using SM = TileSmem<NT, WEIGHTED, false, 1, IO>;
    const RowRef R = geo_row<C>(geo, geo.e0 ? (int64_t)geo.chunk_row[c] : c / geo.m);
    const int64_t e0 = (c - R.c0) * C;
    const int nt = (int)imin64(C, R.n - e0);
    const IO* yr = y + R.e0 + e0;
    const IO* wr = WEIGHTED ? w + R.e0 + e0 : nullptr;

    TileHull H;
    tile_hull_phase<NT, WEIGHTED, false, 1, IO>(yr, wr, nt, true, !increasing, NT, smem, H);

    const int64_t* Sx = reinterpret_cast<const int64_t*>(smem + SM::oSx);
    const int64_t* Wx = reinterpret_cast<const int64_t*>(smem + SM::oWx);
    const size_t cap = (size_t)C + 1;
    uint16_t* sp = ws.slot_p + c * cap;
    int64_t* sS = ws.slot_S + c * cap;
    int64_t* sW = WEIGHTED ? ws.slot_W + c * cap : nullptr;
    int h;
    if (H.all) {
        // every point a vertex: point j = 32 lane + k at its lane's start plus
        // the lane-relative sum (the end point: the tile's total)
        h = nt + 1;
        for (int j = threadIdx.x; j < h; j += NT) {
            const int l = j >> 5, k = j & 31;
            const bool endp = j == nt;
            sp[j] = (uint16_t)j;
            sS[j] = endp ? H.T.LS[NT] : H.T.LS[l] + Sx[l * kRow + k];
            if constexpr (WEIGHTED) sW[j] = endp ? H.T.LW[NT] : H.T.LW[l] + Wx[l * kRow + k];
        }
    } else if (H.list) {
        // the hull of the candidates' list: its vertices (warp 0's bits, lane l
        // holding entries [l K, l K + K)) and the list's last entry, the end point
        __shared__ int s_h;
        if (threadIdx.x < 32) {
            const int wl = threadIdx.x, n = H.list, K = (n - 1 + 31) >> 5;
            const uint16_t* LP = reinterpret_cast<const uint16_t*>(smem + SM::oPx);
            const int64_t* LSv = reinterpret_cast<const int64_t*>(smem + SM::oPx + 2 * kListCap);
            const uint32_t vm = H.T.mask[wl];
            const int cv = __popc(vm);
            int x = cv;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o = __shfl_up_sync(kFull, x, d);
                if (wl >= d) x += o;
            }
            int j = x - cv;
            uint32_t m = vm;
            while (m) {
                const int k = __ffs(m) - 1;
                m &= m - 1u;
                sp[j] = LP[wl * K + k];
                sS[j] = LSv[wl * K + k];
                ++j;
            }
            const int total = __shfl_sync(kFull, x, 31);
            if (wl == 0) { sp[total] = LP[n - 1]; sS[total] = LSv[n - 1]; s_h = total + 1; }
        }
        __syncthreads();
        h = s_h;
    } else {
        // the chunk hull is the compact list of lane 0's row and the chunk's end
        // point: copy them to the slot
        const uint16_t* Px = reinterpret_cast<const uint16_t*>(smem + SM::oPx);
        h = H.bad == 0 ? reinterpret_cast<const int*>(smem + SM::oCnt)[0] + 1 : 0;
        for (int j = threadIdx.x; j < h; j += NT) {
            const bool endp = j == h - 1;
            const int f = j + (j >> 5);                    // flat entry j
            sp[j] = endp ? (uint16_t)nt : Px[f];
            sS[j] = endp ? H.T.LS[NT] : Sx[f];
            if constexpr (WEIGHTED) sW[j] = endp ? H.T.LW[NT] : Wx[f];
        }
    }
    if (threadIdx.x == 0) {
        ChunkMeta mt;
        mt.h = h;
        mt.bad = (int32_t)H.bad;
        mt.qs = H.qs;
        mt.qw = H.qw;
        mt.totS = H.T.LS[NT];
        mt.totW = WEIGHTED ? H.T.LW[NT] : (int64_t)nt;
        ws.meta[c] = mt;
    }
}

// One CTA per chunk; a ragged batch's grid is bounded and its CTAs take the
// chunks in turn.
// CTAs per SM that the chunk kernel's shared memory allows: its registers
// are held to that many (228 KB per SM, 1 KB reserved per CTA).
template <bool WEIGHTED, class IO>
constexpr int chunk_min_blocks() {
    constexpr int b = 233472 / (TileSmem<LongCfg<WEIGHTED>::NT, WEIGHTED, false, 1, IO>::kBytes + 1024);
    return b < 1 ? 1 : (b > 8 ? 8 : b);
}

template <bool WEIGHTED, bool RAGGED, class IO>
__global__ void __launch_bounds__(LongCfg<WEIGHTED>::NT, (chunk_min_blocks<WEIGHTED, IO>()))
chunk_hull_kernel(const IO* __restrict__ y, const IO* __restrict__ w, LongGeo geo,
                  int increasing, LongWs ws) {
    if (!RAGGED) {
        chunk_hull_one<WEIGHTED, IO>(y, w, geo, increasing, ws, blockIdx.x);
        return;
    }
    const int64_t M = geo.count[1];
    for (int64_t c = blockIdx.x; c < M; c += gridDim.x) {
        chunk_hull_one<WEIGHTED, IO>(y, w, geo, increasing, ws, c);
        __syncthreads();   // shared memory is reused by the next chunk
    }
}

// ---------------------------------------------------------------------------
// 2. merge tree over segment lists (one CTA per row)
// ---------------------------------------------------------------------------
extern __shared__ __align__(16) unsigned char merge_smem[];

// A merge's descriptor move: seg[dst + t] = seg[src + t] for t < len (dst < src).
struct Move { int dst, src, len; };

// One segment of a list: a chunk's vertex range, with what its vertices need.
struct Seg {
    int jc, lo, hi;   // chunk (in the row), first and last vertex rank
    int vb;           // first vertex of the chunk in the compact arrays (shared memory)
    int dS, dW;       // chunk-to-row quantum shifts (global memory)
    i128 oS, oW;      // chunk start in row coordinates
};

// Where the merge tree reads a row's chunk hulls and keeps its lists.  SMEM:
// compact copies in shared memory, S and W already on the row's grid; else the
// workspace slots in global memory, converted at every read.
template <bool WEIGHTED, bool SMEM>
struct MView {
    int4* seg;               // (chunk in row, lo, hi, 0)
    int32_t* cnt;
    const i128* offS;
    const i128* offW;
    const int32_t* dS;       // global memory only
    const int32_t* dW;
    const int32_t* vb;       // shared memory only
    const int64_t* S;
    const int64_t* W;
    const uint16_t* P;
    int64_t c0;              // global index of the row's chunk 0
    int C;
    unsigned long long* bst = nullptr;   // bridge-search counters
    int bmax = ISO_BRIDGE_MAX_PASSES;

    __device__ __forceinline__ Seg load(int k) const {
        const int4 s = seg[k];
        Seg g;
        g.jc = s.x; g.lo = s.y; g.hi = s.z;
        g.oS = offS[s.x];
        g.oW = WEIGHTED ? offW[s.x] : (i128)0;
        if constexpr (SMEM) { g.vb = vb[s.x]; g.dS = 0; g.dW = 0; }
        else { g.vb = 0; g.dS = dS[s.x]; g.dW = WEIGHTED ? dW[s.x] : 0; }
        return g;
    }
    __device__ __forceinline__ void at(const Seg& g, int r, i128& Wv, i128& Sv) const {
        if constexpr (SMEM) {
            const int i = g.vb + r;
            Sv = g.oS + S[i];
            if constexpr (WEIGHTED) Wv = g.oW + W[i];
            else Wv = (i128)((int64_t)g.jc * C + P[i]);
        } else {
            const size_t i = (size_t)(c0 + g.jc) * ((size_t)C + 1) + r;
            Sv = g.oS + conv(S[i], g.dS);
            if constexpr (WEIGHTED) Wv = g.oW + conv(W[i], g.dW);
            else Wv = (i128)((int64_t)g.jc * C + P[i]);
        }
    }
};

// The turn o -> a -> b is strictly left, exactly.  Unit weights: every W
// difference is below 2^31 and every S difference below 2^82, so 128-bit
// products are exact (formed from 32 x 32-bit wide products).  Weighted
// rows: a double-precision determinant decides when it is clear of its
// rounding bound, the 256-bit products otherwise.
template <bool WEIGHTED>
__device__ __forceinline__ bool row_turn(i128 Wo, i128 So, i128 Wa, i128 Sa, i128 Wb, i128 Sb) {
    const i128 w1 = Wa - Wo, s1 = Sa - So, w2 = Wb - Wo, s2 = Sb - So;
    if constexpr (!WEIGHTED) {
        // w * s exactly from 32 x 32-bit wide products: |w| < 2^31 (differences
        // of point indices) and |s| < 2^95, so every partial product fits
        auto mul = [](i128 w, i128 s) -> i128 {
            const int64_t wv = (int64_t)(int32_t)(int64_t)w;
            const uint64_t lo = (uint64_t)s;
            const int64_t hi = (int64_t)(s >> 64);
            const int64_t a = wv * (int64_t)(uint32_t)lo;
            const int64_t b = wv * (int64_t)(uint32_t)(lo >> 32);
            return (i128)a + ((i128)b << 32) + ((i128)(wv * hi) << 64);
        };
        return mul(w1, s2) > mul(w2, s1);
    } else {
        if (fits64(w1) && fits64(s1) && fits64(w2) && fits64(s2))
            return left_turn<true>((int64_t)w1, (int64_t)s1, (int64_t)w2, (int64_t)s2);
        const double p = i128_to_double(w1) * i128_to_double(s2);
        const double q = i128_to_double(s1) * i128_to_double(w2);
        const double d = p - q;
        if (fabs(d) > (fabs(p) + fabs(q)) * 0x1p-48) return d > 0.0;
        return sign_det128(w1, s2, s1, w2) > 0;
    }
}

// A position on a list, with its segment and coordinates.
struct Walker {
    int k, r;
    Seg g;
    i128 W, S;
};

// h(x): x strictly below the segment from (AW, AS) to its successor (false
// before the tangent point of A on the right list, true from it on).  B moves
// to the first x in [B, the list's last vertex kRl] with h: bisection over
// segments, then inside one.
template <bool WEIGHTED, class View>
__device__ __forceinline__ void list_tangent_right(const View& V, int kRl, i128 AW, i128 AS, Walker& B) {
    int lo = B.k, hi = kRl;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const Seg gm = V.load(mid), gn = V.load(mid + 1);
        i128 Wm, Sm, Wn, Sn;
        V.at(gm, gm.hi, Wm, Sm);
        V.at(gn, gn.lo, Wn, Sn);
        if (row_turn<WEIGHTED>(AW, AS, Wm, Sm, Wn, Sn)) hi = mid; else lo = mid + 1;
    }
    const Seg g = lo == B.k ? B.g : V.load(lo);
    int rlo = lo == B.k ? B.r : g.lo, rhi = g.hi;
    while (rlo < rhi) {
        const int mid = (rlo + rhi) >> 1;
        i128 Wm, Sm, Wn, Sn;
        V.at(g, mid, Wm, Sm);
        V.at(g, mid + 1, Wn, Sn);
        if (row_turn<WEIGHTED>(AW, AS, Wm, Sm, Wn, Sn)) rhi = mid; else rlo = mid + 1;
    }
    B.k = lo; B.g = g; B.r = rlo;
    V.at(g, rlo, B.W, B.S);
}

// The end of a bridge search whose passes ran out, by nested bisection
// (Theorem 5.2).  a is at or after the bridge's left end on the left list
// (first segment j0) and b is the tangent point of a on the right list (last
// segment kRl).  For x on the left list up to a, t(x) is its tangent point on
// the right list (at or after b); the vertex after x lies strictly below the
// line from x to t(x) for every x before the bridge's left end and for none
// from it on.  The left end is the first x for which it does not: bisection
// over the segments' first vertices, then inside one segment.  The right end
// is t of the left end.
template <bool WEIGHTED, class View>
__device__ __forceinline__ void nested_bridge(const View& V, int j0, int kRl, Walker& a, Walker& b) {
    // x = rank r of segment k (g); its successor is the next rank, else the
    // next segment's first
    auto below = [&](int k, const Seg& g, int r) -> bool {
        i128 Wx, Sx, Wn, Sn;
        V.at(g, r, Wx, Sx);
        if (r < g.hi) {
            V.at(g, r + 1, Wn, Sn);
        } else {
            const Seg h = V.load(k + 1);
            V.at(h, h.lo, Wn, Sn);
        }
        Walker T = b;
        list_tangent_right<WEIGHTED>(V, kRl, Wx, Sx, T);
        return row_turn<WEIGHTED>(Wx, Sx, Wn, Sn, T.W, T.S);
    };
    // the last segment in [j0, a.k] whose first vertex passes (j0 - 1: none)
    const int ak = a.k, ar = a.r;
    int lo = j0 - 1, hi = ak;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const Seg g = V.load(mid);
        if (below(mid, g, g.lo)) lo = mid; else hi = mid - 1;
    }
    int k, r;
    if (lo < j0) {
        k = j0;
        r = V.load(j0).lo;
    } else {
        const Seg g = V.load(lo);
        const int rmax = lo == ak ? ar : g.hi;
        int rl = g.lo + 1, rh = rmax + 1;     // first failing rank; rmax + 1: none here
        while (rl < rh) {
            const int mid = (rl + rh) >> 1;
            if (below(lo, g, mid)) rl = mid + 1; else rh = mid;
        }
        if (rl <= rmax) { k = lo; r = rl; }
        else if (lo < ak) { k = lo + 1; r = V.load(lo + 1).lo; }
        else { k = ak; r = ar; }   // every x up to a passes: ruled out by exact turns
    }
    a.k = k;
    a.g = V.load(k);
    a.r = r;
    V.at(a.g, r, a.W, a.S);
    list_tangent_right<WEIGHTED>(V, kRl, a.W, a.S, b);
}

constexpr int kLinearSteps = 12;   // walk steps before a tangent is found by bisection

// Merge of the lists of the neighbouring nodes starting at j0 and j1
// (Algorithm 1 of the paper, Lemma 4.2): if the two hulls are convex at their
// shared point s, R is appended without s; otherwise the bridge is found by
// alternately moving the left end to its tangent from the right end and the
// right end to its tangent from the left end, a few steps by walking and then
// by bisection over the list (first over segments, then inside one).  The two
// segments the bridge lands in are cut, the merged list's length is set, and
// the move of the right list's tail is returned.  View: MView, or the flat
// arrays of the materialised-copy control (FlatView).  LOOK > 1: inside a
// segment a walk step tests LOOK vertices as independent chains (the group
// merges, whose lists are whole chunk hulls; measured faster there, slower at
// the top levels, where segments hold one or two vertices).
template <bool WEIGHTED, int LOOK = 1, class View>
__device__ __forceinline__ Move merge_plan(const View& V, int j0, int j1) {
    int4* seg = V.seg;
    const int nL = V.cnt[j0], nR = V.cnt[j1];
    const int kLl = j0 + nL - 1, kR0 = j1, kRl = j1 + nR - 1;
    auto turn = [](i128 Wo, i128 So, i128 Wa, i128 Sa, i128 Wb, i128 Sb) {
        return row_turn<WEIGHTED>(Wo, So, Wa, Sa, Wb, Sb);
    };
    // a: the vertex before s on L; b: the vertex after s on R
    Walker a, b;
    i128 Ws, Ss;
    {
        const Seg gl = V.load(kLl);
        V.at(gl, gl.hi, Ws, Ss);
        if (gl.hi > gl.lo) { a.k = kLl; a.g = gl; a.r = gl.hi - 1; }
        else { a.k = kLl - 1; a.g = V.load(kLl - 1); a.r = a.g.hi; }
        V.at(a.g, a.r, a.W, a.S);
        const Seg gr = V.load(kR0);
        if (gr.hi > gr.lo) { b.k = kR0; b.g = gr; b.r = gr.lo + 1; }
        else { b.k = kR0 + 1; b.g = V.load(kR0 + 1); b.r = b.g.lo; }
        V.at(b.g, b.r, b.W, b.S);
    }
    if (turn(a.W, a.S, Ws, Ss, b.W, b.S)) {
        // convex at s: append R without its first vertex s
        int first = kR0;
        const int lo = seg[kR0].y + 1;
        if (lo > seg[kR0].z) first = kR0 + 1;
        else seg[kR0].y = lo;
        const int len = kRl - first + 1;
        V.cnt[j0] = nL + len;
        if (V.bst) atomicAdd(&V.bst[0], 1ull);
        return Move{j0 + nL, first, len};
    }
    // s is not a vertex of the merged hull: the bridge joins L without s to R
    // without s, so a stays before s and b after it.

    // g(x): x strictly below the segment from its predecessor to b (true up to
    // the tangent point of b on L', false after).  Last x in [first, a] with g.
    auto tanL = [&](Walker& A, const Walker& B) {
        // the last segment whose first vertex satisfies g (segment j0: always)
        int lo = j0, hi = A.k;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            const Seg gm = V.load(mid), gp = V.load(mid - 1);
            i128 Wm, Sm, Wp, Sp;
            V.at(gm, gm.lo, Wm, Sm);
            V.at(gp, gp.hi, Wp, Sp);
            if (turn(Wp, Sp, Wm, Sm, B.W, B.S)) lo = mid; else hi = mid - 1;
        }
        const Seg g = lo == A.k ? A.g : V.load(lo);
        int rlo = g.lo, rhi = lo == A.k ? A.r : g.hi;
        while (rlo < rhi) {
            const int mid = (rlo + rhi + 1) >> 1;
            i128 Wm, Sm, Wp, Sp;
            V.at(g, mid, Wm, Sm);
            V.at(g, mid - 1, Wp, Sp);
            if (turn(Wp, Sp, Wm, Sm, B.W, B.S)) rlo = mid; else rhi = mid - 1;
        }
        A.k = lo; A.g = g; A.r = rlo;
        V.at(g, rlo, A.W, A.S);
    };
    // h(x): x strictly below the segment from a to its successor (false before
    // the tangent point of a on R', true from it on).  First x in [b, last] with h.
    auto tanR = [&](const Walker& A, Walker& B) { list_tangent_right<WEIGHTED>(V, kRl, A.W, A.S, B); };

    // Passes of V.bmax at most: a moves only left and b only right, and
    // neither passes the bridge's ends (a tangent point moves right as its
    // source moves left), so each pass leaves a at or after the left end and
    // b at or before the right end; what remains goes to the nested bisection.
    int passes = 0;
    bool nested = false;
    for (;;) {
        if (passes >= V.bmax) { nested = true; break; }
        ++passes;
        bool moved = false;
        // the left end moves to its tangent point from b
        for (int steps = 0;;) {
            const bool hasPrev = a.r > a.g.lo || a.k > j0;
            if (!hasPrev) break;
            if (steps >= kLinearSteps) { tanL(a, b); break; }
            if (LOOK > 1 && a.r - a.g.lo >= LOOK) {
                // LOOK vertices of this segment at once, as independent tests:
                // x_0 = a, x_u = a - u; the walk stops at the first x_u with
                // turn(x_{u+1}, x_u, b)
                i128 Wc[LOOK + 1], Sc[LOOK + 1];
                Wc[0] = a.W; Sc[0] = a.S;
#pragma unroll
                for (int u = 1; u <= LOOK; ++u) V.at(a.g, a.r - u, Wc[u], Sc[u]);
                int u = LOOK;
#pragma unroll
                for (int q = LOOK - 1; q >= 0; --q)
                    if (turn(Wc[q + 1], Sc[q + 1], Wc[q], Sc[q], b.W, b.S)) u = q;
                steps += LOOK;
                if (u > 0) {
                    a.r -= u;
#pragma unroll
                    for (int q = 1; q <= LOOK; ++q)
                        if (q == u) { a.W = Wc[q]; a.S = Sc[q]; }     // no indexed array
                    moved = true;
                }
                if (u < LOOK) break;
                continue;
            }
            ++steps;
            Walker p = a;
            if (a.r > a.g.lo) p.r = a.r - 1;
            else { p.k = a.k - 1; p.g = V.load(p.k); p.r = p.g.hi; }
            V.at(p.g, p.r, p.W, p.S);
            if (turn(p.W, p.S, a.W, a.S, b.W, b.S)) break;
            a = p;
            moved = true;
        }
        // the right end moves to its tangent point from a
        for (int steps = 0;;) {
            const bool hasNext = b.r < b.g.hi || b.k < kRl;
            if (!hasNext) break;
            if (steps >= kLinearSteps) { tanR(a, b); break; }
            if (LOOK > 1 && b.g.hi - b.r >= LOOK) {
                i128 Wc[LOOK + 1], Sc[LOOK + 1];
                Wc[0] = b.W; Sc[0] = b.S;
#pragma unroll
                for (int u = 1; u <= LOOK; ++u) V.at(b.g, b.r + u, Wc[u], Sc[u]);
                int u = LOOK;
#pragma unroll
                for (int q = LOOK - 1; q >= 0; --q)
                    if (turn(a.W, a.S, Wc[q], Sc[q], Wc[q + 1], Sc[q + 1])) u = q;
                steps += LOOK;
                if (u > 0) {
                    b.r += u;
#pragma unroll
                    for (int q = 1; q <= LOOK; ++q)
                        if (q == u) { b.W = Wc[q]; b.S = Sc[q]; }
                    moved = true;
                }
                if (u < LOOK) break;
                continue;
            }
            ++steps;
            Walker q = b;
            if (b.r < b.g.hi) q.r = b.r + 1;
            else { q.k = b.k + 1; q.g = V.load(q.k); q.r = q.g.lo; }
            V.at(q.g, q.r, q.W, q.S);
            if (turn(a.W, a.S, b.W, b.S, q.W, q.S)) break;
            b = q;
            moved = true;
        }
        if (!moved) break;
    }
    if (nested) nested_bridge<WEIGHTED>(V, j0, kRl, a, b);
    if (V.bst) {
        atomicAdd(&V.bst[0], 1ull);
        atomicAdd(&V.bst[1], 1ull);
        atomicAdd(&V.bst[2], (unsigned long long)passes);
        atomicMax(&V.bst[3], (unsigned long long)passes);
        if (nested) atomicAdd(&V.bst[4], 1ull);
    }
    // cut L at a and R at b; R's tail moves down behind L's kept part
    seg[a.k].z = a.r;
    seg[b.k].y = b.r;
    const int len = kRl - b.k + 1;
    V.cnt[j0] = (a.k - j0 + 1) + len;
    return Move{a.k + 1, b.k, len};
}

// Exclusive block-wide scan of one int per thread (blockDim.x <= 1024, a
// multiple of 32); total: the block's sum.
__device__ __forceinline__ int block_excl_scan_int(int v, int* tmp, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(kFull, x, d);
        if (lane >= d) x += o;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nw ? tmp[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(kFull, t, d);
            if (lane >= d) t += o;
        }
        if (lane < nw) tmp[lane] = t;
    }
    __syncthreads();
    const int base = warp ? tmp[warp - 1] : 0;
    total = tmp[nw - 1];
    __syncthreads();
    return base + x - v;
}

// Exclusive block-wide scan of (S, W, H) per thread (blockDim.x <= 1024, a
// multiple of 32); also returns the block totals.
struct Acc3 { i128 s, w; int64_t h; };

__device__ __forceinline__ i128 shfl_up_i128(i128 x, int d) {
    const uint64_t lo = __shfl_up_sync(kFull, (uint64_t)x, d);
    const uint64_t hi = __shfl_up_sync(kFull, (uint64_t)((unsigned __int128)x >> 64), d);
    return (i128)(((unsigned __int128)hi << 64) | lo);
}

__device__ __forceinline__ Acc3 block_excl_scan3(Acc3 v, Acc3* tmp, Acc3& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    Acc3 x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const i128 s = shfl_up_i128(x.s, d);
        const i128 w = shfl_up_i128(x.w, d);
        const int64_t h = __shfl_up_sync(kFull, x.h, d);
        if (lane >= d) { x.s += s; x.w += w; x.h += h; }
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        Acc3 t = lane < nw ? tmp[lane] : Acc3{0, 0, 0};
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const i128 s = shfl_up_i128(t.s, d);
            const i128 w = shfl_up_i128(t.w, d);
            const int64_t h = __shfl_up_sync(kFull, t.h, d);
            if (lane >= d) { t.s += s; t.w += w; t.h += h; }
        }
        if (lane < nw) tmp[lane] = t;
    }
    __syncthreads();
    Acc3 base = warp ? tmp[warp - 1] : Acc3{0, 0, 0};
    total = tmp[nw - 1];
    __syncthreads();
    base.s += x.s - v.s; base.w += x.w - v.w; base.h += x.h - v.h;
    return base;
}

// The merge tree runs in two kernels.  merge_groups_kernel: one CTA per group
// of kGroup consecutive chunks merges them (the tree's first levels), many
// groups at a time across the GPU.  merge_top_kernel: one CTA per row merges
// the groups' lists (the remaining levels) and finds each chunk's root segment.
// Each CTA reads its chunk hulls into shared memory when they fit (noisy rows
// keep few vertices; the top kernel reads only the vertices still inside a
// segment), else it reads them from the slots in global memory.
constexpr int kGroupThreads = 512;   // the most threads of a group CTA (fewer when groups are many)
constexpr int kGroupSmem = 48 * 1024;

// Shared-memory layout for mc chunks and H vertices.
struct MergeLayout {
    size_t oSeg, oOffS, oOffW, oCnt, oVb, oSegOf, oNext, oPrev, oS, oW, oP, bytes;
    __device__ __host__ MergeLayout(int64_t mc, int64_t H, bool weighted, bool ends) {
        size_t o = 0;
        auto take = [&](size_t b, size_t al) { o = (o + al - 1) & ~(al - 1); const size_t r = o; o += b; return r; };
        oSeg = take(16 * mc, 16);
        oOffS = take(16 * mc, 16);
        oOffW = weighted ? take(16 * mc, 16) : 0;
        oS = take(8 * H, 8);
        oW = weighted ? take(8 * H, 8) : 0;
        oCnt = take(4 * mc, 4);
        oVb = take(4 * mc, 4);
        oSegOf = ends ? take(4 * mc, 4) : 0;
        oNext = ends ? take(4 * mc, 4) : 0;
        oPrev = ends ? take(4 * mc, 4) : 0;
        oP = weighted ? 0 : take(2 * H, 2);
        bytes = o;
    }
};

// Row quanta and status: the largest chunk quanta and the or of the chunks'
// status bits, over the m chunks of the row (every thread of the CTA calls it).
struct RowQ { int qs, qw, bad; };

// cache: when not null, the row's chunk records are also copied there (m of
// them), for the caller's next pass.
__device__ __forceinline__ RowQ row_quanta(int64_t m, const LongWs& ws, int64_t c0, int* red,
                                           ChunkMeta* cache = nullptr) {
    const int tid = threadIdx.x, nth = blockDim.x;
    if (tid == 0) { red[0] = -100000; red[1] = -100000; red[2] = 0; }
    __syncthreads();
    int qs = -100000, qw = -100000, bad = 0;
    // four chunks in flight per thread (the loads are independent)
    for (int64_t j0 = tid; j0 < m; j0 += 4 * (int64_t)nth) {
        int4 q4[4], t4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t j = j0 + (int64_t)u * nth;
            q4[u] = j < m ? *reinterpret_cast<const int4*>(&ws.meta[c0 + j]) : make_int4(0, 0, -100000, -100000);
            if (cache && j < m) t4[u] = *(reinterpret_cast<const int4*>(&ws.meta[c0 + j]) + 1);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {   // (h, bad, qs, qw)
            bad |= q4[u].y; qs = max(qs, q4[u].z); qw = max(qw, q4[u].w);
            const int64_t j = j0 + (int64_t)u * nth;
            if (cache && j < m) {
                reinterpret_cast<int4*>(&cache[j])[0] = q4[u];
                reinterpret_cast<int4*>(&cache[j])[1] = t4[u];
            }
        }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        qs = max(qs, __shfl_xor_sync(kFull, qs, d));
        qw = max(qw, __shfl_xor_sync(kFull, qw, d));
        bad |= __shfl_xor_sync(kFull, bad, d);
    }
    if ((tid & 31) == 0) {
        atomicMax(&red[0], qs);
        atomicMax(&red[1], qw);
        if (bad) atomicOr(&red[2], bad);
    }
    __syncthreads();
    const RowQ r{red[0], red[1], red[2]};
    __syncthreads();
    return r;
}

// The levels of the tree whose nodes start at multiples of `span0` chunks,
// inside chunks [jb, je): merges of nodes (j0, j0 + span) for span = span0,
// 2 span0, ... while a node of span chunks is smaller than the range.  A team
// of T threads per merge (T = 1 when merges are many): its first thread finds
// the bridge and cuts the lists, then the team moves the right list's
// descriptors in rounds of T.
template <bool WEIGHTED, bool SMEM, int LOOK = 1>
__device__ __forceinline__ void merge_levels(const MView<WEIGHTED, SMEM>& V, int64_t jb, int64_t je,
                                             int64_t span0) {
    const int tid = threadIdx.x, nth = blockDim.x;
    int4* seg = V.seg;
    for (int64_t half = span0; half < je - jb; half <<= 1) {
        const int64_t span = half << 1;
        const int64_t merges = (je - jb + span - 1) / span;
        int T = 1;
        while (T < 32 && (int64_t)(2 * T) * merges <= nth) T <<= 1;
        const int team = tid / T, tl = tid % T, nteams = nth / T;
        for (int64_t g0 = 0; g0 < merges; g0 += nteams) {
            const int64_t g = g0 + team;
            const int64_t j0 = jb + g * span, j1 = j0 + half;
            const bool act = g < merges && j1 < je;
            Move mv{0, 0, 0};
            if (act && tl == 0) mv = merge_plan<WEIGHTED, LOOK>(V, (int)j0, (int)j1);
            if (T == 1) {
                for (int t = 0; t < mv.len; ++t) seg[mv.dst + t] = seg[mv.src + t];
            } else {
                const int lead = (tid & 31) & ~(T - 1);
                mv.dst = __shfl_sync(kFull, mv.dst, lead);
                mv.src = __shfl_sync(kFull, mv.src, lead);
                mv.len = __shfl_sync(kFull, mv.len, lead);
                int nr = (mv.len + T - 1) / T;
                for (int d = T; d < 32; d <<= 1) nr = max(nr, __shfl_xor_sync(kFull, nr, d));
                for (int q = 0; q < nr; ++q) {
                    const int t = q * T + tl;
                    int4 d = make_int4(0, 0, 0, 0);
                    if (t < mv.len) d = seg[mv.src + t];
                    __syncwarp();
                    if (t < mv.len) seg[mv.dst + t] = d;
                    __syncwarp();
                }
            }
        }
        __syncthreads();
    }
}

// Vertices (chunk jc, ranks lo..lo+len-1) into shared memory at base, on the
// row's grid, for the chunks of [jb, je) with len > 0: vertex i of the range
// total is found by bisection over the bases; four vertices per thread in
// flight.
template <bool WEIGHTED>
__device__ __forceinline__ void copy_vertices(const LongWs& ws, int64_t c0, int jb, int je,
                                              const int32_t* base, const int32_t* lo0, int64_t H,
                                              int64_t* Sw, int64_t* Ww, uint16_t* Pw) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int tid = threadIdx.x, nth = blockDim.x;
    constexpr int U = 4;
    for (int64_t i0 = tid; i0 < H; i0 += (int64_t)U * nth) {
        int jc[U], r[U];
        int64_t sv[U], wv[U];
        uint16_t pv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + (int64_t)u * nth;
            jc[u] = -1;
            if (i < H) {
                int lo = jb, hi = je - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (base[mid] <= i) lo = mid; else hi = mid - 1;
                }
                jc[u] = lo;
                r[u] = (int)(i - base[lo]) + lo0[lo];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (jc[u] < 0) continue;
            const size_t g = (size_t)(c0 + jc[u]) * ((size_t)C + 1) + r[u];
            sv[u] = ws.slot_S[g];
            if (WEIGHTED) wv[u] = ws.slot_W[g]; else pv[u] = ws.slot_p[g];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (jc[u] < 0) continue;
            const int64_t i = i0 + (int64_t)u * nth;
            Sw[i] = conv(sv[u], ws.dS[c0 + jc[u]]);
            if (WEIGHTED) Ww[i] = conv(wv[u], ws.dW[c0 + jc[u]]); else Pw[i] = pv[u];
        }
    }
}

template <bool WEIGHTED, bool SMEM>
__device__ __forceinline__ void merge_group(int64_t m, const LongWs& ws, int64_t c0, int jb, int je,
                                            const i128* gS, const i128* gW, const int32_t* gH,
                                            int64_t Hg) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int tid = threadIdx.x;
    const int mg = je - jb;
    MergeLayout L(mg, SMEM ? Hg : 0, WEIGHTED, false);
    unsigned char* sm = merge_smem;
    MView<WEIGHTED, SMEM> V;
    V.c0 = c0;
    V.C = C;
    V.bst = ws.bst;
    V.bmax = ws.bmax;
    if constexpr (SMEM) {
        // arrays of the group's chunks, indexed by the chunk's index in the row
        V.seg = reinterpret_cast<int4*>(sm + L.oSeg) - jb;
        V.cnt = reinterpret_cast<int32_t*>(sm + L.oCnt) - jb;
        V.offS = reinterpret_cast<i128*>(sm + L.oOffS) - jb;
        V.offW = reinterpret_cast<i128*>(sm + L.oOffW) - jb;
        V.vb = reinterpret_cast<int32_t*>(sm + L.oVb) - jb;
        V.S = reinterpret_cast<int64_t*>(sm + L.oS);
        V.W = reinterpret_cast<int64_t*>(sm + L.oW);
        V.P = reinterpret_cast<uint16_t*>(sm + L.oP);
        V.dS = nullptr; V.dW = nullptr;
    } else {
        V.seg = ws.seg + c0;
        V.cnt = ws.cnt + c0;
        V.offS = ws.offS + c0;
        V.offW = ws.offW + c0;
        V.vb = nullptr;
        V.S = ws.slot_S; V.W = ws.slot_W; V.P = ws.slot_p;
        V.dS = ws.dS + c0; V.dW = ws.dW + c0;
    }
    if (tid < mg) {
        const int j = jb + tid;
        const ChunkMeta mt = ws.meta[c0 + j];
        const_cast<i128*>(V.offS)[j] = gS[tid];
        if (WEIGHTED) const_cast<i128*>(V.offW)[j] = gW[tid];
        if (SMEM) const_cast<int32_t*>(V.vb)[j] = gH[tid];
        V.seg[j] = make_int4(j, 0, mt.h - 1, 0);
        V.cnt[j] = 1;
    }
    __syncthreads();
    if constexpr (SMEM) {
        __shared__ int32_t s_lo0[kGroup];
        if (tid < mg) s_lo0[tid] = 0;
        __syncthreads();
        copy_vertices<WEIGHTED>(ws, c0, jb, je, V.vb, s_lo0 - jb, Hg,
                                const_cast<int64_t*>(V.S), const_cast<int64_t*>(V.W),
                                const_cast<uint16_t*>(V.P));
        __syncthreads();
    }
    merge_levels<WEIGHTED, SMEM, 2>(V, jb, je, 1);
    if constexpr (SMEM) {
        // the group's list back to the workspace
        const int n = V.cnt[jb];
        for (int k = tid; k < n; k += blockDim.x) ws.seg[c0 + jb + k] = V.seg[jb + k];
        if (tid == 0) ws.cnt[c0 + jb] = n;
    }
}

// ---------------------------------------------------------------------------
// Merge levels over flat vertex arrays in shared memory
// ---------------------------------------------------------------------------
// When a group's hull vertices fit in shared memory, each chunk hull becomes a
// contiguous array of its vertices there, with row coordinates formed once (S,
// and W for weights; unit weights: W is the point's index in the row) and a tag
// (chunk in the row << 13 | rank in the chunk's hull).  Neighbouring nodes
// share a point: the left node's last vertex is the right node's first (a
// chunk hull holds both its ends).  A merge keeps the left node's head and
// moves the right node's kept tail down behind it, which in shared memory is a
// few coalesced rounds of one warp; the segment lists of the paper's Section
// 3.3 avoid that copy where the vertices live in global memory.  The bridge is
// found by one warp in a few parallel steps instead of a walk (Lemma 4.2):
//
//   * if the chain is convex at the shared point s, s stays and nothing else
//     changes;
//   * otherwise the bridge joins L = the left node without s to R = the right
//     node without s.  For a vertex x of L, t(x) is its tangent point on R:
//     the first vertex of R that lies strictly below the segment from x to its
//     successor (R's last vertex always does), found by bisection.  The vertex
//     after x (s after L's last) lies strictly below the line from x to t(x)
//     for every x before the bridge's left end and for none from it on, so the
//     left end is the first x for which it does not; the lanes test 32 evenly
//     spaced vertices of the remaining range at once and a ballot narrows it
//     (one round for up to 32 candidates, two for up to 1,024).  The right end
//     is t of the left end.  Ties resolve as in the walks: the left end is the
//     leftmost and the right end the rightmost vertex on the bridge's line.
template <bool WEIGHTED>
struct FlatSm {
    i128* S;          // row coordinates
    i128* Wi;         // weighted rows: W
    int64_t* Wu;      // unit weights: the point's index in the row
    uint32_t* tag;    // chunk << 13 | rank
    unsigned long long* bst = nullptr;   // bridge-search counters
    __device__ __forceinline__ void get(int i, i128& W, i128& Sv) const {
        Sv = S[i];
        if constexpr (WEIGHTED) W = Wi[i]; else W = (i128)Wu[i];
    }
    __device__ __forceinline__ bool turn(int o, int a, int b) const {
        i128 Wo, So, Wa, Sa, Wb, Sb;
        get(o, Wo, So); get(a, Wa, Sa); get(b, Wb, Sb);
        return row_turn<WEIGHTED>(Wo, So, Wa, Sa, Wb, Sb);
    }
    // the same with o's coordinates already at hand
    __device__ __forceinline__ bool turn_from(i128 Wo, i128 So, int a, int b) const {
        i128 Wa, Sa, Wb, Sb;
        get(a, Wa, Sa); get(b, Wb, Sb);
        return row_turn<WEIGHTED>(Wo, So, Wa, Sa, Wb, Sb);
    }
};

constexpr int kFlatTagRank = 13;   // bits of the rank in a tag (C + 1 <= 2^13)

// Merge of the nodes A = [a0, a0 + na) and B = [b0, b0 + nb), b0 >= a0 + na,
// A's last vertex being B's first, by the 32 lanes of one warp.  The merged
// node is left at a0; returns its size (on every lane).
template <bool WEIGHTED>
__device__ int warp_merge(const FlatSm<WEIGHTED>& F, int a0, int na, int b0, int nb) {
    const int lane = threadIdx.x & 31;
    int keepA = na, fromB = 1;            // A[0 .. keepA) then B[fromB .. nb)
    if (!F.turn(a0 + na - 2, b0, b0 + 1)) {
        const int qR = nb - 1;            // R = B[1 .. nb)
        // the tangent point by bisection; on long right hulls first by
        // galloping from R's first vertex (bridges lie near the shared point
        // as a rule)
        auto tangent = [&](int x) -> int {
            i128 Wx, Sx;
            F.get(a0 + x, Wx, Sx);
            auto h = [&](int j) { return j >= qR - 1 || F.turn_from(Wx, Sx, b0 + 1 + j, b0 + 2 + j); };
            int jl = 0, jh = qR - 1;
            if (qR > 32) {
                if (h(0)) return 0;
                int step = 1;
                jl = 1;
                while (!h(jl + step - 1)) { jl += step; step <<= 1; }
                jh = min(jl + step - 1, qR - 1);
            }
            while (jl < jh) {
                const int mid = (jl + jh) >> 1;
                if (h(mid)) jh = mid; else jl = mid + 1;
            }
            return jl;
        };
        // the bridge's left end is in [lo, hi] of L = A[0 .. na-1); P(hi) is
        // false.  The first round tests the 32 vertices nearest the shared
        // point; when the first of them already fails, the left end lies at or
        // before it and 32-fold narrowing follows (8 rounds cover any list; the
        // range never empties).
        int lo = 0, hi = na - 2;
        {
            const int w0 = max(0, hi - 31);
            const int x = w0 + lane;
            bool nf = false;
            int t = 0;
            if (x <= hi) {
                t = tangent(x);
                nf = !F.turn(a0 + x, a0 + x + 1, b0 + 1 + t);
            }
            const unsigned bal = __ballot_sync(kFull, nf);
            if (!(bal & 1u) || w0 == 0) {
                // the window's first vertex passes (or the window is all of L):
                // the left end is the window's first failing vertex
                const int k = bal ? __ffs(bal) - 1 : hi - w0;
                keepA = w0 + k + 1;
                fromB = 1 + __shfl_sync(kFull, t, k);
                lo = hi + 1;                    // done
            } else {
                hi = w0;
            }
        }
        int round = 0;
        for (; round < ISO_BRIDGE_MAX_ROUNDS && lo <= hi; ++round) {
            const int n = hi - lo + 1;
            const int step = (n + 31) >> 5;
            const int x = lo + lane * step;
            bool nf = false;                    // "P(x) is false"
            int t = 0;
            if (x <= hi) {
                t = tangent(x);
                nf = !F.turn(a0 + x, a0 + x + 1, b0 + 1 + t);
            }
            const unsigned bal = __ballot_sync(kFull, nf);
            if (step == 1) {
                // every x in [lo, hi] tested; with exactly convex inputs some P is
                // false, else (inputs convex only up to rounding) the last one
                const int k = bal ? __ffs(bal) - 1 : hi - lo;
                keepA = lo + k + 1;
                fromB = 1 + __shfl_sync(kFull, t, k);
                lo = hi + 1;                    // done
                ++round;
                break;
            }
            if (bal == 0u) {
                const int kmax = (hi - lo) / step;        // last tested sample
                lo = min(lo + kmax * step + 1, hi);
            } else {
                const int k = __ffs(bal) - 1;
                hi = lo + k * step;
                lo = k == 0 ? hi : lo + (k - 1) * step + 1;
            }
        }
        if (F.bst && lane == 0) {
            atomicAdd(&F.bst[5], 1ull);
            atomicMax(&F.bst[6], (unsigned long long)round);
            if (lo <= hi) atomicAdd(&F.bst[7], 1ull);
        }
    }
    // the right node's kept tail moves down behind the left node's kept head
    // (dst < src): 32 U vertices per round, all read before any is written; a
    // round's writes lie below the next round's reads, so one barrier a round
    constexpr int U = WEIGHTED ? 2 : 4;
    const int len = nb - fromB, dst = a0 + keepA, src = b0 + fromB;
    if (dst != src) {
        for (int q = 0; q < len; q += 32 * U) {
            i128 sv[U], wv[U];
            int64_t wu[U];
            uint32_t tg[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = q + 32 * u + lane;
                if (k < len) {
                    sv[u] = F.S[src + k];
                    if constexpr (WEIGHTED) wv[u] = F.Wi[src + k]; else wu[u] = F.Wu[src + k];
                    tg[u] = F.tag[src + k];
                }
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = q + 32 * u + lane;
                if (k < len) {
                    F.S[dst + k] = sv[u];
                    if constexpr (WEIGHTED) F.Wi[dst + k] = wv[u]; else F.Wu[dst + k] = wu[u];
                    F.tag[dst + k] = tg[u];
                }
            }
        }
        __syncwarp();
    }
    return keepA + len;
}

// The ends of chunks 0..m-1 of a row (the first is chunk c0 of the
// workspace) from the row's root hull: n vertices at v0 of the flat arrays F,
// tags in chunk order.  Scratch after the root's tags: first[] (m + 1 ints)
// and the edge slopes (n doubles, 8-byte aligned), which the caller has
// checked fit.  kq: from the row's quanta to values.  Every thread of the CTA
// calls it, after the arrays before v0 + n are dead.
template <bool WEIGHTED>
__device__ __forceinline__ void flat_root_ends(const FlatSm<WEIGHTED>& F, int v0, int n, int64_t m,
                                               const LongWs& ws, int64_t c0, int kq) {
    // ends of every chunk from the root array R (tags in chunk order): first[j]
    // = the first root vertex of a chunk >= j, filled by each root vertex for
    // the chunks since its predecessor's (the nodes' arrays are dead now, so
    // first[] lives in the vertex arrays' space after R)
    const int tid = threadIdx.x, nth = blockDim.x;
    const uint32_t* tg = F.tag + v0;
    int32_t* first = reinterpret_cast<int32_t*>(F.tag + v0 + n);
    constexpr uint32_t kRank = (1u << kFlatTagRank) - 1u;
    for (int k = tid; k <= n; k += nth) {
        const int64_t jlo = k == 0 ? 0 : (int64_t)(tg[k - 1] >> kFlatTagRank) + 1;
        const int64_t jhi = k == n ? m : (int64_t)(tg[k] >> kFlatTagRank);
        for (int64_t j = jlo; j <= jhi && j <= m; ++j) first[j] = k;
    }
    // each root edge's slope once, after first[] (8-byte aligned)
    double* esl = reinterpret_cast<double*>((reinterpret_cast<uintptr_t>(first + m + 1) + 7) & ~(uintptr_t)7);
    for (int k = tid; k + 1 < n; k += nth) {
        i128 Wa, Sa, Wb, Sb;
        F.get(v0 + k, Wa, Sa);
        F.get(v0 + k + 1, Wb, Sb);
        esl[k] = edge_slope(Wa, Sa, Wb, Sb, kq);
    }
    __syncthreads();
    constexpr int C = LongCfg<WEIGHTED>::C;
    for (int64_t j = tid; j < m; j += nth) {
        const int lb = first[j], ub = first[j + 1];
        ChunkEnds ce;
        ce.bad = 0;
        if (lb < ub) { ce.lo = (int)(tg[lb] & kRank); ce.hi = (int)(tg[ub - 1] & kRank); }
        else { ce.lo = 1; ce.hi = 0; }
        ce.pt0_vertex = 0;
        // entering edge: from root vertex lb - 1 to lb (the chunk's first root
        // vertex, else the next); leaving edge: from ub - 1 to ub
        ce.in_sl = j > 0 ? esl[lb - 1] : 0.0;
        ce.out_sl = (lb < ub && j + 1 < m) ? esl[ub - 1] : 0.0;
        if (j > 0) {
            const int k = v0 + lb - 1;
            // the previous root vertex is this chunk's first point (it closes chunk j - 1)
            if constexpr (WEIGHTED) {
                const uint32_t t = F.tag[k];
                ce.pt0_vertex = ((int64_t)(t >> kFlatTagRank) == j - 1 &&
                                 (int)(t & kRank) == ws.meta[c0 + j - 1].h - 1) ? 1 : 0;
            } else {
                ce.pt0_vertex = F.Wu[k] == (int64_t)(j * C) ? 1 : 0;
            }
        }
        store_ends(ws, c0 + j, ce);
    }
}

// Shared-memory bytes of flat_root_ends' scratch past the root's tags.
__host__ __device__ inline size_t flat_root_scratch(int64_t m, int64_t n) {
    return 4 * (size_t)(m + 1) + 8 * (size_t)n + 8;
}

// Shared-memory layout of the flat group merge for mg chunks and H vertices.
struct FlatLayout {
    size_t oS, oW, oTag, oStart, oSize, bytes;
    __host__ __device__ FlatLayout(int64_t mg, int64_t H, bool weighted) {
        size_t o = 0;
        auto take = [&](size_t b, size_t al) { o = (o + al - 1) & ~(al - 1); const size_t r = o; o += b; return r; };
        oS = take(16 * H, 16);
        oW = take((weighted ? 16 : 8) * H, 16);
        oTag = take(4 * H, 4);
        oStart = take(4 * mg, 4);
        oSize = take(4 * mg, 4);
        bytes = o;
    }
};
constexpr int kFlatSmem = 96 * 1024;   // dynamic shared memory of the group kernel
constexpr int kMaxFlatGroups = 2 * kMergeThreads;   // groups of a row whose flat arrays the top merge reads

// The group's chunk hulls [jb, je) (Hg vertices; chunk starts gS/gW in row
// coordinates, vertex bases gH) merged by levels of warp merges over flat
// arrays; the group's root list is written to the workspace as segments, as
// the segment-list merges leave it.  Every thread of the CTA calls it.
template <bool WEIGHTED>
__device__ __forceinline__ void merge_group_flat(const LongWs& ws, int64_t c0, int jb, int je,
                                                 const i128* gS, const i128* gW,
                                                 const int32_t* gH, const int32_t* gDS,
                                                 const int32_t* gDW, int64_t Hg, int64_t g,
                                                 int64_t whole_row, int kq) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nth >> 5;
    const int mg = je - jb;
    const FlatLayout Lo(mg, Hg, WEIGHTED);
    unsigned char* sm = merge_smem;
    FlatSm<WEIGHTED> F;
    F.S = reinterpret_cast<i128*>(sm + Lo.oS);
    F.Wi = reinterpret_cast<i128*>(sm + Lo.oW);
    F.Wu = reinterpret_cast<int64_t*>(sm + Lo.oW);
    F.tag = reinterpret_cast<uint32_t*>(sm + Lo.oTag);
    F.bst = ws.bst;
    int32_t* nstart = reinterpret_cast<int32_t*>(sm + Lo.oStart);
    int32_t* nsize = reinterpret_cast<int32_t*>(sm + Lo.oSize);
    for (int j = tid; j < mg; j += nth) {
        nstart[j] = gH[j];
        nsize[j] = (j + 1 < mg ? gH[j + 1] : (int32_t)Hg) - gH[j];
    }
    // every vertex in row coordinates: its chunk by bisection over the bases
    // (four vertices per thread in flight: their slot loads are independent)
    for (int64_t i0 = tid; i0 < Hg; i0 += 4 * (int64_t)nth) {
        int jl[4], rr[4];
        int64_t sv[4], wv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = i0 + (int64_t)u * nth;
            jl[u] = -1; rr[u] = 0; sv[u] = 0; wv[u] = 0;
            if (i < Hg) {
                int lo = 0, hi = mg - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (gH[mid] <= i) lo = mid; else hi = mid - 1;
                }
                jl[u] = lo;
                rr[u] = (int)(i - gH[lo]);
                const size_t gi = (size_t)(c0 + jb + lo) * ((size_t)C + 1) + rr[u];
                sv[u] = ws.slot_S[gi];
                if constexpr (WEIGHTED) wv[u] = ws.slot_W[gi]; else wv[u] = ws.slot_p[gi];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (jl[u] < 0) continue;
            const int64_t i = i0 + (int64_t)u * nth;
            const int lo = jl[u], j = jb + lo;
            F.S[i] = gS[lo] + conv(sv[u], gDS[lo]);
            if constexpr (WEIGHTED) F.Wi[i] = gW[lo] + conv(wv[u], gDW[lo]);
            else F.Wu[i] = (int64_t)j * C + wv[u];
            F.tag[i] = ((uint32_t)j << kFlatTagRank) | (uint32_t)rr[u];
        }
    }
    __syncthreads();
    for (int half = 1; half < mg; half <<= 1) {
        for (int j = 2 * half * warp; j + half < mg; j += 2 * half * nw) {
            const int n = warp_merge<WEIGHTED>(F, nstart[j], nsize[j], nstart[j + half], nsize[j + half]);
            if (lane == 0) nsize[j] = n;
        }
        __syncthreads();
    }
    // the root list of the group as segments (chunk, first rank, last rank):
    // a segment starts at every vertex whose chunk differs from its predecessor's
    if (warp == 0) {
        const int n = nsize[0], v0 = nstart[0];
        int nseg = 0;
        for (int q = 0; q < n; q += 32) {
            const int k = q + lane;
            uint32_t tg = 0, tp = 0, tn = 0;
            if (k < n) {
                tg = F.tag[v0 + k];
                tp = k > 0 ? F.tag[v0 + k - 1] : ~0u;
                tn = k + 1 < n ? F.tag[v0 + k + 1] : ~0u;
            }
            const bool head = k < n && (tp >> kFlatTagRank) != (tg >> kFlatTagRank);
            const bool tail = k < n && (tn >> kFlatTagRank) != (tg >> kFlatTagRank);
            const unsigned hb = __ballot_sync(kFull, head);
            if (head) {
                // this segment's index; its last rank is found by the segment's tail lane
                const int idx = nseg + __popc(hb & ((1u << lane) - 1u));
                ws.seg[c0 + jb + idx].x = (int)(tg >> kFlatTagRank);
                ws.seg[c0 + jb + idx].y = (int)(tg & ((1u << kFlatTagRank) - 1u));
            }
            // a tail lane belongs to the segment of the last head at or before it
            const unsigned hb_upto = hb & (0xffffffffu >> (31 - lane));
            if (tail) {
                const int idx = nseg + __popc(hb_upto) - 1;
                ws.seg[c0 + jb + idx].z = (int)(tg & ((1u << kFlatTagRank) - 1u));
                ws.seg[c0 + jb + idx].w = 0;
            }
            nseg += __popc(hb);
        }
        if (lane == 0) ws.cnt[c0 + jb] = nseg;
    }
    // the merged hull as a flat array for the top merge, when it fits
    const int n = nsize[0], v0 = nstart[0];
    const bool keep = n <= kGroupFlatCap;
    if (tid == 0) ws.gfN[g] = keep ? n : -1;
    if (keep) {
        const size_t o = (size_t)g * kGroupFlatCap;
        for (int k = tid; k < n; k += nth) {
            ws.gfS[o + k] = F.S[v0 + k];
            if constexpr (WEIGHTED) reinterpret_cast<i128*>(ws.gfW)[o + k] = F.Wi[v0 + k];
            else reinterpret_cast<int64_t*>(ws.gfW)[o + k] = F.Wu[v0 + k];
            ws.gfTag[o + k] = F.tag[v0 + k];
        }
    }
    // a row of this one group: this hull is the row's root hull, and its chunk
    // ends are written here (the top kernel skips the row)
    if (whole_row >= 0) {
        const size_t used = (size_t)(reinterpret_cast<unsigned char*>(F.tag + v0 + n) - merge_smem);
        if (used + flat_root_scratch(mg, n) <= (size_t)kFlatSmem) {
            __syncthreads();              // the hull is written out and nsize, nstart read
            flat_root_ends<WEIGHTED>(F, v0, n, mg, ws, c0, kq);
            if (tid == 0) ws.rowq[whole_row * 4 + 3] = 1;
        }
    }
}

// One group of kGroup chunks: the row's quanta and status, the chunks' starts
// in row coordinates and their grid shifts, then (MERGE) the group's merges.
template <bool WEIGHTED, bool MERGE = true>
__device__ __forceinline__ void merge_group_one(const LongGeo& geo, int64_t ng, const LongWs& ws,
                                                uint32_t* __restrict__ row_status, int64_t g) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    __shared__ Acc3 s_scan[32];
    __shared__ int s_red[3];
    __shared__ i128 s_part[2][kGroupThreads / 32];
    __shared__ i128 s_gS[kGroup], s_gW[kGroup];
    __shared__ int32_t s_gH[kGroup];
    __shared__ int32_t s_gD[2][kGroup];
    __shared__ long long s_Hg;
    const int64_t row = geo.e0 ? (int64_t)geo.group_row[g] : g / ng;
    const RowRef R = geo_row<C>(geo, row);
    const int64_t m = R.m, c0 = R.c0;
    const int64_t gi = g - (geo.e0 ? geo.g0[row] : row * ng);
    const int jb = (int)gi * kGroup;
    const int je = (int)imin64(jb + kGroup, m);
    const int tid = threadIdx.x, nth = blockDim.x;
    // the row's chunk records, read once into the dynamic shared memory when they fit
    // (the merges below use it only after the offsets are done)
    constexpr int64_t kCacheBytes = MERGE ? kFlatSmem : kGroupSmem;
    ChunkMeta* mc = m * (int64_t)sizeof(ChunkMeta) <= kCacheBytes ? reinterpret_cast<ChunkMeta*>(merge_smem)
                                                                   : nullptr;
    const RowQ q = row_quanta(m, ws, c0, s_red, mc);
    if (gi == 0 && tid == 0) {
        ws.rowq[row * 4 + 0] = q.qs; ws.rowq[row * 4 + 1] = q.qw; ws.rowq[row * 4 + 2] = q.bad;
        ws.rowq[row * 4 + 3] = 0;       // set when this group also writes the row's ends
        if (row_status) row_status[R.id] = (uint32_t)q.bad;
    }
    if (q.bad) {
        for (int j = jb + tid; j < je; j += nth) {
            ChunkEnds ce{};
            ce.lo = 1; ce.hi = 0; ce.bad = q.bad;
            store_ends(ws, c0 + j, ce);
        }
        return;
    }
    // the group's start in row coordinates: the converted totals of the chunks before it
    {
        i128 aS = 0, aW = 0;
        // four chunks in flight per thread (the loads are independent)
        for (int64_t j0 = tid; j0 < jb; j0 += 4 * (int64_t)nth) {
            ChunkMeta m4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t j = j0 + (int64_t)u * nth;
                if (j < jb) m4[u] = mc ? mc[j] : ws.meta[c0 + j];
                else { m4[u].qs = q.qs; m4[u].qw = q.qw; m4[u].totS = 0; m4[u].totW = 0; }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                aS += conv(m4[u].totS, q.qs - m4[u].qs);
                aW += WEIGHTED ? (i128)conv(m4[u].totW, q.qw - m4[u].qw) : (i128)m4[u].totW;
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            aS += (i128)(((unsigned __int128)__shfl_xor_sync(kFull, (uint64_t)((unsigned __int128)aS >> 64), d) << 64) |
                         __shfl_xor_sync(kFull, (uint64_t)aS, d));
            aW += (i128)(((unsigned __int128)__shfl_xor_sync(kFull, (uint64_t)((unsigned __int128)aW >> 64), d) << 64) |
                         __shfl_xor_sync(kFull, (uint64_t)aW, d));
        }
        if ((tid & 31) == 0) { s_part[0][tid >> 5] = aS; s_part[1][tid >> 5] = aW; }
        __syncthreads();
        // the group's chunks: starts, shifts and vertex bases by a block scan
        i128 bS = 0, bW = 0;
        for (int w = 0; w < nth / 32; ++w) { bS += s_part[0][w]; bW += s_part[1][w]; }
        const int j = jb + tid;
        const bool valid = tid < kGroup && j < je;
        ChunkMeta mt{};
        if (valid) mt = mc ? mc[j] : ws.meta[c0 + j];
        const int ds = valid ? q.qs - mt.qs : 0;
        const int dw = (valid && WEIGHTED) ? q.qw - mt.qw : 0;
        Acc3 v;
        v.s = valid ? (i128)conv(mt.totS, ds) : (i128)0;
        v.w = valid ? (WEIGHTED ? (i128)conv(mt.totW, dw) : (i128)mt.totW) : (i128)0;
        v.h = valid ? mt.h : 0;
        Acc3 tot;
        const Acc3 e = block_excl_scan3(v, s_scan, tot);
        if (valid) {
            s_gS[tid] = bS + e.s;
            s_gW[tid] = bW + e.w;
            s_gH[tid] = (int32_t)e.h;
            ws.offS[c0 + j] = bS + e.s;
            if (WEIGHTED) ws.offW[c0 + j] = bW + e.w;
            ws.dS[c0 + j] = ds;
            if (WEIGHTED) ws.dW[c0 + j] = dw;
            s_gD[0][tid] = ds;
            s_gD[1][tid] = dw;
        }
        if (tid == 0) s_Hg = tot.h;
        __syncthreads();
    }
    if (!MERGE) return;
    const int64_t Hg = s_Hg;
    if (FlatLayout(je - jb, Hg, WEIGHTED).bytes <= (size_t)kFlatSmem) {
        merge_group_flat<WEIGHTED>(ws, c0, jb, je, s_gS, s_gW, s_gH, s_gD[0], s_gD[1], Hg, g,
                                   m == je - jb ? row : -1, q.qs - (WEIGHTED ? q.qw : 0));
        return;
    }
    if (tid == 0) ws.gfN[g] = -1;
    if (MergeLayout(je - jb, Hg, WEIGHTED, false).bytes <= (size_t)kGroupSmem)
        merge_group<WEIGHTED, true>(m, ws, c0, jb, je, s_gS, s_gW, s_gH, Hg);
    else
        merge_group<WEIGHTED, false>(m, ws, c0, jb, je, s_gS, s_gW, s_gH, Hg);
}

template <bool WEIGHTED, bool RAGGED, bool MERGE = true>
__global__ void __launch_bounds__(kGroupThreads)
merge_groups_kernel(LongGeo geo, int64_t ng, LongWs ws, uint32_t* __restrict__ row_status) {
    wait_prior_grid();
    launch_next_grid();   // the top merge's CTAs may take idle SMs now
    if (!RAGGED) {
        merge_group_one<WEIGHTED, MERGE>(geo, ng, ws, row_status, blockIdx.x);
        return;
    }
    const int64_t G = geo.count[2];
    for (int64_t g = blockIdx.x; g < G; g += gridDim.x) {
        merge_group_one<WEIGHTED>(geo, ng, ws, row_status, g);
        __syncthreads();
    }
}

// Ends: each chunk's root segment, and the root vertices around it, from the
// root list V.seg[0 .. V.cnt[0]) (at most one segment per chunk, in chunk
// order).  Every thread of the CTA calls it; segOf, nextSeg and prevSeg are
// scratch of m entries.
template <bool WEIGHTED, class View>
__device__ __forceinline__ void root_ends(const View& V, int64_t m, const LongWs& ws, int64_t c0,
                                          int32_t* segOf, int32_t* nextSeg, int32_t* prevSeg, int kq) {
    const int tid = threadIdx.x, nth = blockDim.x;
    // With c(j) the number of root segments of chunks <= j (a scan of "chunk j
    // holds one"), the first after chunk j is c(j) and the last before it is
    // c(j) - [j holds one] - 1.
    const int4* seg = V.seg;
    const int nroot = V.cnt[0];
    for (int64_t j = tid; j < m; j += nth) segOf[j] = -1;
    __syncthreads();
    for (int k = tid; k < nroot; k += nth) segOf[seg[k].x] = k;
    __syncthreads();
    {
        __shared__ int s_tmp2[32];
        const int64_t per2 = (m + nth - 1) / nth;
        const int64_t jb2 = imin64(m, tid * per2), je2 = imin64(m, jb2 + per2);
        int c = 0;
        for (int64_t j = jb2; j < je2; ++j) c += segOf[j] >= 0 ? 1 : 0;
        int tot2;
        c = block_excl_scan_int(c, s_tmp2, tot2);
        for (int64_t j = jb2; j < je2; ++j) {
            const int has = segOf[j] >= 0 ? 1 : 0;
            c += has;
            nextSeg[j] = c;                 // first root segment of a chunk > j
            prevSeg[j] = c - has - 1;       // last root segment of a chunk < j
        }
    }
    __syncthreads();
    for (int64_t j = tid; j < m; j += nth) {
        ChunkEnds ce;
        ce.bad = 0;
        const int sk = segOf[j];
        Seg gs{};
        if (sk >= 0) { gs = V.load(sk); ce.lo = gs.lo; ce.hi = gs.hi; }
        else { ce.lo = 1; ce.hi = 0; }
        ce.in_sl = ce.out_sl = 0.0;
        ce.pt0_vertex = 0;
        i128 Wn = 0, Sn = 0;
        if (j + 1 < m) {
            const Seg gn = V.load(nextSeg[j]);
            V.at(gn, gn.lo, Wn, Sn);
        }
        if (j > 0) {
            const int pk = prevSeg[j];
            const Seg gp = V.load(pk);
            i128 Wp, Sp, Wb = Wn, Sb = Sn;
            V.at(gp, gp.hi, Wp, Sp);
            // the previous root vertex is this chunk's first point when it closes chunk j-1
            ce.pt0_vertex = (gp.jc == j - 1 && gp.hi == ws.meta[c0 + gp.jc].h - 1) ? 1 : 0;
            // the entering edge ends at the chunk's first root vertex, else at the next one
            if (sk >= 0) V.at(gs, gs.lo, Wb, Sb);
            ce.in_sl = edge_slope(Wp, Sp, Wb, Sb, kq);
        }
        if (sk >= 0 && j + 1 < m) {
            i128 Wa, Sa;
            V.at(gs, gs.hi, Wa, Sa);
            ce.out_sl = edge_slope(Wa, Sa, Wn, Sn, kq);
        }
        store_ends(ws, c0 + j, ce);
    }
}

template <bool WEIGHTED, bool SMEM>
__device__ __forceinline__ void merge_top(int64_t m, const LongWs& ws, int64_t c0, int64_t Hs,
                                          int32_t* s_len, int32_t* s_lo, int kq) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int tid = threadIdx.x, nth = blockDim.x;
    MergeLayout L(m, SMEM ? Hs : 0, WEIGHTED, true);
    unsigned char* sm = merge_smem;
    MView<WEIGHTED, SMEM> V;
    V.c0 = c0;
    V.C = C;
    V.bst = ws.bst;
    V.bmax = ws.bmax;
    int32_t *segOf, *nextSeg, *prevSeg;
    if constexpr (SMEM) {
        V.seg = reinterpret_cast<int4*>(sm + L.oSeg);
        V.cnt = reinterpret_cast<int32_t*>(sm + L.oCnt);
        V.offS = reinterpret_cast<i128*>(sm + L.oOffS);
        V.offW = reinterpret_cast<i128*>(sm + L.oOffW);
        V.vb = reinterpret_cast<int32_t*>(sm + L.oVb);
        V.S = reinterpret_cast<int64_t*>(sm + L.oS);
        V.W = reinterpret_cast<int64_t*>(sm + L.oW);
        V.P = reinterpret_cast<uint16_t*>(sm + L.oP);
        V.dS = nullptr; V.dW = nullptr;
        segOf = reinterpret_cast<int32_t*>(sm + L.oSegOf);
        nextSeg = reinterpret_cast<int32_t*>(sm + L.oNext);
        prevSeg = reinterpret_cast<int32_t*>(sm + L.oPrev);
        // chunk starts, and the lists of the groups
        for (int64_t j = tid; j < m; j += nth) {
            const_cast<i128*>(V.offS)[j] = ws.offS[c0 + j];
            if (WEIGHTED) const_cast<i128*>(V.offW)[j] = ws.offW[c0 + j];
            V.seg[j] = ws.seg[c0 + j];
            V.cnt[j] = ws.cnt[c0 + j];
        }
        // vertex bases (s_len: the surviving segments' lengths scanned in chunk
        // order) and first ranks (s_lo), staged in the ends scratch; vertex
        // (jc, r) then lives at vb[jc] + r
        for (int64_t j = tid; j < m; j += nth) { segOf[j] = s_len[j]; prevSeg[j] = s_lo[j]; }
        __syncthreads();
        copy_vertices<WEIGHTED>(ws, c0, 0, (int)m, segOf, prevSeg, Hs, const_cast<int64_t*>(V.S),
                                const_cast<int64_t*>(V.W), const_cast<uint16_t*>(V.P));
        for (int64_t j = tid; j < m; j += nth)
            const_cast<int32_t*>(V.vb)[j] = segOf[j] - prevSeg[j];
        __syncthreads();
    } else {
        V.seg = ws.seg + c0;
        V.cnt = ws.cnt + c0;
        V.offS = ws.offS + c0;
        V.offW = ws.offW + c0;
        V.vb = nullptr;
        V.S = ws.slot_S; V.W = ws.slot_W; V.P = ws.slot_p;
        V.dS = ws.dS + c0; V.dW = ws.dW + c0;
        segOf = ws.segOf + c0;
        nextSeg = ws.nextSeg + c0;
        prevSeg = ws.prevSeg + c0;
    }
    merge_levels<WEIGHTED, SMEM>(V, 0, m, kGroup);

    root_ends<WEIGHTED>(V, m, ws, c0, segOf, nextSeg, prevSeg, kq);
}

// The top of the tree over the groups' flat arrays (every group of the row
// kept one, and they fit in shared memory together): the arrays are read as
// the tree's nodes, merged by the warp merges of the group kernel, and each
// chunk's root range and the root vertices around it are found by bisection
// over the root array's tags (Section 3.4, Corollary 4.5).  A root vertex on
// a chunk boundary is tagged with the chunk it ends, as in the segment lists.
template <bool WEIGHTED>
__device__ __forceinline__ void merge_top_flat(const LongWs& ws, int64_t c0, int64_t m, int64_t gb,
                                               int ng, int H, const int32_t* gbase, int kq) {
    const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nth >> 5;
    const FlatLayout Lo(ng, H, WEIGHTED);
    unsigned char* sm = merge_smem;
    FlatSm<WEIGHTED> F;
    F.S = reinterpret_cast<i128*>(sm + Lo.oS);
    F.Wi = reinterpret_cast<i128*>(sm + Lo.oW);
    F.Wu = reinterpret_cast<int64_t*>(sm + Lo.oW);
    F.tag = reinterpret_cast<uint32_t*>(sm + Lo.oTag);
    F.bst = ws.bst;
    int32_t* nstart = reinterpret_cast<int32_t*>(sm + Lo.oStart);
    int32_t* nsize = reinterpret_cast<int32_t*>(sm + Lo.oSize);
    for (int k = tid; k < ng; k += nth) {
        nstart[k] = gbase[k];
        nsize[k] = (k + 1 < ng ? gbase[k + 1] : H) - gbase[k];
    }
    // every vertex at once: its group by bisection over the bases (the last
    // group whose base is at or before it: empty groups are passed over)
    for (int i = tid; i < H; i += nth) {
        int lo = 0, hi = ng - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gbase[mid] <= i) lo = mid; else hi = mid - 1;
        }
        const size_t o = (size_t)(gb + lo) * kGroupFlatCap + (size_t)(i - gbase[lo]);
        F.S[i] = ws.gfS[o];
        if constexpr (WEIGHTED) F.Wi[i] = reinterpret_cast<const i128*>(ws.gfW)[o];
        else F.Wu[i] = reinterpret_cast<const int64_t*>(ws.gfW)[o];
        F.tag[i] = ws.gfTag[o];
    }
    __syncthreads();
    for (int half = 1; half < ng; half <<= 1) {
        for (int k = 2 * half * warp; k + half < ng; k += 2 * half * nw) {
            const int n = warp_merge<WEIGHTED>(F, nstart[k], nsize[k], nstart[k + half], nsize[k + half]);
            if (lane == 0) nsize[k] = n;
        }
        __syncthreads();
    }
    const int n = nsize[0], v0 = nstart[0];
    __syncthreads();                       // nsize and nstart are read: first[] may cover them
    flat_root_ends<WEIGHTED>(F, v0, n, m, ws, c0, kq);
}

template <bool WEIGHTED>
__device__ __forceinline__ void merge_top_row(const LongGeo& geo, const LongWs& ws, int64_t row) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const RowRef R = geo_row<C>(geo, row);
    const int64_t m = R.m, c0 = R.c0;
    const int tid = threadIdx.x, nth = blockDim.x;
    // every group of the row kept a flat array and they fit: the flat top
    const int64_t ng = (m + kGroup - 1) / kGroup;
    const int64_t gb = geo.e0 ? geo.g0[row] : row * ng;
    // the groups' sizes are read with the row's status (a bad row's are unused)
    const int k0 = 2 * tid, k1 = 2 * tid + 1;
    const bool flat_ok = ng <= kMaxFlatGroups;
    const int c0n = flat_ok && k0 < ng ? ws.gfN[gb + k0] : 0;
    const int c1n = flat_ok && k1 < ng ? ws.gfN[gb + k1] : 0;
    // a bad row, or a row of one group: its ends are written
    if (ws.rowq[row * 4 + 2] || ws.rowq[row * 4 + 3]) return;
    // root edge slopes: from the row's quanta to values
    const int kq = ws.rowq[row * 4 + 0] - (WEIGHTED ? ws.rowq[row * 4 + 1] : 0);
    {
        __shared__ int32_t s_gbase[kMaxFlatGroups];
        __shared__ int s_scan2[32];
        if (flat_ok) {
            // bases by a block scan (ng <= blockDim.x * 2)
            const bool ok = __syncthreads_and(c0n >= 0 && c1n >= 0);
            int tot;
            const int b = block_excl_scan_int(c0n + c1n, s_scan2, tot);
            if (k0 < ng) s_gbase[k0] = b;
            if (k1 < ng) s_gbase[k1] = b + c0n;
            __syncthreads();
            if (ok && FlatLayout(ng, tot, WEIGHTED).bytes + flat_root_scratch(m, tot) <= (size_t)kMergeSmem) {
                merge_top_flat<WEIGHTED>(ws, c0, m, gb, (int)ng, tot, s_gbase, kq);
                return;
            }
        }
    }
    // the chunks' surviving segments (each chunk in at most one): lengths into
    // segOf, first ranks into prevSeg (scratch), then bases by a scan
    int32_t* len = ws.segOf + c0;
    int32_t* lo0 = ws.prevSeg + c0;
    for (int64_t j = tid; j < m; j += nth) { len[j] = 0; lo0[j] = 0; }
    __syncthreads();
    for (int64_t g = (int64_t)(tid >> 5) * kGroup; g < m; g += (int64_t)(nth >> 5) * kGroup) {
        const int n = ws.cnt[c0 + g];
        for (int k = tid & 31; k < n; k += 32) {
            const int4 sg = ws.seg[c0 + g + k];
            len[sg.x] = sg.z - sg.y + 1;
            lo0[sg.x] = sg.y;
        }
    }
    __syncthreads();
    // bases: each thread scans a contiguous range of chunks
    __shared__ int s_tmp[32];
    const int64_t per = (m + nth - 1) / nth;
    const int64_t jb = imin64(m, tid * per), je = imin64(m, jb + per);
    int sum = 0;
    for (int64_t j = jb; j < je; ++j) sum += len[j];
    int total;
    int base = block_excl_scan_int(sum, s_tmp, total);
    for (int64_t j = jb; j < je; ++j) {
        const int l = len[j];
        len[j] = base;                                     // now the base of chunk j
        base += l;
    }
    __syncthreads();
    const int64_t Hs = total;
    if (MergeLayout(m, Hs, WEIGHTED, true).bytes <= (size_t)kMergeSmem)
        merge_top<WEIGHTED, true>(m, ws, c0, Hs, len, lo0, kq);
    else
        merge_top<WEIGHTED, false>(m, ws, c0, Hs, len, lo0, kq);
}

template <bool WEIGHTED, bool RAGGED>
__global__ void __launch_bounds__(kMergeThreads, 1)
merge_top_kernel(LongGeo geo, LongWs ws) {
    wait_prior_grid();
    launch_next_grid();   // the expansion's CTAs may take idle SMs now
    if (!RAGGED) {
        merge_top_row<WEIGHTED>(geo, ws, blockIdx.x);
        return;
    }
    const int64_t rows = geo.count[0];
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        merge_top_row<WEIGHTED>(geo, ws, row);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// 3. expansion: each element gets the slope of the root-hull edge above it
// ---------------------------------------------------------------------------
template <bool WEIGHTED, class IO = float>
struct ExpandSmem {
    static constexpr int NT = LongCfg<WEIGHTED>::NT;
    static constexpr int C = LongCfg<WEIGHTED>::C;
    static constexpr int oMask = 0;
    static constexpr int oTmp = oMask + NT * 4;
    static constexpr int oSlope = ((oTmp + (NT / 32 + 2) * 8 + 15) / 16) * 16;   // 16-byte rows
    static constexpr int kBytes = oSlope + C * (int)sizeof(IO);
};

template <bool WEIGHTED, class IO>
__device__ __forceinline__ void expand_one(const IO* __restrict__ y, const LongGeo& geo,
                                           int increasing, const LongWs& ws,
                                           IO* __restrict__ out, uint8_t* __restrict__ blocks,
                                           int64_t c) {
    constexpr int NT = LongCfg<WEIGHTED>::NT;
    constexpr int C = LongCfg<WEIGHTED>::C;
    using XS = ExpandSmem<WEIGHTED, IO>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + XS::oMask);
    int64_t* s_tmp = reinterpret_cast<int64_t*>(smem + XS::oTmp);
    __shared__ IO s_in_sl;                                         // slope of the entering edge
    IO* slope = reinterpret_cast<IO*>(smem + XS::oSlope);   // per point, swizzled rows

    const int64_t row = geo.e0 ? (int64_t)geo.chunk_row[c] : c / geo.m;
    const RowRef R = geo_row<C>(geo, row);
    const int64_t e0 = (c - R.c0) * C;
    const int nt = (int)imin64(C, R.n - e0);
    const int tid = threadIdx.x;
    const ChunkEnds ce = load_ends(ws, c);
    IO* orow = out + R.e0 + e0;
    uint8_t* brow = blocks ? blocks + R.e0 + e0 : nullptr;
    const bool neg = !increasing;

    if (ce.bad) {
        // a rejected row: NaN fit; its block flags are 0, but a ragged
        // segment keeps its first element a block start
        const IO qnan = qnan_t<IO>();
        const bool mark0 = geo.e0 && e0 == 0;
        for (int i = tid; i < nt; i += NT) {
            orow[i] = qnan;
            if (brow) brow[i] = (mark0 && i == 0) ? 1 : 0;
        }
        return;
    }
    const size_t cap = (size_t)C + 1;
    const uint16_t* sp = ws.slot_p + c * cap;
    const int64_t* sS = ws.slot_S + c * cap;
    const int64_t* sW = WEIGHTED ? ws.slot_W + c * cap : nullptr;
    // Every point of the chunk a root vertex (a dense hull): every element is a
    // one-element block, fitted by its own value (an edge's slope is its
    // element's mean; for a decreasing fit the negations cancel).
    if (ce.lo <= ce.hi && ce.hi - ce.lo + sp[ce.lo] == nt && sp[ce.hi] == nt &&
        (sp[ce.lo] == 0 || (sp[ce.lo] == 1 && ce.pt0_vertex))) {
        const IO* yrow = y + R.e0 + e0;
        if ((reinterpret_cast<uintptr_t>(yrow) & 15u) == 0 &&
            (reinterpret_cast<uintptr_t>(orow) & 15u) == 0) {
            using V = typename IoT<IO>::V;
            constexpr int P = IoT<IO>::kPerV;
            const int nv = nt / P;
            for (int i = tid; i < nv; i += NT)
                reinterpret_cast<V*>(orow)[i] = __ldg(reinterpret_cast<const V*>(yrow) + i);
            for (int i = nv * P + tid; i < nt; i += NT) orow[i] = __ldg(yrow + i);
        } else {
            for (int i = tid; i < nt; i += NT) orow[i] = __ldg(yrow + i);
        }
        if (brow) {
            if ((reinterpret_cast<uintptr_t>(brow) & 3u) == 0) {
                const int n4 = nt >> 2;
                for (int i = tid; i < n4; i += NT) reinterpret_cast<uint32_t*>(brow)[i] = 0x01010101u;
                for (int i = (n4 << 2) + tid; i < nt; i += NT) brow[i] = 1;
            } else {
                for (int i = tid; i < nt; i += NT) brow[i] = 1;
            }
        }
        return;
    }
    const ChunkMeta mt = ws.meta[c];

    const int cexp = mt.qs - (WEIGHTED ? mt.qw : 0);   // chunk quanta to values
    s_mask[tid] = 0u;
    __syncthreads();
    // root vertices of this chunk that start one of its elements (point < nt),
    // each with the slope of the root edge leaving it
    const bool has = ce.lo <= ce.hi;
    if (has) {
        for (int r0 = ce.lo; r0 <= ce.hi; r0 += NT) {
            const int r = r0 + tid;
            const int p = r <= ce.hi ? sp[r] : nt;
            // the warp's start bits, one atomic per distinct mask word
            const int word = p < nt ? p >> 5 : -1;
            const unsigned grp = __match_any_sync(kFull, word);
            const unsigned bits = __reduce_or_sync(grp, p < nt ? 1u << (p & 31) : 0u);
            if (word >= 0 && (tid & 31) == __ffs(grp) - 1) atomicOr(&s_mask[word], bits);
            if (p >= nt) continue;
            IO sl;
            if (r < ce.hi) {
                // both ends in the chunk: chunk-relative coordinates, chunk quanta
                const int64_t dS_ = sS[r + 1] - sS[r];
                const int64_t dW_ = WEIGHTED ? sW[r + 1] - sW[r] : (int64_t)(sp[r + 1] - p);
                sl = ratio_t<IO>(dS_, dW_, cexp);
            } else {
                sl = (IO)ce.out_sl;                       // the edge to the next root vertex
            }
            slope[spos_t<IO>(p >> 5, p & 31)] = sl;
        }
    }
    if (tid == 0) {
        // the edge entering the chunk: from the previous root vertex to the first
        // root vertex of the chunk, or to the next root vertex if the chunk has none
        const IO in_sl = e0 > 0 ? (IO)ce.in_sl : IO(0);
        if (ce.pt0_vertex) {
            atomicOr(&s_mask[0], 1u);
            slope[spos_t<IO>(0, 0)] = in_sl;
        }
        s_in_sl = in_sl;
    }
    __syncthreads();
    // the last vertex before each lane: exclusive max-scan of the lanes' last vertices
    const uint32_t mk = s_mask[tid];
    int lastv;
    {
        int v = mk ? (tid << 5) + 31 - __clz(mk) : -1;
        const int wl = tid & 31;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o2 = __shfl_up_sync(kFull, v, d);
            if (wl >= d) v = max(v, o2);
        }
        int* wmax = reinterpret_cast<int*>(s_tmp);
        if (wl == 31) wmax[tid >> 5] = v;
        __syncthreads();
        int before = __shfl_up_sync(kFull, v, 1);
        if (wl == 0) before = -1;
        for (int q = 0; q < (tid >> 5); ++q) before = max(before, wmax[q]);
        lastv = before;
    }
    const IO in_sl = s_in_sl;
    const IO carry = lastv >= 0 ? slope[spos_t<IO>(lastv >> 5, lastv & 31)] : in_sl;
    IO o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const uint32_t upto = k == 31 ? mk : (mk & ((2u << k) - 1u));
        const IO v = upto ? slope[spos_t<IO>(tid, 31 - __clz(upto))] : carry;
        o[k] = neg ? -v : v;
    }
    __syncthreads();   // slopes read: stage the output in their place
    stage_out<IO>(slope, tid, o);
    __syncthreads();
    write_row<IO>(orow, slope, 0, nt, tid, NT, true);
    if (brow) {
        if ((reinterpret_cast<uintptr_t>(brow) & 3u) == 0) {
            const int n4 = nt >> 2;
            for (int i = tid; i < n4; i += NT) {
                const int e4 = i << 2;
                const uint32_t bits = (s_mask[e4 >> 5] >> (e4 & 31)) & 0xfu;
                reinterpret_cast<uint32_t*>(brow)[i] =
                    (bits & 1u) | ((bits & 2u) << 7) | ((bits & 4u) << 14) | ((bits & 8u) << 21);
            }
            for (int i = (n4 << 2) + tid; i < nt; i += NT)
                brow[i] = (uint8_t)((s_mask[i >> 5] >> (i & 31)) & 1u);
        } else {
            for (int i = tid; i < nt; i += NT) brow[i] = (uint8_t)((s_mask[i >> 5] >> (i & 31)) & 1u);
        }
    }
}

template <bool WEIGHTED, bool RAGGED, class IO>
__global__ void __launch_bounds__(LongCfg<WEIGHTED>::NT)
expand_kernel(const IO* __restrict__ y, LongGeo geo, int increasing, LongWs ws,
              IO* __restrict__ out, uint8_t* __restrict__ blocks) {
    wait_prior_grid();
    if (!RAGGED) {
        expand_one<WEIGHTED, IO>(y, geo, increasing, ws, out, blocks, blockIdx.x);
        return;
    }
    const int64_t M = geo.count[1];
    for (int64_t c = blockIdx.x; c < M; c += gridDim.x) {
        expand_one<WEIGHTED, IO>(y, geo, increasing, ws, out, blocks, c);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// 4. ragged batches: the long segments' tables
// ---------------------------------------------------------------------------
// Per-row tables of the long segments of a ragged batch, then the chunk and
// group maps.  One CTA: the long segments are listed (in any order) by the
// classification kernel, at most total / (kRowMax + 1) of them, and their
// chunks and groups fit the bounds the grids were sized for.  (Only
// overlapping segments, which the offsets' checks let through when a rejected
// segment lies between them, could exceed the bounds: the rows past the
// bounds are then rejected with ISO_ROW_BAD_SHAPE.)
template <int C>
__global__ void __launch_bounds__(1024)
long_plan_kernel(const int64_t* __restrict__ off, const int32_t* __restrict__ long_id,
                 const unsigned long long* __restrict__ nlong, int64_t rows_cap,
                 int64_t chunks_cap, int64_t groups_cap, LongGeo geo,
                 uint32_t* __restrict__ row_status) {
    __shared__ Acc3 s_scan[32];
    __shared__ unsigned long long s_keep;
    const int tid = threadIdx.x, nth = blockDim.x;
    int64_t nL = (int64_t)min((unsigned long long)rows_cap, *nlong);
    if (tid == 0) s_keep = (unsigned long long)nL;
    int64_t* e0 = const_cast<int64_t*>(geo.e0);
    int64_t* len = const_cast<int64_t*>(geo.len);
    int64_t* c0 = const_cast<int64_t*>(geo.c0);
    int64_t* g0 = const_cast<int64_t*>(geo.g0);
    int32_t* id = const_cast<int32_t*>(geo.id);
    int64_t carryC = 0, carryG = 0;
    for (int64_t b = 0; b < nL; b += nth) {
        const int64_t r = b + tid;
        Acc3 v{0, 0, 0};
        if (r < nL) {
            const int32_t s = long_id[r];
            const int64_t a = off[s], n = off[s + 1] - a;
            const int64_t m = (n + C - 1) / C;
            e0[r] = a; len[r] = n; id[r] = s;
            v.s = m; v.w = (m + kGroup - 1) / kGroup;
        }
        Acc3 tot;
        const Acc3 e = block_excl_scan3(v, s_scan, tot);
        if (r < nL) {
            c0[r] = carryC + (int64_t)e.s;
            g0[r] = carryG + (int64_t)e.w;
            if (c0[r] + (int64_t)v.s > chunks_cap || g0[r] + (int64_t)v.w > groups_cap)
                atomicMin(&s_keep, (unsigned long long)r);
        }
        carryC += (int64_t)tot.s;
        carryG += (int64_t)tot.w;
    }
    __syncthreads();   // the tables are written
    const int64_t keep = (int64_t)s_keep;
    for (int64_t r = keep + tid; r < nL; r += nth)
        if (row_status) row_status[id[r]] = ISO_ROW_BAD_SHAPE;
    nL = keep;
    if (tid == 0) {
        int64_t* cnt = const_cast<int64_t*>(geo.count);
        cnt[0] = nL;
        cnt[1] = nL > 0 ? c0[nL - 1] + (len[nL - 1] + C - 1) / C : 0;
        cnt[2] = nL > 0 ? g0[nL - 1] + ((len[nL - 1] + C - 1) / C + kGroup - 1) / kGroup : 0;
    }
    // fill the maps, one warp per row
    int32_t* crow = const_cast<int32_t*>(geo.chunk_row);
    int32_t* grow = const_cast<int32_t*>(geo.group_row);
    for (int64_t r = tid >> 5; r < nL; r += nth >> 5) {
        const int64_t m = (len[r] + C - 1) / C, gm = (m + kGroup - 1) / kGroup;
        for (int64_t k = tid & 31; k < m; k += 32) crow[c0[r] + k] = (int32_t)r;
        for (int64_t k = tid & 31; k < gm; k += 32) grow[g0[r] + k] = (int32_t)r;
    }
}

// ---------------------------------------------------------------------------
// 5. materialised-copy control (the paper's Section 7.3, "grid copying")
// ---------------------------------------------------------------------------
// The same chunk hulls, bridge search (merge_plan) and merge schedule as the
// segment lists, but every node of the tree is one contiguous array of
// vertices: after each level's bridges are found, a grid-wide kernel copies
// every merged hull's surviving vertices into the other buffer.  A vertex
// record holds S (and W) on its chunk's grid and a tag, chunk << 32 | rank in
// the chunk's hull << 16 | point index, since a copied vertex leaves its
// chunk's slot.  The root array is turned back into the root list of chunk
// segments, so the ends and the expansion are those of the segment lists and
// the results are identical; only the cost of the merge levels differs.
struct CtlWs {
    int64_t* fS[2];      // [M][C+1] per buffer; a row's region starts at its c0 * (C+1)
    int64_t* fW[2];      // weighted
    uint64_t* tag[2];
    int32_t* base[2];    // [M] node base within the row's region, by the node's first chunk
    int32_t* size[2];    // [M] node vertices
    int4* desc;          // [M] a merged node's sources: (left start, count, right start, count)
    int32_t* runLo;      // [M] first root rank of each chunk, -1 if none
    int32_t* runHi;      // [M]
    int32_t* rowH;       // [rows] vertices of the row at the current level
};

template <bool WEIGHTED>
__host__ __device__ inline size_t carve_ctl(void* base, int64_t rows, int64_t M, CtlWs* cw) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const size_t V = (size_t)M * ((size_t)C + 1);
    size_t off = 0;
    char* b = static_cast<char*>(base);
    auto take = [&](size_t bytes) -> void* {
        void* p = b ? (void*)(b + off) : nullptr;
        off += align256(bytes);
        return p;
    };
    CtlWs w;
    for (int k = 0; k < 2; ++k) {
        w.fS[k] = (int64_t*)take(8 * V);
        w.fW[k] = WEIGHTED ? (int64_t*)take(8 * V) : nullptr;
        w.tag[k] = (uint64_t*)take(8 * V);
        w.base[k] = (int32_t*)take(4 * M);
        w.size[k] = (int32_t*)take(4 * M);
    }
    w.desc = (int4*)take(16 * M);
    w.runLo = (int32_t*)take(4 * M);
    w.runHi = (int32_t*)take(4 * M);
    w.rowH = (int32_t*)take(4 * rows);
    if (cw) *cw = w;
    return off;
}

// merge_plan's view of one level's flat arrays: node j (its first chunk) is
// the single segment (j, lo, hi) of seg[j], over ranks of its array.
template <bool WEIGHTED>
struct FlatView {
    int4* seg;
    int32_t* cnt;
    const int32_t* base;
    const int64_t* S;
    const int64_t* W;
    const uint64_t* tag;
    const i128* offS;
    const i128* offW;
    const int32_t* dS;
    const int32_t* dW;
    int C;
    unsigned long long* bst = nullptr;   // bridge-search counters
    int bmax = ISO_BRIDGE_MAX_PASSES;

    __device__ __forceinline__ Seg load(int k) const {
        const int4 s = seg[k];
        Seg g;
        g.jc = s.x; g.lo = s.y; g.hi = s.z;
        g.vb = base[s.x];
        g.dS = 0; g.dW = 0;
        g.oS = 0; g.oW = 0;
        return g;
    }
    __device__ __forceinline__ void at(const Seg& g, int r, i128& Wv, i128& Sv) const {
        const int64_t i = (int64_t)g.vb + r;
        const uint64_t t = tag[i];
        const int ch = (int)(t >> 32);
        Sv = offS[ch] + conv(S[i], dS[ch]);
        if constexpr (WEIGHTED) Wv = offW[ch] + conv(W[i], dW[ch]);
        else Wv = (i128)((int64_t)ch * C + (int)(t & 0xffffu));
    }
};

__device__ __forceinline__ bool ctl_bad(const LongWs& ws, int64_t row) { return ws.rowq[row * 4 + 2] != 0; }

// Level 0: every chunk hull is a node; bases by a scan of the hull sizes.
// One CTA per row.
template <bool WEIGHTED>
__global__ void __launch_bounds__(kMergeThreads)
ctl_base_kernel(int64_t m, LongWs ws, CtlWs cw) {
    __shared__ int s_tmp[32];
    const int64_t row = blockIdx.x, c0 = row * m;
    if (ctl_bad(ws, row)) return;
    const int tid = threadIdx.x, nth = blockDim.x;
    const int64_t per = (m + nth - 1) / nth;
    const int64_t jb = imin64(m, tid * per), je = imin64(m, jb + per);
    int sum = 0;
    for (int64_t j = jb; j < je; ++j) sum += ws.meta[c0 + j].h;
    int total;
    int b = block_excl_scan_int(sum, s_tmp, total);
    for (int64_t j = jb; j < je; ++j) {
        const int h = ws.meta[c0 + j].h;
        cw.base[0][c0 + j] = b;
        cw.size[0][c0 + j] = h;
        ws.seg[c0 + j] = make_int4((int)j, 0, h - 1, 0);
        ws.cnt[c0 + j] = 1;
        cw.runLo[c0 + j] = -1;
        b += h;
    }
    if (tid == 0) cw.rowH[row] = total;
}

// Level 0: each chunk's slot copied into the flat array, every vertex tagged.
template <bool WEIGHTED>
__global__ void __launch_bounds__(128)
ctl_flatten_kernel(int64_t m, LongWs ws, CtlWs cw) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int64_t c = blockIdx.x, row = c / m, j = c - row * m, c0 = row * m;
    if (ctl_bad(ws, row)) return;
    const int h = ws.meta[c].h;
    const size_t cap = (size_t)C + 1;
    const size_t d = (size_t)c0 * cap + (size_t)cw.base[0][c];
    for (int r = threadIdx.x; r < h; r += blockDim.x) {
        const size_t s = (size_t)c * cap + r;
        cw.fS[0][d + r] = ws.slot_S[s];
        if constexpr (WEIGHTED) cw.fW[0][d + r] = ws.slot_W[s];
        cw.tag[0][d + r] = ((uint64_t)j << 32) | ((uint64_t)r << 16) | ws.slot_p[s];
    }
}

// One level's bridges: one thread per merge of nodes j0 = 2 k half and
// j1 = j0 + half (the paper's first control kernel).
template <bool WEIGHTED>
__global__ void __launch_bounds__(128)
ctl_bridge_kernel(int64_t m, int64_t half, int64_t nmerge, LongWs ws, CtlWs cw, int cur) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int64_t row = blockIdx.y, c0 = row * m;
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= nmerge || ctl_bad(ws, row)) return;
    const size_t R = (size_t)c0 * ((size_t)C + 1);
    FlatView<WEIGHTED> V;
    V.seg = ws.seg + c0;
    V.cnt = ws.cnt + c0;
    V.base = cw.base[cur] + c0;
    V.S = cw.fS[cur] + R;
    V.W = WEIGHTED ? cw.fW[cur] + R : nullptr;
    V.tag = cw.tag[cur] + R;
    V.offS = ws.offS + c0;
    V.offW = ws.offW + c0;
    V.dS = ws.dS + c0;
    V.dW = ws.dW + c0;
    V.C = C;
    V.bst = ws.bst;
    V.bmax = ws.bmax;
    const int64_t j0 = 2 * k * half;
    merge_plan<WEIGHTED>(V, (int)j0, (int)(j0 + half));
}

// One level's layout: each merged node's sources and size, bases by a scan,
// and the nodes' single segments for the next level.  One CTA per row.
__global__ void __launch_bounds__(kMergeThreads)
ctl_scan_kernel(int64_t m, int64_t half, LongWs ws, CtlWs cw, int cur) {
    __shared__ int s_tmp[32];
    const int64_t row = blockIdx.x, c0 = row * m;
    if (ctl_bad(ws, row)) return;
    const int nxt = cur ^ 1;
    const int64_t step = 2 * half, nodes = (m + step - 1) / step;
    const int tid = threadIdx.x, nth = blockDim.x;
    const int64_t per = (nodes + nth - 1) / nth;
    const int64_t kb = imin64(nodes, tid * per), ke = imin64(nodes, kb + per);
    int sum = 0;
    for (int64_t k = kb; k < ke; ++k) {
        const int64_t j = k * step, j1 = j + half;
        int4 d;
        if (j1 < m) {
            const int4 sl = ws.seg[c0 + j], sr = ws.seg[c0 + j1];
            d = make_int4(cw.base[cur][c0 + j] + sl.y, sl.z - sl.y + 1,
                          cw.base[cur][c0 + j1] + sr.y, sr.z - sr.y + 1);
        } else {
            d = make_int4(cw.base[cur][c0 + j], cw.size[cur][c0 + j], 0, 0);
        }
        cw.desc[c0 + j] = d;
        sum += d.y + d.w;
    }
    int total;
    int b = block_excl_scan_int(sum, s_tmp, total);
    for (int64_t k = kb; k < ke; ++k) {
        const int64_t j = k * step;
        const int4 d = cw.desc[c0 + j];
        const int sz = d.y + d.w;
        cw.base[nxt][c0 + j] = b;
        cw.size[nxt][c0 + j] = sz;
        ws.seg[c0 + j] = make_int4((int)j, 0, sz - 1, 0);
        ws.cnt[c0 + j] = 1;
        b += sz;
    }
    if (tid == 0) cw.rowH[row] = total;
}

// One level's copy: every surviving vertex of the row moves to its place in
// the other buffer, the whole grid over the row's vertices (the paper's
// second control kernel).  Each output position finds its node by bisection
// over the level's node bases.
template <bool WEIGHTED>
__global__ void __launch_bounds__(256)
ctl_copy_kernel(int64_t m, int64_t step, LongWs ws, CtlWs cw, int cur) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int64_t row = blockIdx.y, c0 = row * m;
    if (ctl_bad(ws, row)) return;
    const int nxt = cur ^ 1;
    const int64_t H = cw.rowH[row], nodes = (m + step - 1) / step;
    const size_t R = (size_t)c0 * ((size_t)C + 1);
    const int32_t* nb = cw.base[nxt] + c0;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < H;
         p += (int64_t)gridDim.x * blockDim.x) {
        int64_t lo = 0, hi = nodes - 1;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (nb[mid * step] <= p) lo = mid; else hi = mid - 1;
        }
        const int64_t j = lo * step;
        const int64_t q = p - nb[j];
        const int4 d = cw.desc[c0 + j];
        const int64_t src = q < d.y ? d.x + q : d.z + (q - d.y);
        cw.fS[nxt][R + p] = cw.fS[cur][R + src];
        if constexpr (WEIGHTED) cw.fW[nxt][R + p] = cw.fW[cur][R + src];
        cw.tag[nxt][R + p] = cw.tag[cur][R + src];
    }
}

// The root array's runs of equal chunk: each chunk's first and last root rank.
template <bool WEIGHTED>
__global__ void __launch_bounds__(256)
ctl_runs_kernel(int64_t m, LongWs ws, CtlWs cw, int cur) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int64_t row = blockIdx.y, c0 = row * m;
    if (ctl_bad(ws, row)) return;
    const int64_t H = cw.rowH[row];
    const uint64_t* tg = cw.tag[cur] + (size_t)c0 * ((size_t)C + 1);
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < H;
         p += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t t = tg[p];
        const int64_t ch = (int64_t)(t >> 32);
        const int rank = (int)((t >> 16) & 0xffffu);
        if (p == 0 || (int64_t)(tg[p - 1] >> 32) != ch) cw.runLo[c0 + ch] = rank;
        if (p + 1 == H || (int64_t)(tg[p + 1] >> 32) != ch) cw.runHi[c0 + ch] = rank;
    }
}

// The root list from the runs (at most one per chunk, in chunk order), then
// the ends exactly as the segment lists compute them.  One CTA per row.
template <bool WEIGHTED>
__global__ void __launch_bounds__(kMergeThreads)
ctl_root_kernel(int64_t m, LongWs ws, CtlWs cw) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    __shared__ int s_tmp[32];
    const int64_t row = blockIdx.x, c0 = row * m;
    if (ctl_bad(ws, row)) return;
    const int tid = threadIdx.x, nth = blockDim.x;
    const int64_t per = (m + nth - 1) / nth;
    const int64_t jb = imin64(m, tid * per), je = imin64(m, jb + per);
    int sum = 0;
    for (int64_t j = jb; j < je; ++j) sum += cw.runLo[c0 + j] >= 0 ? 1 : 0;
    int total;
    int k = block_excl_scan_int(sum, s_tmp, total);
    for (int64_t j = jb; j < je; ++j)
        if (cw.runLo[c0 + j] >= 0)
            ws.seg[c0 + k++] = make_int4((int)j, cw.runLo[c0 + j], cw.runHi[c0 + j], 0);
    if (tid == 0) ws.cnt[c0] = total;
    __syncthreads();
    MView<WEIGHTED, false> V;
    V.c0 = c0;
    V.C = C;
    V.bst = ws.bst;
    V.bmax = ws.bmax;
    V.seg = ws.seg + c0;
    V.cnt = ws.cnt + c0;
    V.offS = ws.offS + c0;
    V.offW = ws.offW + c0;
    V.vb = nullptr;
    V.S = ws.slot_S; V.W = ws.slot_W; V.P = ws.slot_p;
    V.dS = ws.dS + c0; V.dW = ws.dW + c0;
    root_ends<WEIGHTED>(V, m, ws, c0, ws.segOf + c0, ws.nextSeg + c0, ws.prevSeg + c0,
                        ws.rowq[row * 4 + 0] - (WEIGHTED ? ws.rowq[row * 4 + 1] : 0));
}

// Launch of a kernel that may start while the stream's previous kernel is
// finishing (programmatic dependent launch); the kernel calls
// wait_prior_grid() before reading what that kernel writes.
template <typename... P, typename... A>
static cudaError_t launch_after(void (*kern)(P...), unsigned grid, unsigned block, size_t smem,
                                cudaStream_t stream, A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launch sizes: exact counts for a dense batch, bounds for a ragged one.
struct LongGrid { int64_t rows, chunks, groups, ng; };

template <bool WEIGHTED, bool RAGGED, class IO>
static cudaError_t long_launch(const IO* y, const IO* w, const LongGeo& geo,
                               const LongGrid& gr, int increasing, IO* out, uint8_t* blocks,
                               const LongWs& ws, uint32_t* row_status, cudaStream_t stream) {
    constexpr int NT = LongCfg<WEIGHTED>::NT;
    using SM = TileSmem<NT, WEIGHTED, false, 1, IO>;
    cudaError_t err = cudaFuncSetAttribute(chunk_hull_kernel<WEIGHTED, RAGGED, IO>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    if (err != cudaSuccess) return err;
    chunk_hull_kernel<WEIGHTED, RAGGED, IO><<<(unsigned)gr.chunks, NT, SM::kBytes, stream>>>(y, w, geo,
                                                                                increasing, ws);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "chunk_hull");
    err = cudaFuncSetAttribute(merge_groups_kernel<WEIGHTED, RAGGED>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kFlatSmem);
    if (err != cudaSuccess) return err;
    // one wave of groups: kGroupThreads threads each (shorter chains of merges
    // per warp); more groups: half as many, two CTAs per SM
    const int gthreads = gr.groups <= device_sms() ? kGroupThreads : kGroupThreads / 2;
    err = launch_after(merge_groups_kernel<WEIGHTED, RAGGED>, (unsigned)gr.groups, gthreads, kFlatSmem,
                       stream, geo, gr.ng, ws, row_status);
    if (err != cudaSuccess) return err;
    prof_mark(stream, "merge_groups");
    err = cudaFuncSetAttribute(merge_top_kernel<WEIGHTED, RAGGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMergeSmem);
    if (err != cudaSuccess) return err;
    err = launch_after(merge_top_kernel<WEIGHTED, RAGGED>, (unsigned)gr.rows, kMergeThreads, kMergeSmem, stream,
                       geo, ws);
    if (err != cudaSuccess) return err;
    prof_mark(stream, "merge_top");
    err = cudaFuncSetAttribute(expand_kernel<WEIGHTED, RAGGED, IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               ExpandSmem<WEIGHTED, IO>::kBytes);
    if (err != cudaSuccess) return err;
    err = launch_after(expand_kernel<WEIGHTED, RAGGED, IO>, (unsigned)gr.chunks, NT,
                       (size_t)ExpandSmem<WEIGHTED, IO>::kBytes, stream, y, geo, increasing, ws, out, blocks);
    if (err != cudaSuccess) return err;
    prof_mark(stream, "expand");
    return cudaSuccess;
}

// Bounds of a ragged batch's long part: at most `rows` long segments, whose
// ceil(len / C) chunks number fewer than total / C + rows.
struct RaggedBounds { int64_t rows, chunks, groups; };

template <bool WEIGHTED>
static RaggedBounds ragged_bounds(int64_t rows, int64_t total) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int64_t M = total / C + rows + 1;
    return RaggedBounds{rows, M, M / kGroup + rows + 1};
}

// Tables of the ragged long part, then the workspace of the long path.
template <bool WEIGHTED>
static size_t carve_ragged(void* base, int64_t rows, int64_t total, LongGeo* geo, LongWs* ws) {
    const RaggedBounds B = ragged_bounds<WEIGHTED>(rows, total);
    size_t off = 0;
    char* b = static_cast<char*>(base);
    auto take = [&](size_t bytes) -> void* {
        void* p = b ? (void*)(b + off) : nullptr;
        off += align256(bytes);
        return p;
    };
    LongGeo g;
    g.e0 = (const int64_t*)take(8 * B.rows);
    g.len = (const int64_t*)take(8 * B.rows);
    g.c0 = (const int64_t*)take(8 * B.rows);
    g.g0 = (const int64_t*)take(8 * B.rows);
    g.id = (const int32_t*)take(4 * B.rows);
    g.chunk_row = (const int32_t*)take(4 * B.chunks);
    g.group_row = (const int32_t*)take(4 * B.groups);
    g.count = (const int64_t*)take(8 * 4);
    if (geo) *geo = g;
    off += carve<WEIGHTED>(b ? (void*)(b + off) : nullptr, B.rows, B.chunks, ws);
    return off;
}

}  // namespace


template <bool WEIGHTED, class IO>
static cudaError_t long_fit_t(const IO* y, const IO* w, int64_t rows, int64_t n,
                              int increasing, IO* out, uint8_t* blocks, void* wsp,
                              uint32_t* row_status, cudaStream_t stream) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int64_t m = (n + C - 1) / C;
    LongWs ws;
    carve<WEIGHTED>(wsp, rows, rows * m, &ws);
    LongGeo geo;
    geo.n = n;
    geo.m = m;
    const int64_t ng = (m + kGroup - 1) / kGroup;
    return long_launch<WEIGHTED, false, IO>(y, w, geo, LongGrid{rows, rows * m, rows * ng, ng}, increasing,
                                 out, blocks, ws, row_status, stream);
}

template <class IO>
cudaError_t long_fit(const IO* y, const IO* w, int64_t rows, int64_t n, int increasing, IO* out,
                     uint8_t* blocks, void* ws, size_t ws_bytes, uint32_t* row_status,
                     cudaStream_t stream) {
    (void)ws_bytes;
    return w ? long_fit_t<true, IO>(y, w, rows, n, increasing, out, blocks, ws, row_status, stream)
             : long_fit_t<false, IO>(y, w, rows, n, increasing, out, blocks, ws, row_status, stream);
}


template <bool WEIGHTED, class IO>
static cudaError_t long_fit_ragged_t(const IO* y, const IO* w, const int64_t* off,
                                     const int32_t* long_id, const unsigned long long* nlong,
                                     int64_t rows_max, int64_t total, int increasing, IO* out,
                                     uint8_t* blocks, void* wsp, uint32_t* row_status,
                                     cudaStream_t stream) {
    LongGeo geo;
    LongWs ws;
    carve_ragged<WEIGHTED>(wsp, rows_max, total, &geo, &ws);
    const RaggedBounds B = ragged_bounds<WEIGHTED>(rows_max, total);
    long_plan_kernel<LongCfg<WEIGHTED>::C><<<1, 1024, 0, stream>>>(
        off, long_id, nlong, B.rows, B.chunks, B.groups, geo, row_status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    prof_mark(stream, "long_plan");
    // bounded grids: the CTAs take the chunks (rows) in turn
    const LongGrid gr{std::min<int64_t>(B.rows, kRaggedTopCtas),
                      std::min<int64_t>(B.chunks, kRaggedCtas),
                      std::min<int64_t>(B.groups, kRaggedCtas), 0};
    return long_launch<WEIGHTED, true, IO>(y, w, geo, gr, increasing, out, blocks, ws, row_status, stream);
}

template <class IO>
cudaError_t long_fit_ragged(const IO* y, const IO* w, const int64_t* off,
                            const int32_t* long_id, const unsigned long long* nlong,
                            int64_t rows_max, int64_t total, int increasing, IO* out,
                            uint8_t* blocks, void* ws, uint32_t* row_status, cudaStream_t stream) {
    return w ? long_fit_ragged_t<true, IO>(y, w, off, long_id, nlong, rows_max, total, increasing,
                                           out, blocks, ws, row_status, stream)
             : long_fit_ragged_t<false, IO>(y, w, off, long_id, nlong, rows_max, total, increasing,
                                            out, blocks, ws, row_status, stream);
}


template <bool WEIGHTED, class IO>
static cudaError_t long_control_t(const IO* y, const IO* w, int64_t rows, int64_t n,
                                  int increasing, IO* out, uint8_t* blocks, void* wsp,
                                  uint32_t* row_status, cudaStream_t stream) {
    constexpr int NT = LongCfg<WEIGHTED>::NT;
    constexpr int C = LongCfg<WEIGHTED>::C;
    using SM = TileSmem<NT, WEIGHTED, false, 1, IO>;
    const int64_t m = (n + C - 1) / C, M = rows * m;
    LongWs ws;
    const size_t off = carve<WEIGHTED>(wsp, rows, M, &ws);
    CtlWs cw;
    carve_ctl<WEIGHTED>(static_cast<char*>(wsp) + off, rows, M, &cw);
    LongGeo geo;
    geo.n = n;
    geo.m = m;
    const int64_t ng = (m + kGroup - 1) / kGroup;
    cudaError_t err = cudaFuncSetAttribute(chunk_hull_kernel<WEIGHTED, false, IO>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    if (err != cudaSuccess) return err;
    chunk_hull_kernel<WEIGHTED, false, IO><<<(unsigned)M, NT, SM::kBytes, stream>>>(y, w, geo,
                                                                               increasing, ws);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "chunk_hull");
    // the rows' grids and the chunks' starts, without merging
    err = cudaFuncSetAttribute(merge_groups_kernel<WEIGHTED, false, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kGroupSmem);
    if (err != cudaSuccess) return err;
    merge_groups_kernel<WEIGHTED, false, false><<<(unsigned)(rows * ng), kGroupThreads / 2, kGroupSmem,
                                                  stream>>>(geo, ng, ws, row_status);
    ctl_base_kernel<WEIGHTED><<<(unsigned)rows, kMergeThreads, 0, stream>>>(m, ws, cw);
    ctl_flatten_kernel<WEIGHTED><<<(unsigned)M, 128, 0, stream>>>(m, ws, cw);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "ctl_setup");
    const unsigned xg = (unsigned)std::max<int64_t>(1, (152 * 8) / rows);
    int cur = 0;
    for (int64_t half = 1; half < m; half *= 2) {
        const int64_t nmerge = ((m + half - 1) / half) / 2;
        ctl_bridge_kernel<WEIGHTED><<<dim3((unsigned)((nmerge + 127) / 128), (unsigned)rows), 128, 0,
                                      stream>>>(m, half, nmerge, ws, cw, cur);
        ctl_scan_kernel<<<(unsigned)rows, kMergeThreads, 0, stream>>>(m, half, ws, cw, cur);
        ctl_copy_kernel<WEIGHTED><<<dim3(xg, (unsigned)rows), 256, 0, stream>>>(m, 2 * half, ws, cw,
                                                                                cur);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        cur ^= 1;
    }
    prof_mark(stream, "ctl_merge_levels");
    ctl_runs_kernel<WEIGHTED><<<dim3(xg, (unsigned)rows), 256, 0, stream>>>(m, ws, cw, cur);
    ctl_root_kernel<WEIGHTED><<<(unsigned)rows, kMergeThreads, 0, stream>>>(m, ws, cw);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "ctl_root");
    err = cudaFuncSetAttribute(expand_kernel<WEIGHTED, false, IO>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               ExpandSmem<WEIGHTED, IO>::kBytes);
    if (err != cudaSuccess) return err;
    expand_kernel<WEIGHTED, false, IO><<<(unsigned)M, NT, ExpandSmem<WEIGHTED, IO>::kBytes, stream>>>(
        y, geo, increasing, ws, out, blocks);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "expand");
    return cudaSuccess;
}

template <class IO>
cudaError_t long_fit_control(const IO* y, const IO* w, int64_t rows, int64_t n, int increasing,
                             IO* out, uint8_t* blocks, void* ws, uint32_t* row_status,
                             cudaStream_t stream) {
    return w ? long_control_t<true, IO>(y, w, rows, n, increasing, out, blocks, ws, row_status,
                                        stream)
             : long_control_t<false, IO>(y, w, rows, n, increasing, out, blocks, ws, row_status,
                                         stream);
}

}  // namespace isodev
