// Long rows (n > 8,192): the paper's three-level algorithm (Section 3).
//
//  1. chunk_hull_kernel: one CTA per chunk builds the chunk's hull (lanes ->
//     warps -> CTA, Sections 3.1-3.2) and writes its vertices once into the
//     chunk's slot, with coordinates relative to the chunk (Section 3.3).
//  2. merge_kernel: one CTA per row merges the chunk hulls in a tree.  A node
//     is a list of segments (chunk, first vertex, last vertex), at most one per
//     chunk (Definition 4.3, Theorem 4.4); a merge finds the bridge by a capped
//     walk, or by a nested bisection when the walk gives up (Section 5.2),
//     cuts two segments and moves the right list's descriptors down.  No
//     vertex is ever copied.  It then finds each chunk's range in the root
//     list and the edges into and out of it (Section 3.4, Corollary 4.5).
//  3. expand_kernel: one CTA per chunk writes every element's slope and its
//     block-start byte (Section 3.4).
#include <cstdio>

#include "iso_internal.h"
#include "iso_tile.cuh"

namespace isodev {

namespace {

constexpr int kWalkCap = 64;   // steps of a walk before the bisection takes over (Section 6)

template <bool WEIGHTED> struct LongCfg;
template <> struct LongCfg<false> { static constexpr int NT = 256; static constexpr int C = 8192; };
template <> struct LongCfg<true> { static constexpr int NT = 128; static constexpr int C = 4096; };

struct ChunkMeta {
    int32_t h;      // hull vertices (both ends included)
    int32_t bad;    // ISO_ROW_BAD_* bits
    int32_t qs, qw; // quantum exponents of S and W
    int64_t totS, totW;   // chunk totals (chunk quanta)
};

typedef __int128 i128;

struct ChunkEnds {            // per chunk, from the root list
    int32_t lo, hi;           // rank range of the chunk's root segment, lo > hi if none
    int32_t pt0_vertex;       // 1 if the chunk's first point is a root vertex (closes the previous segment)
    int32_t bad;              // row status bits
    i128 prevW, prevS;        // previous root vertex (row coordinates)
    i128 nextW, nextS;        // next root vertex (row coordinates)
};

struct LongWs {
    ChunkMeta* meta;   // [M]
    int32_t* slot_p;   // [M][C+1] vertex point index within the chunk
    int64_t* slot_S;   // [M][C+1]
    int64_t* slot_W;   // [M][C+1] (weighted)
    int4* seg;         // [M] segment lists: (chunk in row, lo, hi, 0)
    int32_t* cnt;      // [M] list lengths, at a node's first chunk
    int32_t* pre;      // [M] flattened-rank prefixes of a merge's lists
    i128* offS;        // [M] chunk start, row coordinates (row quanta)
    i128* offW;        // [M]
    int32_t* dS;       // [M] shift from chunk to row quantum
    int32_t* dW;       // [M]
    int32_t* segOf;    // [M] root segment of a chunk, or -1
    int32_t* nextSeg;  // [M]
    int32_t* prevSeg;  // [M]
    ChunkEnds* ends;   // [M]
    int32_t* rowq;     // [rows][4]: qs_row, qw_row, bad
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <bool WEIGHTED>
__host__ __device__ inline size_t carve(void* base, int64_t rows, int64_t n, LongWs* ws) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int64_t m = (n + C - 1) / C;
    const int64_t M = rows * m;
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
    w.slot_p = (int32_t*)take(sizeof(int32_t) * cap * M);
    w.slot_S = (int64_t*)take(sizeof(int64_t) * cap * M);
    w.slot_W = WEIGHTED ? (int64_t*)take(sizeof(int64_t) * cap * M) : nullptr;
    w.seg = (int4*)take(sizeof(int4) * M);
    w.cnt = (int32_t*)take(sizeof(int32_t) * M);
    w.pre = (int32_t*)take(sizeof(int32_t) * M);
    w.offS = (i128*)take(sizeof(i128) * M);
    w.offW = (i128*)take(sizeof(i128) * M);
    w.dS = (int32_t*)take(sizeof(int32_t) * M);
    w.dW = (int32_t*)take(sizeof(int32_t) * M);
    w.segOf = (int32_t*)take(sizeof(int32_t) * M);
    w.nextSeg = (int32_t*)take(sizeof(int32_t) * M);
    w.prevSeg = (int32_t*)take(sizeof(int32_t) * M);
    w.ends = (ChunkEnds*)take(sizeof(ChunkEnds) * M);
    w.rowq = (int32_t*)take(sizeof(int32_t) * 4 * rows);
    if (ws) *ws = w;
    return off;
}

// Nearest double of a 128-bit integer (two roundings at most).
__device__ __forceinline__ double i128_to_double(i128 x) {
    const int64_t hi = (int64_t)(x >> 64);
    const uint64_t lo = (uint64_t)x;
    return ldexp((double)hi, 64) + (double)lo;
}

// Round x / 2^d to nearest (half up); d >= 0.
__device__ __forceinline__ int64_t conv(int64_t x, int d) {
    if (d <= 0) return x;
    if (d >= 63) return 0;
    return (x + (1LL << (d - 1))) >> d;
}

// ---------------------------------------------------------------------------
// 1. chunk hulls
// ---------------------------------------------------------------------------
template <bool WEIGHTED>
__global__ void __launch_bounds__(LongCfg<WEIGHTED>::NT)
chunk_hull_kernel(const float* __restrict__ y, const float* __restrict__ w, int64_t n, int64_t m,
                  int increasing, LongWs ws) {
    constexpr int NT = LongCfg<WEIGHTED>::NT;
    constexpr int C = LongCfg<WEIGHTED>::C;
    extern __shared__ __align__(128) unsigned char smem[];
    using SM = TileSmem<NT, WEIGHTED>;
    const int64_t c = blockIdx.x;
    const int64_t row = c / m;
    const int64_t j = c - row * m;
    const int64_t e0 = j * C;
    const int nt = (int)imin64(C, n - e0);
    const float* yr = y + row * n + e0;
    const float* wr = WEIGHTED ? w + row * n + e0 : nullptr;

    TileHull H;
    tile_hull_phase<NT, WEIGHTED>(yr, wr, nt, true, !increasing, NT, smem, H);

    // ranks of the vertices: exclusive scan of the lanes' vertex counts
    int64_t* scan = reinterpret_cast<int64_t*>(smem + SM::oScan);
    const uint32_t mask = H.T.mask[H.lane];
    const int cntl = __popc(mask);
    const int64_t inc = tile_scan_incl<NT>((int64_t)cntl, H.lane, NT, scan);
    int rank = (int)(inc - cntl);
    const size_t cap = (size_t)C + 1;
    int32_t* sp = ws.slot_p + c * cap;
    int64_t* sS = ws.slot_S + c * cap;
    int64_t* sW = WEIGHTED ? ws.slot_W + c * cap : nullptr;
    if (H.bad == 0) {
        uint32_t mm = mask;
        while (mm) {
            const int k = __ffs(mm) - 1;
            mm &= mm - 1u;
            const int p = (H.lane << 5) + k;
            sp[rank] = p;
            sS[rank] = tile_S<WEIGHTED>(H.T, p);
            if constexpr (WEIGHTED) sW[rank] = tile_W<WEIGHTED>(H.T, p);
            ++rank;
        }
    }
    if (threadIdx.x == NT - 1) {
        // the chunk's end point closes the list
        const int h = (int)inc + 1;
        ChunkMeta mt;
        mt.h = h;
        mt.bad = (int32_t)H.bad;
        mt.qs = H.qs;
        mt.qw = H.qw;
        mt.totS = H.T.LS[NT];
        mt.totW = WEIGHTED ? H.T.LW[NT] : (int64_t)nt;
        if (H.bad == 0) {
            sp[h - 1] = nt;
            sS[h - 1] = mt.totS;
            if constexpr (WEIGHTED) sW[h - 1] = mt.totW;
        }
        ws.meta[c] = mt;
    }
}

// ---------------------------------------------------------------------------
// 2. merge tree over segment lists (one CTA per row)
// ---------------------------------------------------------------------------
struct Pos { int k, r; };   // segment index in the row's list array, rank in its chunk

template <bool WEIGHTED>
struct RowView {
    LongWs ws;
    int64_t c0;      // global index of the row's chunk 0
    int64_t m;
    int C;
    int4* seg;       // row's segment array (m entries)
    int32_t* cnt;
    int32_t* pre;

    __device__ __forceinline__ void vertex(int jc, int r, i128& W, i128& S) const {
        const int64_t c = c0 + jc;
        const size_t idx = (size_t)c * ((size_t)C + 1) + r;
        S = ws.offS[c] + conv(ws.slot_S[idx], ws.dS[c]);
        if constexpr (WEIGHTED) W = ws.offW[c] + conv(ws.slot_W[idx], ws.dW[c]);
        else W = (i128)((int64_t)jc * C + ws.slot_p[idx]);
    }
    __device__ __forceinline__ void at(Pos p, i128& W, i128& S) const {
        vertex(seg[p.k].x, p.r, W, S);
    }
    // the turn o -> a -> b is strictly left (exact, 256-bit products)
    __device__ __forceinline__ bool left(Pos o, Pos a, Pos b) const {
        i128 Wo, So, Wa, Sa, Wb, Sb;
        at(o, Wo, So); at(a, Wa, Sa); at(b, Wb, Sb);
        return sign_det128(Wa - Wo, Sb - So, Sa - So, Wb - Wo) > 0;
    }
};

template <bool WEIGHTED>
__device__ void merge_pair(const RowView<WEIGHTED>& V, int j0, int j1) {
    int4* seg = V.seg;
    const int nL = V.cnt[j0], nR = V.cnt[j1];
    const int kLl = j0 + nL - 1, kR0 = j1, kRl = j1 + nR - 1;
    const Pos sL = {kLl, seg[kLl].z};
    const Pos sR = {kR0, seg[kR0].y};
    auto hasPrev = [&](Pos p) { return p.r > seg[p.k].y || p.k > j0; };
    auto prev = [&](Pos p) -> Pos {
        return p.r > seg[p.k].y ? Pos{p.k, p.r - 1} : Pos{p.k - 1, seg[p.k - 1].z};
    };
    auto hasNext = [&](Pos p) { return p.r < seg[p.k].z || p.k < kRl; };
    auto next = [&](Pos p) -> Pos {
        return p.r < seg[p.k].z ? Pos{p.k, p.r + 1} : Pos{p.k + 1, seg[p.k + 1].y};
    };
    const Pos pa = prev(sL);
    const Pos sb = next(sR);
    if (V.left(pa, sL, sb)) {
        // convex at s: append R without its first vertex s
        int first = kR0;
        const int lo = seg[kR0].y + 1;
        if (lo > seg[kR0].z) first = kR0 + 1;
        else seg[kR0].y = lo;
        int dst = j0 + nL;
        for (int k = first; k <= kRl; ++k) seg[dst++] = seg[k];
        V.cnt[j0] = dst - j0;
        return;
    }
    Pos a = pa, b = sb;
    int steps = 0;
    bool gave_up = false;
    for (;;) {
        bool moved = false;
        while (hasPrev(a)) {
            Pos p = prev(a);
            if (V.left(p, a, b)) break;
            a = p; moved = true;
            if (++steps > kWalkCap) { gave_up = true; break; }
        }
        if (gave_up) break;
        while (hasNext(b)) {
            Pos q = next(b);
            if (V.left(a, b, q)) break;
            b = q; moved = true;
            if (++steps > kWalkCap) { gave_up = true; break; }
        }
        if (gave_up || !moved) break;
    }
    if (gave_up) {
        // nested bisection (Section 5.2): over the candidates of L, each tested
        // against its tangent to R, itself found by bisection over R.
        int totL = 0, totR = 0;
        for (int k = j0; k <= kLl; ++k) { V.pre[k] = totL; totL += seg[k].z - seg[k].y + 1; }
        for (int k = kR0; k <= kRl; ++k) { V.pre[k] = totR; totR += seg[k].z - seg[k].y + 1; }
        auto flatL = [&](int f) -> Pos {
            int lo = j0, hi = kLl;
            while (lo < hi) { int mid = (lo + hi + 1) >> 1; if (V.pre[mid] <= f) lo = mid; else hi = mid - 1; }
            return Pos{lo, seg[lo].y + (f - V.pre[lo])};
        };
        auto flatR = [&](int g) -> Pos {
            int lo = kR0, hi = kRl;
            while (lo < hi) { int mid = (lo + hi + 1) >> 1; if (V.pre[mid] <= g) lo = mid; else hi = mid - 1; }
            return Pos{lo, seg[lo].y + (g - V.pre[lo])};
        };
        // tangent point of R seen from L-vertex pa: first g in [1, totR-1] where
        // the next vertex is strictly above the line from pa through it
        auto tangent = [&](Pos ap) -> int {
            int lo = 1, hi = totR - 1;
            while (lo < hi) {
                int mid = (lo + hi) >> 1;
                Pos bm = flatR(mid);
                Pos bn = flatR(mid + 1);
                if (V.left(ap, bm, bn)) hi = mid; else lo = mid + 1;
            }
            return lo;
        };
        int lo = 0, hi = totL - 2;   // candidates: every vertex of L before s
        while (lo < hi) {
            int mid = (lo + hi) >> 1;
            Pos am = flatL(mid);
            Pos an = flatL(mid + 1);
            Pos t = flatR(tangent(am));
            // next vertex of L strictly below the line from am to its tangent: go right
            if (V.left(am, an, t)) lo = mid + 1; else hi = mid;
        }
        a = flatL(lo);
        b = flatR(tangent(a));
    }
    // cut L at a, R at b, and move R's tail down
    seg[a.k].z = a.r;
    seg[b.k].y = b.r;
    int dst = a.k + 1;
    for (int k = b.k; k <= kRl; ++k) seg[dst++] = seg[k];
    V.cnt[j0] = dst - j0;
}

template <bool WEIGHTED>
__global__ void __launch_bounds__(1024)
merge_kernel(int64_t m, LongWs ws, uint32_t* __restrict__ row_status) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    const int64_t row = blockIdx.x;
    const int64_t c0 = row * m;
    const int tid = threadIdx.x, nth = blockDim.x;
    __shared__ int s_qs, s_qw, s_bad;
    __shared__ i128 s_scanS[1024], s_scanW[1024];
    if (tid == 0) { s_qs = -100000; s_qw = -100000; s_bad = 0; }
    __syncthreads();
    int qs = -100000, qw = -100000, bad = 0;
    for (int64_t j = tid; j < m; j += nth) {
        const ChunkMeta mt = ws.meta[c0 + j];
        qs = max(qs, mt.qs); qw = max(qw, mt.qw); bad |= mt.bad;
    }
    atomicMax(&s_qs, qs);
    atomicMax(&s_qw, qw);
    if (bad) atomicOr(&s_bad, bad);
    __syncthreads();
    qs = s_qs; qw = s_qw; bad = s_bad;
    if (tid == 0) {
        ws.rowq[row * 4 + 0] = qs; ws.rowq[row * 4 + 1] = qw; ws.rowq[row * 4 + 2] = bad;
        if (row_status) row_status[row] = (uint32_t)bad;
    }
    if (bad) {
        for (int64_t j = tid; j < m; j += nth) {
            ChunkEnds ce{};
            ce.lo = 1; ce.hi = 0; ce.bad = bad;
            ws.ends[c0 + j] = ce;
        }
        return;
    }
    // chunk starts in row coordinates: exclusive scan of converted chunk totals.
    // Each thread scans a contiguous range of chunks.
    const int64_t per = (m + nth - 1) / nth;
    const int64_t jb = imin64(m, tid * per), je = imin64(m, jb + per);
    i128 accS = 0, accW = 0;
    for (int64_t j = jb; j < je; ++j) {
        const ChunkMeta mt = ws.meta[c0 + j];
        const int ds = qs - mt.qs, dw = WEIGHTED ? qw - mt.qw : 0;
        ws.dS[c0 + j] = ds;
        ws.dW[c0 + j] = dw;
        accS += conv(mt.totS, ds);
        accW += WEIGHTED ? conv(mt.totW, dw) : mt.totW;
    }
    s_scanS[tid] = accS;
    s_scanW[tid] = accW;
    __syncthreads();
    if (tid == 0) {
        i128 a = 0, b = 0;
        for (int t = 0; t < nth; ++t) {
            i128 x = s_scanS[t], y2 = s_scanW[t];
            s_scanS[t] = a; s_scanW[t] = b;
            a += x; b += y2;
        }
    }
    __syncthreads();
    accS = s_scanS[tid];
    accW = s_scanW[tid];
    for (int64_t j = jb; j < je; ++j) {
        const ChunkMeta mt = ws.meta[c0 + j];
        ws.offS[c0 + j] = accS;
        ws.offW[c0 + j] = accW;
        accS += conv(mt.totS, ws.dS[c0 + j]);
        accW += WEIGHTED ? conv(mt.totW, ws.dW[c0 + j]) : mt.totW;
        ws.seg[c0 + j] = make_int4((int)j, 0, mt.h - 1, 0);
        ws.cnt[c0 + j] = 1;
    }
    __threadfence_block();
    __syncthreads();

    RowView<WEIGHTED> V;
    V.ws = ws; V.c0 = c0; V.m = m; V.C = C;
    V.seg = ws.seg + c0; V.cnt = ws.cnt + c0; V.pre = ws.pre + c0;
    for (int r = 0; ((int64_t)1 << r) < m; ++r) {
        const int64_t span = (int64_t)2 << r;
        const int64_t merges = (m + span - 1) / span;
        for (int64_t g = tid; g < merges; g += nth) {
            const int64_t j0 = g * span, j1 = j0 + (span >> 1);
            if (j1 < m) merge_pair<WEIGHTED>(V, (int)j0, (int)j1);
        }
        __threadfence_block();
        __syncthreads();
    }

    // ends: each chunk's root segment, and the root vertices before and after it
    const int nroot = V.cnt[0];
    for (int64_t j = tid; j < m; j += nth) ws.segOf[c0 + j] = -1;
    __syncthreads();
    for (int k = tid; k < nroot; k += nth) ws.segOf[c0 + V.seg[k].x] = k;
    __syncthreads();
    for (int k = tid; k < nroot; k += nth) {
        const int cj = V.seg[k].x;
        const int cprev = k > 0 ? V.seg[k - 1].x : -1;
        const int cnext = k + 1 < nroot ? V.seg[k + 1].x : (int)m;
        for (int q = max(cprev, 0); q < cj; ++q) ws.nextSeg[c0 + q] = k;   // chunks in [cprev, cj)
        for (int q = cj + 1; q <= min(cnext, (int)m - 1); ++q) ws.prevSeg[c0 + q] = k;
    }
    __syncthreads();
    for (int64_t j = tid; j < m; j += nth) {
        ChunkEnds ce;
        ce.bad = 0;
        const int sk = ws.segOf[c0 + j];
        if (sk >= 0) { ce.lo = V.seg[sk].y; ce.hi = V.seg[sk].z; }
        else { ce.lo = 1; ce.hi = 0; }
        ce.prevW = ce.prevS = ce.nextW = ce.nextS = 0;
        ce.pt0_vertex = 0;
        if (j > 0) {
            const int pk = ws.prevSeg[c0 + j];
            const int pc = V.seg[pk].x, pr = V.seg[pk].z;
            V.vertex(pc, pr, ce.prevW, ce.prevS);
            // the previous root vertex is this chunk's first point when it closes chunk j-1
            const ChunkMeta pm = ws.meta[c0 + pc];
            ce.pt0_vertex = (pc == j - 1 && pr == pm.h - 1) ? 1 : 0;
        }
        if (j + 1 < m || sk < 0) {
            if (j + 1 < m) {
                const int nk = ws.nextSeg[c0 + j];
                V.vertex(V.seg[nk].x, V.seg[nk].y, ce.nextW, ce.nextS);
            }
        }
        ws.ends[c0 + j] = ce;
    }
}

// ---------------------------------------------------------------------------
// 3. expansion: each element gets the slope of the root-hull edge above it
// ---------------------------------------------------------------------------
template <bool WEIGHTED>
struct ExpandSmem {
    static constexpr int NT = LongCfg<WEIGHTED>::NT;
    static constexpr int C = LongCfg<WEIGHTED>::C;
    static constexpr int oMask = 0;
    static constexpr int oTmp = oMask + NT * 4;
    static constexpr int oSlope = oTmp + (NT / 32 + 2) * 8;
    static constexpr int oOut = oSlope + ((C + 2) * 4 + 15) / 16 * 16;
    static constexpr int kBytes = oOut + C * 4;
};

template <bool WEIGHTED>
__global__ void __launch_bounds__(LongCfg<WEIGHTED>::NT)
expand_kernel(int64_t n, int64_t m, int increasing, LongWs ws, float* __restrict__ out,
              uint8_t* __restrict__ blocks) {
    constexpr int NT = LongCfg<WEIGHTED>::NT;
    constexpr int C = LongCfg<WEIGHTED>::C;
    using XS = ExpandSmem<WEIGHTED>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + XS::oMask);
    int64_t* s_tmp = reinterpret_cast<int64_t*>(smem + XS::oTmp);
    float* s_slope = reinterpret_cast<float*>(smem + XS::oSlope);
    float* s_out = reinterpret_cast<float*>(smem + XS::oOut);

    const int64_t c = blockIdx.x;
    const int64_t row = c / m;
    const int64_t j = c - row * m;
    const int64_t e0 = j * C;
    const int nt = (int)imin64(C, n - e0);
    const int tid = threadIdx.x;
    const ChunkEnds ce = ws.ends[c];
    float* orow = out + row * n + e0;
    uint8_t* brow = blocks ? blocks + row * n + e0 : nullptr;

    if (ce.bad) {
        const float qnan = __int_as_float(0x7fffffff);
        for (int i = tid; i < nt; i += NT) {
            orow[i] = qnan;
            if (brow) brow[i] = 0;
        }
        return;
    }
    const size_t cap = (size_t)C + 1;
    const int32_t* sp = ws.slot_p + c * cap;
    const int64_t* sS = ws.slot_S + c * cap;
    const int64_t* sW = WEIGHTED ? ws.slot_W + c * cap : nullptr;
    const int qs_row = ws.rowq[row * 4 + 0];
    const int qw_row = WEIGHTED ? ws.rowq[row * 4 + 1] : 0;
    const ChunkMeta mt = ws.meta[c];
    const i128 offS = ws.offS[c], offW = ws.offW[c];
    const int ds = ws.dS[c], dw = ws.dW[c];

    s_mask[tid] = 0u;
    __syncthreads();
    // root vertices of this chunk that start one of its elements (point < nt)
    const bool has = ce.lo <= ce.hi;
    if (has) {
        for (int r = ce.lo + tid; r <= ce.hi; r += NT) {
            const int p = sp[r];
            if (p < nt) atomicOr(&s_mask[p >> 5], 1u << (p & 31));
        }
    }
    if (tid == 0 && ce.pt0_vertex) atomicOr(&s_mask[0], 1u);
    auto row_slope = [&](i128 Wa, i128 Sa, i128 Wb, i128 Sb) -> float {
        const double f = i128_to_double(Sb - Sa) / i128_to_double(Wb - Wa);
        return (float)ldexp(f, qs_row - qw_row);
    };
    auto vrow = [&](int r, i128& W, i128& S) {
        S = offS + conv(sS[r], ds);
        if constexpr (WEIGHTED) W = offW + conv(sW[r], dw);
        else W = (i128)(e0 + sp[r]);
    };
    // s_slope[i]: slope of the edge leaving the i-th vertex of the chunk's mask
    // (point order).  When the chunk's first point closes the previous chunk's
    // segment it is vertex 0 and its edge is the one entering the chunk.
    const int base = ce.pt0_vertex ? 1 : 0;
    if (has) {
        for (int r = ce.lo + tid; r <= ce.hi; r += NT) {
            float sl = 0.0f;
            if (r < ce.hi) {
                // both ends in the chunk: chunk-relative coordinates, chunk quanta
                const int64_t dS_ = sS[r + 1] - sS[r];
                const int64_t dW_ = WEIGHTED ? sW[r + 1] - sW[r] : (int64_t)(sp[r + 1] - sp[r]);
                sl = ldexpf(__ll2float_rn(dS_) / __ll2float_rn(dW_), mt.qs - (WEIGHTED ? mt.qw : 0));
            } else if (sp[r] < nt) {
                i128 Wa, Sa;
                vrow(r, Wa, Sa);
                sl = row_slope(Wa, Sa, ce.nextW, ce.nextS);
            }
            s_slope[base + (r - ce.lo)] = sl;
        }
    }
    if (tid == 0) {
        // the edge entering the chunk: from the previous root vertex to the first
        // root vertex of the chunk, or to the next root vertex if the chunk has none
        float in_sl = 0.0f;
        if (j > 0) {
            i128 Wb, Sb;
            if (has) vrow(ce.lo, Wb, Sb);
            else { Wb = ce.nextW; Sb = ce.nextS; }
            in_sl = row_slope(ce.prevW, ce.prevS, Wb, Sb);
        }
        if (ce.pt0_vertex) s_slope[0] = in_sl;
        s_tmp[NT / 32 + 1] = (int64_t)__float_as_int(in_sl);
    }
    __syncthreads();
    const uint32_t mk = s_mask[tid];
    const int cntl = __popc(mk);
    const int64_t inc = tile_scan_incl<NT>((int64_t)cntl, tid, NT, s_tmp);
    const int pre = (int)(inc - cntl);
    const float in_sl = __int_as_float((int)s_tmp[NT / 32 + 1]);
    const int p0 = tid << 5;
    const int e = min(max(nt - p0, 0), 32);
    for (int k = 0; k < e; ++k) {
        const uint32_t upto = (k == 31) ? mk : (mk & ((2u << k) - 1u));
        const int idx = pre + __popc(upto) - 1;   // the last vertex at or before this element
        float v = idx < 0 ? in_sl : s_slope[idx];
        if (!increasing) v = -v;
        s_out[spos(tid, k)] = v;
    }
    __syncthreads();
    for (int i = tid; i < nt; i += NT) {
        orow[i] = s_out[spos(i >> 5, i & 31)];
        if (brow) brow[i] = (uint8_t)((s_mask[i >> 5] >> (i & 31)) & 1u);
    }
}

}  // namespace

size_t long_fit_workspace(int64_t rows, int64_t n, bool weighted) {
    return weighted ? carve<true>(nullptr, rows, n, nullptr) : carve<false>(nullptr, rows, n, nullptr);
}

template <bool WEIGHTED>
static cudaError_t long_fit_t(const float* y, const float* w, int64_t rows, int64_t n,
                              int increasing, float* out, uint8_t* blocks, void* wsp,
                              uint32_t* row_status, cudaStream_t stream) {
    constexpr int NT = LongCfg<WEIGHTED>::NT;
    constexpr int C = LongCfg<WEIGHTED>::C;
    using SM = TileSmem<NT, WEIGHTED>;
    LongWs ws;
    carve<WEIGHTED>(wsp, rows, n, &ws);
    const int64_t m = (n + C - 1) / C;
    const int64_t M = rows * m;
    cudaError_t err = cudaFuncSetAttribute(chunk_hull_kernel<WEIGHTED>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    if (err != cudaSuccess) return err;
    chunk_hull_kernel<WEIGHTED><<<(unsigned)M, NT, SM::kBytes, stream>>>(y, w, n, m, increasing, ws);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "chunk_hull");
    merge_kernel<WEIGHTED><<<(unsigned)rows, 1024, 0, stream>>>(m, ws, row_status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "merge");
    err = cudaFuncSetAttribute(expand_kernel<WEIGHTED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               ExpandSmem<WEIGHTED>::kBytes);
    if (err != cudaSuccess) return err;
    expand_kernel<WEIGHTED><<<(unsigned)M, NT, ExpandSmem<WEIGHTED>::kBytes, stream>>>(
        n, m, increasing, ws, out, blocks);
    prof_mark(stream, "expand");
    return cudaGetLastError();
}

cudaError_t long_fit(const float* y, const float* w, int64_t rows, int64_t n, int increasing,
                     float* out, uint8_t* blocks, void* ws, size_t ws_bytes, uint32_t* row_status,
                     cudaStream_t stream) {
    (void)ws_bytes;
    return w ? long_fit_t<true>(y, w, rows, n, increasing, out, blocks, ws, row_status, stream)
             : long_fit_t<false>(y, w, rows, n, increasing, out, blocks, ws, row_status, stream);
}

}  // namespace isodev
