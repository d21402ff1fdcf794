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
//     vertex is ever copied between levels.  When a row's chunk hulls fit in
//     shared memory (noisy rows keep few vertices) they are read once into it
//     and the whole tree runs there; otherwise the tree reads them from the
//     slots in global memory.  The kernel then finds each chunk's range in the
//     root list and the root vertices before and after it (Section 3.4,
//     Corollary 4.5).
//  3. expand_kernel: one CTA per chunk writes every element's slope and its
//     block-start byte (Section 3.4).
#include "iso_internal.h"
#include "iso_tile.cuh"

namespace isodev {

namespace {

constexpr int kWalkCap = 64;              // steps of a walk before the bisection (Section 6)
constexpr int kMergeThreads = 512;
constexpr int kMergeSmem = 210 * 1024;    // shared memory of the merge kernel

template <bool WEIGHTED> struct LongCfg;
template <> struct LongCfg<false> { static constexpr int NT = 256; static constexpr int C = 8192; };
template <> struct LongCfg<true> { static constexpr int NT = 128; static constexpr int C = 4096; };

typedef __int128 i128;

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
    i128 prevW, prevS;        // previous root vertex (row coordinates)
    i128 nextW, nextS;        // next root vertex (row coordinates)
};

struct LongWs {
    ChunkMeta* meta;   // [M]
    uint16_t* slot_p;  // [M][C+1] vertex point index within the chunk
    int64_t* slot_S;   // [M][C+1]
    int64_t* slot_W;   // [M][C+1] (weighted)
    int4* seg;         // [M] segment lists (global-memory trees)
    int32_t* cnt;      // [M]
    int32_t* pre;      // [M]
    int32_t* segOf;    // [M]
    int32_t* nextSeg;  // [M]
    int32_t* prevSeg;  // [M]
    i128* offS;        // [M] chunk start, row coordinates (row quanta)
    i128* offW;        // [M]
    int32_t* dS;       // [M] shift from chunk to row quantum
    int32_t* dW;       // [M]
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
    w.slot_p = (uint16_t*)take(sizeof(uint16_t) * cap * M);
    w.slot_S = (int64_t*)take(sizeof(int64_t) * cap * M);
    w.slot_W = WEIGHTED ? (int64_t*)take(sizeof(int64_t) * cap * M) : nullptr;
    w.seg = (int4*)take(sizeof(int4) * M);
    w.cnt = (int32_t*)take(sizeof(int32_t) * M);
    w.pre = (int32_t*)take(sizeof(int32_t) * M);
    w.segOf = (int32_t*)take(sizeof(int32_t) * M);
    w.nextSeg = (int32_t*)take(sizeof(int32_t) * M);
    w.prevSeg = (int32_t*)take(sizeof(int32_t) * M);
    w.offS = (i128*)take(sizeof(i128) * M);
    w.offW = (i128*)take(sizeof(i128) * M);
    w.dS = (int32_t*)take(sizeof(int32_t) * M);
    w.dW = (int32_t*)take(sizeof(int32_t) * M);
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
    using SM = TileSmem<NT, WEIGHTED, false, 1>;
    const int64_t c = blockIdx.x;
    const int64_t row = c / m;
    const int64_t j = c - row * m;
    const int64_t e0 = j * C;
    const int nt = (int)imin64(C, n - e0);
    const float* yr = y + row * n + e0;
    const float* wr = WEIGHTED ? w + row * n + e0 : nullptr;

    TileHull H;
    tile_hull_phase<NT, WEIGHTED, false, 1>(yr, wr, nt, true, !increasing, NT, smem, H);

    // ranks of the vertices: exclusive scan of the lanes' vertex counts
    int64_t* scan = reinterpret_cast<int64_t*>(smem + SM::oScan);
    const uint32_t mask = H.T.mask[H.lane];
    const int cntl = __popc(mask);
    const int64_t inc = tile_scan_incl<NT>((int64_t)cntl, H.lane, NT, scan);
    int rank = (int)(inc - cntl);
    const size_t cap = (size_t)C + 1;
    uint16_t* sp = ws.slot_p + c * cap;
    int64_t* sS = ws.slot_S + c * cap;
    int64_t* sW = WEIGHTED ? ws.slot_W + c * cap : nullptr;
    if (H.bad == 0) {
        uint32_t mm = mask;
        while (mm) {
            const int k = __ffs(mm) - 1;
            mm &= mm - 1u;
            const int p = (H.lane << 5) + k;
            sp[rank] = (uint16_t)p;
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
            sp[h - 1] = (uint16_t)nt;
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

// Where the merge tree finds a row's chunk hulls and keeps its lists: shared
// memory (compact copies) or the workspace slots in global memory.
template <bool WEIGHTED>
struct MStore {
    const int32_t* vb;       // first vertex of each chunk in P/S/W; nullptr: slot layout
    const uint16_t* P;
    const int64_t* S;
    const int64_t* W;
    const i128* offS;
    const i128* offW;
    const int32_t* dS;
    const int32_t* dW;
    int4* seg;               // (chunk in row, lo, hi, 0)
    int32_t* cnt;
    int32_t* pre;
    int64_t c0;              // global index of the row's chunk 0 (slot layout)
    int C;

    __device__ __forceinline__ size_t vidx(int jc, int r) const {
        return vb ? (size_t)vb[jc] + r : (size_t)(c0 + jc) * ((size_t)C + 1) + r;
    }
    __device__ __forceinline__ void vertex(int jc, int r, i128& Wv, i128& Sv) const {
        const size_t i = vidx(jc, r);
        Sv = offS[jc] + conv(S[i], dS[jc]);
        if constexpr (WEIGHTED) Wv = offW[jc] + conv(W[i], dW[jc]);
        else Wv = (i128)((int64_t)jc * C + P[i]);
    }
    __device__ __forceinline__ void at(Pos p, i128& Wv, i128& Sv) const {
        vertex(seg[p.k].x, p.r, Wv, Sv);
    }
    // the turn o -> a -> b is strictly left.  Exact: 128-bit products when the
    // differences fit in 64 bits, 256-bit ones otherwise.
    static __device__ __forceinline__ bool turn(i128 Wo, i128 So, i128 Wa, i128 Sa, i128 Wb,
                                                i128 Sb) {
        const i128 w1 = Wa - Wo, s1 = Sa - So, w2 = Wb - Wo, s2 = Sb - So;
        auto fits = [](i128 x) { return (i128)(int64_t)x == x; };
        if (fits(w1) && fits(s1) && fits(w2) && fits(s2))
            return left_turn<true>((int64_t)w1, (int64_t)s1, (int64_t)w2, (int64_t)s2);
        return sign_det128(w1, s2, s1, w2) > 0;
    }
    __device__ __forceinline__ bool left(Pos o, Pos a, Pos b) const {
        i128 Wo, So, Wa, Sa, Wb, Sb;
        at(o, Wo, So); at(a, Wa, Sa); at(b, Wb, Sb);
        return turn(Wo, So, Wa, Sa, Wb, Sb);
    }
};

// A merge's descriptor move: seg[dst + t] = seg[src + t] for t < len (dst < src).
struct Move { int dst, src, len; };

// Merge of the lists of the neighbouring nodes starting at j0 and j1
// (Algorithm 1): finds the bridge, cuts the two segments it lands in, sets the
// merged list's length, and returns the move of the right list's tail.
template <bool WEIGHTED>
__device__ __forceinline__ Move merge_plan(const MStore<WEIGHTED> V, int j0, int j1) {
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
        const int len = kRl - first + 1;
        V.cnt[j0] = nL + len;
        return Move{j0 + nL, first, len};
    }
    // walk from s's neighbours; the two current ends keep their coordinates in
    // registers, so a step reads one new vertex
    Pos a = pa, b = sb;
    i128 Wa, Sa, Wb, Sb;
    V.at(a, Wa, Sa);
    V.at(b, Wb, Sb);
    int steps = 0;
    bool gave_up = false;
    for (;;) {
        bool moved = false;
        while (hasPrev(a)) {
            const Pos p = prev(a);
            i128 Wp, Sp;
            V.at(p, Wp, Sp);
            if (V.turn(Wp, Sp, Wa, Sa, Wb, Sb)) break;
            a = p; Wa = Wp; Sa = Sp; moved = true;
            if (++steps > kWalkCap) { gave_up = true; break; }
        }
        if (gave_up) break;
        while (hasNext(b)) {
            const Pos q = next(b);
            i128 Wq, Sq;
            V.at(q, Wq, Sq);
            if (V.turn(Wa, Sa, Wb, Sb, Wq, Sq)) break;
            b = q; Wb = Wq; Sb = Sq; moved = true;
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
        // tangent point of R seen from a vertex of L: the first vertex after s
        // whose successor lies strictly above the line through it
        auto tangent = [&](Pos ap) -> int {
            int lo = 1, hi = totR - 1;
            while (lo < hi) {
                int mid = (lo + hi) >> 1;
                if (V.left(ap, flatR(mid), flatR(mid + 1))) hi = mid; else lo = mid + 1;
            }
            return lo;
        };
        int lo = 0, hi = totL - 2;   // candidates: every vertex of L before s
        while (lo < hi) {
            int mid = (lo + hi) >> 1;
            const Pos am = flatL(mid);
            // the next vertex of L strictly below the line from am to its tangent: go right
            if (V.left(am, flatL(mid + 1), flatR(tangent(am)))) lo = mid + 1; else hi = mid;
        }
        a = flatL(lo);
        b = flatR(tangent(a));
    }
    // cut L at a and R at b; R's tail moves down behind L's kept part
    seg[a.k].z = a.r;
    seg[b.k].y = b.r;
    const int len = kRl - b.k + 1;
    V.cnt[j0] = (a.k - j0 + 1) + len;
    return Move{a.k + 1, b.k, len};
}

// Exclusive block-wide scan of one 128-bit value per thread (blockDim.x <= 1024).
__device__ __forceinline__ i128 block_excl_scan_i128(i128 v, i128* tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    i128 x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint64_t lo = __shfl_up_sync(kFull, (uint64_t)x, d);
        const uint64_t hi = __shfl_up_sync(kFull, (uint64_t)((unsigned __int128)x >> 64), d);
        if (lane >= d) x += (i128)(((unsigned __int128)hi << 64) | lo);
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        i128 t = lane < (int)(blockDim.x >> 5) ? tmp[lane] : (i128)0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint64_t lo = __shfl_up_sync(kFull, (uint64_t)t, d);
            const uint64_t hi = __shfl_up_sync(kFull, (uint64_t)((unsigned __int128)t >> 64), d);
            if (lane >= d) t += (i128)(((unsigned __int128)hi << 64) | lo);
        }
        tmp[lane] = t;
    }
    __syncthreads();
    const i128 base = warp ? tmp[warp - 1] : (i128)0;
    __syncthreads();
    return base + x - v;
}

template <bool WEIGHTED>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(int64_t m, LongWs ws, uint32_t* __restrict__ row_status) {
    constexpr int C = LongCfg<WEIGHTED>::C;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ i128 s_tmp[32];
    __shared__ int s_qs, s_qw, s_bad;
    __shared__ unsigned long long s_H;
    const int64_t row = blockIdx.x;
    const int64_t c0 = row * m;
    const int tid = threadIdx.x, nth = blockDim.x;
    if (tid == 0) { s_qs = -100000; s_qw = -100000; s_bad = 0; s_H = 0; }
    __syncthreads();
    {
        int qs = -100000, qw = -100000, bad = 0;
        unsigned long long hsum = 0;
        for (int64_t j = tid; j < m; j += nth) {
            const ChunkMeta mt = ws.meta[c0 + j];
            qs = max(qs, mt.qs); qw = max(qw, mt.qw); bad |= mt.bad; hsum += (unsigned)mt.h;
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            qs = max(qs, __shfl_xor_sync(kFull, qs, d));
            qw = max(qw, __shfl_xor_sync(kFull, qw, d));
            bad |= __shfl_xor_sync(kFull, bad, d);
            hsum += __shfl_xor_sync(kFull, hsum, d);
        }
        if ((tid & 31) == 0) {
            atomicMax(&s_qs, qs);
            atomicMax(&s_qw, qw);
            if (bad) atomicOr(&s_bad, bad);
            atomicAdd(&s_H, hsum);
        }
    }
    __syncthreads();
    const int qs = s_qs, qw = s_qw, bad = s_bad;
    const int64_t Htot = (int64_t)s_H;
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

    // ---- shared-memory layout (used only when the whole row fits) ----
    size_t o = 0;
    auto take = [&](size_t bytes, size_t al) {
        o = (o + al - 1) & ~(al - 1);
        const size_t r = o;
        o += bytes;
        return r;
    };
    const size_t oOffS = take(sizeof(i128) * m, 16);
    const size_t oOffW = WEIGHTED ? take(sizeof(i128) * m, 16) : 0;
    const size_t oSeg = take(sizeof(int4) * m, 16);
    const size_t oS = take(sizeof(int64_t) * Htot, 8);
    const size_t oW = WEIGHTED ? take(sizeof(int64_t) * Htot, 8) : 0;
    const size_t oCnt = take(sizeof(int32_t) * m, 4);
    const size_t oPre = take(sizeof(int32_t) * m, 4);
    const size_t oVb = take(sizeof(int32_t) * m, 4);
    const size_t oDS = take(sizeof(int32_t) * m, 4);
    const size_t oDW = WEIGHTED ? take(sizeof(int32_t) * m, 4) : 0;
    const size_t oSegOf = take(sizeof(int32_t) * m, 4);
    const size_t oNext = take(sizeof(int32_t) * m, 4);
    const size_t oPrev = take(sizeof(int32_t) * m, 4);
    const size_t oP = take(sizeof(uint16_t) * Htot, 2);
    const bool in_smem = o <= (size_t)kMergeSmem;

    i128* offS = in_smem ? (i128*)(smem + oOffS) : ws.offS + c0;
    i128* offW = in_smem ? (i128*)(smem + oOffW) : ws.offW + c0;
    int32_t* dS = in_smem ? (int32_t*)(smem + oDS) : ws.dS + c0;
    int32_t* dW = in_smem ? (int32_t*)(smem + oDW) : ws.dW + c0;
    int4* seg = in_smem ? (int4*)(smem + oSeg) : ws.seg + c0;
    int32_t* cnt = in_smem ? (int32_t*)(smem + oCnt) : ws.cnt + c0;
    int32_t* pre = in_smem ? (int32_t*)(smem + oPre) : ws.pre + c0;
    int32_t* segOf = in_smem ? (int32_t*)(smem + oSegOf) : ws.segOf + c0;
    int32_t* nextSeg = in_smem ? (int32_t*)(smem + oNext) : ws.nextSeg + c0;
    int32_t* prevSeg = in_smem ? (int32_t*)(smem + oPrev) : ws.prevSeg + c0;
    int32_t* vb = in_smem ? (int32_t*)(smem + oVb) : nullptr;
    uint16_t* P = in_smem ? (uint16_t*)(smem + oP) : ws.slot_p;
    int64_t* S = in_smem ? (int64_t*)(smem + oS) : ws.slot_S;
    int64_t* W = in_smem ? (int64_t*)(smem + oW) : ws.slot_W;

    // ---- chunk starts in row coordinates and vertex bases: scans over chunks,
    // each thread owning a contiguous range ----
    const int64_t per = (m + nth - 1) / nth;
    const int64_t jb = imin64(m, tid * per), je = imin64(m, jb + per);
    i128 accS = 0, accW = 0, accH = 0;
    for (int64_t j = jb; j < je; ++j) {
        const ChunkMeta mt = ws.meta[c0 + j];
        const int ds = qs - mt.qs, dw = WEIGHTED ? qw - mt.qw : 0;
        dS[j] = ds;
        if (WEIGHTED) dW[j] = dw;
        accS += conv(mt.totS, ds);
        accW += WEIGHTED ? (i128)conv(mt.totW, dw) : (i128)mt.totW;
        accH += mt.h;
    }
    i128 bS = block_excl_scan_i128(accS, s_tmp);
    i128 bW = block_excl_scan_i128(accW, s_tmp);
    i128 bH = block_excl_scan_i128(accH, s_tmp);
    for (int64_t j = jb; j < je; ++j) {
        const ChunkMeta mt = ws.meta[c0 + j];
        offS[j] = bS;
        if (WEIGHTED) offW[j] = bW;
        if (vb) vb[j] = (int32_t)bH;
        bS += conv(mt.totS, dS[j]);
        bW += WEIGHTED ? (i128)conv(mt.totW, dW[j]) : (i128)mt.totW;
        bH += mt.h;
        seg[j] = make_int4((int)j, 0, mt.h - 1, 0);
        cnt[j] = 1;
    }
    __syncthreads();
    if (in_smem) {
        // read every chunk hull of the row once into shared memory; each thread
        // copies a contiguous range of vertices
        const size_t cap = (size_t)C + 1;
        const int64_t pv = (Htot + nth - 1) / nth;
        const int64_t i0 = imin64(Htot, tid * pv), i1 = imin64(Htot, i0 + pv);
        if (i0 < i1) {
            int lo = 0, hi = (int)m - 1;        // chunk holding vertex i0
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (vb[mid] <= i0) lo = mid; else hi = mid - 1;
            }
            int jc = lo;
            int nextb = jc + 1 < m ? vb[jc + 1] : (int)Htot;
#pragma unroll 4
            for (int64_t i = i0; i < i1; ++i) {
                while (i >= nextb) { ++jc; nextb = jc + 1 < m ? vb[jc + 1] : (int)Htot; }
                const size_t g = (size_t)(c0 + jc) * cap + (size_t)(i - vb[jc]);
                P[i] = ws.slot_p[g];
                S[i] = ws.slot_S[g];
                if (WEIGHTED) W[i] = ws.slot_W[g];
            }
        }
    }
    __syncthreads();

    MStore<WEIGHTED> V;
    V.vb = vb; V.P = P; V.S = S; V.W = W;
    V.offS = offS; V.offW = offW; V.dS = dS; V.dW = dW;
    V.seg = seg; V.cnt = cnt; V.pre = pre;
    V.c0 = c0; V.C = C;
    // Levels with many merges run one thread per merge; the others one warp per
    // merge, whose lanes move the descriptors in coalesced rounds of 32
    // (Section 6, "Merge levels").
    const int warp = tid >> 5, wl = tid & 31, nw = nth >> 5;
    for (int r = 0; ((int64_t)1 << r) < m; ++r) {
        const int64_t span = (int64_t)2 << r;
        const int64_t merges = (m + span - 1) / span;
        if (merges >= nw) {
            for (int64_t g = tid; g < merges; g += nth) {
                const int64_t j0 = g * span, j1 = j0 + (span >> 1);
                if (j1 < m) {
                    const Move mv = merge_plan<WEIGHTED>(V, (int)j0, (int)j1);
                    for (int t = 0; t < mv.len; ++t) seg[mv.dst + t] = seg[mv.src + t];
                }
            }
        } else {
            for (int64_t g = warp; g < merges; g += nw) {
                const int64_t j0 = g * span, j1 = j0 + (span >> 1);
                if (j1 >= m) continue;
                Move mv{0, 0, 0};
                if (wl == 0) mv = merge_plan<WEIGHTED>(V, (int)j0, (int)j1);
                mv.dst = __shfl_sync(kFull, mv.dst, 0);
                mv.src = __shfl_sync(kFull, mv.src, 0);
                mv.len = __shfl_sync(kFull, mv.len, 0);
                __syncwarp();
                for (int t0 = 0; t0 < mv.len; t0 += 32) {
                    const int t = t0 + wl;
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

    // ---- ends: each chunk's root segment, and the root vertices around it ----
    const int nroot = cnt[0];
    for (int64_t j = tid; j < m; j += nth) segOf[j] = -1;
    __syncthreads();
    for (int k = tid; k < nroot; k += nth) {
        const int cj = seg[k].x;
        segOf[cj] = k;
        const int cprev = k > 0 ? seg[k - 1].x : -1;
        const int cnext = k + 1 < nroot ? seg[k + 1].x : (int)m;
        for (int q = max(cprev, 0); q < cj; ++q) nextSeg[q] = k;   // chunks in [cprev, cj)
        for (int q = cj + 1; q <= min(cnext, (int)m - 1); ++q) prevSeg[q] = k;
    }
    __syncthreads();
    for (int64_t j = tid; j < m; j += nth) {
        ChunkEnds ce;
        ce.bad = 0;
        const int sk = segOf[j];
        if (sk >= 0) { ce.lo = seg[sk].y; ce.hi = seg[sk].z; }
        else { ce.lo = 1; ce.hi = 0; }
        ce.prevW = ce.prevS = ce.nextW = ce.nextS = 0;
        ce.pt0_vertex = 0;
        if (j > 0) {
            const int pk = prevSeg[j];
            const int pc = seg[pk].x, pr = seg[pk].z;
            V.vertex(pc, pr, ce.prevW, ce.prevS);
            // the previous root vertex is this chunk's first point when it closes chunk j-1
            ce.pt0_vertex = (pc == j - 1 && pr == ws.meta[c0 + pc].h - 1) ? 1 : 0;
        }
        if (j + 1 < m) {
            const int nk = nextSeg[j];
            V.vertex(seg[nk].x, seg[nk].y, ce.nextW, ce.nextS);
        }
        ws.ends[c0 + j] = ce;
        if (in_smem) {
            ws.offS[c0 + j] = offS[j];
            ws.dS[c0 + j] = dS[j];
            if (WEIGHTED) { ws.offW[c0 + j] = offW[j]; ws.dW[c0 + j] = dW[j]; }
        }
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
    static constexpr int kBytes = oSlope + C * 4;
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
    float* slope = reinterpret_cast<float*>(smem + XS::oSlope);   // per point, swizzled rows

    const int64_t c = blockIdx.x;
    const int64_t row = c / m;
    const int64_t j = c - row * m;
    const int64_t e0 = j * C;
    const int nt = (int)imin64(C, n - e0);
    const int tid = threadIdx.x;
    const ChunkEnds ce = ws.ends[c];
    float* orow = out + row * n + e0;
    uint8_t* brow = blocks ? blocks + row * n + e0 : nullptr;
    const bool neg = !increasing;

    if (ce.bad) {
        const float qnan = __int_as_float(0x7fffffff);
        for (int i = tid; i < nt; i += NT) {
            orow[i] = qnan;
            if (brow) brow[i] = 0;
        }
        return;
    }
    const size_t cap = (size_t)C + 1;
    const uint16_t* sp = ws.slot_p + c * cap;
    const int64_t* sS = ws.slot_S + c * cap;
    const int64_t* sW = WEIGHTED ? ws.slot_W + c * cap : nullptr;
    const int qs_row = ws.rowq[row * 4 + 0];
    const int qw_row = WEIGHTED ? ws.rowq[row * 4 + 1] : 0;
    const ChunkMeta mt = ws.meta[c];
    const i128 offS = ws.offS[c];
    const i128 offW = WEIGHTED ? ws.offW[c] : (i128)0;
    const int ds = ws.dS[c], dw = WEIGHTED ? ws.dW[c] : 0;

    s_mask[tid] = 0u;
    __syncthreads();
    auto row_slope = [&](i128 Wa, i128 Sa, i128 Wb, i128 Sb) -> float {
        const double f = i128_to_double(Sb - Sa) / i128_to_double(Wb - Wa);
        return (float)ldexp(f, qs_row - qw_row);
    };
    auto vrow = [&](int r, i128& Wv, i128& Sv) {
        Sv = offS + conv(sS[r], ds);
        if constexpr (WEIGHTED) Wv = offW + conv(sW[r], dw);
        else Wv = (i128)(e0 + sp[r]);
    };
    // root vertices of this chunk that start one of its elements (point < nt),
    // each with the slope of the root edge leaving it
    const bool has = ce.lo <= ce.hi;
    if (has) {
        for (int r = ce.lo + tid; r <= ce.hi; r += NT) {
            const int p = sp[r];
            if (p >= nt) continue;
            atomicOr(&s_mask[p >> 5], 1u << (p & 31));
            float sl;
            if (r < ce.hi) {
                // both ends in the chunk: chunk-relative coordinates, chunk quanta
                const int64_t dS_ = sS[r + 1] - sS[r];
                const int64_t dW_ = WEIGHTED ? sW[r + 1] - sW[r] : (int64_t)(sp[r + 1] - p);
                sl = ldexpf(__ll2float_rn(dS_) / __ll2float_rn(dW_), mt.qs - (WEIGHTED ? mt.qw : 0));
            } else {
                i128 Wa, Sa;
                vrow(r, Wa, Sa);
                sl = row_slope(Wa, Sa, ce.nextW, ce.nextS);
            }
            slope[spos(p >> 5, p & 31)] = sl;
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
        if (ce.pt0_vertex) {
            atomicOr(&s_mask[0], 1u);
            slope[spos(0, 0)] = in_sl;
        }
        s_tmp[NT / 32 + 1] = (int64_t)__float_as_int(in_sl);
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
    const float in_sl = __int_as_float((int)s_tmp[NT / 32 + 1]);
    const float carry = lastv >= 0 ? slope[spos(lastv >> 5, lastv & 31)] : in_sl;
    float o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const uint32_t upto = k == 31 ? mk : (mk & ((2u << k) - 1u));
        const float v = upto ? slope[spos(tid, 31 - __clz(upto))] : carry;
        o[k] = neg ? -v : v;
    }
    __syncthreads();   // slopes read: stage the output in their place
    float4* st4 = reinterpret_cast<float4*>(slope);
#pragma unroll
    for (int q = 0; q < 8; ++q)
        st4[sunit(tid, q)] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    __syncthreads();
    if ((reinterpret_cast<uintptr_t>(orow) & 15u) == 0) {
        const int n4 = nt >> 2;
        for (int i = tid; i < n4; i += NT) {
            const int e4 = i << 2;
            reinterpret_cast<float4*>(orow)[i] = st4[sunit(e4 >> 5, (e4 & 31) >> 2)];
        }
        for (int i = (n4 << 2) + tid; i < nt; i += NT) orow[i] = slope[spos(i >> 5, i & 31)];
    } else {
        for (int i = tid; i < nt; i += NT) orow[i] = slope[spos(i >> 5, i & 31)];
    }
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
    using SM = TileSmem<NT, WEIGHTED, false, 1>;
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
    err = cudaFuncSetAttribute(merge_kernel<WEIGHTED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMergeSmem);
    if (err != cudaSuccess) return err;
    merge_kernel<WEIGHTED><<<(unsigned)rows, kMergeThreads, kMergeSmem, stream>>>(m, ws, row_status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "merge");
    err = cudaFuncSetAttribute(expand_kernel<WEIGHTED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               ExpandSmem<WEIGHTED>::kBytes);
    if (err != cudaSuccess) return err;
    expand_kernel<WEIGHTED><<<(unsigned)M, NT, ExpandSmem<WEIGHTED>::kBytes, stream>>>(
        n, m, increasing, ws, out, blocks);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    prof_mark(stream, "expand");
    return cudaSuccess;
}

cudaError_t long_fit(const float* y, const float* w, int64_t rows, int64_t n, int increasing,
                     float* out, uint8_t* blocks, void* ws, size_t ws_bytes, uint32_t* row_status,
                     cudaStream_t stream) {
    (void)ws_bytes;
    return w ? long_fit_t<true>(y, w, rows, n, increasing, out, blocks, ws, row_status, stream)
             : long_fit_t<false>(y, w, rows, n, increasing, out, blocks, ws, row_status, stream);
}

}  // namespace isodev
