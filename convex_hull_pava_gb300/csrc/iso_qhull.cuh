// Lower hull of a tile by levels of farthest-point splits.
//
// The hull of a tile (Section 3 of the paper: the lower convex hull of the
// cumulative-sum points (W_p, S_p)) is found here without merging lane hulls
// pair by pair.  The tile's first point and its end point are vertices.  At
// each level every chord (a, b) between two consecutive vertices found so far
// takes the point p strictly below it that lies farthest from it, i.e. that
// maximises
//
//     D_p = (W_p - W_a)(S_b - S_a) - (S_p - S_a)(W_b - W_a)   (> 0 below),
//
// ties going to the smallest p.  That point is a vertex of the hull: the line
// through p parallel to the chord has every point of [a, b] on or above it,
// and p is the leftmost point on it.  A point on or above its chord is not a
// vertex of any chord refined below it and is dropped for good; collinear
// points are never chosen, so the hull's vertices are its strict corners
// (Section 4), the same set the merging rounds produce.  The levels end when
// no point is left below any chord.
//
// Only points that are locally convex can be vertices (Lemma 4.1: element
// p - 1's mean below element p's), so the others are dropped before the
// first level.  Every comparison is exact: D is formed from the tile's
// integer coordinates, in 96 bits for unit weights and in 128 bits for
// weighted tiles.
//
// Work per level: each lane evaluates its live points against the chords they
// lie under; a chord whose points all lie in one lane is finished there; a
// chord spanning lanes is reduced by a segmented scan over the lanes (warp
// shuffles), ending at the lane that holds the chord's right vertex.  A row of
// one block is done after one level (every point lies above the chord from
// the first point to the end), where the pairwise merging rounds walk long
// bridges; rows with many blocks need more levels than the merging rounds
// take time, so the callers keep this for rows whose trend runs against the
// fit (few blocks).
#pragma once

#include "iso_device.cuh"

namespace isodev {

// The farthest candidate of a chord so far: D and the point index p (p < 0:
// none).  Unit weights: D = h 2^32 + l with l < 2^32.  Weighted: D = h 2^64 + l.
template <bool WEIGHTED> struct QBest;
template <> struct QBest<false> {
    int64_t h;
    uint32_t l;
    int p;
};
template <> struct QBest<true> {
    int64_t h;
    uint64_t l;
    int p;
};

template <bool WEIGHTED>
__device__ __forceinline__ QBest<WEIGHTED> qnone() {
    QBest<WEIGHTED> b;
    b.h = 0; b.l = 0; b.p = -1;
    return b;
}

// A is a better candidate than B: larger D, then smaller p.
template <bool WEIGHTED>
__device__ __forceinline__ bool qbetter(const QBest<WEIGHTED>& A, const QBest<WEIGHTED>& B) {
    if (A.p < 0) return false;
    if (B.p < 0) return true;
    if (A.h != B.h) return A.h > B.h;
    if (A.l != B.l) return A.l > B.l;
    return A.p < B.p;
}

template <bool WEIGHTED>
__device__ __forceinline__ QBest<WEIGHTED> qmax(const QBest<WEIGHTED>& A, const QBest<WEIGHTED>& B) {
    return qbetter<WEIGHTED>(A, B) ? A : B;
}

template <bool WEIGHTED>
__device__ __forceinline__ QBest<WEIGHTED> qshfl_up(const QBest<WEIGHTED>& v, int d) {
    QBest<WEIGHTED> r;
    r.h = __shfl_up_sync(kFull, v.h, d);
    r.l = __shfl_up_sync(kFull, v.l, d);
    r.p = __shfl_up_sync(kFull, v.p, d);
    return r;
}

// D of point (Wp, Sp) against the chord from (Wa, Sa) with differences (dW, dS),
// and whether it is > 0.  Unit weights: W differences are point counts below
// 2^14 and S differences below 2^63, so D = h 2^32 + l with two 32 x 32-bit
// products per term.
__device__ __forceinline__ bool qdist(int w1, int64_t s1, int dW, int64_t dS, QBest<false>& b) {
    const int64_t hi = (int64_t)w1 * (int32_t)(dS >> 32) - (int64_t)dW * (int32_t)(s1 >> 32);
    const int64_t lo = (int64_t)w1 * (int64_t)(uint32_t)dS - (int64_t)dW * (int64_t)(uint32_t)s1;
    b.h = hi + (lo >> 32);
    b.l = (uint32_t)lo;
    return b.h > 0 || (b.h == 0 && b.l != 0u);
}
__device__ __forceinline__ bool qdist(int64_t w1, int64_t s1, int64_t dW, int64_t dS, QBest<true>& b) {
    const __int128 d = (__int128)w1 * (__int128)dS - (__int128)s1 * (__int128)dW;
    b.h = (int64_t)(d >> 64);
    b.l = (uint64_t)d;
    return d > 0;
}

// Levels of kQuickLevels at most; a tile that needs more falls back to the
// merging rounds.
constexpr int kQuickLevels = 24;

// The levels, run by each warp on its own (no barrier of the CTA): the lanes of
// a warp form sub-tiles of SL = min(L, 32) lanes (a whole tile when L <= 32),
// each with its first point and its end point as vertices.  The warp keeps
// splitting until none of its sub-tiles has a point below a chord.  Chord ends
// are found by ballots and shuffles; the segmented scan's restarts come from a
// ballot.  On return T.mask holds the vertices of every sub-tile's hull.
// Returns false on every lane of the warp when some sub-tile needed more than
// kQuickLevels levels.
template <bool WEIGHTED>
__device__ bool warp_quickhull(const Tile& T, int lane, int L, int e, bool work, uint32_t cand) {
    using QB = QBest<WEIGHTED>;
    using WT = typename std::conditional<WEIGHTED, int64_t, int>::type;
    const int wl = threadIdx.x & 31;
    const int SL = L < 32 ? L : 32;
    const int wfirst = wl & ~(SL - 1), wlast = wfirst + SL - 1;
    const int lane0 = lane - wl;                       // tile lane of the warp's lane 0
    const int base = lane << 5;
    const int P1 = min((lane - (wl - wfirst) + SL) << 5, T.nt);   // end point of the sub-tile
    const uint32_t sub = (SL == 32 ? 0xffffffffu : ((1u << SL) - 1u)) << wfirst;
    const uint32_t lanebits = e >= 32 ? 0xffffffffu : ((1u << e) - 1u);
    const bool firstlane = wl == wfirst;
    uint32_t vm = (work && firstlane && e > 0) ? 1u : 0u;   // the sub-tile's first point
    uint32_t live = work ? (cand | 1u) & lanebits & ~vm : 0u;
    T.mask[lane] = vm;
    auto Wof = [&](int p) -> WT {
        if constexpr (WEIGHTED) return tile_W<true>(T, p); else return (WT)p;
    };
    bool done = false;
    for (int level = 0; level <= kQuickLevels; ++level) {
        __syncwarp();
        vm = T.mask[lane];
        live &= ~vm;
        if (!__any_sync(kFull, live != 0u)) { done = true; break; }
        if (level == kQuickLevels) break;
        // chord ends around the lane: the last vertex of an earlier lane of the
        // sub-tile and the first vertex of a later one (else the sub-tile's end)
        const uint32_t bal = __ballot_sync(kFull, vm != 0u);
        const int hv = vm ? 31 - __clz(vm) : 0;
        const int lv = vm ? __ffs(vm) - 1 : 0;
        const uint32_t before = bal & sub & ((1u << wl) - 1u);
        const uint32_t after = bal & sub & (wl == 31 ? 0u : ~((2u << wl) - 1u));
        const int qb = before ? 31 - __clz(before) : wl;
        const int qa = after ? __ffs(after) - 1 : wl;
        const int hvq = __shfl_sync(kFull, hv, qb);
        const int lvq = __shfl_sync(kFull, lv, qa);
        const int pa = ((lane0 + qb) << 5) + hvq;
        const int nb = after ? ((lane0 + qa) << 5) + lvq : P1;

        // ---- evaluate the lane's live points, chord by chord ----
        QB F = qnone<WEIGHTED>(), Lst = qnone<WEIGHTED>();
        uint32_t newv = 0u, dead = 0u;
        if (live) {
            int a = (vm & 1u) ? base : pa;
            uint32_t vrest = vm & ~1u;
            bool first = !(vm & 1u);
            int64_t Sa = tile_S<WEIGHTED>(T, a);
            WT Wa = Wof(a);
            for (;;) {
                const int b = vrest ? base + __ffs(vrest) - 1 : nb;
                const int lo = a + 1 - base, hi = b - base;
                uint32_t seg = live;
                if (lo > 0) seg &= lo >= 32 ? 0u : ~((1u << lo) - 1u);
                if (hi < 32) seg &= hi <= 0 ? 0u : ((1u << hi) - 1u);
                const bool last = vrest == 0u;
                int64_t Sb = 0;
                WT Wb = 0;
                if (seg || !last) { Sb = tile_S<WEIGHTED>(T, b); Wb = Wof(b); }
                QB best = qnone<WEIGHTED>();
                if (seg) {
                    const int64_t dS = Sb - Sa;
                    const WT dW = Wb - Wa;
                    const int64_t* row = T.Sx + lane * kRow;
                    uint32_t m = seg;
                    while (m) {
                        const int k = __ffs(m) - 1;
                        m &= m - 1u;
                        QB c;
                        if (!qdist(Wof(base + k) - Wa, row[k] - Sa, dW, dS, c)) { dead |= 1u << k; continue; }
                        c.p = base + k;
                        if (qbetter<WEIGHTED>(c, best)) best = c;
                    }
                }
                if (first) F = best;
                if (last) {
                    if (!first) Lst = best;
                } else if (!first && best.p >= 0) {
                    newv |= 1u << (best.p - base);
                }
                if (last) break;
                a = b; Sa = Sb; Wa = Wb;
                vrest &= vrest - 1u;
                first = false;
            }
        }
        live &= ~dead;

        // ---- chords spanning lanes: segmented scan over the warp, restarting
        // at lanes that hold a vertex and at each sub-tile's first lane ----
        const bool rs = vm != 0u || firstlane;
        const uint32_t rb = __ballot_sync(kFull, rs);
        QB v = vm != 0u ? Lst : F;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const QB o = qshfl_up<WEIGHTED>(v, d);
            // combine while no lane in (wl - d, wl] restarts
            const uint32_t span = wl >= d ? (((2u << wl) - 1u) & ~((2u << (wl - d)) - 1u)) : 0u;
            if (wl >= d && !(rb & span)) v = qmax<WEIGHTED>(o, v);
        }
        QB prev = qshfl_up<WEIGHTED>(v, 1);
        if (firstlane) prev = qnone<WEIGHTED>();
        __syncwarp();
        if (newv) atomicOr(&T.mask[lane], newv);
        if (vm != 0u) {
            const QB fin = qmax<WEIGHTED>(prev, F);
            if (fin.p >= 0) atomicOr(&T.mask[fin.p >> 5], 1u << (fin.p & 31));
        }
        if (wl == wlast && v.p >= 0) atomicOr(&T.mask[v.p >> 5], 1u << (v.p & 31));
    }
    return done;
}

// The hull of every tile of the CTA (tiles of L <= 32 lanes, inside one warp)
// by the levels above; the non-empty-lane bits summ are rebuilt for the
// callers.  Returns false (on every thread) when some tile needed more than
// kQuickLevels levels.  Every thread of the CTA calls it.
template <bool WEIGHTED>
__device__ bool tile_quickhull(const Tile& T, uint32_t* summ, int lane, int L, int e, bool work,
                               uint32_t cand) {
    const bool ok = warp_quickhull<WEIGHTED>(T, lane, L, e, work, cand);
    if (!__syncthreads_and(ok)) return false;
    const uint32_t bal = __ballot_sync(kFull, T.mask[lane] != 0u);
    if ((threadIdx.x & 31) == 0) summ[threadIdx.x >> 5] = bal;
    __syncthreads();
    return true;
}

}  // namespace isodev
