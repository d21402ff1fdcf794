// Candidate filter and list hull for the chunks of long rows (unit weights,
// float32 input).
//
// A point p can be a vertex of the lower hull only if it lies strictly below
// the segment between any two other points a < p < b of the same set (a strict
// vertex has a supporting line with every other point above it).  Lemma 4.1 of
// the paper applies this to a = p - 1, b = p + 1.  Here it is applied with
// points a few dozen elements away, which removes far more on noisy data:
//
//   * after a shear of the diagram by the chunk's mean value (the shear adds
//     the same linear function to every point and changes no turn), the
//     chunk's lowest point g: the chord from the chunk's first point to g and
//     the chord from g to the chunk's end;
//   * for a point of lane l, the lowest points of lanes l - 1, l and l + 1.
//
// The tests run in float32 on sheared prefix sums formed from the staged
// values; a point is dropped only when its float32 test exceeds a bound on
// the float32 rounding error of the quantities involved (derived below), so
// no vertex of the exact hull is ever dropped.  On noisy chunks of 4,096
// elements about 50 of some 2,000 locally convex points survive (170 at the
// most in a sample of 200 chunks), against about 10 hull vertices.
//
// The survivors, with the chunk's first point and end point, are then laid out
// as a list and one warp finds their hull exactly by levels of farthest-point
// splits (the same levels as iso_qhull.cuh, over list entries): the hull of a
// subset of the points that contains every vertex of their hull is that hull.
#pragma once

#include "iso_qhull.cuh"

namespace isodev {

constexpr int kListCap = 512;   // list entries (survivors + the two ends) for the list hull

// Bound on the float32 rounding of the sheared diagram of one lane.  With the
// shear constant c (a float) and the quantum s = 2^q, the exact sheared value
// at the lane's point k is
//     F_k = S_{32l} s - c 32 l + sum_{j<k} (v_j - c),
// v_j the quantised value (|v_j - y_j| <= s/2, y_j the staged float).  The
// lane computes f_0 = G = fl(fl(S_{32l}) s - c 32 l) and
// f_{k+1} = fl(f_k + fl(y_k - c)), where fl(S_{32l}) comes from two 32-bit
// conversions and one fused multiply-add (within 1.5 ulp) and the scaling by
// s is exact.  Each other float operation errs by at most 2^-24 of its
// result, so |f_k - F_k| <= 2^-22 |S_{32l} s| + 2^-24 (|c 32 l| + |G|) +
// sum_j (s/2 + 2^-24 |d_j| + 2^-24 |f_{j+1}|) with d_j = fl(y_j - c).  The
// lane's bound doubles that total (covering the rounding of the bound itself).
//
// A test "p strictly above the segment from x to z" (x < p < z) uses the
// segment's float slope sigma = fl(fl(f_z - f_x) / (z - x)) and intercept
// beta = fl(f_x - sigma x) (one fused multiply-add), the line's value at p
// l = fl(sigma p + beta) (another) and t = fl(f_p - l).  With F the exact
// sheared values, Sigma = (F_z - F_x) / (z - x) and Lambda = F_x + Sigma (p - x):
//   |sigma - Sigma| <= (d_x + d_z + 2^-23 |f_z - f_x|) / (z - x),
//   |l - Lambda|    <= 2 d_x + d_z + 2^-23 |f_z - f_x| + 2^-24 (|beta| + |l|),
//   |t - T|         <= d_p + |l - Lambda| + 2^-24 |t|,   T = F_p - Lambda,
// d the bounds of the three points (p - x <= z - x).  With |l| <= F and
// |t| <= 2 F, F the largest |f| of the lane and of the two ends, p is dropped
// when t exceeds the per-segment constant
//   M = (d_p + 2 d_x + d_z + 2^-23 |f_z - f_x| + 2^-24 |beta| + 2^-22 F)(1 + 2^-20):
// then T >= t - |t - T| > 0, p lies strictly above the exact segment.
struct FSeg {
    float sigma, beta, M;
};

__device__ __forceinline__ FSeg fseg(int x, float fx, float dx, int z, float fz, float dz, float dp,
                                     float F) {
    FSeg r;
    const float num = fz - fx;
    r.sigma = num / (float)(z - x);
    r.beta = fmaf(-r.sigma, (float)x, fx);
    const float Fm = fmaxf(F, fmaxf(fabsf(fx), fabsf(fz)));
    r.M = (dp + 2.0f * dx + dz + 0x1p-23f * fabsf(num) + 0x1p-24f * fabsf(r.beta) + 0x1p-22f * Fm) *
          (1.0f + 0x1p-20f);
    if (!(r.M < 1.0e37f)) r.M = __int_as_float(0x7f800000);   // inf or nan: nothing is dropped
    return r;
}

// Filter of the candidates of every lane of a chunk tile (one tile of L = NT
// lanes).  yv: the lane's staged values (negated for a decreasing fit); e: its
// elements; LS: lane starts (tile-relative, quanta 2^q); cand: Lemma 4.1's
// locally convex points (bits 1 .. e-1).  Returns cand with bit 0 (the lane's
// first point, tested too when lane > 0) and with the points that fail a test
// removed.  Chunks whose quantum is outside float32's normal range keep every
// candidate.  xch: shared scratch of 3 NT + 3 NT / 32 words.  Every thread calls it.
template <int NT>
__device__ uint32_t chunk_filter(const float (&yv)[32], int e, int lane, int nt, int q,
                                 const int64_t* LS, uint32_t cand, float* xch) {
    const int L = NT;
    uint32_t keep = e > 0 ? (cand | (lane > 0 ? 1u : 0u)) : 0u;
    keep &= e >= 32 ? 0xffffffffu : ((1u << e) - 1u);
    if (q < -100 || q > 100) return keep;                     // uniform over the tile
    const float sc = __int_as_float((q + 127) << 23);         // 2^q, exact
    const float tot = i64_to_f32(LS[L]) * sc;
    const float c = tot / (float)(nt > 0 ? nt : 1);           // the shear (any constant works)
    float G, err;
    {
        const float Sl = i64_to_f32(LS[lane]) * sc;
        const float cl = c * (float)(lane << 5);               // rounded: within 2^-24 |cl|
        G = Sl - cl;
        err = 0x1p-22f * fabsf(Sl) + 0x1p-24f * (fabsf(cl) + fabsf(G));
    }
    const float fend = tot - c * (float)nt;
    const float dend = 2.0f * (0x1p-22f * fabsf(tot) + 0x1p-24f * (fabsf(c * (float)nt) + fabsf(fend)));
    float f = G, fmin = G, fabsmax = fabsf(G);
    int kmin = 0;
    const float half_q = 0.5f * sc;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        if (k < e) {
            const float d = yv[k] - c;
            f = f + d;
            err += half_q + 0x1p-24f * (fabsf(d) + fabsf(f));
            fabsmax = fmaxf(fabsmax, fabsf(f));
            if (k + 1 < e && f < fmin) { fmin = f; kmin = k + 1; }
        }
    }
    float delta = 2.0f * err;
    if (!(delta < 1.0e37f)) delta = 1.0e37f;                  // inf or nan: the tests fail, nothing is dropped
    // every lane's lowest point, for its neighbours; each warp's lowest point
    // (smallest f, then smallest index), for the chunk's lowest
    int* xp = reinterpret_cast<int*>(xch);
    float* xf = xch + NT;
    float* xd = xch + 2 * NT;
    xp[lane] = e > 0 ? (lane << 5) + kmin : -1;
    xf[lane] = fmin;
    xd[lane] = delta;
    {
        float wf = e > 0 ? fmin : __int_as_float(0x7f800000);
        int wp = e > 0 ? (lane << 5) + kmin : 0x7fffffff;
        float wd = delta;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float of = __shfl_xor_sync(kFull, wf, d);
            const int op = __shfl_xor_sync(kFull, wp, d);
            const float od = __shfl_xor_sync(kFull, wd, d);
            if (of < wf || (of == wf && op < wp)) { wf = of; wp = op; wd = od; }
        }
        if ((threadIdx.x & 31) == 0) {
            xch[3 * NT + 3 * (threadIdx.x >> 5)] = wf;
            reinterpret_cast<int*>(xch)[3 * NT + 3 * (threadIdx.x >> 5) + 1] = wp;
            xch[3 * NT + 3 * (threadIdx.x >> 5) + 2] = wd;
        }
    }
    __syncthreads();
    // the chunk's lowest sheared point g (a point of the chunk; the two chords
    // through it replace the chunk's own chord)
    float fg = xch[3 * NT];
    int g = reinterpret_cast<const int*>(xch)[3 * NT + 1];
    float dg = xch[3 * NT + 2];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w) {
        const float of = xch[3 * NT + 3 * w];
        const int op = reinterpret_cast<const int*>(xch)[3 * NT + 3 * w + 1];
        if (of < fg || (of == fg && op < g)) { fg = of; g = op; dg = xch[3 * NT + 3 * w + 2]; }
    }
    if (g > nt) { g = 0; fg = 0.0f; dg = 0.0f; }          // no finite point: point 0 (nothing drops)
    // the anchors around this lane: the previous lane's lowest point (point 0,
    // f = 0 exactly, for lane 0) and the next lane's (the end point after the
    // last lane with elements)
    int pa = 0;
    float fa = 0.0f, da = 0.0f;
    if (lane > 0) { pa = xp[lane - 1]; fa = xf[lane - 1]; da = xd[lane - 1]; }
    int pb = nt;
    float fb = fend, db = dend;
    if (lane + 1 < L && xp[lane + 1] >= 0) { pb = xp[lane + 1]; fb = xf[lane + 1]; db = xd[lane + 1]; }
    const int pm = (lane << 5) + kmin;
    const FSeg left = fseg(pa, fa, da, pm, fmin, delta, delta, fabsmax);    // points before the lowest
    const FSeg right = fseg(pm, fmin, delta, pb, fb, db, delta, fabsmax);   // points after it
    const FSeg mid = fseg(pa, fa, da, pb, fb, db, delta, fabsmax);          // the lowest point itself
    const FSeg gl = fseg(0, 0.0f, 0.0f, g, fg, dg, delta, fabsmax);         // chord from point 0 to g
    const FSeg gr = fseg(g, fg, dg, nt, fend, dend, delta, fabsmax);        // chord from g to the end
    // Every point's tests as bit masks (against the chord before the lane's
    // lowest point, the chord after it, and the chunk chord on its side of g),
    // combined once per lane: the same tests, on the same values, as choosing
    // each point's chords one by one.
    const int gk = g - (lane << 5);                        // g's position in this lane
    const FSeg ga = gk > 0 ? gl : gr;                      // the chunk chord of most of the lane
    uint32_t dL = 0u, dR = 0u, dG = 0u;
    f = G;
    float pf = (float)(lane << 5);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const float tl = f - fmaf(left.sigma, pf, left.beta);
        const float tr = f - fmaf(right.sigma, pf, right.beta);
        const float tg = f - fmaf(ga.sigma, pf, ga.beta);
        if (tl > left.M) dL |= 1u << k;
        if (tr > right.M) dR |= 1u << k;
        if (tg > ga.M) dG |= 1u << k;
        if (k < e) f = f + (yv[k] - c);
        pf += 1.0f;
    }
    // before the lowest point the left chord, after it the right one
    uint32_t drop = (dL & ((1u << kmin) - 1u)) | (dR & ~((2u << kmin) - 1u));
    // the lowest point against the chord between the neighbours' lowest points
    if (fmin - fmaf(mid.sigma, (float)pm, mid.beta) > mid.M) drop |= 1u << kmin;
    // the chunk chord on each point's side of g (g itself takes neither)
    const uint32_t sideA = gk > 0 ? (gk >= 32 ? 0xffffffffu : (1u << gk) - 1u)
                                  : (gk < 0 ? 0xffffffffu : ~1u);
    drop |= dG & sideA;
    if (gk > 0 && gk < 31) {
        // g's lane: its points after g against the chord from g to the end
        uint32_t d2 = 0u;
        f = G;
        pf = (float)(lane << 5);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const float t = f - fmaf(gr.sigma, pf, gr.beta);
            if (t > gr.M) d2 |= 1u << k;
            if (k < e) f = f + (yv[k] - c);
            pf += 1.0f;
        }
        drop |= d2 & ~((2u << gk) - 1u);
    }
    return keep & ~drop;
}

// Whether entry t of a sorted list (entries lo..hi, lo <= t <= hi) is a strict
// corner of their lower hull: lo and hi are; an entry between them is when
// the largest slope into it from the left (over entries lo..t-1) is below the
// smallest slope out of it to the right (over t+1..hi), i.e. it lies strictly
// below the segment between the two entries that attain them.  With w = |P_j -
// P_t| and s = S_t - S_j for another entry j, the slope in is the largest s / w
// over j < t and the slope out the smallest -s / w over j > t, i.e. again the
// largest s / w: one running best per side, compared exactly by cross
// products (w below 2^13, |s| below 2^63).  R threads per entry, neighbours in
// a warp, each taking a share (sub) of the others, their bests combined by
// shuffles; every thread of the warp calls it; the result is valid on sub 0.
__device__ __forceinline__ bool list_corner(const uint16_t* P, const int64_t* S, int t, bool act, int lo,
                                            int hi, int R, int sub) {
    // the running bests (entry, w, s) of this thread's share
    int bl = lo, br = hi, wl = 1, wr = 1;
    int64_t sl = 0, sr = 0;
    const bool mine = act && t > lo && t < hi;
    int Pt = 0;
    int64_t St = 0;
    if (mine) {
        Pt = P[t];
        St = S[t];
        wl = Pt - P[lo]; sl = St - S[lo];
        wr = P[hi] - Pt; sr = St - S[hi];
        const int span = (hi - lo - 1 + R - 1) / R;
        const int j0 = lo + 1 + sub * span, j1 = min(hi, j0 + span);
        for (int j = j0; j < j1; ++j) {
            const int w0 = P[j] - Pt;
            const int64_t sv = St - S[j];
            const bool left = j < t;
            const int w = left ? -w0 : w0;
            const int wb = left ? wl : wr;
            const int64_t sb = left ? sl : sr;
            // sv / w > sb / wb  <=>  wb sv - w sb > 0 (w, wb > 0)
            const bool better = j != t && left_turn_w32(wb, sb, w, sv);
            if (better && left) { bl = j; wl = w; sl = sv; }
            if (better && !left) { br = j; wr = w; sr = sv; }
        }
    }
    // the shares' bests combined (lanes of one entry are neighbours in a warp)
    for (int d = 1; d < R; d <<= 1) {
        const int obl = __shfl_xor_sync(kFull, bl, d), owl = __shfl_xor_sync(kFull, wl, d);
        const int64_t osl = __shfl_xor_sync(kFull, sl, d);
        const int obr = __shfl_xor_sync(kFull, br, d), owr = __shfl_xor_sync(kFull, wr, d);
        const int64_t osr = __shfl_xor_sync(kFull, sr, d);
        if (left_turn_w32(wl, sl, owl, osl)) { bl = obl; wl = owl; sl = osl; }
        if (left_turn_w32(wr, sr, owr, osr)) { br = obr; wr = owr; sr = osr; }
    }
    return act && (t == lo || t == hi ||
                   (mine && left_turn_w32(Pt - P[bl], St - S[bl], P[br] - P[bl], S[br] - S[bl])));
}

// Threads per entry for a pass over n entries by NT threads (a power of two,
// at most 32, R n <= NT).
template <int NT>
__device__ __forceinline__ int list_threads_per_entry(int n) {
    int R = 1;
    while (R < 32 && 2 * R * n <= NT) R <<= 1;
    return R;
}

constexpr int kListBlock = 16;      // entries per block of the first pass
constexpr int kListTwoPass = 32;    // longer lists take the first pass
// bytes of cta_list_hull's scratch for NT threads
__host__ __device__ constexpr int list_scratch_bytes(int nt) { return 13 * nt + 16; }

// Lower hull of the n <= NT entries of a list by the CTA: entry i is the point
// with index P[i] (increasing) and tile-relative sum S[i]; entries 0 and n - 1
// are vertices.  An entry is a vertex when no other entry lies on or below the
// line through it with a slope between its in and out slopes: the pairwise
// test of list_corner over all entries.  A list of more than kListTwoPass
// entries first keeps only the corners of its blocks of kListBlock entries (a
// vertex of the whole list's hull is one of the hull of any block holding it),
// then tests the survivors against each other: the same vertices, with far
// fewer pairs.  On return bit t % K of vm[t / K] is set for each vertex t < n - 1,
// K = ceil((n - 1) / 32).  scratch: list_scratch_bytes(NT) bytes of shared
// memory, 8-byte aligned.  Every thread of the CTA calls it.
template <int NT>
__device__ __forceinline__ void cta_list_hull(const uint16_t* P, const int64_t* S, int n, uint32_t* vm,
                                              unsigned char* scratch) {
    const int tid = threadIdx.x;
    if (tid < 32) vm[tid] = 0u;
    const int K = (n - 1 + 31) >> 5;
    const uint16_t* P2 = P;
    const int64_t* S2 = S;
    const uint16_t* Q = nullptr;       // survivor i is entry Q[i]
    int m = n;
    if (n > kListTwoPass) {
        uint16_t* qP = reinterpret_cast<uint16_t*>(scratch);
        uint16_t* qQ = qP + NT;
        int64_t* qS = reinterpret_cast<int64_t*>(scratch + 4 * NT);
        uint8_t* keep = scratch + 12 * NT;
        int* s_m = reinterpret_cast<int*>(scratch + 13 * NT);
        const int R = list_threads_per_entry<NT>(n);
        const int t = tid / R, sub = tid % R;
        const int lo = (t / kListBlock) * kListBlock;
        const int hi = min(lo + kListBlock - 1, n - 1);
        const bool c = list_corner(P, S, t, t < n, lo, hi, R, sub);
        if (sub == 0 && t < n) keep[t] = c ? 1 : 0;
        __syncthreads();
        if (tid < 32) {
            int base = 0;
            for (int q = 0; q < n; q += 32) {
                const int u = q + tid;
                const bool k = u < n && keep[u];
                const unsigned b = __ballot_sync(kFull, k);
                if (k) {
                    const int i = base + __popc(b & ((1u << tid) - 1u));
                    qQ[i] = (uint16_t)u;
                    qP[i] = P[u];
                    qS[i] = S[u];
                }
                base += __popc(b);
            }
            if (tid == 0) *s_m = base;
        }
        __syncthreads();
        m = *s_m;
        P2 = qP; S2 = qS; Q = qQ;
    } else {
        __syncthreads();
    }
    const int R = list_threads_per_entry<NT>(m);
    const int t = tid / R, sub = tid % R;
    const bool c = list_corner(P2, S2, t, t < m, 0, m - 1, R, sub);
    if (sub == 0 && t < m - 1 && c) {
        const int o = Q ? (int)Q[t] : t;
        atomicOr(&vm[o / K], 1u << (o % K));
    }
    __syncthreads();
}

// Lower hull of the entries of a list by one warp: entry i is the point with
// index P[i] (increasing) and tile-relative sum S[i]; entries 0 and n - 1 are
// vertices.  Lane l holds entries [l K, l K + K) of the n - 1 before the last,
// K = ceil((n - 1) / 32) <= 32.  The levels of farthest-point splits of
// iso_qhull.cuh, over entries.  On return vm[l] (shared) holds lane l's vertex
// bits; returns false (on every lane) when more than kQuickLevels levels were
// needed.
__device__ __noinline__ inline bool warp_list_hull(const uint16_t* P, const int64_t* S, int n, uint32_t* vm_sm) {
    using QB = QBest<false>;
    const int wl = threadIdx.x & 31;
    const int K = (n - 1 + 31) >> 5;
    const int base = wl * K;
    const int e = max(0, min(K, n - 1 - base));
    const uint32_t lanebits = e >= 32 ? 0xffffffffu : ((1u << e) - 1u);
    uint32_t vm = wl == 0 ? 1u : 0u;
    uint32_t live = lanebits & ~vm;
    vm_sm[wl] = vm;
    bool done = false;
    for (int level = 0; level <= kQuickLevels; ++level) {
        __syncwarp();
        vm = vm_sm[wl];
        live &= ~vm;
        if (!__any_sync(kFull, live != 0u)) { done = true; break; }
        if (level == kQuickLevels) break;
        const uint32_t bal = __ballot_sync(kFull, vm != 0u);
        const int hv = vm ? 31 - __clz(vm) : 0;
        const int lv = vm ? __ffs(vm) - 1 : 0;
        const uint32_t before = bal & ((1u << wl) - 1u);
        const uint32_t after = bal & (wl == 31 ? 0u : ~((2u << wl) - 1u));
        const int qb = before ? 31 - __clz(before) : wl;
        const int qa = after ? __ffs(after) - 1 : wl;
        const int hvq = __shfl_sync(kFull, hv, qb);
        const int lvq = __shfl_sync(kFull, lv, qa);
        const int ia = qb * K + hvq;
        const int ib = after ? qa * K + lvq : n - 1;

        QB F = qnone<false>(), Lst = qnone<false>();
        uint32_t newv = 0u, dead = 0u;
        if (live) {
            int a = (vm & 1u) ? base : ia;
            uint32_t vrest = vm & ~1u;
            bool first = !(vm & 1u);
            int64_t Sa = S[a];
            int Wa = P[a];
            for (;;) {
                const int b = vrest ? base + __ffs(vrest) - 1 : ib;
                const int lo = a + 1 - base, hi = b - base;
                uint32_t seg = live;
                if (lo > 0) seg &= lo >= 32 ? 0u : ~((1u << lo) - 1u);
                if (hi < 32) seg &= hi <= 0 ? 0u : ((1u << hi) - 1u);
                const bool last = vrest == 0u;
                int64_t Sb = 0;
                int Wb = 0;
                if (seg || !last) { Sb = S[b]; Wb = P[b]; }
                QB best = qnone<false>();
                if (seg) {
                    const int64_t dS = Sb - Sa;
                    const int dW = Wb - Wa;
                    uint32_t m = seg;
                    while (m) {
                        const int k = __ffs(m) - 1;
                        m &= m - 1u;
                        QB c;
                        if (!qdist(P[base + k] - Wa, S[base + k] - Sa, dW, dS, c)) { dead |= 1u << k; continue; }
                        c.p = base + k;
                        if (qbetter<false>(c, best)) best = c;
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
        const bool rs = vm != 0u || wl == 0;
        const uint32_t rb = __ballot_sync(kFull, rs);
        QB v = vm != 0u ? Lst : F;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const QB o = qshfl_up<false>(v, d);
            const uint32_t span = wl >= d ? (((2u << wl) - 1u) & ~((2u << (wl - d)) - 1u)) : 0u;
            if (wl >= d && !(rb & span)) v = qmax<false>(o, v);
        }
        QB prev = qshfl_up<false>(v, 1);
        if (wl == 0) prev = qnone<false>();
        __syncwarp();
        if (newv) atomicOr(&vm_sm[wl], newv);
        if (vm != 0u) {
            const QB fin = qmax<false>(prev, F);
            if (fin.p >= 0) atomicOr(&vm_sm[fin.p / K], 1u << (fin.p % K));
        }
        if (wl == 31 && v.p >= 0) atomicOr(&vm_sm[v.p / K], 1u << (v.p % K));
    }
    return done;
}

}  // namespace isodev
