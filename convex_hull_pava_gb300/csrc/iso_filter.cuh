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
// A test "p strictly above the segment from x to z" computes
//     t = (f_p - f_x)(z - x) - (f_z - f_x)(p - x)
// in float32 and drops p only when t exceeds
//     m = (d_p + d_x)(z - x) + (d_z + d_x)(p - x) + 2^-21 (|f_p - f_x| (z - x) + |f_z - f_x| (p - x)),
// d the bounds of the three points: the first two terms bound the effect of the
// values' errors, the last the rounding of t's own operations (at most four
// roundings of 2^-24 of terms of those sizes).  With point indices exact in
// float (below 2^24), t and m are formed for each side of the lane's lowest
// point from per-lane constants: t = (z - x) f_p - (f_z - f_x) p - k0 and m =
// m0 + m1 p + 2^-21 (z - x) |f_p - f_x|.
struct FSide {
    float w, a, k0, fx, m0, m1;   // segment from x to z: w = z - x, a = f_z - f_x
    float kabs;                   // |w f_x| + |a x|: the size of k0's terms
};

__device__ __forceinline__ FSide side(int x, float fx, float dx, int z, float fz, float dz, float dp) {
    FSide r;
    r.w = (float)(z - x);
    r.a = fz - fx;
    r.fx = fx;
    // t = w (f_p - f_x) - a (p - x) = w f_p - a p - (w f_x - a x)
    r.k0 = fmaf(r.w, fx, -r.a * (float)x);
    r.kabs = fabsf(r.w * fx) + fabsf(r.a * (float)x);
    // m = (dp + dx) w + (dz + dx)(p - x) + 2^-21 (w |f_p - f_x| + |a| (p - x))
    const float g = dz + dx + 0x1p-21f * fabsf(r.a);
    r.m1 = g;
    r.m0 = (dp + dx) * r.w - g * (float)x;
    return r;
}

// p (index pf as a float, sheared value fp) is strictly above the side's segment
// beyond the rounding bound (the bound is inflated by 2^-20 of itself and of the
// sizes of t's terms, for the rounding of t, k0 and m's own arithmetic).
__device__ __forceinline__ bool fabove(float w, float a, float k0, float fx, float m0, float m1,
                                       float kabs, float pf, float fp) {
    const float t = fmaf(w, fp, -fmaf(a, pf, k0));
    const float m = fmaf(m1, pf, m0) + 0x1p-21f * w * fabsf(fp - fx);
    return t > m * (1.0f + 0x1p-20f) + 0x1p-20f * (fabsf(w * fp) + fabsf(a * pf) + kabs);
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
    float f = G, fmin = G;
    int kmin = 0;
    const float half_q = 0.5f * sc;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        if (k < e) {
            const float d = yv[k] - c;
            f = f + d;
            err += half_q + 0x1p-24f * (fabsf(d) + fabsf(f));
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
    const FSide left = side(pa, fa, da, pm, fmin, delta, delta);    // points before the lowest
    const FSide right = side(pm, fmin, delta, pb, fb, db, delta);   // points after it
    const FSide mid = side(pa, fa, da, pb, fb, db, delta);          // the lowest point itself
    const FSide gl = side(0, 0.0f, 0.0f, g, fg, dg, delta);         // chord from point 0 to g
    const FSide gr = side(g, fg, dg, nt, fend, dend, delta);        // chord from g to the end
    uint32_t drop = 0u;
    f = G;
    float pf = (float)(lane << 5);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        if (k < e && ((keep >> k) & 1u)) {
            const int p = (lane << 5) + k;
            const bool lt = p < pm, gt = p > pm;
            // the side of the lane's lowest point that p lies on, field by field
#define ISO_SEL(F) (lt ? left.F : (gt ? right.F : mid.F))
#define ISO_SELG(F) (p < g ? gl.F : gr.F)
            const bool out = (p != g && fabove(ISO_SELG(w), ISO_SELG(a), ISO_SELG(k0), ISO_SELG(fx), ISO_SELG(m0),
                                               ISO_SELG(m1), ISO_SELG(kabs), pf, f)) ||
                             fabove(ISO_SEL(w), ISO_SEL(a), ISO_SEL(k0), ISO_SEL(fx), ISO_SEL(m0), ISO_SEL(m1),
                                    ISO_SEL(kabs), pf, f);
#undef ISO_SELG
#undef ISO_SEL
            if (out) drop |= 1u << k;
        }
        if (k < e) f = f + (yv[k] - c);
        pf += 1.0f;
    }
    return keep & ~drop;
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
