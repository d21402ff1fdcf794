// Device building blocks of the isotonic fit: fixed-point coordinates, the turn
// predicate, lane hulls in a register bit mask, and walking merges of neighbouring
// hulls inside a tile of lanes.
//
// References are to "Merge Hulls Without Copying Vertices: GPU Isotonic
// Regression" (the paper).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <type_traits>

namespace isodev {

constexpr int kPts = 32;        // elements (points) per lane, Section 3.1
constexpr int kRow = 33;        // lane-relative cumulative sums per lane: points 0..32
constexpr unsigned kFull = 0xffffffffu;

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// ---------------------------------------------------------------------------
// Fixed point.  A tile (a short row, or one chunk of a long row) rounds its
// values to integer multiples of a power of two chosen from the largest
// exponent in the tile, so that every value is below 2^50 in magnitude: the
// grid is 2^-50 of the tile's largest value, as fine as an fp64 sum of that
// tile.  Sums of these integers (below 2^63 for 8,192 values) are exact and
// independent of order, and every turn test on them is exact.  The fp32 input
// carries 24 significant bits, so values within 2^26 of the tile's largest
// exponent are represented without any rounding.
// ---------------------------------------------------------------------------

// Biased float32 exponent, with zero and subnormals mapped to 1.
__device__ __forceinline__ int bexp(float v) {
    int e = (__float_as_uint(v) >> 23) & 0xff;
    return e == 0 ? 1 : e;
}

// Biased float64 exponent, with zero and subnormals mapped to 1.
__device__ __forceinline__ int bexp(double v) {
    const int e = (int)(((unsigned long long)__double_as_longlong(v) >> 52) & 0x7ff);
    return e == 0 ? 1 : e;
}

// Inf or NaN.
__device__ __forceinline__ bool nonfinite(float v) { return ((__float_as_uint(v) >> 23) & 0xff) == 0xff; }
__device__ __forceinline__ bool nonfinite(double v) {
    return (((unsigned long long)__double_as_longlong(v) >> 52) & 0x7ff) == 0x7ff;
}

// I/O types.  The grid is the same for float32 and float64 inputs: 2^-50 of the
// power of two above the tile's largest magnitude, i.e. the quantum exponent
// of a tile whose largest biased exponent is e is e - kUnitK (values) or
// pe - kProdK for products w*y whose exponents sum to at most pe.  V: the
// 16-byte vector of staged loads, kPerV elements.
template <class T> struct IoT;
template <> struct IoT<float> {
    static constexpr int kUnitK = 176;    // 127 + 49
    static constexpr int kProdK = 302;    // 2 * 150 + 48 - 46
    using V = float4;
    static constexpr int kPerV = 4;
};
template <> struct IoT<double> {
    static constexpr int kUnitK = 1072;   // 1023 + 49
    static constexpr int kProdK = 2094;   // 2 * 1075 + 48 - 104
    using V = double2;
    static constexpr int kPerV = 2;
};

// round(v / 2^(emax - 176)): |result| < 2^50 when bexp(v) <= emax.  The
// scaling by a power of two is exact in float32 wherever the result is at
// least 1/2 (it only moves the exponent), so one conversion rounds it to the
// nearest integer (ties to even).  Scales above 2^127 (tiles whose values are
// all below 2^-78) take two factors.  A non-finite v gives an arbitrary value
// (the row is flagged and its output discarded).
template <class T> struct QuantT;
template <> struct QuantT<float> {
    float s1, s2;
    __device__ __forceinline__ explicit QuantT(int emax) {
        const int sh = 176 - emax;                 // -78 .. 175
        const int a = sh < 127 ? sh : 127;
        s1 = __int_as_float((a + 127) << 23);
        s2 = __int_as_float((sh - a + 127) << 23);  // 1 unless sh > 127
    }
    __device__ __forceinline__ int64_t operator()(float v) const {
        return __float2ll_rn((v * s1) * s2);
    }
};
using Quant = QuantT<float>;

// The same for float64: round(v / 2^(emax - 1072)), |result| < 2^50 when
// bexp(v) <= emax; the scale 2^(1072 - emax) (2^-974 .. 2^1071) as two
// factors.  A product that falls below the normal range is below 2^-1022 of
// a quantum and rounds to 0 either way.
template <> struct QuantT<double> {
    double s1, s2;
    __device__ __forceinline__ explicit QuantT(int emax) {
        const int sh = 1072 - emax;
        const int a = sh < 1023 ? sh : 1023;
        s1 = __longlong_as_double((long long)(a + 1023) << 52);
        s2 = __longlong_as_double((long long)(sh - a + 1023) << 52);
    }
    __device__ __forceinline__ int64_t operator()(double v) const {
        return __double2ll_rn((v * s1) * s2);
    }
};

__device__ __forceinline__ int64_t quant(float v, int emax) { return Quant(emax)(v); }

// Multiplication by 2^k in float32 as two exact scalings (k within [-252, 254]),
// the product rounded like ldexpf unless it falls below the normal range.
struct Pow2 {
    float a, b;
    __device__ __forceinline__ explicit Pow2(int k) {
        const int k1 = max(min(k, 127), -126);
        const int k2 = max(min(k - k1, 127), -126);
        a = __int_as_float((k1 + 127) << 23);
        b = __int_as_float((k2 + 127) << 23);
    }
    __device__ __forceinline__ float operator()(float x) const { return (x * a) * b; }
};

// float32 of a 64-bit integer from two 32-bit conversions and one fused
// multiply-add on the magnitude: exact when the value is representable, else
// within 1.5 ulp.
__device__ __forceinline__ float i64_to_f32(int64_t x) {
    const uint64_t u = x < 0 ? (uint64_t)0 - (uint64_t)x : (uint64_t)x;
    const float f = __fmaf_rn(__uint2float_rn((unsigned)(u >> 32)), 4294967296.0f,
                              __uint2float_rn((unsigned)u));
    return x < 0 ? -f : f;
}

// round(w*y / 2^(pemax - 302)) from the exact 48-bit product of the mantissas:
// |result| < 2^50 when bexp(w) + bexp(y) <= pemax.
__device__ __forceinline__ int64_t quant_prod(float w, float y, int pemax) {
    const uint32_t bw = __float_as_uint(w), by = __float_as_uint(y);
    int ew = (bw >> 23) & 0xff, ey = (by >> 23) & 0xff;
    uint32_t mw = bw & 0x7fffffu, my = by & 0x7fffffu;
    if (ew) mw |= 0x800000u; else ew = 1;
    if (ey) my |= 0x800000u; else ey = 1;
    const uint64_t prod = (uint64_t)mw * (uint64_t)my;
    const int t = pemax - (ew + ey) - 2;
    uint64_t mag;
    if (t <= 0) {
        mag = prod << min(-t, 2);
    } else {
        mag = t >= 64 ? 0ull : ((prod >> (t - 1)) + 1ull) >> 1;   // round half up
    }
    const int64_t v64 = (int64_t)mag;
    return ((bw ^ by) >> 31) ? -v64 : v64;
}

// round(w*y / 2^(pemax - 2094)) for float64 from the exact 106-bit product of
// the mantissas: |result| < 2^50 when bexp(w) + bexp(y) <= pemax.
__device__ __forceinline__ int64_t quant_prod(double w, double y, int pemax) {
    const uint64_t bw = (uint64_t)__double_as_longlong(w), by = (uint64_t)__double_as_longlong(y);
    int ew = (int)((bw >> 52) & 0x7ff), ey = (int)((by >> 52) & 0x7ff);
    uint64_t mw = bw & 0xfffffffffffffull, my = by & 0xfffffffffffffull;
    if (ew) mw |= 1ull << 52; else ew = 1;
    if (ey) my |= 1ull << 52; else ey = 1;
    const unsigned __int128 prod = (unsigned __int128)mw * my;
    const int t = pemax - (ew + ey) + 56;                    // >= 56
    const uint64_t mag = t >= 128 ? 0ull : (uint64_t)(((prod >> (t - 1)) + 1u) >> 1);
    const int64_t v64 = (int64_t)mag;
    return ((bw ^ by) >> 63) ? -v64 : v64;
}

// Quantum exponents: value = integer * 2^q.
__device__ __forceinline__ int qexp_unit(int emax) { return emax - 176; }
__device__ __forceinline__ int qexp_prod(int pemax) { return pemax - 302; }
template <class T> __device__ __forceinline__ int qexp_unit_t(int emax) { return emax - IoT<T>::kUnitK; }
template <class T> __device__ __forceinline__ int qexp_prod_t(int pemax) { return pemax - IoT<T>::kProdK; }

// A slope (or a ratio) dS / dW * 2^k in the I/O type: float32 from two
// rounded conversions and one division, scaled exactly; float64 likewise in
// double (exact conversions below 2^53).
template <class T> __device__ __forceinline__ T ratio_t(int64_t dS, int64_t dW, int k);
template <> __device__ __forceinline__ float ratio_t<float>(int64_t dS, int64_t dW, int k) {
    return Pow2(k)(i64_to_f32(dS) / i64_to_f32(dW));
}
template <> __device__ __forceinline__ double ratio_t<double>(int64_t dS, int64_t dW, int k) {
    return ldexp((double)dS / (double)dW, k);
}

// Quiet NaN of the I/O type.
template <class T> __device__ __forceinline__ T qnan_t();
template <> __device__ __forceinline__ float qnan_t<float>() { return __int_as_float(0x7fffffff); }
template <> __device__ __forceinline__ double qnan_t<double>() {
    return __longlong_as_double(0x7fffffffffffffffll);
}

// ---------------------------------------------------------------------------
// Turn predicate.  For points O, A, B with A - O = (w1, s1), B - O = (w2, s2),
// the turn O -> A -> B is strictly left (A strictly below the segment O-B on a
// lower hull scanned by increasing W) iff w1*s2 - s1*w2 > 0.  WIDE selects
// 128-bit products: needed everywhere except inside one lane of a unit-weight
// tile, where |w| <= 32 and |s| < 2^56.
// ---------------------------------------------------------------------------
template <bool WIDE>
__device__ __forceinline__ bool left_turn(int64_t w1, int64_t s1, int64_t w2, int64_t s2) {
    if constexpr (WIDE) {
        __int128 a = (__int128)w1 * (__int128)s2;
        __int128 b = (__int128)s1 * (__int128)w2;
        return a > b;
    } else {
        return w1 * s2 > s1 * w2;
    }
}

// Exact sign test w1*s2 - w2*s1 > 0 for |w| < 2^30 (point counts of a tile):
// 32 x 64-bit products split in two halves, without 128-bit arithmetic.
__device__ __forceinline__ bool left_turn_w32(int w1, int64_t s1, int w2, int64_t s2) {
    const int64_t h = (int64_t)w1 * (int32_t)(s2 >> 32) - (int64_t)w2 * (int32_t)(s1 >> 32);
    const int64_t l = (int64_t)w1 * (int64_t)(uint32_t)s2 - (int64_t)w2 * (int64_t)(uint32_t)s1;
    const int64_t H = h + (l >> 32);
    return H > 0 || (H == 0 && (uint32_t)l != 0u);
}

// Exact sign of a*b - c*d for signed 128-bit operands (products up to 256 bits),
// used by the merge levels, whose row coordinates exceed 64 bits.
struct U256 { uint64_t w[4]; };

__device__ __forceinline__ U256 mul_u128(unsigned __int128 a, unsigned __int128 b) {
    const uint64_t a0 = (uint64_t)a, a1 = (uint64_t)(a >> 64);
    const uint64_t b0 = (uint64_t)b, b1 = (uint64_t)(b >> 64);
    const unsigned __int128 p00 = (unsigned __int128)a0 * b0;
    const unsigned __int128 p01 = (unsigned __int128)a0 * b1;
    const unsigned __int128 p10 = (unsigned __int128)a1 * b0;
    const unsigned __int128 p11 = (unsigned __int128)a1 * b1;
    U256 r;
    r.w[0] = (uint64_t)p00;
    unsigned __int128 mid = (p00 >> 64) + (uint64_t)p01 + (uint64_t)p10;
    r.w[1] = (uint64_t)mid;
    unsigned __int128 hi = (mid >> 64) + (p01 >> 64) + (p10 >> 64) + (uint64_t)p11;
    r.w[2] = (uint64_t)hi;
    r.w[3] = (uint64_t)(hi >> 64) + (uint64_t)(p11 >> 64);
    return r;
}

__device__ __forceinline__ int cmp_u256(const U256& x, const U256& y) {
    for (int i = 3; i >= 0; --i) {
        if (x.w[i] != y.w[i]) return x.w[i] > y.w[i] ? 1 : -1;
    }
    return 0;
}

// sign(a*b - c*d)
__device__ __forceinline__ int sign_det128(__int128 a, __int128 b, __int128 c, __int128 d) {
    const int sab = ((a > 0) - (a < 0)) * ((b > 0) - (b < 0));
    const int scd = ((c > 0) - (c < 0)) * ((d > 0) - (d < 0));
    if (sab != scd) return sab > scd ? 1 : -1;        // also covers zero products
    if (sab == 0) return 0;
    auto uabs = [](__int128 x) -> unsigned __int128 {
        return x < 0 ? (unsigned __int128)(-(x + 1)) + 1u : (unsigned __int128)x;
    };
    const int c3 = cmp_u256(mul_u128(uabs(a), uabs(b)), mul_u128(uabs(c), uabs(d)));
    return sab > 0 ? c3 : -c3;
}

// ---------------------------------------------------------------------------
// Lane hull (Section 3.1).  One lane runs the monotone chain over its points
// 0..e (e <= 32 elements), keeping the stack as a bit mask: bit k set while
// point k is on the stack; the top and the entry below it are kept in
// registers and the next entry below is found by count-leading-zeros.  A turn
// of zero pops, so collinear middle points are dropped (Section 4).
//
// Only points that are locally convex can be vertices of any hull that
// contains them (Lemma 4.1); `cand` holds those among 1..e-1, and the chain
// visits only them.  Point e (the lane's end) is always pushed last and is
// not part of the returned mask.
// ---------------------------------------------------------------------------
template <bool WEIGHTED>
__device__ __forceinline__ uint32_t lane_hull(const int64_t* Sx, const int64_t* Wx, uint32_t cand,
                                              int e) {
    if (e <= 0) return 0u;
    // W of a unit-weight lane is a point index (at most 32): 32-bit, and its
    // turn products are 32 x 64-bit (below 2^61, exact in 64 bits)
    using WT = typename std::conditional<WEIGHTED, int64_t, int>::type;
    uint32_t mask = 1u;          // stack membership
    int t = 0, b = -1;           // top and the entry below it
    int64_t St = 0, Sb = 0;
    WT Wt = 0, Wb = 0;
    uint32_t rem = cand & ~1u & (e >= 32 ? 0xffffffffu : ((1u << e) - 1u));
    int k = rem ? (__ffs(rem) - 1) : e;
    rem &= rem - 1u;
    int64_t Sk = Sx[k];
    WT Wk = WEIGHTED ? (WT)Wx[k] : (WT)k;
    // Every iteration pushes or pops; both loads it may need next are issued
    // before the turn is known, so a lane never waits on a dependent load.
    for (int it = 0; it < 2 * kPts + 2; ++it) {
        const int k2 = rem ? (__ffs(rem) - 1) : e;                 // next point after a push
        const uint32_t below = b > 0 ? (mask & ((1u << b) - 1u)) : 0u;
        const int b2 = below ? (31 - __clz(below)) : -1;           // new below-top after a pop
        const int bl = b2 < 0 ? 0 : b2;
        const int64_t Sk2 = Sx[k2];
        const WT Wk2 = WEIGHTED ? (WT)Wx[k2] : (WT)k2;
        const int64_t Sb2 = Sx[bl];
        const WT Wb2 = WEIGHTED ? (WT)Wx[bl] : (WT)bl;
        bool lt;
        if constexpr (WEIGHTED) lt = left_turn<true>(Wt - Wb, St - Sb, Wk - Wb, Sk - Sb);
        else lt = (int64_t)(Wt - Wb) * (Sk - Sb) > (St - Sb) * (int64_t)(Wk - Wb);
        const bool push = (b < 0) || lt;
        if (push) {
            if (k >= e) break;
            mask |= 1u << k;
            b = t; Sb = St; Wb = Wt;
            t = k; St = Sk; Wt = Wk;
            k = k2; Sk = Sk2; Wk = Wk2;
            rem &= rem - 1u;
        } else {
            mask &= ~(1u << t);
            t = b; St = Sb; Wt = Wb;
            b = b2; Sb = Sb2; Wb = Wb2;
        }
    }
    return mask;
}

// ---------------------------------------------------------------------------
// A tile: L consecutive lanes (a power of two) holding one row, or one chunk of
// a row, with nt elements (points 0..nt).  Vertex flags for points 0..nt-1 are
// the lanes' mask bits (point p: lane p/32, bit p%32); point nt, the tile's
// end, is always a vertex.  Coordinates are tile-relative: the lane's start
// plus the lane-relative cumulative sum.
// ---------------------------------------------------------------------------
struct Tile {
    const int64_t* Sx;   // [L][kRow] lane-relative S (row of the tile's lane 0 first)
    const int64_t* Wx;   // [L][kRow] lane-relative W, weighted tiles only
    const int64_t* LS;   // [L+1] lane starts of S, LS[L] = tile total
    const int64_t* LW;   // [L+1] lane starts of W (weighted)
    uint32_t* mask;      // [L] vertex masks
    uint32_t* summ;      // non-empty-lane bits; bit (sbase + lane) for lane of this tile
    int sbase;           // bit offset of the tile's lane 0 in summ
    int L;               // lanes
    int nt;              // elements
};

// Tile-relative coordinates of point p (0..nt).  After the lane hulls are
// built, row l of Sx (Wx) holds the tile-relative cumulative sums at points
// 32l .. 32l+32; the end point of a tile of exactly 32 L elements is LS[L].
template <bool WEIGHTED>
__device__ __forceinline__ int64_t tile_S(const Tile& T, int p) {
    const int l = p >> 5, k = p & 31;
    return l < T.L ? T.Sx[l * kRow + k] : T.LS[T.L];
}
template <bool WEIGHTED>
__device__ __forceinline__ int64_t tile_W(const Tile& T, int p) {
    if constexpr (WEIGHTED) {
        const int l = p >> 5, k = p & 31;
        return l < T.L ? T.Wx[l * kRow + k] : T.LW[T.L];
    } else {
        return (int64_t)p;
    }
}

// Turn test on tile points, with the differences taken from o.
template <bool WEIGHTED>
__device__ __forceinline__ bool tile_turn(int64_t Wo, int64_t So, int64_t Wa, int64_t Sa,
                                          int64_t Wb, int64_t Sb) {
    if constexpr (WEIGHTED) return left_turn<true>(Wa - Wo, Sa - So, Wb - Wo, Sb - So);
    else return left_turn_w32((int)(Wa - Wo), Sa - So, (int)(Wb - Wo), Sb - So);
}

__device__ __forceinline__ bool summ_bit(const Tile& T, int lane) {
    int b = T.sbase + lane;
    return (T.summ[b >> 5] >> (b & 31)) & 1u;
}

// Highest non-empty lane in [lo, hi), or -1.
__device__ __forceinline__ int prev_nonempty(const Tile& T, int lo, int hi) {
    int b = T.sbase + hi - 1, bl = T.sbase + lo;
    while (b >= bl) {
        int wi = b >> 5;
        uint32_t word = T.summ[wi] & (0xffffffffu >> (31 - (b & 31)));
        int wlo = wi << 5;
        if (wlo < bl) word &= ~((1u << (bl - wlo)) - 1u);
        if (word) return wlo + 31 - __clz(word) - T.sbase;
        b = wlo - 1;
    }
    return -1;
}

// Lowest non-empty lane in [lo, hi), or -1.
__device__ __forceinline__ int next_nonempty(const Tile& T, int lo, int hi) {
    int b = T.sbase + lo, bh = T.sbase + hi;
    while (b < bh) {
        int wi = b >> 5;
        int wlo = wi << 5;
        uint32_t word = T.summ[wi] & (0xffffffffu << (b & 31));
        if (bh - wlo < 32) word &= (1u << (bh - wlo)) - 1u;
        if (word) return wlo + __ffs(word) - 1 - T.sbase;
        b = wlo + 32;
    }
    return -1;
}

// Highest vertex < p among lanes [lo_lane, ...); -1 if none.
__device__ __forceinline__ int tile_pred(const Tile& T, int p, int lo_lane) {
    int l = p >> 5, k = p & 31;
    if (l < T.L) {
        uint32_t m = T.mask[l] & ((1u << k) - 1u);
        if (m) return (l << 5) + 31 - __clz(m);
    }
    int q = prev_nonempty(T, lo_lane, min(l, T.L));
    if (q < 0) return -1;
    return (q << 5) + 31 - __clz(T.mask[q]);
}

// Lowest vertex > p among lanes [.., hi_lane); `endp` if none.
__device__ __forceinline__ int tile_succ(const Tile& T, int p, int hi_lane, int endp) {
    int l = p >> 5, k = p & 31;
    uint32_t m = T.mask[l] & ~((2u << k) - 1u);
    if (k == 31) m = 0;
    if (m) return (l << 5) + __ffs(m) - 1;
    int q = next_nonempty(T, l + 1, hi_lane);
    if (q < 0) return endp;
    return (q << 5) + __ffs(T.mask[q]) - 1;
}

// Predecessor / successor vertex for merge groups that lie inside one warp:
// `word` is the warp's non-empty-lane word, so no loop over lanes is needed
// and the leaders of all groups of a warp run the same instructions.
__device__ __forceinline__ int wpred(const Tile& T, uint32_t word, int p, int lo_lane) {
    const int l = p >> 5, k = p & 31;
    const int bl = (T.sbase + l) & 31, blo = (T.sbase + lo_lane) & 31;
    const uint32_t m0 = T.mask[l] & ((1u << k) - 1u);
    const uint32_t below = word & ((1u << bl) - 1u) & ~((1u << blo) - 1u);
    const int q = m0 ? l : max(lo_lane, l - bl + 31 - __clz(below));
    const uint32_t mq = m0 ? m0 : T.mask[q];
    return (q << 5) + 31 - __clz(mq);
}
__device__ __forceinline__ int wsucc(const Tile& T, uint32_t word, int p, int hi_lane, int endp) {
    const int l = p >> 5, k = p & 31;
    const int bl = (T.sbase + l) & 31;
    const int bhi = bl + (hi_lane - l);                  // one past the group's last bit
    const uint32_t m0 = k == 31 ? 0u : (T.mask[l] & ~((2u << k) - 1u));
    uint32_t above = bl == 31 ? 0u : (word & ~((2u << bl) - 1u));
    if (bhi < 32) above &= (1u << bhi) - 1u;
    const int q = m0 ? l : (above ? l - bl + __ffs(above) - 1 : l);
    const uint32_t mq = m0 ? m0 : T.mask[q];
    const int r = (q << 5) + __ffs(mq) - 1;
    return (m0 | above) ? r : endp;
}

// Bridge of the merge of lane groups A = [A0, B0) and B = [B0, Bend) (Section
// 3.2, Lemma 4.2): s = 32*B0 is the last vertex of H(A) and the first of H(B).
// If the chain is convex at s, returns (s, s).  Otherwise walks from s's
// neighbours, the left end left and the right end right, until the line
// between them supports both hulls.  Each step removes a vertex (Lemma 5.1).
// The coordinates of the two current ends stay in registers; a step loads one
// new point.  IN_WARP selects the warp-local lookups.
template <bool WEIGHTED, bool IN_WARP>
__device__ __forceinline__ void tile_bridge(const Tile& T, int A0, int B0, int Bend, int& ra,
                                            int& rb) {
    const int s = B0 << 5;
    const int endB = min(Bend << 5, T.nt);
    const int startA = A0 << 5;
    uint32_t word = 0;
    if constexpr (IN_WARP) word = T.summ[(T.sbase + A0) >> 5];
    auto pred = [&](int p) { return IN_WARP ? wpred(T, word, p, A0) : tile_pred(T, p, A0); };
    auto succ = [&](int p) {
        return IN_WARP ? wsucc(T, word, p, Bend, endB) : tile_succ(T, p, Bend, endB);
    };
    int a = pred(s);
    int b = succ(s);
    int64_t Wa = tile_W<WEIGHTED>(T, a), Sa = tile_S<WEIGHTED>(T, a);
    int64_t Wb = tile_W<WEIGHTED>(T, b), Sb = tile_S<WEIGHTED>(T, b);
    {
        const int64_t Ws = tile_W<WEIGHTED>(T, s), Ss = tile_S<WEIGHTED>(T, s);
        if (tile_turn<WEIGHTED>(Wa, Sa, Ws, Ss, Wb, Sb)) { ra = s; rb = s; return; }
    }
    for (;;) {
        bool moved = false;
        while (a > startA) {
            const int p = pred(a);
            const int64_t Wp = tile_W<WEIGHTED>(T, p), Sp = tile_S<WEIGHTED>(T, p);
            if (tile_turn<WEIGHTED>(Wp, Sp, Wa, Sa, Wb, Sb)) break;   // p -> a -> b convex
            a = p; Wa = Wp; Sa = Sp; moved = true;
        }
        while (b < endB) {
            const int q = succ(b);
            const int64_t Wq = tile_W<WEIGHTED>(T, q), Sq = tile_S<WEIGHTED>(T, q);
            if (tile_turn<WEIGHTED>(Wa, Sa, Wb, Sb, Wq, Sq)) break;   // a -> b -> q convex
            b = q; Wb = Wq; Sb = Sq; moved = true;
        }
        if (!moved) break;
    }
    ra = a; rb = b;
}

// Merge of two neighbouring hulls stored as compact lists (point indices P,
// tile-relative S, and W for weighted tiles; flat entry f at f + f/32), each
// list holding a group's vertices before its end point: L = the cL entries
// from flat fL, R = the cR entries from flat fR, R's
// first entry being L's end point s, and (SE, WE) the end point of R (W: the
// point index for unit weights), index cR below.  If the chain is convex at s,
// R follows L unchanged.  Otherwise the two ends walk to their tangent points
// in turn, from s's neighbours (Lemma 4.2); a walk longer than kCompactLinear
// steps finishes by bisection over the list.  The merged list is L[0..a]
// followed by R[b..cR-1]; the caller moves that tail (returned as flat dst,
// src and len) and the new count is stored in *cntL.
constexpr int kCompactLinear = 8;

template <bool WEIGHTED>
__device__ __forceinline__ void compact_merge(const int64_t* S, const int64_t* W,
                                              const uint16_t* P, int fL, int* cntL, int fR, int cR,
                                              int64_t SE, int64_t WE, int& dst, int& src,
                                              int& len) {
    // flat entry f lives at f + f/32
    const int cL = *cntL;
    auto at = [](int f) { return f + (f >> 5); };
    auto SL = [&](int i) -> int64_t { return S[at(fL + i)]; };
    auto wl = [&](int i) -> int64_t {
        if constexpr (WEIGHTED) return W[at(fL + i)]; else return (int64_t)P[at(fL + i)];
    };
    auto sr = [&](int j) -> int64_t { return j < cR ? S[at(fR + j)] : SE; };
    auto wr = [&](int j) -> int64_t {
        if constexpr (WEIGHTED) return j < cR ? W[at(fR + j)] : WE;
        else return j < cR ? (int64_t)P[at(fR + j)] : WE;
    };
    int a = cL - 1, b = 1;
    int64_t Wa = wl(a), Sa = SL(a), Wb = wr(b), Sb = sr(b);
    if (tile_turn<WEIGHTED>(Wa, Sa, wr(0), sr(0), Wb, Sb)) {
        dst = fL + cL; src = fR; len = cR;
        *cntL = cL + cR;
        return;
    }
    for (;;) {
        bool moved = false;
        // the left end: the last vertex i <= a strictly below the segment from
        // its predecessor to b
        for (int steps = 0; a > 0; ++steps) {
            if (steps == kCompactLinear) {
                int lo = 0, hi = a;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (tile_turn<WEIGHTED>(wl(mid - 1), SL(mid - 1), wl(mid), SL(mid), Wb, Sb)) lo = mid;
                    else hi = mid - 1;
                }
                a = lo; Wa = wl(a); Sa = SL(a);
                break;
            }
            const int64_t Wp = wl(a - 1), Sp = SL(a - 1);
            if (tile_turn<WEIGHTED>(Wp, Sp, Wa, Sa, Wb, Sb)) break;
            --a; Wa = Wp; Sa = Sp; moved = true;
        }
        // the right end: the first vertex j >= b strictly below the segment
        // from a to its successor (R's end point always qualifies)
        for (int steps = 0; b < cR; ++steps) {
            if (steps == kCompactLinear) {
                int lo = b, hi = cR;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (tile_turn<WEIGHTED>(Wa, Sa, wr(mid), sr(mid), wr(mid + 1), sr(mid + 1))) hi = mid;
                    else lo = mid + 1;
                }
                b = lo; Wb = wr(b); Sb = sr(b);
                break;
            }
            const int64_t Wq = wr(b + 1), Sq = sr(b + 1);
            if (tile_turn<WEIGHTED>(Wa, Sa, Wb, Sb, Wq, Sq)) break;
            ++b; Wb = Wq; Sb = Sq; moved = true;
        }
        if (!moved) break;
    }
    dst = fL + a + 1; src = fR + b; len = cR - b;
    *cntL = a + 1 + cR - b;
}

// Clear this lane's vertex bits strictly between a and b.
__device__ __forceinline__ uint32_t clear_between(uint32_t m, int lane, int a, int b) {
    int lo = max(a + 1 - (lane << 5), 0);
    int hi = min(b - (lane << 5), 32);
    if (lo < hi) {
        uint32_t span = (hi - lo == 32) ? 0xffffffffu : (((1u << (hi - lo)) - 1u) << lo);
        m &= ~span;
    }
    return m;
}

}  // namespace isodev
