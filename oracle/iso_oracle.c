/*
 * Reference oracle for weighted isotonic regression.  TEST INFRASTRUCTURE ONLY:
 * nothing on the product path links, loads or calls this file.  Only the tests,
 * the smoke check and the CPU-baseline leg of the benchmark may use it.
 *
 * Plain, slow, obviously correct fp64 CPU code.  It shares no code, header or
 * constant with the CUDA library.
 *
 * What it computes ("Merge Hulls Without Copying Vertices: GPU Isotonic
 * Regression", Section 2.1, eq. (1)): for y_1..y_n and weights w_i > 0, the
 * unique z with z_1 <= ... <= z_n minimising sum_i w_i (z_i - y_i)^2.  The
 * decreasing problem is the increasing one for -y (same section).  The inputs
 * are the float32 values as given, read as doubles; w_i*y_i is then exact
 * (a product of two 24-bit mantissas fits in 53 bits).
 *
 * oracle_pava   -- pool adjacent violators (Section 2.1; "Isotonic Regression
 *                  on GPU", section "A curve that is only allowed to go up"):
 *                  push each element as a block (sum w*y, sum w, start) and pool
 *                  the last two blocks while their means are not increasing.
 *                  Ties are pooled (comparison ">=", cross-multiplied), which
 *                  gives maximal blocks: the canonical hull of Section 2.1 in
 *                  which collinear points are not vertices.
 * oracle_hull   -- a second, independent route: the lower convex hull of the
 *                  cumulative-sum diagram P_k = (W_k, S_k) (eq. (2)) by the
 *                  monotone chain, and z_i = slope of the hull edge above
 *                  [W_{i-1}, W_i] (eq. (3)).  Used only to cross-check PAVA.
 * oracle_backward -- block averaging (Section 6, "Gradient"): with G and W the
 *                  sums of g and w over element i's block,
 *                  d/dy_i = w_i * G / W.  Blocks are given by block-start flags.
 * oracle_backward_w -- the weight gradient of the same section,
 *                  d/dw_i = (y_i - z_i) * G / W.
 *
 * float64 inputs (the paper supports float32 and float64 working types,
 * Section 6 "Implementation"): oracle_pava_f64, oracle_backward_f64 and
 * oracle_backward_w_f64 apply the same definitions to double y, w and g.
 * w_i*y_i and the block sums are then no longer exact in double, so they are
 * kept as unevaluated sums of two doubles (the error-free transformations of
 * Dekker and Knuth: TwoSum for an addition, an FMA for the rounding error of a
 * product), about 106 significant bits, and the pooling test compares the two
 * cross products in the same arithmetic.
 *
 * Error convention ("groupant" page on the Rust PAVA, "arithmetic_resource_
 * partition"): a row with a non-finite y, or a weight that is not finite and
 * positive, is rejected before any arithmetic; the row's status is returned
 * as a bit mask (1 = non-finite y, 2 = bad weight) and its outputs are NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BAD_Y 1u
#define ORACLE_BAD_W 2u

static uint32_t check_row(int64_t n, const float *y, const float *w) {
    uint32_t st = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (!isfinite(y[i])) st |= ORACLE_BAD_Y;
        if (w && (!isfinite(w[i]) || !(w[i] > 0.0f))) st |= ORACLE_BAD_W;
    }
    return st;
}

static void fill_nan(int64_t n, double *z, uint8_t *blocks) {
    for (int64_t i = 0; i < n; ++i) {
        z[i] = NAN;
        if (blocks) blocks[i] = 0;
    }
}

/* One row of weighted PAVA.  Scratch: three arrays of n entries. */
uint32_t oracle_pava(int64_t n, const float *y, const float *w, int increasing,
                     double *z, uint8_t *blocks) {
    uint32_t st = check_row(n, y, w);
    if (st) { fill_nan(n, z, blocks); return st; }
    if (n <= 0) return 0;
    double *bs = (double *)malloc(sizeof(double) * n);   /* block sum of w*y */
    double *bw = (double *)malloc(sizeof(double) * n);   /* block sum of w   */
    int64_t *b0 = (int64_t *)malloc(sizeof(int64_t) * n); /* block start     */
    int64_t top = 0;                                      /* number of blocks */
    const double sgn = increasing ? 1.0 : -1.0;
    for (int64_t i = 0; i < n; ++i) {
        double wi = w ? (double)w[i] : 1.0;
        double yi = sgn * (double)y[i];
        bs[top] = wi * yi;
        bw[top] = wi;
        b0[top] = i;
        ++top;
        /* pool while mean(prev) >= mean(last), i.e. the order is violated or tied */
        while (top >= 2 && bs[top - 2] * bw[top - 1] >= bs[top - 1] * bw[top - 2]) {
            bs[top - 2] += bs[top - 1];
            bw[top - 2] += bw[top - 1];
            --top;
        }
    }
    for (int64_t k = 0; k < top; ++k) {
        int64_t end = (k + 1 < top) ? b0[k + 1] : n;
        double mean = sgn * (bs[k] / bw[k]);
        for (int64_t i = b0[k]; i < end; ++i) {
            z[i] = mean;
            if (blocks) blocks[i] = (uint8_t)(i == b0[k]);
        }
    }
    free(bs); free(bw); free(b0);
    return 0;
}

/* Cumulative-sum diagram, eq. (2): P_0 = (0,0), P_k = (sum_{i<=k} w_i, sum_{i<=k} w_i y_i)
 * with 1-based k; here arrays of n+1 points.  Exposed so that tests can pin it
 * against the running totals the pages print. */
void oracle_points(int64_t n, const float *y, const float *w, int increasing,
                   double *W, double *S) {
    const double sgn = increasing ? 1.0 : -1.0;
    W[0] = 0.0;
    S[0] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double wi = w ? (double)w[i] : 1.0;
        W[i + 1] = W[i] + wi;
        S[i + 1] = S[i] + wi * (sgn * (double)y[i]);
    }
}

/* One row by the lower hull of the cumulative-sum diagram (Section 2.1, eq. (3)). */
uint32_t oracle_hull(int64_t n, const float *y, const float *w, int increasing,
                     double *z, uint8_t *blocks) {
    uint32_t st = check_row(n, y, w);
    if (st) { fill_nan(n, z, blocks); return st; }
    if (n <= 0) return 0;
    double *W = (double *)malloc(sizeof(double) * (n + 1));
    double *S = (double *)malloc(sizeof(double) * (n + 1));
    int64_t *h = (int64_t *)malloc(sizeof(int64_t) * (n + 1)); /* hull vertex indices */
    oracle_points(n, y, w, increasing, W, S);
    int64_t k = 0;
    for (int64_t p = 0; p <= n; ++p) {
        /* drop the top while it is not strictly below the segment from the
           vertex under it to P_p (a turn <= 0: collinear points are removed) */
        while (k >= 2) {
            int64_t o = h[k - 2], a = h[k - 1];
            double cross = (W[a] - W[o]) * (S[p] - S[o]) - (S[a] - S[o]) * (W[p] - W[o]);
            if (cross > 0.0) break;
            --k;
        }
        h[k++] = p;
    }
    const double sgn = increasing ? 1.0 : -1.0;
    for (int64_t e = 0; e + 1 < k; ++e) {
        int64_t a = h[e], b = h[e + 1];
        double slope = sgn * ((S[b] - S[a]) / (W[b] - W[a]));
        for (int64_t i = a; i < b; ++i) {      /* element i lies over [W_i, W_{i+1}] */
            z[i] = slope;
            if (blocks) blocks[i] = (uint8_t)(i == a);
        }
    }
    free(W); free(S); free(h);
    return 0;
}

/* Backward of the fit (Section 6, "Gradient"): out_i = w_i * G_B / W_B where B is
 * element i's block, G_B = sum of grad over B and W_B = sum of w over B (the
 * block's size for unit weights).  blocks[i] != 0 marks a block start;
 * blocks[0] is treated as a start whatever its value. */
void oracle_backward(int64_t n, const float *grad, const uint8_t *blocks, const float *w,
                     double *out) {
    int64_t a = 0;
    while (a < n) {
        int64_t b = a + 1;
        while (b < n && !blocks[b]) ++b;
        double G = 0.0, Wb = 0.0;
        for (int64_t i = a; i < b; ++i) {
            G += (double)grad[i];
            Wb += w ? (double)w[i] : 1.0;
        }
        for (int64_t i = a; i < b; ++i) out[i] = (w ? (double)w[i] : 1.0) * (G / Wb);
        a = b;
    }
}

/* Weight gradient (same section): out_i = (y_i - z_i) * G_B / W_B, with z the
 * fit (in the direction of the call) and the blocks as above. */
void oracle_backward_w(int64_t n, const float *grad, const uint8_t *blocks, const float *w,
                       const float *y, const double *z, double *out) {
    int64_t a = 0;
    while (a < n) {
        int64_t b = a + 1;
        while (b < n && !blocks[b]) ++b;
        double G = 0.0, Wb = 0.0;
        for (int64_t i = a; i < b; ++i) {
            G += (double)grad[i];
            Wb += w ? (double)w[i] : 1.0;
        }
        for (int64_t i = a; i < b; ++i) out[i] = ((double)y[i] - z[i]) * (G / Wb);
        a = b;
    }
}

/* Batched wrappers: rows are independent problems (Section 3, first paragraph).
 * status may be NULL. */
void oracle_pava_rows(int64_t rows, int64_t n, const float *y, const float *w, int increasing,
                      double *z, uint8_t *blocks, uint32_t *status) {
    for (int64_t r = 0; r < rows; ++r) {
        uint32_t st = oracle_pava(n, y + r * n, w ? w + r * n : NULL, increasing, z + r * n,
                                  blocks ? blocks + r * n : NULL);
        if (status) status[r] = st;
    }
}

void oracle_hull_rows(int64_t rows, int64_t n, const float *y, const float *w, int increasing,
                      double *z, uint8_t *blocks, uint32_t *status) {
    for (int64_t r = 0; r < rows; ++r) {
        uint32_t st = oracle_hull(n, y + r * n, w ? w + r * n : NULL, increasing, z + r * n,
                                  blocks ? blocks + r * n : NULL);
        if (status) status[r] = st;
    }
}

void oracle_backward_rows(int64_t rows, int64_t n, const float *grad, const uint8_t *blocks,
                          const float *w, double *out) {
    for (int64_t r = 0; r < rows; ++r)
        oracle_backward(n, grad + r * n, blocks + r * n, w ? w + r * n : NULL, out + r * n);
}

/* ---- float64 inputs ---------------------------------------------------- */

typedef struct { double hi, lo; } dd;   /* the value hi + lo, |lo| <= ulp(hi) / 2 */

/* s + e = a + b exactly (Knuth's TwoSum, no precondition on a and b). */
static dd two_sum(double a, double b) {
    double s = a + b;
    double bb = s - a;
    double e = (a - (s - bb)) + (b - bb);
    dd r = {s, e};
    return r;
}

/* s + e = a + b exactly when |a| >= |b| (Dekker's FastTwoSum). */
static dd fast_two_sum(double a, double b) {
    double s = a + b;
    double e = b - (s - a);
    dd r = {s, e};
    return r;
}

/* p + e = a * b exactly (the FMA gives the product's rounding error). */
static dd two_prod(double a, double b) {
    double p = a * b;
    double e = fma(a, b, -p);
    dd r = {p, e};
    return r;
}

static dd dd_add(dd a, dd b) {
    dd s = two_sum(a.hi, b.hi);
    dd t = two_sum(a.lo, b.lo);
    s.lo += t.hi;
    s = fast_two_sum(s.hi, s.lo);
    s.lo += t.lo;
    return fast_two_sum(s.hi, s.lo);
}

static dd dd_neg(dd a) { dd r = {-a.hi, -a.lo}; return r; }

static dd dd_mul(dd a, dd b) {
    dd p = two_prod(a.hi, b.hi);
    p.lo += a.hi * b.lo + a.lo * b.hi;
    return fast_two_sum(p.hi, p.lo);
}

/* sign of a - b */
static int dd_cmp(dd a, dd b) {
    dd d = dd_add(a, dd_neg(b));
    if (d.hi != 0.0) return d.hi > 0.0 ? 1 : -1;
    return d.lo > 0.0 ? 1 : (d.lo < 0.0 ? -1 : 0);
}

/* a / b rounded to double (two quotient terms, then one rounding). */
static double dd_div(dd a, dd b) {
    double q1 = a.hi / b.hi;
    dd r = dd_add(a, dd_neg(dd_mul(b, (dd){q1, 0.0})));
    double q2 = r.hi / b.hi;
    return q1 + q2;
}

static uint32_t check_row_f64(int64_t n, const double *y, const double *w) {
    uint32_t st = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (!isfinite(y[i])) st |= ORACLE_BAD_Y;
        if (w && (!isfinite(w[i]) || !(w[i] > 0.0))) st |= ORACLE_BAD_W;
    }
    return st;
}

/* One row of weighted PAVA on float64 inputs, sums in double-double. */
uint32_t oracle_pava_f64(int64_t n, const double *y, const double *w, int increasing,
                         double *z, uint8_t *blocks) {
    uint32_t st = check_row_f64(n, y, w);
    if (st) { fill_nan(n, z, blocks); return st; }
    if (n <= 0) return 0;
    dd *bs = (dd *)malloc(sizeof(dd) * n);
    dd *bw = (dd *)malloc(sizeof(dd) * n);
    int64_t *b0 = (int64_t *)malloc(sizeof(int64_t) * n);
    int64_t top = 0;
    const double sgn = increasing ? 1.0 : -1.0;
    for (int64_t i = 0; i < n; ++i) {
        double wi = w ? w[i] : 1.0;
        bs[top] = two_prod(wi, sgn * y[i]);
        bw[top].hi = wi;
        bw[top].lo = 0.0;
        b0[top] = i;
        ++top;
        /* pool while mean(prev) >= mean(last) */
        while (top >= 2 &&
               dd_cmp(dd_mul(bs[top - 2], bw[top - 1]), dd_mul(bs[top - 1], bw[top - 2])) >= 0) {
            bs[top - 2] = dd_add(bs[top - 2], bs[top - 1]);
            bw[top - 2] = dd_add(bw[top - 2], bw[top - 1]);
            --top;
        }
    }
    for (int64_t k = 0; k < top; ++k) {
        int64_t end = (k + 1 < top) ? b0[k + 1] : n;
        double mean = sgn * dd_div(bs[k], bw[k]);
        for (int64_t i = b0[k]; i < end; ++i) {
            z[i] = mean;
            if (blocks) blocks[i] = (uint8_t)(i == b0[k]);
        }
    }
    free(bs); free(bw); free(b0);
    return 0;
}

void oracle_pava_rows_f64(int64_t rows, int64_t n, const double *y, const double *w,
                          int increasing, double *z, uint8_t *blocks, uint32_t *status) {
    for (int64_t r = 0; r < rows; ++r) {
        uint32_t st = oracle_pava_f64(n, y + r * n, w ? w + r * n : NULL, increasing, z + r * n,
                                      blocks ? blocks + r * n : NULL);
        if (status) status[r] = st;
    }
}

/* Block averaging on float64 inputs: out_i = w_i * G / W, G and W summed in
 * double-double over the block that the start flags delimit. */
void oracle_backward_rows_f64(int64_t rows, int64_t n, const double *grad,
                              const uint8_t *blocks, const double *w, double *out) {
    for (int64_t r = 0; r < rows; ++r) {
        const double *g = grad + r * n;
        const uint8_t *b = blocks + r * n;
        const double *wr = w ? w + r * n : NULL;
        double *o = out + r * n;
        int64_t i = 0;
        while (i < n) {
            int64_t j = i + 1;
            while (j < n && !b[j]) ++j;
            dd G = {0.0, 0.0}, W = {0.0, 0.0};
            for (int64_t k = i; k < j; ++k) {
                G = dd_add(G, (dd){g[k], 0.0});
                W = dd_add(W, (dd){wr ? wr[k] : 1.0, 0.0});
            }
            double ratio = dd_div(G, W);
            for (int64_t k = i; k < j; ++k) o[k] = (wr ? wr[k] : 1.0) * ratio;
            i = j;
        }
    }
}

/* The weight gradient on float64 inputs: (y_i - z_i) * G / W. */
void oracle_backward_w_f64(int64_t n, const double *grad, const uint8_t *blocks, const double *w,
                           const double *y, const double *z, double *out) {
    int64_t i = 0;
    while (i < n) {
        int64_t j = i + 1;
        while (j < n && !blocks[j]) ++j;
        dd G = {0.0, 0.0}, W = {0.0, 0.0};
        for (int64_t k = i; k < j; ++k) {
            G = dd_add(G, (dd){grad[k], 0.0});
            W = dd_add(W, (dd){w ? w[k] : 1.0, 0.0});
        }
        double ratio = dd_div(G, W);
        for (int64_t k = i; k < j; ++k) out[k] = (y[k] - z[k]) * ratio;
        i = j;
    }
}
