/*
 * iso.h -- C ABI of the GB300 (sm_103a) isotonic-regression library libiso.so.
 *
 * The operation ("Merge Hulls Without Copying Vertices: GPU Isotonic Regression",
 * Section 2.1, eq. (1)): for every row y_1..y_n with weights w_i > 0, the unique
 * z with z_1 <= z_2 <= ... <= z_n that minimises sum_i w_i (z_i - y_i)^2.  The
 * decreasing problem is the increasing one for -y (same section).  z is taken,
 * as in eq. (3), as the slopes of the lower convex hull of the cumulative-sum
 * diagram P_k = (W_k, S_k), W_k = sum_{i<=k} w_i, S_k = sum_{i<=k} w_i y_i
 * (eq. (2)); the hull's vertices are the starts of the fit's blocks.
 *
 * Conventions shared by every entry point:
 *  - Layout: row-major, contiguous [rows, n] float32 arrays (row r starts at
 *    element r*n).  Any 4-byte alignment is accepted.
 *  - Memory: every array argument ("device" below) must be accessible from
 *    the device: device memory, or pinned (page-locked) host memory, which
 *    under unified addressing is device-accessible at its host address -- the
 *    kernels then read inputs and write outputs in place over the host link
 *    (NVLink-C2C on GB300), with no separate copy.  The workspace is best
 *    kept in device memory.
 *  - Ownership: the caller owns every buffer, the workspace and the stream.
 *    The fit and backward calls allocate no memory, keep no state between
 *    calls (beyond the device's SM count, read once), and never synchronise
 *    the stream: every call only enqueues kernels on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and returns.  Only the optional
 *    benchmarking and debugging switches at the end of this file keep state.
 *  - Errors the host can see (NULL pointers, non-positive or oversized shapes,
 *    a workspace that is too small or misaligned) return a negative status and
 *    enqueue nothing.  A failed kernel launch returns ISO_ERR_CUDA.
 *  - Errors in the data (a non-finite y, a weight that is not finite and
 *    positive) never fail the call: that row's outputs are NaN, its block
 *    flags are 0, and its bit in `row_status` is set (the paper's per-row NaN
 *    flags, Section 6 "Blocks and memory", without its host synchronisation).
 *  - Limits: 1 <= n <= 2^31 - 1, 1 <= rows, rows * n <= 2^40.  An empty call
 *    (rows == 0 or n == 0, neither negative; for ragged batches segments == 0)
 *    does nothing and returns ISO_OK whatever the pointers; a ragged batch
 *    with total == 0 only writes the segments' statuses.
 *  - float64 I/O: every entry point that takes float32 arrays has an _f64
 *    twin taking float64 arrays (the paper supports both working types,
 *    Section 6 "Implementation"), with the same arguments, layout, workspace
 *    sizes, errors and status bits; only the element type differs.
 */
#ifndef ISO_H
#define ISO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ISO_OK = 0,
    ISO_ERR_INVALID_ARG = -1, /* NULL pointer, bad shape or flag                 */
    ISO_ERR_WORKSPACE = -2,   /* workspace NULL / too small / not 256-B aligned */
    ISO_ERR_CUDA = -3,        /* a CUDA call or kernel launch failed            */
    ISO_ERR_TIMEOUT = -4      /* reserved: a bounded device-side wait gave up   */
} iso_status;

/* Bits of a row's status word. */
#define ISO_ROW_BAD_Y 1u /* the row holds a NaN or infinite y                   */
#define ISO_ROW_BAD_W 2u /* the row holds a weight that is not finite and > 0   */
#define ISO_ROW_BAD_SHAPE 4u /* ragged batches: the segment's offsets are out of  */
                             /* order or range, or it is longer than max_len      */

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
int iso_version(void);

/* Human-readable name of a status code (static string). */
const char *iso_status_string(int status);

/*
 * Bytes of device workspace that iso_fit needs for `rows` rows of `n` elements
 * (`weighted` != 0 when w is given).  0 means no workspace is needed.  Returns
 * 0 as well for invalid shapes (iso_fit then reports the error).
 */
size_t iso_fit_workspace_bytes(int64_t rows, int64_t n, int weighted);

/*
 * iso_fit -- forward fit.
 *
 * Defined by eq. (1)-(3) of the paper (Section 2.1); the method is the paper's
 * Section 3: lane hulls kept in register bit masks, lane and chunk merges by
 * walking to the bridge, and, for rows longer than one chunk, a merge tree
 * whose nodes are lists of segments of the chunk hulls (Section 3.3), followed
 * by reconstruction (Section 3.4).
 *
 *  y          [rows, n] float32, device, read only.
 *  w          [rows, n] float32, device, read only, or NULL for unit weights.
 *  rows, n    shape.
 *  increasing 1: non-decreasing fit; 0: non-increasing fit (fit of -y, negated).
 *  out        [rows, n] float32, device, written: the fit.  Every value is
 *             rounded to float32 once from the slope of its hull edge; the
 *             output is not forced to be monotone (no cumulative maximum),
 *             as in the paper's Section 6 "Output".
 *  blocks     [rows, n] uint8, device, written, or NULL: blocks[i] = 1 where
 *             element i starts a block (its left point is a hull vertex; the
 *             paper's block-start byte of Section 6 "Gradient"), else 0.
 *             blocks[0] of a valid row is always 1.  Needed by iso_backward.
 *  workspace  device scratch of at least iso_fit_workspace_bytes(rows, n, w != NULL)
 *             bytes, 256-byte aligned; may be NULL when that size is 0.  Its
 *             contents on entry do not matter.  Calls that share one workspace
 *             must not overlap in time (use one stream).
 *  row_status [rows] uint32, device, written, or NULL: 0 or ISO_ROW_BAD_* bits.
 *  stream     cudaStream_t to enqueue on.
 *
 * Accuracy: cumulative sums are exact integer sums of values rounded to a
 * fixed-point grid of 2^-50 of the largest |w*y| (and |w|) of each chunk; the
 * fit deviates from the exact one by about that amount plus one float32
 * rounding of each slope.
 */
iso_status iso_fit(const float *y, const float *w, int64_t rows, int64_t n, int increasing,
                   float *out, uint8_t *blocks, void *workspace, size_t workspace_bytes,
                   uint32_t *row_status, void *stream);

/*
 * iso_fit_f64 -- iso_fit on float64 arrays.  The same fixed-point arithmetic:
 * values are rounded to 2^-50 of their tile's largest magnitude (a float64
 * value keeps 50 of its 53 bits at the tile's top exponent), sums and turns
 * are exact, and each slope is one float64 quotient of two integers, so the
 * fit deviates from the exact fit of the input by about 2^-49 of the row's
 * largest |y| (times the weights' dynamic range for weighted rows) plus one
 * float64 rounding.
 */
iso_status iso_fit_f64(const double *y, const double *w, int64_t rows, int64_t n, int increasing,
                       double *out, uint8_t *blocks, void *workspace, size_t workspace_bytes,
                       uint32_t *row_status, void *stream);

/* Bytes of device workspace that iso_backward needs (0 = none). */
size_t iso_backward_workspace_bytes(int64_t rows, int64_t n, int weighted);

/*
 * iso_backward -- vector-Jacobian product of the fit with respect to y.
 *
 * The paper's Section 6 "Gradient": the fit is constant on blocks and equals
 * the block's weighted mean, so with G and W the sums of grad and of w over
 * element i's block, d/dy_i = w_i * G / W (G / |block| for unit weights).
 * The blocks are those that iso_fit wrote into `blocks`.
 *
 *  grad       [rows, n] float32, device: gradient with respect to the fit.
 *  blocks     [rows, n] uint8, device: block starts as written by iso_fit
 *             (element 0 of a row is treated as a start whatever its value).
 *  w          [rows, n] float32 or NULL, the weights given to iso_fit.
 *  out        [rows, n] float32, device, written.
 *  workspace  as for iso_fit, of iso_backward_workspace_bytes(rows, n, w != NULL) bytes.
 *  stream     cudaStream_t.
 */
iso_status iso_backward(const float *grad, const uint8_t *blocks, const float *w, int64_t rows,
                        int64_t n, float *out, void *workspace, size_t workspace_bytes,
                        void *stream);

/* iso_backward on float64 arrays (grad, w, out); the blocks are iso_fit_f64's. */
iso_status iso_backward_f64(const double *grad, const uint8_t *blocks, const double *w,
                            int64_t rows, int64_t n, double *out, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * iso_backward_w -- the vector-Jacobian products of the fit with respect to y
 * and to the weights w.
 *
 * The paper's Section 6 "Gradient": on element i's block, with G and W the
 * sums of grad and of w over the block and z_i the block's weighted mean (the
 * fit), d/dy_i = w_i * G / W and d/dw_i = (y_i - z_i) * G / W.  The same
 * formulas hold for increasing and decreasing fits.
 *
 *  grad       [rows, n] float32, device: gradient with respect to the fit.
 *  blocks     [rows, n] uint8, device: block starts as written by iso_fit.
 *  w          [rows, n] float32 or NULL (unit weights), as given to iso_fit.
 *  y          [rows, n] float32, device: the input given to iso_fit.
 *  fit        [rows, n] float32, device: the fit iso_fit wrote.
 *  out_dy     [rows, n] float32, device, written; may be NULL (not wanted).
 *  out_dw     [rows, n] float32, device, written.
 *  workspace  as for iso_backward, of iso_backward_workspace_bytes(rows, n,
 *             w != NULL) bytes.
 *  stream     cudaStream_t.
 *
 * Errors: ISO_ERR_INVALID_ARG for a NULL grad, blocks, y, fit or out_dw or a
 * bad shape, ISO_ERR_WORKSPACE as for iso_backward, ISO_ERR_CUDA for a launch
 * failure.  A row whose forward pass was rejected (its fit is NaN) gets NaN.
 */
iso_status iso_backward_w(const float *grad, const uint8_t *blocks, const float *w,
                          const float *y, const float *fit, int64_t rows, int64_t n,
                          float *out_dy, float *out_dw, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * Bytes of device workspace that iso_fit_ragged needs for `segments` segments
 * covering `total` elements, none longer than max_len (max_len <= 0: total).
 * Returns 0 for invalid arguments (iso_fit_ragged then reports the error).
 */
size_t iso_fit_ragged_workspace_bytes(int64_t segments, int64_t total, int64_t max_len,
                                      int weighted);

/*
 * iso_fit_ragged -- forward fit of a ragged batch: segments of their own
 * lengths laid end to end, each fitted as its own row (eq. (1)-(3), Section
 * 2.1).  The paper fits such batches (many per-segment calibration curves,
 * Section 7.7) by padding them to a rectangle or by laying them end to end in
 * one row with each segment's targets lifted above the previous segment's;
 * here the offsets are given to the library, and every segment gets exactly
 * the fit iso_fit would give it as a row of its own.
 *
 *  y          [total] float32, device, read only: the segments end to end.
 *  w          [total] float32, device, read only, or NULL for unit weights.
 *  offsets    [segments + 1] int64, device, read only: segment s holds elements
 *             offsets[s] .. offsets[s+1]-1.  The offsets are not read by the
 *             host.  Non-decreasing offsets within [0, total] give disjoint
 *             segments; elements outside every segment are not written.
 *  segments   number of segments, 0 <= segments <= 2^31 - 1 (0: nothing to do).
 *  total      length of y (and w, out, blocks), 0 <= total <= 2^40 (with 0, y and
 *             out may be NULL and every segment is empty or rejected).
 *  max_len    an upper bound on the segments' lengths that the caller knows,
 *             or <= 0 for none (total).  It only saves launches and workspace:
 *             a segment longer than it is rejected (ISO_ROW_BAD_SHAPE).  At
 *             most 2^31 - 1.
 *  increasing as for iso_fit.
 *  out        [total] float32, device, written: each segment's fit.
 *  blocks     [total] uint8, device, written, or NULL: block starts as for
 *             iso_fit.  The first element of every non-empty segment that was
 *             not rejected for its shape is flagged 1, also in a segment
 *             rejected for its values (whose other flags are 0), so that
 *             iso_backward / iso_backward_w over the whole array as ONE row
 *             (rows = 1, n = total) give each segment its own backward, when
 *             the segments cover the array end to end.
 *  workspace  device scratch of iso_fit_ragged_workspace_bytes(segments,
 *             total, max_len, w != NULL) bytes, 256-byte aligned.
 *  row_status [segments] uint32, device, written, or NULL: per segment, 0 or
 *             ISO_ROW_BAD_* bits (an empty segment: 0).
 *  stream     cudaStream_t.
 *
 * The segments are sorted on the device into lists by length: up to 8,192
 * elements by the whole-row kernels (by lane class), longer ones by the
 * long-row path; no host synchronisation.  Accuracy as for iso_fit.
 */
iso_status iso_fit_ragged(const float *y, const float *w, const int64_t *offsets,
                          int64_t segments, int64_t total, int64_t max_len, int increasing,
                          float *out, uint8_t *blocks, void *workspace, size_t workspace_bytes,
                          uint32_t *row_status, void *stream);

/* iso_fit_ragged on float64 arrays (y, w, out); offsets and statuses as iso_fit_ragged. */
iso_status iso_fit_ragged_f64(const double *y, const double *w, const int64_t *offsets,
                              int64_t segments, int64_t total, int64_t max_len, int increasing,
                              double *out, uint8_t *blocks, void *workspace,
                              size_t workspace_bytes, uint32_t *row_status, void *stream);

/*
 * iso_fit_copy_control -- a measurement control, not a faster fit: the same
 * fit as iso_fit (bit for bit), with the merge levels of rows longer than
 * 8,192 elements run on materialised hulls instead of segment lists -- the
 * paper's "grid copying" control of Section 7.3: after every level's bridges
 * are found (the same search), every merged hull's surviving vertices are
 * copied into a second flat array by the whole grid.  It measures what the
 * segment lists save; rows of up to 8,192 elements (no merge tree) take the
 * whole-row kernels as in iso_fit.
 *
 * Arguments, results and errors as iso_fit, with a workspace of
 * iso_fit_copy_control_workspace_bytes(rows, n, weighted) bytes (about four
 * times iso_fit's: two flat buffers of C + 1 vertex records per chunk);
 * n <= 2^30.
 */
size_t iso_fit_copy_control_workspace_bytes(int64_t rows, int64_t n, int weighted);
iso_status iso_fit_copy_control(const float *y, const float *w, int64_t rows, int64_t n,
                                int increasing, float *out, uint8_t *blocks, void *workspace,
                                size_t workspace_bytes, uint32_t *row_status, void *stream);

/* iso_backward_w on float64 arrays. */
iso_status iso_backward_w_f64(const double *grad, const uint8_t *blocks, const double *w,
                              const double *y, const double *fit, int64_t rows, int64_t n,
                              double *out_dy, double *out_dw, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * iso_backward_noalloc -- iso_backward for callers that cannot allocate device
 * memory (no counterpart in the paper: it is an interface addition).
 *
 * Same arguments, results and errors as iso_backward, without the workspace:
 * the per-tile records that rows longer than 8,192 elements need live in a
 * fixed 2 MiB array inside the library (device memory that every GPU which
 * loads the library holds until the process exits), which limits such calls to
 * rows * ceil(n / 8192) <= 21,845 tiles; larger calls return ISO_ERR_WORKSPACE
 * and enqueue nothing.  Rows of at most 8,192 elements need no scratch and have
 * no such limit.
 *  - The first call on a device looks up the array's device address (once per
 *    device, on the calling thread's current device); make that first call
 *    before any stream capture.
 *  - Every call shares the one array: calls whose work may overlap on the GPU
 *    (different streams, several host threads) race on it and must be
 *    serialised by the caller.  Each call writes every record it reads, so
 *    nothing needs clearing between calls.
 *  - It calls no allocating function (no cudaMalloc, no cudaFree).
 */
iso_status iso_backward_noalloc(const float *grad, const uint8_t *blocks, const float *w,
                                int64_t rows, int64_t n, float *out, void *stream);

/*
 * Optional per-kernel timing for benchmarks (not part of the fit).
 * iso_profile_enable(1) makes the library create a few CUDA events (once, on
 * first use; the only state the library keeps) and record one before the first
 * kernel of every later iso_fit / iso_backward call and one after each of its
 * kernels, on the call's stream.  iso_profile_enable(0) stops the recording.
 * iso_profile_read waits for the events of the most recent call and writes the
 * duration of each of its kernels in launch order (milliseconds, into ms[0..])
 * and a static name for each (names may be NULL); it returns the number of
 * kernels, or a negative iso_status.  Calls must not run concurrently from
 * several host threads while profiling is enabled.
 */
int iso_profile_enable(int on);
int iso_profile_read(float *ms, const char **names, int max_kernels);

/*
 * Depth of the long-row path's bridge searches (the paper's Section 5.2,
 * Theorem 5.2: the merge depth is bounded by a capped walk followed by a
 * nested bisection over the left hull's vertices, each tested against its
 * tangent point on the right hull).
 *
 * A merge of two segment lists (hull vertices in global memory) moves the
 * bridge's ends alternately to each other's tangent points; after
 * ISO_BRIDGE_MAX_PASSES passes (a pass moves both ends) it finishes with the
 * nested bisection, so no merge takes more than that many passes.  A merge of
 * two flat hulls in shared memory uses the nested bisection from the start,
 * 32 candidates per round, at most ISO_BRIDGE_MAX_ROUNDS rounds after the
 * first window of 32 vertices next to the shared point.
 *
 * iso_bridge_stats_mode (a debugging aid, off by default) makes later long-row
 * fits on the current device count their bridge searches:
 *   mode 0: off;
 *   mode 1: count;
 *   mode 2: count, with every segment-list bridge search taking the nested
 *           bisection from its first pass (to test that path on any input).
 * Switching on allocates the device's eight counters once (cudaMalloc) and
 * zeroes them.  Returns ISO_OK, ISO_ERR_INVALID_ARG for another mode, or
 * ISO_ERR_CUDA.  Calls on several host threads must not change the mode
 * concurrently.
 *
 * iso_bridge_stats_read synchronises the current device and copies its
 * counters into out[0..7] (host memory):
 *   [0] segment-list merges
 *   [1] of those, bridge searches (the chain is not convex at the shared point)
 *   [2] passes, summed over those searches
 *   [3] the most passes of one search (at most ISO_BRIDGE_MAX_PASSES)
 *   [4] searches that ended in the nested bisection
 *   [5] flat merges with a bridge search
 *   [6] the most narrowing rounds of one flat search (at most ISO_BRIDGE_MAX_ROUNDS)
 *   [7] flat searches whose rounds ran out before the bridge was found (0 with
 *       exactly convex hulls; nonzero would mean a wrong merge)
 * It returns ISO_OK, ISO_ERR_INVALID_ARG for a NULL out or counting that was
 * never switched on for the device, or ISO_ERR_CUDA.
 */
#define ISO_BRIDGE_MAX_PASSES 6
#define ISO_BRIDGE_MAX_ROUNDS 8
iso_status iso_bridge_stats_mode(int mode);
iso_status iso_bridge_stats_read(uint64_t *out);

#ifdef __cplusplus
}
#endif

#endif /* ISO_H */
