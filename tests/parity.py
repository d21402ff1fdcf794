"""Parity criteria between the CUDA path and the fp64 oracle.

* Fit: max_i |out_i - z*_i| <= 1e-5 * (1 + max_i |y_i|) per row, with z* the
  oracle's fp64 value (not rounded to fp32).
* Blocks: every oracle block boundary whose adjacent block means differ by more
  than 1e-6 relative (|m_k - m_{k-1}| > 1e-6 * max(|m_k|, |m_{k-1}|)) and by
  more than 2^-44 * max|y| (the data's scale: below it neither the oracle's
  fp64 sums nor the 2^-50 fixed-point grid of the CUDA path decide the order,
  so such a pair is a tie) must be a boundary of the CUDA path; a CUDA boundary that the oracle does not have must
  split a tie (|out_i - out_{i-1}| within the fit tolerance); inside one CUDA
  block the output is constant; element 0 starts a block.

float64 I/O: the fit is within 1e-13 * (1 + max|y|) * max(1, max w / min w).
The CUDA path rounds each value to 2^-50 of its tile's largest magnitude and
vertex coordinates to the row's grid, so its fit moves by about 2^-48 of max|y|
(3.6e-15); for weighted rows the grid of the weights is coarser, relative to a
small weight, by the weights' dynamic range.  The bar leaves a margin of about
30.  Required boundaries: means that differ by more than 1e-12 relative and by
more than 2^-44 * max|y| times the same weight ratio.
"""
import numpy as np

FIT_TOL = 1e-5
GAP_REL = 1e-6
GAP_FLOOR = 2.0 ** -44

FIT_TOL_F64 = 1e-13
GAP_REL_F64 = 1e-12
GAP_FLOOR_F64 = 2.0 ** -44


def f64_params(w):
    """(tol, gap_rel, gap_floor) of float64 parity for a row's weights."""
    ratio = 1.0 if w is None else float(np.max(w) / np.min(w))
    return FIT_TOL_F64 * max(1.0, ratio), GAP_REL_F64, GAP_FLOOR_F64 * max(1.0, ratio)


def fit_tol(y):
    y = np.asarray(y, dtype=np.float64)
    return FIT_TOL * (1.0 + np.abs(y).max(axis=-1))


def check_row(y, out, blocks, z, zb, label="", fit_tol=FIT_TOL, gap_rel=GAP_REL,
              gap_floor=GAP_FLOOR):
    """y: float32 [n]; out: float32 [n] (CUDA); blocks: uint8 [n] (CUDA);
    z: float64 [n] (oracle); zb: uint8 [n] (oracle block starts)."""
    y = np.asarray(y, np.float64)
    out = np.asarray(out, np.float64)
    tol = fit_tol * (1.0 + np.abs(y).max())
    err = np.abs(out - z)
    imax = int(err.argmax())
    assert err[imax] <= tol, f"{label}: fit error {err[imax]:.3e} > {tol:.3e} at {imax} (out {out[imax]!r}, oracle {z[imax]!r})"
    if blocks is None:
        return
    blocks = np.asarray(blocks).astype(bool)
    zb = np.asarray(zb).astype(bool)
    assert blocks[0], f"{label}: element 0 does not start a block"
    n = y.size
    if n > 1:
        inner = ~blocks[1:]
        bad = np.nonzero(inner & (out[1:] != out[:-1]))[0]
        assert bad.size == 0, f"{label}: output not constant inside a block at {bad[:5] + 1}"
        gap = np.abs(z[1:] - z[:-1])
        scale = np.maximum(np.abs(z[1:]), np.abs(z[:-1]))
        required = zb[1:] & (gap > gap_rel * scale) & (gap > gap_floor * np.abs(y).max())
        missing = np.nonzero(required & ~blocks[1:])[0]
        assert missing.size == 0, f"{label}: oracle boundaries missing at {missing[:5] + 1} (gaps {gap[missing[:5]]})"
        extra = np.nonzero(blocks[1:] & ~zb[1:])[0]
        if extra.size:
            d = np.abs(out[1:] - out[:-1])[extra]
            assert d.max() <= tol, f"{label}: extra boundaries that are not ties at {extra[:5] + 1}"


def check_rows(y, out, blocks, z, zb, label=""):
    y = np.atleast_2d(y)
    out = np.atleast_2d(out)
    z = np.atleast_2d(z)
    zb = np.atleast_2d(zb)
    blocks = None if blocks is None else np.atleast_2d(blocks)
    for r in range(y.shape[0]):
        check_row(y[r], out[r], None if blocks is None else blocks[r], z[r], zb[r], f"{label} row {r}")


def check_batch(y, out, blocks, z, zb, label=""):
    """check_row's criteria (float32 I/O) over every row of a [rows, n] batch at
    once, vectorised for batches of many short rows."""
    y = np.atleast_2d(np.asarray(y, np.float64))
    out = np.atleast_2d(np.asarray(out, np.float64))
    z = np.atleast_2d(np.asarray(z, np.float64))
    blocks = np.atleast_2d(np.asarray(blocks)).astype(bool)
    zb = np.atleast_2d(np.asarray(zb)).astype(bool)
    ymax = np.abs(y).max(axis=1, keepdims=True)
    tol = FIT_TOL * (1.0 + ymax)
    err = np.abs(out - z)
    bad = np.nonzero((err > tol).any(axis=1))[0]
    assert bad.size == 0, f"{label}: fit error above tolerance in rows {bad[:5]}"
    assert blocks[:, 0].all(), f"{label}: element 0 does not start a block in rows {np.nonzero(~blocks[:, 0])[0][:5]}"
    if y.shape[1] < 2:
        return
    inner = ~blocks[:, 1:]
    r, c = np.nonzero(inner & (out[:, 1:] != out[:, :-1]))
    assert r.size == 0, f"{label}: output not constant inside a block at rows {r[:5]}, elements {c[:5] + 1}"
    gap = np.abs(z[:, 1:] - z[:, :-1])
    scale = np.maximum(np.abs(z[:, 1:]), np.abs(z[:, :-1]))
    required = zb[:, 1:] & (gap > GAP_REL * scale) & (gap > GAP_FLOOR * ymax)
    r, c = np.nonzero(required & ~blocks[:, 1:])
    assert r.size == 0, f"{label}: oracle boundaries missing at rows {r[:5]}, elements {c[:5] + 1}"
    r, c = np.nonzero(blocks[:, 1:] & ~zb[:, 1:])
    if r.size:
        d = np.abs(out[r, c + 1] - out[r, c])
        assert (d <= tol[r, 0]).all(), f"{label}: extra boundaries that are not ties at rows {r[:5]}"
