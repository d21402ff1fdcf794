"""Reference oracle for weighted isotonic regression (fp64, CPU).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never links, loads or calls it, and it never calls the CUDA library.

The arithmetic lives in ``iso_oracle.c`` (plain C, compiled with gcc by
:func:`build`); this module only marshals numpy arrays.  Citations are to
"Merge Hulls Without Copying Vertices: GPU Isotonic Regression" (the paper):

* :func:`pava` -- weighted pool adjacent violators in fp64, Section 2.1, eq. (1).
* :func:`hull_fit` -- lower hull of the cumulative-sum diagram, Section 2.1,
  eqs. (2)-(3); an independent route used only to cross-check :func:`pava`.
* :func:`points` -- the cumulative-sum diagram itself, eq. (2).
* :func:`backward` / :func:`backward_w` -- block averaging, Section 6, "Gradient".
* :func:`pava_f64`, :func:`backward_f64`, :func:`backward_w_f64` -- the same
  definitions for float64 inputs, with sums in double-double (about 106
  bits), Section 6 "Implementation" (float32 and float64 working types).
* :func:`pava_ragged` -- a ragged batch (segments of unequal lengths laid end
  to end, Section 7.7): each segment fitted as its own row by :func:`pava`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "iso_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libiso_oracle.so")
_lib = None
_lock = threading.Lock()

BAD_Y = 1
BAD_W = 2
BAD_SHAPE = 4


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: it runs on x86_64 and aarch64)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-adds, so every operation rounds as written.
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            for name in ("oracle_pava_rows", "oracle_hull_rows"):
                f = getattr(lib, name)
                f.argtypes = [i64, i64, vp, vp, ci, vp, vp, vp]
                f.restype = None
            lib.oracle_points.argtypes = [i64, vp, vp, ci, vp, vp]
            lib.oracle_points.restype = None
            lib.oracle_backward_rows.argtypes = [i64, i64, vp, vp, vp, vp]
            lib.oracle_backward_rows.restype = None
            lib.oracle_backward_w.argtypes = [i64, vp, vp, vp, vp, vp, vp]
            lib.oracle_backward_w.restype = None
            lib.oracle_pava_rows_f64.argtypes = [i64, i64, vp, vp, ci, vp, vp, vp]
            lib.oracle_pava_rows_f64.restype = None
            lib.oracle_backward_rows_f64.argtypes = [i64, i64, vp, vp, vp, vp]
            lib.oracle_backward_rows_f64.restype = None
            lib.oracle_backward_w_f64.argtypes = [i64, vp, vp, vp, vp, vp, vp]
            lib.oracle_backward_w_f64.restype = None
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _as2d(y, w):
    y = _f32(y)
    squeeze = y.ndim == 1
    y2 = y.reshape(1, -1) if squeeze else y
    w2 = None
    if w is not None:
        w2 = _f32(w).reshape(y2.shape)
    return y2, w2, squeeze


def _rows(fn_name, y, w, increasing):
    y2, w2, squeeze = _as2d(y, w)
    rows, n = y2.shape
    z = np.empty((rows, n), dtype=np.float64)
    blocks = np.empty((rows, n), dtype=np.uint8)
    status = np.empty(rows, dtype=np.uint32)
    getattr(_load(), fn_name)(rows, n, _ptr(y2), _ptr(w2), int(bool(increasing)),
                              _ptr(z), _ptr(blocks), _ptr(status))
    if squeeze:
        return z[0], blocks[0], status[0]
    return z, blocks, status


def pava(y, w=None, increasing=True):
    """Fit by weighted PAVA in fp64.  Returns ``(z, blocks, status)``.

    ``y``: float32 ``[n]`` or ``[rows, n]``; ``w``: same shape or None (unit
    weights).  ``z`` is float64, ``blocks[i] == 1`` where element i starts a
    block, ``status`` is 0 or a mask of :data:`BAD_Y` / :data:`BAD_W` per row
    (that row's z is NaN)."""
    return _rows("oracle_pava_rows", y, w, increasing)


def hull_fit(y, w=None, increasing=True):
    """Fit by the lower hull of the cumulative-sum diagram (fp64 monotone chain)."""
    return _rows("oracle_hull_rows", y, w, increasing)


def points(y, w=None, increasing=True):
    """Cumulative-sum diagram of one row: arrays ``W, S`` of n+1 entries, eq. (2)."""
    y = _f32(y).ravel()
    n = y.size
    w1 = None if w is None else _f32(w).ravel()
    W = np.empty(n + 1, dtype=np.float64)
    S = np.empty(n + 1, dtype=np.float64)
    _load().oracle_points(n, _ptr(y), _ptr(w1), int(bool(increasing)), _ptr(W), _ptr(S))
    return W, S


def backward(grad, blocks, w=None):
    """Block averaging: ``out_i = w_i * G_B / W_B`` over the blocks that
    ``blocks`` marks (uint8 block starts).  fp64 result."""
    g2 = _f32(grad)
    squeeze = g2.ndim == 1
    if squeeze:
        g2 = g2.reshape(1, -1)
    b2 = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(g2.shape)
    w2 = None if w is None else _f32(w).reshape(g2.shape)
    out = np.empty(g2.shape, dtype=np.float64)
    _load().oracle_backward_rows(g2.shape[0], g2.shape[1], _ptr(g2), _ptr(b2), _ptr(w2),
                                 _ptr(out))
    return out[0] if squeeze else out


def backward_w(grad, blocks, w, y, z):
    """Weight gradient of one row: ``(y_i - z_i) * G_B / W_B``."""
    g = _f32(grad).ravel()
    b = np.ascontiguousarray(blocks, dtype=np.uint8).ravel()
    w1 = None if w is None else _f32(w).ravel()
    y1 = _f32(y).ravel()
    z1 = np.ascontiguousarray(z, dtype=np.float64).ravel()
    out = np.empty(g.size, dtype=np.float64)
    _load().oracle_backward_w(g.size, _ptr(g), _ptr(b), _ptr(w1), _ptr(y1), _ptr(z1),
                              _ptr(out))
    return out


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def pava_f64(y, w=None, increasing=True):
    """Fit by weighted PAVA of float64 inputs, block sums in double-double.
    Same shapes and results as :func:`pava`."""
    y2 = _f64(y)
    squeeze = y2.ndim == 1
    if squeeze:
        y2 = y2.reshape(1, -1)
    w2 = None if w is None else _f64(w).reshape(y2.shape)
    rows, n = y2.shape
    z = np.empty((rows, n), dtype=np.float64)
    blocks = np.empty((rows, n), dtype=np.uint8)
    status = np.empty(rows, dtype=np.uint32)
    _load().oracle_pava_rows_f64(rows, n, _ptr(y2), _ptr(w2), int(bool(increasing)), _ptr(z),
                                 _ptr(blocks), _ptr(status))
    if squeeze:
        return z[0], blocks[0], status[0]
    return z, blocks, status


def backward_f64(grad, blocks, w=None):
    """Block averaging of float64 gradients (double-double block sums)."""
    g2 = _f64(grad)
    squeeze = g2.ndim == 1
    if squeeze:
        g2 = g2.reshape(1, -1)
    b2 = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(g2.shape)
    w2 = None if w is None else _f64(w).reshape(g2.shape)
    out = np.empty(g2.shape, dtype=np.float64)
    _load().oracle_backward_rows_f64(g2.shape[0], g2.shape[1], _ptr(g2), _ptr(b2), _ptr(w2),
                                     _ptr(out))
    return out[0] if squeeze else out


def backward_w_f64(grad, blocks, w, y, z):
    """Weight gradient of one float64 row: ``(y_i - z_i) * G_B / W_B``."""
    g = _f64(grad).ravel()
    b = np.ascontiguousarray(blocks, dtype=np.uint8).ravel()
    w1 = None if w is None else _f64(w).ravel()
    out = np.empty(g.size, dtype=np.float64)
    _load().oracle_backward_w_f64(g.size, _ptr(g), _ptr(b), _ptr(w1), _ptr(_f64(y).ravel()),
                                  _ptr(_f64(z).ravel()), _ptr(out))
    return out


def pava_ragged(y, offsets, w=None, increasing=True, max_len=0, f64=False):
    """Fit of a ragged batch: segment s, elements ``offsets[s] .. offsets[s+1]-1``
    of the 1-D ``y`` (and ``w``), fitted on its own by :func:`pava` (or
    :func:`pava_f64` when ``f64``) (Section
    7.7 fits such segments as separate curves).  Returns ``(z, blocks,
    status)``: ``z`` float64 and ``blocks`` uint8 over ``y`` (NaN / 0 outside
    every segment), ``status`` one word per segment.

    Conventions of the library's ragged interface: a segment whose offsets
    are out of order or out of ``[0, len(y)]``, or longer than ``max_len``
    (when > 0), gets :data:`BAD_SHAPE` and no fit; an empty segment gets 0; a
    segment rejected for its values keeps its first element flagged as a
    block start."""
    cast = _f64 if f64 else _f32
    fit = pava_f64 if f64 else pava
    y = cast(y).ravel()
    off = np.asarray(offsets, dtype=np.int64).ravel()
    w1 = None if w is None else cast(w).ravel()
    total, segments = y.size, off.size - 1
    lim = total if max_len is None or max_len <= 0 else min(int(max_len), total)
    z = np.full(total, np.nan)
    blocks = np.zeros(total, dtype=np.uint8)
    status = np.zeros(segments, dtype=np.uint32)
    for s in range(segments):
        a, b = int(off[s]), int(off[s + 1])
        if a < 0 or b < a or b > total or b - a > lim:
            status[s] = BAD_SHAPE
            continue
        if b == a:
            continue
        zs, bs, st = fit(y[a:b], None if w1 is None else w1[a:b], increasing)
        z[a:b] = zs
        blocks[a:b] = bs
        blocks[a] = 1
        status[s] = st
    return z, blocks, status
