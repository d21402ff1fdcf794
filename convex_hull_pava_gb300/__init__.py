"""GB300 (sm_103a) batched and long-row weighted isotonic regression.

Thin Python binding over the C ABI of ``libiso.so`` (declared in
``include/iso.h``): argument marshalling only.  Every step of the fit and of its
backward runs in the library's CUDA kernels; PyTorch supplies device memory
and the current stream.  There is no CPU fallback: without the compiled
library or a CUDA device the calls raise.

Entry points (same names as the C ABI):

* :func:`iso_fit` -- forward fit of ``[rows, n]`` float32 or float64 CUDA
  tensors (float64 calls go to the ABI's ``_f64`` twins).
* :func:`iso_backward` -- block-averaging backward.
* :func:`iso_fit_ragged` -- forward fit of segments of unequal lengths laid
  end to end (int64 offsets on the device).
* :func:`iso_fit_workspace_bytes`, :func:`iso_backward_workspace_bytes`,
  :func:`iso_fit_ragged_workspace_bytes`.
* :func:`isotonic` -- differentiable convenience op (autograd), which also
  accepts host tensors (copied to the GPU and back); :func:`isotonic_ragged`,
  its counterpart for a ragged batch.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libiso.so")

ISO_OK = 0
ISO_ERR_INVALID_ARG = -1
ISO_ERR_WORKSPACE = -2
ISO_ERR_CUDA = -3
ISO_ERR_TIMEOUT = -4
ISO_ROW_BAD_Y = 1
ISO_ROW_BAD_W = 2
ISO_ROW_BAD_SHAPE = 4

EXPORTS = ("iso_version", "iso_status_string", "iso_fit_workspace_bytes", "iso_fit",
           "iso_backward_workspace_bytes", "iso_backward", "iso_backward_w",
           "iso_backward_noalloc", "iso_fit_ragged_workspace_bytes", "iso_fit_ragged",
           "iso_fit_copy_control_workspace_bytes", "iso_fit_copy_control",
           "iso_fit_f64", "iso_backward_f64", "iso_backward_w_f64", "iso_fit_ragged_f64",
           "iso_profile_enable", "iso_profile_read", "iso_bridge_stats_mode",
           "iso_bridge_stats_read")

_lib = None
_lock = threading.Lock()


class IsoError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load_library(path: str | None = None):
    """Load libiso.so (building it first if it is missing and nvcc is present)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            from . import _build
            _build.build()
        lib = ctypes.CDLL(p)
        i64, vp, ci, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.iso_version.argtypes = []
        lib.iso_version.restype = ci
        lib.iso_status_string.argtypes = [ci]
        lib.iso_status_string.restype = ctypes.c_char_p
        lib.iso_fit_workspace_bytes.argtypes = [i64, i64, ci]
        lib.iso_fit_workspace_bytes.restype = sz
        lib.iso_backward_workspace_bytes.argtypes = [i64, i64, ci]
        lib.iso_backward_workspace_bytes.restype = sz
        lib.iso_fit.argtypes = [vp, vp, i64, i64, ci, vp, vp, vp, sz, vp, vp]
        lib.iso_fit.restype = ci
        lib.iso_backward.argtypes = [vp, vp, vp, i64, i64, vp, vp, sz, vp]
        lib.iso_backward.restype = ci
        lib.iso_backward_w.argtypes = [vp, vp, vp, vp, vp, i64, i64, vp, vp, vp, sz, vp]
        lib.iso_backward_w.restype = ci
        lib.iso_backward_noalloc.argtypes = [vp, vp, vp, i64, i64, vp, vp]
        lib.iso_backward_noalloc.restype = ci
        lib.iso_fit_ragged_workspace_bytes.argtypes = [i64, i64, i64, ci]
        lib.iso_fit_ragged_workspace_bytes.restype = sz
        lib.iso_fit_ragged.argtypes = [vp, vp, vp, i64, i64, i64, ci, vp, vp, vp, sz, vp, vp]
        lib.iso_fit_ragged.restype = ci
        lib.iso_fit_copy_control_workspace_bytes.argtypes = [i64, i64, ci]
        lib.iso_fit_copy_control_workspace_bytes.restype = sz
        lib.iso_fit_copy_control.argtypes = [vp, vp, i64, i64, ci, vp, vp, vp, sz, vp, vp]
        lib.iso_fit_copy_control.restype = ci
        for name in ("iso_fit", "iso_backward", "iso_backward_w", "iso_fit_ragged"):
            f64 = getattr(lib, name + "_f64")
            f64.argtypes = getattr(lib, name).argtypes
            f64.restype = ci
        lib.iso_profile_enable.argtypes = [ci]
        lib.iso_profile_enable.restype = ci
        lib.iso_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float),
                                         ctypes.POINTER(ctypes.c_char_p), ci]
        lib.iso_profile_read.restype = ci
        lib.iso_bridge_stats_mode.argtypes = [ci]
        lib.iso_bridge_stats_mode.restype = ci
        lib.iso_bridge_stats_read.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
        lib.iso_bridge_stats_read.restype = ci
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().iso_status_string(int(status)).decode()


def iso_fit_workspace_bytes(rows: int, n: int, weighted: bool) -> int:
    return int(load_library().iso_fit_workspace_bytes(int(rows), int(n), int(bool(weighted))))


def iso_backward_workspace_bytes(rows: int, n: int, weighted: bool) -> int:
    return int(load_library().iso_backward_workspace_bytes(int(rows), int(n), int(bool(weighted))))


def iso_fit_ragged_workspace_bytes(segments: int, total: int, max_len: int, weighted: bool) -> int:
    return int(load_library().iso_fit_ragged_workspace_bytes(int(segments), int(total),
                                                             int(max_len), int(bool(weighted))))


def profile_enable(on: bool = True) -> None:
    """Record CUDA events around every kernel of later calls (benchmarks only)."""
    st = load_library().iso_profile_enable(int(bool(on)))
    if st != ISO_OK:
        raise IsoError(st, "iso_profile_enable")


def profile_read(max_kernels: int = 16):
    """Per-kernel durations (ms) of the most recent call: list of (name, ms)."""
    ms = (ctypes.c_float * max_kernels)()
    names = (ctypes.c_char_p * max_kernels)()
    k = load_library().iso_profile_read(ms, names, max_kernels)
    if k < 0:
        raise IsoError(k, "iso_profile_read")
    return [(names[i].decode(), float(ms[i])) for i in range(k)]


BRIDGE_MAX_PASSES = 6   # ISO_BRIDGE_MAX_PASSES
BRIDGE_MAX_ROUNDS = 8   # ISO_BRIDGE_MAX_ROUNDS
BRIDGE_STATS = ("list_merges", "list_searches", "passes", "max_passes", "nested",
                "flat_searches", "max_rounds", "flat_unfinished")


def bridge_stats_mode(mode: int) -> None:
    """Count the long-row merges' bridge searches on the current device
    (0: off, 1: count, 2: count with every segment-list search taking the
    nested bisection from its first pass).  A debugging aid."""
    st = load_library().iso_bridge_stats_mode(int(mode))
    if st != ISO_OK:
        raise IsoError(st, "iso_bridge_stats_mode")


def bridge_stats_read() -> dict:
    """The current device's bridge-search counters (synchronises the device)."""
    v = (ctypes.c_uint64 * 8)()
    st = load_library().iso_bridge_stats_read(v)
    if st != ISO_OK:
        raise IsoError(st, "iso_bridge_stats_read")
    return {k: int(v[i]) for i, k in enumerate(BRIDGE_STATS)}


def _torch():
    import torch
    return torch


def _check_dev(t, name, dtype):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_io(t, name, dtype):
    """A CUDA tensor, or a pinned (page-locked) host tensor: with unified
    addressing a pinned allocation is device-accessible at the same address,
    so the kernels read and write it in place over the host link."""
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _gpu(t):
    """The device a call on t runs on (the current device for host tensors)."""
    torch = _torch()
    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _empty_io(shape, dtype, like):
    """An output next to `like`: on its device, or pinned host memory."""
    torch = _torch()
    if like.is_cuda:
        return torch.empty(shape, dtype=dtype, device=like.device)
    return torch.empty(shape, dtype=dtype, pin_memory=True)


def _io_dtype(t, name):
    """The I/O type of a call: float32 or float64, taken from its first array."""
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype not in (torch.float32, torch.float64):
        raise ValueError(f"{name} must be a float32 or float64 tensor")
    return t.dtype


def _entry(name, dtype):
    """The ABI function for the I/O type: name, or name + '_f64' for float64."""
    torch = _torch()
    return getattr(load_library(), name + ("_f64" if dtype == torch.float64 else ""))


def _shape2(t):
    if t.dim() == 1:
        return 1, t.shape[0]
    if t.dim() == 2:
        return t.shape[0], t.shape[1]
    raise ValueError("expected a [n] or [rows, n] tensor")


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(nbytes, workspace, device):
    torch = _torch()
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def iso_fit(y, w=None, increasing: bool = True, *, out=None, blocks=None, want_blocks: bool = True,
            row_status=None, workspace=None, stream=None):
    """Fit every row of ``y`` (float32 CUDA, ``[n]`` or ``[rows, n]``).

    Returns ``(out, blocks, row_status)``; ``blocks`` is None when
    ``want_blocks`` is False and none was given.  ``workspace`` may be a uint8
    CUDA tensor of at least :func:`iso_fit_workspace_bytes` bytes (allocated
    here otherwise).  y, w, out and blocks may also be pinned host tensors:
    the kernels then read and write them in place over the host link (outputs
    allocated here follow y)."""
    torch = _torch()
    dt = _io_dtype(y, "y")
    _check_io(y, "y", dt)
    rows, n = _shape2(y)
    if w is not None:
        _check_io(w, "w", dt)
        if w.shape != y.shape:
            raise ValueError("w must have the shape of y")
    if out is None:
        out = _empty_io(y.shape, dt, y)
    _check_io(out, "out", dt)
    if blocks is None and want_blocks:
        blocks = _empty_io(y.shape, torch.uint8, y)
    if blocks is not None:
        _check_io(blocks, "blocks", torch.uint8)
    if row_status is None:
        row_status = _empty_io((rows,), torch.int32, y)
    nbytes = iso_fit_workspace_bytes(rows, n, w is not None)
    ws, ws_bytes = _workspace(nbytes, workspace, _gpu(y))
    st = _entry("iso_fit", dt)(
        y.data_ptr(), None if w is None else w.data_ptr(), rows, n, int(bool(increasing)),
        out.data_ptr(), None if blocks is None else blocks.data_ptr(),
        None if ws is None else ws.data_ptr(), ws_bytes, row_status.data_ptr(), _stream_ptr(stream))
    if st != ISO_OK:
        raise IsoError(st, "iso_fit")
    return out, blocks, row_status


def iso_fit_copy_control_workspace_bytes(rows: int, n: int, weighted: bool) -> int:
    return int(load_library().iso_fit_copy_control_workspace_bytes(int(rows), int(n),
                                                                   int(bool(weighted))))


def iso_fit_copy_control(y, w=None, increasing: bool = True, *, out=None, blocks=None,
                         row_status=None, workspace=None, stream=None):
    """The materialised-copy control (measurement only): :func:`iso_fit`'s
    result, with every merge level's hulls copied into flat arrays instead of
    kept as segment lists.  Returns ``(out, blocks, row_status)``."""
    torch = _torch()
    _check_dev(y, "y", torch.float32)
    rows, n = _shape2(y)
    if w is not None:
        _check_dev(w, "w", torch.float32)
        if w.shape != y.shape:
            raise ValueError("w must have the shape of y")
    if out is None:
        out = torch.empty_like(y)
    if blocks is None:
        blocks = torch.empty(y.shape, dtype=torch.uint8, device=y.device)
    if row_status is None:
        row_status = torch.empty(rows, dtype=torch.int32, device=y.device)
    nbytes = iso_fit_copy_control_workspace_bytes(rows, n, w is not None)
    ws, ws_bytes = _workspace(nbytes, workspace, y.device)
    st = load_library().iso_fit_copy_control(
        y.data_ptr(), None if w is None else w.data_ptr(), rows, n, int(bool(increasing)),
        out.data_ptr(), blocks.data_ptr(), None if ws is None else ws.data_ptr(), ws_bytes,
        row_status.data_ptr(), _stream_ptr(stream))
    if st != ISO_OK:
        raise IsoError(st, "iso_fit_copy_control")
    return out, blocks, row_status


def iso_fit_ragged(y, offsets, w=None, increasing: bool = True, *, max_len: int = 0, out=None,
                   blocks=None, want_blocks: bool = True, row_status=None, workspace=None,
                   stream=None):
    """Fit each segment ``y[offsets[s]:offsets[s+1]]`` of a 1-D float32 CUDA
    tensor as its own row.  ``offsets``: int64 CUDA tensor of ``segments + 1``
    entries (not read by the host).  ``max_len``: an upper bound on the
    segments' lengths, or 0 for none; a longer segment is rejected
    (``ISO_ROW_BAD_SHAPE`` in its status word).  Returns ``(out, blocks,
    row_status)``, ``row_status`` one word per segment."""
    torch = _torch()
    dt = _io_dtype(y, "y")
    _check_io(y, "y", dt)
    _check_io(offsets, "offsets", torch.int64)
    if y.dim() != 1 or offsets.dim() != 1 or offsets.numel() < 2:
        raise ValueError("expected a 1-D y and at least two offsets")
    total, segments = y.numel(), offsets.numel() - 1
    if w is not None:
        _check_io(w, "w", dt)
        if w.shape != y.shape:
            raise ValueError("w must have the shape of y")
    if out is None:
        out = _empty_io(y.shape, dt, y)
    if blocks is None and want_blocks:
        blocks = _empty_io(y.shape, torch.uint8, y)
    if blocks is not None:
        _check_io(blocks, "blocks", torch.uint8)
    if row_status is None:
        row_status = _empty_io((segments,), torch.int32, y)
    nbytes = iso_fit_ragged_workspace_bytes(segments, total, max_len, w is not None)
    ws, ws_bytes = _workspace(nbytes, workspace, _gpu(y))
    _check_io(out, "out", dt)
    st = _entry("iso_fit_ragged", dt)(
        y.data_ptr(), None if w is None else w.data_ptr(), offsets.data_ptr(), segments, total,
        int(max_len), int(bool(increasing)), out.data_ptr(),
        None if blocks is None else blocks.data_ptr(), None if ws is None else ws.data_ptr(),
        ws_bytes, row_status.data_ptr(), _stream_ptr(stream))
    if st != ISO_OK:
        raise IsoError(st, "iso_fit_ragged")
    return out, blocks, row_status


def iso_backward(grad, blocks, w=None, *, out=None, workspace=None, stream=None):
    """Block-averaging backward: ``out_i = w_i * G / W`` over the blocks of ``blocks``."""
    torch = _torch()
    dt = _io_dtype(grad, "grad")
    _check_io(grad, "grad", dt)
    _check_io(blocks, "blocks", torch.uint8)
    rows, n = _shape2(grad)
    if w is not None:
        _check_io(w, "w", dt)
    if out is None:
        out = _empty_io(grad.shape, dt, grad)
    _check_io(out, "out", dt)
    nbytes = iso_backward_workspace_bytes(rows, n, w is not None)
    ws, ws_bytes = _workspace(nbytes, workspace, _gpu(grad))
    st = _entry("iso_backward", dt)(
        grad.data_ptr(), blocks.data_ptr(), None if w is None else w.data_ptr(), rows, n,
        out.data_ptr(), None if ws is None else ws.data_ptr(), ws_bytes, _stream_ptr(stream))
    if st != ISO_OK:
        raise IsoError(st, "iso_backward")
    return out


def iso_backward_w(grad, blocks, w, y, fit, *, out_dy=None, out_dw=None, want_dy=True,
                   workspace=None, stream=None):
    """Gradients with respect to y and to the weights: ``d/dy_i = w_i * G / W`` and
    ``d/dw_i = (y_i - z_i) * G / W`` over the blocks of ``blocks`` (``w`` may be
    None: unit weights).  Returns ``(dy or None, dw)``."""
    torch = _torch()
    dt = _io_dtype(grad, "grad")
    _check_io(grad, "grad", dt)
    _check_io(blocks, "blocks", torch.uint8)
    _check_io(y, "y", dt)
    _check_io(fit, "fit", dt)
    rows, n = _shape2(grad)
    if w is not None:
        _check_io(w, "w", dt)
    if want_dy and out_dy is None:
        out_dy = _empty_io(grad.shape, dt, grad)
    if out_dw is None:
        out_dw = _empty_io(grad.shape, dt, grad)
    nbytes = iso_backward_workspace_bytes(rows, n, w is not None)
    ws, ws_bytes = _workspace(nbytes, workspace, _gpu(grad))
    st = _entry("iso_backward_w", dt)(
        grad.data_ptr(), blocks.data_ptr(), None if w is None else w.data_ptr(), y.data_ptr(),
        fit.data_ptr(), rows, n, None if out_dy is None else out_dy.data_ptr(),
        out_dw.data_ptr(), None if ws is None else ws.data_ptr(), ws_bytes, _stream_ptr(stream))
    if st != ISO_OK:
        raise IsoError(st, "iso_backward_w")
    return out_dy, out_dw


def iso_backward_noalloc(grad, blocks, w=None, *, out=None, stream=None):
    """Backward without a workspace, for callers that cannot allocate device
    memory: long rows use a fixed scratch array inside the library (limit:
    rows * ceil(n / 8192) <= 21,845), and calls that may overlap on the GPU
    must be serialised by the caller."""
    torch = _torch()
    _check_dev(grad, "grad", torch.float32)
    _check_dev(blocks, "blocks", torch.uint8)
    rows, n = _shape2(grad)
    if w is not None:
        _check_dev(w, "w", torch.float32)
    if out is None:
        out = torch.empty_like(grad)
    st = load_library().iso_backward_noalloc(
        grad.data_ptr(), blocks.data_ptr(), None if w is None else w.data_ptr(), rows, n,
        out.data_ptr(), _stream_ptr(stream))
    if st != ISO_OK:
        raise IsoError(st, "iso_backward_noalloc")
    return out


def _make_function():
    torch = _torch()

    class _Isotonic(torch.autograd.Function):
        @staticmethod
        def forward(ctx, y, w, increasing):
            y = y.contiguous()
            w = None if w is None else w.contiguous()
            out, blocks, _ = iso_fit(y, w, increasing)
            ctx.save_for_backward(blocks, w, y, out)
            return out

        @staticmethod
        def backward(ctx, g):
            blocks, w, y, out = ctx.saved_tensors
            g = g.contiguous()
            if w is not None and ctx.needs_input_grad[1]:
                gy, gw = iso_backward_w(g, blocks, w, y, out, want_dy=ctx.needs_input_grad[0])
                return gy, gw, None
            return iso_backward(g, blocks, w), None, None

    class _IsotonicRagged(torch.autograd.Function):
        # Every segment's first element starts a block, so the backward of the
        # whole array as one row is each segment's own backward.
        @staticmethod
        def forward(ctx, y, offsets, w, increasing, max_len):
            y = y.contiguous()
            w = None if w is None else w.contiguous()
            out, blocks, _ = iso_fit_ragged(y, offsets, w, increasing, max_len=max_len)
            ctx.save_for_backward(blocks, w, y, out)
            return out

        @staticmethod
        def backward(ctx, g):
            blocks, w, y, out = ctx.saved_tensors
            g = g.contiguous()
            if w is not None and ctx.needs_input_grad[2]:
                gy, gw = iso_backward_w(g, blocks, w, y, out, want_dy=ctx.needs_input_grad[0])
                return gy, None, gw, None, None
            return iso_backward(g, blocks, w), None, None, None, None

    return _Isotonic, _IsotonicRagged


_Fn = None
_FnRagged = None


def isotonic(y, w=None, increasing: bool = True):
    """Differentiable isotonic regression of each row of ``y`` (gradients with
    respect to ``y`` and, when it requires one, to ``w``).  Host tensors are
    copied to the current CUDA device and the result is copied back."""
    global _Fn, _FnRagged
    torch = _torch()
    if _Fn is None:
        _Fn, _FnRagged = _make_function()
    host = not y.is_cuda
    if host:
        dev = torch.device("cuda", torch.cuda.current_device())
        y = y.to(dev, non_blocking=True)
        w = None if w is None else w.to(dev, non_blocking=True)
    z = _Fn.apply(y, w, bool(increasing))
    if host:
        z = z.to("cpu")
    return z


def isotonic_ragged(y, offsets, w=None, increasing: bool = True, max_len: int = 0):
    """Differentiable fit of each segment ``y[offsets[s]:offsets[s+1]]`` of a
    1-D CUDA tensor (gradients with respect to ``y`` and, when it requires one,
    to ``w``).  The backward assumes the segments cover ``y`` end to end
    (``offsets[0] == 0``, ``offsets[-1] == len(y)``, non-decreasing)."""
    global _Fn, _FnRagged
    if _FnRagged is None:
        _Fn, _FnRagged = _make_function()
    return _FnRagged.apply(y, offsets, w, bool(increasing), int(max_len))
