"""The C ABI library builds, loads and exports every symbol include/iso.h
declares; host-side argument checks work without a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

import convex_hull_pava_gb300 as chp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "iso.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(iso_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_names_match_binding():
    assert set(declared_functions()) == set(chp.EXPORTS)


def test_library_loads_and_exports():
    lib = chp.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.iso_version() >= 100


def test_workspace_queries_host_only():
    assert chp.iso_fit_workspace_bytes(4096, 1024, False) == 0
    assert chp.iso_fit_workspace_bytes(1, 10_000_000, False) > 0
    assert chp.iso_fit_workspace_bytes(16, 4_194_304, True) > chp.iso_fit_workspace_bytes(16, 4_194_304, False)
    assert chp.iso_backward_workspace_bytes(1024, 8192, False) == 0
    assert chp.iso_backward_workspace_bytes(1, 10_000_000, False) > 0
    # invalid shapes report 0
    assert chp.iso_fit_workspace_bytes(0, 10, False) == 0
    assert chp.iso_fit_workspace_bytes(1, 0, False) == 0
    assert chp.iso_fit_workspace_bytes(1, 1 << 31, False) == 0


def test_invalid_arguments_rejected_on_host():
    lib = chp.load_library()
    fake = ctypes.c_void_p(0x1000)
    # NULL y / out, bad shapes, bad flag: rejected before any CUDA call
    assert lib.iso_fit(None, None, 1, 10, 1, fake, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit(fake, None, 1, 10, 1, None, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit(fake, None, -1, 10, 1, fake, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit(fake, None, 1, -3, 1, fake, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit(fake, None, 1, 10, 2, fake, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit(fake, None, 1 << 30, 1 << 30, 1, fake, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    # long rows need a workspace: missing / too small / misaligned
    need = lib.iso_fit_workspace_bytes(1, 100000, 0)
    assert lib.iso_fit(fake, None, 1, 100000, 1, fake, None, None, 0, None, None) == chp.ISO_ERR_WORKSPACE
    assert lib.iso_fit(fake, None, 1, 100000, 1, fake, None, ctypes.c_void_p(0x100000), need - 1, None, None) == chp.ISO_ERR_WORKSPACE
    assert lib.iso_fit(fake, None, 1, 100000, 1, fake, None, ctypes.c_void_p(0x100010), need, None, None) == chp.ISO_ERR_WORKSPACE
    assert lib.iso_backward(None, fake, None, 1, 10, fake, None, 0, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_backward(fake, None, None, 1, 10, fake, None, 0, None) == chp.ISO_ERR_INVALID_ARG
    nb = lib.iso_backward_workspace_bytes(1, 100000, 0)
    assert lib.iso_backward(fake, fake, None, 1, 100000, fake, None, 0, None) == chp.ISO_ERR_WORKSPACE
    assert nb > 0


def test_status_strings():
    assert chp.status_string(0) == "ok"
    assert "workspace" in chp.status_string(chp.ISO_ERR_WORKSPACE)


def test_binding_rejects_host_tensors_without_fallback():
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        chp.iso_fit(torch.zeros(10))


def test_ragged_host_checks():
    lib = chp.load_library()
    fake = ctypes.c_void_p(0x1000)
    # workspace: always needed (the device lists), grows with the long part
    short = chp.iso_fit_ragged_workspace_bytes(1000, 10**6, 8192, False)
    full = chp.iso_fit_ragged_workspace_bytes(1000, 10**6, 0, False)
    assert 0 < short < full
    assert chp.iso_fit_ragged_workspace_bytes(1000, 10**6, 0, True) > full
    assert chp.iso_fit_ragged_workspace_bytes(0, 10, 0, False) == 0
    assert chp.iso_fit_ragged_workspace_bytes(1, 0, 0, False) == 256   # the list counters only
    args = lambda y, off, segs, total, ml, inc, out, ws, wsb: (
        y, None, off, segs, total, ml, inc, out, None, ws, wsb, None, None)
    ws = ctypes.c_void_p(0x100000)
    assert lib.iso_fit_ragged(*args(None, fake, 1, 10, 0, 1, fake, ws, 1 << 30)) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit_ragged(*args(fake, None, 1, 10, 0, 1, fake, ws, 1 << 30)) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit_ragged(*args(fake, fake, -1, 10, 0, 1, fake, ws, 1 << 30)) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit_ragged(*args(fake, fake, 1, 10, 0, 3, fake, ws, 1 << 30)) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit_ragged(*args(fake, fake, 1, 1 << 32, 1 << 31, 1, fake, ws, 1 << 40)) == chp.ISO_ERR_INVALID_ARG
    need = chp.iso_fit_ragged_workspace_bytes(1, 10, 0, False)
    assert lib.iso_fit_ragged(*args(fake, fake, 1, 10, 0, 1, fake, None, 0)) == chp.ISO_ERR_WORKSPACE
    assert lib.iso_fit_ragged(*args(fake, fake, 1, 10, 0, 1, fake, ws, need - 1)) == chp.ISO_ERR_WORKSPACE
    assert lib.iso_fit_ragged(*args(fake, fake, 1, 10, 0, 1, fake, ctypes.c_void_p(0x100010), need)) == chp.ISO_ERR_WORKSPACE


def test_copy_control_host_checks():
    lib = chp.load_library()
    fake = ctypes.c_void_p(0x1000)
    assert chp.iso_fit_copy_control_workspace_bytes(4096, 1024, False) == 0
    big = chp.iso_fit_copy_control_workspace_bytes(1, 10_000_000, False)
    assert big > chp.iso_fit_workspace_bytes(1, 10_000_000, False)
    assert chp.iso_fit_copy_control_workspace_bytes(1, (1 << 30) + 1, False) == 0
    assert lib.iso_fit_copy_control(None, None, 1, 100000, 1, fake, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit_copy_control(fake, None, 1, (1 << 30) + 1, 1, fake, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit_copy_control(fake, None, 1, 100000, 1, fake, None, None, 0, None, None) == chp.ISO_ERR_WORKSPACE


def test_plain_host_tensors_rejected():
    """Host arrays must be pinned (device-accessible); pageable ones are refused
    before any CUDA call."""
    import torch
    with pytest.raises(ValueError):
        chp.iso_fit(torch.zeros(10))
    with pytest.raises(ValueError):
        chp.iso_backward(torch.zeros(10), torch.zeros(10, dtype=torch.uint8))


def test_empty_calls_do_nothing():
    """No rows, or rows of no elements (ragged: no segments): ISO_OK before any
    CUDA call, whatever the pointers; negative sizes are still errors."""
    lib = chp.load_library()
    for rows, n in [(0, 10), (5, 0), (0, 0)]:
        assert lib.iso_fit(None, None, rows, n, 1, None, None, None, 0, None, None) == chp.ISO_OK
        assert lib.iso_fit_f64(None, None, rows, n, 0, None, None, None, 0, None, None) == chp.ISO_OK
        assert lib.iso_backward(None, None, None, rows, n, None, None, 0, None) == chp.ISO_OK
        assert lib.iso_backward_w(None, None, None, None, None, rows, n, None, None, None, 0,
                                  None) == chp.ISO_OK
        assert lib.iso_backward_noalloc(None, None, None, rows, n, None, None) == chp.ISO_OK
        assert lib.iso_fit_copy_control(None, None, rows, n, 1, None, None, None, 0, None,
                                        None) == chp.ISO_OK
        assert chp.iso_fit_workspace_bytes(rows, n, False) == 0
    assert lib.iso_fit(None, None, 0, -1, 1, None, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit(None, None, 0, 10, 2, None, None, None, 0, None, None) == chp.ISO_ERR_INVALID_ARG
    assert lib.iso_fit_ragged(None, None, None, 0, 0, 0, 1, None, None, None, 0, None, None) == chp.ISO_OK


def test_bridge_bounds_match_header():
    src = open(os.path.join(ROOT, "include", "iso.h")).read()
    passes = int(re.search(r"#define ISO_BRIDGE_MAX_PASSES (\d+)", src).group(1))
    rounds = int(re.search(r"#define ISO_BRIDGE_MAX_ROUNDS (\d+)", src).group(1))
    assert (passes, rounds) == (chp.BRIDGE_MAX_PASSES, chp.BRIDGE_MAX_ROUNDS)
    assert len(chp.BRIDGE_STATS) == 8


def test_bridge_stats_mode_checks_host_only():
    # an unknown mode is refused before any CUDA call; mode 0 makes none
    with pytest.raises(chp.IsoError) as e:
        chp.bridge_stats_mode(3)
    assert e.value.status == chp.ISO_ERR_INVALID_ARG
    chp.bridge_stats_mode(0)
