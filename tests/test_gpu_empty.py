"""Empty inputs through the binding: no rows, rows of no elements, a ragged
batch with no elements (every segment empty: statuses 0) or no segments."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(0, 10), (5, 0), (0,)])
@pytest.mark.parametrize("dtype", ["float32", "float64"])
def test_empty_fit_and_backward(cuda_ok, shape, dtype):
    import torch
    import convex_hull_pava_gb300 as chp
    dt = getattr(torch, dtype)
    y = torch.empty(shape, dtype=dt, device="cuda")
    out, blocks, st = chp.iso_fit(y)
    assert out.shape == y.shape and blocks.shape == y.shape
    dy = chp.iso_backward(torch.empty(shape, dtype=dt, device="cuda"), blocks)
    assert dy.shape == y.shape
    yr = y.clone().requires_grad_(True)
    z = chp.isotonic(yr)
    z.sum().backward()
    assert yr.grad.shape == y.shape


def test_empty_ragged(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    y = torch.empty(0, device="cuda")
    off = torch.zeros(4, dtype=torch.int64, device="cuda")
    out, blocks, st = chp.iso_fit_ragged(y, off)
    torch.cuda.synchronize()
    assert out.numel() == 0 and st.cpu().numpy().tolist() == [0, 0, 0]
    out, blocks, st = chp.iso_fit_ragged(torch.arange(3.0, device="cuda"),
                                         torch.tensor([0, 3], device="cuda"))
    torch.cuda.synchronize()
    assert out.cpu().numpy().tolist() == [0.0, 1.0, 2.0]
