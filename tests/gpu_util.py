"""Helpers shared by the GPU parity tests: device copies of oracle-made inputs and the tolerance check
|y_gpu - y_ref| <= tol * sum_k |w_k x_k| (elementwise; NaN must match NaN)."""
import numpy as np
import pytest

# Tolerance classes: binary32 products of the exact-rounded weights with binary32 activations, and the
# tensor-core path where activations and weights are rounded to bfloat16.
TOL_FP32 = 1e-5
TOL_BF16 = 4e-3


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def dev(a):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def x_dev(x_np):
    """Activations to the device: float32 as is; uint16 bfloat16 patterns as a bfloat16 tensor."""
    torch = torch_cuda()
    if x_np.dtype == np.uint16:
        return torch.from_numpy(x_np.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x_np)).cuda()


def check_tol(y_gpu, y_ref, bound, tol, what=""):
    y = np.asarray(y_gpu, dtype=np.float64)
    nan_ref = np.isnan(y_ref)
    assert np.array_equal(np.isnan(y), nan_ref), what + ": NaN pattern differs"
    ok = ~nan_ref
    err = np.abs(y[ok] - y_ref[ok])
    lim = tol * bound[ok]
    bad = err > lim
    if bad.any():
        i = np.argmax(err - lim)
        raise AssertionError("%s: %d of %d outside tolerance; worst err %.3g vs bound %.3g (ratio %.3g)" % (
            what, int(bad.sum()), int(ok.sum()), err[i], bound[ok][i], err[i] / max(bound[ok][i], 1e-300)))
    return float(np.max(err / np.maximum(bound[ok], 1e-300))) if err.size else 0.0


def bit_differences(a, b) -> int:
    """Number of binary32 outputs whose bit patterns differ (the tile-invariance criterion)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    assert a.shape == b.shape
    return int(np.sum(a.view(np.uint32) != b.view(np.uint32)))
