"""Helpers shared by the GPU parity tests."""
import numpy as np
import pytest
import torch

TOL = {"f32": 1e-4, "bf16": 4e-3}   # max |y_gpu - y_ref| / sum_k |w x|


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def x_dev(x: np.ndarray) -> torch.Tensor:
    """float32 array -> fp32 tensor; uint16 (bf16 bits) -> bfloat16 tensor."""
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    return dev(x)


def rel_err(y_gpu: np.ndarray, y_ref: np.ndarray, s_ref: np.ndarray) -> float:
    """max over outputs of |y_gpu - y_ref| / sum|w x|; outputs with a zero sum must be exactly 0."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    zero = s_ref == 0
    assert np.all(y_gpu[zero] == 0), "output with no nonzero term is not exactly 0"
    if np.all(zero):
        return 0.0
    return float(np.max(np.abs(y_gpu[~zero] - y_ref[~zero]) / s_ref[~zero]))
