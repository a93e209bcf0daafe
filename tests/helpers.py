"""Shared helpers for the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

RTOL = 1e-5   # per element: |y - y_ref| <= RTOL * sum_g |dw dx S_g|


def dev():
    return torch.device("cuda", 0)


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        a = a.view(np.float16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.float16:
        return t.numpy().view(np.uint16)
    return t.numpy()


def assert_close(y: np.ndarray, y_ref: np.ndarray, mag: np.ndarray, rtol: float = RTOL):
    """Element-wise condition-aware check; also reports the normwise error."""
    y = y.astype(np.float64)
    ref = y_ref.astype(np.float64)
    err = np.abs(y - ref)
    lim = rtol * mag + 1e-30
    bad = err > lim
    if bad.any():
        i = np.unravel_index(np.argmax(err / lim), err.shape)
        raise AssertionError(
            f"{int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
            f"y={y[i]!r} ref={ref[i]!r} err={err[i]:.3e} limit={lim[i]:.3e}")
    nrm = np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300)
    return float(nrm), float((err / np.maximum(mag, 1e-300)).max())
