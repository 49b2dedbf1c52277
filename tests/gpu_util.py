"""Helpers shared by the GPU tests (device buffers with guard bands, tolerances)."""
import numpy as np
import pytest

GUARD = 1024  # floats of sentinel on each side of every device field (4 KB)
SENTINEL_BITS = 0x7FC0DEAD  # a NaN payload no computation produces


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def sentinel():
    return np.array([SENTINEL_BITS], dtype=np.uint32).view(np.float32)[0]


class Guarded:
    """A device field embedded in a larger buffer whose margins hold sentinels."""

    def __init__(self, torch, host: np.ndarray, fill_sentinel: bool = False):
        n = host.size
        self.shape = host.shape
        self.buf = torch.full((n + 2 * GUARD,), float(sentinel()), dtype=torch.float32, device="cuda")
        self.field = self.buf[GUARD:GUARD + n]
        if not fill_sentinel:
            self.field.copy_(torch.from_numpy(np.ascontiguousarray(host).ravel()))

    @property
    def ptr(self):
        return self.field.data_ptr()

    def numpy(self):
        return self.field.cpu().numpy().reshape(self.shape)

    def guards_intact(self):
        b = self.buf.cpu().numpy().view(np.uint32)
        return bool(np.all(b[:GUARD] == SENTINEL_BITS) and np.all(b[-GUARD:] == SENTINEL_BITS))


def interior_mask(shape, R):
    nz, ny, nx = shape
    m = np.zeros(shape, dtype=bool)
    m[R:nz - R, R:ny - R, R:nx - R] = True
    return m


def sweep_tol(coeffs, u_in) -> float:
    """Per-sweep gate: 1e-5 * sum|c| * max|u_in|."""
    return 1e-5 * float(np.sum(np.abs(np.asarray(coeffs, np.float64)))) * float(np.max(np.abs(u_in)))


def sample_interior(shape, R, n, seed=0, planes=()):
    """Random interior flat indices plus every interior point of the given z planes."""
    nz, ny, nx = shape
    rng = np.random.default_rng(seed)
    x = rng.integers(R, nx - R, n)
    y = rng.integers(R, ny - R, n)
    z = rng.integers(R, nz - R, n)
    idx = [x + nx * (y + ny * z)]
    for zp in planes:
        yy, xx = np.meshgrid(np.arange(R, ny - R), np.arange(R, nx - R), indexing="ij")
        idx.append((xx + nx * (yy + ny * zp)).ravel())
    return np.unique(np.concatenate(idx).astype(np.int64))
