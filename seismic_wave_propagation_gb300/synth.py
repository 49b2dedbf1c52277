"""Seeded synthetic inputs for the star-stencil sweep and the acoustic wave step.

This module only *generates data*; it contains none of the stencil or wave-update
arithmetic. Both the CUDA library's tests/benchmark and the CPU oracle draw their
inputs from here, so the two sides always see bit-identical fields.

Layout: every field is a C-ordered ``float32`` array of shape ``(nz, ny, nx)``, i.e. a
flat 1D array with x innermost and linear index ``i = x + nx*(y + ny*z)``, the layout
the stencil pages describe ("Accelerating High-Order Stencils on GPUs", 3D blocking
with global memory: the grid is stored as a flat 1D array, coalescing along X).

Random numbers come from SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants are the
published ones), evaluated counter-style: value ``i`` of a stream with seed ``s`` is
``mix64(s XOR i)``, so any sub-block of a field can be generated independently and in
parallel. The top 24 bits give a uniform on [-1, 1) that is exact in fp32.

Workload recipes (the grid sizes and values of the five benchmark workloads):

* ``uniform``: u ~ Uniform[-1, 1) from the seed.
* ``wave``: u = u_prev = Gaussian bump (sigma = 3 points) centred on the grid point
  (nx//2, ny//2, nz//2); velocity in 8 piecewise-constant z-layers spaced linearly from
  1500 to 4500 m/s (layer k = floor(8 z / nz)), v2dt2 = (v * dt/h)^2 with
  dt/h = 1e-4 s/m; sponge damping eta = 0.1 * ((16 - d) / 16)^2 where d is the
  distance to the nearest face (d < 16), and 0 elsewhere.
* ``sinusoids``: sum of 4 plane sinusoids with integer wave numbers in [1, 8] per axis
  and random phases, plus Uniform[-0.01, 0.01) noise.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

DEFAULT_SEED = 0x5EED

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_PARAM_SALT = 1 << 63  # keeps parameter draws disjoint from per-point draws


def mix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output function applied to ``x + gamma`` (uint64, wrapping)."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform_from_index(seed: int, idx: np.ndarray) -> np.ndarray:
    """Uniform[-1, 1) values for the given linear indices (float64, exact in fp32)."""
    bits = mix64(np.uint64(seed) ^ np.asarray(idx, dtype=np.uint64)) >> np.uint64(40)
    return bits.astype(np.float64) * (2.0 ** -23) - 1.0


def _param_u64(seed: int, m: int) -> int:
    return int(mix64(np.uint64(seed) ^ np.uint64(_PARAM_SALT | m)))


def _workers() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _fill_by_planes(shape, plane_fn) -> np.ndarray:
    """Allocate a (nz, ny, nx) float32 array and fill it slab by slab in threads."""
    nz, ny, nx = shape
    out = np.empty(shape, dtype=np.float32)
    if nz == 0 or ny == 0 or nx == 0:
        return out
    planes_per_chunk = max(1, (1 << 22) // max(1, nx * ny))
    chunks = [(z0, min(nz, z0 + planes_per_chunk)) for z0 in range(0, nz, planes_per_chunk)]

    def work(c):
        z0, z1 = c
        out[z0:z1] = plane_fn(z0, z1)

    if len(chunks) == 1:
        work(chunks[0])
    else:
        with ThreadPoolExecutor(_workers()) as ex:
            list(ex.map(work, chunks))
    return out


def uniform_field(nx: int, ny: int, nz: int, seed: int = DEFAULT_SEED,
                  scale: float = 1.0) -> np.ndarray:
    """``scale`` * Uniform[-1, 1) on every grid point, value i = f(seed, i)."""
    plane = nx * ny

    def fn(z0, z1):
        idx = np.arange(z0 * plane, z1 * plane, dtype=np.uint64)
        v = uniform_from_index(seed, idx)
        if scale != 1.0:
            v = v * scale
        return v.reshape(z1 - z0, ny, nx)

    return _fill_by_planes((nz, ny, nx), fn)


def gaussian_bump(nx: int, ny: int, nz: int, sigma: float = 3.0,
                  center=None, amplitude: float = 1.0) -> np.ndarray:
    """amplitude * exp(-|p - c|^2 / (2 sigma^2)), c a grid point (default: centre)."""
    cx, cy, cz = center if center is not None else (nx // 2, ny // 2, nz // 2)
    dx2 = (np.arange(nx, dtype=np.float64) - cx) ** 2
    dy2 = (np.arange(ny, dtype=np.float64) - cy) ** 2
    inv = 1.0 / (2.0 * sigma * sigma)

    def fn(z0, z1):
        dz2 = (np.arange(z0, z1, dtype=np.float64) - cz) ** 2
        r2 = dz2[:, None, None] + dy2[None, :, None] + dx2[None, None, :]
        return amplitude * np.exp(-r2 * inv)

    return _fill_by_planes((nz, ny, nx), fn)


def sponge_eta(nx: int, ny: int, nz: int, width: int = 16, eta_max: float = 0.1) -> np.ndarray:
    """Quadratic sponge: eta_max * ((width - d)/width)^2 for d < width, else 0.

    d is the distance (in points) to the nearest of the six faces, so eta = eta_max on
    the faces and 0 from ``width`` points inwards.
    """
    dx = np.minimum(np.arange(nx), nx - 1 - np.arange(nx))
    dy = np.minimum(np.arange(ny), ny - 1 - np.arange(ny))

    def fn(z0, z1):
        zz = np.arange(z0, z1)
        dz = np.minimum(zz, nz - 1 - zz)
        d = np.minimum(np.minimum(dz[:, None, None], dy[None, :, None]), dx[None, None, :])
        t = (width - d.astype(np.float64)) / width
        return np.where(d < width, eta_max * t * t, 0.0)

    return _fill_by_planes((nz, ny, nx), fn)


def layer_velocity(nz: int, nlayers: int = 8, vmin: float = 1500.0, vmax: float = 4500.0) -> np.ndarray:
    """Velocity of each z plane: layer k = floor(nlayers z / nz), v_k linear in k."""
    z = np.arange(nz)
    k = (nlayers * z) // max(1, nz)
    return vmin + (vmax - vmin) * k / (nlayers - 1)


def layered_v2dt2(nx: int, ny: int, nz: int, dt_over_h: float = 1e-4, nlayers: int = 8,
                  vmin: float = 1500.0, vmax: float = 4500.0) -> np.ndarray:
    """(v * dt/h)^2 with v constant in each of ``nlayers`` z-layers."""
    v = layer_velocity(nz, nlayers, vmin, vmax)
    s = (v * dt_over_h) ** 2

    def fn(z0, z1):
        return np.broadcast_to(s[z0:z1, None, None], (z1 - z0, ny, nx))

    return _fill_by_planes((nz, ny, nx), fn)


def sinusoid_params(seed: int = DEFAULT_SEED, nwaves: int = 4):
    """Integer wave numbers (a, b, c) in [1, 8] and phases in [0, 2 pi) per sinusoid."""
    params = []
    for j in range(nwaves):
        q = _param_u64(seed, 2 * j)
        a = 1 + ((q >> 61) & 7)
        b = 1 + ((q >> 58) & 7)
        c = 1 + ((q >> 55) & 7)
        q2 = _param_u64(seed, 2 * j + 1)
        phi = (q2 >> 11) * (2.0 ** -53) * 2.0 * math.pi
        params.append((int(a), int(b), int(c), float(phi)))
    return params


def sinusoid_field(nx: int, ny: int, nz: int, seed: int = DEFAULT_SEED, nwaves: int = 4,
                   noise: float = 0.01) -> np.ndarray:
    """sum_j sin(2 pi (a_j x/nx + b_j y/ny + c_j z/nz) + phi_j) + noise * U[-1, 1)."""
    params = sinusoid_params(seed, nwaves)
    xs = np.arange(nx, dtype=np.float64) / nx
    ys = np.arange(ny, dtype=np.float64) / ny
    plane = nx * ny

    def fn(z0, z1):
        zs = np.arange(z0, z1, dtype=np.float64) / nz
        acc = np.zeros((z1 - z0, ny, nx), dtype=np.float64)
        for a, b, c, phi in params:
            ph = (2.0 * math.pi) * (c * zs[:, None, None] + b * ys[None, :, None] + a * xs[None, None, :]) + phi
            acc += np.sin(ph)
        idx = np.arange(z0 * plane, z1 * plane, dtype=np.uint64)
        acc += noise * uniform_from_index(seed, idx).reshape(z1 - z0, ny, nx)
        return acc

    return _fill_by_planes((nz, ny, nx), fn)


# Coefficient sets. coeffs[0] is the *total* centre weight (summed over the three
# axes); coeffs[r] is the weight of each of the six neighbours at distance r.
LAPLACIAN_8TH_AXIS = (-205.0 / 72.0, 8.0 / 5.0, -1.0 / 5.0, 8.0 / 315.0, -1.0 / 560.0)


def laplacian8_coeffs():
    """25-point 8th-order Laplacian (h = 1): centre 3 * (-205/72), then 8/5, -1/5, 8/315, -1/560."""
    c = list(LAPLACIAN_8TH_AXIS)
    c[0] = 3.0 * c[0]
    return np.asarray(c, dtype=np.float64)


def laplacian2_coeffs():
    """7-point unit-spacing Laplacian: centre -6, neighbours 1."""
    return np.asarray([-6.0, 1.0], dtype=np.float64)


def average7_coeffs():
    """7-point smoothing update: 0.5 * u + (1/12) * (sum of the 6 face neighbours)."""
    return np.asarray([0.5, 1.0 / 12.0], dtype=np.float64)


# The five benchmark workloads. "sweeps" are ping-pong applications of the stencil;
# "steps" are wave time steps with three-buffer rotation.
WORKLOADS = {
    "star7_avg_64": dict(nx=64, ny=64, nz=64, radius=1, coeffs="average7", sweeps=1,
                         init="uniform", shell="copied from input"),
    "star7_lap_512": dict(nx=512, ny=512, nz=512, radius=1, coeffs="laplacian2", sweeps=10,
                          init="uniform", shell="fixed"),
    "star25_lap8_512": dict(nx=512, ny=512, nz=512, radius=4, coeffs="laplacian8", sweeps=1,
                            init="uniform", shell="untouched"),
    "wave25_640": dict(nx=640, ny=640, nz=640, radius=4, coeffs="laplacian8", steps=100,
                       init="wave"),
    "star25_lap8_1536x1536x256": dict(nx=1536, ny=1536, nz=256, radius=4, coeffs="laplacian8",
                                      sweeps=50, init="sinusoids", shell="fixed"),
}


def coeffs_for(name: str) -> np.ndarray:
    return {"average7": average7_coeffs, "laplacian2": laplacian2_coeffs,
            "laplacian8": laplacian8_coeffs}[name]()


def wave_fields(nx: int, ny: int, nz: int, sigma: float = 3.0):
    """(u_prev, u, v2dt2, eta) for the acoustic wave workload."""
    u = gaussian_bump(nx, ny, nz, sigma=sigma)
    return u.copy(), u, layered_v2dt2(nx, ny, nz), sponge_eta(nx, ny, nz)
