"""CPU oracle for the star-stencil sweep and the acoustic wave step (ctypes binding).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The CUDA library never imports or
links it, and it shares no code with the CUDA path. The arithmetic lives in
``stencil_oracle.c`` (plain C, double accumulation, one rounding to fp32); this module
only builds it with gcc and marshals numpy arrays.

Every function follows the definitions written at the top of ``stencil_oracle.c``:
the star stencil of "Accelerating High-Order Stencils on GPUs" (3D blocking with
global memory) and "Thread Coarsening 與 Register Tiling" (Fig 8.10), and the
second-order acoustic update with a pointwise sponge.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "stencil_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_F32P = ctypes.POINTER(ctypes.c_float)
_F64P = ctypes.POINTER(ctypes.c_double)
_I64P = ctypes.POINTER(ctypes.c_int64)
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (OpenMP when available). Returns the path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name, ptr in (("oracle_apply_f64", _F64P), ("oracle_apply_f32", _F32P)):
                fn = getattr(lib, name)
                fn.argtypes = [_I64, _I64, _I64, ctypes.c_int, ptr, ptr, ptr]
                fn.restype = None
            lib.oracle_apply_points_f32.argtypes = [_I64, _I64, _I64, ctypes.c_int, _F32P, _F32P,
                                                    _I64, _I64P, _F32P]
            lib.oracle_wave_step_f64.argtypes = [_I64, _I64, _I64, ctypes.c_int] + [_F64P] * 6
            lib.oracle_wave_step_f32.argtypes = [_I64, _I64, _I64, ctypes.c_int] + [_F32P] * 6
            lib.oracle_wave_points_f32.argtypes = [_I64, _I64, _I64, ctypes.c_int] + [_F32P] * 5 + \
                                                  [_I64, _I64P, _F32P]
            lib.oracle_wave_step_eta7_f64.argtypes = [_I64, _I64, _I64, ctypes.c_int, _F64P, ctypes.c_double,
                                                      ctypes.c_double] + [_F64P] * 5
            lib.oracle_wave_step_eta7_f32.argtypes = [_I64, _I64, _I64, ctypes.c_int, _F32P, ctypes.c_float,
                                                      ctypes.c_float] + [_F32P] * 5
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().oracle_num_threads())


def _grid(a: np.ndarray):
    if a.ndim != 3:
        raise ValueError("fields are (nz, ny, nx) arrays")
    nz, ny, nx = a.shape
    return nx, ny, nz


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _coeffs(coeffs, radius: int, dtype):
    c = np.ascontiguousarray(np.asarray(coeffs, dtype=dtype))
    if not 1 <= radius <= 7 or c.shape != (radius + 1,):
        raise ValueError("need radius in [1, 7] and radius+1 coefficients")
    return c


def _check(a: np.ndarray, dtype, shape=None):
    if a.dtype != dtype or not a.flags.c_contiguous:
        raise ValueError(f"expected a C-contiguous {dtype} array")
    if shape is not None and a.shape != shape:
        raise ValueError("field shapes differ")
    return a


def apply(u: np.ndarray, coeffs, radius: int, out: np.ndarray | None = None) -> np.ndarray:
    """Star stencil on the interior; the shell of ``out`` is left as it was.

    fp32 arrays: double accumulation, one rounding. fp64 arrays: all double.
    If ``out`` is None it starts as a copy of ``u`` (shell copied from the input).
    """
    dt = u.dtype
    if dt not in (np.float32, np.float64):
        raise ValueError("float32 or float64 fields")
    _check(u, dt)
    if out is None:
        out = u.copy()
    _check(out, dt, u.shape)
    nx, ny, nz = _grid(u)
    lib = _load()
    if dt == np.float64:
        c = _coeffs(coeffs, radius, np.float64)
        lib.oracle_apply_f64(nx, ny, nz, radius, _ptr(c, ctypes.c_double), _ptr(u, ctypes.c_double),
                             _ptr(out, ctypes.c_double))
    else:
        c = _coeffs(coeffs, radius, np.float32)
        lib.oracle_apply_f32(nx, ny, nz, radius, _ptr(c, ctypes.c_float), _ptr(u, ctypes.c_float),
                             _ptr(out, ctypes.c_float))
    return out


def apply_points(u: np.ndarray, coeffs, radius: int, idx: np.ndarray) -> np.ndarray:
    """Stencil outputs at the given flat indices (fp32 in, fp32 out; NaN off-interior)."""
    _check(u, np.float32)
    nx, ny, nz = _grid(u)
    c = _coeffs(coeffs, radius, np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    vals = np.empty(idx.shape, dtype=np.float32)
    _load().oracle_apply_points_f32(nx, ny, nz, radius, _ptr(c, ctypes.c_float), _ptr(u, ctypes.c_float),
                                    idx.size, _ptr(idx, ctypes.c_int64), _ptr(vals, ctypes.c_float))
    return vals


def wave_step(u_prev, u, v2dt2, eta, coeffs, radius: int, u_next=None) -> np.ndarray:
    """One acoustic step; returns u_next (shell of u_next left as it was).

    If ``u_next`` is None it starts as a copy of ``u_prev`` (so the shell keeps the
    values of the step before). ``u_next`` may be ``u_prev`` itself.
    """
    dt = u.dtype
    for a in (u_prev, u, v2dt2, eta):
        _check(a, dt, u.shape)
    if u_next is None:
        u_next = u_prev.copy()
    _check(u_next, dt, u.shape)
    if u_next is u:
        raise ValueError("u_next must not be u")
    nx, ny, nz = _grid(u)
    lib = _load()
    if dt == np.float64:
        c = _coeffs(coeffs, radius, np.float64)
        p = lambda a: _ptr(a, ctypes.c_double)  # noqa: E731
        lib.oracle_wave_step_f64(nx, ny, nz, radius, p(c), p(u_prev), p(u), p(u_next), p(v2dt2), p(eta))
    elif dt == np.float32:
        c = _coeffs(coeffs, radius, np.float32)
        p = lambda a: _ptr(a, ctypes.c_float)  # noqa: E731
        lib.oracle_wave_step_f32(nx, ny, nz, radius, p(c), p(u_prev), p(u), p(u_next), p(v2dt2), p(eta))
    else:
        raise ValueError("float32 or float64 fields")
    return u_next


def wave_step_eta7(u_prev, u, v2dt2, eta, coeffs, radius: int, e0: float, e1: float, u_next=None):
    """One acoustic step whose damping at a point is the radius-1 star stencil of eta,
    e0*eta + e1*(its six face neighbours), in place of eta itself (see stencil_oracle.c).
    Same conventions as wave_step."""
    dt = u.dtype
    for a in (u_prev, u, v2dt2, eta):
        _check(a, dt, u.shape)
    if u_next is None:
        u_next = u_prev.copy()
    _check(u_next, dt, u.shape)
    if u_next is u:
        raise ValueError("u_next must not be u")
    nx, ny, nz = _grid(u)
    lib = _load()
    if dt == np.float64:
        c = _coeffs(coeffs, radius, np.float64)
        p = lambda a: _ptr(a, ctypes.c_double)  # noqa: E731
        lib.oracle_wave_step_eta7_f64(nx, ny, nz, radius, p(c), float(e0), float(e1), p(u_prev), p(u),
                                      p(u_next), p(v2dt2), p(eta))
    elif dt == np.float32:
        c = _coeffs(coeffs, radius, np.float32)
        p = lambda a: _ptr(a, ctypes.c_float)  # noqa: E731
        lib.oracle_wave_step_eta7_f32(nx, ny, nz, radius, p(c), float(e0), float(e1), p(u_prev), p(u),
                                      p(u_next), p(v2dt2), p(eta))
    else:
        raise ValueError("float32 or float64 fields")
    return u_next


def wave_points(u_prev, u, v2dt2, eta, coeffs, radius: int, idx: np.ndarray) -> np.ndarray:
    """One wave step evaluated only at the given flat indices (fp32)."""
    for a in (u_prev, u, v2dt2, eta):
        _check(a, np.float32, u.shape)
    nx, ny, nz = _grid(u)
    c = _coeffs(coeffs, radius, np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    vals = np.empty(idx.shape, dtype=np.float32)
    p = lambda a: _ptr(a, ctypes.c_float)  # noqa: E731
    _load().oracle_wave_points_f32(nx, ny, nz, radius, p(c), p(u_prev), p(u), p(v2dt2), p(eta),
                                   idx.size, _ptr(idx, ctypes.c_int64), p(vals))
    return vals


def run_sweeps(u0: np.ndarray, coeffs, radius: int, nsweeps: int) -> np.ndarray:
    """Ping-pong sweeps with a fixed shell: both buffers start as u0."""
    a = u0.copy()
    b = u0.copy()
    for _ in range(nsweeps):
        apply(a, coeffs, radius, out=b)
        a, b = b, a
    return a


def run_wave(u_prev, u, v2dt2, eta, coeffs, radius: int, nsteps: int):
    """nsteps leapfrog steps with three-buffer rotation; returns (u_prev, u)."""
    a, b = u_prev.copy(), u.copy()
    c = u_prev.copy()
    for _ in range(nsteps):
        wave_step(a, b, v2dt2, eta, coeffs, radius, u_next=c)
        a, b, c = b, c, a
    return a, b
