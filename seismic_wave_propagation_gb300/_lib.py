"""ctypes binding of libstencil.so: the same entry points, argument marshalling only.

Every computation runs in the CUDA library.  Fields may be passed as CUDA tensors
(float32, contiguous) or as raw device addresses (int); host-buffer calls take numpy
float32 arrays.  If the library is missing this module raises at the first call: there
is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libstencil.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "libstencil.h")

STENCIL_OK = 0
ERRORS = {-1: "STENCIL_ERR_ARG", -2: "STENCIL_ERR_ALIGNMENT", -3: "STENCIL_ERR_ALIAS",
          -4: "STENCIL_ERR_CUDA", -5: "STENCIL_ERR_TIMEOUT"}
KIND_APPLY, KIND_WAVE, KIND_WAVE_PML, KIND_SEMI, KIND_APPLY2 = 0, 1, 2, 3, 4
LAUNCH_INFO_KEYS = ("grid", "threads", "smem", "ctas_per_sm", "tiles", "zchunks", "tile_x",
                    "tile_y", "stages", "sms", "path")
SWEEP_PATHS = {"auto": 0, "staged": 1, "direct": 2}

_lock = threading.Lock()
_lib = None


class StencilError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{ERRORS.get(code, code)}: {message}")
        self.code = code


def header_functions() -> list[str]:
    """Names of the functions include/libstencil.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text.split('extern "C" {', 1)[1])


def load():
    """Load libstencil.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libstencil.so not built ({LIB_PATH}); run "
                               "python -m seismic_wave_propagation_gb300.build")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, fp = ctypes.c_void_p, ctypes.c_int64, ctypes.POINTER(ctypes.c_float)
        lib.stencil_plan_create.argtypes = [i64, i64, i64, ctypes.c_int, fp]
        lib.stencil_plan_create.restype = vp
        lib.stencil_plan_destroy.argtypes = [vp]
        lib.stencil_plan_destroy.restype = None
        lib.stencil_apply.argtypes = [vp, vp, vp, vp]
        lib.stencil_apply_semi.argtypes = [vp, vp, vp, vp]
        lib.stencil_apply2.argtypes = [vp, vp, vp, vp]
        lib.wave_step.argtypes = [vp] * 7
        lib.wave_step_pml.argtypes = [vp] * 6 + [i64, vp]
        lib.stencil_plan_status.argtypes = [vp, vp]
        lib.stencil_sweeps.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, vp]
        lib.wave_steps.argtypes = [vp] * 6 + [ctypes.c_int, i64, ctypes.c_int, vp]
        lib.stencil_last_error.restype = ctypes.c_char_p
        lib.stencil_apply_host.argtypes = [vp, vp, vp, ctypes.c_int, vp]
        lib.wave_run_host.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, vp]
        lib.stencil_plan_launch_info.argtypes = [vp, ctypes.c_int, ctypes.POINTER(i64), ctypes.c_int]
        lib.stencil_debug_inject.argtypes = [vp, ctypes.c_int]
        lib.stencil_plan_set_sweep_path.argtypes = [vp, ctypes.c_int]
        lib.wave_eta_stencil.argtypes = [vp, vp, vp, ctypes.c_float, ctypes.c_float, vp]
        lib.stencil_plan_host_phases.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.c_int]
        lib.stencil_schedule_query.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.POINTER(i64), ctypes.c_int]
        lib.stencil_version.restype = ctypes.c_char_p
        lib.stencil_slabs_create.argtypes = [i64, i64, i64, ctypes.c_int, fp, ctypes.c_int]
        lib.stencil_slabs_create.restype = vp
        lib.stencil_slabs_destroy.argtypes = [vp]
        lib.stencil_slabs_destroy.restype = None
        lib.stencil_slabs_extent.argtypes = [vp, ctypes.c_int, ctypes.POINTER(i64), ctypes.c_int]
        lib.stencil_slabs_exchange.argtypes = [vp, vp, vp]
        lib.stencil_slabs_apply.argtypes = [vp, vp, vp, vp]
        lib.stencil_slabs_wave_step.argtypes = [vp] * 7
        lib.stencil_slabs_status.argtypes = [vp, vp]
        for fn in ("stencil_apply", "stencil_apply_semi", "stencil_apply2", "wave_step", "wave_step_pml", "stencil_sweeps", "wave_steps",
                   "stencil_plan_status", "stencil_apply_host", "stencil_plan_set_sweep_path",
                   "wave_run_host", "stencil_plan_launch_info", "stencil_debug_inject",
                   "stencil_schedule_query", "stencil_plan_host_phases", "wave_eta_stencil", "stencil_slabs_extent",
                   "stencil_slabs_exchange", "stencil_slabs_apply", "stencil_slabs_wave_step",
                   "stencil_slabs_status"):
            getattr(lib, fn).restype = ctypes.c_int
        _lib = lib
        return lib


def last_error() -> str:
    return load().stencil_last_error().decode()


def _check(rc: int) -> int:
    if rc < 0:
        raise StencilError(rc, last_error())
    return rc


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if x.dtype.__repr__() != "torch.float32" or not x.is_contiguous() or not x.is_cuda:
            raise ValueError("fields must be contiguous float32 CUDA tensors")
        return x.data_ptr()
    raise TypeError(f"cannot take a device address of {type(x)}")


def _stream(stream, *fields) -> int | None:
    if stream is None:
        for f in fields:
            if hasattr(f, "is_cuda") and f.is_cuda:
                import torch
                return torch.cuda.current_stream(f.device).cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host(a: np.ndarray, n: int) -> int:
    if a.dtype != np.float32 or not a.flags.c_contiguous or a.size != n:
        raise ValueError("host fields must be C-contiguous float32 arrays of nx*ny*nz values")
    return a.ctypes.data


class StencilPlan:
    """A star stencil of ``radius`` on an nx x ny x nz grid (see include/libstencil.h)."""

    def __init__(self, nx: int, ny: int, nz: int, radius: int, coeffs):
        lib = load()
        c = np.ascontiguousarray(np.asarray(coeffs, dtype=np.float32))
        if c.ndim != 1:
            raise ValueError("coeffs must be 1D")
        self.nx, self.ny, self.nz, self.radius = int(nx), int(ny), int(nz), int(radius)
        self.coeffs = c.copy()
        self._p = lib.stencil_plan_create(self.nx, self.ny, self.nz, self.radius,
                                          c.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
        if not self._p:
            raise StencilError(-1, last_error())
        self._lib = lib

    @property
    def npoints(self) -> int:
        return self.nx * self.ny * self.nz

    def close(self):
        if getattr(self, "_p", None):
            self._lib.stencil_plan_destroy(self._p)
            self._p = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def apply(self, inp, out, stream=None) -> None:
        _check(self._lib.stencil_apply(self._p, _addr(inp), _addr(out), _stream(stream, inp, out)))

    def apply2(self, inp, out, stream=None) -> None:
        """stencil_apply2: two sweeps in one pass (radius 1): out = S(S(inp))."""
        _check(self._lib.stencil_apply2(self._p, _addr(inp), _addr(out), _stream(stream, inp, out)))

    def apply_semi(self, inp, out, stream=None) -> None:
        """The same sweep in semi-stencil form (an alternative kernel; see the header)."""
        _check(self._lib.stencil_apply_semi(self._p, _addr(inp), _addr(out), _stream(stream, inp, out)))

    def wave_step(self, u_prev, u, u_next, v2dt2, eta, stream=None) -> None:
        fields = (u_prev, u, u_next, v2dt2, eta)
        _check(self._lib.wave_step(self._p, *[_addr(f) for f in fields], _stream(stream, *fields)))

    def wave_step_pml(self, u_prev, u, u_next, v2dt2, eta, pml_width: int, stream=None) -> None:
        fields = (u_prev, u, u_next, v2dt2, eta)
        _check(self._lib.wave_step_pml(self._p, *[_addr(f) for f in fields], int(pml_width),
                                       _stream(stream, *fields)))

    def eta_stencil(self, eta, eta_eff, e0: float, e1: float, stream=None) -> None:
        """wave_eta_stencil: eta_eff = e0*eta + e1*(six face neighbours), once per model."""
        _check(self._lib.wave_eta_stencil(self._p, _addr(eta), _addr(eta_eff), float(e0), float(e1),
                                          _stream(stream, eta, eta_eff)))

    def sweeps(self, a, b, nsweeps: int, use_graph: bool = False, stream=None) -> None:
        """stencil_sweeps: ping-pong sweeps a -> b -> a ...; odd counts end in b."""
        _check(self._lib.stencil_sweeps(self._p, _addr(a), _addr(b), int(nsweeps), int(use_graph),
                                        _stream(stream, a, b)))

    def wave_steps(self, u_prev, u, u_tmp, v2dt2, eta, nsteps: int, pml_width: int = -1,
                   use_graph: bool = False, stream=None) -> None:
        """wave_steps: three-buffer rotation; the newest level ends in [(n+1) % 3]."""
        fields = (u_prev, u, u_tmp, v2dt2, eta)
        _check(self._lib.wave_steps(self._p, *[_addr(f) for f in fields], int(nsteps), int(pml_width),
                                    int(use_graph), _stream(stream, *fields)))

    def status(self, stream=None, *fields) -> None:
        _check(self._lib.stencil_plan_status(self._p, _stream(stream, *fields)))

    def apply_host(self, inp: np.ndarray, out: np.ndarray, nsweeps: int = 1, stream=None) -> None:
        n = self.npoints
        _check(self._lib.stencil_apply_host(self._p, _host(inp, n), _host(out, n), int(nsweeps),
                                            _stream(stream)))

    def wave_run_host(self, u_prev: np.ndarray, u: np.ndarray, v2dt2: np.ndarray, eta: np.ndarray,
                      nsteps: int, stream=None) -> None:
        n = self.npoints
        _check(self._lib.wave_run_host(self._p, _host(u_prev, n), _host(u, n), _host(v2dt2, n),
                                       _host(eta, n), int(nsteps), _stream(stream)))

    def set_sweep_path(self, path) -> None:
        """stencil_plan_set_sweep_path: "auto", "staged" or "direct" (or 0, 1, 2)."""
        if isinstance(path, str):
            if path not in SWEEP_PATHS:
                raise ValueError(f"sweep path must be one of {sorted(SWEEP_PATHS)}, not {path!r}")
            path = SWEEP_PATHS[path]
        _check(self._lib.stencil_plan_set_sweep_path(self._p, int(path)))

    @property
    def sweep_path(self) -> str:
        """The kernel the plan's sweeps run on: "staged" or "direct"."""
        return {1: "staged", 2: "direct"}[self.launch_info(KIND_APPLY)["path"]]

    def launch_info(self, kind: int = KIND_APPLY) -> dict:
        buf = (ctypes.c_int64 * len(LAUNCH_INFO_KEYS))()
        m = _check(self._lib.stencil_plan_launch_info(self._p, kind, buf, len(buf)))
        return {k: int(buf[i]) for i, k in enumerate(LAUNCH_INFO_KEYS[:m])}

    def host_phases(self) -> dict:
        """stencil_plan_host_phases: phase end times (ms) of the last pipelined host sweep."""
        buf = (ctypes.c_float * 5)()
        m = _check(self._lib.stencil_plan_host_phases(self._p, buf, 5))
        keys = ("total_ms", "first_slab_in_ms", "copies_in_done_ms", "sweeps_done_ms", "slabs")
        return {k: float(buf[i]) for i, k in enumerate(keys[:m])}

    def debug_inject(self, mode: int) -> None:
        _check(self._lib.stencil_debug_inject(self._p, int(mode)))


class StencilSlabs:
    """The grid cut along z into slabs, each its own device array with ghost planes
    (stencil_slabs_* in include/libstencil.h).  Fields are lists of per-slab arrays."""

    def __init__(self, nx: int, ny: int, nz: int, radius: int, coeffs, nslabs: int):
        lib = load()
        c = np.ascontiguousarray(np.asarray(coeffs, dtype=np.float32))
        self.nx, self.ny, self.nz, self.radius, self.nslabs = int(nx), int(ny), int(nz), int(radius), int(nslabs)
        self._p = lib.stencil_slabs_create(self.nx, self.ny, self.nz, self.radius,
                                           c.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), self.nslabs)
        if not self._p:
            raise StencilError(-1, last_error())
        self._lib = lib

    def extent(self, k: int) -> dict:
        """Global planes of slab k: stored [begin, end) (ghosts included), owned [own_begin, own_end)."""
        buf = (ctypes.c_int64 * 4)()
        _check(self._lib.stencil_slabs_extent(self._p, int(k), buf, 4))
        return {"begin": buf[0], "end": buf[1], "own_begin": buf[2], "own_end": buf[3]}

    def slab_shape(self, k: int) -> tuple:
        e = self.extent(k)
        return (e["end"] - e["begin"], self.ny, self.nx)

    def _ptrs(self, fields):
        if len(fields) != self.nslabs:
            raise ValueError(f"need {self.nslabs} slab arrays")
        arr = (ctypes.c_void_p * self.nslabs)(*[_addr(f) for f in fields])
        return arr

    def exchange(self, fields, stream=None) -> None:
        _check(self._lib.stencil_slabs_exchange(self._p, self._ptrs(fields), _stream(stream, *fields)))

    def apply(self, inp, out, stream=None) -> None:
        _check(self._lib.stencil_slabs_apply(self._p, self._ptrs(inp), self._ptrs(out),
                                             _stream(stream, *inp, *out)))

    def wave_step(self, u_prev, u, u_next, v2dt2, eta, stream=None) -> None:
        f = (u_prev, u, u_next, v2dt2, eta)
        _check(self._lib.stencil_slabs_wave_step(self._p, *[self._ptrs(x) for x in f],
                                                 _stream(stream, *u)))

    def status(self, stream=None, *fields) -> None:
        _check(self._lib.stencil_slabs_status(self._p, _stream(stream, *fields)))

    def close(self):
        if getattr(self, "_p", None):
            self._lib.stencil_slabs_destroy(self._p)
            self._p = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


SCHEDULE_KEYS = ("grid", "tiles", "zchunks", "items", "tile_x", "tile_y", "x_origin")


def schedule_query(nx: int, ny: int, nz: int, radius: int, kind: int, num_sms: int,
                   ctas_per_sm: int) -> dict:
    """stencil_schedule_query: the plan's z-chunk schedule for a given GPU, host-only."""
    buf = (ctypes.c_int64 * len(SCHEDULE_KEYS))()
    m = _check(load().stencil_schedule_query(int(nx), int(ny), int(nz), int(radius), int(kind),
                                             int(num_sms), int(ctas_per_sm), buf, len(buf)))
    return {k: int(buf[i]) for i, k in enumerate(SCHEDULE_KEYS[:m])}


def version() -> str:
    return load().stencil_version().decode()


def apply_noalloc(nx: int, ny: int, nz: int, radius: int, coeffs, inp, out, stream=None) -> None:
    """stencil_apply_noalloc: one sweep that allocates nothing on the device.

    For callers that cannot allocate device memory when they need the sweep; its scratch
    is a fixed 256-byte device array inside the library (see include/libstencil.h).
    """
    lib = load()
    fn = lib.stencil_apply_noalloc
    fn.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                   ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    c = np.ascontiguousarray(np.asarray(coeffs, dtype=np.float32))
    _check(fn(int(nx), int(ny), int(nz), int(radius), c.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
              _addr(inp), _addr(out), _stream(stream, inp, out)))
