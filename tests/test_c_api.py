"""The C ABI from C: tests/c_api_example.c compiles and links against include/libstencil.h and
libstencil.so with a plain C compiler (CPU), and on a GPU its two sweeps (device buffers and
host buffers) match the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from seismic_wave_propagation_gb300 import build as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def cuda_root() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def compile_example(out_dir) -> str:
    lib = b.build()
    libdir = os.path.dirname(lib)
    cuda = cuda_root()
    exe = os.path.join(str(out_dir), "c_api_example")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_api_example.c"), "-o", exe,
           "-L", libdir, "-l:libstencil.so", f"-Wl,-rpath,{libdir}",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_example_compiles_and_links(tmp_path):
    exe = compile_example(tmp_path)
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_c_example_matches_oracle(tmp_path):
    import oracle
    from seismic_wave_propagation_gb300 import synth
    from gpu_util import interior_mask, sweep_tol
    exe = compile_example(tmp_path)
    nx, ny, nz = 136, 75, 41
    u = synth.uniform_field(nx, ny, nz, seed=77)
    paths = [str(tmp_path / f) for f in ("in.bin", "out_dev.bin", "out_host.bin")]
    u.tofile(paths[0])
    r = subprocess.run([exe, str(nx), str(ny), str(nz)] + paths, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok libstencil")
    c = synth.laplacian8_coeffs().astype(np.float32)
    want = oracle.apply(u, c, 4, out=np.zeros_like(u))
    m = interior_mask(u.shape, 4)
    tol = sweep_tol(c, u)
    for p in paths[1:]:
        got = np.fromfile(p, dtype=np.float32).reshape(u.shape)
        assert np.max(np.abs(got[m].astype(np.float64) - want[m])) <= tol
        np.testing.assert_array_equal(got[~m], u[~m])  # shell: the input's values
