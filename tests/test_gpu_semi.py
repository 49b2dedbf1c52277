"""Parity of the semi-stencil sweep (stencil_apply_semi) against the CPU oracle, through the
C ABI: the same cases and bar as stencil_apply, since both compute the same definition."""
import numpy as np
import pytest

import oracle
from seismic_wave_propagation_gb300 import KIND_SEMI, StencilError, StencilPlan, synth
from gpu_util import Guarded, interior_mask, sweep_tol, torch_cuda
from test_gpu_apply import CASES

pytestmark = pytest.mark.gpu


def run_semi(torch, u, coeffs, R):
    nz, ny, nx = u.shape
    plan = StencilPlan(nx, ny, nz, R, coeffs)
    gin = Guarded(torch, u)
    gout = Guarded(torch, u, fill_sentinel=True)
    plan.apply_semi(gin.ptr, gout.ptr)
    plan.status()
    out = gout.numpy()
    assert gin.guards_intact() and gout.guards_intact()
    np.testing.assert_array_equal(gin.numpy(), u)  # input untouched
    plan.close()
    return out


def check(u, out, coeffs, R):
    c32 = np.asarray(coeffs, np.float32)
    m = interior_mask(u.shape, R)
    want = oracle.apply(u, c32, R, out=np.zeros_like(u))
    err = np.abs(out[m].astype(np.float64) - want[m])
    tol = sweep_tol(c32, u)
    assert err.size == 0 or err.max() <= tol, f"max err {err.max()} > {tol}"
    assert np.all(out.view(np.uint32)[~m] == 0x7FC0DEAD), "shell written"
    return err.max() if err.size else 0.0


@pytest.mark.parametrize("nx,ny,nz,R", CASES)
def test_semi_matches_oracle(nx, ny, nz, R):
    torch = torch_cuda()
    u = synth.uniform_field(nx, ny, nz, seed=2000 + nx + R)
    c = np.random.default_rng(10 + R).uniform(-1, 1, R + 1)
    check(u, run_semi(torch, u, c, R), c, R)


def test_semi_star25_512_full_grid():
    """The 25-point 8th-order Laplacian at 512^3, every interior point against the oracle."""
    torch = torch_cuda()
    u = synth.uniform_field(512, 512, 512)
    c = synth.laplacian8_coeffs()
    err = check(u, run_semi(torch, u, c, 4), c, 4)
    print(f"semi star25 512^3: max |gpu - oracle| = {err:.3e}")


def test_semi_checkerboard_closed_form():
    """Checkerboard input: the 25-point Laplacian gives -sum|c| = -2048/105 times the input."""
    torch = torch_cuda()
    n = 40
    z, y, x = np.indices((n, n, n))
    cb = np.where((x + y + z) % 2 == 0, 1.0, -1.0).astype(np.float32)
    out = run_semi(torch, cb, synth.laplacian8_coeffs(), 4)
    m = interior_mask(cb.shape, 4)
    np.testing.assert_allclose(out[m], -2048.0 / 105.0 * cb[m], rtol=0, atol=1e-4)


def test_semi_launch_geometry_and_errors():
    torch = torch_cuda()
    n = 32
    plan = StencilPlan(n, n, n, 4, synth.laplacian8_coeffs())
    info = plan.launch_info(KIND_SEMI)
    assert info["stages"] >= 2 * 4 + 1  # the ring keeps R planes behind the lead
    assert 1 <= info["grid"] <= info["sms"] * info["ctas_per_sm"]
    a = torch.zeros(n ** 3 + 64, device="cuda")
    for bad, code in (((a.data_ptr(), a.data_ptr()), -3), ((a.data_ptr() + 4, a.data_ptr() + 1024), -2),
                      ((0, a.data_ptr()), -1)):
        with pytest.raises(StencilError) as ei:
            plan.apply_semi(*bad)
        assert ei.value.code == code
    plan.close()
