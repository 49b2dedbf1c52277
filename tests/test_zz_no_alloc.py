"""The allocation-free sweep entry point (stencil_apply_noalloc) through the C ABI.

Some callers cannot allocate device memory at the moment they need a sweep (their
framework's pool owns the free memory, or their footprint is fixed at start-up); this
entry point serves them by keeping its scratch in a fixed device array inside the
library.  Its output must match the plan-based stencil_apply on the same input, on two
calls in a row (the second call reuses the scratch the first one left behind).
This file is collected last so that a failure here never hides the other tests.
"""
import numpy as np
import pytest

from seismic_wave_propagation_gb300 import StencilError, StencilPlan, synth
from seismic_wave_propagation_gb300._lib import apply_noalloc
from gpu_util import interior_mask, sweep_tol, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nx,ny,nz,R,coeffs", [
    (136, 75, 41, 4, "laplacian8"),
    (64, 64, 64, 1, "average7"),
])
def test_noalloc_matches_plan_apply_twice(nx, ny, nz, R, coeffs):
    torch = torch_cuda()
    c = synth.coeffs_for(coeffs)
    plan = StencilPlan(nx, ny, nz, R, c)
    m = interior_mask((nz, ny, nx), R)
    for call, seed in enumerate((11, 12)):
        u = synth.uniform_field(nx, ny, nz, seed=seed)
        d_in = torch.from_numpy(u.ravel()).cuda()
        ref = d_in.clone()
        got = d_in.clone()
        plan.apply(d_in, ref)
        plan.status(None, ref)
        apply_noalloc(nx, ny, nz, R, c, d_in, got)
        ref_h = ref.cpu().numpy().reshape(u.shape)
        got_h = got.cpu().numpy().reshape(u.shape)
        tol = sweep_tol(c, u)
        assert np.max(np.abs(got_h[m].astype(np.float64) - ref_h[m])) <= tol, f"call {call}"
        np.testing.assert_array_equal(got_h[~m], u[~m])  # shell untouched
    plan.close()


def test_noalloc_rejects_bad_sizes():
    torch = torch_cuda()
    c = synth.laplacian8_coeffs()
    a = torch.zeros(64, device="cuda")
    with pytest.raises(StencilError) as ei:
        apply_noalloc(1 << 31, 4, 4, 4, c, a, a)
    assert ei.value.code == -1 and "maximum" in str(ei.value)
    with pytest.raises(StencilError) as ei:
        apply_noalloc(30, 16, 16, 4, c, a, a)
    assert ei.value.code == -2
