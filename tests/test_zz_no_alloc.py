"""The allocation-free sweep entry point (stencil_apply_noalloc) through the C ABI.

Some callers cannot allocate device memory at the moment they need a sweep (their
framework's pool owns the free memory, or their footprint is fixed at start-up); this
entry point serves them by keeping its scratch in a fixed device array inside the
library.  Its output must match the CPU oracle and the plan-based stencil_apply on the
same input, on two calls in a row (the second call reuses the scratch the first one left
behind), and a call must not take any device memory.
This file is collected last so that a failure here never hides the other tests.
"""
import numpy as np
import pytest

import oracle
from seismic_wave_propagation_gb300 import StencilError, StencilPlan, synth
from seismic_wave_propagation_gb300._lib import apply_noalloc
from gpu_util import interior_mask, sweep_tol, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nx,ny,nz,R,coeffs", [
    (136, 75, 41, 4, "laplacian8"),    # the direct sweep (the automatic path of this size)
    (64, 64, 64, 1, "average7"),       # the direct sweep
    (256, 256, 160, 4, "laplacian8"),  # the staged sweep
])
def test_noalloc_matches_oracle_and_plan_apply_twice(nx, ny, nz, R, coeffs):
    torch = torch_cuda()
    c = synth.coeffs_for(coeffs)
    c32 = c.astype(np.float32)
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
        want = oracle.apply(u, c32, R)
        tol = sweep_tol(c32, u)
        assert np.max(np.abs(got_h[m].astype(np.float64) - want[m])) <= tol, f"call {call} vs oracle"
        assert np.max(np.abs(got_h[m].astype(np.float64) - ref_h[m])) <= tol, f"call {call} vs stencil_apply"
        np.testing.assert_array_equal(got_h[~m], u[~m])  # shell untouched
    plan.close()


def test_noalloc_takes_no_device_memory():
    """After a first call (which may load the library's device code), a call on a grid of
    another shape leaves the device's free memory unchanged."""
    torch = torch_cuda()
    c = synth.laplacian8_coeffs()
    a = torch.from_numpy(synth.uniform_field(72, 40, 30, seed=5).ravel()).cuda()
    b = a.clone()
    apply_noalloc(72, 40, 30, 4, c, a, b)
    u = synth.uniform_field(200, 66, 52, seed=6)
    d_in = torch.from_numpy(u.ravel()).cuda()
    d_out = d_in.clone()
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    apply_noalloc(200, 66, 52, 4, c, d_in, d_out)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after >= free_before, f"free device memory fell by {free_before - free_after} bytes"
    got = d_out.cpu().numpy().reshape(u.shape)
    want = oracle.apply(u, c.astype(np.float32), 4)
    m = interior_mask(u.shape, 4)
    assert np.max(np.abs(got[m].astype(np.float64) - want[m])) <= sweep_tol(c.astype(np.float32), u)


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
