"""The device watchdog: a staged load that never arrives ends in STENCIL_ERR_TIMEOUT.

The plan's test hook makes every CTA skip one of its TMA loads (nothing sets that
mbarrier), so the bounded wait for it runs out after about two seconds; the kernel
records the failure, waits for its own copies still in flight and returns.  No GPU fault
is involved.  Afterwards the plan works normally again.
"""
import time

import numpy as np
import pytest

import oracle
from seismic_wave_propagation_gb300 import StencilError, StencilPlan, synth
from gpu_util import interior_mask, sweep_tol, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind,R,dims", [("apply", 4, (136, 75, 41)), ("apply", 4, (1032, 1020, 14)),
                                         ("apply", 1, (136, 75, 41)), ("semi", 4, (136, 75, 41)),
                                         ("wave", 4, (136, 75, 41))])
def test_lost_load_times_out_and_plan_recovers(kind, R, dims):
    """R = 4 sweeps meet at a CTA barrier every plane (small planes) or every two planes
    (planes of 2^20 points or more), R = 1 sweeps release ring slots warp by warp: every
    protocol must turn a lost load into a timeout."""
    torch = torch_cuda()
    nx, ny, nz = dims
    c = synth.laplacian8_coeffs() if R == 4 else synth.laplacian2_coeffs()
    plan = StencilPlan(nx, ny, nz, R, c)
    plan.set_sweep_path("staged")  # the direct sweep has no staged loads to lose
    u = synth.uniform_field(nx, ny, nz)
    d = torch.from_numpy(u.ravel()).cuda()
    out = d.clone()
    aux = [d.clone() * 0.0 + 0.1, d.clone() * 0.0]

    def run():
        if kind == "apply":
            plan.apply(d, out)
        elif kind == "semi":
            plan.apply_semi(d, out)
        else:
            plan.wave_step(aux[1], d, out, aux[0], aux[1])

    plan.debug_inject(1)
    t0 = time.time()
    run()
    with pytest.raises(StencilError) as ei:
        plan.status(None, d)
    assert ei.value.code == -5, ei.value
    assert time.time() - t0 < 30
    plan.debug_inject(0)
    run()
    plan.status(None, d)  # status was cleared by the previous read; this run is clean
    if kind in ("apply", "semi"):
        m = interior_mask(u.shape, R)
        want = oracle.apply(u, c.astype(np.float32), R)
        got = out.cpu().numpy().reshape(u.shape)
        assert np.max(np.abs(got[m] - want[m])) <= sweep_tol(c, u)
    plan.close()
