"""The native time loops and host-buffer calls against the CPU oracle (through the C ABI).

stencil_sweeps (with and without its CUDA graph), stencil_apply_host (one pipelined
sweep, several sweeps) and wave_run_host each run a whole workload inside the library;
their final fields are compared with the oracle's own loops (run_sweeps, run_wave) from
the same inputs.

Sweep tolerance: each GPU sweep is within 1e-5 * sum|c| * max|u_in| of the exact
operator applied to its own input, and the coefficients here are scaled so that the
operator's max-norm gain |c0| + 6 * sum_r |c_r| is 1: it does not amplify earlier errors,
and after k sweeps the difference to the oracle's run is at most k * 1e-5 * max|u0|.
"""
import numpy as np
import pytest

import oracle
from seismic_wave_propagation_gb300 import StencilPlan, synth
from gpu_util import interior_mask, torch_cuda

pytestmark = pytest.mark.gpu


def unit_coeffs(R, seed):
    """Coefficients scaled to a max-norm gain |c0| + 6 sum_r |c_r| of 1 (non-expanding)."""
    if R == 4:
        c = synth.laplacian8_coeffs()
    else:
        c = np.random.default_rng(seed).uniform(-1, 1, R + 1)
    return (c / (abs(c[0]) + 6.0 * np.sum(np.abs(c[1:])))).astype(np.float32)


@pytest.mark.parametrize("path", ["staged", "auto"])
@pytest.mark.parametrize("use_graph", [True, False])
@pytest.mark.parametrize("nsweeps", [3, 4])
@pytest.mark.parametrize("dims,R", [((136, 75, 41), 4), ((200, 33, 57), 1), ((68, 130, 30), 2),
                                    ((256, 96, 70), 3), ((256, 256, 128), 1)])
def test_native_sweeps_match_oracle_run_sweeps(dims, R, nsweeps, use_graph, path):
    """On the staged path and on the automatic one: the direct kernel at these sizes, and
    at 256 x 256 x 128 (radius 1, above 8 million points) two-sweep passes with the odd
    sweeps on the direct kernel."""
    torch = torch_cuda()
    nx, ny, nz = dims
    c = unit_coeffs(R, nx + R)
    u0 = synth.uniform_field(nx, ny, nz, seed=500 + R)
    plan = StencilPlan(nx, ny, nz, R, c)
    plan.set_sweep_path(path)
    a = torch.from_numpy(u0.ravel()).cuda()
    b = a.clone()
    for _ in range(2):  # the second call replays the cached graph
        a.copy_(torch.from_numpy(u0.ravel()))
        b.copy_(a)
        plan.sweeps(a, b, nsweeps, use_graph=use_graph)
        plan.status(None, a)
    got = (a if nsweeps % 2 == 0 else b).cpu().numpy().reshape(u0.shape)
    want = oracle.run_sweeps(u0, c, R, nsweeps)
    m = interior_mask(u0.shape, R)
    tol = nsweeps * 1e-5 * float(np.max(np.abs(u0)))
    err = float(np.max(np.abs(got[m].astype(np.float64) - want[m])))
    assert err <= tol, f"{err} > {tol}"
    np.testing.assert_array_equal(got[~m], u0[~m])  # fixed shell
    plan.close()


@pytest.mark.parametrize("nsweeps", [1, 3, 5])
@pytest.mark.parametrize("dims,R", [((136, 75, 200), 4), ((64, 40, 140), 1), ((32, 32, 20), 4)])
def test_host_buffer_sweeps_match_oracle(dims, R, nsweeps):
    """stencil_apply_host: one sweep runs pipelined over z-slabs on three streams, several
    sweeps run back to back on the device (radius 1: four of five in two-sweep passes);
    both from host to host."""
    torch_cuda()
    nx, ny, nz = dims
    c = unit_coeffs(R, 7)
    u0 = synth.uniform_field(nx, ny, nz, seed=77)
    plan = StencilPlan(nx, ny, nz, R, c)
    out_h = np.full_like(u0, 3.0)
    for _ in range(2):
        plan.apply_host(u0, out_h, nsweeps)
    want = oracle.run_sweeps(u0, c, R, nsweeps)
    m = interior_mask(u0.shape, R)
    tol = nsweeps * 1e-5 * float(np.max(np.abs(u0)))
    assert float(np.max(np.abs(out_h[m].astype(np.float64) - want[m]))) <= tol
    np.testing.assert_array_equal(out_h[~m], u0[~m])
    if nsweeps == 1:
        ph = plan.host_phases()
        assert ph["slabs"] >= 1 and 0 < ph["first_slab_in_ms"] <= ph["copies_in_done_ms"] <= ph["total_ms"]
        assert ph["sweeps_done_ms"] <= ph["total_ms"]
    plan.close()


def rel_l2(x, y):
    return float(np.linalg.norm((x.astype(np.float64) - y).ravel()) / np.linalg.norm(y.ravel().astype(np.float64)))


@pytest.mark.parametrize("nsteps", [1, 7, 30])
def test_wave_run_host_matches_oracle_run_wave(nsteps):
    """wave_run_host (two-buffer stepping on the device, host to host) against run_wave."""
    torch_cuda()
    nx, ny, nz = 96, 40, 36
    up, u, s, e = synth.wave_fields(nx, ny, nz)
    e = synth.sponge_eta(nx, ny, nz, width=8)
    c = synth.laplacian8_coeffs()
    plan = StencilPlan(nx, ny, nz, 4, c)
    hp, hu = up.copy(), u.copy()
    plan.wave_run_host(hp, hu, s, e, nsteps)
    o_prev, o_cur = oracle.run_wave(up, u, s, e, c.astype(np.float32), 4, nsteps)
    assert rel_l2(hu, o_cur) <= 1e-5
    assert rel_l2(hp, o_prev) <= 1e-5
    m = interior_mask(u.shape, 4)
    np.testing.assert_array_equal(hu[~m], u[~m])
    plan.close()
