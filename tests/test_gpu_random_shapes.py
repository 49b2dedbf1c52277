"""Seeded random grid shapes against the oracle: every radius, both ring protocols of the
staged sweep (radius 4 meets at a CTA barrier, radii 1-3 release slots warp by warp), the
direct-load sweep, the semi-stencil sweep and the wave step, on sizes that are ragged in every axis (partial x and y tiles, short and
uneven z-chunks, empty interiors)."""
import numpy as np
import pytest

import oracle
from seismic_wave_propagation_gb300 import StencilPlan, synth
from gpu_util import Guarded, interior_mask, sweep_tol, torch_cuda

pytestmark = pytest.mark.gpu


def shapes(seed: int, count: int):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        R = int(rng.integers(1, 5))
        nx = 4 * int(rng.integers(1, 80))  # 4 .. 316, x rows stay 16-byte aligned
        ny = int(rng.integers(1, 140))
        nz = int(rng.integers(1, 70))
        out.append((nx, ny, nz, R))
    return out


SWEEP_SHAPES = shapes(2024, 24)
WAVE_SHAPES = shapes(2025, 10)


@pytest.mark.parametrize("kernel", ["staged", "direct", "semi"])
@pytest.mark.parametrize("nx,ny,nz,R", SWEEP_SHAPES)
def test_random_shape_sweep(nx, ny, nz, R, kernel):
    torch = torch_cuda()
    u = synth.uniform_field(nx, ny, nz, seed=nx * 7 + ny * 11 + nz * 13 + R)
    c = np.random.default_rng(nx + ny + nz).uniform(-1, 1, R + 1)
    plan = StencilPlan(nx, ny, nz, R, c)
    if kernel != "semi":
        plan.set_sweep_path(kernel)
    gin = Guarded(torch, u)
    gout = Guarded(torch, u, fill_sentinel=True)
    (plan.apply_semi if kernel == "semi" else plan.apply)(gin.ptr, gout.ptr)
    plan.status()
    got = gout.numpy()
    assert gin.guards_intact() and gout.guards_intact()
    plan.close()
    c32 = np.asarray(c, np.float32)
    m = interior_mask(u.shape, R)
    want = oracle.apply(u, c32, R, out=np.zeros_like(u))
    if m.any():
        assert np.max(np.abs(got[m].astype(np.float64) - want[m])) <= sweep_tol(c32, u)
    assert np.all(got.view(np.uint32)[~m] == 0x7FC0DEAD), "shell written"


@pytest.mark.parametrize("nx,ny,nz,R", WAVE_SHAPES)
def test_random_shape_wave_step(nx, ny, nz, R):
    torch = torch_cuda()
    seed = nx + 3 * ny + 5 * nz + R
    up = synth.uniform_field(nx, ny, nz, seed=seed)
    u = synth.uniform_field(nx, ny, nz, seed=seed + 1)
    s = synth.uniform_field(nx, ny, nz, seed=seed + 2, scale=0.1) + np.float32(0.1)
    e = synth.sponge_eta(nx, ny, nz, width=6)
    c = np.random.default_rng(seed).uniform(-0.3, 0.3, R + 1)
    plan = StencilPlan(nx, ny, nz, R, c)
    gs = [Guarded(torch, a) for a in (up, u, s, e)]
    gn = Guarded(torch, u, fill_sentinel=True)
    plan.wave_step(gs[0].ptr, gs[1].ptr, gn.ptr, gs[2].ptr, gs[3].ptr)
    plan.status()
    got = gn.numpy()
    assert all(g.guards_intact() for g in gs + [gn])
    plan.close()
    want = oracle.wave_step(up, u, s, e, np.asarray(c, np.float32), R, u_next=np.zeros_like(u))
    m = interior_mask(u.shape, R)
    if m.any():
        tol = 1e-5 * (2 + 0.2 * float(np.sum(np.abs(c)))) * 2.0
        assert np.max(np.abs(got[m] - want[m])) <= tol
    assert np.all(got.view(np.uint32)[~m] == 0x7FC0DEAD)


def split_shapes(seed: int, count: int):
    """Shapes (all radii) on which wave_step_pml runs as two launches: the inner region
    holds at least 0.6 of the tiles x planes (64-wide tiles from x = 0, 16-high tiles from
    y = R).  Band widths are drawn from 0-6, but at these sizes only width 0 passes, so
    these cases run the no-eta kernel on ragged grids beside a thin band launch; wider
    bands are covered on larger grids in the wave tests."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(100 * count):
        if len(out) == count:
            break
        R = int(rng.integers(1, 5))
        nx, ny, nz = 64 * int(rng.integers(2, 7)), int(rng.integers(60, 200)), int(rng.integers(20, 70))
        pml = int(rng.integers(0, 7))
        ntx, nty = -(-nx // 64), -(-(ny - 2 * R) // 16)
        bx = max(0, min(ntx, (nx - pml) // 64) - (-(-pml // 64)))
        by = max(0, min(nty, (ny - pml - R) // 16) - max(0, -(-(pml - R) // 16)))
        bz = max(0, min(nz - R, nz - pml) - max(R, pml))
        if bx * by * bz >= 0.6 * ntx * nty * (nz - 2 * R):
            out.append((nx, ny, nz, R, pml))
    return out


@pytest.mark.parametrize("nx,ny,nz,R,pml", split_shapes(2026, 10))
def test_random_shape_region_split_step(nx, ny, nz, R, pml):
    torch = torch_cuda()
    seed = nx + 3 * ny + 5 * nz + R + 7 * pml
    up = synth.uniform_field(nx, ny, nz, seed=seed)
    u = synth.uniform_field(nx, ny, nz, seed=seed + 1)
    s = synth.uniform_field(nx, ny, nz, seed=seed + 2, scale=0.1) + np.float32(0.1)
    z, y, x = np.meshgrid(*[np.arange(n) for n in (nz, ny, nx)], indexing="ij")
    d = np.minimum.reduce([x, nx - 1 - x, y, ny - 1 - y, z, nz - 1 - z])
    e = np.where(d < pml, synth.uniform_field(nx, ny, nz, seed=seed + 3, scale=0.05) + np.float32(0.05),
                 np.float32(0.0)).astype(np.float32)
    c = np.random.default_rng(seed).uniform(-0.3, 0.3, R + 1)
    plan = StencilPlan(nx, ny, nz, R, c)
    gs = [Guarded(torch, a) for a in (up, u, s, e)]
    gn = Guarded(torch, u, fill_sentinel=True)
    plan.wave_step_pml(gs[0].ptr, gs[1].ptr, gn.ptr, gs[2].ptr, gs[3].ptr, pml)
    plan.status()
    got = gn.numpy()
    assert all(g.guards_intact() for g in gs + [gn])
    plan.close()
    want = oracle.wave_step(up, u, s, e, np.asarray(c, np.float32), R, u_next=np.zeros_like(u))
    m = interior_mask(u.shape, R)
    tol = 1e-5 * (2 + 0.2 * float(np.sum(np.abs(c)))) * 2.0
    assert np.max(np.abs(got[m] - want[m])) <= tol
    assert np.all(got.view(np.uint32)[~m] == 0x7FC0DEAD)


def two_sweep_shapes(seed: int, count: int):
    rng = np.random.default_rng(seed)
    return [(4 * int(rng.integers(1, 80)), int(rng.integers(1, 140)), int(rng.integers(1, 70)))
            for _ in range(count)]


TWO_SWEEP_SHAPES = two_sweep_shapes(2027, 16)


@pytest.mark.parametrize("nx,ny,nz", TWO_SWEEP_SHAPES)
def test_random_shape_two_sweep_pass(nx, ny, nz):
    """stencil_apply2 (radius 1) on seeded shapes ragged in every axis: 30-row tiles whose
    last row group runs past the tile, partial x tiles, short z, empty interiors; against
    two oracle sweeps with a fixed shell, guard bands and shell sentinels kept."""
    torch = torch_cuda()
    u = synth.uniform_field(nx, ny, nz, seed=nx * 5 + ny * 3 + nz)
    c = np.random.default_rng(nx + ny).uniform(-1, 1, 2)
    c = (c / (abs(c[0]) + 6.0 * abs(c[1]))).astype(np.float32)  # max-norm gain 1
    plan = StencilPlan(nx, ny, nz, 1, c)
    gin = Guarded(torch, u)
    gout = Guarded(torch, u, fill_sentinel=True)
    plan.apply2(gin.ptr, gout.ptr)
    plan.status()
    got = gout.numpy()
    assert gin.guards_intact() and gout.guards_intact()
    plan.close()
    want = oracle.run_sweeps(u, c, 1, 2)
    m = interior_mask(u.shape, 1)
    if m.any():
        assert np.max(np.abs(got[m].astype(np.float64) - want[m])) <= 2e-5 * float(np.max(np.abs(u)))
    assert np.all(got.view(np.uint32)[~m] == 0x7FC0DEAD), "shell written"
