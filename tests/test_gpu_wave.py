"""Parity of the fused CUDA wave step against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest

import oracle
from seismic_wave_propagation_gb300 import StencilPlan, synth
from gpu_util import Guarded, interior_mask, sample_interior, torch_cuda

pytestmark = pytest.mark.gpu


def gpu_wave(torch, up, u, s, e, c, R, nsteps, two_buffers=False):
    nz, ny, nx = u.shape
    plan = StencilPlan(nx, ny, nz, R, c)
    d = [torch.from_numpy(np.ascontiguousarray(a).ravel()).cuda() for a in (up, u, s, e)]
    a, b, sv, ev = d
    nxt = a.clone()
    for _ in range(nsteps):
        if two_buffers:
            plan.wave_step(a, b, a, sv, ev)
            a, b = b, a
        else:
            plan.wave_step(a, b, nxt, sv, ev)
            a, b, nxt = b, nxt, a
    plan.status(None, a)
    out = (a.cpu().numpy().reshape(u.shape), b.cpu().numpy().reshape(u.shape))
    plan.close()
    return out


def rel_l2(x, y):
    return float(np.linalg.norm((x.astype(np.float64) - y).ravel()) / np.linalg.norm(y.ravel().astype(np.float64)))


@pytest.mark.parametrize("R", [1, 2, 3, 4])
def test_single_step_matches_oracle(R):
    torch = torch_cuda()
    nx, ny, nz = 136, 70, 40
    c = np.random.default_rng(R).uniform(-0.3, 0.3, R + 1)
    up = synth.uniform_field(nx, ny, nz, seed=7)
    u = synth.uniform_field(nx, ny, nz, seed=8)
    s = synth.uniform_field(nx, ny, nz, seed=9, scale=0.1) + np.float32(0.1)
    e = synth.sponge_eta(nx, ny, nz, width=10)
    plan = StencilPlan(nx, ny, nz, R, c)
    gs = [Guarded(torch, a) for a in (up, u, s, e)]
    gn = Guarded(torch, u, fill_sentinel=True)
    plan.wave_step(gs[0].ptr, gs[1].ptr, gn.ptr, gs[2].ptr, gs[3].ptr)
    plan.status()
    got = gn.numpy()
    assert all(g.guards_intact() for g in gs + [gn])
    want = oracle.wave_step(up, u, s, e, np.asarray(c, np.float32), R, u_next=np.zeros_like(u))
    m = interior_mask(u.shape, R)
    # one step: rounding of the stencil sum (scaled by v2dt2 <= 0.2) plus the update
    tol = 1e-5 * (2 + 0.2 * float(np.sum(np.abs(c)))) * 2.0
    assert np.max(np.abs(got[m] - want[m])) <= tol
    assert np.all(got.view(np.uint32)[~m] == 0x7FC0DEAD)
    plan.close()


@pytest.mark.parametrize("two_buffers", [False, True])
def test_multi_step_small(two_buffers):
    torch = torch_cuda()
    nx, ny, nz = 96, 80, 72
    up, u, s, e = synth.wave_fields(nx, ny, nz)
    c = synth.laplacian8_coeffs()
    g_prev, g_cur = gpu_wave(torch, up, u, s, e, c, 4, 30, two_buffers)
    o_prev, o_cur = oracle.run_wave(up, u, s, e, c.astype(np.float32), 4, 30)
    assert rel_l2(g_cur, o_cur) <= 1e-5
    assert rel_l2(g_prev, o_prev) <= 1e-5


def test_sponge_absorbs_pulse_near_face():
    """Pulse 6 points from a face on a 64^3 grid, 200 steps through the sponge."""
    torch = torch_cuda()
    n = 64
    u = synth.gaussian_bump(n, n, n, sigma=3.0, center=(6, 32, 32))
    s = synth.layered_v2dt2(n, n, n)
    e = synth.sponge_eta(n, n, n)
    c = synth.laplacian8_coeffs()
    g_prev, g_cur = gpu_wave(torch, u.copy(), u, s, e, c, 4, 200)
    o_prev, o_cur = oracle.run_wave(u.copy(), u, s, e, c.astype(np.float32), 4, 200)
    assert rel_l2(g_cur, o_cur) <= 1e-4
    assert np.all(np.isfinite(g_cur))


def test_host_buffer_entry_matches_device_path():
    torch = torch_cuda()
    nx, ny, nz = 96, 40, 36
    up, u, s, e = synth.wave_fields(nx, ny, nz)
    c = synth.laplacian8_coeffs()
    plan = StencilPlan(nx, ny, nz, 4, c)
    hp, hu = up.copy(), u.copy()
    plan.wave_run_host(hp, hu, s, e, 7)
    g_prev, g_cur = gpu_wave(torch, up, u, s, e, c, 4, 7, two_buffers=True)
    np.testing.assert_array_equal(hu, g_cur)
    np.testing.assert_array_equal(hp, g_prev)
    plan.close()


@pytest.fixture(scope="module")
def wave640():
    """The 640^3 acoustic workload's inputs and the oracle's independent 100-step run."""
    n = 640
    up, u, s, e = synth.wave_fields(n, n, n)
    c = synth.laplacian8_coeffs()
    o_prev, o_cur = oracle.run_wave(up, u, s, e, c.astype(np.float32), 4, 100)
    return {"fields": (up, u, s, e), "c": c, "o_prev": o_prev, "o_cur": o_cur}


def test_wave25_640_hundred_steps(wave640):
    """The 640^3 acoustic run: 100 steps on the GPU and in the oracle from identical
    inputs, relative L2 <= 1e-4; plus a per-step sampled check on the GPU's own state."""
    torch = torch_cuda()
    n = 640
    up, u, s, e = wave640["fields"]
    c = wave640["c"]
    c32 = c.astype(np.float32)
    plan = StencilPlan(n, n, n, 4, c)
    d = [torch.from_numpy(a.ravel()).cuda() for a in (up, u, s, e)]
    a, b, sv, ev = d
    nxt = a.clone()
    idx = sample_interior(u.shape, 4, 100000, planes=(320,))
    for k in range(100):
        if k in (0, 50):
            hp, hc = a.cpu().numpy().reshape(u.shape), b.cpu().numpy().reshape(u.shape)
        plan.wave_step(a, b, nxt, sv, ev)
        if k in (0, 50):
            plan.status(None, nxt)
            want = oracle.wave_points(hp, hc, s, e, c32, 4, idx)
            got = nxt.cpu().numpy()[idx]
            assert np.max(np.abs(got - want)) <= 1e-5 * (2 + 0.2025 * 19.51) * float(np.max(np.abs(hc)))
        a, b, nxt = b, nxt, a
    plan.status(None, b)
    g_cur = b.cpu().numpy().reshape(u.shape)
    plan.close()
    r = rel_l2(g_cur, wave640["o_cur"])
    print(f"wave25 640^3 x100: relative L2 {r:.3e}, |u|_2 {np.linalg.norm(wave640['o_cur']):.4f}")
    assert r <= 1e-4


@pytest.mark.parametrize("pml", [-1, 16])
def test_native_wave_steps_640_match_oracle(wave640, pml):
    """The 640^3 workload as the benchmark runs it: wave_steps, all 100 steps captured once
    as a CUDA graph (pml < 0: wave_step; 16: wave_step_pml with the 16-point sponge band),
    against the oracle's run: relative L2 <= 1e-4 for the last two levels."""
    torch = torch_cuda()
    n = 640
    up, u, s, e = wave640["fields"]
    c = wave640["c"]
    plan = StencilPlan(n, n, n, 4, c)
    f = [torch.from_numpy(x.ravel()).cuda() for x in (up, u, s, e)]
    bufs = [f[0], f[1], f[0].clone()]
    plan.wave_steps(bufs[0], bufs[1], bufs[2], f[2], f[3], 100, pml_width=pml, use_graph=True)
    plan.status(None, bufs[0])
    cur = bufs[101 % 3].cpu().numpy().reshape(u.shape)
    prev = bufs[100 % 3].cpu().numpy().reshape(u.shape)
    plan.close()
    del f, bufs
    r_cur, r_prev = rel_l2(cur, wave640["o_cur"]), rel_l2(prev, wave640["o_prev"])
    print(f"wave_steps 640^3 x100 (pml {pml}): relative L2 {r_cur:.3e} / {r_prev:.3e}")
    assert r_cur <= 1e-4 and r_prev <= 1e-4


def band_mask(shape, width):
    """True at points closer than `width` to a face."""
    nz, ny, nx = shape
    d = np.minimum.reduce(np.meshgrid(np.minimum(np.arange(nz), nz - 1 - np.arange(nz)),
                                      np.minimum(np.arange(ny), ny - 1 - np.arange(ny)),
                                      np.minimum(np.arange(nx), nx - 1 - np.arange(nx)), indexing="ij"))
    return d < width


@pytest.mark.parametrize("pml,dims", [(16, (200, 150, 90)), (10, (136, 75, 41)), (0, (136, 75, 41)),
                                      (1000, (136, 75, 41)), (5, (96, 70, 60)),
                                      (6, (1088, 320, 128)), (4, (1024, 128, 64)), (0, (512, 96, 40))])
def test_wave_step_pml_matches_oracle(pml, dims):
    """Region-split step on fields whose eta vanishes beyond `pml` points from the faces
    (random inside the band): identical to the full update, which the oracle computes."""
    torch = torch_cuda()
    nx, ny, nz = dims
    c = synth.laplacian8_coeffs()
    c32 = c.astype(np.float32)
    up = synth.uniform_field(nx, ny, nz, seed=21)
    u = synth.uniform_field(nx, ny, nz, seed=22)
    s = synth.uniform_field(nx, ny, nz, seed=23, scale=0.05) + np.float32(0.1)
    e = synth.uniform_field(nx, ny, nz, seed=24, scale=0.05) + np.float32(0.05)
    e = np.where(band_mask(u.shape, pml), e, np.float32(0.0)).astype(np.float32)
    plan = StencilPlan(nx, ny, nz, 4, c)
    d = [torch.from_numpy(a.ravel()).cuda() for a in (up, u, s, e)]
    nxt = torch.full_like(d[0], 7.0)
    plan.wave_step_pml(d[0], d[1], nxt, d[2], d[3], pml)
    plan.status(None, nxt)
    got = nxt.cpu().numpy().reshape(u.shape)
    want = oracle.wave_step(up, u, s, e, c32, 4, u_next=np.full_like(u, 7.0))
    m = interior_mask(u.shape, 4)
    assert np.max(np.abs(got[m] - want[m])) <= 1e-5 * (2 + 0.15 * 19.51) * 2
    assert np.all(got[~m] == 7.0)
    plan.close()


def test_wave_step_pml_on_the_sponge_model_equals_wave_step():
    """On the sponge model (eta = 0 beyond 16 points) the split step reproduces wave_step."""
    torch = torch_cuda()
    n = 96
    up, u, s, e = synth.wave_fields(n, n, n)
    c = synth.laplacian8_coeffs()
    plan = StencilPlan(n, n, n, 4, c)
    d = [torch.from_numpy(a.ravel()).cuda() for a in (up, u, s, e)]
    a, b = d[0].clone(), d[1].clone()
    ap, bp = d[0].clone(), d[1].clone()
    for _ in range(20):
        plan.wave_step(a, b, a, d[2], d[3])
        a, b = b, a
        plan.wave_step_pml(ap, bp, ap, d[2], d[3], 16)
        ap, bp = bp, ap
    plan.status(None, a)
    g, gp = b.cpu().numpy(), bp.cpu().numpy()
    assert rel_l2(gp, g.astype(np.float64)) <= 1e-6
    plan.close()


@pytest.mark.parametrize("use_graph", [False, True])
@pytest.mark.parametrize("pml", [-1, 16])
def test_native_step_loop_matches_step_by_step(use_graph, pml):
    torch = torch_cuda()
    n, steps = 80, 7
    up, u, s, e = synth.wave_fields(n, n, n)
    c = synth.laplacian8_coeffs()
    plan = StencilPlan(n, n, n, 4, c)
    f = [torch.from_numpy(x.ravel()).cuda() for x in (up, u, s, e)]
    for _ in range(2):  # the second call replays the cached graph
        bufs = [f[0].clone(), f[1].clone(), f[0].clone()]
        plan.wave_steps(bufs[0], bufs[1], bufs[2], f[2], f[3], steps, pml_width=pml, use_graph=use_graph)
        plan.status(None, bufs[0])
    a, b, t = f[0].clone(), f[1].clone(), f[0].clone()
    for _ in range(steps):
        if pml < 0:
            plan.wave_step(a, b, t, f[2], f[3])
        else:
            plan.wave_step_pml(a, b, t, f[2], f[3], pml)
        a, b, t = b, t, a
    plan.status(None, a)
    assert torch.equal(bufs[(steps + 1) % 3], b)
    assert torch.equal(bufs[steps % 3], a)
    plan.close()


def test_eta_stencil_damping_field_matches_oracle():
    """wave_eta_stencil: the radius-1 star stencil of eta everywhere but on the faces, which
    it leaves untouched; new weights on a second call take effect."""
    torch = torch_cuda()
    nx, ny, nz = 136, 75, 41
    e = synth.uniform_field(nx, ny, nz, seed=61, scale=0.05) + np.float32(0.05)
    plan = StencilPlan(nx, ny, nz, 4, synth.laplacian8_coeffs())
    d = torch.from_numpy(e.ravel()).cuda()
    out = torch.full_like(d, 9.0)
    for e0, e1 in ((0.5, 1.0 / 12.0), (0.25, 0.125)):
        plan.eta_stencil(d, out, e0, e1)
        plan.status(None, out)
        got = out.cpu().numpy().reshape(e.shape)
        want = oracle.apply(e, np.float32([e0, e1]), 1)
        m1 = interior_mask(e.shape, 1)
        assert np.max(np.abs(got[m1].astype(np.float64) - want[m1])) <= 1e-6 * 0.1
        assert np.all(got[~m1] == 9.0)
    plan.close()


@pytest.mark.parametrize("nsteps,dims", [(1, (136, 75, 41)), (25, (96, 80, 72))])
def test_wave_with_7_point_eta_stencil_matches_oracle(nsteps, dims):
    """The PML step whose damping is the 7-point stencil of eta: wave_eta_stencil once, then
    wave_steps (one CUDA graph) on the result, against the oracle's direct 7-point step."""
    torch = torch_cuda()
    nx, ny, nz = dims
    c = synth.laplacian8_coeffs()
    c32 = c.astype(np.float32)
    e0, e1 = 0.5, 1.0 / 12.0
    up, u, s, _ = synth.wave_fields(nx, ny, nz)
    u = (u + synth.uniform_field(nx, ny, nz, seed=62, scale=0.01)).astype(np.float32)
    e = synth.sponge_eta(nx, ny, nz, width=10) + synth.uniform_field(nx, ny, nz, seed=63, scale=0.01) + \
        np.float32(0.01)
    e = e.astype(np.float32)
    plan = StencilPlan(nx, ny, nz, 4, c)
    f = [torch.from_numpy(x.ravel()).cuda() for x in (up, u, s, e)]
    eff = torch.empty_like(f[3])
    plan.eta_stencil(f[3], eff, e0, e1)
    bufs = [f[0], f[1], f[0].clone()]
    plan.wave_steps(bufs[0], bufs[1], bufs[2], f[2], eff, nsteps, use_graph=True)
    plan.status(None, bufs[0])
    got = bufs[(nsteps + 1) % 3].cpu().numpy().reshape(u.shape)
    a, b, t = up.copy(), u.copy(), up.copy()
    for _ in range(nsteps):
        oracle.wave_step_eta7(a, b, s, e, c32, 4, e0, e1, u_next=t)
        a, b, t = b, t, a
    m = interior_mask(u.shape, 4)
    if nsteps == 1:
        assert np.max(np.abs(got[m] - b[m])) <= 1e-5 * (2 + 0.2025 * 19.51) * float(np.max(np.abs(u)))
    else:
        assert rel_l2(got, b) <= 1e-5
    np.testing.assert_array_equal(got[~m], b[~m])
    plan.close()


def inner_share(dims, pml, R=4, ty=16):
    """Share of the step's tiles x planes in the inner region of wave_step_pml (64-wide
    tiles from x = 0, tile_y-high tiles from y = R)."""
    nx, ny, nz = dims
    ntx, nty = -(-nx // 64), -(-(ny - 2 * R) // ty)
    bx = max(0, min(ntx, (nx - pml) // 64) - (-(-pml // 64)))
    by = max(0, min(nty, (ny - pml - R) // ty) - max(0, -(-(pml - R) // ty)))
    bz = max(0, min(nz - R, nz - pml) - max(R, pml))
    return bx * by * bz / (ntx * nty * (nz - 2 * R))


@pytest.mark.parametrize("pml,dims", [(6, (1088, 320, 128)), (4, (1024, 128, 64))])
def test_region_split_step_loop_matches_oracle(pml, dims):
    """Grids where wave_step_pml runs as two launches (inner region without eta beside the
    band with the full update): 6 steps through wave_steps in one CUDA graph, against the
    oracle's steps on the same fields."""
    assert inner_share(dims, pml) >= 0.6  # the split path, not the single launch
    torch = torch_cuda()
    nx, ny, nz = dims
    c = synth.laplacian8_coeffs()
    c32 = c.astype(np.float32)
    up = synth.uniform_field(nx, ny, nz, seed=71)
    u = synth.uniform_field(nx, ny, nz, seed=72)
    s = synth.uniform_field(nx, ny, nz, seed=73, scale=0.05) + np.float32(0.1)
    e = synth.uniform_field(nx, ny, nz, seed=74, scale=0.05) + np.float32(0.05)
    e = np.where(band_mask(u.shape, pml), e, np.float32(0.0)).astype(np.float32)
    plan = StencilPlan(nx, ny, nz, 4, c)
    f = [torch.from_numpy(x.ravel()).cuda() for x in (up, u, s, e)]
    bufs = [f[0], f[1], f[0].clone()]
    steps = 6
    for _ in range(2):  # the second call replays the captured graph
        bufs = [torch.from_numpy(up.ravel()).cuda(), torch.from_numpy(u.ravel()).cuda(),
                torch.from_numpy(up.ravel()).cuda()]
        plan.wave_steps(bufs[0], bufs[1], bufs[2], f[2], f[3], steps, pml_width=pml, use_graph=True)
        plan.status(None, bufs[0])
    got = bufs[(steps + 1) % 3].cpu().numpy().reshape(u.shape)
    a, b, t = up.copy(), u.copy(), up.copy()
    for _ in range(steps):
        oracle.wave_step(a, b, s, e, c32, 4, u_next=t)
        a, b, t = b, t, a
    assert rel_l2(got, b) <= 1e-5
    m = interior_mask(u.shape, 4)
    np.testing.assert_array_equal(got[~m], b[~m])
    plan.close()


def test_wave_step_beyond_2pow31_points():
    """64-bit indexing of the fused wave step: 2048 x 1024 x 1030 = 2.16e9 points (8.6 GB
    per field), sampled against the oracle, including the last interior row.  u_prev and u
    are one field and v2dt2 and eta another (allowed: only u_next must not overlap them)."""
    torch = torch_cuda()
    nx, ny, nz, R = 2048, 1024, 1030, 4
    if torch.cuda.get_device_properties(0).total_memory < 60 * 2 ** 30:
        pytest.skip("needs ~30 GB of device memory")
    c = synth.laplacian8_coeffs()
    c32 = c.astype(np.float32)
    u = synth.uniform_field(nx, ny, nz, seed=98)
    s = (np.abs(u) * np.float32(0.05)).astype(np.float32)  # v2dt2 and eta in [0, 0.05]
    plan = StencilPlan(nx, ny, nz, R, c)
    du = torch.from_numpy(u.ravel()).cuda()
    ds = torch.from_numpy(s.ravel()).cuda()
    dn = torch.full_like(du, 5.0)
    plan.wave_step(du, du, dn, ds, ds)
    plan.status(None, dn)
    idx = sample_interior(u.shape, R, 200000, seed=4)
    top = (nz - R - 1) * nx * ny + (ny - R - 1) * nx + np.arange(R, nx - R, dtype=np.int64)  # last interior row
    idx = np.unique(np.concatenate([idx, top]))
    assert idx.max() > 2 ** 31
    got = dn[torch.from_numpy(idx).cuda()].cpu().numpy().astype(np.float64)
    want = oracle.wave_points(u, u, s, s, c32, R, idx)
    tol = 1e-5 * (3 + 0.05 * float(np.sum(np.abs(c32)))) * float(np.max(np.abs(u))) * 2.0
    assert np.max(np.abs(got - want)) <= tol
    assert np.all(dn[(nz - 1) * nx * ny:].cpu().numpy() == 5.0)  # the shell's last plane is untouched
    plan.close()
