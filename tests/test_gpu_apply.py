"""Parity of the CUDA stencil sweep against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest

import oracle
from seismic_wave_propagation_gb300 import StencilError, StencilPlan, synth
from gpu_util import Guarded, interior_mask, sample_interior, sweep_tol, torch_cuda

pytestmark = pytest.mark.gpu


def run_apply(torch, u, coeffs, R, shell_from_input=False, path=None):
    nz, ny, nx = u.shape
    plan = StencilPlan(nx, ny, nz, R, coeffs)
    if path is not None:
        plan.set_sweep_path(path)
        assert plan.sweep_path == path
    gin = Guarded(torch, u)
    gout = Guarded(torch, u, fill_sentinel=not shell_from_input)
    plan.apply(gin.ptr, gout.ptr)
    plan.status()
    out = gout.numpy()
    assert gin.guards_intact() and gout.guards_intact()
    np.testing.assert_array_equal(gin.numpy(), u)  # input untouched
    plan.close()
    return out


def check(u, out, coeffs, R, shell_bits=None):
    c32 = np.asarray(coeffs, np.float32)
    m = interior_mask(u.shape, R)
    want = oracle.apply(u, c32, R, out=np.zeros_like(u))
    err = np.abs(out[m].astype(np.float64) - want[m])
    tol = sweep_tol(c32, u)
    assert err.size == 0 or err.max() <= tol, f"max err {err.max()} > {tol}"
    if shell_bits is None:
        assert np.all(out.view(np.uint32)[~m] == 0x7FC0DEAD), "shell written"
    else:
        np.testing.assert_array_equal(out[~m], shell_bits[~m])
    return err.max() if err.size else 0.0


CASES = [
    # (nx, ny, nz, R): several x tiles with a ragged last tile, ragged y tiles, odd nz
    (136, 75, 41, 1), (136, 75, 41, 2), (136, 75, 41, 3), (136, 75, 41, 4),
    (64, 64, 64, 4), (200, 33, 17, 4), (12, 12, 12, 4), (12, 9, 9, 4), (4, 5, 6, 1),
    (8, 40, 7, 2), (20, 21, 11, 3), (256, 96, 200, 4), (68, 130, 30, 1),
    # planes of 2^20 points or more: the radius-4 sweep's 64 x 24 tiles, ragged in x and y;
    # one narrow tile column 4167 tiles tall; a plane just past 2^20 points
    (1100, 1000, 19, 4), (12, 100000, 10, 4), (2052, 520, 13, 4),
]


@pytest.mark.parametrize("path", ["staged", "direct"])
@pytest.mark.parametrize("nx,ny,nz,R", CASES)
def test_apply_matches_oracle(nx, ny, nz, R, path):
    """Both sweep kernels on the same ragged grids (the automatic choice takes the direct
    one for all of them)."""
    torch = torch_cuda()
    u = synth.uniform_field(nx, ny, nz, seed=1000 + nx + R)
    c = np.random.default_rng(R).uniform(-1, 1, R + 1)
    out = run_apply(torch, u, c, R, path=path)
    check(u, out, c, R)


@pytest.mark.parametrize("dims,R,want", [((64, 64, 64), 1, "direct"), ((448, 448, 448), 1, "direct"),
                                         ((480, 480, 480), 1, "staged"), ((224, 224, 224), 2, "direct"),
                                         ((232, 232, 232), 2, "staged"), ((168, 168, 168), 3, "direct"),
                                         ((172, 172, 172), 3, "staged"), ((148, 148, 148), 4, "direct"),
                                         ((152, 152, 152), 4, "staged"), ((512, 512, 512), 4, "staged")])
def test_automatic_sweep_path(dims, R, want):
    """The automatic choice: the direct kernel up to 100, 12, 5 and 3.5 million points for
    radius 1..4; launch_info reports the chosen kernel's launch."""
    torch_cuda()
    plan = StencilPlan(*dims, R, np.ones(R + 1, np.float32))
    assert plan.sweep_path == want
    info = plan.launch_info(0)
    if want == "direct":
        nx, ny, nz = dims
        cols = ((nx - R - 1) >> 2) + 1 - (R >> 2)
        assert info["grid"] == -(-cols * (ny - 2 * R) * (nz - 2 * R) // 256)
        assert (info["threads"], info["smem"], info["tiles"], info["zchunks"]) == (256, 0, 0, 0)
    else:
        assert info["smem"] > 0 and info["tiles"] > 0
    plan.set_sweep_path("staged" if want == "direct" else "direct")
    assert plan.sweep_path != want
    plan.set_sweep_path("auto")
    assert plan.sweep_path == want
    with pytest.raises(StencilError) as ei:
        plan.set_sweep_path(3)
    assert ei.value.code == -1
    with pytest.raises(ValueError):
        plan.set_sweep_path("fast")
    plan.close()


@pytest.mark.parametrize("R", [1, 4])
def test_laplacian_coefficients(R):
    torch = torch_cuda()
    c = synth.laplacian8_coeffs() if R == 4 else synth.laplacian2_coeffs()
    u = synth.uniform_field(192, 80, 50)
    check(u, run_apply(torch, u, c, R), c, R)


def test_empty_interior_is_noop():
    torch = torch_cuda()
    u = synth.uniform_field(8, 8, 8)
    out = run_apply(torch, u, synth.laplacian8_coeffs(), 4)
    assert np.all(out.view(np.uint32) == 0x7FC0DEAD)


@pytest.mark.parametrize("nx,ny,nz,R", [(1024, 1024, 20, 1), (2048, 512, 24, 2), (1024, 1024, 30, 3)])
def test_several_items_per_cta(nx, ny, nz, R):
    """More work items than resident CTAs: each CTA streams several tiles in turn, and the
    ring's refills run from one item into the next (the radii 1-3 release slots warp by
    warp and locate each refill themselves)."""
    torch = torch_cuda()
    u = synth.uniform_field(nx, ny, nz, seed=3000 + R)
    c = np.random.default_rng(20 + R).uniform(-1, 1, R + 1)
    plan = StencilPlan(nx, ny, nz, R, c)
    plan.set_sweep_path("staged")
    info = plan.launch_info(0)
    assert info["tiles"] * info["zchunks"] > info["grid"], info  # several items per CTA
    plan.close()
    out = run_apply(torch, u, c, R, path="staged")
    check(u, out, c, R)


def test_star7_avg_64_shell_copied():
    """7-point smoothing on 64^3 with the shell copied from the input."""
    torch = torch_cuda()
    u = synth.uniform_field(64, 64, 64)
    c = synth.average7_coeffs()
    out = run_apply(torch, u, c, 1, shell_from_input=True)
    check(u, out, c, 1, shell_bits=u)


def test_constant_field_and_checkerboard():
    torch = torch_cuda()
    c = synth.laplacian8_coeffs()
    u = np.full((40, 36, 72), 0.75, np.float32)
    out = run_apply(torch, u, c, 4)
    m = interior_mask(u.shape, 4)
    assert np.max(np.abs(out[m])) <= 1e-6 * 19.51
    z, y, x = np.meshgrid(*[np.arange(n) for n in u.shape], indexing="ij")
    cb = np.where((x + y + z) % 2 == 0, 1.0, -1.0).astype(np.float32)
    out = run_apply(torch, cb, c, 4)
    np.testing.assert_allclose(out[m], -2048.0 / 105.0 * cb[m], rtol=0, atol=1e-4)


def test_star25_512_full_grid():
    """The 25-point 8th-order Laplacian at 512^3, every interior point against the oracle."""
    torch = torch_cuda()
    u = synth.uniform_field(512, 512, 512)
    c = synth.laplacian8_coeffs()
    out = run_apply(torch, u, c, 4)
    err = check(u, out, c, 4)
    print(f"star25 512^3: max |gpu - oracle| = {err:.3e}")


def _sweeps(torch, u0, c, R, nsweeps, check_at, samples, planes):
    """Ping-pong sweeps on the GPU; at the listed sweeps check the GPU's own input/output
    pair at sampled points against the oracle (per-sweep gate)."""
    nz, ny, nx = u0.shape
    plan = StencilPlan(nx, ny, nz, R, c)
    a = torch.from_numpy(u0.ravel()).cuda()
    b = a.clone()
    c32 = np.asarray(c, np.float32)
    idx = sample_interior(u0.shape, R, samples, planes=planes)
    worst, report = 0.0, []
    for k in range(nsweeps):
        host_in = a.cpu().numpy().reshape(u0.shape) if k in check_at else None
        plan.apply(a, b)
        if host_in is not None:
            plan.status(None, b)
            amax = float(np.max(np.abs(host_in)))
            got = b.cpu().numpy()[idx]
            if amax <= 1e30:
                want = oracle.apply_points(host_in, c32, R, idx)
                err = float(np.max(np.abs(got.astype(np.float64) - want)))
                tol = sweep_tol(c32, host_in)
                assert err <= tol, f"sweep {k}: {err} > {tol}"
                worst = max(worst, err / tol)
            report.append((k, amax))
        a, b = b, a
    plan.status(None, a)
    host = a.cpu().numpy().reshape(u0.shape)
    m = interior_mask(u0.shape, R)
    np.testing.assert_array_equal(host[~m], u0[~m])  # fixed shell
    plan.close()
    return worst, report, host


def test_star7_lap_512_ten_sweeps():
    torch = torch_cuda()
    u0 = synth.uniform_field(512, 512, 512)
    worst, report, _ = _sweeps(torch, u0, synth.laplacian2_coeffs(), 1, 10, set(range(10)),
                               200000, planes=(1, 255, 510))
    print(f"star7 512^3 x10: worst err/tol {worst:.3f}; max|u_in| per sweep {report}")


def test_star25_1536x1536x256_fifty_sweeps():
    """50 ping-pong sweeps; gated while max|u_in| <= 1e30 (fp32 overflows near sweep 33)."""
    torch = torch_cuda()
    u0 = synth.sinusoid_field(1536, 1536, 256)
    worst, report, final = _sweeps(torch, u0, synth.laplacian8_coeffs(), 4, 50,
                                   {0, 1, 2, 10, 20, 29, 30, 31}, 100000, planes=(4, 128, 251))
    print(f"star25 1536x1536x256 x50: worst err/tol {worst:.3f}; max|u_in| {report}; "
          f"final finite fraction {np.isfinite(final).mean():.4f}")


def test_star25_1536x1536x256_sweep_time_is_value_independent():
    """The 50-sweep run overflows to inf and then NaN; the sweep time must not change with
    the values (no slow path for non-finite or subnormal operands): the median time of
    sweeps 1-30 (finite) against that of sweeps 35-50 (inf / NaN)."""
    torch = torch_cuda()
    nx, ny, nz, R = 1536, 1536, 256, 4
    u0 = synth.sinusoid_field(nx, ny, nz)
    plan = StencilPlan(nx, ny, nz, R, synth.laplacian8_coeffs())
    a = torch.from_numpy(u0.ravel()).cuda()
    b = a.clone()
    del u0
    s = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    finite = []
    for k in range(50):
        if k in (30, 34):
            finite.append((k, bool(torch.isfinite(a).all())))
        ev[k][0].record(s)
        plan.apply(a, b, s)
        ev[k][1].record(s)
        a, b = b, a
    plan.status(s)
    ms = [x.elapsed_time(y) for x, y in ev]
    early, late = float(np.median(ms[0:30])), float(np.median(ms[34:50]))
    print(f"star25 1536x1536x256: median ms per sweep, sweeps 1-30 {early:.4f}, 35-50 {late:.4f}; "
          f"input finite at sweeps {finite}")
    assert finite == [(30, True), (34, False)]  # the late sweeps really run on inf / NaN
    assert 0.9 < late / early < 1.1
    plan.close()


def test_host_buffer_entry_matches_device_path():
    torch = torch_cuda()
    nx, ny, nz, R = 136, 75, 41, 4
    u = synth.uniform_field(nx, ny, nz)
    c = synth.laplacian8_coeffs()
    plan = StencilPlan(nx, ny, nz, R, c)
    out_h = np.empty_like(u)
    plan.apply_host(u, out_h, 3)
    a = torch.from_numpy(u.ravel()).cuda()
    b = a.clone()
    for _ in range(3):
        plan.apply(a, b)
        a, b = b, a
    plan.status(None, a)
    np.testing.assert_array_equal(out_h.ravel(), a.cpu().numpy())
    plan.apply_host(u, out_h, 0)
    np.testing.assert_array_equal(out_h, u)
    plan.close()


def test_launch_geometry():
    torch_cuda()
    plan = StencilPlan(512, 512, 512, 4, synth.laplacian8_coeffs())
    info = plan.launch_info(0)
    assert 1 <= info["grid"] <= info["sms"] * info["ctas_per_sm"]
    assert info["grid"] <= info["tiles"] * info["zchunks"]
    assert info["tile_x"] == 64
    plan.close()


@pytest.mark.parametrize("use_graph", [False, True])
@pytest.mark.parametrize("nsweeps", [3, 4])
@pytest.mark.parametrize("path", ["staged", "direct"])
def test_native_sweep_loop_matches_launch_by_launch(use_graph, nsweeps, path):
    torch = torch_cuda()
    nx, ny, nz, R = 136, 75, 41, 4
    c = synth.laplacian8_coeffs()
    u = synth.uniform_field(nx, ny, nz)
    plan = StencilPlan(nx, ny, nz, R, c)
    plan.set_sweep_path(path)
    a = torch.from_numpy(u.ravel()).cuda()
    b = a.clone()
    ra, rb = a.clone(), a.clone()
    for _ in range(2):  # the second call replays the cached graph
        a.copy_(ra)
        b.copy_(ra)
        plan.sweeps(a, b, nsweeps, use_graph=use_graph)
        plan.status(None, a)
    x, y = ra, rb
    for _ in range(nsweeps):
        plan.apply(x, y)
        x, y = y, x
    plan.status(None, x)
    got = a if nsweeps % 2 == 0 else b
    assert torch.equal(got, x)
    plan.close()


@pytest.mark.parametrize("path", ["staged", "direct"])
@pytest.mark.parametrize("dims,R", [((136, 75, 200), 4), ((64, 40, 140), 1), ((32, 32, 20), 4)])
def test_pipelined_host_sweep_matches_device_path(dims, R, path):
    """One host-to-host sweep runs pipelined over z-slabs (each slab a z-range launch of
    the plan's sweep kernel); it must equal the device path."""
    torch = torch_cuda()
    nx, ny, nz = dims
    c = synth.laplacian8_coeffs()[:R + 1] if R == 4 else synth.laplacian2_coeffs()
    u = synth.uniform_field(nx, ny, nz, seed=77)
    plan = StencilPlan(nx, ny, nz, R, c)
    plan.set_sweep_path(path)
    out_h = np.full_like(u, 3.0)
    for _ in range(2):
        plan.apply_host(u, out_h, 1)
    a = torch.from_numpy(u.ravel()).cuda()
    b = a.clone()
    plan.apply(a, b)
    plan.status(None, b)
    np.testing.assert_array_equal(out_h.ravel(), b.cpu().numpy())
    plan.close()


def test_grid_beyond_2pow31_points():
    """64-bit indexing: 2048 x 1024 x 1030 = 2.16e9 points (8.6 GB per field), on both
    sweep kernels (the direct one forced: the automatic choice is the staged one here)."""
    torch = torch_cuda()
    nx, ny, nz, R = 2048, 1024, 1030, 4
    if torch.cuda.get_device_properties(0).total_memory < 40 * 2 ** 30:
        pytest.skip("needs ~20 GB of device memory")
    c = synth.laplacian8_coeffs()
    u = synth.uniform_field(nx, ny, nz, seed=99)
    plan = StencilPlan(nx, ny, nz, R, c)
    assert plan.sweep_path == "staged"
    a = torch.from_numpy(u.ravel()).cuda()
    idx = sample_interior(u.shape, R, 200000, seed=3)
    top = (nz - R - 1) * nx * ny + (ny - R - 1) * nx + np.arange(R, nx - R, dtype=np.int64)  # last interior row
    idx = np.unique(np.concatenate([idx, top]))
    assert idx.max() > 2 ** 31
    want = oracle.apply_points(u, c.astype(np.float32), R, idx)
    for path in ("staged", "direct"):
        plan.set_sweep_path(path)
        b = torch.full_like(a, 5.0)
        plan.apply(a, b)
        plan.status(None, b)
        got = b[torch.from_numpy(idx).cuda()].cpu().numpy()
        assert np.max(np.abs(got.astype(np.float64) - want)) <= sweep_tol(c, u), path
        last = b[(nz - 1) * nx * ny:].cpu().numpy()
        assert np.all(last == 5.0), path  # the shell's last plane is untouched
        del b
    plan.close()


def test_two_plans_on_two_streams_concurrently():
    """Plans own their state; sweeps of two plans overlapping on two streams are unaffected."""
    torch = torch_cuda()
    dims = [(136, 75, 120, 4), (200, 64, 90, 1)]
    plans, ins, outs, refs = [], [], [], []
    for nx, ny, nz, R in dims:
        c = synth.laplacian8_coeffs() if R == 4 else synth.laplacian2_coeffs()
        u = synth.uniform_field(nx, ny, nz, seed=nx + R)
        plans.append(StencilPlan(nx, ny, nz, R, c))
        ins.append(torch.from_numpy(u.ravel()).cuda())
        outs.append(ins[-1].clone())
        ref = ins[-1].clone()
        plans[-1].apply(ins[-1], ref)
        plans[-1].status(None, ref)
        refs.append(ref)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(20):
        for p, a, b, s in zip(plans, ins, outs, streams):
            p.apply(a, b, s)
    for p, b, ref, s in zip(plans, outs, refs, streams):
        p.status(s)
        assert torch.equal(b, ref)
        p.close()


TWO_SWEEP_CASES = [(136, 75, 41), (64, 64, 64), (4, 5, 6), (8, 40, 7), (200, 33, 17), (68, 130, 30),
                   (512, 62, 9), (132, 31, 3), (260, 94, 70)]


@pytest.mark.parametrize("nx,ny,nz", TWO_SWEEP_CASES)
def test_two_sweeps_in_one_pass_match_oracle(nx, ny, nz):
    """stencil_apply2 (radius 1): S(S(u)) in one pass, against two oracle sweeps with a fixed
    shell; ragged tiles in x and y (30-row tiles), short z, the shell and guard bands kept."""
    torch = torch_cuda()
    u = synth.uniform_field(nx, ny, nz, seed=4000 + nx + ny + nz)
    c = np.random.default_rng(nx + nz).uniform(-1, 1, 2)
    c = (c / (abs(c[0]) + 6.0 * abs(c[1]))).astype(np.float32)  # max-norm gain 1
    plan = StencilPlan(nx, ny, nz, 1, c)
    gin = Guarded(torch, u)
    gout = Guarded(torch, u, fill_sentinel=True)
    plan.apply2(gin.ptr, gout.ptr)
    plan.status()
    got = gout.numpy()
    assert gin.guards_intact() and gout.guards_intact()
    np.testing.assert_array_equal(gin.numpy(), u)
    plan.close()
    want = oracle.run_sweeps(u, c, 1, 2)
    m = interior_mask(u.shape, 1)
    if m.any():
        assert np.max(np.abs(got[m].astype(np.float64) - want[m])) <= 2e-5 * float(np.max(np.abs(u)))
    assert np.all(got.view(np.uint32)[~m] == 0x7FC0DEAD), "shell written"


@pytest.mark.parametrize("path", ["staged", "direct"])
@pytest.mark.parametrize("nsweeps", [2, 5, 6, 9, 10])
def test_radius1_sweep_loops_with_two_sweep_passes_match_oracle(nsweeps, path):
    """stencil_sweeps at radius 1 on the staged path runs 2*floor(n/4) two-sweep passes plus
    single sweeps, on the direct path n single sweeps; the result lands in the buffer the
    sweep count says, and matches the oracle's loop."""
    torch = torch_cuda()
    nx, ny, nz = 200, 97, 45
    u0 = synth.uniform_field(nx, ny, nz, seed=77)
    c = np.float32([-0.5, 1.0 / 12.0])
    plan = StencilPlan(nx, ny, nz, 1, c)
    plan.set_sweep_path(path)
    for use_graph in (False, True):
        a = torch.from_numpy(u0.ravel()).cuda()
        b = a.clone()
        plan.sweeps(a, b, nsweeps, use_graph=use_graph)
        plan.status(None, a)
        got = (a if nsweeps % 2 == 0 else b).cpu().numpy().reshape(u0.shape)
        want = oracle.run_sweeps(u0, c, 1, nsweeps)
        m = interior_mask(u0.shape, 1)
        assert np.max(np.abs(got[m].astype(np.float64) - want[m])) <= nsweeps * 1e-5 * float(np.max(np.abs(u0)))
        np.testing.assert_array_equal(got[~m], u0[~m])
    plan.close()


def test_two_sweep_pass_only_for_radius_1():
    torch = torch_cuda()
    plan = StencilPlan(64, 64, 64, 4, synth.laplacian8_coeffs())
    a = torch.zeros(64 ** 3, device="cuda")
    b = torch.zeros(64 ** 3, device="cuda")
    with pytest.raises(Exception) as ei:
        plan.apply2(a, b)
    assert "radius 1" in str(ei.value)
    plan.close()


def test_star7_lap_512_ten_sweeps_as_two_sweep_passes():
    """The 10-sweep 512^3 7-point workload as five two-sweep passes (stencil_apply2).  Each
    pass is checked on the GPU's own input v: with |S(w) - exact| <= 1e-5 sum|c| max|w| per
    sweep and S's max-norm gain g = |c0| + 6|c1|, a pass is within 2e-5 sum|c| g max|v| of
    S(S(v)), at sampled points and on three whole planes."""
    torch = torch_cuda()
    n = 512
    u0 = synth.uniform_field(n, n, n)
    c = synth.laplacian2_coeffs()
    c32 = np.asarray(c, np.float32)
    sc = float(np.sum(np.abs(c32)))
    gain = abs(float(c32[0])) + 6.0 * abs(float(c32[1]))
    plan = StencilPlan(n, n, n, 1, c)
    a = torch.from_numpy(u0.ravel()).cuda()
    b = a.clone()
    idx = sample_interior(u0.shape, 1, 200000, seed=5, planes=(1, 255, 510))
    worst = 0.0
    for k in range(5):
        v = a.cpu().numpy().reshape(u0.shape)
        plan.apply2(a, b)
        plan.status(None, b)
        s1 = oracle.apply(v, c32, 1)  # the first sweep, shell copied from v
        want = oracle.apply_points(s1, c32, 1, idx)
        got = b.cpu().numpy()[idx]
        tol = 2e-5 * sc * gain * float(np.max(np.abs(v)))
        err = float(np.max(np.abs(got.astype(np.float64) - want)))
        assert err <= tol, f"pass {k}: {err} > {tol}"
        worst = max(worst, err / tol)
        a, b = b, a
    host = a.cpu().numpy().reshape(u0.shape)
    m = interior_mask(u0.shape, 1)
    np.testing.assert_array_equal(host[~m], u0[~m])
    plan.close()
    print(f"star7 512^3 x10 as two-sweep passes: worst err/tol {worst:.3f}")


def test_sweep_path_change_recaptures_the_loop_graph():
    """The cached graph of stencil_sweeps belongs to one sweep path: after a change of path
    the next call captures the new kernel's loop, and both results match the oracle."""
    torch = torch_cuda()
    nx, ny, nz, R = 96, 50, 40, 2
    u0 = synth.uniform_field(nx, ny, nz, seed=5)
    c = np.float32([0.4, 0.05, -0.025])
    plan = StencilPlan(nx, ny, nz, R, c)
    want = oracle.run_sweeps(u0, c, R, 3)
    m = interior_mask(u0.shape, R)
    for path in ("direct", "staged", "direct"):
        plan.set_sweep_path(path)
        a = torch.from_numpy(u0.ravel()).cuda()
        b = a.clone()
        plan.sweeps(a, b, 3, use_graph=True)
        plan.status(None, a)
        got = b.cpu().numpy().reshape(u0.shape)
        assert np.max(np.abs(got[m].astype(np.float64) - want[m])) <= 3e-5 * float(np.max(np.abs(u0)))
        np.testing.assert_array_equal(got[~m], u0[~m])
    plan.close()
