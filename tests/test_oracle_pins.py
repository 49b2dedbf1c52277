"""Pins for the CPU oracle: each test checks it against something other than itself.

The oracle computes the star stencil of "Accelerating High-Order Stencils on GPUs"
(3D blocking with global memory) / "Thread Coarsening 與 Register Tiling" (Fig 8.10)
and the acoustic update with a pointwise sponge. The checks below come from linear
algebra (Kronecker-sum operator), a library routine (scipy.ndimage.correlate), closed
forms (polynomial exactness and the exact truncation error, plane-wave eigenvalues,
the checkerboard eigenvalue, the exact discrete leapfrog solution of an eigenmode,
damped or not) and invariants (linearity, axis symmetry, untouched shell).
"""
import math

import numpy as np
import pytest
import scipy.sparse as sp
from scipy import ndimage

from seismic_wave_propagation_gb300 import synth

LAP8 = synth.laplacian8_coeffs()
LAP2 = synth.laplacian2_coeffs()


def rng(seed=1):
    return np.random.default_rng(seed)


def interior(shape, R):
    nz, ny, nx = shape
    m = np.zeros(shape, dtype=bool)
    m[R:nz - R, R:ny - R, R:nx - R] = True
    return m


def kron_operator(nx, ny, nz, coeffs):
    """Kronecker-sum form: a banded matrix per axis, centre weight split over the axes."""
    R = len(coeffs) - 1

    def band(n):
        diags, offs = [np.full(n, coeffs[0] / 3.0)], [0]
        for r in range(1, R + 1):
            diags += [np.full(n - r, coeffs[r]), np.full(n - r, coeffs[r])]
            offs += [r, -r]
        return sp.diags(diags, offs, shape=(n, n), format="csr")

    ix, iy, iz = sp.identity(nx), sp.identity(ny), sp.identity(nz)
    op = (sp.kron(iz, sp.kron(iy, band(nx))) + sp.kron(iz, sp.kron(band(ny), ix))
          + sp.kron(band(nz), sp.kron(iy, ix)))
    return op.tocsr()


def star_kernel(coeffs):
    R = len(coeffs) - 1
    k = np.zeros((2 * R + 1,) * 3)
    k[R, R, R] = coeffs[0]
    for r in range(1, R + 1):
        for s in (R - r, R + r):
            k[s, R, R] = k[R, s, R] = k[R, R, s] = coeffs[r]
    return k


@pytest.mark.parametrize("R,shape", [(1, (6, 7, 8)), (2, (7, 9, 8)), (3, (9, 8, 10)), (4, (10, 11, 12)),
                                     (4, (13, 9, 16))])
def test_matches_kronecker_sum_operator(oracle_mod, R, shape):
    c = rng(R).uniform(-2, 2, R + 1)
    u = rng(10 + R).standard_normal(shape)
    nz, ny, nx = shape
    ref = (kron_operator(nx, ny, nz, c) @ u.ravel()).reshape(shape)
    out = oracle_mod.apply(u, c, R)
    m = interior(shape, R)
    np.testing.assert_allclose(out[m], ref[m], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(out[~m], u[~m])


@pytest.mark.parametrize("R", [1, 2, 3, 4])
def test_matches_ndimage_correlate(oracle_mod, R):
    shape = (2 * R + 5, 2 * R + 4, 2 * R + 7)
    c = rng(20 + R).uniform(-1, 1, R + 1)
    u = rng(30 + R).standard_normal(shape)
    ref = ndimage.correlate(u, star_kernel(c), mode="constant", cval=0.0)
    out = oracle_mod.apply(u, c, R, out=np.zeros_like(u))
    m = interior(shape, R)
    np.testing.assert_allclose(out[m], ref[m], rtol=0, atol=1e-12)


def test_brute_force_neighbour_sum_8cube(oracle_mod):
    """R=1 on an 8^3 grid (interior 6^3): sum over an explicit offset list."""
    u = rng(3).standard_normal((8, 8, 8))
    c = [0.7, -0.3]
    offsets = [(0, 0, 0, 0)] + [(dz, dy, dx, 1) for dz, dy, dx in
                                [(1, 0, 0), (-1, 0, 0), (0, 1, 0), (0, -1, 0), (0, 0, 1), (0, 0, -1)]]
    out = oracle_mod.apply(u, c, 1)
    for z in range(1, 7):
        for y in range(1, 7):
            for x in range(1, 7):
                want = sum(c[w] * u[z + dz, y + dy, x + dx] for dz, dy, dx, w in offsets)
                assert abs(out[z, y, x] - want) < 1e-13


def test_empty_interior_is_a_noop(oracle_mod):
    u = rng(4).standard_normal((8, 8, 8)).astype(np.float32)
    out = np.full_like(u, 7.0)
    oracle_mod.apply(u, LAP8.astype(np.float32), 4, out=out)
    assert np.all(out == 7.0)


def _monomial(shape, a, b, c, scale):
    nz, ny, nx = shape
    z, y, x = np.meshgrid(*[(np.arange(n) - (n - 1) / 2.0) / scale for n in (nz, ny, nx)], indexing="ij")
    return x, y, z, x ** a * y ** b * z ** c


def _lap_monomial(x, y, z, a, b, c, scale):
    t = 0.0
    if a >= 2:
        t = t + a * (a - 1) * x ** (a - 2) * y ** b * z ** c
    if b >= 2:
        t = t + b * (b - 1) * x ** a * y ** (b - 2) * z ** c
    if c >= 2:
        t = t + c * (c - 1) * x ** a * y ** b * z ** (c - 2)
    return t / scale ** 2 + 0 * x


@pytest.mark.parametrize("R,coeffs,maxdeg", [(4, LAP8, 9), (1, LAP2, 3)])
def test_polynomial_exactness(oracle_mod, R, coeffs, maxdeg):
    """Each axis' stencil differentiates polynomials up to degree 2R+1 exactly (h = 1)."""
    shape, scale = (2 * R + 9, 2 * R + 8, 2 * R + 10), 2.0 * R + 5
    m = interior(shape, R)
    degs = [(a, b, c) for a in range(maxdeg + 1) for b in range(maxdeg + 1) for c in range(maxdeg + 1)
            if (a + b + c) % 3 == 0 or max(a, b, c) == maxdeg]
    for a, b, c in degs:
        x, y, z, u = _monomial(shape, a, b, c, scale)
        out = oracle_mod.apply(u, coeffs, R)
        want = _lap_monomial(x, y, z, a, b, c, scale)
        err = np.max(np.abs(out[m] - want[m]))
        assert err < 1e-12, (a, b, c, err)


@pytest.mark.parametrize("R,coeffs,order", [(4, LAP8, 8), (1, LAP2, 2)])
def test_leading_truncation_error(oracle_mod, R, coeffs, order):
    """On x^(order+2) the error is exactly the leading term 2 (p!)^2/(2p+2)! * f^(2p+2), p = order/2.

    (1/12 for the 3-point and 1/3150 for the 9-point second-difference weights.)
    """
    p = order // 2
    k = order + 2
    shape, scale = (2 * R + 3, 2 * R + 3, 2 * R + 12), 6.0
    x, y, z, u = _monomial(shape, k, 0, 0, scale)
    out = oracle_mod.apply(u, coeffs, R)
    m = interior(shape, R)
    err = out[m] - (k * (k - 1) * x ** (k - 2) / scale ** 2)[m]
    const = 2.0 * math.factorial(p) ** 2 / math.factorial(2 * p + 2) * math.factorial(k) / scale ** k
    np.testing.assert_allclose(np.abs(err), const, rtol=1e-6)
    assert np.ptp(err) < 1e-9 * const + 1e-13


@pytest.mark.parametrize("R", [1, 2, 4])
def test_plane_wave_eigenvalue(oracle_mod, R):
    c = rng(40 + R).uniform(-1, 1, R + 1)
    shape = (2 * R + 6, 2 * R + 7, 2 * R + 8)
    th = np.array([0.37, 1.1, 2.3])
    z, y, x = np.meshgrid(*[np.arange(n, dtype=float) for n in shape], indexing="ij")
    u = np.cos(th[0] * x + th[1] * y + th[2] * z + 0.4)
    lam = c[0] + 2.0 * sum(c[r] * sum(math.cos(r * t) for t in th) for r in range(1, R + 1))
    out = oracle_mod.apply(u, c, R)
    m = interior(shape, R)
    np.testing.assert_allclose(out[m], lam * u[m], rtol=0, atol=1e-12)


def test_modified_wavenumber_of_8th_order(oracle_mod):
    """Small wave numbers: lambda = -|k|^2 up to O(k^10)."""
    shape = (16, 16, 16)
    th = np.array([0.05, 0.08, 0.11])
    z, y, x = np.meshgrid(*[np.arange(n, dtype=float) for n in shape], indexing="ij")
    u = np.cos(th[0] * x + th[1] * y + th[2] * z)
    out = oracle_mod.apply(u, LAP8, 4)
    m = interior(shape, 4)
    np.testing.assert_allclose(out[m], -np.sum(th ** 2) * u[m], rtol=0, atol=1e-13)


@pytest.mark.parametrize("R,coeffs,lam", [(4, LAP8, -2048.0 / 105.0), (1, LAP2, -12.0)])
def test_checkerboard_eigenvalue(oracle_mod, R, coeffs, lam):
    shape = (12, 13, 14)
    z, y, x = np.meshgrid(*[np.arange(n) for n in shape], indexing="ij")
    u = np.where((x + y + z) % 2 == 0, 1.0, -1.0)
    out = oracle_mod.apply(u, coeffs, R)
    m = interior(shape, R)
    np.testing.assert_allclose(out[m], lam * u[m], rtol=0, atol=1e-13)
    assert abs(np.sum(np.abs(coeffs[1:])) * 6 + abs(coeffs[0]) + lam) < 1e-13


def _golden_gpuflight():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "gpuflight_7pt.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    R, c0, c1 = rows[0]
    return int(R), [float(c0), float(c1)]


@pytest.mark.parametrize("R,coeffs,gain", [(4, LAP8, 0.0), (1, LAP2, 0.0),
                                           (1, list(synth.average7_coeffs()), 1.0),
                                           (1, _golden_gpuflight()[1], 1.0)])
def test_constant_field(oracle_mod, R, coeffs, gain):
    u = np.full((11, 12, 13), 0.625)
    out = oracle_mod.apply(u, coeffs, R)
    m = interior(u.shape, R)
    np.testing.assert_allclose(out[m], gain * 0.625, rtol=0, atol=1e-14)


@pytest.mark.parametrize("R", [1, 3, 4])
def test_shell_untouched_bitwise(oracle_mod, R):
    shape = (2 * R + 5, 2 * R + 6, 2 * R + 4)
    u = rng(5).uniform(-1, 1, shape).astype(np.float32)
    sentinel = np.array([0x7FC0DEAD], dtype=np.uint32).view(np.float32)[0]
    out = np.full(shape, sentinel, dtype=np.float32)
    c = synth.laplacian8_coeffs()[:R + 1].astype(np.float32)
    oracle_mod.apply(u, c, R, out=out)
    m = interior(shape, R)
    assert np.all(out.view(np.uint32)[~m] == 0x7FC0DEAD)
    assert np.all(np.isfinite(out[m]))


def test_linearity_and_axis_symmetry(oracle_mod):
    u = rng(6).standard_normal((14, 14, 14))
    v = rng(7).standard_normal((14, 14, 14))
    a, b = 0.37, -1.9
    lhs = oracle_mod.apply(a * u + b * v, LAP8, 4, out=np.zeros_like(u))
    rhs = a * oracle_mod.apply(u, LAP8, 4, out=np.zeros_like(u)) + b * oracle_mod.apply(v, LAP8, 4, out=np.zeros_like(u))
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)
    base = oracle_mod.apply(u, LAP8, 4, out=np.zeros_like(u))
    for perm in [(0, 2, 1), (1, 0, 2), (2, 1, 0), (1, 2, 0)]:
        ut = np.ascontiguousarray(u.transpose(perm))
        got = oracle_mod.apply(ut, LAP8, 4, out=np.zeros_like(ut))
        np.testing.assert_allclose(got, base.transpose(perm), rtol=0, atol=1e-12)


def test_f32_entry_is_rounded_f64(oracle_mod):
    shape = (13, 11, 12)
    u = rng(8).uniform(-1, 1, shape).astype(np.float32)
    c32 = LAP8.astype(np.float32)
    got = oracle_mod.apply(u, c32, 4)
    ref = oracle_mod.apply(u.astype(np.float64), c32.astype(np.float64), 4)
    np.testing.assert_array_equal(got, ref.astype(np.float32))
    # wave step likewise
    up = rng(9).uniform(-1, 1, shape).astype(np.float32)
    s = rng(10).uniform(0, 0.2, shape).astype(np.float32)
    e = rng(11).uniform(0, 0.1, shape).astype(np.float32)
    got = oracle_mod.wave_step(up, u, s, e, c32, 4)
    d = lambda a: a.astype(np.float64)  # noqa: E731
    ref = oracle_mod.wave_step(d(up), d(u), d(s), d(e), c32.astype(np.float64), 4)
    np.testing.assert_array_equal(got, ref.astype(np.float32))


def test_points_entry_matches_full_sweep(oracle_mod):
    shape = (15, 14, 16)
    u = rng(12).uniform(-1, 1, shape).astype(np.float32)
    c32 = LAP8.astype(np.float32)
    full = oracle_mod.apply(u, c32, 4)
    m = interior(shape, 4)
    idx = np.flatnonzero(m.ravel())[::7]
    np.testing.assert_array_equal(oracle_mod.apply_points(u, c32, 4, idx), full.ravel()[idx])
    assert np.isnan(oracle_mod.apply_points(u, c32, 4, np.array([0, 3]))).all()
    up = rng(13).uniform(-1, 1, shape).astype(np.float32)
    s = np.full(shape, 0.1, np.float32)
    e = rng(14).uniform(0, 0.1, shape).astype(np.float32)
    full = oracle_mod.wave_step(up, u, s, e, c32, 4)
    np.testing.assert_array_equal(oracle_mod.wave_points(up, u, s, e, c32, 4, idx), full.ravel()[idx])


def test_wave_reduces_to_leapfrog_without_velocity(oracle_mod):
    shape = (12, 12, 12)
    u = rng(15).standard_normal(shape)
    up = rng(16).standard_normal(shape)
    z = np.zeros(shape)
    out = oracle_mod.wave_step(up, u, z, z, LAP8, 4)
    m = interior(shape, 4)
    np.testing.assert_array_equal(out[m], (2.0 * u - up)[m])
    np.testing.assert_array_equal(out[~m], up[~m])


def test_wave_constant_field_is_steady(oracle_mod):
    shape = (12, 13, 12)
    K = np.full(shape, -0.8125)
    s = rng(17).uniform(0, 0.2, shape)
    e = rng(18).uniform(0, 0.1, shape)
    out = oracle_mod.wave_step(K.copy(), K, s, e, LAP8, 4)
    np.testing.assert_allclose(out, K, rtol=0, atol=1e-14)


def _eigenmode(shape, th):
    z, y, x = np.meshgrid(*[np.arange(n, dtype=float) for n in shape], indexing="ij")
    return np.cos(th[0] * x) * np.cos(th[1] * y) * np.cos(th[2] * z)


@pytest.mark.parametrize("eta", [0.0, 0.05])
def test_exact_discrete_leapfrog(oracle_mod, eta):
    """Eigenmode u0 with stencil eigenvalue lam, constant s and eta, u_prev = u = u0.

    The update is the recurrence (1+eta) g[n+1] = (2 + s lam) g[n] - (1-eta) g[n-1] per
    mode, with g[-1] = g[0] = 1; its closed form is A rho1^n + B rho2^n over the roots
    of (1+eta) rho^2 - (2 + s lam) rho + (1-eta). For eta = 0 it is
    cos((n+1/2) phi) / cos(phi/2), cos phi = 1 + s lam / 2. The shell carries the exact
    solution (Dirichlet data), so the whole interior stays exact.
    """
    shape, th, s = (20, 22, 24), (0.7, 1.3, 2.1), 0.2
    lam = sum(LAP8[0] / 3.0 + 2.0 * sum(LAP8[r] * math.cos(r * t) for r in range(1, 5)) for t in th)
    roots = np.roots([1.0 + eta, -(2.0 + s * lam), 1.0 - eta]).astype(complex)
    r1, r2 = roots
    # A + B = 1, A/r1 + B/r2 = 1
    A, B = np.linalg.solve(np.array([[1.0, 1.0], [1.0 / r1, 1.0 / r2]]), np.array([1.0, 1.0]))
    g = lambda n: (A * r1 ** n + B * r2 ** n).real  # noqa: E731
    if eta == 0.0:
        phi = math.acos(1.0 + s * lam / 2.0)
        for n in range(5):
            assert abs(g(n) - math.cos((n + 0.5) * phi) / math.cos(phi / 2)) < 1e-12
    u0 = _eigenmode(shape, th)
    S = np.full(shape, s)
    E = np.full(shape, eta)
    m = interior(shape, 4)
    prev, cur = u0.copy(), u0.copy()
    for n in range(1, 41):
        nxt = oracle_mod.wave_step(prev, cur, S, E, LAP8, 4, u_next=np.empty_like(cur))
        nxt[~m] = g(n) * u0[~m]
        prev, cur = cur, nxt
        np.testing.assert_allclose(cur, g(n) * u0, rtol=0, atol=1e-10)
    assert abs(g(40)) > 1e-3 or eta > 0


def _leapfrog_gain(lam, s, eta):
    """g(n) of the per-mode recurrence (1+eta) g[n+1] = (2 + s lam) g[n] - (1-eta) g[n-1],
    g[-1] = g[0] = 1, evaluated by the recurrence itself in exact rational-free floats."""
    g = {-1: 1.0, 0: 1.0}

    def at(n):
        for k in range(max(g) + 1, n + 1):
            g[k] = ((2.0 + s * lam) * g[k - 1] - (1.0 - eta) * g[k - 2]) / (1.0 + eta)
        return g[n]
    return at


def _face_distance(shape):
    nz, ny, nx = shape
    return np.minimum.reduce(np.meshgrid(np.minimum(np.arange(nz), nz - 1 - np.arange(nz)),
                                         np.minimum(np.arange(ny), ny - 1 - np.arange(ny)),
                                         np.minimum(np.arange(nx), nx - 1 - np.arange(nx)), indexing="ij"))


@pytest.mark.parametrize("R,coeffs,nsteps,shape", [(4, "lap8", 6, (60, 58, 62)),
                                                    (1, "lap2", 17, (48, 46, 44))])
@pytest.mark.parametrize("eta", [0.0, 0.05])
def test_run_wave_time_loop_on_an_eigenmode(oracle_mod, R, coeffs, nsteps, shape, eta):
    """The oracle's own time loop (three-buffer rotation, fixed shell) on an eigenmode.

    run_wave keeps every buffer's shell at its starting value u0, so its levels differ
    from the exact g(n) u0 only where the fixed shell has reached: level n is exact at
    every point at least n*R from the nearest face (level 1 reads only level 0 and its
    shell, which are exact; each later level moves the front R points inward). On that
    core both returned levels must equal g(n-1) u0 and g(n) u0, the per-mode leapfrog
    recurrence; a slip in the rotation (levels swapped, a level reused) breaks it at once.
    Outside the core the fixed shell must have made a difference, or the pin would not
    see the rotation of the shell values either.
    """
    c = LAP8 if coeffs == "lap8" else LAP2
    th, s = (0.7, 1.3, 2.1), 0.2
    lam = sum(c[0] / 3.0 + 2.0 * sum(c[r] * math.cos(r * t) for r in range(1, R + 1)) for t in th)
    g = _leapfrog_gain(lam, s, eta)
    u0 = _eigenmode(shape, th)
    S = np.full(shape, s)
    E = np.full(shape, eta)
    prev, cur = oracle_mod.run_wave(u0, u0, S, E, c, R, nsteps)
    core = _face_distance(shape) >= nsteps * R
    assert core.sum() > 1000
    np.testing.assert_allclose(cur[core], g(nsteps) * u0[core], rtol=0, atol=1e-10)
    np.testing.assert_allclose(prev[core], g(nsteps - 1) * u0[core], rtol=0, atol=1e-10)
    ring = (_face_distance(shape) >= R) & ~core
    assert np.max(np.abs(cur[ring] - g(nsteps) * u0[ring])) > 1e-6
    # the inputs are not modified
    np.testing.assert_array_equal(u0, _eigenmode(shape, th))


def test_run_wave_zero_and_one_step(oracle_mod):
    """Zero steps return the inputs; one step equals one wave_step."""
    shape = (14, 13, 12)
    up = rng(31).uniform(-1, 1, shape)
    u = rng(32).uniform(-1, 1, shape)
    s = rng(33).uniform(0, 0.2, shape)
    e = rng(34).uniform(0, 0.1, shape)
    a, b = oracle_mod.run_wave(up, u, s, e, LAP8, 4, 0)
    np.testing.assert_array_equal(a, up)
    np.testing.assert_array_equal(b, u)
    a, b = oracle_mod.run_wave(up, u, s, e, LAP8, 4, 1)
    np.testing.assert_array_equal(a, u)
    np.testing.assert_array_equal(b, oracle_mod.wave_step(up, u, s, e, LAP8, 4))


def test_eta7_constant_eta_gives_the_pointwise_step(oracle_mod):
    """Weights with e0 + 6 e1 = 1 (the register-rotation lab's 1/4 and 1/8, exact in binary)
    keep a constant eta unchanged, so the step equals the pointwise one bit for bit."""
    shape = (14, 13, 15)
    up = rng(41).uniform(-1, 1, shape)
    u = rng(42).uniform(-1, 1, shape)
    s = rng(43).uniform(0, 0.2, shape)
    K = np.full(shape, 0.0625)
    a = oracle_mod.wave_step_eta7(up, u, s, K, LAP8, 4, 0.25, 0.125)
    b = oracle_mod.wave_step(up, u, s, K, LAP8, 4)
    np.testing.assert_array_equal(a, b)


def test_eta7_centre_weight_alone_is_the_pointwise_step(oracle_mod):
    shape = (13, 14, 12)
    up, u = rng(44).uniform(-1, 1, shape), rng(45).uniform(-1, 1, shape)
    s, e = rng(46).uniform(0, 0.2, shape), rng(47).uniform(0, 0.1, shape)
    np.testing.assert_array_equal(oracle_mod.wave_step_eta7(up, u, s, e, LAP8, 4, 1.0, 0.0),
                                  oracle_mod.wave_step(up, u, s, e, LAP8, 4))


def test_eta7_brute_force(oracle_mod):
    """Every interior point of a small grid from an explicit neighbour list."""
    shape = (10, 11, 9)
    up, u = rng(48).standard_normal(shape), rng(49).standard_normal(shape)
    s, e = rng(50).uniform(0, 0.2, shape), rng(51).uniform(0, 0.1, shape)
    c = [-6.0, 1.0]
    e0, e1 = 0.3, 0.07
    got = oracle_mod.wave_step_eta7(up, u, s, e, c, 1, e0, e1, u_next=np.zeros(shape))
    nbrs = [(1, 0, 0), (-1, 0, 0), (0, 1, 0), (0, -1, 0), (0, 0, 1), (0, 0, -1)]
    for z in range(1, shape[0] - 1):
        for y in range(1, shape[1] - 1):
            for x in range(1, shape[2] - 1):
                lap = c[0] * u[z, y, x] + c[1] * sum(u[z + a, y + b, x + d] for a, b, d in nbrs)
                eff = e0 * e[z, y, x] + e1 * sum(e[z + a, y + b, x + d] for a, b, d in nbrs)
                want = (2 * u[z, y, x] - (1 - eff) * up[z, y, x] + s[z, y, x] * lap) / (1 + eff)
                assert abs(got[z, y, x] - want) < 1e-13


def test_eta7_equals_the_pointwise_step_on_the_smoothed_damping(oracle_mod):
    """Since eta does not change in time, the step is the pointwise step on the damping field
    e0*eta + e1*(six neighbours), which the (pinned) radius-1 stencil computes."""
    shape = (16, 15, 17)
    up, u = rng(52).standard_normal(shape), rng(53).standard_normal(shape)
    s, e = rng(54).uniform(0, 0.2, shape), rng(55).uniform(0, 0.1, shape)
    eff = oracle_mod.apply(e, [0.5, 1.0 / 12.0], 1)
    np.testing.assert_allclose(oracle_mod.wave_step_eta7(up, u, s, e, LAP8, 4, 0.5, 1.0 / 12.0),
                               oracle_mod.wave_step(up, u, s, eff, LAP8, 4), rtol=0, atol=1e-14)
    f = [x.astype(np.float32) for x in (up, u, s, e)]
    eff32 = oracle_mod.apply(f[3], np.float32([0.5, 1.0 / 12.0]), 1)
    a = oracle_mod.wave_step_eta7(f[0], f[1], f[2], f[3], LAP8.astype(np.float32), 4, 0.5, 1.0 / 12.0)
    b = oracle_mod.wave_step(f[0], f[1], f[2], eff32, LAP8.astype(np.float32), 4)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-6)


def test_sweeps_keep_a_fixed_shell(oracle_mod):
    u0 = rng(19).uniform(-1, 1, (10, 11, 12)).astype(np.float32)
    out = oracle_mod.run_sweeps(u0, LAP2.astype(np.float32), 1, 3)
    m = interior(u0.shape, 1)
    np.testing.assert_array_equal(out[~m], u0[~m])
    one = oracle_mod.apply(u0, LAP2.astype(np.float32), 1)
    two = oracle_mod.apply(one, LAP2.astype(np.float32), 1)
    three = oracle_mod.apply(two, LAP2.astype(np.float32), 1)
    np.testing.assert_array_equal(out, three)


def test_planted_sign_error_is_caught(oracle_mod):
    """A flipped neighbour weight (the kind of slip the pins exist for) fails the checkerboard pin."""
    bad = LAP8.copy()
    bad[2] = -bad[2]
    shape = (12, 12, 12)
    z, y, x = np.meshgrid(*[np.arange(n) for n in shape], indexing="ij")
    u = np.where((x + y + z) % 2 == 0, 1.0, -1.0)
    out = oracle_mod.apply(u, bad, 4)
    m = interior(shape, 4)
    assert np.max(np.abs(out[m] - (-2048.0 / 105.0) * u[m])) > 0.1


def test_oracle_regression_fixture(oracle_mod):
    """Bitwise against stored oracle outputs (x86 and Arm give the same bits: no FMA contraction)."""
    import importlib.util
    import os
    here = os.path.join(os.path.dirname(__file__), "golden")
    spec = importlib.util.spec_from_file_location("mk", os.path.join(here, "make_oracle_regression.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    rows = [ln.split() for ln in open(os.path.join(here, "oracle_regression.txt")) if not ln.startswith("#")]
    for kind, R, cname, dims in mk.CASES:
        idx, vals = mk.case_values(kind, R, cname, dims)
        want = {int(r[6]): int(r[7], 16) for r in rows
                if (r[0], int(r[1]), r[2], tuple(map(int, r[3:6]))) == (kind, R, cname, dims)}
        assert len(want) == len(idx)
        for i, v in zip(idx, vals):
            assert int(np.float32(v).view(np.uint32)) == want[int(i)], (kind, cname, i)
