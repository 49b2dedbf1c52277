"""The z-slab decomposition on one GPU (stencil_slabs_*) against the CPU oracle.

The grid is cut into slabs along z, each stored as its own device array with ghost
planes; a sweep or step of the whole grid exchanges ghost planes between the slab arrays
and runs the kernels on every slab, the planes away from the cuts overlapped with the
exchange.  Put back together, the owned planes must match the oracle's run on the whole
grid, and the exchange must deliver every ghost plane bit for bit from its owner.
"""
import numpy as np
import pytest

import oracle
from seismic_wave_propagation_gb300 import StencilError, StencilSlabs, synth, zslab
from gpu_util import interior_mask, torch_cuda

pytestmark = pytest.mark.gpu


def to_slabs(torch, slabs, field):
    out = []
    for k in range(slabs.nslabs):
        e = slabs.extent(k)
        out.append(torch.from_numpy(np.ascontiguousarray(field[e["begin"]:e["end"]]).ravel()).cuda())
    return out


def from_slabs(slabs, arrays, shape):
    nz, ny, nx = shape
    parts = []
    for k, a in enumerate(arrays):
        e = slabs.extent(k)
        h = a.cpu().numpy().reshape(e["end"] - e["begin"], ny, nx)
        parts.append(h[e["own_begin"] - e["begin"]:e["own_end"] - e["begin"]])
    return np.concatenate(parts)


@pytest.mark.parametrize("dims,R,P", [((136, 75, 41), 4, 2), ((200, 33, 97), 4, 3), ((68, 130, 60), 1, 4),
                                      ((96, 40, 12), 3, 4), ((128, 64, 257), 4, 7), ((64, 64, 64), 2, 1)])
def test_partition_matches_the_rank_schedule(dims, R, P):
    torch_cuda()
    nx, ny, nz = dims
    slabs = StencilSlabs(nx, ny, nz, R, synth.laplacian8_coeffs()[:R + 1], P)
    want = zslab.partition(nz, P, R)
    for k in range(P):
        e = slabs.extent(k)
        assert (e["begin"], e["end"], e["own_begin"], e["own_end"]) == (
            want[k]["begin"], want[k]["end"], want[k]["own_begin"], want[k]["own_end"])
    slabs.close()


@pytest.mark.parametrize("dims,R,P", [((136, 75, 41), 4, 2), ((200, 33, 97), 4, 3), ((68, 130, 60), 1, 4),
                                      ((128, 64, 257), 4, 7)])
def test_exchange_delivers_every_ghost_plane(dims, R, P):
    torch = torch_cuda()
    nx, ny, nz = dims
    u = synth.uniform_field(nx, ny, nz, seed=41)
    slabs = StencilSlabs(nx, ny, nz, R, synth.laplacian8_coeffs()[:R + 1], P)
    arrs = to_slabs(torch, slabs, u)
    for k, a in enumerate(arrs):  # stale ghost planes
        e = slabs.extent(k)
        h = a.view(e["end"] - e["begin"], ny, nx)
        h[:e["own_begin"] - e["begin"]] = float("nan")
        h[e["own_end"] - e["begin"]:] = float("nan")
    slabs.exchange(arrs)
    slabs.status(None, *arrs)
    for k, a in enumerate(arrs):
        e = slabs.extent(k)
        np.testing.assert_array_equal(a.cpu().numpy().reshape(-1, ny, nx), u[e["begin"]:e["end"]])
    slabs.close()


@pytest.mark.parametrize("nsweeps", [1, 3])
@pytest.mark.parametrize("dims,R,P", [((136, 75, 41), 4, 2), ((200, 33, 97), 4, 3), ((68, 130, 60), 1, 4),
                                      ((96, 40, 30), 3, 3), ((128, 64, 257), 4, 7), ((64, 64, 64), 2, 1)])
def test_slab_sweeps_match_oracle(dims, R, P, nsweeps):
    torch = torch_cuda()
    nx, ny, nz = dims
    c = synth.laplacian8_coeffs()[:R + 1] if R == 4 else np.random.default_rng(R).uniform(-1, 1, R + 1)
    c = (c / (abs(c[0]) + 6.0 * np.sum(np.abs(c[1:])))).astype(np.float32)  # max-norm gain 1
    u0 = synth.uniform_field(nx, ny, nz, seed=42 + R)
    slabs = StencilSlabs(nx, ny, nz, R, c, P)
    a = to_slabs(torch, slabs, u0)
    b = [x.clone() for x in a]
    for _ in range(nsweeps):
        slabs.apply(a, b)
        a, b = b, a
    slabs.status(None, *a)
    got = from_slabs(slabs, a, u0.shape)
    want = oracle.run_sweeps(u0, c, R, nsweeps)
    m = interior_mask(u0.shape, R)
    tol = nsweeps * 1e-5 * float(np.max(np.abs(u0)))
    assert float(np.max(np.abs(got[m].astype(np.float64) - want[m]))) <= tol
    np.testing.assert_array_equal(got[~m], u0[~m])
    slabs.close()


@pytest.mark.parametrize("two_buffers", [False, True])
@pytest.mark.parametrize("P", [2, 5])
def test_slab_wave_steps_match_oracle(P, two_buffers):
    torch = torch_cuda()
    nx, ny, nz, steps = 96, 80, 72, 20
    up, u, s, e = synth.wave_fields(nx, ny, nz)
    c = synth.laplacian8_coeffs()
    slabs = StencilSlabs(nx, ny, nz, 4, c, P)
    prev, cur, vv, ee = [to_slabs(torch, slabs, f) for f in (up, u, s, e)]
    nxt = [x.clone() for x in prev]
    for _ in range(steps):
        if two_buffers:
            slabs.wave_step(prev, cur, prev, vv, ee)
            prev, cur = cur, prev
        else:
            slabs.wave_step(prev, cur, nxt, vv, ee)
            prev, cur, nxt = cur, nxt, prev
    slabs.status(None, *cur)
    got = from_slabs(slabs, cur, u.shape)
    o_prev, o_cur = oracle.run_wave(up, u, s, e, c.astype(np.float32), 4, steps)
    rel = np.linalg.norm((got.astype(np.float64) - o_cur).ravel()) / np.linalg.norm(o_cur.ravel())
    assert rel <= 1e-5
    slabs.close()


def test_slab_argument_errors():
    torch = torch_cuda()
    c = synth.laplacian8_coeffs()
    with pytest.raises(StencilError):
        StencilSlabs(64, 64, 12, 4, c, 4)  # slabs of 3 planes < R
    with pytest.raises(StencilError):
        StencilSlabs(64, 64, 64, 4, c, 0)
    slabs = StencilSlabs(64, 32, 40, 4, c, 2)
    u = synth.uniform_field(64, 32, 40)
    a = to_slabs(torch, slabs, u)
    with pytest.raises(StencilError) as ei:
        slabs.apply(a, a)  # in and out the same arrays
    assert ei.value.code == -3
    with pytest.raises(ValueError):
        slabs.apply(a[:1], a[:1])
    slabs.close()
