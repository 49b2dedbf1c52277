"""The z-slab decomposition's rank-level exchange on CPU (gloo, world sizes 2 and 3).

Each rank holds one slab of a global field (owned planes plus ghost planes), exchanges
ghost planes with its neighbours through torch.distributed, and sweeps its slab with the
CPU oracle.  The owned planes, put back together, must equal the oracle's sweeps of the
whole grid bit for bit (every point is computed by the same arithmetic from the same
values), and after an exchange every ghost plane must hold its owner's values.
"""
import os
import sys

import numpy as np
import pytest

from seismic_wave_propagation_gb300 import synth, zslab

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("nz,P,R", [(41, 2, 4), (40, 3, 1), (100, 7, 4), (9, 2, 4), (64, 1, 4), (37, 4, 3)])
def test_partition_tiles_the_grid(nz, P, R):
    parts = zslab.partition(nz, P, R)
    assert parts[0]["own_begin"] == 0 and parts[-1]["own_end"] == nz
    for a, b in zip(parts, parts[1:]):
        assert a["own_end"] == b["own_begin"]
    for p in parts:
        assert p["own_end"] - p["own_begin"] >= R
        assert p["begin"] == max(0, p["own_begin"] - R) and p["end"] == min(nz, p["own_end"] + R)


@pytest.mark.parametrize("nz,P,R", [(41, 2, 4), (40, 3, 1), (100, 7, 4), (37, 4, 3)])
def test_messages_fill_every_ghost_plane_once_from_its_owner(nz, P, R):
    parts = zslab.partition(nz, P, R)
    got = {k: [] for k in range(P)}
    for m in zslab.ghost_messages(nz, P, R):
        src, dst = parts[m["src"]], parts[m["dst"]]
        for i in range(m["planes"]):
            g_src = src["begin"] + m["src_plane"] + i
            g_dst = dst["begin"] + m["dst_plane"] + i
            assert g_src == g_dst  # the same global plane
            assert src["own_begin"] <= g_src < src["own_end"]  # sent by its owner
            got[m["dst"]].append(g_dst)
    for k, p in enumerate(parts):
        ghosts = [z for z in range(p["begin"], p["end"]) if not p["own_begin"] <= z < p["own_end"]]
        assert sorted(got[k]) == ghosts


def test_too_many_slabs_rejected():
    with pytest.raises(ValueError):
        zslab.partition(10, 4, 4)


def _worker(rank, world, port, kind, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), OMP_NUM_THREADS="1")
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle
    from seismic_wave_propagation_gb300 import synth as sy, zslab as zs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        nx, ny, nz, R, steps = 24, 20, 41, 4, 3
        c = sy.laplacian8_coeffs().astype(np.float32) / np.float32(20.0)
        part = zs.partition(nz, world, R)[rank]
        b, e = part["begin"], part["end"]
        if kind == "sweep":
            g = sy.uniform_field(nx, ny, nz, seed=3)
            a = torch.from_numpy(g[b:e].copy())
            out = a.clone()
            a[:part["own_begin"] - b] = float("nan")  # stale ghost planes: the exchange must fill them
            a[part["own_end"] - b:] = float("nan")
            for step in range(steps):
                zs.exchange_ghosts(dist, a, rank, world, nz, R)
                if step == 0:  # every ghost plane now holds its owner's values
                    np.testing.assert_array_equal(a.numpy(), g[b:e])
                oracle.apply(a.numpy(), c, R, out=out.numpy())
                a, out = out, a
            mine = a.numpy()[part["own_begin"] - b:part["own_end"] - b]
        else:
            up, u, s, et = sy.wave_fields(nx, ny, nz)
            u = u + sy.uniform_field(nx, ny, nz, seed=4, scale=0.01)
            fs = [torch.from_numpy(np.ascontiguousarray(x[b:e])) for x in (up, u, s, et)]
            prev, cur, vv, ee = fs
            nxt = prev.clone()  # three-buffer rotation, as the oracle's time loop
            for _ in range(steps):
                zs.exchange_ghosts(dist, cur, rank, world, nz, R)
                oracle.wave_step(prev.numpy(), cur.numpy(), vv.numpy(), ee.numpy(), c * 20, R, u_next=nxt.numpy())
                prev, cur, nxt = cur, nxt, prev
            mine = cur.numpy()[part["own_begin"] - b:part["own_end"] - b]
        q.put((rank, mine.copy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("kind", ["sweep", "wave"])
def test_slab_sweeps_over_gloo_equal_the_whole_grid(world, kind):
    import oracle
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + 10 * world + (0 if kind == "sweep" else 1)
    procs = [ctx.Process(target=_worker, args=(r, world, port, kind, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got = np.concatenate([res[r] for r in range(world)])
    nx, ny, nz, R, steps = 24, 20, 41, 4, 3
    c = synth.laplacian8_coeffs().astype(np.float32) / np.float32(20.0)
    if kind == "sweep":
        want = oracle.run_sweeps(synth.uniform_field(nx, ny, nz, seed=3), c, R, steps)
    else:
        up, u, s, et = synth.wave_fields(nx, ny, nz)
        u = u + synth.uniform_field(nx, ny, nz, seed=4, scale=0.01)
        want = oracle.run_wave(up, u, s, et, c * 20, R, steps)[1]
    np.testing.assert_array_equal(got, want)
