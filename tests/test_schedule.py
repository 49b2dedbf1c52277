"""The launch planner's z-chunk choice (host only, no GPU): stencil_schedule_query.

The plan scores every chunk count n by the round-robin step count
rounds(n) * (ceil(nzi / n) + 0.7 R) and takes, among the counts within 0.5 % of the best,
the one that keeps the most CTA slots busy.  The library scans only the largest chunk
count of each round count; these tests check that it picks what a scan over every
chunk count picks, and that its cost does not grow with nz.
"""
import math
import time

import pytest

from seismic_wave_propagation_gb300 import _lib
from seismic_wave_propagation_gb300 import build as b

TILE_X = 64


@pytest.fixture(scope="module", autouse=True)
def lib():
    b.build()
    return _lib.load()


def full_scan(nx, ny, nz, R, tile_y, kind, sms, occ, x_origin=0):
    """Every chunk count from 1 to nzi, scored as the planner scores them (tiles cover x
    from 0, or from the interior origin x = R)."""
    nzi = nz - 2 * R
    ntiles = math.ceil((nx - 2 * x_origin) / TILE_X) * math.ceil((ny - 2 * R) / tile_y)
    slots = sms * occ

    def score(n):
        items = ntiles * n
        g = min(items, slots)
        rounds = -(-items // g)
        return rounds * (-(-nzi // n) + 0.35 * 2 * R), items / (rounds * slots)

    max_n = min(nzi, (1 << 30) // ntiles)
    best = min(score(n)[0] for n in range(1, max_n + 1))
    pick, pick_busy = 1, -1.0
    for n in range(1, max_n + 1):
        cost, busy = score(n)
        if cost <= best * 1.005 and busy > pick_busy + 1e-12:
            pick, pick_busy = n, busy
    if kind in (0, 3) and R <= 2:
        pick = min(nzi, -(-sms // ntiles))
    return ntiles, pick


SHAPES = [(512, 512, 512), (640, 640, 640), (1536, 1536, 256), (64, 64, 64), (136, 75, 41),
          (2048, 512, 512), (256, 96, 200), (4096, 4096, 40), (64, 64, 3000), (384, 384, 384),
          (1024, 1024, 20), (12, 12, 12), (200, 33, 17), (8192, 2048, 16)]


@pytest.mark.parametrize("nx,ny,nz", SHAPES)
@pytest.mark.parametrize("R,kind,occ", [(4, 0, 2), (4, 1, 2), (1, 0, 4), (2, 0, 3), (3, 1, 2), (4, 3, 2),
                                        (4, 2, 2), (1, 4, 2)])
@pytest.mark.parametrize("sms", [152, 148, 7])
def test_choice_matches_a_scan_over_every_chunk_count(nx, ny, nz, R, kind, occ, sms):
    got = _lib.schedule_query(nx, ny, nz, R, kind, sms, occ)
    tile_y = got["tile_y"]
    assert got["x_origin"] in (0, R)
    ntiles, pick = full_scan(nx, ny, nz, R, tile_y, kind, sms, occ, got["x_origin"])
    assert got["tiles"] == ntiles
    assert got["zchunks"] == pick
    assert got["items"] == ntiles * pick
    assert got["grid"] == min(ntiles * pick, sms * occ)


def test_measured_choices_are_kept():
    """The schedules measured on GB300 (152 SMs): the radius-4 sweep (three CTAs per SM)
    at 512^3 in 7 chunks of 64 x 32 tiles (the fastest of 1-16 chunks within 0.4 %), at
    1536 x 1536 x 256 in 2 chunks of 64 x 24 tiles (2 % behind the best, 3-4); the 640^3
    wave step (three CTAs per SM) in 9, the fastest of 2-12."""
    got = _lib.schedule_query(512, 512, 512, 4, 0, 152, 3)
    assert (got["tile_y"], got["zchunks"]) == (32, 7)
    got = _lib.schedule_query(1536, 1536, 256, 4, 0, 152, 3)
    assert (got["tile_y"], got["zchunks"]) == (24, 2)
    assert _lib.schedule_query(640, 640, 640, 4, 1, 152, 3)["zchunks"] == 9


def test_tall_grid_plans_quickly():
    t0 = time.perf_counter()
    got = _lib.schedule_query(64, 64, 1 << 28, 4, 0, 152, 2)
    dt = time.perf_counter() - t0
    assert dt < 0.05, f"planning took {dt:.3f} s"
    assert got["tiles"] == 2 and got["zchunks"] >= 152 and got["grid"] == 304


def test_two_sweep_kind_only_for_radius_1():
    got = _lib.schedule_query(512, 512, 512, 1, 4, 152, 2)
    assert got["tile_y"] == 30 and got["tiles"] == 8 * 17
    with pytest.raises(_lib.StencilError):
        _lib.schedule_query(512, 512, 512, 4, 4, 152, 2)


def test_empty_interior_and_bad_arguments():
    got = _lib.schedule_query(8, 8, 8, 4, 0, 152, 2)
    assert got["grid"] == 0 and got["zchunks"] == 0
    for args in [(64, 64, 64, 0, 0, 152, 2), (64, 64, 64, 4, 4, 152, 2), (64, 64, 64, 4, 0, 0, 2),
                 (64, 64, 64, 4, 0, 152, 0), (1 << 31, 4, 4, 4, 0, 152, 2), (64, 64, 64, 1, 5, 152, 2)]:
        with pytest.raises(_lib.StencilError):
            _lib.schedule_query(*args)
