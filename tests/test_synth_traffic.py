"""Input generator and traffic-model checks (no GPU)."""
import os

import numpy as np
import pytest

from seismic_wave_propagation_gb300 import synth, traffic


def test_splitmix64_published_sequence():
    # SplitMix64 with state 0: the generator adds gamma before mixing, so its k-th
    # output is mix(k * gamma) (k = 1, 2, 3), i.e. mix64((k-1) * gamma) here.
    g = 0x9E3779B97F4A7C15
    xs = np.array([0, g, (2 * g) % (1 << 64)], dtype=np.uint64)
    got = [int(v) for v in synth.mix64(xs)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_uniform_is_exact_fp32_and_in_range():
    u = synth.uniform_field(37, 5, 3)
    assert u.dtype == np.float32 and u.shape == (3, 5, 37)
    assert u.min() >= -1.0 and u.max() < 1.0
    idx = np.arange(u.size, dtype=np.uint64)
    np.testing.assert_array_equal(u.ravel(), synth.uniform_from_index(synth.DEFAULT_SEED, idx).astype(np.float32))
    assert np.all(synth.uniform_from_index(synth.DEFAULT_SEED, idx).astype(np.float32).astype(np.float64)
                  == synth.uniform_from_index(synth.DEFAULT_SEED, idx))
    assert abs(float(u.mean())) < 0.05


def test_uniform_chunking_is_invisible():
    a = synth.uniform_field(1024, 1024, 9)  # several chunks, threaded
    idx = np.arange(a.size, dtype=np.uint64)
    np.testing.assert_array_equal(a.ravel(), synth.uniform_from_index(synth.DEFAULT_SEED, idx).astype(np.float32))


def test_wave_inputs():
    n = 64
    up, u, s, e = synth.wave_fields(n, n, n)
    assert u[32, 32, 32] == 1.0 and np.array_equal(u, up)
    assert abs(u[32, 32, 35] - np.exp(-9 / 18)) < 1e-7
    assert e[0, 20, 20] == np.float32(0.1) and e[32, 32, 32] == 0.0
    assert e[16, 32, 32] == 0.0 and abs(e[15, 32, 32] - 0.1 / 256) < 1e-9
    vz = s[:, 0, 0]
    np.testing.assert_allclose(vz[0], 0.0225, rtol=1e-6)
    np.testing.assert_allclose(vz[-1], 0.2025, rtol=1e-6)
    assert len(np.unique(vz)) == 8
    assert np.all(np.diff(vz) >= 0)


def test_sinusoids():
    p = synth.sinusoid_params()
    assert len(p) == 4 and all(1 <= a <= 8 and 1 <= b <= 8 and 1 <= c <= 8 for a, b, c, _ in p)
    f = synth.sinusoid_field(32, 24, 16)
    assert f.shape == (16, 24, 32) and np.all(np.abs(f) <= 4.01)


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pmpp_opb.txt")


def _golden():
    vals = {}
    for ln in open(GOLDEN):
        if ln.strip() and not ln.startswith("#"):
            k, v = ln.split()[:2]
            vals[k] = float(v)
    return vals


def _close(printed, got):
    s = repr(printed)
    decimals = len(s.split(".")[1]) if "." in s and not s.endswith(".0") else 0
    return abs(got - printed) <= 0.5 * 10 ** (-decimals) + 1e-12


def test_page_figures_pin_the_counting_helpers():
    g = _golden()
    assert _close(g["naive_op_per_byte_R1"], traffic.naive_op_per_byte(1))
    assert _close(g["tiled_op_per_byte_T8_R1"], traffic.tiled_op_per_byte(8, 1))
    assert _close(g["tiled_op_per_byte_T32_R1"], traffic.tiled_op_per_byte(32, 1))
    assert _close(g["tiled_op_per_byte_limit_R1"], traffic.tiled_op_per_byte_limit(1))
    assert _close(g["halo_fraction_T8_R1"], traffic.halo_fraction(8, 1))
    assert traffic.shared_bytes_plane_buffers(32, 3) == g["shared_bytes_3planes_T32"]
    assert traffic.shared_bytes_plane_buffers(32, 1) == g["shared_bytes_1plane_T32"]
    i, o, opb = traffic.coarsened_tile_counts(32, 16, 1)
    assert i == g["exercise_inputs_T32_C16"] and o == g["exercise_outputs_T32_C16"]
    assert _close(g["exercise_op_per_byte_T32_C16"], opb)
    assert traffic.flops_per_point(1, True) == g["flops_per_point_7pt"]


def test_compulsory_bytes():
    assert traffic.interior_points(512, 512, 512, 4) == 504 ** 3
    assert traffic.apply_bytes(512, 512, 512, 4) == 4 * 512 ** 3 + 4 * 504 ** 3
    assert traffic.wave_bytes(640, 640, 640, 4) == 4 * 640 ** 3 + 16 * 632 ** 3
    assert traffic.interior_points(8, 8, 8, 4) == 0
    assert traffic.flops_per_point(4) == 29
