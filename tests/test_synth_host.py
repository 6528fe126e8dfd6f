"""Host side of the seeded input generator: determinism, slicing and distributions."""

import math

import numpy as np

from synth import host_fill, normal_K, uniform_K, NORMAL, UNIFORM, get


def test_slices_are_consistent():
    full = host_fill(0, 4, 0, 10000, NORMAL, normal_K(1.0), True)
    part = host_fill(0, 4, 1234, 500, NORMAL, normal_K(1.0), True)
    assert np.array_equal(full[1234:1734], part)
    assert np.array_equal(full, host_fill(0, 4, 0, 10000, NORMAL, normal_K(1.0), True))
    assert not np.array_equal(full, host_fill(1, 4, 0, 10000, NORMAL, normal_K(1.0), True))
    assert not np.array_equal(full, host_fill(0, 5, 0, 10000, NORMAL, normal_K(1.0), True))


def test_bf16_is_rne_of_fp32():
    f = host_fill(3, 7, 0, 4096, NORMAL, normal_K(0.3), False)
    b = host_fill(3, 7, 0, 4096, NORMAL, normal_K(0.3), True)
    u = f.view(np.uint32).astype(np.uint64)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(b, ref)


def test_normal_moments():
    v = host_fill(0, 1, 0, 200000, NORMAL, normal_K(2.0), False).astype(np.float64)
    assert abs(v.mean()) < 0.02
    assert abs(v.std() - 2.0) < 0.02
    assert np.abs(v).max() <= 2.0 * 2 * math.sqrt(3) + 1e-6


def test_uniform_range():
    v = host_fill(0, 2, 0, 100000, UNIFORM, uniform_K(0.5), False).astype(np.float64)
    assert v.min() >= -0.5 and v.max() <= 0.5
    assert abs(v.mean()) < 0.01
    assert abs(v.var() - 0.25 / 3) < 0.002


def test_workload_shapes_and_zipf_bias():
    w = get("mixtral")
    gb = w.gate_bias_host()
    p = np.exp(gb.astype(np.float64))
    assert abs(p.sum() - 1) < 1e-6
    assert np.allclose(p, [0.398, 0.186, 0.119, 0.087, 0.068, 0.056, 0.047, 0.040], atol=1e-3)
    t = get("tiny")
    assert t.x_host().shape == (64, 8) and t.wg_host().shape == (8, 4)
    assert t.w1_host(3).shape == (8, 8) and t.b1_host(3).shape == (8,)
    assert np.array_equal(t.x_host(rows=[5, 2]), t.x_host()[[5, 2]])
    s = get("switch")
    assert s.N1 == 4096 and s.w1_host(0).dtype == np.uint16
