"""The seeded input generator: determinism, shapes, per-request regeneration."""
import numpy as np

import workloads
from workloads import bf16_bits_to_f32, f32_to_bf16_bits


def test_subset_regeneration_matches_full():
    w = workloads.scaled(workloads.get("qwen3_4b_like"), B=6, V=512, r=16, H=32)
    full = workloads.generate(w)
    sub = workloads.generate(w, requests=[4, 1])
    np.testing.assert_array_equal(sub.U, full.U[[4, 1]])
    np.testing.assert_array_equal(sub.T, full.T[[4, 1]])
    np.testing.assert_array_equal(sub.h, full.h[[4, 1]])
    np.testing.assert_array_equal(sub.anchor, full.anchor[[4, 1]])
    again = workloads.generate(w)
    np.testing.assert_array_equal(again.U, full.U)
    np.testing.assert_array_equal(again.W2, full.W2)


def test_shapes_and_types():
    for w in workloads.WORKLOADS:
        s = workloads.scaled(w, B=2, V=256)
        x = workloads.generate(s)
        assert x.U.shape == (2, s.gamma, 256) and x.U.dtype == np.float32
        assert x.T.shape == (2, s.gamma + 1, 256)
        assert x.W1.shape == (256, s.r) and x.W1.dtype == np.uint16
        assert x.W2.shape == (s.r, 256)
        assert x.h.shape == (2, s.gamma, s.H)
        assert x.w_c.shape == (s.H + s.r,)
        assert x.sps.shape == (2 * (s.gamma + 1) + 1,) and np.all(x.sps > 0)
        assert np.all((x.anchor >= 0) & (x.anchor < 256))


def test_bf16_round_trip_and_rounding():
    x = np.array([1.0, -2.5, 3.140625, 1.0 + 2**-8, 1.0 + 3 * 2**-9], np.float32)
    y = bf16_bits_to_f32(f32_to_bf16_bits(x))
    np.testing.assert_array_equal(y[:3], x[:3])
    assert y[3] == 1.0                       # tie rounds to even
    assert y[4] == np.float32(1.0 + 2**-7)   # above the tie rounds up


def test_spikes_and_target_noise():
    w = workloads.scaled(workloads.get("long_block"), B=2, V=20000)
    x = workloads.generate(w)
    frac = np.mean(x.U - np.round(x.U) == 0)   # no exact structure expected
    assert frac < 0.01
    d1 = (x.T[:, 0] - x.U[:, 0]).std()
    d15 = (x.T[:, 14] - x.U[:, 14]).std()
    assert abs(d1 - 0.5) < 0.02 and abs(d15 - 2.0) < 0.05
