"""The seeded input recipes: determinism and distribution shape."""
import numpy as np

from bit_quantized_gemv_tq1_gb300 import synth


def test_matvec_is_deterministic_and_exact():
    a = synth.matvec(16, 512, 2, p_zero=0.4, d_lo=0.005, d_hi=0.05, seed=2)
    b = synth.matvec(16, 512, 2, p_zero=0.4, d_lo=0.005, d_hi=0.05, seed=2)
    np.testing.assert_array_equal(a.w, b.w)
    np.testing.assert_array_equal(a.x, b.x)
    # weights are exactly d * t
    w = a.trits.reshape(16, 2, 256) * a.scales.astype(np.float32)[:, :, None]
    np.testing.assert_array_equal(a.w, w.reshape(16, 512))


def test_trit_distribution():
    t = synth.draw_trits(np.random.default_rng(0), (400, 1000), 0.4)
    f0 = np.mean(t == 0)
    assert abs(f0 - 0.4) < 0.01
    assert abs(np.mean(t == 1) - 0.3) < 0.01 and abs(np.mean(t == -1) - 0.3) < 0.01
    u = synth.draw_trits(np.random.default_rng(0), (400, 1000), 1.0 / 3.0)
    assert set(np.unique(u)) == {-1, 0, 1}


def test_scales_range():
    s = synth.draw_scales(np.random.default_rng(1), (1000,), 0.005, 0.05)
    assert s.dtype == np.float16
    assert s.min() >= np.float16(0.005) and s.max() <= np.float16(0.05)


def test_zipf_routing():
    ids = synth.zipf_topk(np.random.default_rng(2), 64, 128, 8, 1.1)
    assert ids.shape == (64, 8) and ids.min() >= 0 and ids.max() < 128
    for row in ids:
        assert len(set(row.tolist())) == 8
    counts = np.bincount(ids.ravel(), minlength=128)
    assert counts.max() > 3 * counts.mean()   # skewed, not uniform


def test_moe_prefix_consistency():
    a = synth.moe(16, 8, 256, 1, 4, seed=4)
    b = synth.moe(16, 8, 256, 5, 4, seed=4)
    np.testing.assert_array_equal(a.ids[0], b.ids[0])
    np.testing.assert_array_equal(a.x[0], b.x[0])
    np.testing.assert_array_equal(a.expert_weights(3), b.expert_weights(3))
