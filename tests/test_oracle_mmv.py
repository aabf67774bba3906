"""Pins of the oracle's dot products against definitions it does not share.

* brute force: the dense fp64 product W @ X of the generator's own trits and
  scales with the dequantised activations (numpy matmul), on tiny shapes;
* integer identity per 32-element chunk: I = sum(trit * q8), computed from the
  generator's trits with numpy;
* closed forms (all trits +1 and q = 127 gives I = 32*127 = 4064);
* mat-vec-id reduces to per-slot dense products.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth


def _dense_x(q8, t, k):
    d, _, q = orc.q8_1_fields(q8, t, k)
    return q.astype(np.float64) * np.repeat(d.astype(np.float64), 32, axis=1)


def _dense_w(p):
    return p.trits.astype(np.float64) * np.repeat(p.scales.astype(np.float64), 256, axis=1)


@pytest.mark.parametrize("n", [1, 2, 3, 5])
@pytest.mark.parametrize("k", [256, 512])
@pytest.mark.parametrize("t", [1, 2, 3])
def test_brute_force_dense_product(n, k, t):
    p = synth.matvec(n, k, t, seed=100 + n * 10 + t)
    blocks = orc.tq1_encode_rows(p.w)
    q8 = orc.q8_1_quantize(p.x)
    y = orc.mmv_f64(blocks, q8, n, k, t)
    ref = _dense_x(q8, t, k) @ _dense_w(p).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", [(4, 256, 2), (3, 1024, 3), (2, 2048, 1)])
def test_integer_partials_identity(shape):
    n, k, t = shape
    p = synth.matvec(n, k, t, p_zero=0.4, seed=7)
    blocks = orc.tq1_encode_rows(p.w)
    q8 = orc.q8_1_quantize(p.x)
    part = orc.mmv_partials(blocks, q8, n, k, t)
    _, _, q = orc.q8_1_fields(q8, t, k)
    ref = np.einsum("nbe,tbe->tnb", p.trits.reshape(n, k // 32, 32).astype(np.int64),
                    q.reshape(t, k // 32, 32).astype(np.int64))
    np.testing.assert_array_equal(part, ref)


def test_extreme_partials_closed_form():
    w = np.full((2, 256), np.float32(0.5))
    w[1] = -0.5
    x = np.full((1, 256), np.float32(3.0))
    part = orc.mmv_partials(orc.tq1_encode_rows(w), orc.q8_1_quantize(x), 2, 256, 1)
    assert np.all(part[0, 0] == 4064) and np.all(part[0, 1] == -4064)
    y = orc.mmv_f64(orc.tq1_encode_rows(w), orc.q8_1_quantize(x), 2, 256, 1)
    d_a = float(np.float16(np.float32(3.0) / np.float32(127.0)))
    np.testing.assert_allclose(y[0], [0.5 * d_a * 4064 * 8, -0.5 * d_a * 4064 * 8], rtol=1e-15)


def test_one_hot_layout_probe():
    # weight element e = +1 (all others 0) against an activation one-hot at e':
    # the output is nonzero exactly when e == e'.
    k = 256
    for e in (0, 37, 159, 160, 201, 239, 240, 255):
        w = np.zeros((1, k), np.float32)
        w[0, e] = 1.0
        blocks = orc.tq1_encode_rows(w)
        for e2 in (e, (e + 1) % k, (e + 32) % k):
            x = np.zeros((1, k), np.float32)
            x[0, e2] = 1.0
            y = orc.mmv_f64(blocks, orc.q8_1_quantize(x), 1, k, 1)[0, 0]
            assert (y != 0.0) == (e == e2)


def test_sampled_rows_match_full():
    p = synth.matvec(9, 512, 2, seed=3)
    blocks, q8 = orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x)
    full = orc.mmv_f64(blocks, q8, 9, 512, 2)
    rows = [8, 0, 4, 4]
    np.testing.assert_array_equal(orc.mmv_f64_rows(blocks, q8, 9, 512, 2, rows), full[:, rows])


def test_mmv_id_reduces_to_dense_slots():
    m = synth.moe(n_experts=6, n=5, k=512, t=3, top_k=2, seed=9)
    ws = [m.expert(e) for e in range(6)]
    blocks = np.stack([orc.tq1_encode_rows(w) for (_, _, w) in ws])
    q8 = orc.q8_1_quantize(m.x)
    ids = m.ids.copy()
    ids[2, 1] = 99  # out of range: slot left untouched
    y = orc.mmv_id_f64(blocks, 6, q8, ids, 5, 512, 3, 2)
    xd = _dense_x(q8, 3, 512)
    for t in range(3):
        for s in range(2):
            e = ids[t, s]
            if e >= 6:
                assert np.all(np.isnan(y[t, s]))
                continue
            tr, sc, _ = ws[e]
            wd = tr.astype(np.float64) * np.repeat(sc.astype(np.float64), 256, axis=1)
            np.testing.assert_allclose(y[t, s], wd @ xd[t], rtol=1e-12, atol=1e-12)
    rows = [4, 1]
    ys = orc.mmv_id_f64_rows(blocks, 6, q8, ids, 5, 512, 3, 2, rows)
    np.testing.assert_array_equal(ys[:2], y[:2][:, :, rows])
