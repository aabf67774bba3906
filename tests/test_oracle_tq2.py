"""Pins of the oracle's TQ2_0 functions (the 2-bit sibling format, reading R6
of the oracle: qs[64] with four 2-bit codes per byte, fp16 d at byte 64).

The pages name TQ2_0 but give no layout, so the layout itself is a reading
("parity unpinned" by the pages).  What is pinned is everything built on it:

* the element order is a bijection of the 256 (byte, field) slots, and each
  32-element chunk reads one field of 32 consecutive bytes (the chunk
  contract of PrismML-Eng/llama.cpp issue #139, "Current behavior");
* encode -> decode returns the generator's own trits and fp16 scales;
* cross-format: the same weights encoded as TQ1_0 (whose oracle is pinned by
  its own tests) and as TQ2_0 give identical trits, identical integer
  partials and bit-identical fp64 outputs;
* brute force: the dense fp64 product of the generator's trits and scales with
  the dequantised activations;
* the unused code 3 decodes to +2 (value = code - 1).
"""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth


def test_element_order_is_a_bijection_with_the_chunk_contract():
    seen = set()
    for e in range(256):
        bi, f = orc.tq2_elem_pos(e)
        assert 0 <= bi < 64 and 0 <= f < 4
        seen.add((bi, f))
        c = e // 32
        # chunk c: one field of 32 consecutive bytes, element order within the chunk
        assert f == c % 4 and bi == 32 * (c // 4) + e % 32
    assert len(seen) == 256


def test_code_field_extraction_all_byte_values():
    # A block whose qs bytes are all equal to b: element e's code is field
    # f of b, for every byte value (independent bit arithmetic here).
    for b in range(256):
        blk = np.zeros(orc.TQ2_BYTES, dtype=np.uint8)
        blk[:64] = b
        for e in (0, 31, 32, 100, 127, 128, 200, 255):
            f = (e // 32) % 4
            assert orc.tq2_code(blk, e) == (b >> (2 * f)) & 3


@pytest.mark.parametrize("n,k,p_zero", [(1, 256, 1 / 3), (5, 1024, 0.4), (3, 2048, 0.0), (2, 512, 1.0)])
def test_round_trip_synthetic_weights(n, k, p_zero):
    p = synth.matvec(n, k, 1, p_zero=p_zero, seed=11 + n + k)
    blocks = orc.tq2_encode_rows(p.w)
    assert blocks.shape == (n, k // 256, 66)
    trits, scales = orc.tq2_decode_rows(blocks, n, k)
    np.testing.assert_array_equal(trits, p.trits)
    # An all-zero block has amax 0 -> d = 0; every other block keeps its scale.
    nz = np.any(p.trits.reshape(n, k // 256, 256) != 0, axis=2)
    np.testing.assert_array_equal(scales[nz], p.scales.astype(np.float32)[nz])
    assert np.all(scales[~nz] == 0)
    # Codes written by the encoder are 0, 1 or 2 only.
    codes = np.stack([(blocks[:, :, :64] >> (2 * f)) & 3 for f in range(4)])
    assert codes.max() <= 2


@pytest.mark.parametrize("shape", [(4, 256, 1), (7, 1024, 3), (3, 2048, 2)])
def test_cross_format_identical_results(shape):
    n, k, t = shape
    p = synth.matvec(n, k, t, p_zero=0.4, seed=3 * n + t)
    b1, b2 = orc.tq1_encode_rows(p.w), orc.tq2_encode_rows(p.w)
    np.testing.assert_array_equal(orc.tq1_decode_rows(b1, n, k)[0], orc.tq2_decode_rows(b2, n, k)[0])
    np.testing.assert_array_equal(orc.tq1_decode_rows(b1, n, k)[1], orc.tq2_decode_rows(b2, n, k)[1])
    q8 = orc.q8_1_quantize(p.x)
    np.testing.assert_array_equal(orc.mmv_partials(b1, q8, n, k, t), orc.tq2_mmv_partials(b2, q8, n, k, t))
    np.testing.assert_array_equal(orc.mmv_f64(b1, q8, n, k, t), orc.tq2_mmv_f64(b2, q8, n, k, t))
    rows = np.array([n - 1, 0], dtype=np.int64)
    np.testing.assert_array_equal(orc.tq2_mmv_f64_rows(b2, q8, n, k, t, rows), orc.tq2_mmv_f64(b2, q8, n, k, t)[:, rows])


@pytest.mark.parametrize("n", [1, 3])
@pytest.mark.parametrize("k", [256, 768])
@pytest.mark.parametrize("t", [1, 2])
def test_brute_force_dense_product(n, k, t):
    p = synth.matvec(n, k, t, seed=200 + n * 10 + t)
    blocks = orc.tq2_encode_rows(p.w)
    q8 = orc.q8_1_quantize(p.x)
    d, _, q = orc.q8_1_fields(q8, t, k)
    x = q.astype(np.float64) * np.repeat(d.astype(np.float64), 32, axis=1)
    w = p.trits.astype(np.float64) * np.repeat(p.scales.astype(np.float64), 256, axis=1)
    np.testing.assert_allclose(orc.tq2_mmv_f64(blocks, q8, n, k, t), x @ w.T, rtol=1e-12, atol=1e-12)


def test_unused_code_decodes_to_plus_two():
    blk = np.zeros((1, 1, orc.TQ2_BYTES), dtype=np.uint8)
    blk[0, 0, 5] = 0b11  # element 5: code 3; every other element code 0 (-1)
    blk[0, 0, 64:66] = np.frombuffer(np.float16(0.5).tobytes(), dtype=np.uint8)
    trits, scales = orc.tq2_decode_rows(blk, 1, 256)
    assert trits[0, 5] == 2 and np.all(np.delete(trits[0], 5) == -1) and scales[0, 0] == 0.5
    x = np.ones((1, 256), dtype=np.float32)
    q8 = orc.q8_1_quantize(x)  # q = 127 everywhere, d = 1/127
    part = orc.tq2_mmv_partials(blk, q8, 1, 256, 1)
    assert part[0, 0, 0] == 127 * (2 - 31) and np.all(part[0, 0, 1:] == -127 * 32)


def test_dequantize_is_trits_times_scales():
    p = synth.matvec(6, 768, 1, p_zero=0.4, seed=8)
    got = orc.tq2_dequantize_rows(orc.tq2_encode_rows(p.w), 6, 768)
    want = p.trits.astype(np.float32) * np.repeat(p.scales.astype(np.float32), 256, axis=1)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(got, p.w)  # the synthetic weights round-trip exactly


def test_mmv_id_cross_format():
    # Expert-routed mat-vec: the same experts encoded as TQ1_0 and TQ2_0 give
    # bit-identical fp64 outputs (reading R5 of the oracle for the routing).
    E, n, k, t, top_k = 5, 12, 512, 3, 2
    p = synth.matvec(E * n, k, t, p_zero=0.4, seed=77)
    ids = np.array([[0, 4], [2, 2], [1, 3]], dtype=np.int32)
    q8 = orc.q8_1_quantize(p.x)
    y1 = orc.mmv_id_f64(orc.tq1_encode_rows(p.w), E, q8, ids, n, k, t, top_k)
    y2 = orc.tq2_mmv_id_f64(orc.tq2_encode_rows(p.w), E, q8, ids, n, k, t, top_k)
    np.testing.assert_array_equal(y1, y2)
    # and slot (c, s) is the dense mat-vec of expert ids[c, s] against token c
    dense = orc.tq2_mmv_f64(orc.tq2_encode_rows(p.w), q8, E * n, k, t)
    for c in range(t):
        for s in range(top_k):
            e = ids[c, s]
            np.testing.assert_array_equal(y2[c, s], dense[c, e * n:(e + 1) * n])
