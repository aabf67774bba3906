"""Pins of the oracle's TQ1_0 byte code, element order and fp16 conversion.

Nothing here compares the oracle with itself: the checks are exhaustive
round trips over every trit pattern, a closed form of the byte code,
hand-worked fixtures (tests/golden/), the element order stated on
PrismML-Eng/llama.cpp issue #139 ("Current behavior": chunk c reads digit c
of bytes qs[0..31]), and numpy's own binary16 conversion.
"""
import itertools
import os

import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_five_trit_bytes_round_trip_exhaustive():
    seen = set()
    for u in itertools.product(range(3), repeat=5):
        b = orc.pack_byte(u)
        assert 0 <= b <= 255
        assert tuple(orc.digit(b, k) for k in range(5)) == u
        v = sum(ui * 3 ** (4 - i) for i, ui in enumerate(u))
        # closed form: the ceil code is inverted by floor(b*243/256)
        assert (b * 243) // 256 == v
        seen.add(b)
    assert len(seen) == 243
    assert min(seen) == 0 and max(seen) == 255


def test_four_trit_bytes_round_trip_exhaustive():
    seen = set()
    for u in itertools.product(range(3), repeat=4):
        b = orc.pack_byte(list(u) + [0])
        assert tuple(orc.digit(b, k) for k in range(4)) == u
        assert orc.digit(b, 4) == 0
        seen.add(b)
    assert len(seen) == 81


def test_byte_code_golden():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "tq1_byte_code.txt")) if ln.strip() and ln[0] != "#"]
    assert len(rows) >= 10
    for r in rows:
        u = [int(x) for x in r[:5]]
        v, b = int(r[5]), int(r[6])
        assert sum(ui * 3 ** (4 - i) for i, ui in enumerate(u)) == v
        assert orc.pack_byte(u) == b, (u, b)
        assert [orc.digit(b, k) for k in range(5)] == u


def test_element_order_first_160_from_the_page():
    # Chunk c (elements 32c..32c+31) reads digit c of bytes qs[0..31].
    for e in range(160):
        assert orc.elem_pos(e) == (e % 32, e // 32)


def test_element_order_is_a_bijection_onto_digit_slots():
    slots = [orc.elem_pos(e) for e in range(256)]
    assert len(set(slots)) == 256
    assert all(0 <= b < 48 and 0 <= d < 5 for b, d in slots[:240])
    assert all(48 <= b < 52 and 0 <= d < 4 for b, d in slots[240:])


@pytest.mark.parametrize("e", [0, 1, 31, 32, 77, 159, 160, 175, 176, 239, 240, 243, 244, 255])
def test_one_hot_block_touches_one_digit(e):
    d = np.float32(np.float16(0.0625))
    w = np.zeros((1, 256), dtype=np.float32)
    w[0, e] = d
    blk = orc.tq1_encode_rows(w).reshape(-1)
    zero = orc.pack_byte([1, 1, 1, 1, 1])
    zero_qh = orc.pack_byte([1, 1, 1, 1, 0])
    bi, dg = orc.elem_pos(e)
    for j in range(52):
        base = zero if j < 48 else zero_qh
        if j != bi:
            assert blk[j] == base
    digits = [orc.digit(int(blk[bi]), k) for k in range(5)]
    expect = [1, 1, 1, 1, 1 if bi < 48 else 0]
    expect[dg] = 2
    assert digits == expect
    if e < 160:
        assert bi == e % 32 and dg == e // 32
    assert int(blk[52]) | (int(blk[53]) << 8) == int(np.float16(d).view(np.uint16))


@pytest.mark.parametrize("p_zero", [1.0 / 3.0, 0.4])
def test_encode_decode_round_trip(p_zero):
    p = synth.matvec(7, 1024, 1, p_zero=p_zero, seed=11)
    blocks = orc.tq1_encode_rows(p.w)
    tr, sc = orc.tq1_decode_rows(blocks, p.n, p.k)
    np.testing.assert_array_equal(tr, p.trits)
    np.testing.assert_array_equal(sc, p.scales.astype(np.float32))


def test_all_zero_block_has_zero_scale():
    blocks = orc.tq1_encode_rows(np.zeros((2, 512), np.float32))
    tr, sc = orc.tq1_decode_rows(blocks, 2, 512)
    assert not tr.any() and not sc.any()


def test_weight_rounding_ties_go_away_from_zero():
    # amax = 1: 0.5 and -0.5 are exact ties of the trit rounding.
    w = np.zeros((1, 256), np.float32)
    w[0, :4] = [1.0, 0.5, -0.5, 0.49]
    tr, sc = orc.tq1_decode_rows(orc.tq1_encode_rows(w), 1, 256)
    assert list(tr[0, :4]) == [1, 1, -1, 0]
    assert sc[0, 0] == 1.0


def test_f16_from_f32_matches_numpy():
    rng = np.random.default_rng(0)
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 6.1035156e-05, 6.0e-08, 5.96e-08,
            2.98e-08, 2.9802322e-08, 1e-10, 1.00048828125, 1.0009765625, 1.00146484375, 2049.0, 2051.0,
            float(np.float32(0.1)), float(np.nextafter(np.float32(65504), np.float32(0)))]
    vals += list(rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-9, 5, 20000))
    vals += list(np.float32(2.0) ** rng.integers(-30, 17, 2000) * (1 + np.float32(2.0) ** -11))  # exact ties
    with np.errstate(over="ignore"):
        for v in vals:
            v32 = np.float32(v)
            expect = int(np.array([v32], np.float32).astype(np.float16).view(np.uint16)[0])
            assert orc.f16_from_f32(float(v32)) == expect, v


def test_f32_from_f16_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    for h in range(0, 65536, 7):
        got = orc.f32_from_f16(h)
        r = ref[h]
        if np.isnan(r):
            assert np.isnan(got)
        else:
            assert got == r and np.signbit(got) == np.signbit(r), h


@pytest.mark.parametrize("p_zero", [1.0 / 3.0, 0.4])
def test_dequantize_returns_the_synthetic_weights(p_zero):
    # The generator draws fp32 weights that are exactly fp16(d) * trit, so the
    # values the blocks encode are those weights, element for element.
    p = synth.matvec(19, 1024, 1, p_zero=p_zero, seed=17)
    blocks = orc.tq1_encode_rows(p.w)
    np.testing.assert_array_equal(orc.tq1_dequantize_rows(blocks, p.n, p.k), p.w)
