"""Pins of the oracle's Q8_1 activation quantiser.

The pages give only the block's fields (fp16 scale, fp16 sum, 32 int8
values); the rounding is a stated reading.  These checks pin it from
outside: a hand-worked block (tests/golden/q8_1_example.txt) and invariants
any correct implementation of the reading satisfies.
"""
import os

import numpy as np
import pytest

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    rows = [ln for ln in open(os.path.join(GOLDEN, "q8_1_example.txt")) if ln.strip() and ln[0] != "#"]
    x = np.array([float(v) for v in rows[0].split()], np.float32)
    q = np.array([int(v) for v in rows[1].split()], np.int8)
    d16, s, s16 = rows[2].split()
    return x, q, int(d16, 16), int(s), int(s16, 16)


def test_hand_worked_block():
    x, q, d16, s, s16 = _golden()
    assert x.size == 32 and q.size == 32 and int(q.astype(np.int64).sum()) == s
    out = orc.q8_1_quantize(x[None, :]).reshape(-1)
    assert int(out[0]) | (int(out[1]) << 8) == d16
    assert int(out[2]) | (int(out[3]) << 8) == s16
    np.testing.assert_array_equal(out[4:].view(np.int8), q)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_invariants_random(seed):
    rng = np.random.default_rng(seed)
    t, k = 3, 32 * 64
    x = (rng.standard_normal((t, k)) * 10.0 ** rng.uniform(-3, 3, (t, 1))).astype(np.float32)
    d, s, q = orc.q8_1_fields(orc.q8_1_quantize(x), t, k)
    xb = x.reshape(t, k // 32, 32).astype(np.float64)
    qb = q.reshape(t, k // 32, 32).astype(np.int64)
    amax = np.abs(xb).max(axis=2)
    dd = amax / 127.0
    # the extreme element maps to +-127 and the rest stays in range
    arg = np.abs(xb).argmax(axis=2)
    ext = np.take_along_axis(qb, arg[:, :, None], axis=2)[:, :, 0]
    assert np.all(np.abs(ext) == 127)
    assert np.all(np.abs(qb) <= 127)
    # rounding error at most half a step (small slack for the fp32 divide)
    assert np.all(np.abs(xb / dd[:, :, None] - qb) <= 0.5 + 1e-4)
    # signs agree
    assert np.all((qb == 0) | (np.sign(qb) == np.sign(xb)))
    # stored scale is the fp16 rounding of amax/127: within half an ulp,
    # which is relative 2^-11 for normals and the fixed 2^-25 below 2^-14
    half_ulp = lambda v: np.maximum(np.abs(v) * 2.0 ** -11, 2.0 ** -25)
    assert np.all(np.abs(d - dd) <= half_ulp(dd) * (1 + 1e-6))
    # stored sum is the fp16 rounding of d * sum(q) (d itself rounded in fp32)
    ss = dd * qb.sum(axis=2)
    assert np.all(np.abs(s - ss) <= half_ulp(ss) * (1 + 1e-5) + np.abs(ss) * 1e-6)


def test_zero_block():
    d, s, q = orc.q8_1_fields(orc.q8_1_quantize(np.zeros((1, 64), np.float32)), 1, 64)
    assert not d.any() and not s.any() and not q.any()


def test_single_nonzero_and_negative_extreme():
    x = np.zeros((1, 32), np.float32)
    x[0, 31] = -3.0
    d, s, q = orc.q8_1_fields(orc.q8_1_quantize(x), 1, 32)
    assert q[0, 31] == -127 and not q[0, :31].any()
    assert np.isclose(d[0, 0], 3.0 / 127, rtol=2 ** -11)


def test_denormal_inputs():
    x = np.full((1, 32), np.float32(1e-40))
    x[0, 0] = np.float32(3e-40)
    d, s, q = orc.q8_1_fields(orc.q8_1_quantize(x), 1, 32)
    # amax/127 is a tiny fp32 denormal: the fp16 scale is 0, the int8 codes
    # are still finite (x/d = 214102/1686 and 71367/1686 in units of 2^-149)
    assert d[0, 0] == 0.0
    assert int(q[0, 0]) == 127 and np.all(q[0, 1:] == 42)
