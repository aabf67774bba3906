"""Quantisers on the GPU vs the oracle, byte for byte."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_quantize_rows_configs(name):
    p = synth.config_matvec(name)
    got = G.host(G.quantize_rows(p.w))
    want = orc.tq1_encode_rows(p.w).reshape(-1)
    np.testing.assert_array_equal(got, want)


def test_quantize_rows_edges():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((9, 512)) * 0.3).astype(np.float32)
    w[0, :256] = 0.0                                  # all-zero block
    w[1, :256] = 0.0
    w[1, 0], w[1, 1], w[1, 2] = 1.0, 0.5, -0.5        # exact ties
    w[2, 255] = 40.0                                   # amax at the last element
    w[3, 0] = -40.0                                    # amax at the first element
    w[4, :256] = np.float32(1e-40)                     # denormals
    w[4, 7] = np.float32(-3e-40)
    w[5] = np.float32(np.float16(0.07)) * rng.integers(-1, 2, 512)  # exact d * t
    w[6, 256:] = 70000.0                               # scale overflows fp16
    got = G.host(G.quantize_rows(w))
    want = orc.tq1_encode_rows(w).reshape(-1)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("t,k", [(1, 1024), (1, 6144), (32, 6144), (3, 32 * 7)])
def test_quantize_acts_random(t, k):
    x = np.random.default_rng(t * 1000 + k).standard_normal((t, k)).astype(np.float32)
    got = G.host(G.quantize_acts(x))
    want = orc.q8_1_quantize(x).reshape(-1)
    np.testing.assert_array_equal(got, want)


def test_quantize_acts_edges():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((1, 32 * 8)) * 10.0 ** rng.uniform(-6, 6, (1, 32 * 8))).astype(np.float32)
    b = x.reshape(8, 32)
    b[0] = 0.0                                                   # zero block
    b[1] = np.array([127, 63.5, -63.5, 0.5, -0.5, 1.5, 2.5, -2.5] * 4, np.float32)   # ties
    b[2, 31] = 1e6                                               # amax last
    b[3, 0] = -1e6                                               # amax first
    b[4] = np.float32(1e-40)                                     # denormals
    b[4, 0] = np.float32(3e-40)
    b[5] = np.float32(1e-30)                                     # fp16 scale underflow
    b[6] = np.float32(3e6)                                       # fp16 sum overflow
    got = G.host(G.quantize_acts(x))
    want = orc.q8_1_quantize(x).reshape(-1)
    np.testing.assert_array_equal(got, want)


def test_quantize_empty_is_noop():
    L = G.lib()
    L.tq1_quantize_rows(0, 0, 0, 256)
    L.q8_1_quantize_acts(0, 0, 0, 256)
    assert L.tq1_sync_status() == 0
