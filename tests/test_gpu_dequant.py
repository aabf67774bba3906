"""Dequantisation and row gathers on the GPU vs the oracle: the values are
exact (fp16 scale times -1, 0 or +1), so fp32 and fp16 outputs must equal the
oracle's bit for bit."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _dequant(blocks, n, k, f16):
    t = G.torch()
    out = t.full((n, k), float("nan"), dtype=t.float16 if f16 else t.float32, device="cuda")
    G.lib().tq1_dequantize_rows(blocks, out, n, k, f16)
    assert G.lib().tq1_sync_status() == 0
    return G.host(out)


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("n,k", [(1, 256), (7, 512), (300, 2048), (33, 1280), (129, 6144)])
def test_dequantize_rows_exact(n, k, f16):
    p = synth.matvec(n, k, 1, p_zero=0.4, seed=n + k)
    blocks = G.quantize_rows(p.w)
    got = _dequant(blocks, n, k, f16)
    ref = orc.tq1_dequantize_rows(orc.tq1_encode_rows(p.w), n, k)
    np.testing.assert_array_equal(got, ref.astype(np.float16) if f16 else ref)


def test_dequantize_config2_full_size():
    # The bench's workload: N=5120, K=6144 to fp32 and fp16.
    p = synth.config_matvec("c2")
    blocks = G.quantize_rows(p.w)
    ref = orc.tq1_dequantize_rows(orc.tq1_encode_rows(p.w), p.n, p.k)
    np.testing.assert_array_equal(_dequant(blocks, p.n, p.k, False), ref)
    np.testing.assert_array_equal(_dequant(blocks, p.n, p.k, True), ref.astype(np.float16))


@pytest.mark.parametrize("f16", [False, True])
def test_get_rows_repeats_and_bad_ids(f16):
    n, k = 50, 1024
    p = synth.matvec(n, k, 1, seed=3)
    blocks = G.quantize_rows(p.w)
    ids = np.array([4, 4, 0, 49, 17, -1, 50, 3], dtype=np.int32)
    t = G.torch()
    out = t.full((ids.size, k), 123.0, dtype=t.float16 if f16 else t.float32, device="cuda")
    G.lib().tq1_get_rows(blocks, G.dev(ids), ids.size, out, n, k, f16)
    assert G.lib().tq1_sync_status() == -8  # TQ1_ERR_BAD_ID for -1 and 50
    got = G.host(out)
    ref = orc.tq1_dequantize_rows(orc.tq1_encode_rows(p.w), n, k)
    for i, r in enumerate(ids):
        if 0 <= r < n:
            np.testing.assert_array_equal(got[i], ref[r].astype(np.float16) if f16 else ref[r])
        else:
            assert np.all(got[i] == 123.0)  # untouched
    assert G.lib().tq1_sync_status() == 0  # cleared
