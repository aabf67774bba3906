"""Dequantisation and row gathers on the GPU vs the oracle, TQ1_0 and TQ2_0:
the values are exact (fp16 scale times -1, 0 or +1; +2 for TQ2_0's unused
code), so fp32 and fp16 outputs must equal the oracle's bit for bit."""
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
@pytest.mark.parametrize("n,k", [(1, 256), (7, 512), (300, 2048), (33, 1280), (129, 6144), (61, 2816)])
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


# ------------------------------------------------------------------ TQ2_0 --
def _tq2_blocks(w):
    t = G.torch()
    n, k = w.shape
    b = t.empty(n * (k // 256) * 66, dtype=t.uint8, device="cuda")
    G.lib().tq2_quantize_rows(G.dev(w.astype(np.float32)), b, n, k)
    return b



def test_get_rows_many_ids_ragged_segments():
    # 16000 gathered rows of 11 blocks each: every warp takes several row
    # segments (8 blocks and a ragged 3) in turn, rows start at every even
    # offset modulo 16, and some ids are out of range.
    n, k = 300, 2816
    p = synth.matvec(n, k, 1, p_zero=0.3, seed=31)
    blocks = G.quantize_rows(p.w)
    rng = np.random.default_rng(32)
    ids = rng.integers(-2, n + 2, size=16000).astype(np.int32)
    t = G.torch()
    out = t.full((ids.size, k), 7.0, dtype=t.float16, device="cuda")
    G.lib().tq1_get_rows(blocks, G.dev(ids), ids.size, out, n, k, 1)
    assert G.lib().tq1_sync_status() == -8
    got = G.host(out)
    ref = orc.tq1_dequantize_rows(orc.tq1_encode_rows(p.w), n, k).astype(np.float16)
    ok = (ids >= 0) & (ids < n)
    np.testing.assert_array_equal(got[ok], ref[ids[ok]])
    assert np.all(got[~ok] == 7.0)

def _tq2_dequant(blocks, n, k, f16):
    t = G.torch()
    out = t.full((n, k), float("nan"), dtype=t.float16 if f16 else t.float32, device="cuda")
    G.lib().tq2_dequantize_rows(blocks, out, n, k, f16)
    assert G.lib().tq1_sync_status() == 0
    return G.host(out)


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("n,k", [(1, 256), (7, 512), (300, 2048), (33, 1280), (129, 6144), (61, 2816)])
def test_tq2_dequantize_rows_exact(n, k, f16):
    p = synth.matvec(n, k, 1, p_zero=0.4, seed=n + 2 * k)
    got = _tq2_dequant(_tq2_blocks(p.w), n, k, f16)
    ref = orc.tq2_dequantize_rows(orc.tq2_encode_rows(p.w), n, k)
    np.testing.assert_array_equal(got, ref.astype(np.float16) if f16 else ref)


@pytest.mark.parametrize("f16", [False, True])
def test_tq2_dequantize_raw_codes_including_three(f16):
    # Every code, the unused 3 (+2 d) included, and scales up to 1e4.
    n, k = 40, 1024
    rng = np.random.default_rng(12)
    raw = rng.integers(0, 256, size=(n, k // 256, 66), dtype=np.uint8)
    d = rng.uniform(-1e4, 1e4, size=(n, k // 256)).astype(np.float16)
    raw[:, :, 64:66] = d.view(np.uint8).reshape(n, k // 256, 2)
    got = _tq2_dequant(G.dev(raw.reshape(-1)), n, k, f16)
    ref = orc.tq2_dequantize_rows(raw, n, k)
    np.testing.assert_array_equal(got, ref.astype(np.float16) if f16 else ref)


@pytest.mark.parametrize("f16", [False, True])
def test_tq2_get_rows_repeats_and_bad_ids(f16):
    n, k = 50, 1024
    p = synth.matvec(n, k, 1, seed=4)
    blocks = _tq2_blocks(p.w)
    ids = np.array([4, 4, 0, 49, 17, -1, 50, 3], dtype=np.int32)
    t = G.torch()
    out = t.full((ids.size, k), 123.0, dtype=t.float16 if f16 else t.float32, device="cuda")
    G.lib().tq2_get_rows(blocks, G.dev(ids), ids.size, out, n, k, f16)
    assert G.lib().tq1_sync_status() == -8  # TQ1_ERR_BAD_ID for -1 and 50
    got = G.host(out)
    ref = orc.tq2_dequantize_rows(orc.tq2_encode_rows(p.w), n, k)
    for i, r in enumerate(ids):
        if 0 <= r < n:
            np.testing.assert_array_equal(got[i], ref[r].astype(np.float16) if f16 else ref[r])
        else:
            assert np.all(got[i] == 123.0)
