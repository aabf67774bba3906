"""Prefill (t >= 256) vs the oracle: fp32 outputs within max(1e-3 |ref|,
1e-4) on ragged and full-size shapes, through the tcgen05 tile path
(tq1_mmv_ws with a workspace) and through the allocation-free tq1_mmv."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,k,t", [(128, 256, 256), (300, 512, 256), (129, 256, 300), (64, 1024, 385),
                                   (257, 4096, 256), (1000, 768, 260)])
def test_prefill_small_full(n, k, t):
    p = synth.matvec(n, k, t, seed=n + 3 * t)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    ref = orc.mmv_f64(orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x), n, k, t)
    G.assert_close(G.mmv_ws(blocks, q8, n, k, t), ref)
    G.assert_close(G.mmv(blocks, q8, n, k, t), ref)


def test_config5_sampled_rows():
    p = synth.config_matvec("c5")
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    rows = np.unique(np.concatenate([[0, 127, 128, p.n - 1], np.random.default_rng(5).integers(0, p.n, 44)]))
    ref = orc.mmv_f64(orc.tq1_encode_rows(p.w[rows]), orc.q8_1_quantize(p.x), rows.size, p.k, p.t)
    G.assert_close(G.mmv_ws(blocks, q8, p.n, p.k, p.t)[:, rows], ref)
    G.assert_close(G.mmv(blocks, q8, p.n, p.k, p.t)[:, rows], ref)


def test_prefill_large_and_tiny_activations():
    # Activations up to ~1e6 force the per-token power-of-two pre-scale; a
    # token of zeros and one of tiny values exercise the other end.
    p = synth.matvec(200, 1024, 256, seed=77)
    x = p.x.copy()
    x[3] *= 1e6
    x[4, :512] *= 3e5
    x[5] = 0.0
    x[6] *= 1e-6
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(x)
    ref = orc.mmv_f64(orc.tq1_encode_rows(p.w), orc.q8_1_quantize(x), p.n, p.k, p.t)
    for y in (G.mmv_ws(blocks, q8, p.n, p.k, p.t), G.mmv(blocks, q8, p.n, p.k, p.t)):
        G.assert_close(y, ref)
        assert np.all(y[5] == 0.0)


def test_prefill_zero_weight_rows_and_determinism():
    p = synth.matvec(256, 512, 300, seed=9)
    w = p.w.copy()
    w[10] = 0.0
    w[200:256] = 0.0
    blocks, q8 = G.quantize_rows(w), G.quantize_acts(p.x)
    a = G.mmv_ws(blocks, q8, p.n, p.k, p.t)
    b = G.mmv_ws(blocks, q8, p.n, p.k, p.t)
    np.testing.assert_array_equal(a, b)
    assert np.all(a[:, 10] == 0.0) and np.all(a[:, 200:] == 0.0)
    ref = orc.mmv_f64(orc.tq1_encode_rows(w), orc.q8_1_quantize(p.x), p.n, p.k, p.t)
    G.assert_close(a, ref)


def test_config5_partials_sampled_rows():
    """The exact integer partials of config 5 (N=14336, K=4096, T=512) through
    the debug entry: tq1_mmv's kernel for this t (16 slices of 32 columns on the
    tensor-core rungs), bit for bit against the oracle on sampled rows."""
    p = synth.config_matvec("c5")
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    rows = np.unique(np.concatenate([[0, 15, 16, p.n - 1], np.random.default_rng(55).integers(0, p.n, 20)]))
    L, torch = G.lib(), G.torch()
    part = torch.full((p.t, p.n, p.k // 32), -2 ** 31, dtype=torch.int32, device="cuda")  # 3.5 GiB
    L.tq1_mmv_partials(blocks, q8, part, p.n, p.k, p.t)
    assert L.tq1_sync_status() == 0
    got = G.host(part[:, torch.from_numpy(rows).cuda()])  # only the sampled rows come back
    del part
    ref = orc.mmv_partials(orc.tq1_encode_rows(p.w[rows]), orc.q8_1_quantize(p.x), rows.size, p.k, p.t)
    np.testing.assert_array_equal(got, ref)

