"""The warp-level tensor-core rungs (8..32 token columns, mma.sync over exact
fp16 operands) against the oracle: integer partials bit-exact, fp32 outputs
within max(1e-3 |ref|, 1e-4), on the full-size sweep shape (sampled rows) and
on ragged shapes that exercise partial M-tiles, short K ranges, odd block
counts and every n-tile count; TQ2_0 weights, the residual epilogue and
bitwise determinism."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TQ2_BYTES = 66


def _sample_rows(n, seed, extra=61):
    rng = np.random.default_rng(seed)
    # matrix edges, M-tile edges (rows 15/16, 31/32) and random rows
    fixed = [0, 1, 7, 8, 15, 16, 31, 32, n // 2, n - 17, n - 16, n - 9, n - 1]
    return np.unique(np.clip(np.concatenate([fixed, rng.integers(0, n, extra)]), 0, n - 1))


@pytest.mark.parametrize("t", [7, 8, 9, 16, 17, 24, 25, 31, 32, 33])
def test_c3_rungs_partials_and_outputs_sampled_rows(t):
    p = synth.config_matvec("c3")
    blocks = G.quantize_rows(p.w)
    x = np.concatenate([p.x, -0.5 * p.x])[:t]  # config 3 holds 32 activation rows
    assert x.shape[0] == t
    q8 = G.quantize_acts(x)
    rows = _sample_rows(p.n, t)
    ob, oq = orc.tq1_encode_rows(p.w[rows]), orc.q8_1_quantize(x)
    np.testing.assert_array_equal(G.partials(blocks, q8, p.n, p.k, t)[:, rows],
                                  orc.mmv_partials(ob, oq, rows.size, p.k, t))
    G.assert_close(G.mmv(blocks, q8, p.n, p.k, t)[:, rows], orc.mmv_f64(ob, oq, rows.size, p.k, t))


# (n, k, t): partial last M-tile, a single block per row (no K split), odd
# block counts, K ranges of unequal length, rows beyond one wave of groups.
RAGGED = [(1, 256, 8), (15, 256, 9), (17, 512, 31), (33, 768, 8), (100, 2304, 16), (129, 256 * 63, 12),
          (300, 1024, 24), (513, 6144, 32), (2000, 2048, 40), (4099, 4096, 20), (77, 256 * 7, 8)]


@pytest.mark.parametrize("n,k,t", RAGGED)
def test_ragged_shapes_all_rows(n, k, t):
    p = synth.matvec(n, k, t, p_zero=0.4, seed=n + 3 * k + t)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    ob, oq = orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x)
    np.testing.assert_array_equal(G.partials(blocks, q8, n, k, t), orc.mmv_partials(ob, oq, n, k, t))
    G.assert_close(G.mmv(blocks, q8, n, k, t), orc.mmv_f64(ob, oq, n, k, t))


def test_extreme_partials_on_the_tensor_cores():
    # All-(+1) / all-(-1) rows against q = +-127 chunks: partials of +-4064,
    # the largest a chunk can hold (the fp32 accumulator stays exact).
    k = 512
    w = np.full((20, k), np.float32(0.25))
    w[1] = -0.25
    w[2, ::2] = -0.25
    x = np.full((9, k), np.float32(5.0))
    x[1, 100:] = -5.0
    x[5] = -5.0
    blocks, q8 = G.quantize_rows(w), G.quantize_acts(x)
    part = G.partials(blocks, q8, 20, k, 9)
    np.testing.assert_array_equal(part, orc.mmv_partials(orc.tq1_encode_rows(w), orc.q8_1_quantize(x), 20, k, 9))
    assert part[0, 0, 0] == 4064 and part[0, 1, 0] == -4064 and part[5, 1, 0] == 4064


@pytest.mark.parametrize("t", [8, 16, 32])
def test_residual_add_in_place(t):
    n, k = 1000, 2048
    p = synth.matvec(n, k, t, seed=77 + t)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    res = np.random.default_rng(t).standard_normal((t, n)).astype(np.float32)
    L, torch = G.lib(), G.torch()
    r = G.dev(res)
    L.tq1_mmv_add(blocks, q8, r, r, n, k, t)
    assert L.tq1_sync_status() == 0
    ref = orc.mmv_f64(orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x), n, k, t) + res.astype(np.float64)
    G.assert_close(G.host(r), ref)


def test_deterministic_repeat():
    p = synth.matvec(5120, 6144, 32, seed=91)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    for t in (8, 16, 32):
        np.testing.assert_array_equal(G.mmv(blocks, q8, p.n, p.k, t), G.mmv(blocks, q8, p.n, p.k, t))


def _quantize_tq2(w):
    t = G.torch()
    n, k = w.shape
    blocks = t.empty(n * (k // 256) * TQ2_BYTES, dtype=t.uint8, device="cuda")
    G.lib().tq2_quantize_rows(G.dev(w.astype(np.float32)), blocks, n, k)
    return blocks


@pytest.mark.parametrize("n,k,t", [(5120, 6144, 16), (5120, 6144, 32), (17, 512, 9), (300, 2304, 8)])
def test_tq2_rungs(n, k, t):
    p = synth.matvec(n, k, t, seed=5 * n + t)
    blocks, q8 = _quantize_tq2(p.w), G.quantize_acts(p.x)
    rows = _sample_rows(n, t) if n > 1000 else np.arange(n)
    ob, oq = orc.tq2_encode_rows(p.w[rows]), orc.q8_1_quantize(p.x)
    L, torch = G.lib(), G.torch()
    part = torch.full((t, n, k // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    y = torch.full((t, n), float("nan"), dtype=torch.float32, device="cuda")
    L.tq2_mmv_partials(blocks, q8, part, n, k, t)
    L.tq2_mmv(blocks, q8, y, n, k, t)
    assert L.tq1_sync_status() == 0
    np.testing.assert_array_equal(G.host(part)[:, rows], orc.tq2_mmv_partials(ob, oq, rows.size, k, t))
    G.assert_close(G.host(y)[:, rows], orc.tq2_mmv_f64(ob, oq, rows.size, k, t))
