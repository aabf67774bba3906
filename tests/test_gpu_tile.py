"""The tcgen05 tile path (tq1_mmv_ws with a workspace, t >= its threshold) vs
the oracle: fp32 outputs within max(1e-3 |ref|, 1e-4).  The shapes pick
single and ragged row tiles, ragged 64-token tiles, several persistent tiles
per CTA, and two shapes whose row stride keeps them on the allocation-free
kernels (no workspace asked for)."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 2048, 33),      # one row, one tile: 127 zero-filled rows
    (129, 2048, 40),    # two row tiles
    (77, 6144, 48),     # 24 blocks per tile, a partial row tile
    (256, 4096, 33),    # two row tiles, 31 padding tokens
    (64, 2048, 64),
    (200, 2048, 65),    # two token tiles
    (130, 4096, 129),   # three token tiles, ragged
    (2000, 2048, 200),
    (5000, 2048, 520),  # more tiles than SMs: two tiles per CTA, accumulators reused
    (300, 10240, 40),   # k > 8192: the prep kernel reads each token's blocks twice
    (300, 1280, 40),    # row stride not a multiple of 16 bytes: no workspace, other kernels
    (1000, 768, 37),
]


@pytest.mark.parametrize("n,k,t", SHAPES)
def test_tile_shapes(n, k, t):
    p = synth.matvec(n, k, t, p_zero=0.4, seed=5 * n + k + t)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    assert (G.lib().tq1_mmv_workspace_size(n, k, t) > 0) == (k % 2048 == 0)
    y = G.mmv_ws(blocks, q8, n, k, t)
    G.assert_close(y, orc.mmv_f64(orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x), n, k, t))


def test_tile_activation_scale_extremes():
    # Tokens up to ~1e6 need the per-token power-of-two pre-scale in every
    # split; a zero token and a tiny one exercise the other end.
    p = synth.matvec(300, 2048, 40, seed=41)
    x = p.x.copy()
    x[1] *= 1e6
    x[2, :1024] *= 3e5
    x[3] = 0.0
    x[4] *= 1e-6
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(x)
    y = G.mmv_ws(blocks, q8, p.n, p.k, p.t)
    G.assert_close(y, orc.mmv_f64(orc.tq1_encode_rows(p.w), orc.q8_1_quantize(x), p.n, p.k, p.t))
    assert np.all(y[3] == 0.0)


def test_tile_deterministic_and_zero_rows():
    p = synth.matvec(700, 4096, 70, seed=42)
    w = p.w.copy()
    w[5] = 0.0
    w[600:] = 0.0
    blocks, q8 = G.quantize_rows(w), G.quantize_acts(p.x)
    a = G.mmv_ws(blocks, q8, p.n, p.k, p.t)
    b = G.mmv_ws(blocks, q8, p.n, p.k, p.t)
    np.testing.assert_array_equal(a, b)
    assert np.all(a[:, 5] == 0.0) and np.all(a[:, 600:] == 0.0)
    G.assert_close(a, orc.mmv_f64(orc.tq1_encode_rows(w), orc.q8_1_quantize(p.x), p.n, p.k, p.t))


def test_tile_config3_sampled_rows_back_to_back():
    # Several calls in a row on one stream (the next call's weight expansion
    # overlaps the previous call), alternating the tile path (with a
    # workspace) and the allocation-free rungs, sharing one workspace.
    p = synth.config_matvec("c3")
    blocks = G.quantize_rows(p.w)
    rows = np.unique(np.concatenate([[0, 127, 128, p.n - 1], np.random.default_rng(34).integers(0, p.n, 60)]))
    ob = orc.tq1_encode_rows(p.w[rows])
    L = G.lib()
    torch = G.torch()
    x = np.concatenate([p.x, p.x[:32] * 0.5])
    ws_bytes = L.tq1_mmv_workspace_size(p.n, p.k, 64)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    outs = []
    for t in (64, 7, 40, 16):
        q8 = G.quantize_acts(x[:t])
        y = torch.full((t, p.n), float("nan"), dtype=torch.float32, device="cuda")
        L.tq1_mmv_ws(blocks, q8, y, p.n, p.k, t, ws, ws_bytes)
        outs.append((t, y))
    assert L.tq1_sync_status() == 0
    for t, y in outs:
        G.assert_close(G.host(y)[:, rows], orc.mmv_f64(ob, orc.q8_1_quantize(x[:t]), rows.size, p.k, t))


def test_workspace_too_small_is_refused_before_launch():
    n, k, t = 300, 2048, 64
    p = synth.matvec(n, k, t, seed=3)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    L = G.lib()
    torch = G.torch()
    need = L.tq1_mmv_workspace_size(n, k, t)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = torch.full((t, n), 7.0, dtype=torch.float32, device="cuda")
    rc = L.library().tq1_mmv_ws(blocks.data_ptr(), q8.data_ptr(), None, y.data_ptr(), n, k, t, ws.data_ptr(),
                                need - 1, None)
    assert rc == -5  # TQ1_ERR_WORKSPACE
    assert L.tq1_sync_status() == 0
    assert np.all(G.host(y) == 7.0)  # nothing ran


@pytest.mark.parametrize("in_place", [False, True])
def test_tile_residual_epilogue(in_place):
    # y = res + W x through the tile path's epilogue (tq1_mmv_ws with res),
    # a separate residual buffer and in place (y is the residual).
    n, k, t = 200, 2048, 140
    p = synth.matvec(n, k, t, seed=303)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    res = np.random.default_rng(5).standard_normal((t, n)).astype(np.float32)
    L, torch = G.lib(), G.torch()
    ws_bytes = L.tq1_mmv_workspace_size(n, k, t)
    assert ws_bytes > 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    r = G.dev(res)
    y = r if in_place else torch.full((t, n), float("nan"), dtype=torch.float32, device="cuda")
    L.tq1_mmv_ws(blocks, q8, y, n, k, t, ws, ws_bytes, res=r)
    assert L.tq1_sync_status() == 0
    ref = orc.mmv_f64(orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x), n, k, t) + res.astype(np.float64)
    G.assert_close(G.host(y), ref)
