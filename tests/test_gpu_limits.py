"""Sizes at the library's limits and degenerate shapes, every route, against
the oracle (integer partials bit-exact, fp32 outputs within max(1e-3 |ref|,
1e-4)): the largest accepted K (62720 = 245 blocks: the rungs' staging does
not fit, so calls fall back to the kernels that can stage it), a single row
on every route, column counts past 32 (slices) and past 64 (several token
tiles of the tile path), and single-expert routing."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

K_MAX = 62720


@pytest.mark.parametrize("t", [1, 4, 8, 16, 32])
def test_largest_k(t):
    n = 37
    p = synth.matvec(n, K_MAX, t, p_zero=0.4, seed=1000 + t)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    ob, oq = orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x)
    np.testing.assert_array_equal(G.partials(blocks, q8, n, K_MAX, t), orc.mmv_partials(ob, oq, n, K_MAX, t))
    G.assert_close(G.mmv(blocks, q8, n, K_MAX, t), orc.mmv_f64(ob, oq, n, K_MAX, t))


@pytest.mark.parametrize("t", [1, 2, 5, 8, 9, 24, 33, 70])
def test_single_row_every_route(t):
    k = 2048
    p = synth.matvec(1, k, t, seed=2000 + t)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    ob, oq = orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x)
    ref = orc.mmv_f64(ob, oq, 1, k, t)
    np.testing.assert_array_equal(G.partials(blocks, q8, 1, k, t), orc.mmv_partials(ob, oq, 1, k, t))
    G.assert_close(G.mmv(blocks, q8, 1, k, t), ref)
    G.assert_close(G.mmv_ws(blocks, q8, 1, k, t), ref)


@pytest.mark.parametrize("n,k,t", [(333, 4096, 100), (70, 2048, 193)])
def test_many_columns_both_entries(n, k, t):
    # tq1_mmv: 32-column slices of the tensor-core rungs (a ragged last slice);
    # tq1_mmv_ws: the tcgen05 tile path, several 64-token tiles, a ragged last one.
    p = synth.matvec(n, k, t, p_zero=0.4, seed=n + t)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    ob, oq = orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x)
    ref = orc.mmv_f64(ob, oq, n, k, t)
    np.testing.assert_array_equal(G.partials(blocks, q8, n, k, t), orc.mmv_partials(ob, oq, n, k, t))
    G.assert_close(G.mmv(blocks, q8, n, k, t), ref)
    G.assert_close(G.mmv_ws(blocks, q8, n, k, t), ref)


@pytest.mark.parametrize("t,top_k", [(1, 1), (40, 1), (3, 4)])
def test_single_expert(t, top_k):
    # One expert holds every (token, slot) pair, the same expert repeated in a
    # token's slots included: the direct mode for few pairs, the compacted
    # mode above 32.  (The synthetic routing draws distinct experts, so the
    # draw uses top_k experts and the ids are then all set to expert 0.)
    m = synth.moe(top_k, 200, 1024, t, top_k, seed=50 + t)
    ids = np.zeros((t, top_k), np.int32)
    torch = G.torch()
    w0 = m.expert_weights(0)
    blocks = G.quantize_rows(w0)
    q8 = G.quantize_acts(m.x)
    L = G.lib()
    ws = torch.zeros(L.tq1_mmv_id_workspace_size(1, t, top_k), dtype=torch.uint8, device="cuda")
    y = torch.full((t, top_k, m.n), float("nan"), dtype=torch.float32, device="cuda")
    L.tq1_mmv_id(blocks, 1, q8, G.dev(ids), y, m.n, m.k, t, top_k, ws)
    assert L.tq1_sync_status() == 0
    ob = orc.tq1_encode_rows(w0).reshape(1, -1)
    G.assert_close(G.host(y), orc.mmv_id_f64(ob, 1, orc.q8_1_quantize(m.x), ids, m.n, m.k, t, top_k))
