"""tq1_mmv_id_noalloc: the expert-routed mat-vec for callers that cannot
allocate device memory (stream-capture regions, fixed memory budgets,
latency-critical loops, plain C callers without an allocator).  Its routing
table lives in a fixed array inside the library instead of a caller
workspace.

Checked through the C ABI against tq1_mmv_id (which takes a workspace) and
against the oracle's per-slot products, on two calls in a row with different
routings.  Both calls route more than 32
(token, slot) pairs, so they go through the compacted routing table that the
fixed array holds (fewer pairs are served without a table); the second call
routes to fewer experts than the first, so a table left over from the first
call cannot leak into the second unnoticed.  A decode-sized call (no table)
follows.  This file is collected last on purpose."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _experts_gpu(m):
    t = G.torch()
    eb = m.n * (m.k // 256) * 54
    blocks = t.empty(m.n_experts * eb, dtype=t.uint8, device="cuda")
    for e in range(m.n_experts):
        blocks[e * eb:(e + 1) * eb] = G.quantize_rows(m.expert_weights(e))
    return blocks


def _with_workspace(L, blocks, m, q8, ids, t_tok):
    t = G.torch()
    ws_bytes = L.tq1_mmv_id_workspace_size(m.n_experts, t_tok, m.top_k)
    ws = t.zeros(ws_bytes, dtype=t.uint8, device="cuda")
    y = t.full((t_tok, m.top_k, m.n), float("nan"), dtype=t.float32, device="cuda")
    L.tq1_mmv_id(blocks, m.n_experts, q8, ids, y, m.n, m.k, t_tok, m.top_k, ws)
    assert L.tq1_sync_status() == 0
    return G.host(y)


def _no_alloc(L, blocks, m, q8, ids, t_tok):
    t = G.torch()
    y = t.full((t_tok, m.top_k, m.n), float("nan"), dtype=t.float32, device="cuda")
    L.tq1_mmv_id_noalloc(blocks, m.n_experts, q8, ids, y, m.n, m.k, t_tok, m.top_k)
    assert L.tq1_sync_status() == 0
    return G.host(y)


def test_no_alloc_matches_workspace_entry_on_two_calls():
    L = G.lib()
    m = synth.moe(n_experts=24, n=320, k=1024, t=12, top_k=4, seed=31)
    assert m.t * m.top_k > 32  # the routing-table path
    blocks = _experts_gpu(m)
    q8 = G.quantize_acts(m.x)
    oq = orc.q8_1_quantize(m.x)
    ob = np.stack([orc.tq1_encode_rows(m.expert_weights(e)).reshape(-1) for e in range(m.n_experts)])
    first = m.ids.astype(np.int32)
    # Second call: only seven experts, each token's four ids distinct.
    second = np.array([[c % 3, 3 + c % 2, 5, 6] for c in range(m.t)], dtype=np.int32)
    assert all(len(set(row)) == m.top_k for row in second)
    assert len(np.unique(second)) < len(np.unique(first))
    for ids_np in (first, second):
        ids = G.dev(ids_np)
        ref = _with_workspace(L, blocks, m, q8, ids, m.t)
        got = _no_alloc(L, blocks, m, q8, ids, m.t)
        assert np.isfinite(got).all()
        G.assert_close(got, ref)
        G.assert_close(got, orc.mmv_id_f64(ob, m.n_experts, oq, ids_np, m.n, m.k, m.t, m.top_k))
    # A decode-sized call (one token, 4 pairs) after the table-sized ones.
    q8_1 = G.quantize_acts(m.x[:1])
    ids = G.dev(first[:1].copy())
    G.assert_close(_no_alloc(L, blocks, m, q8_1, ids, 1), _with_workspace(L, blocks, m, q8_1, ids, 1))
