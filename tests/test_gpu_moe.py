"""Expert-routed mat-vec on the GPU vs the oracle."""
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


def _mmv_id(blocks, m, ids, q8, fill=float("nan")):
    L = G.lib()
    t = G.torch()
    ws_bytes = L.tq1_mmv_id_workspace_size(m.n_experts, m.t, m.top_k)
    ws = t.zeros(ws_bytes, dtype=t.uint8, device="cuda")
    y = t.full((m.t, m.top_k, m.n), fill, dtype=t.float32, device="cuda")
    L.tq1_mmv_id(blocks, m.n_experts, q8, G.dev(ids.astype(np.int32)), y, m.n, m.k, m.t, m.top_k, ws)
    return y, L.tq1_sync_status()


def _mmv_id_partials(blocks, m, ids, q8, fmt="tq1"):
    L = G.lib()
    t = G.torch()
    ws_bytes = L.tq1_mmv_id_workspace_size(m.n_experts, m.t, m.top_k)
    ws = t.zeros(ws_bytes, dtype=t.uint8, device="cuda")
    part = t.full((m.t, m.top_k, m.n, m.k // 32), -2 ** 31, dtype=t.int32, device="cuda")
    fn = L.tq1_mmv_id_partials if fmt == "tq1" else L.tq2_mmv_id_partials
    fn(blocks, m.n_experts, q8, G.dev(ids.astype(np.int32)), part, m.n, m.k, m.t, m.top_k, ws)
    assert L.tq1_sync_status() == 0
    return G.host(part)


def _oracle_id_partials(m, ids, rows, fmt="tq1"):
    """Per routed (token, slot) pair: the oracle's dense partials of that
    expert's sampled rows against the token's activations (the routed
    product reduces to per-expert mat-vecs)."""
    enc = orc.tq1_encode_rows if fmt == "tq1" else orc.tq2_encode_rows
    dense = orc.mmv_partials if fmt == "tq1" else orc.tq2_mmv_partials
    oq = orc.q8_1_quantize(m.x).reshape(m.t, -1)
    cache = {}
    out = np.zeros((m.t, m.top_k, len(rows), m.k // 32), np.int32)
    for c in range(m.t):
        for s in range(m.top_k):
            e = int(ids[c, s])
            if e not in cache:
                cache[e] = enc(m.expert_weights(e)[rows])
            out[c, s] = dense(cache[e], oq[c], len(rows), m.k, 1)[0]
    return out


def _oracle_blocks(m, experts):
    eb = m.n * (m.k // 256) * 54
    out = np.zeros((m.n_experts, eb), np.uint8)
    for e in experts:
        out[e] = orc.tq1_encode_rows(m.expert_weights(e)).reshape(-1)
    return out


@pytest.mark.parametrize("t", [1, 32])
def test_config4_sampled_rows(t):
    m = synth.config_moe(t)
    blocks = _experts_gpu(m)
    q8 = G.quantize_acts(m.x)
    y, st = _mmv_id(blocks, m, m.ids, q8)
    assert st == 0
    used = np.unique(m.ids)
    ob = _oracle_blocks(m, used)
    rows = np.unique(np.concatenate([[0, m.n - 1], np.random.default_rng(t).integers(0, m.n, 62)]))
    ref = orc.mmv_id_f64_rows(ob, m.n_experts, orc.q8_1_quantize(m.x), m.ids, m.n, m.k, m.t, m.top_k, rows)
    G.assert_close(G.host(y)[:, :, rows], ref)


@pytest.mark.parametrize("t", [1, 32])
def test_config4_partials_sampled_rows(t):
    """The routed decode kernels' own integer partials (direct mode at T=1,
    the compacted mode at T=32) against the oracle's, bit for bit."""
    m = synth.config_moe(t)
    blocks = _experts_gpu(m)
    q8 = G.quantize_acts(m.x)
    part = _mmv_id_partials(blocks, m, m.ids, q8)
    rows = np.unique(np.concatenate([[0, 1, m.n - 1], np.random.default_rng(t + 5).integers(0, m.n, 45)]))
    np.testing.assert_array_equal(part[:, :, rows], _oracle_id_partials(m, m.ids, rows))


ROUTINGS = {
    "repeated_and_unused": np.array([[0, 3], [3, 0], [3, 5], [0, 3], [5, 3]]),
    "all_on_one": np.array([[2], [2], [2], [2], [2]]),
    "top1": np.array([[1], [4], [1], [0], [6]]),
    "every_expert": np.array([[0, 1, 2, 3, 4, 5, 6], [6, 5, 4, 3, 2, 1, 0], [1, 3, 5, 0, 2, 4, 6],
                              [2, 2, 2, 2, 2, 2, 2], [0, 6, 0, 6, 0, 6, 0]]),
}


@pytest.mark.parametrize("name", sorted(ROUTINGS))
def test_small_routings_full(name):
    ids = ROUTINGS[name].astype(np.int32)
    t, top_k = ids.shape
    m = synth.moe(7, 300, 1024, t, top_k, seed=41)
    m.ids = ids
    blocks = _experts_gpu(m)
    q8 = G.quantize_acts(m.x)
    y, st = _mmv_id(blocks, m, ids, q8)
    assert st == 0
    ob = _oracle_blocks(m, range(7))
    ref = orc.mmv_id_f64(ob, 7, orc.q8_1_quantize(m.x), ids, m.n, m.k, t, top_k)
    G.assert_close(G.host(y), ref)
    part = _mmv_id_partials(blocks, m, ids, q8)
    np.testing.assert_array_equal(part, _oracle_id_partials(m, ids, np.arange(m.n)))


def test_many_tokens_one_expert_beyond_32_columns():
    m = synth.moe(4, 96, 512, 40, 2, seed=3)
    m.ids = np.stack([np.full(40, 1), np.arange(40) % 4], axis=1).astype(np.int32)
    blocks = _experts_gpu(m)
    y, st = _mmv_id(blocks, m, m.ids, G.quantize_acts(m.x))
    assert st == 0
    ref = orc.mmv_id_f64(_oracle_blocks(m, range(4)), 4, orc.q8_1_quantize(m.x), m.ids, m.n, m.k, m.t, m.top_k)
    G.assert_close(G.host(y), ref)


@pytest.mark.parametrize("fmt", ["tq1", "tq2"])
def test_grouped_tasks_ragged_rows_blocks_and_pairs(fmt):
    # 144 pairs (the compacted mode) on 9 experts, 200 rows (ragged last
    # task), 6 blocks, one expert with at least 19 pairs (several 4-pair
    # chunks and a ragged one): outputs and exact partials.
    m = synth.moe(9, 200, 1536, 48, 3, seed=88)
    ids = m.ids.copy()
    ids[:19, 0] = 4
    ids[:19, 1:] = np.where(ids[:19, 1:] == 4, 5, ids[:19, 1:])
    ids[:19, 2] = np.where(ids[:19, 2] == ids[:19, 1], (ids[:19, 1] + 1) % 9, ids[:19, 2])
    ids[:19, 2] = np.where(ids[:19, 2] == 4, 6, ids[:19, 2])
    m.ids = ids.astype(np.int32)
    q8 = G.quantize_acts(m.x)
    oq = orc.q8_1_quantize(m.x)
    if fmt == "tq1":
        blocks = _experts_gpu(m)
        y, st = _mmv_id(blocks, m, m.ids, q8)
        assert st == 0
        ref = orc.mmv_id_f64(_oracle_blocks(m, range(9)), 9, oq, m.ids, m.n, m.k, m.t, m.top_k)
        G.assert_close(G.host(y), ref)
    else:
        blocks = _experts_gpu_tq2(m)
        y = _tq2_id(blocks, m, m.ids, q8)
        ref = orc.tq2_mmv_id_f64(_oracle_blocks_tq2(m, range(9)), 9, oq, m.ids, m.n, m.k, m.t, m.top_k)
        G.assert_close(y, ref)
    part = _mmv_id_partials(blocks, m, m.ids, q8, fmt)
    np.testing.assert_array_equal(part, _oracle_id_partials(m, m.ids, np.arange(m.n), fmt))


def test_equals_per_expert_mmv():
    m = synth.moe(6, 256, 2048, 4, 3, seed=12)
    blocks = _experts_gpu(m)
    q8 = G.quantize_acts(m.x)
    y, st = _mmv_id(blocks, m, m.ids, q8)
    assert st == 0
    y = G.host(y)
    eb = m.n * 8 * 54
    for c in range(m.t):
        q1 = G.quantize_acts(m.x[c:c + 1])
        for s in range(m.top_k):
            e = int(m.ids[c, s])
            ref = G.mmv(blocks[e * eb:(e + 1) * eb], q1, m.n, m.k, 1)[0]
            G.assert_close(y[c, s], ref)


def test_bad_id_sets_status_and_skips_slot():
    m = synth.moe(5, 64, 512, 3, 2, seed=5)
    ids = m.ids.copy()
    ids[1, 0] = 9
    ids[2, 1] = -1
    blocks = _experts_gpu(m)
    y, st = _mmv_id(blocks, m, ids, G.quantize_acts(m.x), fill=123.0)
    assert st == -8
    y = G.host(y)
    assert np.all(y[1, 0] == 123.0) and np.all(y[2, 1] == 123.0)
    ref = orc.mmv_id_f64(_oracle_blocks(m, range(5)), 5, orc.q8_1_quantize(m.x), ids, m.n, m.k, m.t, m.top_k)
    ok = ~np.isnan(ref)
    G.assert_close(y[ok], ref[ok])
    assert G.lib().tq1_sync_status() == 0  # cleared


def test_deterministic_repeat():
    m = synth.config_moe(32)
    blocks = _experts_gpu(m)
    q8 = G.quantize_acts(m.x)
    a, _ = _mmv_id(blocks, m, m.ids, q8)
    b, _ = _mmv_id(blocks, m, m.ids, q8)
    np.testing.assert_array_equal(G.host(a), G.host(b))


@pytest.mark.parametrize("t,top_k,n_experts", [(1, 8, 16), (3, 4, 6), (40, 2, 5), (70, 2, 5)])
def test_per_slot_activations(t, top_k, n_experts):
    # One activation row per (token, slot): direct mode (few pairs) and the
    # compacted path (80 pairs).
    m = synth.moe(n_experts, 160, 1024, t, top_k, seed=9 + t)
    blocks = _experts_gpu(m)
    x = np.random.default_rng(t).standard_normal((t * top_k, m.k)).astype(np.float32)
    q8 = G.quantize_acts(x)
    L, torch = G.lib(), G.torch()
    ws_bytes = L.tq1_mmv_id_workspace_size(m.n_experts, t, top_k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    y = torch.full((t, top_k, m.n), float("nan"), dtype=torch.float32, device="cuda")
    L.tq1_mmv_id_slots(blocks, m.n_experts, q8, G.dev(m.ids.astype(np.int32)), y, m.n, m.k, t, top_k, ws)
    assert L.tq1_sync_status() == 0
    ob = _oracle_blocks(m, np.unique(m.ids))
    oq = orc.q8_1_quantize(x).reshape(t * top_k, -1)
    ref = np.zeros((t, top_k, m.n))
    for c in range(t):
        for s in range(top_k):
            e = int(m.ids[c, s])
            ref[c, s] = orc.mmv_f64(ob[e], oq[c * top_k + s], m.n, m.k, 1)[0]
    G.assert_close(G.host(y), ref)


# ------------------------------------------------------------------ TQ2_0 --
def _experts_gpu_tq2(m):
    t = G.torch()
    eb = m.n * (m.k // 256) * 66
    blocks = t.empty(m.n_experts * eb, dtype=t.uint8, device="cuda")
    for e in range(m.n_experts):
        w = G.dev(m.expert_weights(e).astype(np.float32))
        G.lib().tq2_quantize_rows(w, blocks[e * eb:(e + 1) * eb], m.n, m.k)
    return blocks


def _oracle_blocks_tq2(m, experts):
    eb = m.n * (m.k // 256) * 66
    out = np.zeros((m.n_experts, eb), np.uint8)
    for e in experts:
        out[e] = orc.tq2_encode_rows(m.expert_weights(e)).reshape(-1)
    return out


def _tq2_id(blocks, m, ids, q8, slots=False, t=None):
    L, torch = G.lib(), G.torch()
    t = m.t if t is None else t
    ws_bytes = L.tq1_mmv_id_workspace_size(m.n_experts, t, m.top_k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    y = torch.full((t, m.top_k, m.n), float("nan"), dtype=torch.float32, device="cuda")
    fn = L.tq2_mmv_id_slots if slots else L.tq2_mmv_id
    fn(blocks, m.n_experts, q8, G.dev(ids.astype(np.int32)), y, m.n, m.k, t, m.top_k, ws)
    assert L.tq1_sync_status() == 0
    return G.host(y)


@pytest.mark.parametrize("t", [1, 32])
def test_tq2_config4_sampled_rows(t):
    # Direct mode (t = 1: 8 pairs) and the compacted path (t = 32: 256 pairs).
    m = synth.config_moe(t)
    blocks = _experts_gpu_tq2(m)
    q8 = G.quantize_acts(m.x)
    y = _tq2_id(blocks, m, m.ids, q8)
    ob = _oracle_blocks_tq2(m, np.unique(m.ids))
    ref = orc.tq2_mmv_id_f64(ob, m.n_experts, orc.q8_1_quantize(m.x), m.ids, m.n, m.k, m.t, m.top_k)
    G.assert_close(y, ref)
    part = _mmv_id_partials(blocks, m, m.ids, q8, fmt="tq2")
    rows = np.unique(np.concatenate([[0, m.n - 1], np.random.default_rng(t + 9).integers(0, m.n, 30)]))
    np.testing.assert_array_equal(part[:, :, rows], _oracle_id_partials(m, m.ids, rows, fmt="tq2"))


def test_tq2_routings_long_rows():
    # Repeated, unused and all-expert routings with long rows (k = 256 * 63,
    # 4158 bytes per TQ2_0 row).
    for ids in (ROUTINGS["repeated_and_unused"], ROUTINGS["every_expert"]):
        ids = ids.astype(np.int32)
        t, top_k = ids.shape
        m = synth.moe(7, 40, 256 * 63, t, top_k, seed=43)
        m.ids = ids
        y = _tq2_id(_experts_gpu_tq2(m), m, ids, G.quantize_acts(m.x))
        ref = orc.tq2_mmv_id_f64(_oracle_blocks_tq2(m, range(7)), 7, orc.q8_1_quantize(m.x), ids, m.n, m.k, t, top_k)
        G.assert_close(y, ref)


@pytest.mark.parametrize("t,top_k,n_experts", [(1, 8, 16), (40, 2, 5)])
def test_tq2_per_slot_activations(t, top_k, n_experts):
    m = synth.moe(n_experts, 160, 1024, t, top_k, seed=19 + t)
    x = np.random.default_rng(t + 5).standard_normal((t * top_k, m.k)).astype(np.float32)
    y = _tq2_id(_experts_gpu_tq2(m), m, m.ids, G.quantize_acts(x), slots=True)
    ob = _oracle_blocks_tq2(m, np.unique(m.ids))
    oq = orc.q8_1_quantize(x).reshape(t * top_k, -1)
    ref = np.zeros((t, top_k, m.n))
    for c in range(t):
        for s in range(top_k):
            e = int(m.ids[c, s])
            ref[c, s] = orc.tq2_mmv_f64(ob[e], oq[c * top_k + s], m.n, m.k, 1)[0]
    G.assert_close(y, ref)


def test_large_expert_count_runs_the_compaction_kernel():
    # 1100 experts: the routing table (four words per expert plus one per
    # pair) is larger than the routed kernel builds in shared memory, so the
    # compaction kernel writes it into the workspace first; 160 pairs take the
    # compacted mode.  Outputs and exact partials against the oracle.
    m = synth.moe(1100, 64, 512, 80, 2, seed=77)
    t_ = G.torch()
    eb = m.n * (m.k // 256) * 54
    used = np.unique(m.ids)
    blocks = t_.zeros(m.n_experts * eb, dtype=t_.uint8, device="cuda")
    for e in used:
        blocks[e * eb:(e + 1) * eb] = G.quantize_rows(m.expert_weights(int(e)))
    q8 = G.quantize_acts(m.x)
    y, st = _mmv_id(blocks, m, m.ids, q8)
    assert st == 0
    ob = _oracle_blocks(m, used)
    G.assert_close(G.host(y), orc.mmv_id_f64(ob, m.n_experts, orc.q8_1_quantize(m.x), m.ids, m.n, m.k, m.t, m.top_k))
    rows = np.arange(m.n)
    np.testing.assert_array_equal(_mmv_id_partials(blocks, m, m.ids, q8), _oracle_id_partials(m, m.ids, rows))
