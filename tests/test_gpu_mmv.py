"""Mat-vec on the GPU vs the oracle: exact integer partials, fp32 outputs
within max(1e-3 |ref|, 1e-4), layout probes, ladder consistency and
determinism.  Full-size workloads are checked on sampled rows."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _run(p):
    blocks = G.quantize_rows(p.w)
    q8 = G.quantize_acts(p.x)
    return blocks, q8


def _oracle(p):
    return orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x)


# Small shapes spanning several passes (256 units each), several CTAs and
# ragged tails: all outputs compared.
SMALL = [
    (1, 256, 1), (3, 256, 2), (7, 512, 3), (33, 1024, 1), (256, 1024, 1), (100, 2048, 4),
    (77, 6144, 5), (301, 768 * 4, 8), (64, 4096, 16), (130, 2048, 32), (45, 256 * 9, 31),
    (17, 6144, 2), (1000, 512, 1), (5, 256 * 63, 1),
    # the 8-column decode rung (t = 5): one row and block, long K (records
    # beyond the two-CTA budget), ragged rows
    (1, 256, 5), (9, 256 * 63, 5), (130, 2304, 5),
    # the one-n-tile tensor-core rung below and at 8 columns
    (1, 256, 8), (9, 256 * 63, 6), (130, 2304, 7),
]


@pytest.mark.parametrize("n,k,t", SMALL)
def test_partials_bit_exact_small(n, k, t):
    p = synth.matvec(n, k, t, seed=n + k + t)
    blocks, q8 = _run(p)
    ob, oq = _oracle(p)
    np.testing.assert_array_equal(G.partials(blocks, q8, n, k, t), orc.mmv_partials(ob, oq, n, k, t))


@pytest.mark.parametrize("n,k,t", SMALL)
def test_mmv_small(n, k, t):
    p = synth.matvec(n, k, t, p_zero=0.4, seed=2 * n + k + t)
    blocks, q8 = _run(p)
    ob, oq = _oracle(p)
    G.assert_close(G.mmv(blocks, q8, n, k, t), orc.mmv_f64(ob, oq, n, k, t))


def test_config1_full():
    p = synth.config_matvec("c1")
    blocks, q8 = _run(p)
    ob, oq = _oracle(p)
    G.assert_close(G.mmv(blocks, q8, p.n, p.k, p.t), orc.mmv_f64(ob, oq, p.n, p.k, p.t))
    np.testing.assert_array_equal(G.partials(blocks, q8, p.n, p.k, p.t), orc.mmv_partials(ob, oq, p.n, p.k, p.t))


def test_config2_full():
    p = synth.config_matvec("c2")
    blocks, q8 = _run(p)
    ob, oq = _oracle(p)
    G.assert_close(G.mmv(blocks, q8, p.n, p.k, p.t), orc.mmv_f64(ob, oq, p.n, p.k, p.t))
    np.testing.assert_array_equal(G.partials(blocks, q8, p.n, p.k, p.t), orc.mmv_partials(ob, oq, p.n, p.k, p.t))


def test_config3_every_t_sampled_rows():
    p = synth.config_matvec("c3")
    blocks = G.quantize_rows(p.w)
    rng = np.random.default_rng(33)
    rows = np.unique(np.concatenate([[0, 1, p.n - 1], rng.integers(0, p.n, 125)]))
    ob = orc.tq1_encode_rows(p.w[rows])  # the oracle encodes only the sampled rows
    for t in range(1, 33):
        x = p.x[:t]
        q8 = G.quantize_acts(x)
        y = G.mmv(blocks, q8, p.n, p.k, t)
        ref = orc.mmv_f64(ob, orc.q8_1_quantize(x), rows.size, p.k, t)
        G.assert_close(y[:, rows], ref)


def _cta_rows(n, ctas=152):
    """Rows of a few whole CTAs (first, middle, last) of the decode kernel's
    one-CTA-per-SM split, plus their neighbours."""
    bounds = [(n * i) // ctas for i in range(ctas + 1)]
    out = []
    for i in (0, 1, ctas // 2, ctas - 1):
        out.extend(range(bounds[i], bounds[i + 1]))
    return np.unique(np.array(out))


def test_decode_rungs_several_rounds_sampled_rows():
    """N=5700, K=6144: a CTA holds 37 or 38 rows, more than the 8-column rung's
    weight slab takes at once (36 rows: a second round) and more tasks than
    the 2-column rung's warps pre-expand (30 > 28: tasks expanded after the
    wait); the last 4-row group holds one or two rows (a paired lane whose
    second row is missing).  Every rung, whole CTAs compared with the oracle."""
    p = synth.matvec(5700, 6144, 8, p_zero=0.4, seed=57)
    blocks = G.quantize_rows(p.w)
    rows = _cta_rows(p.n)
    ob = orc.tq1_encode_rows(p.w[rows])
    for t in (1, 2, 3, 4, 6, 8):
        x = p.x[:t]
        q8 = G.quantize_acts(x)
        y = G.mmv(blocks, q8, p.n, p.k, t)
        G.assert_close(y[:, rows], orc.mmv_f64(ob, orc.q8_1_quantize(x), rows.size, p.k, t))


def test_config3_partials_t32_sampled_rows():
    p = synth.config_matvec("c3")
    blocks, q8 = _run(p)
    rows = np.arange(0, p.n, 97)
    part = G.partials(blocks, q8, p.n, p.k, 32)
    ref = orc.mmv_partials(orc.tq1_encode_rows(p.w[rows]), orc.q8_1_quantize(p.x), rows.size, p.k, 32)
    np.testing.assert_array_equal(part[:, rows], ref)


def test_columns_beyond_32_use_slices():
    p = synth.matvec(90, 1024, 75, seed=75)
    blocks, q8 = _run(p)
    ob, oq = _oracle(p)
    G.assert_close(G.mmv(blocks, q8, p.n, p.k, p.t), orc.mmv_f64(ob, oq, p.n, p.k, p.t))
    np.testing.assert_array_equal(G.partials(blocks, q8, p.n, p.k, p.t), orc.mmv_partials(ob, oq, p.n, p.k, p.t))


def test_extreme_partials():
    w = np.full((3, 512), np.float32(0.25))
    w[1] = -0.25
    w[2, ::2] = -0.25
    x = np.full((2, 512), np.float32(5.0))
    x[1, 100:] = -5.0
    blocks, q8 = G.quantize_rows(w), G.quantize_acts(x)
    part = G.partials(blocks, q8, 3, 512, 2)
    np.testing.assert_array_equal(part, orc.mmv_partials(orc.tq1_encode_rows(w), orc.q8_1_quantize(x), 3, 512, 2))
    assert part[0, 0, 0] == 4064 and part[0, 1, 0] == -4064


def _one_hot_columns(k, cols):
    x = np.zeros((len(cols), k), np.float32)
    x[np.arange(len(cols)), cols] = 1.0
    return x


# Layout probes on every route: weight row e holds +1 at element e and zeros
# elsewhere; activation column c is one-hot at element e'_c.  y[c][e] != 0
# exactly when e == e'_c, and (where partials exist) the only nonzero partial
# of row e'_c is 127 at chunk e'_c / 32.  A transposed element order, a wrong
# digit or a chunk mapped to the wrong activation word fails these.
# (k, t, cols): k = 256 with t = 32 runs the general kernel (k not a multiple
# of 2048); k = 2048 with t <= 5 the decode rungs, with t >= 6 the
# tensor-core rungs.  cols: every element of the first and the last block.
ONE_HOT = [(256, 32, range(256)), (2048, 1, list(range(0, 256, 5)) + list(range(1792, 2048, 7))),
           (2048, 2, list(range(256)) + list(range(1792, 2048))), (2048, 4, range(0, 256, 3)),
           (2048, 5, list(range(256)) + list(range(1792, 2048))), (2048, 6, list(range(256)) + list(range(1792, 2048))),
           (2048, 8, list(range(256)) + list(range(1792, 2048))), (2048, 32, list(range(256)) + list(range(1792, 2048)))]


@pytest.mark.parametrize("k,t,cols", ONE_HOT, ids=[f"k{k}-t{t}" for k, t, _ in ONE_HOT])
def test_one_hot_layout_probes(k, t, cols):
    cols = np.array(list(cols))
    cols = np.concatenate([cols, cols[:(-len(cols)) % t]])  # whole groups of t columns
    w = np.eye(k, dtype=np.float32)
    blocks = G.quantize_rows(w)
    for g in range(0, len(cols), t):
        cg = cols[g:g + t]
        q8 = G.quantize_acts(_one_hot_columns(k, cg))
        y = G.mmv(blocks, q8, k, k, t)
        expect = np.zeros((t, k), bool)
        expect[np.arange(t), cg] = True
        np.testing.assert_array_equal(y != 0, expect)
        if t <= 8 or k % 2048 == 0:
            part = G.partials(blocks, q8, k, k, t)
            ref = np.zeros_like(part)
            ref[np.arange(t), cg, cg // 32] = 127
            np.testing.assert_array_equal(part, ref)


def test_decode_kernel_partials_c3_whole_ctas():
    """The integer partials of the kernels tq1_mmv runs (the decode kernel's
    rungs, pair mode included, at t = 1..5; the one-n-tile tensor-core rung
    at 6..8) against the oracle's, bit for bit, on whole decode-kernel CTAs
    of config 3's shape (N=5120, K=6144)."""
    p = synth.config_matvec("c3")
    blocks = G.quantize_rows(p.w)
    rows = _cta_rows(p.n)
    ob = orc.tq1_encode_rows(p.w[rows])
    for t in range(1, 9):
        x = p.x[:t]
        q8 = G.quantize_acts(x)
        part = G.partials(blocks, q8, p.n, p.k, t)
        np.testing.assert_array_equal(part[:, rows], orc.mmv_partials(ob, orc.q8_1_quantize(x), rows.size, p.k, t))


def test_decode_kernel_partials_several_rounds():
    """Partials through the decode kernel where a CTA's rows take a second
    slab round and a paired lane has no second row (N=5700, K=6144)."""
    p = synth.matvec(5700, 6144, 8, p_zero=0.4, seed=58)
    blocks = G.quantize_rows(p.w)
    rows = _cta_rows(p.n)
    ob = orc.tq1_encode_rows(p.w[rows])
    for t in (1, 2, 3, 5, 8):
        x = p.x[:t]
        q8 = G.quantize_acts(x)
        part = G.partials(blocks, q8, p.n, p.k, t)
        np.testing.assert_array_equal(part[:, rows], orc.mmv_partials(ob, orc.q8_1_quantize(x), rows.size, p.k, t))


@pytest.mark.parametrize("t", [2, 3, 4, 8, 32])
def test_multi_column_equals_single_columns(t):
    # strata PR #1418 method: a multi-column call equals single-column calls.
    # Integer partials always bit-exact; fp32 outputs within the float
    # tolerance (t = 1 runs the dp4a decode kernel, t >= 6 the tensor-core
    # rungs, whose accumulation orders differ).
    p = synth.matvec(5120, 6144, t, seed=8)
    blocks, q8 = _run(p)
    y = G.mmv(blocks, q8, p.n, p.k, t)
    part = G.partials(blocks, q8, p.n, p.k, t)
    for c in range(t):
        q1 = G.quantize_acts(p.x[c:c + 1])
        np.testing.assert_array_equal(G.partials(blocks, q1, p.n, p.k, 1)[0], part[c])
        G.assert_close(y[c], G.mmv(blocks, q1, p.n, p.k, 1)[0])


def test_deterministic_repeat():
    p = synth.matvec(5120, 6144, 3, seed=9)
    blocks, q8 = _run(p)
    a = G.mmv(blocks, q8, p.n, p.k, 3)
    b = G.mmv(blocks, q8, p.n, p.k, 3)
    np.testing.assert_array_equal(a, b)


def test_empty_is_noop():
    L = G.lib()
    L.tq1_mmv(0, 0, 0, 0, 256, 1)
    L.tq1_mmv(0, 0, 0, 7, 256, 0)
    assert L.tq1_sync_status() == 0


@pytest.mark.parametrize("n,k,t", [(300, 2048, 1), (5120, 6144, 2), (77, 1024, 4), (257, 2048, 5), (129, 4096, 9),
                                   (300, 2048, 40)])
def test_mmv_add_residual(n, k, t):
    # Every route (decode rungs, general kernel, tile path with split-K and
    # persistent tiles): y = res + W x, separately and in place.
    p = synth.matvec(n, k, t, p_zero=0.4, seed=n + 7 * t)
    blocks, q8 = G.quantize_rows(p.w), G.quantize_acts(p.x)
    res = np.random.default_rng(t).standard_normal((t, n)).astype(np.float32)
    L, torch = G.lib(), G.torch()
    y = torch.full((t, n), float("nan"), dtype=torch.float32, device="cuda")
    r = G.dev(res)
    L.tq1_mmv_add(blocks, q8, r, y, n, k, t)
    ref = orc.mmv_f64(orc.tq1_encode_rows(p.w), orc.q8_1_quantize(p.x), n, k, t) + res.astype(np.float64)
    G.assert_close(G.host(y), ref)
    L.tq1_mmv_add(blocks, q8, r, r, n, k, t)  # in place
    np.testing.assert_array_equal(G.host(r), G.host(y))
    assert L.tq1_sync_status() == 0


@pytest.mark.parametrize("n,k,t", [(5120, 6144, 1), (300, 2048, 2), (77, 1024, 3), (129, 4096, 4), (1, 256, 1)])
def test_mmv_f32_fused_quantisation_matches_two_step(n, k, t):
    # Quantisation inside the decode kernel gives the records, hence the
    # outputs, of q8_1_quantize_acts followed by tq1_mmv, bit for bit; the
    # activations include an all-zero chunk and ties.
    p = synth.matvec(n, k, t, p_zero=0.4, seed=3 * n + t)
    x = p.x.copy()
    x[0, :32] = 0.0
    x[-1, -32:] = np.arange(32, dtype=np.float32) - 15.5
    blocks = G.quantize_rows(p.w)
    L, torch = G.lib(), G.torch()
    y1 = torch.full((t, n), float("nan"), dtype=torch.float32, device="cuda")
    y2 = torch.full((t, n), float("nan"), dtype=torch.float32, device="cuda")
    xd = G.dev(x)
    L.tq1_mmv_f32(blocks, xd, y1, n, k, t)
    L.tq1_mmv(blocks, G.quantize_acts(x), y2, n, k, t)
    assert L.tq1_sync_status() == 0
    # the same decode kernel on the same records: bitwise
    np.testing.assert_array_equal(G.host(y1), G.host(y2))
    for c in range(t):  # each column equals its own one-column two-step call, bitwise
        y3 = torch.full((1, n), float("nan"), dtype=torch.float32, device="cuda")
        L.tq1_mmv(blocks, G.quantize_acts(x[c:c + 1]), y3, n, k, 1)
        y4 = torch.full((1, n), float("nan"), dtype=torch.float32, device="cuda")
        L.tq1_mmv_f32(blocks, G.dev(x[c:c + 1]), y4, n, k, 1)
        np.testing.assert_array_equal(G.host(y3), G.host(y4))
    G.assert_close(G.host(y1), orc.mmv_f64(orc.tq1_encode_rows(p.w), orc.q8_1_quantize(x), n, k, t))


def test_bounded_wait_timeout_reports_status_and_recovers():
    # Failure detection without a GPU fault: the test hook makes one CTA skip
    # a weight copy, its bounded waits give up (about 2 s each), the call
    # reports TQ1_ERR_TIMEOUT through the status word, and the next call on
    # the same context is correct.
    n, k = 640, 2048
    p = synth.matvec(n, k, 1, seed=31)
    blocks, q8 = _run(p)
    L = G.lib()
    L.library().tq1_debug_inject_wait_timeout()
    torch = G.torch()
    y = torch.zeros((1, n), dtype=torch.float32, device="cuda")
    L.tq1_mmv(blocks, q8, y, n, k, 1)
    assert L.tq1_sync_status() == -7  # TQ1_ERR_TIMEOUT
    ob, oq = _oracle(p)
    G.assert_close(G.mmv(blocks, q8, n, k, 1), orc.mmv_f64(ob, oq, n, k, 1))
