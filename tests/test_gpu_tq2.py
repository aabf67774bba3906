"""TQ2_0 (2-bit ternary codes) on the GPU vs the oracle: encoder bytes
bit-exact, integer partials bit-exact, fp32 outputs within max(1e-3 |ref|,
1e-4), over the decode kernel (t = 1 and the fused-quantisation entry), the
tensor-core rungs (t >= 6), the tcgen05 tile path (tq2_mmv_ws with a
workspace) and the full-size decode and prefill shapes (sampled rows)."""
import numpy as np
import pytest

from oracle import oracle as orc
from bit_quantized_gemv_tq1_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

TQ2_BYTES = 66


def _quantize_tq2(w):
    t = G.torch()
    n, k = w.shape
    blocks = t.empty(n * (k // 256) * TQ2_BYTES, dtype=t.uint8, device="cuda")
    G.lib().tq2_quantize_rows(G.dev(w.astype(np.float32)), blocks, n, k)
    return blocks


def _mmv(blocks, q8, n, k, t):
    tt = G.torch()
    y = tt.full((t, n), float("nan"), dtype=tt.float32, device="cuda")
    G.lib().tq2_mmv(blocks, q8, y, n, k, t)
    assert G.lib().tq1_sync_status() == 0
    return G.host(y)


def _partials(blocks, q8, n, k, t):
    tt = G.torch()
    p = tt.full((t, n, k // 32), -2 ** 31, dtype=tt.int32, device="cuda")
    G.lib().tq2_mmv_partials(blocks, q8, p, n, k, t)
    assert G.lib().tq1_sync_status() == 0
    return G.host(p)


SHAPES = [
    (1, 256, 1), (3, 256, 2), (7, 512, 3), (33, 1024, 4), (256, 1024, 1), (100, 2048, 4),
    (77, 6144, 5), (301, 768 * 4, 8), (64, 4096, 16), (130, 2048, 32), (45, 256 * 9, 33),
    (17, 6144, 2), (1000, 512, 1), (5, 256 * 63, 1), (299, 2304, 2),
    (1, 256, 8), (9, 256 * 63, 6), (130, 2304, 7),
]


@pytest.mark.parametrize("n,k", [(1, 256), (7, 512), (300, 2048), (129, 6144)])
def test_encoder_bytes_bit_exact(n, k):
    p = synth.matvec(n, k, 1, p_zero=0.4, seed=n * 7 + k)
    got = G.host(_quantize_tq2(p.w)).reshape(n, k // 256, TQ2_BYTES)
    np.testing.assert_array_equal(got, orc.tq2_encode_rows(p.w))


def test_encoder_rounding_and_zero_blocks():
    # Values at the rounding boundary (|w| = amax / 2 rounds away from zero),
    # a zero block, and one-hot blocks.
    w = np.zeros((3, 512), dtype=np.float32)
    w[0, :256] = np.linspace(-1.0, 1.0, 256, dtype=np.float32)
    w[0, 7] = 0.5
    w[0, 8] = -0.5
    w[2, 300] = -3.0
    got = G.host(_quantize_tq2(w)).reshape(3, 2, TQ2_BYTES)
    np.testing.assert_array_equal(got, orc.tq2_encode_rows(w))


@pytest.mark.parametrize("n,k,t", SHAPES)
def test_partials_bit_exact(n, k, t):
    p = synth.matvec(n, k, t, seed=n + k + t)
    blocks, q8 = _quantize_tq2(p.w), G.quantize_acts(p.x)
    ref = orc.tq2_mmv_partials(orc.tq2_encode_rows(p.w), orc.q8_1_quantize(p.x), n, k, t)
    np.testing.assert_array_equal(_partials(blocks, q8, n, k, t), ref)


@pytest.mark.parametrize("n,k,t", SHAPES)
def test_mmv(n, k, t):
    p = synth.matvec(n, k, t, p_zero=0.4, seed=2 * n + k + t)
    blocks, q8 = _quantize_tq2(p.w), G.quantize_acts(p.x)
    ref = orc.tq2_mmv_f64(orc.tq2_encode_rows(p.w), orc.q8_1_quantize(p.x), n, k, t)
    G.assert_close(_mmv(blocks, q8, n, k, t), ref)


def test_same_trits_as_tq1_give_the_same_outputs():
    # Both formats hold the same trits and scales for the same weights, and
    # both kernels sum exact integer partials in the same per-block order.
    p = synth.matvec(640, 2048, 2, seed=5)
    q8 = G.quantize_acts(p.x)
    y1 = G.mmv(G.quantize_rows(p.w), q8, 640, 2048, 2)
    y2 = _mmv(_quantize_tq2(p.w), q8, 640, 2048, 2)
    G.assert_close(y2, y1, rtol=1e-5, atol=1e-6)


def test_unused_code_three():
    # Code 3 is never written by the encoder; it decodes to +2 (oracle).
    n, k = 5, 512
    rng = np.random.default_rng(9)
    raw = rng.integers(0, 256, size=(n, k // 256, TQ2_BYTES), dtype=np.uint8)
    raw[:, :, 64:66] = np.frombuffer(np.float16(0.03125).tobytes(), dtype=np.uint8)
    x = synth.matvec(1, k, 2, seed=1).x
    q8 = G.quantize_acts(x)
    oq = orc.q8_1_quantize(x)
    blocks = G.dev(raw.reshape(-1))
    np.testing.assert_array_equal(_partials(blocks, q8, n, k, 2), orc.tq2_mmv_partials(raw, oq, n, k, 2))
    G.assert_close(_mmv(blocks, q8, n, k, 2), orc.tq2_mmv_f64(raw, oq, n, k, 2))


def test_decode_workload_full_size_sampled_rows():
    # N=5120, K=6144 (the decode workload) at t = 1, 2, 4, 8: all outputs of
    # the GPU call, sampled rows against the oracle.
    p = synth.config_matvec("c2")
    blocks = _quantize_tq2(p.w)
    rng = np.random.default_rng(21)
    rows = np.unique(np.concatenate([[0, 1, p.n - 1], rng.integers(0, p.n, 125)]))
    ob = orc.tq2_encode_rows(p.w[rows])
    xs = synth.matvec(1, p.k, 8, seed=77).x
    for t in (1, 2, 4, 8):
        x = xs[:t]
        y = _mmv(blocks, G.quantize_acts(x), p.n, p.k, t)
        G.assert_close(y[:, rows], orc.tq2_mmv_f64(ob, orc.q8_1_quantize(x), rows.size, p.k, t))


def test_decode_rungs_several_rounds_sampled_rows():
    """TQ2_0 on the decode rungs where a CTA's rows need a second slab round
    or tasks expanded after the wait (N=5700, K=6144: 37-38 rows per CTA),
    whole CTAs compared with the oracle."""
    p = synth.matvec(5700, 6144, 8, p_zero=0.4, seed=58)
    blocks = _quantize_tq2(p.w)
    bounds = [(p.n * i) // 152 for i in range(153)]
    rows = np.unique(np.concatenate([np.arange(bounds[i], bounds[i + 1]) for i in (0, 1, 76, 151)]))
    ob = orc.tq2_encode_rows(p.w[rows])
    for t in (1, 2, 4, 8):
        x = p.x[:t]
        q8 = G.quantize_acts(x)
        y = _mmv(blocks, q8, p.n, p.k, t)
        G.assert_close(y[:, rows], orc.tq2_mmv_f64(ob, orc.q8_1_quantize(x), rows.size, p.k, t))


def test_decode_kernel_partials_whole_ctas():
    """The integer partials on TQ2_0 weights of the kernels tq2_mmv runs (the
    decode kernel's rungs at t = 1..5, the one-n-tile tensor-core rung at
    6..8) against the oracle's, bit for bit, on whole decode-kernel CTAs of
    N=5120, K=6144."""
    p = synth.matvec(5120, 6144, 8, seed=61)
    blocks = _quantize_tq2(p.w)
    ctas = 152
    bounds = [(p.n * i) // ctas for i in range(ctas + 1)]
    rows = np.unique(np.concatenate([np.arange(bounds[i], bounds[i + 1]) for i in (0, 75, ctas - 1)]))
    ob = orc.tq2_encode_rows(p.w[rows])
    for t in range(1, 9):
        x = p.x[:t]
        q8 = G.quantize_acts(x)
        part = _partials(blocks, q8, p.n, p.k, t)
        np.testing.assert_array_equal(part[:, rows], orc.tq2_mmv_partials(ob, orc.q8_1_quantize(x), rows.size, p.k, t))


def test_determinism():
    p = synth.matvec(700, 4096, 3, seed=4)
    blocks, q8 = _quantize_tq2(p.w), G.quantize_acts(p.x)
    y0 = _mmv(blocks, q8, 700, 4096, 3)
    for _ in range(3):
        np.testing.assert_array_equal(_mmv(blocks, q8, 700, 4096, 3), y0)


# tq2_mmv runs the tensor-core rungs; tq2_mmv_ws with a workspace runs the
# tcgen05 tile path where tq1_mmv_workspace_size asks for one.
TILE = [(300, 2048, 7), (129, 4096, 12), (640, 6144, 16), (257, 2048, 33), (1000, 4096, 64), (200, 2048, 100)]


@pytest.mark.parametrize("n,k,t", TILE)
def test_tile_path(n, k, t):
    p = synth.matvec(n, k, t, p_zero=0.4, seed=3 * n + k + t)
    blocks, q8 = _quantize_tq2(p.w), G.quantize_acts(p.x)
    ref = orc.tq2_mmv_f64(orc.tq2_encode_rows(p.w), orc.q8_1_quantize(p.x), n, k, t)
    G.assert_close(_mmv(blocks, q8, n, k, t), ref)
    G.assert_close(G.mmv_ws(blocks, q8, n, k, t, fmt="tq2"), ref)


def test_tile_path_code_three():
    # Raw blocks with every code, including the unused 3 (+2 d), through the
    # fp16 table of the tensor-core expansion.
    n, k, t = 130, 2048, 40
    rng = np.random.default_rng(19)
    raw = rng.integers(0, 256, size=(n, k // 256, TQ2_BYTES), dtype=np.uint8)
    d = rng.uniform(0.01, 0.1, size=(n, k // 256)).astype(np.float16)
    raw[:, :, 64:66] = d.view(np.uint8).reshape(n, k // 256, 2)
    x = synth.matvec(1, k, t, seed=2).x
    ref = orc.tq2_mmv_f64(raw, orc.q8_1_quantize(x), n, k, t)
    rb, q8 = G.dev(raw.reshape(-1)), G.quantize_acts(x)
    G.assert_close(_mmv(rb, q8, n, k, t), ref)                   # tensor-core rungs
    G.assert_close(G.mmv_ws(rb, q8, n, k, t, fmt="tq2"), ref)     # tcgen05 tile path


def test_prefill_shape_sampled_rows():
    # N=14336, K=4096, T=512 (the prefill workload's shape) in TQ2_0.
    p = synth.config_matvec("c5")
    blocks = _quantize_tq2(p.w)
    rng = np.random.default_rng(55)
    rows = np.unique(np.concatenate([[0, 127, 128, p.n - 1], rng.integers(0, p.n, 60)]))
    q8 = G.quantize_acts(p.x)
    ref = orc.tq2_mmv_f64(orc.tq2_encode_rows(p.w[rows]), orc.q8_1_quantize(p.x), rows.size, p.k, p.t)
    G.assert_close(_mmv(blocks, q8, p.n, p.k, p.t)[:, rows], ref)
    G.assert_close(G.mmv_ws(blocks, q8, p.n, p.k, p.t, fmt="tq2")[:, rows], ref)


@pytest.mark.parametrize("n,k,t", [(5120, 6144, 1), (300, 2048, 2), (77, 1024, 3), (129, 4096, 4)])
def test_fused_quantisation_matches_two_step(n, k, t):
    # tq2_mmv_f32 quantises in the decode kernel's prologue with the same
    # operations as q8_1_quantize_acts: bit-identical per column.
    p = synth.matvec(n, k, t, seed=n + 3 * t)
    blocks = _quantize_tq2(p.w)
    two = _mmv(blocks, G.quantize_acts(p.x), n, k, t)
    tt = G.torch()
    y = tt.full((t, n), float("nan"), dtype=tt.float32, device="cuda")
    G.lib().tq2_mmv_f32(blocks, G.dev(p.x.astype(np.float32)), y, n, k, t)
    assert G.lib().tq1_sync_status() == 0
    np.testing.assert_array_equal(G.host(y), two)  # the same decode kernel on the same records
    if t > 1:
        for c in range(t):  # each column equals its own one-column two-step call, bitwise
            one = _mmv(blocks, G.quantize_acts(p.x[c:c + 1]), n, k, 1)
            y1 = tt.full((1, n), float("nan"), dtype=tt.float32, device="cuda")
            G.lib().tq2_mmv_f32(blocks, G.dev(p.x[c:c + 1].astype(np.float32)), y1, n, k, 1)
            np.testing.assert_array_equal(G.host(y1), one)


@pytest.mark.parametrize("n,k,t", [(640, 2048, 1), (300, 2304, 3), (257, 2048, 9), (100, 2304, 40)])
def test_residual_add(n, k, t):
    # y = res + W x: the decode rungs, the tile path (t = 9) and the general
    # kernel (k not a multiple of 2048); also in place (res is y).
    p = synth.matvec(n, k, t, seed=7 * n + t)
    blocks, q8 = _quantize_tq2(p.w), G.quantize_acts(p.x)
    plain = _mmv(blocks, q8, n, k, t)
    res = np.random.default_rng(t).standard_normal((t, n)).astype(np.float32)
    tt = G.torch()
    y = tt.full((t, n), float("nan"), dtype=tt.float32, device="cuda")
    G.lib().tq2_mmv_add(blocks, q8, G.dev(res), y, n, k, t)
    assert G.lib().tq1_sync_status() == 0
    np.testing.assert_array_equal(G.host(y), (plain + res).astype(np.float32))
    yy = G.dev(res)
    G.lib().tq2_mmv_add(blocks, q8, yy, yy, n, k, t)
    assert G.lib().tq1_sync_status() == 0
    np.testing.assert_array_equal(G.host(yy), (plain + res).astype(np.float32))
