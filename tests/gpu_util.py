"""Helpers for the GPU parity tests: move numpy inputs to the device, call
the library through its C ABI binding, and compare with the oracle."""
import numpy as np

QK, BLOCK_BYTES, QK8, Q8_BYTES = 256, 54, 32, 36

# Float tolerance of the mat-vec outputs: max relative error 1e-3 with an
# absolute floor of 1e-4 (the library accumulates in fp32, the oracle is exact
# up to fp64 rounding).
RTOL, ATOL = 1e-3, 1e-4


def torch():
    import torch as _t
    return _t


def dev(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def host(x):
    return x.cpu().numpy()


def lib():
    from bit_quantized_gemv_tq1_gb300 import _lib
    from bit_quantized_gemv_tq1_gb300 import build
    build.build()
    return _lib


def quantize_rows(w: np.ndarray):
    L = lib()
    n, k = w.shape
    blocks = torch().empty(n * (k // QK) * BLOCK_BYTES, dtype=torch().uint8, device="cuda")
    L.tq1_quantize_rows(dev(w.astype(np.float32)), blocks, n, k)
    return blocks


def quantize_acts(x: np.ndarray):
    L = lib()
    t, k = x.shape
    q8 = torch().empty(t * (k // QK8) * Q8_BYTES, dtype=torch().uint8, device="cuda")
    L.q8_1_quantize_acts(dev(x.astype(np.float32)), q8, t, k)
    return q8


def mmv(blocks, q8, n, k, t):
    L = lib()
    y = torch().full((t, n), float("nan"), dtype=torch().float32, device="cuda")
    L.tq1_mmv(blocks, q8, y, n, k, t)
    assert L.tq1_sync_status() == 0
    return host(y)


def mmv_ws(blocks, q8, n, k, t, fmt="tq1", res=None):
    """tq1_mmv_ws / tq2_mmv_ws with a workspace of the size the library asks
    for (the tcgen05 tile path wherever that size is nonzero)."""
    L = lib()
    tt = torch()
    ws_bytes = L.tq1_mmv_workspace_size(n, k, t)
    ws = tt.empty(max(ws_bytes, 16), dtype=tt.uint8, device="cuda")
    y = tt.full((t, n), float("nan"), dtype=tt.float32, device="cuda")
    fn = L.tq1_mmv_ws if fmt == "tq1" else L.tq2_mmv_ws
    fn(blocks, q8, y, n, k, t, ws, ws_bytes, res=res)
    assert L.tq1_sync_status() == 0
    return host(y)


def partials(blocks, q8, n, k, t):
    L = lib()
    p = torch().full((t, n, k // QK8), -2 ** 31, dtype=torch().int32, device="cuda")
    L.tq1_mmv_partials(blocks, q8, p, n, k, t)
    assert L.tq1_sync_status() == 0
    return host(p)


def assert_close(y, ref, rtol=RTOL, atol=ATOL):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert y.shape == ref.shape
    assert np.all(np.isfinite(y)), "non-finite output"
    err = np.abs(y - ref)
    bound = np.maximum(rtol * np.abs(ref), atol)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"got {y[tuple(i)]!r}, want {ref[tuple(i)]!r}")
