"""The C ABI: the library loads, exports every function include/tq1.h
declares, and rejects bad arguments on the host without launching anything
(these checks run before any CUDA call, so they need no GPU)."""
import ctypes
import os
import re

import pytest

from bit_quantized_gemv_tq1_gb300 import _lib as L
from bit_quantized_gemv_tq1_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tq1.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("tq1_quantize_rows", "q8_1_quantize_acts", "tq1_mmv", "tq1_mmv_id", "tq1_mmv_partials",
                 "tq1_mmv_id_workspace_size", "tq1_sync_status", "tq1_status_string", "tq1_dequantize_rows",
                 "tq1_get_rows", "tq2_quantize_rows", "tq2_mmv", "tq2_mmv_partials", "tq2_blocks_bytes", "tq2_dequantize_rows", "tq2_get_rows", "tq2_mmv_id",
                 "tq2_mmv_id_slots", "tq2_mmv_f32", "tq2_mmv_add", "tq1_mmv_id_partials",
                 "tq2_mmv_id_partials", "tq1_mmv_id_noalloc"):
        assert want in names


def test_every_declaration_cites_a_passage():
    # The comment block nearest above each declaration names the passage
    # that defines the operation, or says that it is a convention of this
    # library.
    src = open(HEADER).read()
    missing = []
    for m in re.finditer(r"^(?:const\s+char\s*\*|int|size_t|void)\s+(\w+)\s*\(", src, flags=re.M):
        before = src[:m.start()]
        end = before.rfind("*/")
        start = before.rfind("/*", 0, end)
        block = before[start:end] if start >= 0 and end >= 0 else ""
        if "Source:" not in block and "No passage" not in block:
            missing.append(m.group(1))
    assert not missing, missing


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in L.STATUS:
        assert lib.tq1_status_string(code)
    assert lib.tq1_version() == b"0.1.0"


def test_sizes(lib):
    assert L.tq1_blocks_bytes(5120, 6144) == 5120 * 24 * 54
    assert L.tq1_q8_1_bytes(3, 6144) == 3 * 192 * 36
    assert L.tq1_mmv_id_workspace_size(128, 32, 8) >= 4 * (1 + 129 + 128 + 256)
    assert L.tq1_mmv_id_workspace_size(128, 32, 8) % 256 == 0


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced


@pytest.mark.parametrize("args,code", [
    ((FAKE, FAKE, FAKE, 10, 300, 1), -2),   # k not a multiple of 256
    ((FAKE, FAKE, FAKE, -1, 256, 1), -2),   # negative n
    ((FAKE, FAKE, FAKE, 10, 0, 1), -2),     # k == 0
    ((FAKE, FAKE, FAKE, 10, 256, -3), -2),  # negative t
    ((None, FAKE, FAKE, 10, 256, 1), -1),   # null weights
    ((FAKE, FAKE, None, 10, 256, 1), -1),   # null output
    ((FAKE + 4, FAKE, FAKE, 10, 256, 1), -3),  # misaligned
    ((FAKE, FAKE, FAKE, 10, 256 * 246, 1), -4),  # k beyond the staging limit
    ((None, None, None, 0, 256, 1), 0),     # empty: nothing to do
    ((None, None, None, 5, 256, 0), 0),
])
def test_mmv_host_checks(lib, args, code):
    assert lib.tq1_mmv(*args, None) == code


def test_other_host_checks(lib):
    assert lib.tq1_quantize_rows(FAKE, FAKE, 4, 100, None) == -2
    assert lib.tq1_quantize_rows(None, FAKE, 4, 256, None) == -1
    assert lib.q8_1_quantize_acts(FAKE, FAKE, 1, 48, None) == -2
    assert lib.q8_1_quantize_acts(FAKE + 8, FAKE, 1, 64, None) == -3
    assert lib.tq1_mmv_partials(FAKE, FAKE, None, 4, 256, 1, None) == -1
    ws = L.tq1_mmv_id_workspace_size(8, 2, 2)
    assert lib.tq1_mmv_id(FAKE, 8, FAKE, FAKE, FAKE, 16, 256, 2, 2, FAKE, ws - 1, None) == -5
    assert lib.tq1_mmv_id(FAKE, 0, FAKE, FAKE, FAKE, 16, 256, 2, 2, FAKE, ws, None) == -2
    assert lib.tq1_mmv_id(FAKE, 8, FAKE, None, FAKE, 16, 256, 2, 2, FAKE, ws, None) == -1
    assert lib.tq1_mmv_id(FAKE, 8, FAKE, FAKE, FAKE, 16, 256, 0, 2, FAKE, ws, None) == 0


def test_mmv_f32_host_checks(lib):
    assert lib.tq1_mmv_f32(FAKE, FAKE, FAKE, 10, 256, 5, None) == -4   # t > 4: not fused
    assert lib.tq1_mmv_f32(FAKE, None, FAKE, 10, 256, 1, None) == -1
    assert lib.tq1_mmv_f32(FAKE, FAKE + 4, FAKE, 10, 256, 1, None) == -3
    assert lib.tq1_mmv_f32(FAKE, FAKE, FAKE, 10, 300, 1, None) == -2
    assert lib.tq1_mmv_f32(None, None, None, 0, 256, 1, None) == 0


def test_mmv_add_host_checks(lib):
    assert lib.tq1_mmv_add(FAKE, FAKE, None, FAKE, 10, 256, 1, None) == -1   # null residual
    assert lib.tq1_mmv_add(FAKE, FAKE, FAKE + 4, FAKE, 10, 256, 1, None) == -3
    assert lib.tq1_mmv_add(FAKE, FAKE, FAKE, FAKE, 10, 300, 1, None) == -2
    assert lib.tq1_mmv_add(None, None, None, None, 0, 256, 1, None) == 0


def test_dequant_host_checks(lib):
    assert lib.tq1_dequantize_rows(FAKE, FAKE, 4, 100, 0, None) == -2
    assert lib.tq1_dequantize_rows(FAKE, FAKE, -1, 256, 0, None) == -2
    assert lib.tq1_dequantize_rows(None, FAKE, 4, 256, 0, None) == -1
    assert lib.tq1_dequantize_rows(FAKE, FAKE + 8, 4, 256, 1, None) == -3
    assert lib.tq1_dequantize_rows(None, None, 0, 256, 0, None) == 0
    assert lib.tq1_get_rows(FAKE, None, 3, FAKE, 4, 256, 0, None) == -1
    assert lib.tq1_get_rows(FAKE, FAKE, -1, FAKE, 4, 256, 0, None) == -2
    assert lib.tq1_get_rows(FAKE, FAKE + 4, 3, FAKE, 4, 256, 0, None) == -3
    assert lib.tq1_get_rows(None, None, 0, None, 4, 256, 0, None) == 0


def test_tq2_host_checks(lib):
    assert L.tq2_blocks_bytes(5120, 6144) == 5120 * 24 * 66
    assert lib.tq2_quantize_rows(FAKE, FAKE, 4, 100, None) == -2
    assert lib.tq2_quantize_rows(None, FAKE, 4, 256, None) == -1
    assert lib.tq2_quantize_rows(FAKE, FAKE + 2, 4, 256, None) == -3
    assert lib.tq2_mmv(FAKE, FAKE, FAKE, 10, 300, 1, None) == -2
    assert lib.tq2_mmv(FAKE, None, FAKE, 10, 256, 1, None) == -1
    assert lib.tq2_mmv(FAKE + 4, FAKE, FAKE, 10, 256, 1, None) == -3
    assert lib.tq2_mmv(FAKE, FAKE, FAKE, 10, 256 * 246, 1, None) == -4
    assert lib.tq2_mmv(None, None, None, 0, 256, 3, None) == 0
    assert lib.tq2_mmv_partials(FAKE, FAKE, None, 4, 256, 1, None) == -1


def test_tq2_dequant_host_checks(lib):
    assert lib.tq2_dequantize_rows(FAKE, FAKE, 4, 100, 0, None) == -2
    assert lib.tq2_dequantize_rows(None, FAKE, 4, 256, 0, None) == -1
    assert lib.tq2_dequantize_rows(FAKE, FAKE + 8, 4, 256, 1, None) == -3
    assert lib.tq2_dequantize_rows(None, None, 0, 256, 0, None) == 0
    assert lib.tq2_get_rows(FAKE, None, 3, FAKE, 4, 256, 0, None) == -1
    assert lib.tq2_get_rows(FAKE, FAKE, -1, FAKE, 4, 256, 0, None) == -2
    assert lib.tq2_get_rows(FAKE, FAKE + 4, 3, FAKE, 4, 256, 0, None) == -3
    assert lib.tq2_get_rows(None, None, 0, None, 4, 256, 0, None) == 0


def test_tq2_mmv_id_host_checks(lib):
    ws = L.tq1_mmv_id_workspace_size(8, 2, 2)
    assert lib.tq2_mmv_id(FAKE, 8, FAKE, FAKE, FAKE, 16, 256, 2, 2, FAKE, ws - 1, None) == -5
    assert lib.tq2_mmv_id(FAKE, 0, FAKE, FAKE, FAKE, 16, 256, 2, 2, FAKE, ws, None) == -2
    assert lib.tq2_mmv_id(FAKE, 8, FAKE, None, FAKE, 16, 256, 2, 2, FAKE, ws, None) == -1
    assert lib.tq2_mmv_id_slots(FAKE, 8, FAKE, FAKE, FAKE, 16, 300, 2, 2, FAKE, ws, None) == -2
    assert lib.tq2_mmv_id_slots(FAKE, 8, FAKE, FAKE, FAKE, 16, 256, 0, 2, FAKE, ws, None) == 0


def test_tq2_fused_entry_host_checks(lib):
    assert lib.tq2_mmv_f32(FAKE, FAKE, FAKE, 10, 256, 5, None) == -4
    assert lib.tq2_mmv_f32(FAKE, None, FAKE, 10, 256, 1, None) == -1
    assert lib.tq2_mmv_add(FAKE, FAKE, None, FAKE, 10, 256, 1, None) == -1
    assert lib.tq2_mmv_add(FAKE, FAKE, FAKE + 4, FAKE, 10, 256, 1, None) == -3


def test_mmv_id_partials_host_checks(lib):
    ws = L.tq1_mmv_id_workspace_size(8, 2, 2)
    for fn in (lib.tq1_mmv_id_partials, lib.tq2_mmv_id_partials):
        assert fn(FAKE, 8, FAKE, FAKE, FAKE, 16, 256, 2, 2, FAKE, ws - 1, None) == -5
        assert fn(FAKE, 8, FAKE, FAKE, None, 16, 256, 2, 2, FAKE, ws, None) == -1
        assert fn(FAKE, 8, FAKE, FAKE, FAKE + 4, 16, 256, 2, 2, FAKE, ws, None) == -3
        assert fn(FAKE, 0, FAKE, FAKE, FAKE, 16, 256, 2, 2, FAKE, ws, None) == -2
        assert fn(FAKE, 8, FAKE, FAKE, FAKE, 16, 256, 0, 2, FAKE, ws, None) == 0


def test_no_alloc_rejects_calls_beyond_its_table(lib):
    # tq1_mmv_id_noalloc's fixed routing table holds 1024 experts and 16384
    # routed pairs; larger calls are refused on the host, before any launch.
    fake = 1 << 20
    assert lib.tq1_mmv_id_noalloc(fake, 1025, fake, fake, fake, 16, 256, 1, 1, None) == -5
    assert lib.tq1_mmv_id_noalloc(fake, 8, fake, fake, fake, 16, 256, 4097, 4, None) == -5
    assert lib.tq1_mmv_id_noalloc(fake, 8, fake, fake, fake, 16, 256, 1, 1 << 40, None) == -5


def test_mmv_ws_host_checks(lib):
    # The tile path's workspace: asked for only where the tile path runs (k a
    # multiple of 2048, t at its threshold or above), refused when too small
    # or misaligned, before anything is launched.
    assert L.tq1_mmv_workspace_size(300, 2048, 1) == 0
    assert L.tq1_mmv_workspace_size(300, 1280, 512) == 0
    need = L.tq1_mmv_workspace_size(300, 2048, 512)
    assert need >= 2 * 2 * 512 * 2048 + 4 * 512 and need % 256 == 0
    for fn in (lib.tq1_mmv_ws, lib.tq2_mmv_ws):
        assert fn(FAKE, FAKE, None, FAKE, 300, 2048, 512, FAKE, need - 1, None) == -5
        assert fn(FAKE, FAKE, None, FAKE, 300, 2048, 512, FAKE + 8, need, None) == -3
        assert fn(FAKE, FAKE, None, None, 300, 2048, 512, FAKE, need, None) == -1
        assert fn(FAKE, FAKE, None, FAKE, 300, 2000, 512, FAKE, need, None) == -2
        assert fn(FAKE, FAKE, None, FAKE, 0, 2048, 512, FAKE, need, None) == 0


def test_k_past_the_limit_is_refused(lib):
    # 62720 (245 blocks) is the largest k the mat-vec entries accept.
    assert lib.tq1_mmv(FAKE, FAKE, FAKE, 4, 62720 + 256, 1, None) == -4
    assert lib.tq1_mmv_partials(FAKE, FAKE, FAKE, 4, 62720 + 256, 1, None) == -4
    assert lib.tq2_mmv(FAKE, FAKE, FAKE, 4, 62720 + 256, 9, None) == -4

