"""Python face of the plain C oracle (tq1_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the benchmark's CPU-baseline leg, never by the product path.  It shares
no code with the CUDA library in ``bit_quantized_gemv_tq1_gb300``.

Every function here is argument marshalling around the C routine of the same
purpose; the arithmetic lives in tq1_oracle.c, which cites the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq1_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 256
BLOCK_BYTES = 54
TQ2_BYTES = 66
QK8 = 32
Q8_BYTES = 36


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE fp32, no contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.orc_f16_from_f32.restype = ctypes.c_uint16
        lib.orc_f16_from_f32.argtypes = [ctypes.c_float]
        lib.orc_f32_from_f16.restype = ctypes.c_float
        lib.orc_f32_from_f16.argtypes = [ctypes.c_uint16]
        lib.orc_tq1_pack_byte.restype = ctypes.c_uint8
        lib.orc_tq1_pack_byte.argtypes = [P]
        lib.orc_tq1_digit.restype = ctypes.c_int
        lib.orc_tq1_digit.argtypes = [ctypes.c_uint8, ctypes.c_int]
        lib.orc_tq1_elem_pos.restype = None
        lib.orc_tq1_elem_pos.argtypes = [ctypes.c_int, P, P]
        lib.orc_tq1_encode_rows.argtypes = [P, P, I64, I64]
        lib.orc_tq1_decode_rows.argtypes = [P, P, P, I64, I64]
        lib.orc_q8_1_quantize.argtypes = [P, P, I64, I64]
        lib.orc_mmv_partials.argtypes = [P, P, P, I64, I64, I64]
        lib.orc_mmv_f64.argtypes = [P, P, P, I64, I64, I64]
        lib.orc_mmv_f64_rows.argtypes = [P, P, P, I64, I64, I64, P, I64]
        lib.orc_mmv_id_f64.argtypes = [P, I64, P, P, P, I64, I64, I64, I64]
        lib.orc_mmv_id_f64_rows.argtypes = [P, I64, P, P, P, I64, I64, I64, I64, P, I64]
        lib.orc_tq2_elem_pos.restype = None
        lib.orc_tq2_elem_pos.argtypes = [ctypes.c_int, P, P]
        lib.orc_tq2_code.restype = ctypes.c_int
        lib.orc_tq2_code.argtypes = [P, ctypes.c_int]
        lib.orc_tq2_encode_rows.argtypes = [P, P, I64, I64]
        lib.orc_tq2_decode_rows.argtypes = [P, P, P, I64, I64]
        lib.orc_tq2_mmv_partials.argtypes = [P, P, P, I64, I64, I64]
        lib.orc_tq2_mmv_f64.argtypes = [P, P, P, I64, I64, I64]
        lib.orc_tq2_mmv_f64_rows.argtypes = [P, P, P, I64, I64, I64, P, I64]
        lib.orc_tq2_mmv_id_f64.argtypes = [P, I64, P, P, P, I64, I64, I64, I64]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_set_num_threads.restype = None
        lib.orc_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- fp16 ----
def f16_from_f32(x: float) -> int:
    return int(_load().orc_f16_from_f32(ctypes.c_float(x)))


def f32_from_f16(h: int) -> float:
    return float(_load().orc_f32_from_f16(ctypes.c_uint16(h)))


# ------------------------------------------------------------ byte code ---
def pack_byte(digits) -> int:
    u = np.zeros(5, dtype=np.int32)
    u[: len(digits)] = digits
    return int(_load().orc_tq1_pack_byte(_ptr(u)))


def digit(b: int, k: int) -> int:
    return int(_load().orc_tq1_digit(ctypes.c_uint8(b), ctypes.c_int(k)))


def elem_pos(e: int) -> tuple[int, int]:
    bi, dg = ctypes.c_int(), ctypes.c_int()
    _load().orc_tq1_elem_pos(e, ctypes.byref(bi), ctypes.byref(dg))
    return bi.value, dg.value


# -------------------------------------------------------------- encoding --
def tq1_encode_rows(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    assert k % QK == 0
    out = np.zeros((n, k // QK, BLOCK_BYTES), dtype=np.uint8)
    _load().orc_tq1_encode_rows(_ptr(w), _ptr(out), n, k)
    return out


def tq1_decode_rows(blocks: np.ndarray, n: int, k: int) -> tuple[np.ndarray, np.ndarray]:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert blocks.size == n * (k // QK) * BLOCK_BYTES
    trits = np.zeros((n, k), dtype=np.int8)
    scales = np.zeros((n, k // QK), dtype=np.float32)
    _load().orc_tq1_decode_rows(_ptr(blocks), _ptr(trits), _ptr(scales), n, k)
    return trits, scales


def tq1_dequantize_rows(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    """Values the blocks encode, fp32 [n][k]: trit * d per element (the decode
    above, scaled by its block's fp16 scale; exact in fp32)."""
    trits, scales = tq1_decode_rows(blocks, n, k)
    return (trits.astype(np.float32).reshape(n, k // QK, QK) * scales[:, :, None]).reshape(n, k)


def q8_1_quantize(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    t, k = x.shape
    assert k % QK8 == 0
    out = np.zeros((t, k // QK8, Q8_BYTES), dtype=np.uint8)
    _load().orc_q8_1_quantize(_ptr(x), _ptr(out), t, k)
    return out


def q8_1_fields(q8: np.ndarray, t: int, k: int):
    """Split Q8_1 bytes into (d fp32 [t][k/32], s fp32 [t][k/32], q int8 [t][k]).
    Pure byte reinterpretation (little-endian fp16 fields)."""
    b = np.ascontiguousarray(q8, dtype=np.uint8).reshape(t, k // QK8, Q8_BYTES)
    d = b[:, :, 0:2].copy().view(np.float16).reshape(t, k // QK8).astype(np.float32)
    s = b[:, :, 2:4].copy().view(np.float16).reshape(t, k // QK8).astype(np.float32)
    q = b[:, :, 4:].copy().view(np.int8).reshape(t, k)
    return d, s, q


# ------------------------------------------------------------ dot products -
def mmv_partials(blocks: np.ndarray, q8: np.ndarray, n: int, k: int, t: int) -> np.ndarray:
    out = np.zeros((t, n, k // QK8), dtype=np.int32)
    _load().orc_mmv_partials(_ptr(np.ascontiguousarray(blocks)), _ptr(np.ascontiguousarray(q8)),
                             _ptr(out), n, k, t)
    return out


def mmv_f64(blocks: np.ndarray, q8: np.ndarray, n: int, k: int, t: int) -> np.ndarray:
    out = np.zeros((t, n), dtype=np.float64)
    _load().orc_mmv_f64(_ptr(np.ascontiguousarray(blocks)), _ptr(np.ascontiguousarray(q8)), _ptr(out), n, k, t)
    return out


def mmv_f64_rows(blocks: np.ndarray, q8: np.ndarray, n: int, k: int, t: int, rows) -> np.ndarray:
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < n)
    out = np.zeros((t, rows.size), dtype=np.float64)
    _load().orc_mmv_f64_rows(_ptr(np.ascontiguousarray(blocks)), _ptr(np.ascontiguousarray(q8)), _ptr(out),
                             n, k, t, _ptr(rows), rows.size)
    return out


def mmv_id_f64(expert_blocks: np.ndarray, n_experts: int, q8: np.ndarray, ids: np.ndarray,
               n: int, k: int, t: int, top_k: int, fill: float = np.nan) -> np.ndarray:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.full((t, top_k, n), fill, dtype=np.float64)
    _load().orc_mmv_id_f64(_ptr(np.ascontiguousarray(expert_blocks)), n_experts, _ptr(np.ascontiguousarray(q8)),
                           _ptr(ids), _ptr(out), n, k, t, top_k)
    return out


def mmv_id_f64_rows(expert_blocks: np.ndarray, n_experts: int, q8: np.ndarray, ids: np.ndarray,
                    n: int, k: int, t: int, top_k: int, rows, fill: float = np.nan) -> np.ndarray:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.full((t, top_k, rows.size), fill, dtype=np.float64)
    _load().orc_mmv_id_f64_rows(_ptr(np.ascontiguousarray(expert_blocks)), n_experts,
                                _ptr(np.ascontiguousarray(q8)), _ptr(ids), _ptr(out), n, k, t, top_k,
                                _ptr(rows), rows.size)
    return out


# ------------------------------------------------------------------ TQ2_0 --
# The 2-bit sibling format (reading R6 of tq1_oracle.c): qs[64] with four
# 2-bit codes per byte, fp16 d at byte 64, 66 bytes per 256-block.
def tq2_elem_pos(e: int) -> tuple[int, int]:
    bi, f = ctypes.c_int(), ctypes.c_int()
    _load().orc_tq2_elem_pos(e, ctypes.byref(bi), ctypes.byref(f))
    return bi.value, f.value


def tq2_code(block: np.ndarray, e: int) -> int:
    block = np.ascontiguousarray(block, dtype=np.uint8)
    assert block.size == TQ2_BYTES
    return int(_load().orc_tq2_code(_ptr(block), e))


def tq2_encode_rows(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    assert k % QK == 0
    out = np.zeros((n, k // QK, TQ2_BYTES), dtype=np.uint8)
    _load().orc_tq2_encode_rows(_ptr(w), _ptr(out), n, k)
    return out


def tq2_decode_rows(blocks: np.ndarray, n: int, k: int) -> tuple[np.ndarray, np.ndarray]:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert blocks.size == n * (k // QK) * TQ2_BYTES
    trits = np.zeros((n, k), dtype=np.int8)
    scales = np.zeros((n, k // QK), dtype=np.float32)
    _load().orc_tq2_decode_rows(_ptr(blocks), _ptr(trits), _ptr(scales), n, k)
    return trits, scales


def tq2_mmv_partials(blocks: np.ndarray, q8: np.ndarray, n: int, k: int, t: int) -> np.ndarray:
    out = np.zeros((t, n, k // QK8), dtype=np.int32)
    _load().orc_tq2_mmv_partials(_ptr(np.ascontiguousarray(blocks)), _ptr(np.ascontiguousarray(q8)),
                                 _ptr(out), n, k, t)
    return out


def tq2_mmv_f64(blocks: np.ndarray, q8: np.ndarray, n: int, k: int, t: int) -> np.ndarray:
    out = np.zeros((t, n), dtype=np.float64)
    _load().orc_tq2_mmv_f64(_ptr(np.ascontiguousarray(blocks)), _ptr(np.ascontiguousarray(q8)), _ptr(out), n, k, t)
    return out


def tq2_mmv_f64_rows(blocks: np.ndarray, q8: np.ndarray, n: int, k: int, t: int, rows) -> np.ndarray:
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < n)
    out = np.zeros((t, rows.size), dtype=np.float64)
    _load().orc_tq2_mmv_f64_rows(_ptr(np.ascontiguousarray(blocks)), _ptr(np.ascontiguousarray(q8)), _ptr(out),
                                 n, k, t, _ptr(rows), rows.size)
    return out


def tq2_dequantize_rows(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    """Values TQ2_0 blocks encode, fp32 [n][k]: (code - 1) * d per element
    (the oracle decode scaled by its block's fp16 scale; exact in fp32)."""
    trits, scales = tq2_decode_rows(blocks, n, k)
    return (trits.astype(np.float32).reshape(n, k // QK, QK) * scales[:, :, None]).reshape(n, k)


def tq2_mmv_id_f64(expert_blocks: np.ndarray, n_experts: int, q8: np.ndarray, ids: np.ndarray,
                   n: int, k: int, t: int, top_k: int, fill: float = np.nan) -> np.ndarray:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.full((t, top_k, n), fill, dtype=np.float64)
    _load().orc_tq2_mmv_id_f64(_ptr(np.ascontiguousarray(expert_blocks)), n_experts, _ptr(np.ascontiguousarray(q8)),
                               _ptr(ids), _ptr(out), n, k, t, top_k)
    return out
