"""ctypes binding of libtq1 (include/tq1.h): argument marshalling only.

Every function has the name of the C entry point it calls and takes torch
CUDA tensors (or raw device addresses as ints) plus sizes; all computation
happens in the library's CUDA kernels.  There is no CPU path: if the
library is not built, or a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

TQ1_OK = 0
STATUS = {
    0: "TQ1_OK", -1: "TQ1_ERR_NULL", -2: "TQ1_ERR_SHAPE", -3: "TQ1_ERR_ALIGN", -4: "TQ1_ERR_UNSUPPORTED",
    -5: "TQ1_ERR_WORKSPACE", -6: "TQ1_ERR_CUDA", -7: "TQ1_ERR_TIMEOUT", -8: "TQ1_ERR_BAD_ID",
}
BLOCK_BYTES = 54
Q8_BYTES = 36


class Tq1Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {STATUS.get(code, code)} ({library().tq1_status_string(code).decode()})"
        if code == -6:
            msg += f": {library().tq1_last_cuda_error().decode()}"
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB


def library() -> ctypes.CDLL:
    """Load libtq1.so (must have been built by build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libtq1 is not built ({path} missing): run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        lib.tq1_status_string.restype = ctypes.c_char_p
        lib.tq1_status_string.argtypes = [ctypes.c_int]
        lib.tq1_version.restype = ctypes.c_char_p
        lib.tq1_version.argtypes = []
        lib.tq1_debug_inject_wait_timeout.restype = None
        lib.tq1_debug_inject_wait_timeout.argtypes = []
        lib.tq1_last_cuda_error.restype = ctypes.c_char_p
        lib.tq1_last_cuda_error.argtypes = []
        lib.tq1_blocks_bytes.restype = SZ
        lib.tq1_blocks_bytes.argtypes = [I64, I64]
        lib.tq2_blocks_bytes.restype = SZ
        lib.tq2_blocks_bytes.argtypes = [I64, I64]
        lib.tq2_quantize_rows.argtypes = [P, P, I64, I64, P]
        lib.tq2_mmv.argtypes = [P, P, P, I64, I64, I64, P]
        lib.tq2_mmv_partials.argtypes = [P, P, P, I64, I64, I64, P]
        lib.tq2_dequantize_rows.argtypes = [P, P, I64, I64, ctypes.c_int, P]
        lib.tq2_mmv_f32.argtypes = [P, P, P, I64, I64, I64, P]
        lib.tq2_mmv_add.argtypes = [P, P, P, P, I64, I64, I64, P]
        lib.tq2_mmv_id.argtypes = [P, I64, P, P, P, I64, I64, I64, I64, P, SZ, P]
        lib.tq2_mmv_id_slots.argtypes = [P, I64, P, P, P, I64, I64, I64, I64, P, SZ, P]
        lib.tq2_get_rows.argtypes = [P, P, I64, P, I64, I64, ctypes.c_int, P]
        lib.tq1_q8_1_bytes.restype = SZ
        lib.tq1_q8_1_bytes.argtypes = [I64, I64]
        lib.tq1_quantize_rows.argtypes = [P, P, I64, I64, P]
        lib.q8_1_quantize_acts.argtypes = [P, P, I64, I64, P]
        lib.tq1_mmv.argtypes = [P, P, P, I64, I64, I64, P]
        lib.tq1_mmv_partials.argtypes = [P, P, P, I64, I64, I64, P]
        lib.tq1_mmv_add.argtypes = [P, P, P, P, I64, I64, I64, P]
        lib.tq1_mmv_f32.argtypes = [P, P, P, I64, I64, I64, P]
        lib.tq1_mmv_id_workspace_size.restype = SZ
        lib.tq1_mmv_id_workspace_size.argtypes = [I64, I64, I64]
        lib.tq1_mmv_id.argtypes = [P, I64, P, P, P, I64, I64, I64, I64, P, SZ, P]
        lib.tq1_mmv_id_slots.argtypes = [P, I64, P, P, P, I64, I64, I64, I64, P, SZ, P]
        lib.tq1_mmv_id_noalloc.argtypes = [P, I64, P, P, P, I64, I64, I64, I64, P]
        lib.tq1_mmv_workspace_size.restype = SZ
        lib.tq1_mmv_workspace_size.argtypes = [I64, I64, I64]
        lib.tq1_mmv_ws.argtypes = [P, P, P, P, I64, I64, I64, P, SZ, P]
        lib.tq2_mmv_ws.argtypes = [P, P, P, P, I64, I64, I64, P, SZ, P]
        lib.tq1_mmv_id_partials.argtypes = [P, I64, P, P, P, I64, I64, I64, I64, P, SZ, P]
        lib.tq2_mmv_id_partials.argtypes = [P, I64, P, P, P, I64, I64, I64, I64, P, SZ, P]
        lib.tq1_dequantize_rows.argtypes = [P, P, I64, I64, ctypes.c_int, P]
        lib.tq1_get_rows.argtypes = [P, P, I64, P, I64, I64, ctypes.c_int, P]
        lib.tq1_sync_status.argtypes = [P]
        for name in ("tq1_quantize_rows", "q8_1_quantize_acts", "tq1_mmv", "tq1_mmv_add", "tq1_mmv_f32",
                     "tq1_mmv_partials", "tq1_mmv_id", "tq1_mmv_id_slots", "tq1_mmv_id_noalloc",
                     "tq1_dequantize_rows", "tq1_get_rows", "tq1_sync_status", "tq2_quantize_rows",
                     "tq2_mmv", "tq2_mmv_partials", "tq2_dequantize_rows", "tq2_get_rows", "tq2_mmv_id",
                     "tq2_mmv_id_slots", "tq2_mmv_f32", "tq2_mmv_add", "tq1_mmv_id_partials",
                     "tq2_mmv_id_partials", "tq1_mmv_ws", "tq2_mmv_ws"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _addr(x) -> int | None:
    """Device address of a CUDA tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("libtq1 takes CUDA tensors only")
    if not x.is_contiguous():
        raise ValueError("libtq1 takes contiguous tensors only")
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> None:
    if rc != TQ1_OK:
        raise Tq1Error(rc, where)


def tq1_blocks_bytes(n: int, k: int) -> int:
    return int(library().tq1_blocks_bytes(n, k))


def tq1_q8_1_bytes(t: int, k: int) -> int:
    return int(library().tq1_q8_1_bytes(t, k))


def tq1_quantize_rows(w, blocks, n: int, k: int, stream=None) -> None:
    _check(library().tq1_quantize_rows(_addr(w), _addr(blocks), n, k, _stream(stream)), "tq1_quantize_rows")


def q8_1_quantize_acts(x, q8, t: int, k: int, stream=None) -> None:
    _check(library().q8_1_quantize_acts(_addr(x), _addr(q8), t, k, _stream(stream)), "q8_1_quantize_acts")


def tq1_mmv(blocks, q8, y, n: int, k: int, t: int, stream=None) -> None:
    _check(library().tq1_mmv(_addr(blocks), _addr(q8), _addr(y), n, k, t, _stream(stream)), "tq1_mmv")


def tq1_mmv_f32(blocks, x, y, n: int, k: int, t: int, stream=None) -> None:
    """Decode mat-vec from fp32 activations, quantised to Q8_1 inside the kernel (t <= 4)."""
    _check(library().tq1_mmv_f32(_addr(blocks), _addr(x), _addr(y), n, k, t, _stream(stream)), "tq1_mmv_f32")


def tq1_mmv_add(blocks, q8, res, y, n: int, k: int, t: int, stream=None) -> None:
    """y = res + W x (res may be y itself)."""
    _check(library().tq1_mmv_add(_addr(blocks), _addr(q8), _addr(res), _addr(y), n, k, t, _stream(stream)),
           "tq1_mmv_add")


def tq1_mmv_workspace_size(n: int, k: int, t: int) -> int:
    """Bytes tq1_mmv_ws / tq2_mmv_ws need (0: the call takes the allocation-free kernels)."""
    return int(library().tq1_mmv_workspace_size(n, k, t))


def tq1_mmv_ws(blocks, q8, y, n: int, k: int, t: int, ws, ws_bytes: int | None = None, res=None,
               stream=None) -> None:
    """tq1_mmv (res None) or tq1_mmv_add with a caller workspace: the tcgen05 tile path at prefill-sized t."""
    wsb = ws_bytes if ws_bytes is not None else (0 if ws is None else ws.numel() * ws.element_size())
    _check(library().tq1_mmv_ws(_addr(blocks), _addr(q8), _addr(res), _addr(y), n, k, t, _addr(ws), wsb,
                                _stream(stream)), "tq1_mmv_ws")


def tq2_mmv_ws(blocks, q8, y, n: int, k: int, t: int, ws, ws_bytes: int | None = None, res=None,
               stream=None) -> None:
    wsb = ws_bytes if ws_bytes is not None else (0 if ws is None else ws.numel() * ws.element_size())
    _check(library().tq2_mmv_ws(_addr(blocks), _addr(q8), _addr(res), _addr(y), n, k, t, _addr(ws), wsb,
                                _stream(stream)), "tq2_mmv_ws")


def tq1_mmv_partials(blocks, q8, part, n: int, k: int, t: int, stream=None) -> None:
    _check(library().tq1_mmv_partials(_addr(blocks), _addr(q8), _addr(part), n, k, t, _stream(stream)),
           "tq1_mmv_partials")


def tq1_mmv_id_workspace_size(n_experts: int, t: int, top_k: int) -> int:
    return int(library().tq1_mmv_id_workspace_size(n_experts, t, top_k))


def tq1_mmv_id(expert_blocks, n_experts: int, q8, ids, y, n: int, k: int, t: int, top_k: int, ws,
               ws_bytes: int | None = None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(library().tq1_mmv_id(_addr(expert_blocks), n_experts, _addr(q8), _addr(ids), _addr(y), n, k, t, top_k,
                                _addr(ws), ws_bytes, _stream(stream)), "tq1_mmv_id")


def tq1_mmv_id_slots(expert_blocks, n_experts: int, q8, ids, y, n: int, k: int, t: int, top_k: int, ws,
                     ws_bytes: int | None = None, stream=None) -> None:
    """tq1_mmv_id with one Q8_1 activation row per (token, slot): q8 [t][top_k][k/32]."""
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(library().tq1_mmv_id_slots(_addr(expert_blocks), n_experts, _addr(q8), _addr(ids), _addr(y), n, k, t,
                                      top_k, _addr(ws), ws_bytes, _stream(stream)), "tq1_mmv_id_slots")


def tq1_mmv_id_partials(expert_blocks, n_experts: int, q8, ids, part, n: int, k: int, t: int, top_k: int, ws,
                        ws_bytes: int | None = None, stream=None) -> None:
    """Debug: the exact int32 partials part[t][top_k][n][k/32] of tq1_mmv_id."""
    wsb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(library().tq1_mmv_id_partials(_addr(expert_blocks), n_experts, _addr(q8), _addr(ids), _addr(part), n, k,
                                         t, top_k, _addr(ws), wsb, _stream(stream)), "tq1_mmv_id_partials")


def tq2_mmv_id_partials(expert_blocks, n_experts: int, q8, ids, part, n: int, k: int, t: int, top_k: int, ws,
                        ws_bytes: int | None = None, stream=None) -> None:
    """Debug: the exact int32 partials part[t][top_k][n][k/32] of tq2_mmv_id."""
    wsb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(library().tq2_mmv_id_partials(_addr(expert_blocks), n_experts, _addr(q8), _addr(ids), _addr(part), n, k,
                                         t, top_k, _addr(ws), wsb, _stream(stream)), "tq2_mmv_id_partials")


def tq1_mmv_id_noalloc(expert_blocks, n_experts: int, q8, ids, y, n: int, k: int, t: int, top_k: int,
                       stream=None) -> None:
    """tq1_mmv_id for callers that cannot allocate a workspace: the routing
    table lives in a fixed array inside the library (limits: 1024 experts,
    16384 routed token/slot pairs).  Make the first call on a device before
    any stream capture; calls that may overlap on the GPU race on the array."""
    _check(library().tq1_mmv_id_noalloc(_addr(expert_blocks), n_experts, _addr(q8), _addr(ids), _addr(y), n, k, t,
                                        top_k, _stream(stream)), "tq1_mmv_id_noalloc")


def tq1_dequantize_rows(blocks, out, n: int, k: int, out_f16: bool = False, stream=None) -> None:
    """out[n][k] (fp32, or fp16 when out_f16) = the values the TQ1_0 blocks encode."""
    _check(library().tq1_dequantize_rows(_addr(blocks), _addr(out), n, k, int(bool(out_f16)), _stream(stream)),
           "tq1_dequantize_rows")


def tq1_get_rows(blocks, row_ids, n_ids: int, out, n: int, k: int, out_f16: bool = False, stream=None) -> None:
    """out[i] = dequantised row row_ids[i] of the n x k TQ1_0 matrix."""
    _check(library().tq1_get_rows(_addr(blocks), _addr(row_ids), n_ids, _addr(out), n, k, int(bool(out_f16)),
                                  _stream(stream)), "tq1_get_rows")


def tq2_blocks_bytes(n: int, k: int) -> int:
    return int(library().tq2_blocks_bytes(n, k))


def tq2_quantize_rows(w, blocks, n: int, k: int, stream=None) -> None:
    _check(library().tq2_quantize_rows(_addr(w), _addr(blocks), n, k, _stream(stream)), "tq2_quantize_rows")


def tq2_mmv(blocks, q8, y, n: int, k: int, t: int, stream=None) -> None:
    _check(library().tq2_mmv(_addr(blocks), _addr(q8), _addr(y), n, k, t, _stream(stream)), "tq2_mmv")


def tq2_mmv_f32(blocks, x, y, n: int, k: int, t: int, stream=None) -> None:
    _check(library().tq2_mmv_f32(_addr(blocks), _addr(x), _addr(y), n, k, t, _stream(stream)), "tq2_mmv_f32")


def tq2_mmv_add(blocks, q8, res, y, n: int, k: int, t: int, stream=None) -> None:
    _check(library().tq2_mmv_add(_addr(blocks), _addr(q8), _addr(res), _addr(y), n, k, t, _stream(stream)),
           "tq2_mmv_add")


def tq2_mmv_partials(blocks, q8, part, n: int, k: int, t: int, stream=None) -> None:
    _check(library().tq2_mmv_partials(_addr(blocks), _addr(q8), _addr(part), n, k, t, _stream(stream)),
           "tq2_mmv_partials")


def tq2_mmv_id(expert_blocks, n_experts: int, q8, ids, y, n: int, k: int, t: int, top_k: int, ws,
               ws_bytes: int | None = None, stream=None) -> None:
    wsb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(library().tq2_mmv_id(_addr(expert_blocks), n_experts, _addr(q8), _addr(ids), _addr(y), n, k, t, top_k,
                                _addr(ws), wsb, _stream(stream)), "tq2_mmv_id")


def tq2_mmv_id_slots(expert_blocks, n_experts: int, q8, ids, y, n: int, k: int, t: int, top_k: int, ws,
                     ws_bytes: int | None = None, stream=None) -> None:
    wsb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(library().tq2_mmv_id_slots(_addr(expert_blocks), n_experts, _addr(q8), _addr(ids), _addr(y), n, k, t,
                                      top_k, _addr(ws), wsb, _stream(stream)), "tq2_mmv_id_slots")


def tq2_dequantize_rows(blocks, out, n: int, k: int, out_f16: bool = False, stream=None) -> None:
    _check(library().tq2_dequantize_rows(_addr(blocks), _addr(out), n, k, int(out_f16), _stream(stream)),
           "tq2_dequantize_rows")


def tq2_get_rows(blocks, row_ids, n_ids: int, out, n: int, k: int, out_f16: bool = False, stream=None) -> None:
    _check(library().tq2_get_rows(_addr(blocks), _addr(row_ids), n_ids, _addr(out), n, k, int(out_f16),
                                  _stream(stream)), "tq2_get_rows")


def tq1_sync_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status code."""
    return int(library().tq1_sync_status(_stream(stream)))
