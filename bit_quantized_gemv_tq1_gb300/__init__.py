"""TQ1_0 ternary mat-vec for GB300 (sm_103a): Python binding of libtq1.

Importing the package loads nothing; the CUDA library is loaded on first use
of a binding function.  The functions carry the names of the C entry points
declared in include/tq1.h.
"""
_EXPORTS = (
    "tq1_quantize_rows", "q8_1_quantize_acts", "tq1_mmv", "tq1_mmv_add", "tq1_mmv_f32", "tq1_mmv_partials",
    "tq1_mmv_id", "tq1_mmv_id_slots", "tq1_mmv_id_noalloc", "tq1_mmv_id_workspace_size", "tq1_dequantize_rows",
    "tq1_get_rows", "tq1_sync_status", "tq1_blocks_bytes", "tq1_q8_1_bytes", "tq2_quantize_rows", "tq2_mmv",
    "tq2_mmv_partials", "tq2_blocks_bytes", "tq2_dequantize_rows", "tq2_get_rows", "tq2_mmv_id",
    "tq2_mmv_id_slots", "tq2_mmv_f32", "tq2_mmv_add", "Tq1Error", "library", "library_path", "STATUS",
)
__all__ = list(_EXPORTS)


def __getattr__(name):
    if name in _EXPORTS:
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
