"""ctypes view of libbgtq.so (the C ABI in include/bgtq.h).

Only argument marshalling lives here.  Loading fails loudly when the library
has not been built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes as C
import os

from . import build as _build

_LIB = None


class BgtqCache(C.Structure):
    _fields_ = [("k_codes", C.c_void_p), ("k_norm", C.c_void_p), ("v_codes", C.c_void_p),
                ("v_norm", C.c_void_p), ("capacity", C.c_int64), ("k_recent", C.c_void_p), ("recent", C.c_int64),
                ("page_table", C.c_void_p), ("max_pages", C.c_int64), ("page_tokens", C.c_int64),
                ("n_pages", C.c_int64)]


class BgtqHeadTables(C.Structure):
    _fields_ = [("n_coded", C.c_int), ("perm", C.POINTER(C.c_uint8)), ("width", C.POINTER(C.c_uint8)),
                ("piece", C.POINTER(C.c_uint8)), ("sign_k", C.POINTER(C.c_int8)), ("sign_v", C.POINTER(C.c_int8)),
                ("whiten", C.POINTER(C.c_float)), ("dewhiten", C.POINTER(C.c_float)),
                ("slot_pair", C.POINTER(C.c_uint8)), ("slot_offset", C.POINTER(C.c_uint16))]


EXPORTS = {
    "bgtq_last_error": (C.c_char_p, []),
    "bgtq_alloc_bits": (C.c_int, [C.c_void_p, C.c_int64, C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "bgtq_plan_create": (C.c_int, [C.POINTER(C.c_void_p), C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                   C.c_void_p, C.c_void_p, C.c_uint64, C.c_int, C.c_int]),
    "bgtq_plan_destroy": (C.c_int, [C.c_void_p]),
    "bgtq_plan_save": (C.c_int, [C.c_void_p, C.c_void_p, C.c_size_t, C.POINTER(C.c_size_t)]),
    "bgtq_plan_load": (C.c_int, [C.POINTER(C.c_void_p), C.c_void_p, C.c_size_t, C.c_int]),
    "bgtq_plan_get_head": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(BgtqHeadTables)]),
    "bgtq_plan_get_codebook": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(C.POINTER(C.c_float)),
                                         C.POINTER(C.POINTER(C.c_float)), C.POINTER(C.c_int)]),
    "bgtq_plan_code": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_int64, C.c_void_p]),
    "bgtq_cache_bytes": (C.c_int, [C.c_void_p, C.c_int, C.c_int64, C.POINTER(C.c_size_t),
                                   C.POINTER(C.c_size_t), C.POINTER(C.c_size_t)]),
    "bgtq_quantize_append": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                       C.c_void_p, C.POINTER(BgtqCache), C.c_void_p]),
    "bgtq_decode_attn_workspace": (C.c_int, [C.c_void_p, C.c_int, C.c_int64, C.POINTER(C.c_size_t)]),
    "bgtq_decode_attn": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(BgtqCache), C.c_void_p, C.c_int64,
                                   C.c_int, C.c_void_p, C.c_int, C.c_float, C.c_void_p, C.c_size_t, C.c_void_p]),
    "bgtq_decode_step": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                   C.POINTER(BgtqCache), C.c_void_p, C.c_int64, C.c_int, C.c_void_p, C.c_int, C.c_float,
                                   C.c_void_p, C.c_size_t, C.c_void_p]),
    "bgtq_prefill_attn": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                    C.POINTER(BgtqCache), C.c_void_p, C.c_int, C.c_float, C.c_void_p]),
    "bgtq_prefill_chunk_workspace": (C.c_int, [C.c_void_p, C.c_int, C.c_int64, C.POINTER(C.c_size_t)]),
    "bgtq_prefill_chunk_attn": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                          C.c_void_p, C.c_int64, C.POINTER(BgtqCache), C.c_void_p, C.c_int, C.c_float,
                                          C.c_void_p, C.c_size_t, C.c_void_p]),
    "bgtq_decode_attn_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(BgtqCache), C.c_void_p,
                                           C.c_int64, C.c_int, C.c_void_p, C.c_int, C.c_float, C.c_void_p]),
    "bgtq_logit_mae": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(BgtqCache), C.c_int64,
                                 C.c_int, C.c_float, C.c_void_p]),
    "bgtq_dequant_debug": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(BgtqCache), C.c_int, C.c_int, C.c_int,
                                     C.c_int64, C.c_int64, C.c_void_p, C.c_void_p, C.c_int]),
}


def debug_bounds() -> bool:
    """BGTQ_DEBUG_BOUNDS=1 in the environment selects the range-checked build
    of the library (for the whole process)."""
    return os.environ.get("BGTQ_DEBUG_BOUNDS", "0") not in ("", "0")


def library_path() -> str:
    return _build.LIB_DEBUG if debug_bounds() else _build.LIB


def lib(build_if_missing: bool = True):
    """The loaded CDLL; builds it first when asked and the sources changed."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if build_if_missing:
        path = _build.build(debug_bounds=debug_bounds())
    if not os.path.exists(path):
        raise RuntimeError(f"libbgtq.so is not built ({path}); run rope_aware_quantized_gb300.build.build()")
    L = C.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L
