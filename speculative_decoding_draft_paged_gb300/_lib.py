"""ctypes view of the C ABI in ``include/dflash.h``.

Argument marshalling only.  The library must have been built
(``speculative_decoding_draft_paged_gb300.build.build()``); there is no
fallback when it is missing.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

DFLASH_OK = 0
DFLASH_ERR_INVALID = -1
DFLASH_ERR_WORKSPACE = -2
DFLASH_ERR_DEVICE = -3
DFLASH_ERR_LAUNCH = -4

DFLASH_STATUS_BAD_PAGE = 1
DFLASH_STATUS_BAD_CTX_LEN = 2
DFLASH_STATUS_TIMEOUT = 4
DFLASH_STATUS_FP8_RANGE = 8

DFLASH_TEST_WITHHOLD_LOADS = 1

KV_BF16 = 0
KV_FP8_E4M3 = 1

PATH_AUTO = 0
PATH_MMA = 1
PATH_TCGEN05 = 2



def _header_static_scratch_bytes() -> int:
    """DFLASH_STATIC_SCRATCH_BYTES as the public header defines it."""
    import re

    with open(os.path.join(_build.INCLUDE, "dflash.h")) as f:
        m = re.search(r"#define\s+DFLASH_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", f.read())
    if m is None:
        raise RuntimeError("DFLASH_STATIC_SCRATCH_BYTES not found in include/dflash.h")
    return int(m[1]) << int(m[2])


# Size of the library-held scratch array of dflash_block_attn_static_ws.
STATIC_SCRATCH_BYTES = _header_static_scratch_bytes()

EXPORTS = (
    "dflash_workspace_size",
    "dflash_plan",
    "dflash_block_attn",
    "dflash_block_attn_timed",
    "dflash_block_attn_static_ws",
    "dflash_block_placement",
    "dflash_append_block_kv",
    "dflash_block_attn_append",
    "dflash_block_attn_dense_suffix",
    "dflash_block_attn_fp8_context",
    "dflash_block_attn_fp8_context_timed",
    "dflash_partial_workspace_size",
    "dflash_block_attn_partial",
    "dflash_combine_partials",
    "dflash_status_string",
    "dflash_read_device_status",
    "dflash_clear_device_status",
    "dflash_version",
)


class Params(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("future_keys", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("max_ctx_len", ctypes.c_int32),
        ("force_path", ctypes.c_int32),
        ("force_split_tiles", ctypes.c_int32),
        ("right_window", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("test_flags", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 1),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int32),
        ("rows", ctypes.c_int32),
        ("rows_padded", ctypes.c_int32),
        ("tile_keys", ctypes.c_int32),
        ("split_tiles", ctypes.c_int32),
        ("max_splits", ctypes.c_int32),
        ("units", ctypes.c_int64),
        ("threads", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("flat", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 1),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Open ``libdflash.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library not built ({path}); run "
                    "speculative_decoding_draft_paged_gb300.build.build()")
            lib = ctypes.CDLL(path)
            vp, i32 = ctypes.c_void_p, ctypes.c_int
            lib.dflash_workspace_size.argtypes = [ctypes.POINTER(Params)]
            lib.dflash_workspace_size.restype = ctypes.c_size_t
            lib.dflash_plan.argtypes = [ctypes.POINTER(Params), ctypes.POINTER(PlanInfo)]
            lib.dflash_plan.restype = i32
            lib.dflash_block_attn.argtypes = [ctypes.POINTER(Params), vp, vp, vp, vp, vp, vp, vp, vp,
                                              ctypes.c_size_t, vp]
            lib.dflash_block_attn.restype = i32
            lib.dflash_block_attn_timed.argtypes = lib.dflash_block_attn.argtypes + [vp, vp]
            lib.dflash_block_attn_timed.restype = i32
            lib.dflash_block_attn_static_ws.argtypes = [ctypes.POINTER(Params)] + [vp] * 8
            lib.dflash_block_attn_static_ws.restype = i32
            lib.dflash_block_placement.argtypes = [ctypes.POINTER(Params)] + [vp] * 5
            lib.dflash_block_placement.restype = i32
            lib.dflash_append_block_kv.argtypes = [ctypes.POINTER(Params)] + [vp] * 8
            lib.dflash_append_block_kv.restype = i32
            lib.dflash_block_attn_append.argtypes = [ctypes.POINTER(Params)] + [vp] * 10 + \
                [ctypes.c_size_t, vp]
            lib.dflash_block_attn_append.restype = i32
            lib.dflash_block_attn_dense_suffix.argtypes = lib.dflash_block_attn_append.argtypes
            lib.dflash_block_attn_dense_suffix.restype = i32
            f32 = ctypes.c_float
            lib.dflash_block_attn_fp8_context.argtypes = [ctypes.POINTER(Params)] + [vp] * 5 + \
                [f32, f32] + [vp] * 5 + [ctypes.c_size_t, vp]
            lib.dflash_block_attn_fp8_context.restype = i32
            lib.dflash_block_attn_fp8_context_timed.argtypes = \
                lib.dflash_block_attn_fp8_context.argtypes + [vp, vp]
            lib.dflash_block_attn_fp8_context_timed.restype = i32
            lib.dflash_partial_workspace_size.argtypes = [ctypes.POINTER(Params)]
            lib.dflash_partial_workspace_size.restype = ctypes.c_size_t
            lib.dflash_block_attn_partial.argtypes = [ctypes.POINTER(Params)] + [vp] * 10 + \
                [ctypes.c_size_t, vp]
            lib.dflash_block_attn_partial.restype = i32
            lib.dflash_combine_partials.argtypes = [ctypes.POINTER(Params), i32] + [vp] * 5
            lib.dflash_combine_partials.restype = i32
            lib.dflash_status_string.argtypes = [i32]
            lib.dflash_status_string.restype = ctypes.c_char_p
            lib.dflash_read_device_status.argtypes = [vp, vp]
            lib.dflash_read_device_status.restype = i32
            lib.dflash_clear_device_status.argtypes = [vp, vp]
            lib.dflash_clear_device_status.restype = i32
            lib.dflash_version.argtypes = []
            lib.dflash_version.restype = i32
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().dflash_status_string(int(code)).decode()
