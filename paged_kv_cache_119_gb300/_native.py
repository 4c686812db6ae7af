"""ctypes declarations of libpa.so's C ABI (include/pa.h).  Loading fails loudly
when the library has not been built: there is no fallback implementation."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2, 3
PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = 0, -1, -2, -3, -4
PA_DEVERR_BLOCK_ID, PA_DEVERR_CONTEXT_LEN, PA_DEVERR_SLOT, PA_DEVERR_TIMEOUT = 1, 2, 4, 8
PA_DEVERR_RANGE = 0x10
PA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

# Every symbol include/pa.h and include/pa_block_manager.h declare, with (restype, argtypes).
_i32, _i64, _sz, _vp, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, \
    ctypes.c_float
SIGNATURES = {
    "pa_decode_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_decode": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _vp, ctypes.c_int, _i64, _vp, _i64,
                                 _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp, _sz,
                                 _vp]),
    "pa_decode_noalloc": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _vp, ctypes.c_int, _i64, _vp,
                                         _i64, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32,
                                         _i32, _vp]),
    "pa_decode_fp8": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _i64,
                                     _vp, _i64, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32,
                                     _vp, _sz, _vp]),
    "pa_chunk_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32, _i32]),
    "pa_chunk_attention_fp8": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp, _vp,
                                              _vp, _i64, _vp, _i64, _vp, _vp, _i64, _i32, _i32,
                                              _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp, _sz,
                                              _vp]),
    "pa_decode_partition_tokens": (_i32, [ctypes.c_int, ctypes.c_int, _i32, _i32, _i32, _i32, _i32,
                                          _i32, _i32]),
    "pa_decode_orders_sequences": (_i32, [ctypes.c_int, ctypes.c_int, _i32, _i32, _i32, _i32, _i32,
                                          _i32, _i32]),
    "pa_chunk_partition_tokens": (_i32, [ctypes.c_int, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                         _i32]),
    "pa_chunk_attention": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, _vp, ctypes.c_int, _i64, _vp,
                                          _i64, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _i32, _i32,
                                          _i32, _f32, _i32, _vp, _sz, _vp]),
    "pa_reshape_and_cache_fp8": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                                                _i64, _i32, _i32, _i32, _i64, _vp]),
    "pa_reshape_and_cache": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i64,
                                            ctypes.c_int, _vp]),
    "pa_copy_blocks": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32,
                                      ctypes.POINTER(_i64), _i64, _i64, _i64, _vp]),
    "pa_swap_blocks": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32,
                                      ctypes.POINTER(_i64), _i64, _i64, _i64, _i64, _vp]),
    "pa_decode_kernel_name": (ctypes.c_char_p, [ctypes.c_int, _i32, _i32, _i32]),
    "pa_chunk_kernel_name": (ctypes.c_char_p, [ctypes.c_int, _i32, _i32, _i32, _i32]),
    "pa_stream_read": (ctypes.c_int, [_vp, _sz, _vp, _vp]),
    "pa_stream_read_runs": (ctypes.c_int, [_vp, _sz, ctypes.c_uint32, _vp, ctypes.c_int64, _vp, _vp]),
    "pa_test_arm_wait_timeout": (ctypes.c_int, [_i32, ctypes.c_uint32]),
    "pa_get_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), _vp]),
    "pa_bm_create": (_vp, [_i32, _i32, ctypes.POINTER(_i32)]),
    "pa_bm_destroy": (None, [_vp]),
    "pa_bm_add_sequence": (ctypes.c_int, [_vp, _i64, _i32, ctypes.POINTER(_i64)]),
    "pa_bm_fork": (ctypes.c_int, [_vp, _i64, _i64]),
    "pa_bm_append": (ctypes.c_int, [_vp, ctypes.POINTER(_i64), _i32, ctypes.POINTER(_i64),
                                    ctypes.POINTER(_i64), ctypes.POINTER(_i32)]),
    "pa_bm_free": (ctypes.c_int, [_vp, _i64]),
    "pa_bm_block_tables": (ctypes.c_int, [_vp, ctypes.POINTER(_i64), _i32, ctypes.POINTER(_i32),
                                          _i32, ctypes.POINTER(_i32)]),
    "pa_bm_num_free_blocks": (_i32, [_vp]),
    "pa_bm_ref_count": (_i32, [_vp, _i32]),
    "pa_bm_num_tokens": (_i32, [_vp, _i64]),
    "pa_bm_set_cpu_pool": (ctypes.c_int, [_vp, _i32]),
    "pa_bm_swap_out": (ctypes.c_int, [_vp, ctypes.POINTER(_i64), _i32, ctypes.POINTER(_i64), _i32,
                                      ctypes.POINTER(_i32)]),
    "pa_bm_swap_in": (ctypes.c_int, [_vp, ctypes.POINTER(_i64), _i32, ctypes.POINTER(_i64), _i32,
                                     ctypes.POINTER(_i32)]),
    "pa_bm_num_free_cpu_blocks": (_i32, [_vp]),
    "pa_bm_cpu_ref_count": (_i32, [_vp, _i32]),
    "pa_bm_is_swapped": (_i32, [_vp, _i64]),
    "pa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pa_version": (ctypes.c_char_p, []),
}


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libpa.so.  Raises RuntimeError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libpa.so is not built ({path} missing): run "
                    "`python -c \"import __graft_entry__ as g; g.build()\"` first. "
                    "paged_kv_cache_119_gb300 has no non-CUDA fallback.")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


class PAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = load().pa_status_string(status).decode()
        super().__init__(f"{fn} failed with status {status} ({msg})")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PAError(fn, status)
