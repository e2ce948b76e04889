"""ctypes declarations of the C ABI in include/pkv.h (argument marshalling only).

The shared library is built in-tree (``paged_kv_cache_222_gb300/libpkv.so``).
If it is missing, loading raises: there is no fallback implementation.
"""

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_CUDA = 3
PKV_ERR_WORKSPACE = 4
PKV_ERR_OUT_OF_BLOCKS = 5

PKV_BF16 = 0
PKV_F32 = 1
PKV_E4M3 = 2

DEVERR_NAMES = {0: "none", 1: "wait timeout", 2: "block id out of range",
                3: "context length out of range", 4: "slot out of range"}


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class DecodePlan(ctypes.Structure):
    _fields_ = [("split_tokens", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("mode", ctypes.c_int32),
                ("workers", ctypes.c_int32), ("prefix_split_tokens", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class TraceEntry(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_double)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float

SIGNATURES = {
    "pkv_append": (_I32, [_P, _P, _I32, _I64, _P, _P, _P, ctypes.POINTER(CacheDesc), _P, _P, _I64, _P]),
    "pkv_slot_mapping": (_I32, [_P, _I32, _I32, _P, _P, _I64, ctypes.POINTER(CacheDesc), _P, _P]),
    "pkv_decode_attention": (_I32, [_P, _I32, _I32, _P, _P, ctypes.POINTER(CacheDesc), _P, _I32, _P,
                                    _I32, _F, _P, _P, _P, _I64, _P]),
    "pkv_decode_plan": (_I32, [_I32, _I32, ctypes.POINTER(CacheDesc), _I32, _I32, _I32,
                               ctypes.POINTER(DecodePlan)]),
    "pkv_decode_attention_ex": (_I32, [_P, _I32, _I32, _P, _P, ctypes.POINTER(CacheDesc), _P, _I32,
                                       _P, _I32, _F, _P, _P, _P, _I64, _P, ctypes.c_size_t, _I32, _P]),
    "pkv_decode_attention_noalloc": (_I32, [_P, _I32, _I32, _P, _P, ctypes.POINTER(CacheDesc), _P, _I32,
                                            _P, _I32, _F, _P, _P, _P, _I64, _P]),
    "pkv_decode_attention_append": (_I32, [_P, _I32, _I32, _P, _P, ctypes.POINTER(CacheDesc), _P, _P, _I32,
                                           _P, _I32, _P, _I32, _F, _P, _P, _P, _I64, _P, ctypes.c_size_t,
                                           _I32, _P]),
    "pkv_cascade_plan": (_I32, [_I32, _I32, ctypes.POINTER(CacheDesc), _I32, _I32, _I32,
                                ctypes.POINTER(DecodePlan)]),
    "pkv_cascade_decode_attention": (_I32, [_P, _I32, _I32, _P, _P, ctypes.POINTER(CacheDesc), _P, _I32,
                                            _P, _I32, _P, _I32, _F, _P, _P, ctypes.c_size_t, _P]),
    "pkv_multi_query_plan": (_I32, [_I32, _I32, _I32, ctypes.POINTER(CacheDesc), _I32, _I32, _I32,
                                    ctypes.POINTER(DecodePlan)]),
    "pkv_multi_query_attention": (_I32, [_P, _I32, _I32, _I32, _P, _P, ctypes.POINTER(CacheDesc), _P, _I32,
                                         _P, _I32, _F, _P, _P, ctypes.c_size_t, _I32, _P]),
    "pkv_copy_blocks": (_I32, [_P, _P, ctypes.POINTER(CacheDesc), _P, _P, _I32, _P]),
    "pkv_bm_create": (_I32, [_I64, _I32, ctypes.POINTER(_P)]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_num_free": (_I64, [_P]),
    "pkv_bm_ref_count": (_I32, [_P, _I64]),
    "pkv_bm_seq_len": (_I64, [_P, _I64]),
    "pkv_bm_num_sequences": (_I64, [_P]),
    "pkv_bm_add_sequence": (_I32, [_P, _I64]),
    "pkv_bm_fork": (_I32, [_P, _I64, _I64]),
    "pkv_bm_free_sequence": (_I32, [_P, _I64]),
    "pkv_bm_append": (_I32, [_P, _I32, _P, _P, _P, _P, _P, _I32, ctypes.POINTER(_I32)]),
    "pkv_bm_blocks_needed": (_I32, [_P, _I32, _P, _P, ctypes.POINTER(_I64)]),
    "pkv_bm_block_tables": (_I32, [_P, _I32, _P, _I32, _P, _P]),
    "pkv_bm_set_host_blocks": (_I32, [_P, _I64]),
    "pkv_bm_num_free_host": (_I64, [_P]),
    "pkv_bm_host_entries": (_I64, [_P, _I64]),
    "pkv_bm_evict": (_I32, [_P, _I64, _I32, _P, _P, _P, ctypes.POINTER(_I32)]),
    "pkv_bm_stage": (_I32, [_P, _I64, _I32, _P, _P, _P, ctypes.POINTER(_I32)]),
    "pkv_bm_table_entries": (_I32, [_P, _I64, _I32, _P, _P, ctypes.POINTER(_I32)]),
    "pkv_bm_prefetch_candidates": (_I32, [_P, _I64, _P, _F, _I32, _P, ctypes.POINTER(_I32)]),
    "pkv_copy_blocks_between": (_I32, [_P, _P, _I64, _P, _P, _I64, ctypes.POINTER(CacheDesc), _P, _P, _I32, _I32,
                                       _P]),
    "pkv_host_alloc": (_I32, [ctypes.c_size_t, ctypes.POINTER(_P)]),
    "pkv_host_free": (_I32, [_P]),
    "pkv_selftest_wait_timeout": (_I32, [_I32, _I32, _P]),
    "pkv_get_device_error": (_I32, [_P]),
    "pkv_status_string": (ctypes.c_char_p, [_I32]),
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_abi_version": (_I32, []),
    "pkv_trace_enable": (_I32, [_I32]),
    "pkv_trace_read": (_I32, [ctypes.POINTER(TraceEntry), _I32]),
    "pkv_shutdown": (_I32, []),
}

_lock = threading.Lock()
_lib = None


def load(path=LIB_PATH):
    """Load libpkv.so once and declare every entry point."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is not built; run `python -m paged_kv_cache_222_gb300.build` "
                "(the CUDA library is required; there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class PkvError(RuntimeError):
    def __init__(self, status, where):
        lib = load()
        detail = lib.pkv_last_error().decode()
        name = lib.pkv_status_string(status).decode()
        super().__init__(f"{where}: {name}: {detail}")
        self.status = status


def check(status, where):
    if status != PKV_OK:
        raise PkvError(status, where)
