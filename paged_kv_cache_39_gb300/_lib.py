"""ctypes loader for ``libkvpaged.so`` (the C ABI of ``include/kvpaged.h``).

There is no fallback: if the library has not been built (``build()`` in the
repository's entry module, or ``python -m paged_kv_cache_39_gb300.build``),
loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvpaged.so")

KV_OK, KV_EINVAL, KV_EUNSUPPORTED, KV_ECUDA = 0, -1, -2, -3
ERR_BITS = {
    "BAD_BLOCK": 1,
    "BAD_SLOT": 2,
    "BAD_POSITION": 4,
    "BAD_RANGE": 8,
    "NULL_WRITE": 16,
    "BAD_QSL": 32,
    "OUT_OF_SPACE": 64,
    "TIMEOUT": 128,
}
PAD_SLOT_ID = -1
NULL_BLOCK_ID = 0
MAX_RANGES_PER_REQ = 256
MAX_GATHER_REQS = 4096
MAX_TOKENS = 2147418112  # largest max_num_tokens of one slot-mapping call (2^31 - 65536)

# Every entry point the header declares, with its argument and result types.
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
SIGNATURES = {
    "kv_slot_mapping_paged": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _P, _P, _P],
                              ctypes.c_int),
    "kv_slot_mapping_paged_cp": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _I32, _I32, _I32,
                                  _P, _P, _P], ctypes.c_int),
    "kv_slot_mapping_range": ([_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _P, _P, _P],
                              ctypes.c_int),
    "kv_cache_write": ([_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _P, _P],
                       ctypes.c_int),
    "kv_slot_mapping_paged_write": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _P, _P, _P,
                                     _P, _I32, _I32, _I32, _P, _P, _P], ctypes.c_int),
    "kv_slot_mapping_range_write": ([_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _P,
                                     _P, _P, _P, _I32, _I32, _I32, _P, _P, _P], ctypes.c_int),
    "kv_cache_gather": ([_P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _P, _I32, _P, _P, _I32, _P, _P,
                         _I64, _P, _P], ctypes.c_int),
    "kv_cache_gather_bulk": ([_P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _P, _I32, _P, _P, _I32, _P,
                              _P, _I64, _P, _P], ctypes.c_int),
    "kv_expand_kernel_blocks": ([_P, _I32, _I32, _I32, _I32, _P, _I32, _P, _P], ctypes.c_int),
    "kv_table_from_ranges": ([_P, _P, _P, _I32, _I32, _P, _I32, _P, _P], ctypes.c_int),
    "kv_cache_gather_range": ([_P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _P, _P, _P, _I32, _P, _P,
                               _I32, _P, _P, _I64, _P, _P], ctypes.c_int),
    "kv_copy_blocks": ([_P, _P, _I32, _I64, _I32, _I32, _I32, _P, _P, _I32, _P, _P], ctypes.c_int),
    "kv_copy_blocks_bulk": ([_P, _P, _I32, _I64, _I32, _I32, _I32, _P, _P, _I32, _P, _P],
                            ctypes.c_int),
    "kv_diag_bounded_wait": ([_I32, _P, _P], ctypes.c_int),
    "kv_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "kv_abi_version": ([], ctypes.c_int),
}

_lock = threading.Lock()
_lib = None


class KVError(RuntimeError):
    """A kv_* call returned a negative kv_status."""

    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def check(fn: str, status: int) -> None:
    if status != KV_OK:
        msg = load().kv_status_string(status).decode()
        raise KVError(fn, status, msg)
