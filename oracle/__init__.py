"""CPU oracle of the paged KV-cache hot path (numpy front end over kv_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
the benchmark's CPU-baseline leg and reference arm may import this package.  It shares no code
with the CUDA library and never imports it; both sides are fed by the seeded
generators in ``paged_kv_cache_39_gb300.workloads``.

Each function mirrors one entry point of the C oracle and cites, in
``kv_oracle.c``, the page passage it follows.  Arrays are numpy; bf16 values
are carried as their raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

from .build import build_oracle, library_path

PAD_SLOT = -1
NULL_BLOCK = 0
RANGE_CAP = 256
ERR_BITS = {
    "BAD_BLOCK": 1,
    "BAD_SLOT": 2,
    "BAD_POSITION": 4,
    "BAD_RANGE": 8,
    "NULL_WRITE": 16,
    "BAD_QSL": 32,
    "OUT_OF_SPACE": 64,
}
OK, EINVAL, EUNSUPPORTED = 0, -1, -2

_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("KV_ORACLE_LIB") or library_path()
    if not os.path.exists(path):
        build_oracle()
    lib = ctypes.CDLL(path)
    sigs = {
        "orc_coord": ([_I64, _I64, _I64, _I64, _I64], _I64),
        "orc_slot_mapping_paged": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _P, _P], ctypes.c_int),
        "orc_slot_mapping_paged_cp": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _I32, _I32,
                                       _I32, _P, _P], ctypes.c_int),
        "orc_slot_mapping_range": ([_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, _P, _P],
                                   ctypes.c_int),
        "orc_table_from_ranges": ([_P, _P, _P, _I32, _I32, _I32, _P, _P], ctypes.c_int),
        "orc_gather_rows_range": ([_I32, _I64, _I32, _P, _P, _P, _I32, _P, _P, _I32, _I64, _P, _P],
                                  ctypes.c_int),
        "orc_copy_blocks": ([_P, _P, _I32, _I64, _I32, _I32, _I32, _P, _P, _I32, _P], ctypes.c_int),
        "orc_cache_write": ([_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _P], ctypes.c_int),
        "orc_write_rows": ([_P, _I32, _I32, _I64, _I32, _P, _P], ctypes.c_int),
        "orc_gather_rows": ([_I32, _I64, _I32, _P, _I32, _P, _P, _I32, _I64, _P, _P], ctypes.c_int),
        "orc_cache_gather": ([_P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _P, _I32, _P, _P, _I32,
                              _P, _P, _I64, _P, _P], ctypes.c_int),
        "orc_expand_kernel_blocks": ([_P, _I32, _I32, _I32, _I32, _P, _I32, _P], ctypes.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"oracle rejected the arguments (status {status})")
        self.status = status


def _check(rc: int):
    if rc != OK:
        raise OracleError(rc)


def coord(layer: int, block: int, token: int, num_blocks: int, block_size: int) -> int:
    return int(_load().orc_coord(layer, block, token, num_blocks, block_size))


def slot_mapping_paged(qsl, positions, block_table, num_tokens: int, max_num_tokens: int,
                       block_size: int, num_blocks: int) -> Tuple[np.ndarray, int]:
    """Per-token slots through the block table; returns (slot_mapping, error word)."""
    qsl = _c(qsl, np.int32)
    positions = _c(positions, np.int64)
    table = _c(block_table, np.int32)
    if table.ndim != 2:
        raise ValueError("block_table must be [rows, stride]")
    R = len(qsl) - 1
    out = np.empty(max_num_tokens, dtype=np.int64)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_slot_mapping_paged(_ptr(qsl), _ptr(positions), _ptr(table), table.shape[1], R,
                                          num_tokens, max_num_tokens, block_size, num_blocks,
                                          _ptr(out), _ptr(err)))
    return out, int(err[0])


def slot_mapping_paged_cp(qsl, positions, block_table, num_tokens: int, max_num_tokens: int,
                          block_size: int, num_blocks: int, cp_world_size: int, cp_rank: int,
                          cp_interleave: int) -> Tuple[np.ndarray, int]:
    """Context-parallel paged slot mapping (parity unpinned beyond world size 1)."""
    qsl = _c(qsl, np.int32)
    positions = _c(positions, np.int64)
    table = _c(block_table, np.int32)
    R = len(qsl) - 1
    out = np.empty(max_num_tokens, dtype=np.int64)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_slot_mapping_paged_cp(_ptr(qsl), _ptr(positions), _ptr(table),
                                             table.shape[1], R, num_tokens, max_num_tokens,
                                             block_size, num_blocks, cp_world_size, cp_rank,
                                             cp_interleave, _ptr(out), _ptr(err)))
    return out, int(err[0])


def slot_mapping_range(qsl, positions, range_start, range_len, num_ranges, num_tokens: int,
                       max_num_tokens: int, block_size: int, num_blocks: int
                       ) -> Tuple[np.ndarray, int]:
    """Per-token slots from contiguous range descriptors; returns (slots, error word)."""
    qsl = _c(qsl, np.int32)
    positions = _c(positions, np.int64)
    rs = _c(range_start, np.int32)
    rl = _c(range_len, np.int32)
    nr = _c(num_ranges, np.int32)
    R = len(qsl) - 1
    out = np.empty(max_num_tokens, dtype=np.int64)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_slot_mapping_range(_ptr(qsl), _ptr(positions), _ptr(rs), _ptr(rl), _ptr(nr),
                                          rs.shape[1], R, num_tokens, max_num_tokens, block_size,
                                          num_blocks, _ptr(out), _ptr(err)))
    return out, int(err[0])


def table_from_ranges(range_start, range_len, num_ranges, table_stride: int,
                      with_error: bool = False):
    """Block table [rows, table_stride] expanded from the range descriptors."""
    rs = _c(range_start, np.int32)
    rl = _c(range_len, np.int32)
    nr = _c(num_ranges, np.int32)
    R = rs.shape[0]
    table = np.empty((R, table_stride), dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_table_from_ranges(_ptr(rs), _ptr(rl), _ptr(nr), rs.shape[1], R,
                                         table_stride, _ptr(table), _ptr(err)))
    return (table, int(err[0])) if with_error else table


def cache_write(key, value, k_cache, v_cache, slot_mapping, num_blocks: int,
                block_size: int) -> int:
    """Scatter key/value [L, N, H, D] (uint16 bits) into k_cache/v_cache in place.

    ``k_cache``/``v_cache`` are uint16 ``[L, B, T, H, D]`` arrays, modified in
    place.  Returns the error word.
    """
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    slot = _c(slot_mapping, np.int64)
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags["C_CONTIGUOUS"]:
            raise ValueError("caches must be C-contiguous uint16 arrays")
    L, N, H, D = key.shape
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_cache_write(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot),
                                   N, L, num_blocks, block_size, H, D, _ptr(err)))
    return int(err[0])


def write_rows(slot_mapping, num_tokens: int, num_layers: int, num_blocks: int,
               block_size: int) -> Tuple[np.ndarray, int]:
    """Destination cache row of every (layer, token), -1 where skipped: [L, N]."""
    slot = _c(slot_mapping, np.int64)
    out = np.empty((num_layers, num_tokens), dtype=np.int64)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_write_rows(_ptr(slot), num_tokens, num_layers, num_blocks, block_size,
                                  _ptr(out), _ptr(err)))
    return out, int(err[0])


def gather_rows(layer: int, num_blocks: int, block_size: int, block_table, gather_start,
                gather_end, out_rows: int) -> Tuple[np.ndarray, int]:
    """Source row of each output row (>=0 cache row, -1 zero, -2 not written)."""
    table = _c(block_table, np.int32)
    g0 = _c(gather_start, np.int32)
    g1 = _c(gather_end, np.int32)
    out = np.empty(out_rows, dtype=np.int64)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_gather_rows(layer, num_blocks, block_size, _ptr(table), table.shape[1],
                                   _ptr(g0), _ptr(g1), len(g0), out_rows, _ptr(out), _ptr(err)))
    return out, int(err[0])


def gather_rows_range(layer: int, num_blocks: int, block_size: int, range_start, range_len,
                      num_ranges, gather_start, gather_end, out_rows: int) -> Tuple[np.ndarray, int]:
    """Source row of each output row of the range-addressed gather."""
    rs = _c(range_start, np.int32)
    rl = _c(range_len, np.int32)
    nr = _c(num_ranges, np.int32)
    g0 = _c(gather_start, np.int32)
    g1 = _c(gather_end, np.int32)
    out = np.empty(out_rows, dtype=np.int64)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_gather_rows_range(layer, num_blocks, block_size, _ptr(rs), _ptr(rl),
                                         _ptr(nr), rs.shape[1], _ptr(g0), _ptr(g1), len(g0),
                                         out_rows, _ptr(out), _ptr(err)))
    return out, int(err[0])


def copy_blocks(k_cache, v_cache, src_blocks, dst_blocks) -> int:
    """Copy whole blocks src -> dst in every layer of both caches (in place)."""
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags["C_CONTIGUOUS"] or c.ndim != 5:
            raise ValueError("caches must be C-contiguous uint16 [L, B, T, H, D] arrays")
    L, B, T, H, D = k_cache.shape
    src = _c(src_blocks, np.int32)
    dst = _c(dst_blocks, np.int32)
    if len(src) != len(dst):
        raise ValueError("src and dst differ in length")
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), L, B, T, H, D, _ptr(src),
                                   _ptr(dst), len(src), _ptr(err)))
    return int(err[0])


def cache_gather(k_cache, v_cache, layer: int, num_blocks: int, block_size: int, block_table,
                 gather_start, gather_end, k_out, v_out) -> int:
    """Gather rows into k_out/v_out (uint16 [out_rows, H, D], modified in place)."""
    L, B, T, H, D = k_cache.shape
    assert B == num_blocks and T == block_size
    table = _c(block_table, np.int32)
    g0 = _c(gather_start, np.int32)
    g1 = _c(gather_end, np.int32)
    out_rows = k_out.shape[0]
    scratch = np.empty(out_rows, dtype=np.int64)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_cache_gather(_ptr(k_cache), _ptr(v_cache), layer, L, num_blocks, block_size,
                                    H, D, _ptr(table), table.shape[1], _ptr(g0), _ptr(g1), len(g0),
                                    _ptr(k_out), _ptr(v_out), out_rows, _ptr(scratch), _ptr(err)))
    return int(err[0])


def expand_kernel_blocks(mgr_table, mgr_block_size: int, kernel_block_size: int,
                         kernel_stride: Optional[int] = None) -> Tuple[np.ndarray, int]:
    table = _c(mgr_table, np.int32)
    R, Ms = table.shape
    if kernel_stride is None:
        if kernel_block_size <= 0 or mgr_block_size % kernel_block_size != 0:
            kernel_stride = Ms
        else:
            kernel_stride = Ms * (mgr_block_size // kernel_block_size)
    out = np.empty((R, kernel_stride), dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    _check(_load().orc_expand_kernel_blocks(_ptr(table), R, Ms, mgr_block_size, kernel_block_size,
                                            _ptr(out), kernel_stride, _ptr(err)))
    return out, int(err[0])
