"""Torch-facing wrappers of the C ABI (argument marshalling only).

Each function has the name of the C entry point it calls, takes CUDA tensors,
checks their dtype, device and contiguity, passes raw pointers and the
current CUDA stream, and raises ``KVError`` on a negative status.  All work
runs in the CUDA kernels; nothing here computes on the host.

``err`` is an optional int32 CUDA tensor of one element: data errors the
kernels detect are OR-ed into it (see ``ERR_BITS``).

``prepare=True`` validates the arguments once and returns a ``Prepared``
call instead of launching: calling it launches the same kernel on the
then-current stream with the cached pointers, so a loop over persistent
buffers (a serving step) pays for the C call alone.  The prepared call
keeps its tensors alive; their contents may change between calls, their
storage must not.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from ._lib import check, load

__all__ = [
    "Prepared",
    "kv_slot_mapping_paged",
    "kv_slot_mapping_paged_cp",
    "kv_slot_mapping_range",
    "kv_cache_write",
    "kv_slot_mapping_paged_write",
    "kv_slot_mapping_range_write",
    "kv_cache_gather",
    "kv_expand_kernel_blocks",
    "kv_table_from_ranges",
    "kv_cache_gather_range",
    "kv_copy_blocks",
    "new_error_word",
]


class Prepared:
    """A validated call of one entry point; calling it launches again."""

    __slots__ = ("name", "_fn", "_args", "_device", "_keep", "result")

    def __init__(self, name, fn, args, device, keep, result):
        self.name, self._fn, self._args, self._device = name, fn, args, device
        self._keep, self.result = keep, result

    def __call__(self):
        check(self.name, self._fn(*self._args,
                                  torch.cuda.current_stream(self._device).cuda_stream))
        return self.result


def _run(name: str, args: tuple, device: int, keep: tuple, result, prepare: bool):
    fn = getattr(load(), name)
    if prepare:
        return Prepared(name, fn, args, device, keep, result)
    check(name, fn(*args, torch.cuda.current_stream(device).cuda_stream))
    return result


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None or t.numel() == 0:
        return None
    return t.data_ptr()


def _cuda_check(t, name: str) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the kernels take device pointers), "
                         f"got {t.device}")


def _device_of(t: torch.Tensor, name: str) -> int:
    _cuda_check(t, name)
    return t.get_device()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device: int) -> None:
    _cuda_check(t, name)
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.get_device() != device:
        raise ValueError(f"{name} must live on cuda:{device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _err_ptr(err: Optional[torch.Tensor], device: int) -> Optional[int]:
    if err is None:
        return None
    _need(err, "err", torch.int32, device)
    if err.numel() < 1:
        raise ValueError("err needs one element")
    return err.data_ptr()


def new_error_word(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def _slot_common(query_start_loc, positions, max_num_tokens, slot_mapping, num_tokens):
    """Shared argument checks of the slot maps: (device, num_reqs, n, n_max, output)."""
    dev = _device_of(positions, "positions")
    _need(query_start_loc, "query_start_loc", torch.int32, dev)
    _need(positions, "positions", torch.int64, dev)
    n = positions.numel() if num_tokens is None else int(num_tokens)
    if n > positions.numel():
        raise ValueError("num_tokens exceeds positions")
    n_max = n if max_num_tokens is None else int(max_num_tokens)
    if slot_mapping is None:
        slot_mapping = torch.empty(n_max, dtype=torch.int64, device=positions.device)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    if slot_mapping.numel() < n_max:
        raise ValueError("slot_mapping is shorter than max_num_tokens")
    return dev, max(query_start_loc.numel() - 1, 0), n, n_max, slot_mapping


def _table_check(block_table, dev, num_reqs):
    _need(block_table, "block_table", torch.int32, dev)
    if block_table.dim() != 2:
        raise ValueError("block_table must be [num_reqs, table_stride]")
    if block_table.shape[0] < num_reqs:
        raise ValueError("block_table has fewer rows than requests")


def _ranges_check(range_start, range_len, num_ranges, dev, num_reqs):
    for name, t in (("range_start", range_start), ("range_len", range_len),
                    ("num_ranges", num_ranges)):
        _need(t, name, torch.int32, dev)
    if range_start.dim() != 2 or range_len.shape != range_start.shape:
        raise ValueError("range_start/range_len must both be [num_reqs, range_stride]")
    if range_start.shape[0] < num_reqs or num_ranges.numel() < num_reqs:
        raise ValueError("descriptor arrays have fewer rows than requests")


def kv_slot_mapping_paged(query_start_loc: torch.Tensor, positions: torch.Tensor,
                          block_table: torch.Tensor, block_size: int, num_blocks: int,
                          max_num_tokens: Optional[int] = None,
                          slot_mapping: Optional[torch.Tensor] = None,
                          num_tokens: Optional[int] = None,
                          err: Optional[torch.Tensor] = None, prepare: bool = False):
    """slot_mapping[t] through ``block_table`` [num_reqs, stride] (int32)."""
    dev, R, n, n_max, slot_mapping = _slot_common(query_start_loc, positions, max_num_tokens,
                                                  slot_mapping, num_tokens)
    _table_check(block_table, dev, R)
    args = (_ptr(query_start_loc), _ptr(positions), _ptr(block_table), block_table.shape[1], R,
            n, n_max, int(block_size), int(num_blocks), _ptr(slot_mapping), _err_ptr(err, dev))
    return _run("kv_slot_mapping_paged", args, dev,
                (query_start_loc, positions, block_table, slot_mapping, err), slot_mapping,
                prepare)


def kv_slot_mapping_paged_cp(query_start_loc: torch.Tensor, positions: torch.Tensor,
                             block_table: torch.Tensor, block_size: int, num_blocks: int,
                             cp_world_size: int, cp_rank: int, cp_interleave: int = 1,
                             max_num_tokens: Optional[int] = None,
                             slot_mapping: Optional[torch.Tensor] = None,
                             num_tokens: Optional[int] = None,
                             err: Optional[torch.Tensor] = None, prepare: bool = False):
    """kv_slot_mapping_paged for one rank of context parallelism (see the header)."""
    dev, R, n, n_max, slot_mapping = _slot_common(query_start_loc, positions, max_num_tokens,
                                                  slot_mapping, num_tokens)
    _table_check(block_table, dev, R)
    args = (_ptr(query_start_loc), _ptr(positions), _ptr(block_table), block_table.shape[1], R,
            n, n_max, int(block_size), int(num_blocks), int(cp_world_size), int(cp_rank),
            int(cp_interleave), _ptr(slot_mapping), _err_ptr(err, dev))
    return _run("kv_slot_mapping_paged_cp", args, dev,
                (query_start_loc, positions, block_table, slot_mapping, err), slot_mapping,
                prepare)


def kv_slot_mapping_range(query_start_loc: torch.Tensor, positions: torch.Tensor,
                          range_start: torch.Tensor, range_len: torch.Tensor,
                          num_ranges: torch.Tensor, block_size: int, num_blocks: int,
                          max_num_tokens: Optional[int] = None,
                          slot_mapping: Optional[torch.Tensor] = None,
                          num_tokens: Optional[int] = None,
                          err: Optional[torch.Tensor] = None, prepare: bool = False):
    """slot_mapping[t] through per-request range descriptors [num_reqs, range_stride]."""
    dev, R, n, n_max, slot_mapping = _slot_common(query_start_loc, positions, max_num_tokens,
                                                  slot_mapping, num_tokens)
    _ranges_check(range_start, range_len, num_ranges, dev, R)
    args = (_ptr(query_start_loc), _ptr(positions), _ptr(range_start), _ptr(range_len),
            _ptr(num_ranges), range_start.shape[1], R, n, n_max, int(block_size),
            int(num_blocks), _ptr(slot_mapping), _err_ptr(err, dev))
    return _run("kv_slot_mapping_range", args, dev,
                (query_start_loc, positions, range_start, range_len, num_ranges, slot_mapping,
                 err), slot_mapping, prepare)


def _cache_dims(k_cache: torch.Tensor, v_cache: torch.Tensor, dev: int
                ) -> Tuple[int, int, int, int, int]:
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    if k_cache.dim() != 5:
        raise ValueError("caches must be [num_layers, num_blocks, block_size, kv_heads, head_dim]")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    return tuple(int(x) for x in k_cache.shape)


def kv_cache_write(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                   num_tokens: Optional[int] = None,
                   err: Optional[torch.Tensor] = None, prepare: bool = False):
    """Scatter key/value [L, N, H, D] (bf16) into the [L, B, T, H, D] caches.

    Returns None (or the ``Prepared`` call)."""
    dev = _device_of(key, "key")
    _need(key, "key", torch.bfloat16, dev)
    _need(value, "value", torch.bfloat16, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    L, B, T, H, D = _cache_dims(k_cache, v_cache, dev)
    if key.dim() != 4 or key.shape[0] != L or key.shape[2:] != (H, D) or value.shape != key.shape:
        raise ValueError("key/value must be [num_layers, num_tokens, kv_heads, head_dim]")
    n = key.shape[1] if num_tokens is None else int(num_tokens)
    if n > key.shape[1] or slot_mapping.numel() < n:
        raise ValueError("num_tokens exceeds key rows or slot_mapping")
    if n != key.shape[1] and L > 1:
        raise ValueError("num_tokens must equal key.shape[1] for multi-layer writes")
    args = (_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), n, L, B,
            T, H, D, _err_ptr(err, dev))
    return _run("kv_cache_write", args, dev, (key, value, k_cache, v_cache, slot_mapping, err),
                None, prepare)


def _rows_check(key, value, k_cache, v_cache, dev, n):
    """Shapes of the write half of the fused calls: (L, H, D, row arguments)."""
    _need(key, "key", torch.bfloat16, dev)
    _need(value, "value", torch.bfloat16, dev)
    L, B, T, H, D = _cache_dims(k_cache, v_cache, dev)
    if key.dim() != 4 or key.shape[0] != L or key.shape[2:] != (H, D) or value.shape != key.shape:
        raise ValueError("key/value must be [num_layers, num_tokens, kv_heads, head_dim]")
    if n > key.shape[1]:
        raise ValueError("num_tokens exceeds key rows")
    if n != key.shape[1] and L > 1:
        raise ValueError("num_tokens must equal key.shape[1] for multi-layer writes")
    return (_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), L, H, D)


def kv_slot_mapping_paged_write(query_start_loc: torch.Tensor, positions: torch.Tensor,
                                block_table: torch.Tensor, block_size: int, num_blocks: int,
                                key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                                v_cache: torch.Tensor, max_num_tokens: Optional[int] = None,
                                slot_mapping: Optional[torch.Tensor] = None,
                                num_tokens: Optional[int] = None,
                                err: Optional[torch.Tensor] = None, prepare: bool = False):
    """kv_slot_mapping_paged then kv_cache_write on its slots, in one launch.

    ``num_blocks`` must equal the caches' block count.  Returns slot_mapping."""
    dev, R, n, n_max, slot_mapping = _slot_common(query_start_loc, positions, max_num_tokens,
                                                  slot_mapping, num_tokens)
    _table_check(block_table, dev, R)
    rows = _rows_check(key, value, k_cache, v_cache, dev, n)
    if int(num_blocks) != k_cache.shape[1]:
        raise ValueError("num_blocks differs from the caches' block count")
    if int(block_size) != k_cache.shape[2]:
        raise ValueError("block_size differs from the caches' block size")
    args = (_ptr(query_start_loc), _ptr(positions), _ptr(block_table), block_table.shape[1], R,
            n, n_max, int(block_size), int(num_blocks), *rows, _ptr(slot_mapping),
            _err_ptr(err, dev))
    return _run("kv_slot_mapping_paged_write", args, dev,
                (query_start_loc, positions, block_table, key, value, k_cache, v_cache,
                 slot_mapping, err), slot_mapping, prepare)


def kv_slot_mapping_range_write(query_start_loc: torch.Tensor, positions: torch.Tensor,
                                range_start: torch.Tensor, range_len: torch.Tensor,
                                num_ranges: torch.Tensor, block_size: int, num_blocks: int,
                                key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                                v_cache: torch.Tensor, max_num_tokens: Optional[int] = None,
                                slot_mapping: Optional[torch.Tensor] = None,
                                num_tokens: Optional[int] = None,
                                err: Optional[torch.Tensor] = None, prepare: bool = False):
    """kv_slot_mapping_range then kv_cache_write on its slots, in one launch."""
    dev, R, n, n_max, slot_mapping = _slot_common(query_start_loc, positions, max_num_tokens,
                                                  slot_mapping, num_tokens)
    _ranges_check(range_start, range_len, num_ranges, dev, R)
    rows = _rows_check(key, value, k_cache, v_cache, dev, n)
    if int(num_blocks) != k_cache.shape[1]:
        raise ValueError("num_blocks differs from the caches' block count")
    if int(block_size) != k_cache.shape[2]:
        raise ValueError("block_size differs from the caches' block size")
    args = (_ptr(query_start_loc), _ptr(positions), _ptr(range_start), _ptr(range_len),
            _ptr(num_ranges), range_start.shape[1], R, n, n_max, int(block_size),
            int(num_blocks), *rows, _ptr(slot_mapping), _err_ptr(err, dev))
    return _run("kv_slot_mapping_range_write", args, dev,
                (query_start_loc, positions, range_start, range_len, num_ranges, key, value,
                 k_cache, v_cache, slot_mapping, err), slot_mapping, prepare)


def _gather_outputs(k_cache, gather_start, gather_end, k_out, v_out, out_rows, H, D, dev):
    _need(gather_start, "gather_start", torch.int32, dev)
    _need(gather_end, "gather_end", torch.int32, dev)
    if k_out is None:
        if out_rows is None:
            # the total span length lives on the device: reading it back here
            # would synchronise the stream inside an asynchronous call
            raise ValueError("give out_rows (or k_out/v_out) for the gather")
        k_out = torch.empty((out_rows, H, D), dtype=torch.bfloat16, device=k_cache.device)
        v_out = torch.empty((out_rows, H, D), dtype=torch.bfloat16, device=k_cache.device)
    _need(k_out, "k_out", torch.bfloat16, dev)
    _need(v_out, "v_out", torch.bfloat16, dev)
    rows = k_out.shape[0] if out_rows is None else int(out_rows)
    for t in (k_out, v_out):
        if t.dim() < 1 or t.shape[0] < rows or t.numel() < rows * H * D:
            raise ValueError("outputs are smaller than out_rows rows of kv_heads x head_dim")
    return k_out, v_out, rows


def kv_cache_gather(k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                    gather_start: torch.Tensor, gather_end: torch.Tensor, layer: int = 0,
                    k_out: Optional[torch.Tensor] = None, v_out: Optional[torch.Tensor] = None,
                    out_rows: Optional[int] = None,
                    err: Optional[torch.Tensor] = None, bulk: bool = False,
                    prepare: bool = False):
    """Gather positions [start_r, end_r) of every request into packed [rows, H, D] buffers.

    ``out_rows`` (or, when it is None, the given outputs' row count) must be
    at least the total span length.  Without outputs ``out_rows`` is required:
    the spans live on the device, and the call never reads them back (it does
    not synchronise and can be captured in a CUDA graph).
    ``bulk=True`` calls kv_cache_gather_bulk (bulk-copy engine) instead.
    Returns (k_out, v_out).
    """
    dev = _device_of(k_cache, "k_cache")
    L, B, T, H, D = _cache_dims(k_cache, v_cache, dev)
    _need(block_table, "block_table", torch.int32, dev)
    if block_table.dim() != 2:
        raise ValueError("block_table must be [num_reqs, table_stride]")
    R = gather_start.numel()
    if gather_end.numel() != R or block_table.shape[0] < R:
        raise ValueError("gather spans and block_table rows disagree")
    k_out, v_out, rows = _gather_outputs(k_cache, gather_start, gather_end, k_out, v_out,
                                         out_rows, H, D, dev)
    name = "kv_cache_gather_bulk" if bulk else "kv_cache_gather"
    args = (_ptr(k_cache), _ptr(v_cache), int(layer), L, B, T, H, D, _ptr(block_table),
            block_table.shape[1], _ptr(gather_start), _ptr(gather_end), R, _ptr(k_out),
            _ptr(v_out), rows, _err_ptr(err, dev))
    return _run(name, args, dev,
                (k_cache, v_cache, block_table, gather_start, gather_end, k_out, v_out, err),
                (k_out, v_out), prepare)


def kv_expand_kernel_blocks(mgr_table: torch.Tensor, mgr_block_size: int,
                            kernel_block_size: int,
                            kernel_table: Optional[torch.Tensor] = None,
                            err: Optional[torch.Tensor] = None, prepare: bool = False):
    """Expand an int32 [R, Ms] manager table into an int32 [R, Ks] kernel table."""
    dev = _device_of(mgr_table, "mgr_table")
    _need(mgr_table, "mgr_table", torch.int32, dev)
    if mgr_table.dim() != 2:
        raise ValueError("mgr_table must be [num_reqs, mgr_stride]")
    R, Ms = mgr_table.shape
    if kernel_table is None:
        k = mgr_block_size // kernel_block_size if kernel_block_size > 0 else 1
        kernel_table = torch.empty((R, Ms * max(k, 1)), dtype=torch.int32,
                                   device=mgr_table.device)
    _need(kernel_table, "kernel_table", torch.int32, dev)
    if kernel_table.dim() != 2 or kernel_table.shape[0] != R:
        raise ValueError("kernel_table must be [num_reqs, kernel_stride]")
    args = (_ptr(mgr_table), R, Ms, int(mgr_block_size), int(kernel_block_size),
            _ptr(kernel_table), kernel_table.shape[1], _err_ptr(err, dev))
    return _run("kv_expand_kernel_blocks", args, dev, (mgr_table, kernel_table, err),
                kernel_table, prepare)


def kv_table_from_ranges(range_start: torch.Tensor, range_len: torch.Tensor,
                         num_ranges: torch.Tensor, table_stride: Optional[int] = None,
                         block_table: Optional[torch.Tensor] = None,
                         err: Optional[torch.Tensor] = None, prepare: bool = False):
    """Block table int32 [num_reqs, table_stride] expanded from range descriptors."""
    dev = _device_of(range_start, "range_start")
    R = range_start.shape[0] if range_start.dim() == 2 else 0
    _ranges_check(range_start, range_len, num_ranges, dev, R)
    if block_table is None:
        if table_stride is None:
            raise ValueError("give table_stride or block_table")
        block_table = torch.empty((R, int(table_stride)), dtype=torch.int32,
                                  device=range_start.device)
    _need(block_table, "block_table", torch.int32, dev)
    if block_table.dim() != 2 or block_table.shape[0] != R:
        raise ValueError("block_table must be [num_reqs, table_stride]")
    args = (_ptr(range_start), _ptr(range_len), _ptr(num_ranges), range_start.shape[1], R,
            _ptr(block_table), block_table.shape[1], _err_ptr(err, dev))
    return _run("kv_table_from_ranges", args, dev,
                (range_start, range_len, num_ranges, block_table, err), block_table, prepare)


def kv_cache_gather_range(k_cache: torch.Tensor, v_cache: torch.Tensor,
                          range_start: torch.Tensor, range_len: torch.Tensor,
                          num_ranges: torch.Tensor, gather_start: torch.Tensor,
                          gather_end: torch.Tensor, layer: int = 0,
                          k_out: Optional[torch.Tensor] = None,
                          v_out: Optional[torch.Tensor] = None, out_rows: Optional[int] = None,
                          err: Optional[torch.Tensor] = None, prepare: bool = False):
    """kv_cache_gather with the blocks found from range descriptors."""
    dev = _device_of(k_cache, "k_cache")
    L, B, T, H, D = _cache_dims(k_cache, v_cache, dev)
    R = gather_start.numel()
    _ranges_check(range_start, range_len, num_ranges, dev, R)
    if gather_end.numel() != R:
        raise ValueError("gather_start and gather_end differ in length")
    k_out, v_out, rows = _gather_outputs(k_cache, gather_start, gather_end, k_out, v_out,
                                         out_rows, H, D, dev)
    args = (_ptr(k_cache), _ptr(v_cache), int(layer), L, B, T, H, D, _ptr(range_start),
            _ptr(range_len), _ptr(num_ranges), range_start.shape[1], _ptr(gather_start),
            _ptr(gather_end), R, _ptr(k_out), _ptr(v_out), rows, _err_ptr(err, dev))
    return _run("kv_cache_gather_range", args, dev,
                (k_cache, v_cache, range_start, range_len, num_ranges, gather_start, gather_end,
                 k_out, v_out, err), (k_out, v_out), prepare)


def kv_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_blocks: torch.Tensor,
                   dst_blocks: torch.Tensor, err: Optional[torch.Tensor] = None,
                   bulk: bool = False, prepare: bool = False):
    """Copy whole blocks src -> dst (every layer, K and V) in place.

    ``bulk=True`` calls kv_copy_blocks_bulk (bulk-copy engine) instead.
    Returns None (or the ``Prepared`` call)."""
    dev = _device_of(k_cache, "k_cache")
    L, B, T, H, D = _cache_dims(k_cache, v_cache, dev)
    _need(src_blocks, "src_blocks", torch.int32, dev)
    _need(dst_blocks, "dst_blocks", torch.int32, dev)
    if src_blocks.numel() != dst_blocks.numel():
        raise ValueError("src_blocks and dst_blocks differ in length")
    args = (_ptr(k_cache), _ptr(v_cache), L, B, T, H, D, _ptr(src_blocks), _ptr(dst_blocks),
            src_blocks.numel(), _err_ptr(err, dev))
    return _run("kv_copy_blocks_bulk" if bulk else "kv_copy_blocks", args, dev,
                (k_cache, v_cache, src_blocks, dst_blocks, err), None, prepare)
