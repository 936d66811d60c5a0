"""Torch-facing wrappers of the C ABI (argument marshalling only).

Each function has the name of the C entry point it calls, takes CUDA tensors,
checks their dtype, device and contiguity, passes raw pointers and the
current CUDA stream, and raises ``KVError`` on a negative status.  All work
runs in the CUDA kernels; nothing here computes on the host.

``err`` is an optional int32 CUDA tensor of one element: data errors the
kernels detect are OR-ed into it (see ``ERR_BITS``).
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from ._lib import check, load

__all__ = [
    "kv_slot_mapping_paged",
    "kv_slot_mapping_paged_cp",
    "kv_slot_mapping_range",
    "kv_cache_write",
    "kv_cache_gather",
    "kv_expand_kernel_blocks",
    "kv_table_from_ranges",
    "kv_cache_gather_range",
    "kv_copy_blocks",
    "new_error_word",
]


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None or t.numel() == 0:
        return None
    return t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device: torch.device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (the kernels take device pointers), "
                         f"got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must live on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _err_ptr(err: Optional[torch.Tensor], device: torch.device) -> Optional[int]:
    if err is None:
        return None
    _need(err, "err", torch.int32, device)
    if err.numel() < 1:
        raise ValueError("err needs one element")
    return err.data_ptr()


def new_error_word(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def kv_slot_mapping_paged(query_start_loc: torch.Tensor, positions: torch.Tensor,
                          block_table: torch.Tensor, block_size: int, num_blocks: int,
                          max_num_tokens: Optional[int] = None,
                          slot_mapping: Optional[torch.Tensor] = None,
                          num_tokens: Optional[int] = None,
                          err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """slot_mapping[t] through ``block_table`` [num_reqs, stride] (int32)."""
    dev = positions.device
    _need(query_start_loc, "query_start_loc", torch.int32, dev)
    _need(positions, "positions", torch.int64, dev)
    _need(block_table, "block_table", torch.int32, dev)
    if block_table.dim() != 2:
        raise ValueError("block_table must be [num_reqs, table_stride]")
    num_reqs = query_start_loc.numel() - 1
    if block_table.shape[0] < num_reqs:
        raise ValueError("block_table has fewer rows than requests")
    n = positions.numel() if num_tokens is None else int(num_tokens)
    if n > positions.numel():
        raise ValueError("num_tokens exceeds positions")
    n_max = n if max_num_tokens is None else int(max_num_tokens)
    if slot_mapping is None:
        slot_mapping = torch.empty(n_max, dtype=torch.int64, device=dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    if slot_mapping.numel() < n_max:
        raise ValueError("slot_mapping is shorter than max_num_tokens")
    lib = load()
    check("kv_slot_mapping_paged", lib.kv_slot_mapping_paged(
        _ptr(query_start_loc), _ptr(positions), _ptr(block_table), block_table.shape[1],
        max(num_reqs, 0), n, n_max, int(block_size), int(num_blocks), _ptr(slot_mapping),
        _err_ptr(err, dev), _stream(dev)))
    return slot_mapping


def kv_slot_mapping_paged_cp(query_start_loc: torch.Tensor, positions: torch.Tensor,
                             block_table: torch.Tensor, block_size: int, num_blocks: int,
                             cp_world_size: int, cp_rank: int, cp_interleave: int = 1,
                             max_num_tokens: Optional[int] = None,
                             slot_mapping: Optional[torch.Tensor] = None,
                             num_tokens: Optional[int] = None,
                             err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """kv_slot_mapping_paged for one rank of context parallelism (see the header)."""
    dev = positions.device
    _need(query_start_loc, "query_start_loc", torch.int32, dev)
    _need(positions, "positions", torch.int64, dev)
    _need(block_table, "block_table", torch.int32, dev)
    if block_table.dim() != 2:
        raise ValueError("block_table must be [num_reqs, table_stride]")
    num_reqs = query_start_loc.numel() - 1
    if block_table.shape[0] < num_reqs:
        raise ValueError("block_table has fewer rows than requests")
    n = positions.numel() if num_tokens is None else int(num_tokens)
    if n > positions.numel():
        raise ValueError("num_tokens exceeds positions")
    n_max = n if max_num_tokens is None else int(max_num_tokens)
    if slot_mapping is None:
        slot_mapping = torch.empty(n_max, dtype=torch.int64, device=dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    if slot_mapping.numel() < n_max:
        raise ValueError("slot_mapping is shorter than max_num_tokens")
    lib = load()
    check("kv_slot_mapping_paged_cp", lib.kv_slot_mapping_paged_cp(
        _ptr(query_start_loc), _ptr(positions), _ptr(block_table), block_table.shape[1],
        max(num_reqs, 0), n, n_max, int(block_size), int(num_blocks), int(cp_world_size),
        int(cp_rank), int(cp_interleave), _ptr(slot_mapping), _err_ptr(err, dev), _stream(dev)))
    return slot_mapping


def kv_slot_mapping_range(query_start_loc: torch.Tensor, positions: torch.Tensor,
                          range_start: torch.Tensor, range_len: torch.Tensor,
                          num_ranges: torch.Tensor, block_size: int, num_blocks: int,
                          max_num_tokens: Optional[int] = None,
                          slot_mapping: Optional[torch.Tensor] = None,
                          num_tokens: Optional[int] = None,
                          err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """slot_mapping[t] through per-request range descriptors [num_reqs, range_stride]."""
    dev = positions.device
    _need(query_start_loc, "query_start_loc", torch.int32, dev)
    _need(positions, "positions", torch.int64, dev)
    for name, t in (("range_start", range_start), ("range_len", range_len),
                    ("num_ranges", num_ranges)):
        _need(t, name, torch.int32, dev)
    if range_start.dim() != 2 or range_len.shape != range_start.shape:
        raise ValueError("range_start/range_len must both be [num_reqs, range_stride]")
    num_reqs = query_start_loc.numel() - 1
    if range_start.shape[0] < num_reqs or num_ranges.numel() < num_reqs:
        raise ValueError("descriptor arrays have fewer rows than requests")
    n = positions.numel() if num_tokens is None else int(num_tokens)
    if n > positions.numel():
        raise ValueError("num_tokens exceeds positions")
    n_max = n if max_num_tokens is None else int(max_num_tokens)
    if slot_mapping is None:
        slot_mapping = torch.empty(n_max, dtype=torch.int64, device=dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    if slot_mapping.numel() < n_max:
        raise ValueError("slot_mapping is shorter than max_num_tokens")
    lib = load()
    check("kv_slot_mapping_range", lib.kv_slot_mapping_range(
        _ptr(query_start_loc), _ptr(positions), _ptr(range_start), _ptr(range_len),
        _ptr(num_ranges), range_start.shape[1], max(num_reqs, 0), n, n_max, int(block_size),
        int(num_blocks), _ptr(slot_mapping), _err_ptr(err, dev), _stream(dev)))
    return slot_mapping


def _cache_dims(k_cache: torch.Tensor) -> Tuple[int, int, int, int, int]:
    if k_cache.dim() != 5:
        raise ValueError("caches must be [num_layers, num_blocks, block_size, kv_heads, head_dim]")
    return tuple(int(x) for x in k_cache.shape)


def kv_cache_write(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                   num_tokens: Optional[int] = None,
                   err: Optional[torch.Tensor] = None) -> None:
    """Scatter key/value [L, N, H, D] (bf16) into the [L, B, T, H, D] caches."""
    dev = key.device
    for name, t in (("key", key), ("value", value), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, torch.bfloat16, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    L, B, T, H, D = _cache_dims(k_cache)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if key.dim() != 4 or key.shape[0] != L or key.shape[2:] != (H, D) or value.shape != key.shape:
        raise ValueError("key/value must be [num_layers, num_tokens, kv_heads, head_dim]")
    n = key.shape[1] if num_tokens is None else int(num_tokens)
    if n > key.shape[1] or slot_mapping.numel() < n:
        raise ValueError("num_tokens exceeds key rows or slot_mapping")
    if n != key.shape[1] and L > 1:
        raise ValueError("num_tokens must equal key.shape[1] for multi-layer writes")
    lib = load()
    check("kv_cache_write", lib.kv_cache_write(
        _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), n, L, B, T, H, D,
        _err_ptr(err, dev), _stream(dev)))


def kv_cache_gather(k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                    gather_start: torch.Tensor, gather_end: torch.Tensor, layer: int = 0,
                    k_out: Optional[torch.Tensor] = None, v_out: Optional[torch.Tensor] = None,
                    out_rows: Optional[int] = None,
                    err: Optional[torch.Tensor] = None, bulk: bool = False
                    ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Gather positions [start_r, end_r) of every request into packed [rows, H, D] buffers.

    ``out_rows`` (or the given outputs' row count) must be at least the total
    span length; when it is None and no outputs are given, the total is read
    back from the device spans (a synchronising convenience for tests).
    ``bulk=True`` calls kv_cache_gather_bulk (bulk-copy engine) instead.
    """
    dev = k_cache.device
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(gather_start, "gather_start", torch.int32, dev)
    _need(gather_end, "gather_end", torch.int32, dev)
    L, B, T, H, D = _cache_dims(k_cache)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if block_table.dim() != 2:
        raise ValueError("block_table must be [num_reqs, table_stride]")
    R = gather_start.numel()
    if gather_end.numel() != R or block_table.shape[0] < R:
        raise ValueError("gather spans and block_table rows disagree")
    if k_out is None:
        if out_rows is None:
            out_rows = int((gather_end.long() - gather_start.long()).clamp_min(0).sum().item())
        k_out = torch.empty((out_rows, H, D), dtype=torch.bfloat16, device=dev)
        v_out = torch.empty((out_rows, H, D), dtype=torch.bfloat16, device=dev)
    _need(k_out, "k_out", torch.bfloat16, dev)
    _need(v_out, "v_out", torch.bfloat16, dev)
    rows = k_out.shape[0] if out_rows is None else int(out_rows)
    for t in (k_out, v_out):
        if t.dim() < 1 or t.shape[0] < rows or t.numel() < rows * H * D:
            raise ValueError("outputs are smaller than out_rows rows of kv_heads x head_dim")
    lib = load()
    name = "kv_cache_gather_bulk" if bulk else "kv_cache_gather"
    check(name, getattr(lib, name)(
        _ptr(k_cache), _ptr(v_cache), int(layer), L, B, T, H, D, _ptr(block_table),
        block_table.shape[1], _ptr(gather_start), _ptr(gather_end), R, _ptr(k_out), _ptr(v_out),
        rows, _err_ptr(err, dev), _stream(dev)))
    return k_out, v_out


def kv_expand_kernel_blocks(mgr_table: torch.Tensor, mgr_block_size: int,
                            kernel_block_size: int,
                            kernel_table: Optional[torch.Tensor] = None,
                            err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Expand an int32 [R, Ms] manager table into an int32 [R, Ks] kernel table."""
    dev = mgr_table.device
    _need(mgr_table, "mgr_table", torch.int32, dev)
    if mgr_table.dim() != 2:
        raise ValueError("mgr_table must be [num_reqs, mgr_stride]")
    R, Ms = mgr_table.shape
    if kernel_table is None:
        k = mgr_block_size // kernel_block_size if kernel_block_size > 0 else 1
        kernel_table = torch.empty((R, Ms * max(k, 1)), dtype=torch.int32, device=dev)
    _need(kernel_table, "kernel_table", torch.int32, dev)
    if kernel_table.dim() != 2 or kernel_table.shape[0] != R:
        raise ValueError("kernel_table must be [num_reqs, kernel_stride]")
    lib = load()
    check("kv_expand_kernel_blocks", lib.kv_expand_kernel_blocks(
        _ptr(mgr_table), R, Ms, int(mgr_block_size), int(kernel_block_size), _ptr(kernel_table),
        kernel_table.shape[1], _err_ptr(err, dev), _stream(dev)))
    return kernel_table


def kv_table_from_ranges(range_start: torch.Tensor, range_len: torch.Tensor,
                         num_ranges: torch.Tensor, table_stride: Optional[int] = None,
                         block_table: Optional[torch.Tensor] = None,
                         err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Block table int32 [num_reqs, table_stride] expanded from range descriptors."""
    dev = range_start.device
    for name, t in (("range_start", range_start), ("range_len", range_len),
                    ("num_ranges", num_ranges)):
        _need(t, name, torch.int32, dev)
    if range_start.dim() != 2 or range_len.shape != range_start.shape:
        raise ValueError("range_start/range_len must both be [num_reqs, range_stride]")
    R = range_start.shape[0]
    if num_ranges.numel() < R:
        raise ValueError("num_ranges has fewer entries than descriptor rows")
    if block_table is None:
        if table_stride is None:
            raise ValueError("give table_stride or block_table")
        block_table = torch.empty((R, int(table_stride)), dtype=torch.int32, device=dev)
    _need(block_table, "block_table", torch.int32, dev)
    if block_table.dim() != 2 or block_table.shape[0] != R:
        raise ValueError("block_table must be [num_reqs, table_stride]")
    lib = load()
    check("kv_table_from_ranges", lib.kv_table_from_ranges(
        _ptr(range_start), _ptr(range_len), _ptr(num_ranges), range_start.shape[1], R,
        _ptr(block_table), block_table.shape[1], _err_ptr(err, dev), _stream(dev)))
    return block_table


def kv_cache_gather_range(k_cache: torch.Tensor, v_cache: torch.Tensor,
                          range_start: torch.Tensor, range_len: torch.Tensor,
                          num_ranges: torch.Tensor, gather_start: torch.Tensor,
                          gather_end: torch.Tensor, layer: int = 0,
                          k_out: Optional[torch.Tensor] = None,
                          v_out: Optional[torch.Tensor] = None, out_rows: Optional[int] = None,
                          err: Optional[torch.Tensor] = None
                          ) -> Tuple[torch.Tensor, torch.Tensor]:
    """kv_cache_gather with the blocks found from range descriptors."""
    dev = k_cache.device
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    for name, t in (("range_start", range_start), ("range_len", range_len),
                    ("num_ranges", num_ranges), ("gather_start", gather_start),
                    ("gather_end", gather_end)):
        _need(t, name, torch.int32, dev)
    L, B, T, H, D = _cache_dims(k_cache)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if range_start.dim() != 2 or range_len.shape != range_start.shape:
        raise ValueError("range_start/range_len must both be [num_reqs, range_stride]")
    R = gather_start.numel()
    if gather_end.numel() != R or range_start.shape[0] < R or num_ranges.numel() < R:
        raise ValueError("gather spans and descriptor rows disagree")
    if k_out is None:
        if out_rows is None:
            out_rows = int((gather_end.long() - gather_start.long()).clamp_min(0).sum().item())
        k_out = torch.empty((out_rows, H, D), dtype=torch.bfloat16, device=dev)
        v_out = torch.empty((out_rows, H, D), dtype=torch.bfloat16, device=dev)
    _need(k_out, "k_out", torch.bfloat16, dev)
    _need(v_out, "v_out", torch.bfloat16, dev)
    rows = k_out.shape[0] if out_rows is None else int(out_rows)
    for t in (k_out, v_out):
        if t.dim() < 1 or t.shape[0] < rows or t.numel() < rows * H * D:
            raise ValueError("outputs are smaller than out_rows rows of kv_heads x head_dim")
    lib = load()
    check("kv_cache_gather_range", lib.kv_cache_gather_range(
        _ptr(k_cache), _ptr(v_cache), int(layer), L, B, T, H, D, _ptr(range_start),
        _ptr(range_len), _ptr(num_ranges), range_start.shape[1], _ptr(gather_start),
        _ptr(gather_end), R, _ptr(k_out), _ptr(v_out), rows, _err_ptr(err, dev), _stream(dev)))
    return k_out, v_out


def kv_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_blocks: torch.Tensor,
                   dst_blocks: torch.Tensor, err: Optional[torch.Tensor] = None) -> None:
    """Copy whole blocks src -> dst (every layer, K and V) in place."""
    dev = k_cache.device
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(src_blocks, "src_blocks", torch.int32, dev)
    _need(dst_blocks, "dst_blocks", torch.int32, dev)
    L, B, T, H, D = _cache_dims(k_cache)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if src_blocks.numel() != dst_blocks.numel():
        raise ValueError("src_blocks and dst_blocks differ in length")
    lib = load()
    check("kv_copy_blocks", lib.kv_copy_blocks(
        _ptr(k_cache), _ptr(v_cache), L, B, T, H, D, _ptr(src_blocks), _ptr(dst_blocks),
        src_blocks.numel(), _err_ptr(err, dev), _stream(dev)))
