"""Seeded synthetic workloads for the paged KV-cache hot path.

This module only builds *structure*: which requests exist, which positions each
token has, which physical blocks a request owns (as a block-table row and as
contiguous ranges), and which positions a read-path gather asks for.  It holds
none of the hot path's arithmetic (no slot ids, no cache offsets, no copies):
both the CPU oracle and the CUDA library are fed from here and nothing here
depends on either of them.

The shapes follow the workloads the pages describe:

* a block table is an int32 ``[rows, max_blocks_per_req]`` array whose row is a
  request and whose column j is the physical block of logical block j
  ("Blocktabelle", Verantwortung); its stride is rounded up to a multiple of
  ``128 // block_size`` (same page, Grenzen und Fehler, TRTLLM alignment);
* block 0 is the null block and is never handed to a request
  ("vLLM Block Table Management", Symbol Map and Deep Dive section 1);
* a request's blocks may also be described as contiguous ranges
  ``(range_start, range_len)`` in logical order, at most 256 per request
  ("Range-addressed KV cache blocks ...", The Fork Implementation);
* CUDA-graph padding rows own no tokens and an all-null table row
  ("Blocktabelle", Entwurfsmotivation, CUDA-Graph-Padding);
* sliding-window recycling replaces every block that lies wholly before
  ``num_computed - window + 1`` with the null block
  ("vLLM Block Table Management", Deep Dive section 6).

The public benchmark the pages use for their serving runs (ShareGPT) is not
available; these generators stand in for its 16K/128K shapes with uniform
context-length draws.  Every function takes an explicit seed.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

NULL_BLOCK = 0
RANGE_CAP = 256  # per-request descriptor cap of the range backend


def table_stride_for(max_blocks: int, block_size: int) -> int:
    """Round a per-request block count up to the TRTLLM-friendly multiple."""
    mult = max(1, 128 // block_size)
    return max(mult, -(-max_blocks // mult) * mult)


def range_stride_for(max_runs: int) -> int:
    """Descriptor capacity per request for a layout whose requests hold at
    most ``max_runs`` ranges: that cap rounded up to a multiple of 4 (16-byte
    rows, so a row head loads as one vector), never above the backend's cap."""
    return min(RANGE_CAP, max(4, -(-max_runs // 4) * 4))


def blocks_for(num_tokens: int, block_size: int) -> int:
    """Number of blocks a request holding ``num_tokens`` tokens owns."""
    return -(-num_tokens // block_size)


def swa_null_prefix(num_computed: int, window: int, block_size: int) -> int:
    """Leading blocks that sliding-window recycling has replaced by the null block.

    Tokens before ``num_computed - window + 1`` are freed; a block is freed only
    when all of its tokens are ("vLLM Block Table Management", Deep Dive 6).
    """
    first_kept_token = num_computed - window + 1
    if first_kept_token <= 0:
        return 0
    return first_kept_token // block_size


@dataclass
class Layout:
    """One physical placement of every request's blocks."""

    table: np.ndarray                  # int32 [rows, table_stride]
    range_start: Optional[np.ndarray]  # int32 [rows, range_stride] or None
    range_len: Optional[np.ndarray]    # int32 [rows, range_stride] or None
    num_ranges: Optional[np.ndarray]   # int32 [rows] or None

    @property
    def table_stride(self) -> int:
        return int(self.table.shape[1])

    @property
    def range_stride(self) -> int:
        return int(self.range_start.shape[1]) if self.range_start is not None else 0


@dataclass
class Workload:
    """Inputs of one pass of the hot path for one KV-cache group."""

    name: str
    seed: int
    block_size: int
    num_blocks: int          # physical blocks in the pool, block 0 included
    num_layers: int
    num_kv_heads: int
    head_dim: int
    num_reqs: int            # rows handed to the kernels (padding rows included)
    num_real_reqs: int
    qsl: np.ndarray          # int32 [num_reqs + 1]
    positions: np.ndarray    # int64 [num_tokens]
    num_tokens: int
    max_num_tokens: int
    layouts: Dict[str, Layout] = field(default_factory=dict)
    gather_start: Optional[np.ndarray] = None  # int32 [num_reqs]
    gather_end: Optional[np.ndarray] = None    # int32 [num_reqs]
    blocks_per_req: Optional[np.ndarray] = None  # int64 [num_reqs]
    notes: str = ""

    @property
    def row_elems(self) -> int:
        return self.num_kv_heads * self.head_dim

    @property
    def row_bytes(self) -> int:
        return self.row_elems * 2


@dataclass
class HybridGroup:
    """One KV-cache group of the hybrid workload, in manager-block units."""

    name: str
    mgr_block_size: int
    kernel_block_size: int
    mgr_num_blocks: int      # manager pool size, null block 0 included
    mgr_table: np.ndarray    # int32 [num_reqs, mgr_stride]
    gather_start: np.ndarray  # int32 [num_reqs]
    gather_end: np.ndarray    # int32 [num_reqs]

    @property
    def kernel_num_blocks(self) -> int:
        return self.mgr_num_blocks * (self.mgr_block_size // self.kernel_block_size)


@dataclass
class HybridWorkload:
    name: str
    seed: int
    num_reqs: int            # padded rows
    num_real_reqs: int
    ctx: np.ndarray          # int64 [num_real_reqs]
    qsl: np.ndarray
    positions: np.ndarray
    num_tokens: int
    max_num_tokens: int
    num_kv_heads: int
    head_dim: int
    window: int
    groups: Dict[str, HybridGroup] = field(default_factory=dict)
    num_layers: int = 1


# --------------------------------------------------------------------------
# placement helpers (structure only)
# --------------------------------------------------------------------------

def _split_into_runs(rng: np.random.Generator, n: int, max_runs: int) -> np.ndarray:
    """Split ``n`` blocks into ``U{1..min(max_runs, n)}`` runs of random length."""
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    k = int(rng.integers(1, min(max_runs, n) + 1))
    if k == 1:
        return np.array([n], dtype=np.int64)
    cuts = np.sort(rng.choice(n - 1, size=k - 1, replace=False) + 1)
    return np.diff(np.concatenate([[0], cuts, [n]])).astype(np.int64)


def _place_runs(rng: np.random.Generator, lengths: np.ndarray, lo: int, hi: int,
                packed: bool) -> np.ndarray:
    """Place runs of the given lengths at random disjoint offsets of ``[lo, hi)``.

    The runs are laid out in a random order with random gaps (or no gaps when
    ``packed``).  Returns each run's first block, indexed like ``lengths``.
    """
    m = len(lengths)
    total = int(lengths.sum())
    free = (hi - lo) - total
    if free < 0:
        raise ValueError(f"pool [{lo},{hi}) too small for {total} blocks")
    order = rng.permutation(m)
    if packed or m == 0:
        gaps = np.zeros(m, dtype=np.int64)
    else:
        cuts = np.sort(rng.integers(0, free + 1, size=m))
        gaps = np.diff(np.concatenate([[0], cuts])).astype(np.int64)
    ordered_len = lengths[order]
    advance = gaps + np.concatenate([[0], ordered_len[:-1]]).astype(np.int64)
    starts_ordered = lo + np.cumsum(advance)
    starts = np.empty(m, dtype=np.int64)
    starts[order] = starts_ordered
    return starts


def _runs_of(blocks: Sequence[int]) -> List[Tuple[int, int]]:
    """Maximal runs of consecutive block ids in a block list."""
    runs: List[Tuple[int, int]] = []
    for b in blocks:
        b = int(b)
        if runs and runs[-1][0] + runs[-1][1] == b:
            runs[-1] = (runs[-1][0], runs[-1][1] + 1)
        else:
            runs.append((b, 1))
    return runs


def _layout_from_block_lists(block_lists: List[np.ndarray], rows: int, table_stride: int,
                             run_lists: Optional[List[List[Tuple[int, int]]]],
                             range_stride: int) -> Layout:
    table = np.zeros((rows, table_stride), dtype=np.int32)
    for r, bl in enumerate(block_lists):
        table[r, :len(bl)] = bl
    if run_lists is None:
        return Layout(table, None, None, None)
    rs = np.zeros((rows, range_stride), dtype=np.int32)
    rl = np.zeros((rows, range_stride), dtype=np.int32)
    nr = np.zeros(rows, dtype=np.int32)
    for r, runs in enumerate(run_lists):
        if len(runs) > range_stride:
            raise ValueError("more runs than the descriptor stride")
        nr[r] = len(runs)
        for i, (s, ln) in enumerate(runs):
            rs[r, i] = s
            rl[r, i] = ln
    return Layout(table, rs, rl, nr)


def _runs_layout(rng: np.random.Generator, nblocks: np.ndarray, max_runs: int, pool: int,
                 rows: int, table_stride: int, range_stride: int, packed: bool) -> Layout:
    """Layout "G": each request's blocks as a few contiguous runs in the pool."""
    per_req = [_split_into_runs(rng, int(n), max_runs) for n in nblocks]
    lengths = np.concatenate(per_req) if per_req else np.zeros(0, dtype=np.int64)
    starts = _place_runs(rng, lengths, 1, pool, packed)
    block_lists, run_lists, k = [], [], 0
    for runs in per_req:
        rl = []
        bl = []
        for ln in runs:
            s = int(starts[k])
            k += 1
            rl.append((s, int(ln)))
            bl.append(np.arange(s, s + ln, dtype=np.int64))
        run_lists.append(rl)
        block_lists.append(np.concatenate(bl) if bl else np.zeros(0, dtype=np.int64))
    return _layout_from_block_lists(block_lists, rows, table_stride, run_lists, range_stride)


def _perm_layout(rng: np.random.Generator, nblocks: np.ndarray, pool: int, rows: int,
                 table_stride: int, range_stride: Optional[int]) -> Layout:
    """Layout "P": a random permutation of the pool dealt to requests in order.

    When ``range_stride`` is given, each request's block list is also described
    by its maximal runs of consecutive ids (only possible when they fit).
    """
    perm = rng.permutation(np.arange(1, pool, dtype=np.int64))
    need = int(nblocks.sum())
    if need > len(perm):
        raise ValueError("pool too small")
    block_lists, k = [], 0
    for n in nblocks:
        block_lists.append(perm[k:k + int(n)])
        k += int(n)
    run_lists = None
    if range_stride is not None:
        run_lists = [_runs_of(bl) for bl in block_lists]
    return _layout_from_block_lists(block_lists, rows, table_stride, run_lists, range_stride or 0)


def _qsl_from_lengths(lengths: Sequence[int], rows: int) -> np.ndarray:
    q = np.zeros(rows + 1, dtype=np.int64)
    q[1:len(lengths) + 1] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    q[len(lengths) + 1:] = q[len(lengths)]
    return q.astype(np.int32)


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    """4 prompts of U{7..50} tokens, block size 16, 64-block pool, 8x64 heads."""
    rng = np.random.default_rng(seed)
    T, B, R = 16, 64, 4
    lens = rng.integers(7, 51, size=R)
    nblocks = np.array([blocks_for(int(n), T) for n in lens], dtype=np.int64)
    stride = table_stride_for(int(nblocks.max()), T)
    lay_p = _perm_layout(rng, nblocks, B, R, stride, RANGE_CAP)
    lay_g = _runs_layout(rng, nblocks, 3, B, R, stride, range_stride_for(3), packed=False)
    positions = np.concatenate([np.arange(n, dtype=np.int64) for n in lens])
    N = int(lens.sum())
    n_max = -(-(N + 1) // 256) * 256
    g0 = np.zeros(R, dtype=np.int32)
    g1 = lens.astype(np.int32)
    return Workload("tiny", seed, T, B, 1, 8, 64, R, R, _qsl_from_lengths(lens, R), positions,
                    N, n_max, {"P": lay_p, "G": lay_g}, g0, g1, nblocks,
                    notes="prompts from position 0; max_num_tokens rounded up to 256")


def decode(seed: int = 1, num_blocks: int = 40960, ctx_max: int = 4096) -> Workload:
    """256 decode requests, context U{512..ctx_max}, one new token each, num_blocks pool."""
    rng = np.random.default_rng(seed)
    T, B, R = 16, num_blocks, 256
    ctx = rng.integers(512, ctx_max + 1, size=R)
    nblocks = np.array([blocks_for(int(c), T) for c in ctx], dtype=np.int64)
    assert int(nblocks.sum()) < B - 1
    stride = table_stride_for(blocks_for(ctx_max, T), T)
    lay_g = _runs_layout(rng, nblocks, 4, B, R, stride, range_stride_for(4), packed=False)
    positions = (ctx - 1).astype(np.int64)
    g0 = np.zeros(R, dtype=np.int32)
    g1 = ctx.astype(np.int32)
    return Workload("decode", seed, T, B, 1, 8, 128, R, R, _qsl_from_lengths([1] * R, R),
                    positions, R, R, {"G": lay_g}, g0, g1, nblocks,
                    notes="new token at position ctx-1; 1-4 runs per request")


def mixed(seed: int = 2, num_blocks: int = 49152, decode_ctx_max: int = 4096) -> Workload:
    """240 decode tokens plus 16 prefill chunks of 8192 tokens total, 32 layers."""
    rng = np.random.default_rng(seed)
    T, L = 16, 32
    n_dec, n_pre, pre_total = 240, 16, 8192
    dec_ctx = rng.integers(512, decode_ctx_max + 1, size=n_dec)
    cuts = np.sort(rng.choice(pre_total - 1, size=n_pre - 1, replace=False) + 1)
    pre_len = np.diff(np.concatenate([[0], cuts, [pre_total]])).astype(np.int64)
    pre_prior = rng.integers(0, 8193, size=n_pre)
    lens = np.concatenate([np.ones(n_dec, dtype=np.int64), pre_len])
    owned = np.concatenate([dec_ctx, pre_prior + pre_len]).astype(np.int64)
    nblocks = np.array([blocks_for(int(c), T) for c in owned], dtype=np.int64)
    assert int(nblocks.sum()) < num_blocks - 1
    R = n_dec + n_pre
    stride = table_stride_for(int(nblocks.max()), T)
    lay_g = _runs_layout(rng, nblocks, 8, num_blocks, R, stride, range_stride_for(8),
                         packed=False)
    positions = np.concatenate(
        [(dec_ctx - 1).astype(np.int64)]
        + [np.arange(int(c), int(c) + int(n), dtype=np.int64) for c, n in zip(pre_prior, pre_len)])
    N = int(lens.sum())
    g0 = np.zeros(R, dtype=np.int32)
    g1 = owned.astype(np.int32)
    return Workload("mixed", seed, T, num_blocks, L, 8, 128, R, R, _qsl_from_lengths(lens, R),
                    positions, N, N, {"G": lay_g}, g0, g1, nblocks,
                    notes="decode requests first, then prefill chunks with prior context U{0..8192}")


def long_context(seed: int = 3, num_reqs: int = 8, tokens_per_req: int = 131072) -> Workload:
    """8 requests x 131072 tokens, block size 16, permuted vs 1-16 packed runs."""
    rng = np.random.default_rng(seed)
    T = 16
    per = blocks_for(tokens_per_req, T)
    B = num_reqs * per + 1
    nblocks = np.full(num_reqs, per, dtype=np.int64)
    stride = table_stride_for(per, T)
    lay_p = _perm_layout(rng, nblocks, B, num_reqs, stride, None)
    lay_g = _runs_layout(rng, nblocks, 16, B, num_reqs, stride, range_stride_for(16), packed=True)
    positions = np.tile(np.arange(tokens_per_req, dtype=np.int64), num_reqs)
    N = num_reqs * tokens_per_req
    g0 = np.zeros(num_reqs, dtype=np.int32)
    g1 = np.full(num_reqs, tokens_per_req, dtype=np.int32)
    return Workload("long", seed, T, B, 1, 8, 128, num_reqs, num_reqs,
                    _qsl_from_lengths([tokens_per_req] * num_reqs, num_reqs), positions, N, N,
                    {"P": lay_p, "G": lay_g}, g0, g1, nblocks,
                    notes="whole-context gather; P = permutation, G = packed runs")


def hybrid(seed: int = 4, num_real: int = 512, num_padded: int = 640, ctx_max: int = 32768,
           full_pool: int = 270336, window: int = 4096) -> HybridWorkload:
    """Full-attention + sliding-window groups, manager block 32 over kernel block 16.

    512 decode requests with context U{1..ctx_max} are padded to 640 rows for
    CUDA-graph capture: padding rows own no tokens and an all-null table row,
    and the slot-mapping tail is padded.
    """
    rng = np.random.default_rng(seed)
    mbs, kbs = 32, 16
    ctx = rng.integers(1, ctx_max + 1, size=num_real).astype(np.int64)
    mgr_stride = table_stride_for(blocks_for(ctx_max, mbs), mbs)
    # full-attention group: every block kept, pool permuted
    full_need = np.array([blocks_for(int(c), mbs) for c in ctx], dtype=np.int64)
    full_pool_blocks = full_pool + 1
    assert int(full_need.sum()) <= full_pool
    full_lay = _perm_layout(rng, np.concatenate([full_need, np.zeros(num_padded - num_real, np.int64)]),
                            full_pool_blocks, num_padded, mgr_stride, None)
    # sliding-window group: leading recycled blocks are null, the rest permuted
    keep_max = blocks_for(window, mbs) + 1
    swa_pool_blocks = num_real * keep_max + 1
    swa_null = np.array([swa_null_prefix(int(c) - 1, window, mbs) for c in ctx], dtype=np.int64)
    swa_keep = full_need - swa_null
    assert int(swa_keep.max()) <= keep_max
    perm = rng.permutation(np.arange(1, swa_pool_blocks, dtype=np.int64))
    swa_table = np.zeros((num_padded, mgr_stride), dtype=np.int32)
    k = 0
    for r in range(num_real):
        n0, n1 = int(swa_null[r]), int(full_need[r])
        swa_table[r, n0:n1] = perm[k:k + (n1 - n0)]
        k += n1 - n0
    zeros_pad = np.zeros(num_padded - num_real, dtype=np.int64)
    full_g0 = np.zeros(num_padded, dtype=np.int32)
    full_g1 = np.concatenate([ctx, zeros_pad]).astype(np.int32)
    swa_g0 = np.concatenate([np.maximum(ctx - window, 0), zeros_pad]).astype(np.int32)
    swa_g1 = full_g1.copy()
    groups = {
        "full": HybridGroup("full", mbs, kbs, full_pool_blocks, full_lay.table, full_g0, full_g1),
        "swa": HybridGroup("swa", mbs, kbs, swa_pool_blocks, swa_table, swa_g0, swa_g1),
    }
    qsl = _qsl_from_lengths([1] * num_real, num_padded)
    positions = (ctx - 1).astype(np.int64)
    return HybridWorkload("hybrid", seed, num_padded, num_real, ctx, qsl, positions, num_real,
                          num_padded, 8, 128, window, groups)


CONFIGS = {
    "tiny": tiny,
    "decode": decode,
    "mixed": mixed,
    "long": long_context,
    "hybrid": hybrid,
}


# --------------------------------------------------------------------------
# K/V values: bf16 draws of N(0, 1)
# --------------------------------------------------------------------------

def bf16_normal(shape, seed: int, device="cpu"):
    """Seeded N(0,1) bf16 tensor (torch generator on the target device)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.bfloat16)
