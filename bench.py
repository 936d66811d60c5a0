#!/usr/bin/env python3
"""Benchmark of the paged KV-cache hot path on GB300.

The headline is the metric's first half on the decode step: 256 requests with
one new token each, contexts U{512..4096}, block size 16, a 40960-block pool,
8 KV heads x 128 bf16, each request's blocks in 1-4 contiguous ranges.  One
step is

  1. kv_slot_mapping_paged   (block-table strategy)
  2. kv_slot_mapping_range   (range strategy, same layout, side by side)
  3. kv_cache_write          (the new tokens' K/V rows to their slots)

captured once in a CUDA graph and replayed, as a serving loop runs its decode
steps.  The range map reads nothing the other two write (it fills its own slot
buffer), so the graph runs it on a second branch beside the paged map -> write
chain.  `value` is new tokens per second over the whole job.  The L2 is
flushed (a 256 MiB write, then a 256 MiB read) between timed steps, outside
the timed events.  Beside it, in the same JSON line:

  paged_vs_range   the two strategies' slot map + write, as separate launches
                   and as the fused calls, each replayed from a CUDA graph;
  gather_GBps      the metric's second half: the whole-context gather of the
                   long-context workload (8 x 131072 tokens) through the
                   permuted table P, with its own roofline (table G and the
                   range-addressed and bulk-copy gathers under "gather");
  decode_step_with_gather  the decode step followed by the gather of every
                   request's whole context (597k rows);
  e2e              the headline step through the public API from host memory.

Rank 0 prints one JSON line.  `--impl reference` times the CPU oracle on the
same step instead.  The mixed, long-context and hybrid workloads are timed per
kernel after the headline and reported under "configs".
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "KV write+slot-map tokens/s and gather GB/s (frac of ~8 TB/s), paged vs range"
FLUSH_BYTES = 512 << 20  # two halves of 256 MiB, each twice the 129 MB L2
DECODE_DESC = ("decode step: 256 requests x 1 new token, context U{512..4096}, block_size 16, "
               "40960-block pool, KV 8x128 bf16 (one layer), 1-4 contiguous ranges per request; "
               "step = paged slot map + range slot map + KV write (one CUDA graph: paged map -> "
               "write, the range map on a second branch)")
GATHER_DESC = ("long-context gather: 8 requests x 131072 tokens, block_size 16, KV 8x128 bf16, "
               "whole context of every request into packed K/V buffers (8.59 GB moved)")


# --------------------------------------------------------------------------
# peaks, clocks, profile-derived traffic
# --------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


_REASONS = [(0x1, "gpu_idle"), (0x2, "applications_clocks_setting"), (0x4, "sw_power_cap"),
            (0x8, "hw_slowdown"), (0x10, "sync_boost"), (0x20, "sw_thermal_slowdown"),
            (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"),
            (0x100, "display_clock_setting")]


class ClockSampler:
    """Samples the SM clock and clock-event reasons through NVML (read only)."""

    def __init__(self, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._h = None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            bus = self._bus_id()
            ok = False
            if bus:
                ok = nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            if not ok and nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self._nvml, self._h = nvml, h
            m = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = int(m.value)
            self._reasons_fn = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except Exception:
            self._nvml = None

    @staticmethod
    def _bus_id():
        try:
            import torch
            p = torch.cuda.get_device_properties(torch.cuda.current_device())
            return "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            return None

    def _sample(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0:
            self.samples.append(int(clk.value))
        if self._reasons_fn(self._h, ctypes.byref(rs)) == 0:
            self.reasons |= int(rs.value)

    def _loop(self):
        while not self._stop.wait(self.period):
            self._sample()

    def __enter__(self):
        # a sample as the region starts, every period inside it, one as it ends:
        # a short region (20 steps take a few ms) still gets several
        if self._nvml is not None:
            self._sample()
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
            self._sample()

    def summary(self):
        if self._nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        names = [n for bit, n in _REASONS if self.reasons & bit and n != "gpu_idle"]
        med = statistics.median(self.samples) if self.samples else None
        return {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(self.samples)}


def kernel_source_sha(kernel: str) -> str:
    """Hash of the sources a kernel is built from (its .cu file and the
    library headers it includes)."""
    files = {"cache_gather_kernel": "kv_cache_gather.cu", "cache_write_kernel": "kv_cache_write.cu",
             "slot_mapping_paged_kernel": "kv_slot_mapping.cu",
             "slot_mapping_range_kernel": "kv_slot_mapping.cu",
             "slot_mapping_range_staged_kernel": "kv_slot_mapping.cu",
             "expand_kernel": "kv_expand.cu",
             "cache_gather_range_kernel": "kv_cache_gather.cu",
             "table_from_ranges_kernel": "kv_range_table.cu",
             "copy_blocks_kernel": "kv_copy_blocks.cu",
             "cache_gather_bulk_kernel": "kv_cache_gather.cu",
             "slot_write_kernel": "kv_slot_write.cu",
             "copy_blocks_bulk_kernel": "kv_copy_blocks.cu"}
    csrc = os.path.join(ROOT, "paged_kv_cache_39_gb300", "csrc")
    # the .cu file and, recursively, the library headers it includes
    order, todo = [], [files[kernel]]
    while todo:
        f = todo.pop(0)
        if f in order or not os.path.exists(os.path.join(csrc, f)):
            continue
        order.append(f)
        with open(os.path.join(csrc, f)) as fh:
            todo += re.findall(r'^#include "([^"]+)"', fh.read(), flags=re.M)
    h = hashlib.sha256()
    for f in order:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current source of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[workload][kernel]
        if e.get("source_sha256") != kernel_source_sha(kernel):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# --------------------------------------------------------------------------
# workloads as lists of launches
# --------------------------------------------------------------------------

class Launch:
    """One timed call of the C ABI; `launches` kernels are enqueued per call."""

    def __init__(self, name, kernel, fn, alg_bytes, units=0, launches=1):
        self.name, self.kernel, self.fn, self.alg_bytes = name, kernel, fn, alg_bytes
        self.units, self.launches = units, launches


def _touched_blocks(g0, g1, T):
    g0 = g0.astype(np.int64)
    g1 = g1.astype(np.int64)
    n = np.where(g1 > g0, (g1 - 1) // T - g0 // T + 1, 0)
    return int(n.sum())


def slotmap_bytes(N, n_max, R):
    return n_max * 8 + N * 8 + N * 4 + (R + 1) * 4


def range_bytes(N, n_max, R, nr):
    return n_max * 8 + N * 8 + (R + 1) * 4 + R * 4 + int(nr[:R].sum()) * 8


def write_bytes(L, N_valid, N, row_bytes):
    return L * N_valid * row_bytes * 4 + N * 8


def fused_bytes(slot_bytes, L, N_valid, N, row_bytes):
    """Slot map plus write, without the write's re-read of the slot mapping."""
    return slot_bytes + write_bytes(L, N_valid, N, row_bytes) - N * 8


def gather_bytes(rows, row_bytes, blocks, R):
    return rows * row_bytes * 4 + blocks * 4 + R * 8


class Built:
    """A workload's launches in stream order.  `branch` lists the indices of
    launches that read nothing the others write and write nothing they read:
    a step's graph runs those on a second branch (see step_fn)."""

    def __init__(self, name, desc, launches, tokens, keep, branch=()):
        self.name, self.desc, self.launches, self.tokens, self.keep = name, desc, launches, tokens, keep
        self.branch = tuple(branch)


def forked(torch, side, chain, branch):
    """One function running `chain` in order on the current stream and
    `branch` in order on `side`, forked from the current stream's state and
    joined back into it; captured in a CUDA graph, the two lists become two
    branches of the graph."""
    def run():
        cur = torch.cuda.current_stream()
        side.wait_stream(cur)
        for fn in chain:
            fn()
        with torch.cuda.stream(side):
            for fn in branch:
                fn()
        cur.wait_stream(side)
    return run


def step_fn(torch, built, side, extra=()):
    """The whole step of `built` (plus `extra` launches after its chain) as
    one function: the independent launches on a second branch."""
    chain = [l.fn for i, l in enumerate(built.launches) if i not in built.branch]
    branch = [built.launches[i].fn for i in built.branch]
    return forked(torch, side, chain + [l.fn for l in extra], branch)


def build_decode(torch, kv, wl, dev, seed=1, extras=False, small=False):
    # small: the same 256-token batch over a 20480-block pool and contexts
    # U{512..1024} (a few GB on the device, for profiler captures)
    w = wl.decode(seed, 20480, 1024) if small else wl.decode(seed)
    lay = w.layouts["G"]
    T, B, H, D = w.block_size, w.num_blocks, w.num_kv_heads, w.head_dim
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    qsl, pos, table = t(w.qsl), t(w.positions), t(lay.table)
    rs, rl, nr = t(lay.range_start), t(lay.range_len), t(lay.num_ranges)
    g0, g1 = t(w.gather_start), t(w.gather_end)
    key = wl.bf16_normal((1, w.num_tokens, H, D), 11, dev)
    val = wl.bf16_normal((1, w.num_tokens, H, D), 12, dev)
    kc = wl.bf16_normal((1, B, T, H, D), 13, dev)
    vc = wl.bf16_normal((1, B, T, H, D), 14, dev)
    slot_p = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
    slot_r = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    rows = int((w.gather_end.astype(np.int64) - w.gather_start).sum())
    k_out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)
    v_out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)
    N, n_max, R = w.num_tokens, w.max_num_tokens, w.num_reqs
    rb = w.row_bytes
    launches = [
        Launch("slot_mapping_paged", "slot_mapping_paged_kernel",
               lambda: kv.kv_slot_mapping_paged(qsl, pos, table, T, B, max_num_tokens=n_max,
                                                slot_mapping=slot_p, err=err),
               slotmap_bytes(N, n_max, R), N),
        Launch("slot_mapping_range", "slot_mapping_range_kernel",
               lambda: kv.kv_slot_mapping_range(qsl, pos, rs, rl, nr, T, B, max_num_tokens=n_max,
                                                slot_mapping=slot_r, err=err),
               range_bytes(N, n_max, R, lay.num_ranges), N),
        Launch("cache_write", "cache_write_kernel",
               lambda: kv.kv_cache_write(key, val, kc, vc, slot_p, err=err),
               write_bytes(1, N, N, rb), N),
    ]
    # the read path after the step: every request's whole context
    gather = Launch("cache_gather", "cache_gather_kernel",
                    lambda: kv.kv_cache_gather(kc, vc, table, g0, g1, k_out=k_out, v_out=v_out,
                                               out_rows=rows, err=err),
                    gather_bytes(rows, rb, _touched_blocks(w.gather_start, w.gather_end, T), R),
                    rows)
    if extras:
        table2 = torch.empty_like(table)
        slot_cp = torch.empty_like(slot_p)
        slot_f = torch.empty_like(slot_p)
        launches += [
            gather,
            Launch("slot_mapping_paged_write", "slot_write_kernel",
                   lambda: kv.kv_slot_mapping_paged_write(qsl, pos, table, T, B, key, val, kc, vc,
                                                          max_num_tokens=n_max,
                                                          slot_mapping=slot_f, err=err),
                   fused_bytes(slotmap_bytes(N, n_max, R), 1, N, N, rb), N),
            Launch("slot_mapping_range_write", "slot_write_kernel",
                   lambda: kv.kv_slot_mapping_range_write(qsl, pos, rs, rl, nr, T, B, key, val,
                                                          kc, vc, max_num_tokens=n_max,
                                                          slot_mapping=slot_f, err=err),
                   fused_bytes(range_bytes(N, n_max, R, lay.num_ranges), 1, N, N, rb), N),
            Launch("slot_mapping_paged_cp[W=4,rank1]", "slot_mapping_paged_kernel",
                   lambda: kv.kv_slot_mapping_paged_cp(qsl, pos, table, T, B, 4, 1, 1,
                                                       max_num_tokens=n_max, slot_mapping=slot_cp,
                                                       err=err),
                   slotmap_bytes(N, n_max, R), N),
            Launch("table_from_ranges", "table_from_ranges_kernel",
                   lambda: kv.kv_table_from_ranges(rs, rl, nr, block_table=table2, err=err),
                   lay.table.size * 4 + int(lay.num_ranges.sum()) * 8 + R * 4, R),
            Launch("cache_gather_bulk", "cache_gather_bulk_kernel",
                   lambda: kv.kv_cache_gather(kc, vc, table, g0, g1, k_out=k_out, v_out=v_out,
                                              out_rows=rows, err=err, bulk=True),
                   gather_bytes(rows, rb, _touched_blocks(w.gather_start, w.gather_end, T), R),
                   rows),
            Launch("cache_gather_range", "cache_gather_range_kernel",
                   lambda: kv.kv_cache_gather_range(kc, vc, rs, rl, nr, g0, g1, k_out=k_out,
                                                    v_out=v_out, out_rows=rows, err=err),
                   rows * rb * 4 + int(lay.num_ranges.sum()) * 8 + R * 12, rows),
        ]
    keep = dict(w=w, lay=lay, qsl=qsl, pos=pos, table=table, rs=rs, rl=rl, nr=nr, g0=g0, g1=g1,
                key=key, val=val, kc=kc, vc=vc, slot_p=slot_p, slot_r=slot_r, err=err,
                k_out=k_out, v_out=v_out, rows=rows, gather=gather)
    # the range map (its own slot buffer) is independent of the paged map and
    # the write, which reads the paged map's slots
    return Built("decode", DECODE_DESC, launches, N, keep, branch=(1,))


def build_mixed(torch, kv, wl, dev, small=False):
    free, _ = torch.cuda.mem_get_info(dev)
    L = 1 if small else 32
    w = wl.mixed()
    note = ""
    if not small and free < 2 * 32 * 49152 * 16 * 2048 + (8 << 30):
        w = wl.mixed(num_blocks=32768, decode_ctx_max=2048)
        note = " (reduced: 32768 blocks, decode ctx U{512..2048}, for free memory)"
    lay = w.layouts["G"]
    T, B, H, D = w.block_size, w.num_blocks, w.num_kv_heads, w.head_dim
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    qsl, pos, table = t(w.qsl), t(w.positions), t(lay.table)
    rs, rl, nr = t(lay.range_start), t(lay.range_len), t(lay.num_ranges)
    key = wl.bf16_normal((L, w.num_tokens, H, D), 21, dev)
    val = wl.bf16_normal((L, w.num_tokens, H, D), 22, dev)
    kc = torch.full((L, B, T, H, D), 0x3C01, dtype=torch.int16, device=dev).view(torch.bfloat16)
    vc = torch.full((L, B, T, H, D), 0x3C01, dtype=torch.int16, device=dev).view(torch.bfloat16)
    slot_p = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
    slot_r = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
    slot_f = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    N, n_max, R = w.num_tokens, w.max_num_tokens, w.num_reqs
    # copy-on-write fork of 1024 blocks (every layer): disjoint sources and targets
    perm = np.random.default_rng(5).permutation(np.arange(1, B, dtype=np.int32))
    n_cow = 1024
    cow_src, cow_dst = t(perm[:n_cow]), t(perm[n_cow:2 * n_cow])
    launches = [
        Launch("slot_mapping_paged", "slot_mapping_paged_kernel",
               lambda: kv.kv_slot_mapping_paged(qsl, pos, table, T, B, max_num_tokens=n_max,
                                                slot_mapping=slot_p, err=err),
               slotmap_bytes(N, n_max, R), N),
        Launch("slot_mapping_range", "slot_mapping_range_kernel",
               lambda: kv.kv_slot_mapping_range(qsl, pos, rs, rl, nr, T, B, max_num_tokens=n_max,
                                                slot_mapping=slot_r, err=err),
               range_bytes(N, n_max, R, lay.num_ranges), N),
        Launch("cache_write", "cache_write_kernel",
               lambda: kv.kv_cache_write(key, val, kc, vc, slot_p, err=err),
               write_bytes(L, N, N, w.row_bytes), N * L),
        Launch("slot_mapping_paged_write", "slot_write_kernel",
               lambda: kv.kv_slot_mapping_paged_write(qsl, pos, table, T, B, key, val, kc, vc,
                                                      max_num_tokens=n_max, slot_mapping=slot_f,
                                                      err=err),
               fused_bytes(slotmap_bytes(N, n_max, R), L, N, N, w.row_bytes), N * L),
        Launch("slot_mapping_range_write", "slot_write_kernel",
               lambda: kv.kv_slot_mapping_range_write(qsl, pos, rs, rl, nr, T, B, key, val, kc,
                                                      vc, max_num_tokens=n_max,
                                                      slot_mapping=slot_f, err=err),
               fused_bytes(range_bytes(N, n_max, R, lay.num_ranges), L, N, N, w.row_bytes),
               N * L),
        Launch("copy_blocks[cow 1024]", "copy_blocks_kernel",
               lambda: kv.kv_copy_blocks(kc, vc, cow_src, cow_dst, err=err),
               n_cow * L * T * w.row_bytes * 4 + n_cow * 8, n_cow * L),
        Launch("copy_blocks_bulk[cow 1024]", "copy_blocks_bulk_kernel",
               lambda: kv.kv_copy_blocks(kc, vc, cow_src, cow_dst, err=err, bulk=True),
               n_cow * L * T * w.row_bytes * 4 + n_cow * 8, n_cow * L),
    ]
    desc = (f"mixed prefill+decode: 16 prefill chunks (8192 tokens) + 240 decode tokens, "
            f"{L} layers, {B}-block pool per layer, KV 8x128 bf16, 1-8 ranges/request{note}")
    keep = dict(kc=kc, vc=vc, key=key, val=val, err=err)
    return Built("mixed", desc, launches, N, keep)


def build_long(torch, kv, wl, dev, small=False):
    w = wl.long_context(num_reqs=2 if small else 8)
    T, B, H, D = w.block_size, w.num_blocks, w.num_kv_heads, w.head_dim
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    qsl, pos = t(w.qsl), t(w.positions)
    tp, tg = t(w.layouts["P"].table), t(w.layouts["G"].table)
    lg = w.layouts["G"]
    rs, rl, nr = t(lg.range_start), t(lg.range_len), t(lg.num_ranges)
    g0, g1 = t(w.gather_start), t(w.gather_end)
    tg_rebuilt = torch.empty_like(tg)
    # copy-on-write of 4096 blocks (disjoint sources and targets), 537 MB moved
    n_cow = 4096
    perm = np.random.default_rng(6).permutation(np.arange(1, B, dtype=np.int32))
    cow_src, cow_dst = t(perm[:n_cow]), t(perm[n_cow:2 * n_cow])
    kc = wl.bf16_normal((1, B, T, H, D), 31, dev)
    vc = wl.bf16_normal((1, B, T, H, D), 32, dev)
    rows = w.num_tokens
    k_out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)
    v_out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)
    slot = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
    slot_pre = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
    key = wl.bf16_normal((1, w.num_tokens, H, D), 33, dev)
    val = wl.bf16_normal((1, w.num_tokens, H, D), 34, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    N, R = w.num_tokens, w.num_reqs
    gb = gather_bytes(rows, w.row_bytes, _touched_blocks(w.gather_start, w.gather_end, T), R)
    # the prompt's K/V written once (prefill) through the permuted table, so the
    # write kernel also runs on inputs far larger than L2
    kv.kv_slot_mapping_paged(qsl, pos, tp, T, B, slot_mapping=slot_pre, err=err)
    launches = [
        Launch("cache_write[prefill,P]", "cache_write_kernel",
               lambda: kv.kv_cache_write(key, val, kc, vc, slot_pre, err=err),
               write_bytes(1, N, N, w.row_bytes), N),
        Launch("slot_mapping_paged[P]", "slot_mapping_paged_kernel",
               lambda: kv.kv_slot_mapping_paged(qsl, pos, tp, T, B, slot_mapping=slot, err=err),
               slotmap_bytes(N, N, R), N),
        Launch("slot_mapping_paged[G]", "slot_mapping_paged_kernel",
               lambda: kv.kv_slot_mapping_paged(qsl, pos, tg, T, B, slot_mapping=slot, err=err),
               slotmap_bytes(N, N, R), N),
        Launch("slot_mapping_range[G]", "slot_mapping_range_kernel",
               lambda: kv.kv_slot_mapping_range(qsl, pos, rs, rl, nr, T, B, slot_mapping=slot,
                                                err=err),
               range_bytes(N, N, R, lg.num_ranges), N),
        Launch("cache_gather[P]", "cache_gather_kernel",
               lambda: kv.kv_cache_gather(kc, vc, tp, g0, g1, k_out=k_out, v_out=v_out,
                                          out_rows=rows, err=err), gb, rows),
        Launch("cache_gather[G]", "cache_gather_kernel",
               lambda: kv.kv_cache_gather(kc, vc, tg, g0, g1, k_out=k_out, v_out=v_out,
                                          out_rows=rows, err=err), gb, rows),
        Launch("cache_gather_bulk[P]", "cache_gather_bulk_kernel",
               lambda: kv.kv_cache_gather(kc, vc, tp, g0, g1, k_out=k_out, v_out=v_out,
                                          out_rows=rows, err=err, bulk=True), gb, rows),
        Launch("cache_gather_bulk[G]", "cache_gather_bulk_kernel",
               lambda: kv.kv_cache_gather(kc, vc, tg, g0, g1, k_out=k_out, v_out=v_out,
                                          out_rows=rows, err=err, bulk=True), gb, rows),
        Launch("cache_gather_range[G]", "cache_gather_range_kernel",
               lambda: kv.kv_cache_gather_range(kc, vc, rs, rl, nr, g0, g1, k_out=k_out,
                                                v_out=v_out, out_rows=rows, err=err),
               rows * w.row_bytes * 4 + int(lg.num_ranges.sum()) * 8 + R * 12, rows),
        Launch("table_from_ranges[G]", "table_from_ranges_kernel",
               lambda: kv.kv_table_from_ranges(rs, rl, nr, block_table=tg_rebuilt, err=err),
               lg.table.size * 4 + int(lg.num_ranges.sum()) * 8 + R * 4, R),
        Launch(f"copy_blocks[cow {n_cow}]", "copy_blocks_kernel",
               lambda: kv.kv_copy_blocks(kc, vc, cow_src, cow_dst, err=err),
               n_cow * T * w.row_bytes * 4 + n_cow * 8, n_cow),
        Launch(f"copy_blocks_bulk[cow {n_cow}]", "copy_blocks_bulk_kernel",
               lambda: kv.kv_copy_blocks(kc, vc, cow_src, cow_dst, err=err, bulk=True),
               n_cow * T * w.row_bytes * 4 + n_cow * 8, n_cow),
    ]
    desc = (f"long-context gather: {R} requests x 131072 tokens, block_size 16, KV 8x128 bf16; "
            "P = permuted block table, G = 1-16 packed ranges per request; plus the prompt's "
            "prefill write through P and a 4096-block copy-on-write")
    keep = dict(kc=kc, vc=vc, k_out=k_out, v_out=v_out, key=key, val=val, err=err)
    return Built("long", desc, launches, N, keep)


def build_hybrid(torch, kv, wl, dev, small=False):
    h = wl.hybrid(num_real=128 if small else 512, num_padded=160 if small else 640)
    H, D = h.num_kv_heads, h.head_dim
    rb = H * D * 2
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    qsl, pos = t(h.qsl), t(h.positions)
    key = wl.bf16_normal((1, h.num_tokens, H, D), 41, dev)
    val = wl.bf16_normal((1, h.num_tokens, H, D), 42, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    launches, keep = [], dict(key=key, val=val, err=err)
    R, N, n_max = h.num_reqs, h.num_tokens, h.max_num_tokens
    for name, g in h.groups.items():
        kbs, mbs, Bk = g.kernel_block_size, g.mgr_block_size, g.kernel_num_blocks
        k = mbs // kbs
        mgr = t(g.mgr_table)
        kt = torch.empty((R, g.mgr_table.shape[1] * k), dtype=torch.int32, device=dev)
        kc = wl.bf16_normal((1, Bk, kbs, H, D), 43 + len(name), dev)
        vc = wl.bf16_normal((1, Bk, kbs, H, D), 45 + len(name), dev)
        slot = torch.empty(n_max, dtype=torch.int64, device=dev)
        # gather calls: 64 real requests per call, then the padding rows in one call
        calls = [(c, min(c + 64, h.num_real_reqs)) for c in range(0, h.num_real_reqs, 64)]
        calls.append((h.num_real_reqs, R))
        max_rows = max(int((g.gather_end[a:b].astype(np.int64) - g.gather_start[a:b]).sum())
                       for a, b in calls)
        k_out = torch.empty((max(max_rows, 1), H, D), dtype=torch.bfloat16, device=dev)
        v_out = torch.empty((max(max_rows, 1), H, D), dtype=torch.bfloat16, device=dev)
        g0, g1 = t(g.gather_start), t(g.gather_end)
        keep.update({f"{name}_{x}": y for x, y in dict(mgr=mgr, kt=kt, kc=kc, vc=vc, slot=slot,
                                                         k_out=k_out, v_out=v_out, g0=g0,
                                                         g1=g1).items()})
        rows_total = int((g.gather_end.astype(np.int64) - g.gather_start).sum())

        def gather_all(kc=kc, vc=vc, kt=kt, g0=g0, g1=g1, k_out=k_out, v_out=v_out, calls=calls,
                       g=g):
            for a, b in calls:
                rows = int((g.gather_end[a:b].astype(np.int64) - g.gather_start[a:b]).sum())
                kv.kv_cache_gather(kc, vc, kt[a:b], g0[a:b], g1[a:b], k_out=k_out, v_out=v_out,
                                   out_rows=rows, err=err)

        launches += [
            Launch(f"expand[{name}]", "expand_kernel",
                   lambda mgr=mgr, kt=kt, mbs=mbs, kbs=kbs: kv.kv_expand_kernel_blocks(
                       mgr, mbs, kbs, kernel_table=kt, err=err),
                   g.mgr_table.size * 4 + R * g.mgr_table.shape[1] * k * 4, R),
            Launch(f"slot_mapping_paged[{name}]", "slot_mapping_paged_kernel",
                   lambda kt=kt, slot=slot, kbs=kbs, Bk=Bk: kv.kv_slot_mapping_paged(
                       qsl, pos, kt, kbs, Bk, max_num_tokens=n_max, slot_mapping=slot, err=err),
                   slotmap_bytes(N, n_max, R), N),
            Launch(f"cache_write[{name}]", "cache_write_kernel",
                   lambda kc=kc, vc=vc, slot=slot: kv.kv_cache_write(key, val, kc, vc, slot[:N],
                                                                      err=err),
                   write_bytes(1, N, N, rb), N),
            Launch(f"cache_gather[{name}]", "cache_gather_kernel", gather_all,
                   gather_bytes(rows_total, rb, _touched_blocks(g.gather_start, g.gather_end, kbs),
                                R), rows_total, launches=len(calls)),
        ]
    desc = (f"hybrid groups: {h.num_real_reqs} requests padded to {R}, context U{{1..32768}}, "
            "manager block 32 -> kernel block 16, full-attention + sliding-window 4096 groups, "
            "KV 8x128 bf16; gather in calls of 64 requests + one call on the padding rows")
    return Built("hybrid", desc, launches, N, keep)


def build_slotmap(torch, kv, wl, dev, small=False, reqs=None):
    """The long-context slot maps alone (1M positions, no caches): a small
    device footprint for full profiler captures of the two strategies.
    `reqs` requests of 131072 positions instead of 8 scale the same maps up
    (4M, 16M positions); beside them a plain copy kernel over the same bytes
    (positions read, one int64 per token written) gives the floor a kernel of
    this shape reaches at that size."""
    w = wl.long_context(num_reqs=reqs or (2 if small else 8))
    T, B = w.block_size, w.num_blocks
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    qsl, pos = t(w.qsl), t(w.positions)
    tp, tg = t(w.layouts["P"].table), t(w.layouts["G"].table)
    lg = w.layouts["G"]
    rs, rl, nr = t(lg.range_start), t(lg.range_len), t(lg.num_ranges)
    slot = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    N, R = w.num_tokens, w.num_reqs
    launches = [
        Launch("slot_mapping_paged[P]", "slot_mapping_paged_kernel",
               lambda: kv.kv_slot_mapping_paged(qsl, pos, tp, T, B, slot_mapping=slot, err=err),
               slotmap_bytes(N, N, R), N),
        Launch("slot_mapping_paged[G]", "slot_mapping_paged_kernel",
               lambda: kv.kv_slot_mapping_paged(qsl, pos, tg, T, B, slot_mapping=slot, err=err),
               slotmap_bytes(N, N, R), N),
        Launch("slot_mapping_range[G]", "slot_mapping_range_kernel",
               lambda: kv.kv_slot_mapping_range(qsl, pos, rs, rl, nr, T, B, slot_mapping=slot,
                                                err=err),
               range_bytes(N, N, R, lg.num_ranges), N),
    ]
    floor_out = torch.empty_like(slot)
    launches.append(Launch("copy_floor[torch add: positions in, int64 out]", "elementwise_kernel",
                           lambda: torch.add(pos, 1, out=floor_out), 16 * N, N))
    desc = f"long-context slot maps only: {R} requests x 131072 positions, block_size 16"
    return Built("slotmap", desc, launches, N, dict(err=err))


BUILDERS = {"decode": build_decode, "mixed": build_mixed, "long": build_long,
            "hybrid": build_hybrid, "slotmap": build_slotmap}


# --------------------------------------------------------------------------
# timing
# --------------------------------------------------------------------------

def flush_l2(buf):
    """Write a buffer larger than L2, then read another one: the read evicts the
    dirty lines the write left, so their write-back happens here and not
    inside the next timed step.  The read is an int32 max (a sum would first
    cast the half to int64 through a freshly written temporary, leaving L2
    dirty again)."""
    n = buf.numel() // 2
    buf[:n].add_(1)
    buf[n:].max()


def time_steps(torch, built, steps, flush_buf, stream):
    """Per-step and per-launch device times (ms) over `steps` steps, L2 flushed
    between steps (launches inside a step share what the step reuses)."""
    nl = len(built.launches)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(steps)]
    for s in range(steps):
        flush_l2(flush_buf)
        evs[s][0].record(stream)
        for i, l in enumerate(built.launches):
            l.fn()
            evs[s][i + 1].record(stream)
    torch.cuda.synchronize()
    step_ms = [evs[s][0].elapsed_time(evs[s][nl]) for s in range(steps)]
    per = [[evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)] for i in range(nl)]
    return step_ms, per


def time_each(torch, built, reps, flush_buf, stream):
    """Per-launch device times (ms) with the L2 flushed before every launch, so
    no launch finds another's inputs in cache."""
    nl = len(built.launches)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(nl)] for _ in range(reps)]
    for s in range(reps):
        for i, l in enumerate(built.launches):
            flush_l2(flush_buf)
            evs[s][i][0].record(stream)
            l.fn()
            evs[s][i][1].record(stream)
    torch.cuda.synchronize()
    return [[evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(reps)] for i in range(nl)]


def kernel_report(built, per, peak):
    out = {}
    for l, times in zip(built.launches, per):
        avg = sum(times) / len(times)
        gbs = l.alg_bytes / (avg * 1e-3) / 1e9
        out[l.name] = {"us": round(avg * 1e3, 2), "us_median": round(statistics.median(times) * 1e3, 2),
                       "alg_bytes": int(l.alg_bytes), "GB/s": round(gbs, 1),
                       "frac_of_measured_hbm": round(gbs / peak, 4),
                       "frac_of_8TBps": round(gbs / 8000.0, 4)}
    return out


# --------------------------------------------------------------------------
# CPU oracle runs (baseline leg and reference arm)
# --------------------------------------------------------------------------

def oracle_write_step(oracle, w, lay, kc_h, vc_h, key_h, val_h):
    """One oracle pass of the headline step on the whole decode batch: both
    slot maps, then the write of every new token's K/V rows."""
    n, T, B = w.num_tokens, w.block_size, w.num_blocks
    sp, _ = oracle.slot_mapping_paged(w.qsl, w.positions, lay.table, n, w.max_num_tokens, T, B)
    oracle.slot_mapping_range(w.qsl, w.positions, lay.range_start, lay.range_len, lay.num_ranges,
                              n, w.max_num_tokens, T, B)
    oracle.cache_write(key_h, val_h, kc_h, vc_h, sp[:n], B, T)
    return n


def oracle_gather_step(oracle, w, lay, kc_h, vc_h, n_req):
    """The oracle's context gather of the first n_req requests of the decode batch."""
    g0, g1 = w.gather_start[:n_req], w.gather_end[:n_req]
    rows = int((g1.astype(np.int64) - g0).sum())
    ko = np.empty((rows, w.num_kv_heads, w.head_dim), np.uint16)
    vo = np.empty_like(ko)
    oracle.cache_gather(kc_h, vc_h, 0, w.num_blocks, w.block_size, lay.table[:n_req], g0, g1, ko,
                        vo)
    return rows


def host_decode_state(wl, seed=1):
    w = wl.decode(seed)
    lay = w.layouts["G"]
    rng = np.random.default_rng(99)
    shape = (1, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    # zero-filled host caches: their contents do not change the oracle's work
    kc_h = np.zeros(shape, np.uint16)
    vc_h = np.zeros(shape, np.uint16)
    key_h = rng.integers(0, 1 << 16, size=(1, w.num_tokens, w.num_kv_heads, w.head_dim),
                         dtype=np.uint16)
    val_h = rng.integers(0, 1 << 16, size=key_h.shape, dtype=np.uint16)
    return w, lay, kc_h, vc_h, key_h, val_h


def host_cpu():
    """The host CPU's model as the OS reports it ("unknown" when it does not)."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        m = re.search(r"^model name\s*:\s*(.+)$", info, flags=re.M)
        if m:
            return m.group(1).strip()
        # Arm cores name the implementer and the part number instead
        impl = re.search(r"^CPU implementer\s*:\s*(\S+)", info, flags=re.M)
        part = re.search(r"^CPU part\s*:\s*(\S+)", info, flags=re.M)
        if impl and part:
            parts = {("0x41", "0xd4f"): "Arm Neoverse V2", ("0x41", "0xd40"): "Arm Neoverse V1",
                     ("0x41", "0xd0c"): "Arm Neoverse N1"}
            key = (impl.group(1).lower(), part.group(1).lower())
            return parts.get(key, f"{platform.machine()} implementer {key[0]} part {key[1]}")
    except OSError:
        pass
    return platform.processor() or platform.machine() or "unknown"


def cpu_baseline(seconds, rounds=5):
    """The oracle's headline step on one host core, timed in the pages' host-bench
    manner: `rounds` rounds, one warm-up call per round, then whole steps for
    seconds / rounds; value = mean of the per-round rates, with their stddev."""
    import oracle
    from paged_kv_cache_39_gb300 import workloads as wl
    w, lay, kc_h, vc_h, key_h, val_h = host_decode_state(wl)
    rates, steps_total, el_total = [], 0, 0.0
    for _ in range(rounds):
        oracle_write_step(oracle, w, lay, kc_h, vc_h, key_h, val_h)  # warm-up call
        t0 = time.perf_counter()
        steps, toks = 0, 0
        while True:
            toks += oracle_write_step(oracle, w, lay, kc_h, vc_h, key_h, val_h)
            steps += 1
            el = time.perf_counter() - t0
            if el >= seconds / rounds:
                break
        rates.append(toks / el)
        steps_total += steps
        el_total += el
    return {"value": round(statistics.mean(rates), 1),
            "stddev": round(statistics.stdev(rates), 1) if rounds > 1 else 0.0,
            "rounds": rounds, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps_total} whole headline steps of the oracle (paged and range slot "
                      f"maps and the KV write of all 256 decode tokens) in {rounds} rounds, "
                      f"single-threaded, {el_total:.1f} s",
            "host_cores": os.cpu_count(), "host_cpu": host_cpu(),
            "cores_note": f"1 of {os.cpu_count()} cores"}


def oracle_rows(seconds_cap=4.0):
    """The oracle timed per row on bounded samples of the workloads (one host
    core); units per second, each with its sample.  A baseline beside the GPU
    figures, not a target."""
    import oracle
    from paged_kv_cache_39_gb300 import workloads as wl
    out = {}

    def timed(name, unit, n_units, sample, fn):
        fn()  # warm
        t0 = time.perf_counter()
        reps = 0
        while True:
            fn()
            reps += 1
            el = time.perf_counter() - t0
            if el >= seconds_cap or reps >= 3:
                break
        per = el / reps
        out[name] = {"seconds": round(per, 5), "value": round(n_units / per, 1), "unit": unit,
                     "sample": sample}

    lw = wl.long_context()
    lp, lg = lw.layouts["P"], lw.layouts["G"]
    T, B, N = lw.block_size, lw.num_blocks, lw.num_tokens
    timed("slot_mapping_paged", "positions/s", N, "long context, 8 x 131072 positions, table P",
          lambda: oracle.slot_mapping_paged(lw.qsl, lw.positions, lp.table, N, N, T, B))
    timed("slot_mapping_range", "positions/s", N, "long context, 8 x 131072 positions, 1-16 ranges",
          lambda: oracle.slot_mapping_range(lw.qsl, lw.positions, lg.range_start, lg.range_len,
                                            lg.num_ranges, N, N, T, B))
    timed("slot_mapping_paged_cp", "positions/s", N, "long context, table P, W=4 rank 1",
          lambda: oracle.slot_mapping_paged_cp(lw.qsl, lw.positions, lp.table, N, N, T, B, 4, 1,
                                               1))
    timed("table_from_ranges", "entries/s", lg.table.size, "long context, 8 x 8192 entries",
          lambda: oracle.table_from_ranges(lg.range_start, lg.range_len, lg.num_ranges,
                                           lg.table_stride))
    # one request's whole context (131072 rows of K and V) from a long-context cache
    shape = (1, B, T, lw.num_kv_heads, lw.head_dim)
    kc = np.full(shape, 0x3C01, np.uint16)
    vc = np.full(shape, 0x3C02, np.uint16)
    rows = 131072
    ko = np.empty((rows, lw.num_kv_heads, lw.head_dim), np.uint16)
    vo = np.empty_like(ko)
    timed("cache_gather", "rows/s", rows, "long context, one request's 131072 rows (table P)",
          lambda: oracle.cache_gather(kc, vc, 0, B, T, lp.table[:1], lw.gather_start[:1],
                                      lw.gather_end[:1], ko, vo))
    src, _ = oracle.gather_rows_range(0, B, T, lg.range_start[:1], lg.range_len[:1],
                                      lg.num_ranges[:1], lw.gather_start[:1], lw.gather_end[:1],
                                      rows)
    timed("cache_gather_range (row resolution only)", "rows/s", rows,
          "long context, one request's 131072 rows through its ranges (source rows only)",
          lambda: oracle.gather_rows_range(0, B, T, lg.range_start[:1], lg.range_len[:1],
                                           lg.num_ranges[:1], lw.gather_start[:1],
                                           lw.gather_end[:1], rows))
    key = np.full((1, rows, lw.num_kv_heads, lw.head_dim), 0x3C03, np.uint16)
    slots, _ = oracle.slot_mapping_paged(lw.qsl[:2], lw.positions[:rows], lp.table[:1], rows,
                                         rows, T, B)
    timed("cache_write", "rows/s", rows, "long context, one request's 131072-row prefill write",
          lambda: oracle.cache_write(key, key, kc, vc, slots, B, T))
    perm = np.random.default_rng(5).permutation(np.arange(1, B, dtype=np.int32))
    timed("copy_blocks", "blocks/s", 1024, "1024 block copies in a one-layer long-context cache",
          lambda: oracle.copy_blocks(kc, vc, perm[:1024], perm[1024:2048]))
    del kc, vc, ko, vo, key
    h = wl.hybrid()
    g = h.groups["full"]
    timed("expand_kernel_blocks", "entries/s", g.mgr_table.size * 2,
          "hybrid full-attention table 640 x 1024 -> 640 x 2048",
          lambda: oracle.expand_kernel_blocks(g.mgr_table, 32, 16))

    # Large host caches are zero-filled by the allocator, so only the pages a
    # call touches are ever backed: the blocks a gather reads are written
    # first (a read of a never-written page would see one shared zero page),
    # the rows a write fills are backed by its warm-up call.
    # hybrid full-attention group: one gather call of 64 requests, as issued
    kt, _ = oracle.expand_kernel_blocks(g.mgr_table, g.mgr_block_size, g.kernel_block_size)
    kbs, Bk = g.kernel_block_size, g.kernel_num_blocks
    shape = (1, Bk, kbs, h.num_kv_heads, h.head_dim)
    kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    g0, g1 = g.gather_start[:64], g.gather_end[:64]
    rows = int((g1.astype(np.int64) - g0).sum())
    touched = np.unique(np.concatenate([kt[r, :-(-int(g1[r]) // kbs)] for r in range(64)]))
    touched = touched[touched > 0]
    kc[0, touched] = 0x3C01
    vc[0, touched] = 0x3C02
    ko = np.empty((rows, h.num_kv_heads, h.head_dim), np.uint16)
    vo = np.empty_like(ko)
    timed("cache_gather (hybrid full, one 64-request call)", "rows/s", rows,
          f"hybrid full-attention group: the first gather call (64 requests, {rows} rows)",
          lambda: oracle.cache_gather(kc, vc, 0, Bk, kbs, kt[:64], g0, g1, ko, vo))
    full_rows = int((g.gather_end.astype(np.int64) - g.gather_start).sum())
    e = out["cache_gather (hybrid full, one 64-request call)"]
    e["scaled_full_group_s"] = round(full_rows / e["value"], 2)
    e["scaled"] = f"the whole group ({full_rows} rows in 9 calls) at this call's rate"
    del kc, vc, ko, vo
    # mixed prefill+decode: the 32-layer write of all 8432 tokens
    mw = wl.mixed()
    L, T, B = mw.num_layers, mw.block_size, mw.num_blocks
    shape = (L, B, T, mw.num_kv_heads, mw.head_dim)
    kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    key = np.full((L, mw.num_tokens, mw.num_kv_heads, mw.head_dim), 0x3C03, np.uint16)
    slots, _ = oracle.slot_mapping_paged(mw.qsl, mw.positions, mw.layouts["G"].table,
                                         mw.num_tokens, mw.num_tokens, T, B)
    timed("cache_write (mixed, 32 layers)", "rows/s", L * mw.num_tokens,
          f"mixed prefill+decode: all {mw.num_tokens} tokens x {L} layers (full size)",
          lambda: oracle.cache_write(key, key, kc, vc, slots, B, T))
    del kc, vc, key
    return out


def run_reference(args, rk):
    """The oracle as the reference arm: the headline step (both slot maps and
    the write of all 256 decode tokens) on one host core."""
    if not rk.is_main:
        return
    import oracle
    from paged_kv_cache_39_gb300 import workloads as wl
    w, lay, kc_h, vc_h, key_h, val_h = host_decode_state(wl)
    for _ in range(args.warmup):
        oracle_write_step(oracle, w, lay, kc_h, vc_h, key_h, val_h)
    t0 = time.perf_counter()
    toks = 0
    for _ in range(args.steps):
        toks += oracle_write_step(oracle, w, lay, kc_h, vc_h, key_h, val_h)
    el = time.perf_counter() - t0
    value = toks / el
    sample = ("each step: the oracle's headline step on all 256 requests of the decode batch "
              "(paged and range slot maps, KV write), single-threaded")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int64", "data": "synthetic",
            "config": {"workload": DECODE_DESC, "parallelism": "host cores, rank 0"},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": 1,
                             "kind": "oracle", "sample": sample, "host_cores": os.cpu_count(),
                             "host_cpu": host_cpu()},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class GraphStep:
    """`fns` captured once in a CUDA graph (on a side stream first, so lazy
    set-up stays out of the capture); replay() launches the whole step."""

    def __init__(self, torch, fns):
        self.torch = torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for fn in fns:
                fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g):
            for fn in fns:
                fn()
        for _ in range(3):
            self.g.replay()
        torch.cuda.synchronize()

    def replay(self):
        self.g.replay()

    def times_ms(self, steps, flush_buf):
        """Device time of each of `steps` replays (CUDA events on the launching
        stream), L2 flushed between replays outside the events."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush_l2(flush_buf)
            a.record()
            self.g.replay()
            b.record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]


def graph_replay_ms(torch, fns, steps, flush_buf):
    """Mean device time (ms) of one replay of `fns` captured in a CUDA graph."""
    g = GraphStep(torch, fns)
    ms = sum(g.times_ms(steps, flush_buf)) / steps
    del g
    return ms


def launch_floor_us(torch, dev, steps, flush_buf):
    """One replay of a graph holding a single one-element torch kernel: the
    launch-and-complete floor every latency-bound kernel here sits on."""
    z = torch.zeros(1, dtype=torch.int32, device=dev)
    return round(graph_replay_ms(torch, [lambda: z.add_(1)], steps, flush_buf) * 1e3, 2)


def paged_vs_range(torch, kv, built, steps, reps, flush_buf, stream):
    """Slot map + KV write of the decode batch by each strategy: the separate
    slot-map and write launches, and the fused calls, each replayed from one
    CUDA graph (L2 flushed between replays) and, per launch, timed alone with
    the L2 flushed before it."""
    k = built.keep
    w = k["w"]
    T, B, n_max = w.block_size, w.num_blocks, w.max_num_tokens
    q, p, kc, vc, key, val, err = k["qsl"], k["pos"], k["kc"], k["vc"], k["key"], k["val"], k["err"]
    slot_p, slot_r = k["slot_p"], k["slot_r"]
    # every variant writes (and its write reads) one shared slot buffer: where
    # a buffer lies moves these latency-bound pairs by up to ~1.5 us, which
    # would otherwise pass for a difference between the strategies
    s = torch.empty_like(slot_p)
    calls = {
        "slot_mapping_paged": lambda: kv.kv_slot_mapping_paged(q, p, k["table"], T, B,
                                                               max_num_tokens=n_max,
                                                               slot_mapping=s, err=err),
        "slot_mapping_range": lambda: kv.kv_slot_mapping_range(q, p, k["rs"], k["rl"], k["nr"],
                                                               T, B, max_num_tokens=n_max,
                                                               slot_mapping=s, err=err),
        "cache_write": lambda: kv.kv_cache_write(key, val, kc, vc, s, err=err),
        "slot_mapping_paged_write": lambda: kv.kv_slot_mapping_paged_write(
            q, p, k["table"], T, B, key, val, kc, vc, max_num_tokens=n_max, slot_mapping=s,
            err=err),
        "slot_mapping_range_write": lambda: kv.kv_slot_mapping_range_write(
            q, p, k["rs"], k["rl"], k["nr"], T, B, key, val, kc, vc, max_num_tokens=n_max,
            slot_mapping=s, err=err),
    }
    graphs = {
        "paged": [calls["slot_mapping_paged"], calls["cache_write"]],
        "range": [calls["slot_mapping_range"], calls["cache_write"]],
        "paged_fused": [calls["slot_mapping_paged_write"]],
        "range_fused": [calls["slot_mapping_range_write"]],
    }
    gs = {n: GraphStep(torch, fns) for n, fns in graphs.items()}
    # replays interleaved round robin, so drift affects every variant alike
    evs = {n: [] for n in gs}
    for _ in range(steps):
        for n, g in gs.items():
            flush_l2(flush_buf)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            evs[n].append((a, b))
    torch.cuda.synchronize()
    g_us = {n: sum(a.elapsed_time(b) for a, b in l) / len(l) * 1e3 for n, l in evs.items()}
    del gs
    per_launch = Built("pvr", "", [Launch(n, "", f, 0) for n, f in calls.items()], 0, k)
    per = time_each(torch, per_launch, reps, flush_buf, stream)
    us = {l.name: round(sum(t) / len(t) * 1e3, 2) for l, t in zip(per_launch.launches, per)}
    for name in ("slot_mapping_paged", "slot_mapping_range_write"):
        calls[name]()
        torch.cuda.synchronize()
        if not torch.equal(s, slot_p) or not torch.equal(slot_p, slot_r):
            raise RuntimeError(f"{name}: slot mappings differ between the calls")
    n = built.tokens
    return {
        "tokens_per_s": {name: round(n / (v * 1e-6), 1) for name, v in g_us.items()},
        "graph_replay_us": {name: round(v, 2) for name, v in g_us.items()},
        "range_over_paged": {"separate": round(g_us["range"] / g_us["paged"], 3),
                             "fused": round(g_us["range_fused"] / g_us["paged_fused"], 3)},
        "per_launch_us": us,
        "replays": steps, "per_launch_reps": reps,
        "note": "paged/range: that strategy's slot-map launch then the write launch, captured "
                "in one CUDA graph; *_fused: kv_slot_mapping_{paged,range}_write, one launch "
                "in a graph; the four graphs replayed round robin with the L2 flushed before "
                "each replay, all writing one shared slot buffer.  per_launch_us: each call "
                "alone, L2 flushed before it (the means are over all reps: a single "
                "latency-bound launch varies by about 1 us)",
    }


def gather_long(torch, kv, wl, dev, reps, flush_buf, stream, peak, same_run_copy, small=False):
    """The metric's second half: the whole-context gather of the long-context
    workload through the permuted table P (the general case) and the packed
    ranges' table G, the range-addressed and the bulk-copy gathers beside it."""
    w = wl.long_context(num_reqs=2 if small else 8)
    T, B, H, D = w.block_size, w.num_blocks, w.num_kv_heads, w.head_dim
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    tp, tg = t(w.layouts["P"].table), t(w.layouts["G"].table)
    lg = w.layouts["G"]
    rs, rl, nr = t(lg.range_start), t(lg.range_len), t(lg.num_ranges)
    g0, g1 = t(w.gather_start), t(w.gather_end)
    kc = wl.bf16_normal((1, B, T, H, D), 31, dev)
    vc = wl.bf16_normal((1, B, T, H, D), 32, dev)
    rows = w.num_tokens
    k_out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)
    v_out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    R = w.num_reqs
    gb = gather_bytes(rows, w.row_bytes, _touched_blocks(w.gather_start, w.gather_end, T), R)
    gr = rows * w.row_bytes * 4 + int(lg.num_ranges.sum()) * 8 + R * 12
    b = Built("gather", GATHER_DESC, [
        Launch("cache_gather[P]", "cache_gather_kernel",
               lambda: kv.kv_cache_gather(kc, vc, tp, g0, g1, k_out=k_out, v_out=v_out,
                                          out_rows=rows, err=err), gb, rows),
        Launch("cache_gather[G]", "cache_gather_kernel",
               lambda: kv.kv_cache_gather(kc, vc, tg, g0, g1, k_out=k_out, v_out=v_out,
                                          out_rows=rows, err=err), gb, rows),
        Launch("cache_gather_range[G]", "cache_gather_range_kernel",
               lambda: kv.kv_cache_gather_range(kc, vc, rs, rl, nr, g0, g1, k_out=k_out,
                                                v_out=v_out, out_rows=rows, err=err), gr, rows),
        Launch("cache_gather_bulk[P]", "cache_gather_bulk_kernel",
               lambda: kv.kv_cache_gather(kc, vc, tp, g0, g1, k_out=k_out, v_out=v_out,
                                          out_rows=rows, err=err, bulk=True), gb, rows),
        Launch("cache_gather_bulk[G]", "cache_gather_bulk_kernel",
               lambda: kv.kv_cache_gather(kc, vc, tg, g0, g1, k_out=k_out, v_out=v_out,
                                          out_rows=rows, err=err, bulk=True), gb, rows),
    ], rows, dict(err=err))
    for _ in range(3):
        for l in b.launches:
            l.fn()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit(f"long-context gathers reported data errors: {int(err.item())}")
    per = time_each(torch, b, reps, flush_buf, stream)
    rep = kernel_report(b, per, peak[0])
    p = b.launches[0]
    avg_ms = sum(per[0]) / len(per[0])
    achieved = p.alg_bytes / (avg_ms * 1e-3) / 1e9
    traffic = profiled_traffic(p.kernel, "long")
    if traffic is not None and small:
        traffic = None
    out = {"GBps": round(achieved, 1), "workload": GATHER_DESC + (" [small]" if small else ""),
           "kernels": rep,
           "roofline": {"bound": "hbm", "kernel": p.kernel + " (table P)",
                        "achieved": round(achieved, 1), "peak": peak[0],
                        "peak_kind": f"{peak[1]} hbm_gbs (copy, read+write)", "unit": "GB/s",
                        "frac": round(achieved / peak[0], 4), "traffic": traffic,
                        "alg_bytes_per_launch": int(p.alg_bytes),
                        "avg_launch_us": round(avg_ms * 1e3, 2),
                        "same_run_copy_GBps": same_run_copy,
                        "frac_of_same_run_copy": round(achieved / same_run_copy, 4),
                        "frac_of_8TBps": round(achieved / 8000.0, 4)},
           "l2": "inputs and outputs (4.3 GB each way) far larger than L2; flushed before "
                 "every launch as well", "reps": reps}
    del b, kc, vc, k_out, v_out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def decode_step_with_gather(torch, built, steps, flush_buf, stream, peak, args):
    """The decode step followed by the read path: the three calls of the
    headline step, then the gather of every request's whole context (597k
    rows, 4.9 GB moved), timed per launch within each step and replayed from
    one CUDA graph."""
    b = Built("decode+gather", "", built.launches + [built.keep["gather"]], built.tokens,
              built.keep)
    step_ms, per = time_steps(torch, b, steps, flush_buf, stream)
    rep = kernel_report(b, per, peak[0])
    g = b.launches[-1]
    avg_ms = sum(per[-1]) / len(per[-1])
    achieved = g.alg_bytes / (avg_ms * 1e-3) / 1e9
    ms = sum(step_ms) / len(step_ms)
    side = torch.cuda.Stream(device=built.keep["qsl"].device)
    g_ms = graph_replay_ms(torch, [step_fn(torch, built, side, extra=[b.launches[-1]])], steps,
                           flush_buf)
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(b.tokens / (ms * 1e-3), 1),
            "graph_ms_per_step": round(g_ms, 4),
            "graph_tokens_per_s": round(b.tokens / (g_ms * 1e-3), 1),
            "steps": steps, "kernels": rep,
            "gather_roofline": {"bound": "hbm", "kernel": g.kernel,
                                "achieved": round(achieved, 1), "peak": peak[0],
                                "unit": "GB/s", "frac": round(achieved / peak[0], 4),
                                "traffic": profiled_traffic(g.kernel, "decode"),
                                "alg_bytes_per_launch": int(g.alg_bytes),
                                "avg_launch_us": round(avg_ms * 1e3, 2)},
            "note": "per-launch events inside each step, in stream order (L2 flushed between "
                    "steps); graph: the four calls in one CUDA graph, the range map on a second "
                    "branch"}


# --------------------------------------------------------------------------
# end to end through the public API with host buffers
# --------------------------------------------------------------------------

def device_alias(torch, host, dev):
    """A CUDA int32 tensor over the same bytes as the pinned host tensor
    `host` (page-locked memory is mapped into the device's address space, at
    the same address), or None when the driver reports no such mapping."""
    try:
        cudart = ctypes.CDLL("libcudart.so.13")
        attr = (ctypes.c_char * 256)()
        if cudart.cudaPointerGetAttributes(attr, ctypes.c_void_p(host.data_ptr())) != 0:
            return None
        kind = ctypes.c_int.from_buffer(attr, 0).value
        dptr = ctypes.c_void_p.from_buffer(attr, 8).value
        if kind != 1 or dptr != host.data_ptr():  # 1: page-locked host memory
            return None

        class _Iface:
            __cuda_array_interface__ = {"shape": (host.numel() * host.element_size() // 4,),
                                        "typestr": "<i4", "data": (host.data_ptr(), False),
                                        "version": 3, "strides": None}
        alias = torch.as_tensor(_Iface(), device=dev)
    except Exception:
        return None
    return alias if alias.data_ptr() == host.data_ptr() else None


def e2e_step(torch, kv, built, steps, flush_buf, stream, upload="sm", download="ce"):
    """The headline step through the public API from host memory: every step
    copies its inputs from pinned host memory (packed, one copy: an
    elementwise kernel reading the pinned buffer through its device mapping,
    13.5-13.6 against 13.8-14.3 us per step by the copy engine, which is used
    where the driver reports no mapping or with upload="ce"; download="sm"
    reads the outputs back the same way, measured slower: 15.2-15.6 against
    14.1-14.3 us), runs the
    three prepared calls (paged map -> write, the range map on a second
    branch, as in the device-resident step), and copies both slot mappings and
    the error word back to pinned host memory, where the host checks them.
    The packed upload ends with zero bytes over the set's error word, so the
    copy that brings a step's inputs also clears its error word.

    Measured the way a pipelined serving loop runs it, inputs prepared one
    step ahead and results checked two steps behind: three buffer sets, and
    for set j a CUDA graph that runs step j on it while two forked branches
    upload step j+1's inputs into the next set and read step j-1's outputs
    back from the previous one.  One graph launch per step, each moving one
    step's inputs up and one step's outputs down; after launching step j the
    host waits for step j-1 and checks the error word and a slot of step j-2;
    value = steps / wall time.  The same step run serially (upload, calls,
    read-back) and waited for is reported as `sync_ms_per_step`."""
    k = built.keep
    w, lay = k["w"], k["lay"]
    dev = k["qsl"].device
    names = ["qsl", "pos", "table", "rs", "rl", "nr", "key", "val"]
    host_src = {"qsl": w.qsl, "pos": w.positions, "table": lay.table, "rs": lay.range_start,
                "rl": lay.range_len, "nr": lay.num_ranges, "key": k["key"].cpu(),
                "val": k["val"].cpu()}
    # one pinned staging buffer, each input at a 256-byte offset, then 256
    # zero bytes that land on the set's error word: the upload of a step's
    # inputs also clears its error word, with no reset of its own in the graph
    offs, total = {}, 0
    for n in names:
        offs[n] = total
        total += -(-k[n].numel() * k[n].element_size() // 256) * 256
    h_stage = torch.zeros(total + 256, dtype=torch.uint8).pin_memory()
    for n in names:
        nbytes = k[n].numel() * k[n].element_size()
        src = host_src[n]
        src = torch.from_numpy(np.ascontiguousarray(src)) if isinstance(src, np.ndarray) else src
        h_stage[offs[n]:offs[n] + nbytes].copy_(src.contiguous().view(-1).view(torch.uint8))
    h_alias = device_alias(torch, h_stage, dev) if upload == "sm" else None
    T, B, n_max = w.block_size, w.num_blocks, w.max_num_tokens
    n_slot = k["slot_p"].numel()
    out_bytes = 256 + 2 * n_slot * 8  # error word (256-byte slot), both slot mappings
    exp_p = k["slot_p"].cpu().numpy()
    exp_r = k["slot_r"].cpu().numpy()
    probe = int(np.argmax(exp_p >= 0))

    class Set:
        """One set of device buffers, its read-back buffer and prepared calls."""

        def __init__(self):
            # [inputs | error word | slot_p | slot_r]: the upload covers the
            # inputs and the error word, the read-back the error word and slots
            buf = torch.zeros(total + out_bytes, dtype=torch.uint8, device=dev)
            self.d_in, self.d_out = buf[:total + 256], buf[total:]
            self.d_in32 = self.d_in.view(torch.int32)
            d = {n: buf[offs[n]:offs[n] + k[n].numel() * k[n].element_size()]
                 .view(k[n].dtype).view(k[n].shape) for n in names}
            self.h_out = torch.zeros(out_bytes, dtype=torch.uint8).pin_memory()
            self.h_out_alias = (device_alias(torch, self.h_out, dev) if download == "sm"
                                else None)
            self.d_out32 = self.d_out.view(torch.int32)
            h = self.h_out.numpy()
            self.h_err = h[:4].view(np.int32)
            self.h_slot_p = h[256:256 + n_slot * 8].view(np.int64)
            self.h_slot_r = h[256 + n_slot * 8:256 + 2 * n_slot * 8].view(np.int64)
            self.err = self.d_out[:4].view(torch.int32)
            slot_p = self.d_out[256:256 + n_slot * 8].view(torch.int64)
            slot_r = self.d_out[256 + n_slot * 8:256 + 2 * n_slot * 8].view(torch.int64)
            # validated once; the graphs replay them with the cached pointers
            self.calls = [
                kv.kv_slot_mapping_paged(d["qsl"], d["pos"], d["table"], T, B,
                                         max_num_tokens=n_max, slot_mapping=slot_p,
                                         err=self.err, prepare=True),
                kv.kv_slot_mapping_range(d["qsl"], d["pos"], d["rs"], d["rl"], d["nr"], T, B,
                                         max_num_tokens=n_max, slot_mapping=slot_r,
                                         err=self.err, prepare=True),
                kv.kv_cache_write(d["key"], d["val"], k["kc"], k["vc"], slot_p, err=self.err,
                                  prepare=True),
            ]
            self.done = torch.cuda.Event()

        def upload(self):
            if h_alias is not None:
                # the SMs read the pinned inputs over the chip-to-chip link
                torch.bitwise_or(h_alias, 0, out=self.d_in32)
            else:
                self.d_in.copy_(h_stage, non_blocking=True)

        def compute(self):
            paged, rng, write = self.calls
            forked(torch, range_stream, [paged, write], [rng])()

        def download(self):
            if self.h_out_alias is not None:
                # the SMs store the outputs into the pinned buffer's device mapping
                torch.bitwise_or(self.d_out32, 0, out=self.h_out_alias)
            else:
                self.h_out.copy_(self.d_out, non_blocking=True)

        def check(self):
            if int(self.h_err[0]) != 0:
                raise RuntimeError("end-to-end step reported data errors")
            if int(self.h_slot_p[probe]) != int(exp_p[probe]):
                raise RuntimeError("end-to-end step read back a wrong slot")

    sets = [Set(), Set(), Set()]
    up_stream = torch.cuda.Stream(device=dev)
    down_stream = torch.cuda.Stream(device=dev)
    range_stream = torch.cuda.Stream(device=dev)

    def pipelined(j):
        """Step j on set j; step j+1's inputs up into set j+1, step j-1's
        outputs back from set j-1 (sets modulo 3), on two side branches."""
        cur = torch.cuda.current_stream()
        up_stream.wait_stream(cur)
        down_stream.wait_stream(cur)
        with torch.cuda.stream(up_stream):
            sets[(j + 1) % 3].upload()
        with torch.cuda.stream(down_stream):
            sets[(j + 2) % 3].download()
        sets[j % 3].compute()
        cur.wait_stream(up_stream)
        cur.wait_stream(down_stream)

    def capture(fn):
        for st in sets:
            st.upload()
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize()
        return g

    graphs = [capture(lambda j=j: pipelined(j)) for j in range(3)]
    serial = capture(lambda: (sets[0].upload(), sets[0].compute(), sets[0].download()))
    step_no = [0]

    def run(n):
        """n more steps; returns after all of them have been checked."""
        first = step_no[0]
        for j in range(first, first + n + 2):  # two more launches read the last steps back
            graphs[j % 3].replay()
            sets[j % 3].done.record()
            if j > first:
                sets[(j - 1) % 3].done.synchronize()
                if j - 2 >= first:
                    sets[(j - 2) % 3].check()
        step_no[0] = first + n + 2

    for st in sets:
        st.upload()
    run(6)  # warm-up
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    wall = time.perf_counter() - t0
    n_steps = steps + 2  # the two extra launches each did a whole step's work too

    # every step on its own, serially: upload, calls, read-back, waited for
    # (L2 flushed before)
    times = []
    for s in range(min(steps, 200)):
        flush_l2(flush_buf)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        serial.replay()
        sets[0].done.record()
        sets[0].done.synchronize()
        sets[0].check()
        times.append(time.perf_counter() - t1)
    # what came back is the device path's answer on the same inputs
    for st in sets:
        if (int(st.h_err[0]) != 0 or not np.array_equal(st.h_slot_p, exp_p)
                or not np.array_equal(st.h_slot_r, exp_r)):
            raise RuntimeError("end-to-end read-back differs from the device-resident step")
    ms = wall / n_steps * 1e3
    del graphs, serial, sets
    return {"value": round(built.tokens / (ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(total + 256), "d2h_bytes_per_step": int(out_bytes),
            "upload": ("an elementwise kernel reading the pinned buffer" if h_alias is not None
                       else "the copy engine"),
            "ms_per_step": round(ms, 4), "steps": n_steps,
            "sync_ms_per_step": round(statistics.median(times) * 1e3, 4),
            "note": "wall time over all steps: each step copies one step's packed inputs "
                    "(positions, query_start_loc, block table, range descriptors, new K/V "
                    "rows) from pinned host memory and reads one step's slot mappings and "
                    "error word back to pinned host memory; three buffer sets, each with a "
                    "CUDA graph that runs its step while forked branches upload the next "
                    "step's inputs and read the previous step's outputs back; the host checks "
                    "every step's error word and a slot two steps behind; steps run back to "
                    "back with no L2 flush (each step's inputs arrive fresh by its upload, "
                    "through L2), so a step can be a little faster than the flushed "
                    "device-resident one; sync_ms_per_step: median of one step run serially "
                    "(upload, calls, read-back) and waited for, L2 flushed before it"}


# --------------------------------------------------------------------------
# main
# --------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="decode", choices=list(BUILDERS))
    ap.add_argument("--small", action="store_true",
                    help="shrink the workload (profiling captures); not a bench line")
    ap.add_argument("--no-detail", action="store_true", help="skip the other workloads")
    ap.add_argument("--reqs", type=int, default=None,
                    help="--workload slotmap: requests of 131072 positions (default 8)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--detail-reps", type=int, default=10)
    args = ap.parse_args()
    args.steps = max(1, args.steps)
    args.warmup = max(3, args.warmup)

    from paged_kv_cache_39_gb300 import dist as kdist
    if args.impl == "reference":
        run_reference(args, kdist.from_env())
        return

    import torch
    import paged_kv_cache_39_gb300 as kv
    from paged_kv_cache_39_gb300 import workloads as wl

    rk = kdist.init("nccl")
    dev = torch.device("cuda", rk.local_rank)
    torch.cuda.set_device(dev)
    kv.load()
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = load_peaks()
    flush_buf = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    if args.workload != "decode":
        return profile_run(torch, kv, wl, dev, args, rk, flush_buf, stream, peak, kdist)

    built = build_decode(torch, kv, wl, dev, small=args.small)
    for _ in range(args.warmup):
        flush_l2(flush_buf)
        for l in built.launches:
            l.fn()
    torch.cuda.synchronize()
    if int(built.keep["err"].item()) != 0:
        raise SystemExit(f"kernels reported data errors: {int(built.keep['err'].item())}")
    side = torch.cuda.Stream(device=dev)
    step = GraphStep(torch, [step_fn(torch, built, side)])

    with ClockSampler() as clocks:
        kdist.barrier(dev)
        torch.cuda.synchronize()
        step_ms = step.times_ms(args.steps, flush_buf)
        torch.cuda.synchronize()
        kdist.barrier(dev)
    if int(built.keep["err"].item()) != 0:
        raise SystemExit(f"kernels reported data errors: {int(built.keep['err'].item())}")
    ms_per_step = sum(step_ms) / len(step_ms)
    ms_max = kdist.max_over_ranks(ms_per_step, dev)
    value = built.tokens * rk.world_size / (ms_max * 1e-3)
    del step

    # the step's kernels one by one (L2 flushed before each) for the roofline
    reps = min(max(args.steps, 100), 1000)
    per = time_each(torch, built, reps, flush_buf, stream)
    kernels = kernel_report(built, per, peak)
    dom_i = max(range(len(built.launches)), key=lambda i: sum(per[i]))
    dom = built.launches[dom_i]
    dom_avg_ms = sum(per[dom_i]) / len(per[dom_i])
    achieved = dom.alg_bytes / (dom_avg_ms * 1e-3) / 1e9
    floor_us = launch_floor_us(torch, dev, min(max(args.steps, 100), 1000), flush_buf)
    roofline = {"bound": "hbm", "kernel": dom.kernel, "achieved": round(achieved, 1),
                "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs (copy, read+write)",
                "unit": "GB/s", "frac": round(achieved / peak, 6),
                "traffic": profiled_traffic(dom.kernel, "decode"),
                "alg_bytes_per_launch": int(dom.alg_bytes),
                "avg_launch_us": round(dom_avg_ms * 1e3, 2),
                "launch_floor_us": floor_us,
                "frac_of_launch_floor": round(floor_us / (dom_avg_ms * 1e3), 4),
                "regime": "latency: 256 tokens move a few KB to 2 MB per kernel, so every "
                          "kernel of the step is a chain of dependent DRAM round trips on top "
                          "of the launch; launch_floor_us is one replay of a graph holding a "
                          "single one-element kernel, timed the same way, and "
                          "frac_of_launch_floor that floor over this kernel's time",
                "timing": f"each call alone, L2 flushed before it, mean of {reps} launches"}
    same_run_copy = copy_ceiling(torch, dev, flush_buf, reps=5)["torch_copy_GBps_median"]

    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": rk.world_size, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_max, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int64", "payload": "bf16 bits copied",
            "data": "synthetic",
            "config": {"workload": built.desc + (" [small]" if args.small else ""),
                       "l2": "flushed between timed steps outside the events (256 MiB written, then "
                             "another 256 MiB read)",
                       "timing": "the step's three calls captured once in a CUDA graph (paged "
                                 "map -> write; the range map on a second branch), one replay "
                                 "per step, CUDA events around each replay",
                       "parallelism": "replicas" if rk.world_size > 1 else "single GPU",
                       "per_gpu_tokens_per_step": built.tokens},
            "kernels": kernels, "roofline": roofline,
            "gpu_launches": args.steps * len(built.launches),
            "clocks": clocks.summary()}
    line["paged_vs_range"] = paged_vs_range(torch, kv, built, min(max(args.steps, 500), 2000),
                                            reps, flush_buf, stream)
    gather = gather_long(torch, kv, wl, dev, max(args.detail_reps, 5), flush_buf, stream,
                         (peak, peak_kind), same_run_copy, small=args.small)
    line["gather_GBps"] = gather["GBps"]
    line["gather_roofline"] = gather["roofline"]  # the metric's second half
    line["gather"] = gather
    line["decode_step_with_gather"] = decode_step_with_gather(
        torch, built, min(args.steps, 500), flush_buf, stream, (peak, peak_kind), args)
    e2e = e2e_step(torch, kv, built, min(max(args.steps, 500), 5000), flush_buf, stream)
    if rk.world_size > 1:
        # whole job, like `value`: every rank's tokens over the slowest rank's step
        kdist.barrier(dev)
        e2e_ms = kdist.max_over_ranks(e2e["ms_per_step"], dev)
        e2e["per_gpu_value"] = e2e["value"]
        e2e["ms_per_step"] = round(e2e_ms, 4)
        e2e["value"] = round(built.tokens * rk.world_size / (e2e_ms * 1e-3), 1)
    line["e2e"] = e2e

    if rk.is_main and rk.world_size == 1:
        if args.cpu_seconds > 0:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        if not args.no_detail:
            built = None
            torch.cuda.empty_cache()
            line["configs"] = detail(torch, kv, wl, dev, args, flush_buf, stream, peak)
            if args.cpu_seconds > 0:
                line["oracle_rows"] = oracle_rows()
    if rk.is_main:
        print(json.dumps(line), flush=True)
    kdist.finalize()


def profile_run(torch, kv, wl, dev, args, rk, flush_buf, stream, peak, kdist):
    """`--workload X` (X not the decode step): the workload's launches in
    order, per-launch events, L2 flushed between steps.  For profiler captures
    and kernel A/B runs; the line is marked as not a bench line."""
    kw = {"reqs": args.reqs} if args.workload == "slotmap" and args.reqs else {}
    built = BUILDERS[args.workload](torch, kv, wl, dev, small=args.small, **kw)
    for _ in range(args.warmup):
        flush_l2(flush_buf)
        for l in built.launches:
            l.fn()
    torch.cuda.synchronize()
    if int(built.keep["err"].item()) != 0:
        raise SystemExit(f"kernels reported data errors: {int(built.keep['err'].item())}")
    step_ms, _ = time_steps(torch, built, args.steps, flush_buf, stream)
    per = time_each(torch, built, args.steps, flush_buf, stream)
    line = {"not_a_bench_line": f"--workload {args.workload}", "workload": built.desc +
            (" [small]" if args.small else ""), "steps": args.steps,
            "ms_per_step": round(sum(step_ms) / len(step_ms), 4),
            "kernels": kernel_report(built, per, peak),
            "timing": "ms_per_step: the launches back to back, L2 flushed between steps; "
                      "kernels: each launch alone, L2 flushed before it, CUDA events"}
    if rk.is_main:
        print(json.dumps(line), flush=True)
    kdist.finalize()


def copy_ceiling(torch, dev, flush_buf, reps=10):
    """Device-to-device copy of 1 Gi bf16 elements (read + write bytes), the
    same copy the measured peak is taken from, timed in this run."""
    src = torch.empty(1 << 30, dtype=torch.bfloat16, device=dev).fill_(1)
    dst = torch.empty_like(src)
    dst.copy_(src)
    times = []
    for _ in range(reps):
        flush_l2(flush_buf)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src)
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    best = min(times)
    del src, dst
    torch.cuda.empty_cache()
    return {"torch_copy_GBps_best": round(2 * (2 << 30) / (best * 1e-3) / 1e9, 1),
            "torch_copy_GBps_median": round(2 * (2 << 30) / (statistics.median(times) * 1e-3) / 1e9,
                                            1),
            "bytes": 2 * (2 << 30)}


def detail(torch, kv, wl, dev, args, flush_buf, stream, peak):
    out = {"copy_ceiling": copy_ceiling(torch, dev, flush_buf)}
    for name in ("decode", "mixed", "long", "hybrid"):
        b = (build_decode(torch, kv, wl, dev, extras=True) if name == "decode"
             else BUILDERS[name](torch, kv, wl, dev))
        for _ in range(3):
            for l in b.launches:
                l.fn()
        torch.cuda.synchronize()
        per = time_each(torch, b, args.detail_reps, flush_buf, stream)
        rep = kernel_report(b, per, peak)
        entry = {"workload": b.desc, "kernels": rep, "errors": int(b.keep["err"].item()),
                 "l2": "flushed before every launch", "reps": args.detail_reps}
        if name == "mixed":
            tw = rep["cache_write"]["us"]
            entry["write_slotmap_tokens_per_s"] = {
                "paged": round(b.tokens / ((rep["slot_mapping_paged"]["us"] + tw) * 1e-6), 1),
                "range": round(b.tokens / ((rep["slot_mapping_range"]["us"] + tw) * 1e-6), 1),
                "paged_fused": round(b.tokens / (rep["slot_mapping_paged_write"]["us"] * 1e-6),
                                     1),
                "range_fused": round(b.tokens / (rep["slot_mapping_range_write"]["us"] * 1e-6),
                                     1)}
        out[name] = entry
        del b
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    main()
