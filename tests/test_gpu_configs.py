"""GPU parity at the workloads' full sizes, in the launch configurations the
benchmark times.

Slot maps and expanded tables are compared whole with the oracle.  For the
KV copies, the oracle computes the destination (write) or source (gather)
row of every output row; every row is then checked on the device (torch only
moves the bytes being compared) and a random sample of rows is checked on
the host against cache rows fetched one by one.  Caches that the write does
not address must keep their fill pattern, the null block included.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_39_gb300 as kv
from paged_kv_cache_39_gb300 import workloads as wl
from gpu_helpers import (FILL, SAMPLE, check_write, check_write_vs_before, cuda, dev,
                         device_rows_equal, err_word, filled_cache, free_bytes, rows_view,
                         sample_host_check)

pytestmark = pytest.mark.gpu

@pytest.fixture(autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    torch.cuda.set_device(dev())
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def slot_maps_match(w, lay, check_range=True):
    T, B = w.block_size, w.num_blocks
    exp, exp_e = oracle.slot_mapping_paged(w.qsl, w.positions, lay.table, w.num_tokens,
                                           w.max_num_tokens, T, B)
    qsl, pos = cuda(w.qsl), cuda(w.positions)
    e = err_word()
    sp = kv.kv_slot_mapping_paged(qsl, pos, cuda(lay.table), T, B,
                                  max_num_tokens=w.max_num_tokens, err=e)
    assert int(e.item()) == exp_e == 0
    assert np.array_equal(sp.cpu().numpy(), exp)
    if check_range and lay.range_start is not None:
        exp_r, exp_re = oracle.slot_mapping_range(w.qsl, w.positions, lay.range_start,
                                                  lay.range_len, lay.num_ranges, w.num_tokens,
                                                  w.max_num_tokens, T, B)
        e = err_word()
        sr = kv.kv_slot_mapping_range(qsl, pos, cuda(lay.range_start), cuda(lay.range_len),
                                      cuda(lay.num_ranges), T, B,
                                      max_num_tokens=w.max_num_tokens, err=e)
        assert int(e.item()) == exp_re == 0
        assert np.array_equal(sr.cpu().numpy(), exp_r)
        assert np.array_equal(exp_r, exp)  # range == paged slot for slot
    return sp, exp


def test_decode_full():
    """The decode batch: slot maps, the write into caches of random contents
    (every other row unchanged), then the gather of every request's whole
    context (597k rows, all distinct), checked row by row against the
    oracle's source rows."""
    w = wl.decode()
    lay = w.layouts["G"]
    T, B, H, D, E = w.block_size, w.num_blocks, w.num_kv_heads, w.head_dim, w.row_elems
    sp, exp = slot_maps_match(w, lay)
    key = wl.bf16_normal((1, w.num_tokens, H, D), 101, dev())
    val = wl.bf16_normal((1, w.num_tokens, H, D), 102, dev())
    kc = wl.bf16_normal((1, B, T, H, D), 103, dev())
    vc = wl.bf16_normal((1, B, T, H, D), 104, dev())
    kc0, vc0 = kc.clone(), vc.clone()
    e = err_word()
    kv.kv_cache_write(key, val, kc, vc, sp, err=e)
    exp_e = check_write_vs_before(key, val, kc, vc, kc0, vc0, exp, 1, w.num_tokens, B, T, E,
                                  np.random.default_rng(1))
    assert int(e.item()) == exp_e == 0
    del kc0, vc0
    # the decode batch's contexts read back through the table: the new token
    # is the last row of each request's span
    rows = int(w.gather_end.sum())
    src, exp_ge = oracle.gather_rows(0, B, T, lay.table, w.gather_start, w.gather_end, rows)
    assert (src >= 0).all() and len(np.unique(src)) == rows
    for bulk in (False, True):
        e = err_word()
        k_out, v_out = kv.kv_cache_gather(kc, vc, cuda(lay.table), cuda(w.gather_start),
                                          cuda(w.gather_end), out_rows=rows, err=e, bulk=bulk)
        assert int(e.item()) == exp_ge == 0
        assert device_rows_equal(k_out, kc, src, E) and device_rows_equal(v_out, vc, src, E)
        last = np.cumsum(w.gather_end.astype(np.int64)) - 1
        sel = torch.from_numpy(last).to(dev())
        assert torch.equal(rows_view(k_out, E)[sel], rows_view(key[0], E))
        assert torch.equal(rows_view(v_out, E)[sel], rows_view(val[0], E))
        sample = np.sort(np.random.default_rng(11).choice(rows, size=SAMPLE, replace=False))
        kflat = rows_view(kc, E)
        sample_host_check(k_out, lambda n: kflat[n].cpu().numpy().view(np.uint16), src, E,
                          sample)
        del k_out, v_out


def test_mixed_full():
    w = mixed_workload()
    lay = w.layouts["G"]
    T, B, L, H, D, E = (w.block_size, w.num_blocks, w.num_layers, w.num_kv_heads, w.head_dim,
                        w.row_elems)
    sp, exp = slot_maps_match(w, lay)
    key = wl.bf16_normal((L, w.num_tokens, H, D), 201, dev())
    val = wl.bf16_normal((L, w.num_tokens, H, D), 202, dev())
    kc, vc = filled_cache((L, B, T, H, D)), filled_cache((L, B, T, H, D))
    e = err_word()
    kv.kv_cache_write(key, val, kc, vc, sp, err=e)
    exp_e = check_write(key, val, kc, vc, exp, L, w.num_tokens, B, T, E, np.random.default_rng(2))
    assert int(e.item()) == exp_e == 0
    # null block 0 of every layer is untouched
    assert (kc.view(torch.int16)[:, 0] == FILL).all() and (vc.view(torch.int16)[:, 0] == FILL).all()


def mixed_workload():
    if free_bytes() >= 2 * 32 * 49152 * 16 * 2048 + (12 << 30):
        return wl.mixed()
    print("mixed: reduced to 32768 blocks / decode ctx U{512..2048} for free memory")
    return wl.mixed(num_blocks=32768, decode_ctx_max=2048)


def test_mixed_gather_layers():
    """Gathers from the 32-layer mixed caches (51.5 GB each, random contents)
    at layers 0, 17 and 31, where layer * num_blocks * block_size * row_bytes
    puts byte offsets far past 2^32: the table gather, its bulk-copy form and
    the range-addressed gather, every row against the oracle's source rows.
    The batch is written first, so the gathered spans also hold the new
    tokens' rows (gather after write returns what was written).  Then the
    copy-on-write kernels on the same caches, every layer."""
    w = mixed_workload()
    lay = w.layouts["G"]
    T, B, L, H, D, E = (w.block_size, w.num_blocks, w.num_layers, w.num_kv_heads, w.head_dim,
                        w.row_elems)
    N = w.num_tokens
    kc = wl.bf16_normal((L, B, T, H, D), 501, dev())
    vc = wl.bf16_normal((L, B, T, H, D), 502, dev())
    key = wl.bf16_normal((L, N, H, D), 503, dev())
    val = wl.bf16_normal((L, N, H, D), 504, dev())
    exp_s, _ = oracle.slot_mapping_paged(w.qsl, w.positions, lay.table, N, N, T, B)
    e = err_word()
    sp = kv.kv_slot_mapping_paged(cuda(w.qsl), cuda(w.positions), cuda(lay.table), T, B, err=e)
    kv.kv_cache_write(key, val, kc, vc, sp, err=e)
    assert int(e.item()) == 0
    dest, _ = oracle.write_rows(exp_s, N, L, B, T)  # absolute cache row of (layer, token)
    rows = int((w.gather_end.astype(np.int64) - w.gather_start).sum())
    table, g0, g1 = cuda(lay.table), cuda(w.gather_start), cuda(w.gather_end)
    rs, rl, nr = cuda(lay.range_start), cuda(lay.range_len), cuda(lay.num_ranges)
    kflat = rows_view(kc, E)
    rng = np.random.default_rng(12)
    for layer in (0, 17, 31):
        src, exp_ge = oracle.gather_rows(layer, B, T, lay.table, w.gather_start, w.gather_end,
                                         rows)
        assert exp_ge == 0 and (src >= 0).all()
        assert src.min() >= layer * B * T and src.max() < (layer + 1) * B * T
        # output rows whose source is a row the write just filled, and its token
        order = np.argsort(dest[layer])
        at = np.searchsorted(dest[layer][order], src)
        hit = (at < N) & (dest[layer][order][np.minimum(at, N - 1)] == src)
        assert int(hit.sum()) == N  # every new token is read back exactly once
        o_new = torch.from_numpy(np.nonzero(hit)[0]).to(dev())
        t_new = torch.from_numpy(order[at[hit]]).to(dev())
        outs = {}
        for form in ("table", "bulk", "range"):
            e = err_word()
            if form == "range":
                ko, vo = kv.kv_cache_gather_range(kc, vc, rs, rl, nr, g0, g1, layer=layer,
                                                  out_rows=rows, err=e)
            else:
                ko, vo = kv.kv_cache_gather(kc, vc, table, g0, g1, layer=layer, out_rows=rows,
                                            err=e, bulk=form == "bulk")
            assert int(e.item()) == 0, (layer, form)
            assert device_rows_equal(ko, kc, src, E) and device_rows_equal(vo, vc, src, E), \
                (layer, form)
            assert torch.equal(rows_view(ko, E)[o_new], rows_view(key[layer], E)[t_new])
            assert torch.equal(rows_view(vo, E)[o_new], rows_view(val[layer], E)[t_new])
            outs[form] = (ko, vo)
        sample = np.sort(rng.choice(rows, size=SAMPLE, replace=False))
        sample_host_check(outs["table"][0], lambda n: kflat[n].cpu().numpy().view(np.uint16),
                          src, E, sample)
        del outs
    # copy-on-write on the same caches: 1024 forks by the vector kernel and
    # 1024 by the bulk-copy kernel, disjoint blocks, every layer (offsets past
    # 2^32 bytes); each destination block of every layer must equal its
    # source's earlier contents, and untouched blocks keep theirs
    perm = rng.permutation(np.arange(1, B, dtype=np.int32))
    untouched = torch.from_numpy(perm[4096:4096 + 64].astype(np.int64)).to(dev())
    k_keep, v_keep = kc[:, untouched].clone(), vc[:, untouched].clone()
    for n, bulk in ((0, False), (1, True)):
        src_b = perm[2048 * n:2048 * n + 1024]
        dst_b = perm[2048 * n + 1024:2048 * n + 2048]
        s_idx = torch.from_numpy(src_b.astype(np.int64)).to(dev())
        d_idx = torch.from_numpy(dst_b.astype(np.int64)).to(dev())
        k_src, v_src = kc[:, s_idx].clone(), vc[:, s_idx].clone()
        e = err_word()
        kv.kv_copy_blocks(kc, vc, cuda(src_b), cuda(dst_b), err=e, bulk=bulk)
        assert int(e.item()) == 0
        assert torch.equal(kc[:, d_idx].view(torch.int16), k_src.view(torch.int16)), bulk
        assert torch.equal(vc[:, d_idx].view(torch.int16), v_src.view(torch.int16)), bulk
        assert torch.equal(kc[:, s_idx].view(torch.int16), k_src.view(torch.int16))
        del k_src, v_src
    assert torch.equal(kc[:, untouched].view(torch.int16), k_keep.view(torch.int16))
    assert torch.equal(vc[:, untouched].view(torch.int16), v_keep.view(torch.int16))


@pytest.mark.parametrize("layout", ["P", "G"])
def test_long_context_full(layout):
    w = wl.long_context()
    lay = w.layouts[layout]
    T, B, H, D, E = w.block_size, w.num_blocks, w.num_kv_heads, w.head_dim, w.row_elems
    slot_maps_match(w, lay)
    kc = wl.bf16_normal((1, B, T, H, D), 301, dev())
    vc = wl.bf16_normal((1, B, T, H, D), 302, dev())
    rows = w.num_tokens
    e = err_word()
    k_out, v_out = kv.kv_cache_gather(kc, vc, cuda(lay.table), cuda(w.gather_start),
                                      cuda(w.gather_end), out_rows=rows, err=e)
    src, exp_e = oracle.gather_rows(0, B, T, lay.table, w.gather_start, w.gather_end, rows)
    assert int(e.item()) == exp_e == 0
    assert device_rows_equal(k_out, kc, src, E) and device_rows_equal(v_out, vc, src, E)
    # the bulk-copy gather gives the same bytes
    kb, vb = torch.empty_like(k_out), torch.empty_like(v_out)
    kv.kv_cache_gather(kc, vc, cuda(lay.table), cuda(w.gather_start), cuda(w.gather_end),
                       k_out=kb, v_out=vb, out_rows=rows, err=e, bulk=True)
    assert int(e.item()) == 0
    assert torch.equal(rows_view(kb, E), rows_view(k_out, E))
    assert torch.equal(rows_view(vb, E), rows_view(v_out, E))
    del kb, vb
    rng = np.random.default_rng(3)
    sample = np.sort(rng.choice(rows, size=SAMPLE, replace=False))
    kflat = rows_view(kc, E)
    sample_host_check(k_out, lambda n: kflat[n].cpu().numpy().view(np.uint16), src, E, sample)
    if layout == "G":
        # one packed run per range: the first range of request 0 is one contiguous copy
        s0, ln0 = int(lay.range_start[0, 0]), int(lay.range_len[0, 0])
        assert torch.equal(rows_view(k_out, E)[:ln0 * T], kflat[s0 * T:(s0 + ln0) * T])


def test_hybrid_full():
    h = wl.hybrid()
    H, D, E = h.num_kv_heads, h.head_dim, h.num_kv_heads * h.head_dim
    qsl, pos = cuda(h.qsl), cuda(h.positions)
    rng = np.random.default_rng(4)
    key = wl.bf16_normal((1, h.num_tokens, H, D), 401, dev())
    val = wl.bf16_normal((1, h.num_tokens, H, D), 402, dev())
    for name, g in h.groups.items():
        kbs = g.kernel_block_size
        Bk = g.kernel_num_blocks
        # 32 -> 16 expansion of the manager table
        exp_kt, exp_xe = oracle.expand_kernel_blocks(g.mgr_table, g.mgr_block_size, kbs)
        e = err_word()
        kt = kv.kv_expand_kernel_blocks(cuda(g.mgr_table), g.mgr_block_size, kbs, err=e)
        assert int(e.item()) == exp_xe == 0
        assert np.array_equal(kt.cpu().numpy(), exp_kt)
        # decode slot map over the kernel table, padded rows and tail PAD
        exp_s, exp_se = oracle.slot_mapping_paged(h.qsl, h.positions, exp_kt, h.num_tokens,
                                                  h.max_num_tokens, kbs, Bk)
        e = err_word()
        sp = kv.kv_slot_mapping_paged(qsl, pos, kt, kbs, Bk, max_num_tokens=h.max_num_tokens,
                                      err=e)
        assert int(e.item()) == exp_se == 0
        assert np.array_equal(sp.cpu().numpy(), exp_s)
        assert (exp_s[h.num_tokens:] == -1).all()
        # decode write of one token per real request
        kc = wl.bf16_normal((1, Bk, kbs, H, D), 410 + len(name), dev())
        vc = wl.bf16_normal((1, Bk, kbs, H, D), 420 + len(name), dev())
        dest, exp_we = oracle.write_rows(exp_s[:h.num_tokens], h.num_tokens, 1, Bk, kbs)
        e = err_word()
        kv.kv_cache_write(key, val, kc, vc, sp[:h.num_tokens], err=e)
        assert int(e.item()) == exp_we == 0
        drow = torch.from_numpy(dest[0]).to(dev())
        assert torch.equal(rows_view(kc, E)[drow], rows_view(key, E))
        assert torch.equal(rows_view(vc, E)[drow], rows_view(val, E))
        # gather: 8 calls of 64 requests, then the 128 padding rows (no rows, no error)
        kflat = rows_view(kc, E)
        for c in range(0, h.num_reqs, 64):
            hi = min(h.num_reqs, c + 64) if c < h.num_real_reqs else h.num_reqs
            g0, g1 = g.gather_start[c:hi], g.gather_end[c:hi]
            rows = int((g1.astype(np.int64) - g0).sum())
            e = err_word()
            k_out, v_out = kv.kv_cache_gather(kc, vc, kt[c:hi].contiguous(), cuda(g0), cuda(g1),
                                              out_rows=rows, err=e)
            src, exp_ge = oracle.gather_rows(0, Bk, kbs, exp_kt[c:hi], g0, g1, rows)
            assert int(e.item()) == exp_ge == 0
            if rows:
                assert device_rows_equal(k_out, kc, src, E)
                assert device_rows_equal(v_out, vc, src, E)
                kb, vb = torch.empty_like(k_out), torch.empty_like(v_out)
                kv.kv_cache_gather(kc, vc, kt[c:hi].contiguous(), cuda(g0), cuda(g1), k_out=kb,
                                   v_out=vb, out_rows=rows, err=e, bulk=True)
                assert int(e.item()) == 0
                assert torch.equal(rows_view(kb, E), rows_view(k_out, E))
                assert torch.equal(rows_view(vb, E), rows_view(v_out, E))
                del kb, vb
                sample = np.sort(rng.choice(rows, size=min(256, rows), replace=False))
                sample_host_check(v_out, lambda n: rows_view(vc, E)[n].cpu().numpy().view(np.uint16),
                                  src, E, sample)
                assert (src >= 0).all()  # SWA windows never touch recycled blocks
            if c >= h.num_real_reqs:
                assert rows == 0
                break
        del kc, vc, kt, kflat
        torch.cuda.empty_cache()
