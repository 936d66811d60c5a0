"""GPU parity of the fused slot-mapping + KV write calls.

kv_slot_mapping_paged_write (kv_slot_mapping_range_write) must give exactly
what the oracle's paged (range) slot map followed by the oracle's KV write
gives: the same slot mapping with its PAD tail, the same cache bytes and the
same error word ("Blocktabelle", Datenfluss and Verantwortung;
"Range-addressed KV cache blocks ...", The Innovation).  Two tokens given the
same slot (a table that repeats a block) race for it in either form, one
16-byte store at a time; there each 16-byte piece of the row must be one of
theirs, and every other row is compared exactly."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_39_gb300 as kv
from paged_kv_cache_39_gb300 import workloads as wl
from gpu_helpers import (bits, check_write, cuda, dev, err_word, filled_cache, free_bytes,
                         random_slot_case)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    torch.cuda.set_device(dev())
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def random_ranges(rng, rows, B):
    rstride = int(rng.choice([1, 4, 40, 256]))
    rs = rng.integers(-2, B + 2, size=(rows, rstride)).astype(np.int32)
    rl = rng.integers(-1, 12, size=(rows, rstride)).astype(np.int32)
    if rng.random() < 0.5:
        rl = np.maximum(rl, 1)
    nr = rng.integers(0, rstride + 1, size=rows).astype(np.int32)
    if rng.random() < 0.3:
        nr[rng.integers(0, rows)] = rstride + 1
    return rs, rl, nr


ROW_SHAPES = [(1, 8), (8, 64), (8, 128), (16, 128), (2, 72)]  # 16 B .. 4 KiB rows


@pytest.mark.parametrize("kind", ["paged", "range"])
@pytest.mark.parametrize("seed", range(30))
def test_fused_adversarial(seed, kind):
    rng = np.random.default_rng(7000 + seed)
    T, R, q, N, n_max, stride, B, table, pos = random_slot_case(rng)
    H, D = ROW_SHAPES[seed % len(ROW_SHAPES)]
    L = 1 + seed % 3
    if kind == "paged":
        exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, n_max, T, B)
    else:
        rs, rl, nr = random_ranges(rng, max(R, 1), B)
        exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, n_max, T, B)
    key = wl.bf16_normal((L, N, H, D), 40 + seed)
    val = wl.bf16_normal((L, N, H, D), 80 + seed)
    kc = wl.bf16_normal((L, B, T, H, D), 120 + seed)
    vc = wl.bf16_normal((L, B, T, H, D), 160 + seed)
    kb, vb = bits(key), bits(val)
    # slots that several tokens share race; the oracle writes the others
    s_tok = exp_s[:N]
    valid = s_tok[s_tok >= 0]
    uniq, counts = np.unique(valid, return_counts=True)
    shared = uniq[counts > 1]
    s_unique = np.where(np.isin(s_tok, shared), -1, s_tok)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_we = oracle.cache_write(kb, vb, ek, ev, s_unique, B, T)
    assert exp_we == 0  # the slot map never yields a slot the write refuses

    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    slot = torch.full((n_max,), 12345, dtype=torch.int64, device=dev())
    e = err_word()
    if kind == "paged":
        kv.kv_slot_mapping_paged_write(cuda(q), cuda(pos), cuda(table), T, B, key.to(dev()),
                                       val.to(dev()), kc_d, vc_d, max_num_tokens=n_max,
                                       slot_mapping=slot, num_tokens=N, err=e)
    else:
        kv.kv_slot_mapping_range_write(cuda(q), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B,
                                       key.to(dev()), val.to(dev()), kc_d, vc_d,
                                       max_num_tokens=n_max, slot_mapping=slot, num_tokens=N,
                                       err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(slot.cpu().numpy(), exp_s)
    gk, gv = bits(kc_d), bits(vc_d)
    for s in shared:
        b, o = divmod(int(s), T)
        toks = np.nonzero(s_tok == s)[0]
        for l in range(L):
            for got, src in ((gk[l, b, o], kb), (gv[l, b, o], vb)):
                # stores race per 16-byte vector: each piece is one token's
                pieces = got.reshape(-1, 8)
                cands = np.stack([src[l, t].reshape(-1, 8) for t in toks])
                assert (cands == pieces[None]).all(axis=2).any(axis=0).all()
            ek[l, b, o], ev[l, b, o] = gk[l, b, o], gv[l, b, o]
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


def _fused(kind, w, lay, key, val, kc, vc, e):
    qsl, pos = cuda(w.qsl), cuda(w.positions)
    if kind == "paged":
        return kv.kv_slot_mapping_paged_write(qsl, pos, cuda(lay.table), w.block_size,
                                              w.num_blocks, key, val, kc, vc,
                                              max_num_tokens=w.max_num_tokens, err=e)
    return kv.kv_slot_mapping_range_write(qsl, pos, cuda(lay.range_start), cuda(lay.range_len),
                                          cuda(lay.num_ranges), w.block_size, w.num_blocks,
                                          key, val, kc, vc, max_num_tokens=w.max_num_tokens,
                                          err=e)


@pytest.mark.parametrize("kind", ["paged", "range"])
@pytest.mark.parametrize("name", ["tiny", "decode", "mixed"])
def test_fused_full_configs(name, kind):
    if name == "mixed":
        need = 2 * 32 * 49152 * 16 * 2048 + (8 << 30)
        w = (wl.mixed() if free_bytes() >= need
             else wl.mixed(num_blocks=32768, decode_ctx_max=2048))
    else:
        w = wl.CONFIGS[name]()
    lay = w.layouts["G"]
    T, B, L, H, D, E = (w.block_size, w.num_blocks, w.num_layers, w.num_kv_heads, w.head_dim,
                        w.row_elems)
    exp, exp_e = oracle.slot_mapping_paged(w.qsl, w.positions, lay.table, w.num_tokens,
                                           w.max_num_tokens, T, B)
    key = wl.bf16_normal((L, w.num_tokens, H, D), 501, dev())
    val = wl.bf16_normal((L, w.num_tokens, H, D), 502, dev())
    kc, vc = filled_cache((L, B, T, H, D)), filled_cache((L, B, T, H, D))
    e = err_word()
    slot = _fused(kind, w, lay, key, val, kc, vc, e)
    assert int(e.item()) == exp_e == 0
    assert np.array_equal(slot.cpu().numpy(), exp)
    assert check_write(key, val, kc, vc, exp, L, w.num_tokens, B, T, E,
                       np.random.default_rng(5)) == 0


@pytest.mark.parametrize("kind", ["paged", "range"])
@pytest.mark.parametrize("R", [2047, 2048, 6000])
def test_fused_many_requests(R, kind):
    """Up to 2047 requests the CTA stages query_start_loc in shared memory;
    past that each warp searches it in global memory."""
    rng = np.random.default_rng(7500 + R)
    T, H, D, stride = 16, 1, 64, 4
    lens = rng.integers(0, 3, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    B = R * stride + 1
    table = rng.permutation(np.arange(1, B)).astype(np.int32)[:R * stride].reshape(R, stride)
    # distinct positions within a request, so no two tokens share a slot
    pos = np.concatenate([rng.choice(stride * T + 8, size=n, replace=False)
                          for n in lens]).astype(np.int64)
    rs, rl = table[:, :1].copy(), np.ones((R, 1), np.int32)  # one single-block range per row
    nr = np.ones(R, np.int32)
    if kind == "paged":
        exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, N + 5, T, B)
    else:
        exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N + 5, T, B)
    key = wl.bf16_normal((1, N, H, D), 7600 + R)
    val = wl.bf16_normal((1, N, H, D), 7700 + R)
    kc = torch.zeros((1, B, T, H, D), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    assert oracle.cache_write(bits(key), bits(val), ek, ev, exp_s[:N], B, T) == 0
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    if kind == "paged":
        s = kv.kv_slot_mapping_paged_write(cuda(q), cuda(pos), cuda(table), T, B, key.to(dev()),
                                           val.to(dev()), kc_d, vc_d, max_num_tokens=N + 5,
                                           err=e)
    else:
        s = kv.kv_slot_mapping_range_write(cuda(q), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T,
                                           B, key.to(dev()), val.to(dev()), kc_d, vc_d,
                                           max_num_tokens=N + 5, err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(s.cpu().numpy(), exp_s)
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)


@pytest.mark.parametrize("fused", [False, True])
def test_row_check_covers_rows_past_the_grid(fused):
    """A batch of 1000 descriptor rows and only 16 tokens runs on one CTA
    (256 threads, or 2 CTAs for the fused call): the grid-wide row check
    must still loop over every row and flag the malformed ones."""
    rng = np.random.default_rng(7900)
    R, T, B, S = 1000, 16, 5000, 4
    rs = rng.permutation(np.arange(1, B))[:R * S].reshape(R, S).astype(np.int32)  # distinct
    rl = np.ones((R, S), np.int32)
    nr = rng.integers(1, S + 1, size=R).astype(np.int32)
    nr[300] = S + 2                   # count above the stride
    rl[999, 0] = 0                    # zero-length first range
    nr[999] = max(nr[999], 1)
    lens = np.zeros(R, np.int64)
    lens[[0, 5, 700]] = [6, 6, 4]
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.int64)
    exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N, T, B)
    assert exp_e == kv.ERR_BITS["BAD_RANGE"]
    e = err_word()
    if fused:
        H, D = 1, 8
        key = wl.bf16_normal((1, N, H, D), 7901)
        kc = torch.zeros((1, B, T, H, D), dtype=torch.bfloat16)
        ek, ev = bits(kc).copy(), bits(kc).copy()
        oracle.cache_write(bits(key), bits(key), ek, ev, exp_s, B, T)
        kc_d, vc_d = kc.to(dev()), kc.clone().to(dev())
        s = kv.kv_slot_mapping_range_write(cuda(q), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B,
                                           key.to(dev()), key.to(dev()), kc_d, vc_d, err=e)
        assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)
    else:
        s = kv.kv_slot_mapping_range(cuda(q), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B, err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(s.cpu().numpy(), exp_s)


@pytest.mark.parametrize("call", ["paged", "range", "paged_write"])
def test_qsl_check_covers_entries_past_the_grid(call):
    """query_start_loc decreasing at entry 2500 of 3000, with 16 tokens (one
    or two CTAs): the grid-wide check still reaches it and sets BAD_QSL."""
    R, T, B, S = 3000, 16, 4000, 4
    lens = np.zeros(R, np.int64)
    lens[[1, 2]] = [10, 6]
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q[2500] = q[2501] + 1  # decreasing once
    N = 16
    pos = np.arange(N, dtype=np.int64)
    table = np.arange(1, R * S + 1, dtype=np.int32).reshape(R, S) % (B - 1) + 1
    rs, rl, nr = table[:, :1].copy(), np.ones((R, 1), np.int32), np.ones(R, np.int32)
    _, exp_e = oracle.slot_mapping_paged(q, pos, table, N, N, T, B)
    assert exp_e & kv.ERR_BITS["BAD_QSL"]
    e = err_word()
    if call == "paged":
        kv.kv_slot_mapping_paged(cuda(q), cuda(pos), cuda(table), T, B, err=e)
    elif call == "range":
        _, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N, T, B)
        kv.kv_slot_mapping_range(cuda(q), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B, err=e)
    else:
        key = torch.zeros((1, N, 1, 8), dtype=torch.bfloat16, device=dev())
        kc = torch.zeros((1, B, T, 1, 8), dtype=torch.bfloat16, device=dev())
        kv.kv_slot_mapping_paged_write(cuda(q), cuda(pos), cuda(table), T, B, key, key, kc,
                                       kc.clone(), err=e)
    # slot values are unspecified under a bad qsl; the error word is not
    assert int(e.item()) & kv.ERR_BITS["BAD_QSL"]
    assert int(e.item()) == exp_e
