"""Seeded stress of the hot path against the oracle: many adversarial cases
per call (slot maps, fused slot map + write, the three gathers, both block
copies), bit-exact, error word included.  KV_STRESS_SEEDS scales the number
of seeds (default 60 per group)."""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_39_gb300 as kv
from paged_kv_cache_39_gb300 import workloads as wl
from gpu_helpers import bits, cuda, dev, err_word, random_slot_case

pytestmark = pytest.mark.gpu

SEEDS = range(int(os.environ.get("KV_STRESS_SEEDS", "60")))
ROW_SHAPES = [(1, 8), (8, 64), (2, 72), (8, 128), (16, 128)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    torch.cuda.set_device(dev())
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _ranges(rng, rows, B):
    rstride = int(rng.choice([1, 4, 40, 256]))
    rs = rng.integers(-2, B + 2, size=(rows, rstride)).astype(np.int32)
    rl = rng.integers(-1, 12, size=(rows, rstride)).astype(np.int32)
    if rng.random() < 0.5:
        rl = np.maximum(rl, 1)
    nr = rng.integers(0, rstride + 1, size=rows).astype(np.int32)
    if rng.random() < 0.3:
        nr[rng.integers(0, rows)] = rstride + 1
    return rs, rl, nr


def _dev_bits(a):
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev())


@pytest.mark.parametrize("seed", SEEDS)
def test_slot_maps_and_fused_stress(seed):
    rng = np.random.default_rng(100000 + seed)
    T, R, q, N, n_max, stride, B, table, pos = random_slot_case(rng)
    pad = int(rng.choice([0, 0, 400_000]))
    n_max += pad
    rs, rl, nr = _ranges(rng, max(R, 1), B)
    exp = {"paged": oracle.slot_mapping_paged(q, pos, table, N, n_max, T, B),
           "range": oracle.slot_mapping_range(q, pos, rs, rl, nr, N, n_max, T, B)}
    e = err_word()
    s = kv.kv_slot_mapping_paged(cuda(q), cuda(pos), cuda(table), T, B, max_num_tokens=n_max,
                                 num_tokens=N, err=e)
    assert int(e.item()) == exp["paged"][1] and np.array_equal(s.cpu().numpy(), exp["paged"][0])
    e = err_word()
    s = kv.kv_slot_mapping_range(cuda(q), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B,
                                 max_num_tokens=n_max, num_tokens=N, err=e)
    assert int(e.item()) == exp["range"][1] and np.array_equal(s.cpu().numpy(), exp["range"][0])
    if pad or B * T > 20000:
        return
    H, D = ROW_SHAPES[seed % len(ROW_SHAPES)]
    L = 1 + seed % 2
    key = wl.bf16_normal((L, N, H, D), seed)
    kc = wl.bf16_normal((L, B, T, H, D), seed + 1)
    kb = bits(key)
    for kind in ("paged", "range"):
        exp_s, exp_e = exp[kind]
        s_tok = exp_s[:N]
        uniq, cnt = np.unique(s_tok[s_tok >= 0], return_counts=True)
        shared = uniq[cnt > 1]
        ek, ev = bits(kc).copy(), bits(kc).copy()
        oracle.cache_write(kb, kb, ek, ev, np.where(np.isin(s_tok, shared), -1, s_tok), B, T)
        kd, vd = kc.to(dev()), kc.to(dev())
        e = err_word()
        if kind == "paged":
            out = kv.kv_slot_mapping_paged_write(cuda(q), cuda(pos), cuda(table), T, B,
                                                 key.to(dev()), key.to(dev()), kd, vd,
                                                 max_num_tokens=n_max, num_tokens=N, err=e)
        else:
            out = kv.kv_slot_mapping_range_write(cuda(q), cuda(pos), cuda(rs), cuda(rl),
                                                 cuda(nr), T, B, key.to(dev()), key.to(dev()),
                                                 kd, vd, max_num_tokens=n_max, num_tokens=N,
                                                 err=e)
        assert int(e.item()) == exp_e and np.array_equal(out.cpu().numpy(), exp_s)
        gk, gv = bits(kd), bits(vd)
        for sl in shared:  # shared slots race per 16-byte store
            b, o = divmod(int(sl), T)
            toks = np.nonzero(s_tok == sl)[0]
            for l in range(L):
                for got in (gk[l, b, o], gv[l, b, o]):
                    cands = np.stack([kb[l, t].reshape(-1, 8) for t in toks])
                    assert (cands == got.reshape(-1, 8)[None]).all(axis=2).any(axis=0).all()
                ek[l, b, o], ev[l, b, o] = gk[l, b, o], gv[l, b, o]
        assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


@pytest.mark.parametrize("seed", SEEDS)
def test_gathers_and_copies_stress(seed):
    rng = np.random.default_rng(200000 + seed)
    R = int(rng.integers(1, 300))
    T = int(rng.choice([1, 4, 6, 8, 12, 16]))
    stride = int(rng.integers(1, 12))
    B = int(rng.integers(2, 80))
    L = int(rng.integers(1, 3))
    H, D = ROW_SHAPES[seed % len(ROW_SHAPES)]
    table = rng.integers(-1, B + 2, size=(R, stride)).astype(np.int32)
    table[rng.random(table.shape) < 0.2] = 0
    g0 = rng.integers(-1, stride * T + 2, size=R).astype(np.int32)
    g1 = (g0 + rng.integers(-2, 3 * T + 2, size=R)).astype(np.int32)
    total = int(np.where((g0 >= 0) & (g1 >= g0), g1 - g0, 0).sum())
    out_rows = max(0, total + int(rng.integers(-3, 4)))
    layer = int(rng.integers(0, L))
    kc = wl.bf16_normal((L, B, T, H, D), seed)
    vc = wl.bf16_normal((L, B, T, H, D), seed + 7)
    kcb, vcb = bits(kc), bits(vc)
    kcd, vcd = kc.to(dev()), vc.to(dev())
    fill = lambda v: np.full((out_rows, H, D), v, np.uint16)  # noqa: E731
    ko, vo = fill(0x1234), fill(0x4321)
    exp_e = oracle.cache_gather(kcb, vcb, layer, B, T, table, g0, g1, ko, vo)
    for bulk in (False, True):
        k_out, v_out = _dev_bits(fill(0x1234)), _dev_bits(fill(0x4321))
        e = err_word()
        kv.kv_cache_gather(kcd, vcd, cuda(table), cuda(g0), cuda(g1), layer=layer, k_out=k_out,
                           v_out=v_out, out_rows=out_rows, err=e, bulk=bulk)
        assert int(e.item()) == exp_e
        assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)
    # the range-addressed gather on random (partly malformed) descriptors
    S = int(rng.choice([1, 4, 9, 40]))
    rs = rng.integers(-1, B + 2, size=(R, S)).astype(np.int32)
    rl = rng.integers(-1, 6, size=(R, S)).astype(np.int32)
    if rng.random() < 0.5:
        rl = np.maximum(rl, 1)
    nr = rng.integers(0, S + 1, size=R).astype(np.int32)
    src, exp_re = oracle.gather_rows_range(layer, B, T, rs, rl, nr, g0, g1, out_rows)
    E = H * D
    ko2, vo2 = fill(0x1234).reshape(-1, E), fill(0x4321).reshape(-1, E)
    kf, vf = kcb.reshape(-1, E), vcb.reshape(-1, E)
    for o, n in enumerate(src):
        if n >= 0:
            ko2[o], vo2[o] = kf[n], vf[n]
        elif n == -1:
            ko2[o], vo2[o] = 0, 0
    k_out, v_out = _dev_bits(fill(0x1234)), _dev_bits(fill(0x4321))
    e = err_word()
    kv.kv_cache_gather_range(kcd, vcd, cuda(rs), cuda(rl), cuda(nr), cuda(g0), cuda(g1),
                             layer=layer, k_out=k_out, v_out=v_out, out_rows=out_rows, err=e)
    assert int(e.item()) == exp_re
    assert np.array_equal(bits(k_out).reshape(-1, E), ko2)
    assert np.array_equal(bits(v_out).reshape(-1, E), vo2)
    # block copies: distinct destinations, none the source of another pair
    P = int(rng.integers(0, min(20, (B - 1) // 2) + 1))
    perm = rng.permutation(np.arange(1, B)).astype(np.int32)
    sb, db = perm[:P].copy(), perm[P:2 * P].copy()
    if P > 2:
        sb[0] = int(rng.choice([0, -1, B]))
        db[1] = int(rng.choice([0, -3, B + 1]))
    for bulk in (False, True):
        ek, ev = kcb.copy(), vcb.copy()
        exp_ce = oracle.copy_blocks(ek, ev, sb, db)
        kd2, vd2 = kc.to(dev()), vc.to(dev())
        e = err_word()
        kv.kv_copy_blocks(kd2, vd2, cuda(sb), cuda(db), err=e, bulk=bulk)
        assert int(e.item()) == exp_ce
        assert np.array_equal(bits(kd2), ek) and np.array_equal(bits(vd2), ev)


def _prefill_batch(rng):
    """A large prefill-like batch (170k-700k tokens over at most 12 requests):
    the size at which the range map stages each tile's descriptors in shared
    memory.  Positions mostly run on from a random start, with jumps,
    negative and out-of-range values; descriptor rows are adversarial: empty,
    negative and zero lengths, null starts, starts whose ranges run past the
    pool, counts above the stride, rows of more than 32 ranges."""
    R = int(rng.integers(1, 13))
    N = int(rng.integers(170_000, 700_000))
    cuts = np.sort(rng.integers(0, N + 1, size=R - 1))
    lens = np.diff(np.concatenate([[0], cuts, [N]]))
    shift = int(rng.choice([0, 0, 7]))
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64) + shift
    q[-1] = min(q[-1], N)
    n_max = N + int(rng.choice([0, 5, 3000]))
    T = int(rng.choice([16, 16, 24, 32]))
    B = 400_000
    pos = np.empty(N, np.int64)
    for r in range(R):
        lo, hi = int(q[r]), int(q[r + 1])
        pos[lo:hi] = int(rng.integers(0, 20_000)) + np.arange(hi - lo)
    pos[:q[0]] = rng.integers(0, 1000, size=int(q[0]))
    jumps = rng.integers(0, N, size=int(rng.integers(0, 50)))
    pos[jumps] = rng.integers(-3, 2_000_000, size=len(jumps))
    S = int(rng.choice([8, 32, 40, 256]))
    rs = rng.integers(1, B - 3000, size=(R, S)).astype(np.int32)
    rl = rng.integers(1, 3000, size=(R, S)).astype(np.int32)
    nr = rng.integers(0, min(S, 40) + 1, size=R).astype(np.int32)
    mask = rng.random((R, S))
    rl[mask < 0.03] = 0
    rl[(mask >= 0.03) & (mask < 0.05)] = -1
    rs[(mask >= 0.05) & (mask < 0.08)] = 0
    rs[(mask >= 0.08) & (mask < 0.11)] = B - 10
    rs[(mask >= 0.11) & (mask < 0.12)] = -5
    if R > 1 and rng.random() < 0.3:
        nr[rng.integers(0, R)] = S + 1
    return T, R, q.astype(np.int32), N, n_max, B, pos, rs, rl, nr


@pytest.mark.parametrize("seed", range(max(1, len(SEEDS) // 4)))
def test_range_staged_stress(seed):
    rng = np.random.default_rng(90_000 + seed)
    T, R, q, N, n_max, B, pos, rs, rl, nr = _prefill_batch(rng)
    exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, n_max, T, B)
    e = err_word()
    s = kv.kv_slot_mapping_range(cuda(q), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B,
                                 max_num_tokens=n_max, err=e)
    assert int(e.item()) == exp_e
    got = s.cpu().numpy()
    assert np.array_equal(got, exp_s), f"first difference at token {int(np.argmax(got != exp_s))}"
    # the paged map over the same blocks agrees wherever the table holds them
    if (nr >= 0).all() and (nr <= rs.shape[1]).all() and (rl[:, :] > 0).all():
        stride = wl.table_stride_for(int(np.maximum(rl, 0).sum(axis=1).max()) + 1, T)
        table = oracle.table_from_ranges(rs, rl, nr, stride)
        ep, _ = oracle.slot_mapping_paged(q, pos, table, N, n_max, T, B)
        e2 = err_word()
        sp = kv.kv_slot_mapping_paged(cuda(q), cuda(pos), cuda(table), T, B,
                                      max_num_tokens=n_max, err=e2)
        assert np.array_equal(sp.cpu().numpy(), ep)
