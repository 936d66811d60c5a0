"""Large shapes through the whole path: both slot maps, the fused calls,
the write, the three gathers and both block copies at 128 to 2048 tokens per
block (528, not a power of two, is a size hybrid attention/state-space models
give their attention blocks); expansion ratios of 11 to 128; 80 and 128
layers; rows of 32 and 40 KiB.  Every result is compared with the oracle bit
for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_39_gb300 as kv
from paged_kv_cache_39_gb300 import workloads as wl
from gpu_helpers import bits, cuda, dev, err_word

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    torch.cuda.set_device(dev())
    yield
    torch.cuda.synchronize()


def _case(T, seed):
    """Three requests over one contiguous range of `stride` blocks each (the
    table row is that range expanded): a prefill crossing a block boundary, a
    decode token, and a prefill whose last positions run past the row."""
    rng = np.random.default_rng(seed)
    stride, R = 4, 3
    B = 1 + R * stride + 3
    firsts = 1 + rng.permutation(R) * stride
    table = np.stack([np.arange(f, f + stride) for f in firsts]).astype(np.int32)
    rs = np.zeros((R, 4), np.int32)
    rl = np.zeros((R, 4), np.int32)
    rs[:, 0], rl[:, 0] = firsts, stride
    nr = np.ones(R, np.int32)
    p0 = int(rng.integers(0, T))
    pos = [np.arange(p0, p0 + T + T // 2 + 1),
           np.array([int(rng.integers(0, stride * T))]),
           np.arange(stride * T - 5, stride * T + 3)]
    lens = [len(p) for p in pos]
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return B, table, rs, rl, nr, qsl, np.concatenate(pos).astype(np.int64)


@pytest.mark.parametrize("T,H,D", [(128, 1, 8), (528, 1, 8), (2048, 1, 8), (528, 2, 64)])
def test_large_block_sizes(T, H, D):
    L = 2
    B, table, rs, rl, nr, qsl, pos = _case(T, 15000 + T + H + D)
    N = int(qsl[-1])
    n_max = N + 7
    exp_s, exp_e = oracle.slot_mapping_paged(qsl, pos, table, N, n_max, T, B)
    exp_r, exp_re = oracle.slot_mapping_range(qsl, pos, rs, rl, nr, N, n_max, T, B)
    assert np.array_equal(exp_s, exp_r) and exp_e == exp_re
    assert (exp_s[:N] >= 0).sum() == N - 3  # the three positions past the row are PAD

    e = err_word()
    s = kv.kv_slot_mapping_paged(cuda(qsl), cuda(pos), cuda(table), T, B, max_num_tokens=n_max,
                                 err=e)
    assert np.array_equal(s.cpu().numpy(), exp_s) and int(e.item()) == exp_e
    e = err_word()
    s = kv.kv_slot_mapping_range(cuda(qsl), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B,
                                 max_num_tokens=n_max, err=e)
    assert np.array_equal(s.cpu().numpy(), exp_s) and int(e.item()) == exp_e

    # write, and the fused calls from the same starting caches
    key = wl.bf16_normal((L, N, H, D), 150)
    val = wl.bf16_normal((L, N, H, D), 151)
    kc = wl.bf16_normal((L, B, T, H, D), 152)
    vc = wl.bf16_normal((L, B, T, H, D), 153)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_we = oracle.cache_write(bits(key), bits(val), ek, ev, exp_s[:N], B, T)
    kd, vd = key.to(dev()), val.to(dev())
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    kv.kv_cache_write(kd, vd, kc_d, vc_d, cuda(exp_s[:N]), err=e)
    assert int(e.item()) == exp_we
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)
    for fused in ("paged", "range"):
        kc_f, vc_f = kc.to(dev()), vc.to(dev())
        e = err_word()
        if fused == "paged":
            s = kv.kv_slot_mapping_paged_write(cuda(qsl), cuda(pos), cuda(table), T, B, kd, vd,
                                               kc_f, vc_f, max_num_tokens=n_max, err=e)
        else:
            s = kv.kv_slot_mapping_range_write(cuda(qsl), cuda(pos), cuda(rs), cuda(rl),
                                               cuda(nr), T, B, kd, vd, kc_f, vc_f,
                                               max_num_tokens=n_max, err=e)
        assert np.array_equal(s.cpu().numpy(), exp_s), fused
        assert int(e.item()) == exp_e | exp_we, fused
        assert np.array_equal(bits(kc_f), ek) and np.array_equal(bits(vc_f), ev), fused

    # gathers of layer 1 over spans that start and end inside blocks
    rng = np.random.default_rng(T + 7)
    R, stride = table.shape
    g0 = rng.integers(0, stride * T // 2, size=R).astype(np.int32)
    g1 = np.minimum(g0 + rng.integers(1, 2 * T + 3, size=R), stride * T).astype(np.int32)
    out_rows = int((g1 - g0).sum())
    ko = np.zeros((out_rows, H, D), np.uint16)
    vo = np.zeros((out_rows, H, D), np.uint16)
    exp_ge = oracle.cache_gather(ek, ev, 1, B, T, table, g0, g1, ko, vo)
    for bulk in (False, True):
        e = err_word()
        k_out, v_out = kv.kv_cache_gather(kc_d, vc_d, cuda(table), cuda(g0), cuda(g1), layer=1,
                                          out_rows=out_rows, err=e, bulk=bulk)
        assert int(e.item()) == exp_ge
        assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo), bulk
    e = err_word()
    k_out, v_out = kv.kv_cache_gather_range(kc_d, vc_d, cuda(rs), cuda(rl), cuda(nr), cuda(g0),
                                            cuda(g1), layer=1, out_rows=out_rows, err=e)
    src, exp_rge = oracle.gather_rows_range(1, B, T, rs, rl, nr, g0, g1, out_rows)
    assert int(e.item()) == exp_rge
    k_rows = ek.reshape(-1, H * D)
    v_rows = ev.reshape(-1, H * D)
    assert (src >= 0).all()
    assert np.array_equal(bits(k_out).reshape(-1, H * D), k_rows[src])
    assert np.array_equal(bits(v_out).reshape(-1, H * D), v_rows[src])
    assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)

    # copy-on-write of whole blocks (a block is T rows: up to 264 KiB here)
    src_b = table[:, 0].copy()
    dst_b = np.array([B - 3, B - 2, B - 1], np.int32)
    for bulk in (False, True):
        ck, cv = ek.copy(), ev.copy()
        exp_ce = oracle.copy_blocks(ck, cv, src_b, dst_b)
        kc_c, vc_c = kc_d.clone(), vc_d.clone()
        e = err_word()
        kv.kv_copy_blocks(kc_c, vc_c, cuda(src_b), cuda(dst_b), err=e, bulk=bulk)
        assert int(e.item()) == exp_ce
        assert np.array_equal(bits(kc_c), ck) and np.array_equal(bits(vc_c), cv), bulk


@pytest.mark.parametrize("mgr_bs,kern_bs,extra", [(528, 16, 0), (1056, 16, 5), (2048, 16, 0),
                                                  (528, 48, 2)])
def test_expand_large_ratios(mgr_bs, kern_bs, extra):
    """Manager blocks of 528 to 2048 tokens unfolded into 16- or 48-token
    kernel blocks (k = 11 to 128 kernel entries per manager entry), with null
    and negative entries and one whose last kernel block overflows int32."""
    k = mgr_bs // kern_bs
    rng = np.random.default_rng(16000 + mgr_bs + kern_bs)
    R, Ms = 9, 7
    mgr = rng.integers(-2, (1 << 31) // k, size=(R, Ms)).astype(np.int32)
    mgr[rng.random(mgr.shape) < 0.3] = 0
    mgr[1, 2] = (1 << 31) // k  # m * k + (k - 1) passes INT32_MAX
    mgr[2, 0], mgr[4, 6] = -1, -7
    Ks = Ms * k + extra
    exp, exp_e = oracle.expand_kernel_blocks(mgr, mgr_bs, kern_bs, Ks)
    assert exp_e != 0  # the negative and the overflowing entries
    e = err_word()
    out = kv.kv_expand_kernel_blocks(cuda(mgr), mgr_bs, kern_bs,
                                     kernel_table=torch.full((R, Ks), 77, dtype=torch.int32,
                                                             device=dev()), err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(out.cpu().numpy(), exp)


@pytest.mark.parametrize("L,H,D", [(80, 1, 8), (128, 2, 16), (2, 64, 256), (3, 20, 1024)])
def test_many_layers_and_wide_rows(L, H, D):
    """80 and 128 layers of small rows, and rows of 32 and 40 KiB (64 heads x
    256, 20 x 1024), through the write, the fused paged call, the gather of
    the last layer and both block copies (the bulk forms refuse rows past 32
    KiB, where the vector forms run)."""
    T = 16
    B, table, rs, rl, nr, qsl, pos = _case(T, 17000 + L + H + D)
    N = int(qsl[-1])
    exp_s, exp_e = oracle.slot_mapping_paged(qsl, pos, table, N, N, T, B)
    key = wl.bf16_normal((L, N, H, D), 170)
    val = wl.bf16_normal((L, N, H, D), 171)
    kc = wl.bf16_normal((L, B, T, H, D), 172)
    vc = wl.bf16_normal((L, B, T, H, D), 173)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_we = oracle.cache_write(bits(key), bits(val), ek, ev, exp_s, B, T)
    kd, vd = key.to(dev()), val.to(dev())
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    kv.kv_cache_write(kd, vd, kc_d, vc_d, cuda(exp_s), err=e)
    assert int(e.item()) == exp_we
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)
    kc_f, vc_f = kc.to(dev()), vc.to(dev())
    e = err_word()
    s = kv.kv_slot_mapping_paged_write(cuda(qsl), cuda(pos), cuda(table), T, B, kd, vd, kc_f,
                                       vc_f, err=e)
    assert np.array_equal(s.cpu().numpy(), exp_s) and int(e.item()) == exp_e | exp_we
    assert np.array_equal(bits(kc_f), ek) and np.array_equal(bits(vc_f), ev)
    del kc_f, vc_f

    R, stride = table.shape
    g0 = np.array([0, 5, 17], np.int32)
    g1 = np.array([stride * T, 38, 17 + T], np.int32)
    out_rows = int((g1 - g0).sum())
    ko = np.zeros((out_rows, H, D), np.uint16)
    vo = np.zeros((out_rows, H, D), np.uint16)
    exp_ge = oracle.cache_gather(ek, ev, L - 1, B, T, table, g0, g1, ko, vo)
    for bulk in (False, True):
        e = err_word()
        args = (kc_d, vc_d, cuda(table), cuda(g0), cuda(g1))
        if bulk and H * D * 2 > 32768:
            with pytest.raises(kv.KVError) as ei:
                kv.kv_cache_gather(*args, layer=L - 1, out_rows=out_rows, err=e, bulk=True)
            assert ei.value.status == kv.KV_EUNSUPPORTED
            continue
        k_out, v_out = kv.kv_cache_gather(*args, layer=L - 1, out_rows=out_rows, err=e,
                                          bulk=bulk)
        assert int(e.item()) == exp_ge
        assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo), bulk

    src_b = np.array([table[0, 1], table[2, 3], 0], np.int32)
    dst_b = np.array([B - 1, B - 2, B - 3], np.int32)
    for bulk in (False, True):
        ck, cv = ek.copy(), ev.copy()
        exp_ce = oracle.copy_blocks(ck, cv, src_b, dst_b)
        kc_c, vc_c = kc_d.clone(), vc_d.clone()
        e = err_word()
        kv.kv_copy_blocks(kc_c, vc_c, cuda(src_b), cuda(dst_b), err=e, bulk=bulk)
        assert int(e.item()) == exp_ce
        assert np.array_equal(bits(kc_c), ck) and np.array_equal(bits(vc_c), cv), bulk
