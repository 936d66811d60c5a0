"""GPU parity of the next-step entry points (range expansion, range-addressed
gather, copy-on-write block copy) against the CPU oracle, bit-exact, with the
error word."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_39_gb300 as kv
from paged_kv_cache_39_gb300 import workloads as wl
from gpu_helpers import bits, cuda, dev, device_rows_equal, err_word, rows_view

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    torch.cuda.set_device(dev())
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def random_ranges(rng, R, S, B, malformed=True):
    rs = rng.integers(-1 if malformed else 1, B + 2, size=(R, S)).astype(np.int32)
    rl = rng.integers(-1 if malformed else 1, 6, size=(R, S)).astype(np.int32)
    nr = rng.integers(0, S + 1, size=R).astype(np.int32)
    if malformed and R > 1:
        nr[int(rng.integers(0, R))] = S + 3
    return rs, rl, nr


# ------------------------------------------------------ range expansion


@pytest.mark.parametrize("seed,R,S,TS", [(0, 5, 6, 12), (1, 64, 256, 300), (2, 1, 256, 2048),
                                         (3, 40, 4, 7), (4, 3, 1, 1), (5, 9, 33, 64)])
def test_table_from_ranges_parity(seed, R, S, TS):
    rng = np.random.default_rng(9000 + seed)
    rs, rl, nr = random_ranges(rng, R, S, 1 << 20)
    if seed == 1:
        rs[0, 0] = (1 << 31) - 2  # the second block of this range overflows int32
        rl[0, 0] = 3
        nr[0] = max(nr[0], 1)
    exp, exp_e = oracle.table_from_ranges(rs, rl, nr, TS, with_error=True)
    e = err_word()
    out = kv.kv_table_from_ranges(cuda(rs), cuda(rl), cuda(nr),
                                  block_table=torch.full((R, TS), 77, dtype=torch.int32,
                                                         device=dev()), err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(out.cpu().numpy(), exp)


@pytest.mark.parametrize("name,layout", [("tiny", "G"), ("tiny", "P"), ("decode", "G"),
                                         ("mixed", "G"), ("long", "G")])
def test_table_from_ranges_rebuilds_workload_tables(name, layout):
    w = wl.CONFIGS[name]()
    lay = w.layouts[layout]
    e = err_word()
    t = kv.kv_table_from_ranges(cuda(lay.range_start), cuda(lay.range_len), cuda(lay.num_ranges),
                                table_stride=lay.table_stride, err=e)
    assert int(e.item()) == 0
    assert np.array_equal(t.cpu().numpy(), lay.table)
    # the paged slot map over the rebuilt table equals the range slot map
    qsl, pos = cuda(w.qsl), cuda(w.positions)
    e = err_word()
    sp = kv.kv_slot_mapping_paged(qsl, pos, t, w.block_size, w.num_blocks,
                                  max_num_tokens=w.max_num_tokens, err=e)
    sr = kv.kv_slot_mapping_range(qsl, pos, cuda(lay.range_start), cuda(lay.range_len),
                                  cuda(lay.num_ranges), w.block_size, w.num_blocks,
                                  max_num_tokens=w.max_num_tokens, err=e)
    assert int(e.item()) == 0 and torch.equal(sp, sr)


# ------------------------------------------------ range-addressed gather


@pytest.mark.parametrize("seed,R,S,H,D", [(0, 1, 4, 8, 128), (1, 6, 6, 8, 64), (2, 300, 3, 1, 8),
                                          (3, 4096, 2, 1, 16), (4, 17, 40, 16, 128),
                                          (5, 9, 256, 2, 72), (6, 4093, 2, 1, 8),
                                          (7, 4095, 1, 1, 8)])
def test_gather_range_random_parity(seed, R, S, H, D):
    rng = np.random.default_rng(9100 + seed)
    T, B, L = 8, 60, 2
    rs, rl, nr = random_ranges(rng, R, S, B)
    g0 = rng.integers(-1, 30 * T, size=R).astype(np.int32)
    g1 = (g0 + rng.integers(-2, 24, size=R)).astype(np.int32)
    total = int(np.where((g0 >= 0) & (g1 >= g0), g1 - g0, 0).sum())
    out_rows = max(0, total - int(rng.integers(0, 3))) if seed % 2 else total + 3
    layer = seed % L
    kc = wl.bf16_normal((L, B, T, H, D), 60 + seed)
    vc = wl.bf16_normal((L, B, T, H, D), 70 + seed)
    ko = np.full((out_rows, H, D), 0x1234, np.uint16)
    vo = np.full((out_rows, H, D), 0x4321, np.uint16)
    src, exp_e = oracle.gather_rows_range(layer, B, T, rs, rl, nr, g0, g1, out_rows)
    kc_h, vc_h = bits(kc).reshape(-1, H * D), bits(vc).reshape(-1, H * D)
    for o, n in enumerate(src):
        if n >= 0:
            ko.reshape(-1, H * D)[o] = kc_h[n]
            vo.reshape(-1, H * D)[o] = vc_h[n]
        elif n == -1:
            ko.reshape(-1, H * D)[o] = 0
            vo.reshape(-1, H * D)[o] = 0
    k_out = torch.from_numpy(np.full((out_rows, H, D), 0x1234, np.int16)).view(
        torch.bfloat16).to(dev())
    v_out = torch.from_numpy(np.full((out_rows, H, D), 0x4321, np.int16)).view(
        torch.bfloat16).to(dev())
    e = err_word()
    kv.kv_cache_gather_range(kc.to(dev()), vc.to(dev()), cuda(rs), cuda(rl), cuda(nr), cuda(g0),
                             cuda(g1), layer=layer, k_out=k_out, v_out=v_out, out_rows=out_rows,
                             err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)


@pytest.mark.parametrize("name", ["tiny", "decode", "long"])
def test_gather_range_equals_table_gather_full_size(name):
    w = wl.CONFIGS[name]()
    lay = w.layouts["G"]
    T, B, H, D, E = w.block_size, w.num_blocks, w.num_kv_heads, w.head_dim, w.row_elems
    kc = wl.bf16_normal((1, B, T, H, D), 80, dev())
    vc = wl.bf16_normal((1, B, T, H, D), 81, dev())
    rows = int((w.gather_end.astype(np.int64) - w.gather_start).sum())
    g0, g1 = cuda(w.gather_start), cuda(w.gather_end)
    e = err_word()
    kr, vr = kv.kv_cache_gather_range(kc, vc, cuda(lay.range_start), cuda(lay.range_len),
                                      cuda(lay.num_ranges), g0, g1, out_rows=rows, err=e)
    src, exp_e = oracle.gather_rows_range(0, B, T, lay.range_start, lay.range_len, lay.num_ranges,
                                          w.gather_start, w.gather_end, rows)
    assert int(e.item()) == exp_e == 0
    assert device_rows_equal(kr, kc, src, E) and device_rows_equal(vr, vc, src, E)
    kt, vt = kv.kv_cache_gather(kc, vc, cuda(lay.table), g0, g1, out_rows=rows, err=e)
    assert int(e.item()) == 0
    assert torch.equal(rows_view(kt, E), rows_view(kr, E))
    assert torch.equal(rows_view(vt, E), rows_view(vr, E))


# ------------------------------------------------------- copy-on-write


@pytest.mark.parametrize("bulk", [False, True])
@pytest.mark.parametrize("L,H,D", [(1, 8, 128), (3, 8, 64), (2, 16, 128), (2, 1, 128), (0, 8, 64)])
def test_copy_blocks_parity(L, H, D, bulk):
    rng = np.random.default_rng(9200 + L * 7 + H + D)
    B, T, P = 64, 16, 20
    perm = rng.permutation(np.arange(1, B))
    src = perm[:P].astype(np.int32)
    dst = perm[P:2 * P].astype(np.int32)
    src[3] = 0          # null source
    dst[5] = 0          # null destination
    src[7] = B + 4      # bad source
    dst[9] = -2         # bad destination
    kc = wl.bf16_normal((L, B, T, H, D), 90 + L)
    vc = wl.bf16_normal((L, B, T, H, D), 95 + L)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_e = oracle.copy_blocks(ek, ev, src, dst)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    kv.kv_copy_blocks(kc_d, vc_d, cuda(src), cuda(dst), err=e, bulk=bulk)
    assert int(e.item()) == exp_e
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)


@pytest.mark.parametrize("T,H,D", [(12, 16, 128), (16, 32, 128), (3, 1, 8), (1, 8, 128)])
def test_copy_blocks_bulk_piece_sizes(T, H, D):
    """Blocks of 48 KiB and 128 KiB move as 32 KiB pieces plus a remainder;
    tiny blocks (48 B, 2 KiB) as one piece each."""
    rng = np.random.default_rng(9250 + T + H + D)
    L, B, P = 2, 40, 12
    perm = rng.permutation(np.arange(1, B))
    src = perm[:P].astype(np.int32)
    dst = perm[P:2 * P].astype(np.int32)
    src[2], dst[4] = 0, B  # a null source, an out-of-range destination
    kc = wl.bf16_normal((L, B, T, H, D), 300 + T)
    vc = wl.bf16_normal((L, B, T, H, D), 310 + T)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_e = oracle.copy_blocks(ek, ev, src, dst)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    kv.kv_copy_blocks(kc_d, vc_d, cuda(src), cuda(dst), err=e, bulk=True)
    assert int(e.item()) == exp_e
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)


def test_copy_then_write_diverges_only_the_copy():
    B, T, H, D = 32, 16, 8, 128
    kc = wl.bf16_normal((2, B, T, H, D), 99, dev())
    vc = wl.bf16_normal((2, B, T, H, D), 98, dev())
    orig = kc.clone()
    e = err_word()
    kv.kv_copy_blocks(kc, vc, cuda(np.array([4], np.int32)), cuda(np.array([20], np.int32)), err=e)
    key = wl.bf16_normal((2, 1, H, D), 97, dev())
    kv.kv_cache_write(key, key, kc, vc, cuda(np.array([20 * T + 3], np.int64)), err=e)
    assert int(e.item()) == 0
    assert torch.equal(kc[:, 4], orig[:, 4])
    same = (kc[:, 20] == orig[:, 4]).all(dim=(2, 3))
    exp = torch.ones_like(same)
    exp[:, 3] = False
    assert torch.equal(same, exp)


@pytest.mark.parametrize("bulk", [False, True])
@pytest.mark.parametrize("P,L,T", [(1000, 3, 16), (2000, 4, 6)])
def test_copy_blocks_grouped_path(P, L, T, bulk):
    """Batches of tens of thousands of rows copy four rows per warp step; a
    block size of 6 leaves a two-row remainder in every block."""
    rng = np.random.default_rng(9300 + P + T)
    H, D = 1, 32
    B = 2 * P + 50
    perm = rng.permutation(np.arange(1, B)).astype(np.int32)
    src, dst = perm[:P].copy(), perm[P:2 * P].copy()
    src[5], dst[9], src[11] = 0, 0, B + 1
    kc = wl.bf16_normal((L, B, T, H, D), 400 + T)
    vc = wl.bf16_normal((L, B, T, H, D), 410 + T)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_e = oracle.copy_blocks(ek, ev, src, dst)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    kv.kv_copy_blocks(kc_d, vc_d, cuda(src), cuda(dst), err=e, bulk=bulk)
    assert int(e.item()) == exp_e
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)
