"""GPU parity on small and adversarial cases: every output of every kernel is
compared element by element with the CPU oracle (bit-exact, tolerance 0:
outputs are integers or copied bf16 bits), together with the error word."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_39_gb300 as kv
from paged_kv_cache_39_gb300 import workloads as wl
from gpu_helpers import bits, cuda, dev, err_word, random_slot_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()  # fails loudly when the CUDA library is missing
    torch.cuda.set_device(dev())
    yield
    torch.cuda.synchronize()


def run_paged(qsl, pos, table, N, n_max, T, B):
    e = err_word()
    s = kv.kv_slot_mapping_paged(cuda(np.asarray(qsl, np.int32)), cuda(np.asarray(pos, np.int64)),
                                 cuda(np.asarray(table, np.int32)), T, B, max_num_tokens=n_max,
                                 num_tokens=N, err=e)
    return s.cpu().numpy(), int(e.item())


def run_range(qsl, pos, rs, rl, nr, N, n_max, T, B):
    e = err_word()
    s = kv.kv_slot_mapping_range(cuda(np.asarray(qsl, np.int32)), cuda(np.asarray(pos, np.int64)),
                                 cuda(np.asarray(rs, np.int32)), cuda(np.asarray(rl, np.int32)),
                                 cuda(np.asarray(nr, np.int32)), T, B, max_num_tokens=n_max,
                                 num_tokens=N, err=e)
    return s.cpu().numpy(), int(e.item())


# ------------------------------------------------------------------ golden


def test_figure6_on_gpu(golden):
    g = golden("figure6_bs4.json")
    T = g["block_size"]
    for step in g["steps"]:
        row = np.zeros((1, 8), np.int32)
        row[0, :len(step["row"])] = step["row"]
        n = len(step["positions"])
        s, e = run_paged([0, n], step["positions"], row, n, n, T, 16)
        assert e == 0 and s.tolist() == step["slots"]
    rs = np.zeros((1, 256), np.int32)
    rl = np.zeros((1, 256), np.int32)
    for i, (a, b) in enumerate(g["ranges_final_row"]):
        rs[0, i], rl[0, i] = a, b
    pos = sum((st["positions"] for st in g["steps"]), [])
    s, e = run_range([0, len(pos)], pos, rs, rl, [3], len(pos), len(pos), T, 16)
    assert e == 0 and s.tolist() == sum((st["slots"] for st in g["steps"]), [])


def test_page3_on_gpu(golden):
    g = golden("page3_bs16.json")
    row = np.zeros((1, 8), np.int32)
    row[0, :2] = g["row"]
    n = len(g["positions"])
    s, e = run_paged([0, n], g["positions"], row, n, n + 3, g["block_size"], 16)
    assert e == 0
    assert s[:16].tolist() == list(range(112, 128)) and s[16] == 16 and (s[n:] == -1).all()


def test_expand_golden_on_gpu(golden):
    g = golden("expand_32_16.json")
    e = err_word()
    out = kv.kv_expand_kernel_blocks(cuda(np.array([g["mgr_row"]], np.int32)),
                                     g["mgr_block_size"], g["kernel_block_size"], err=e)
    assert out.cpu().numpy()[0].tolist() == g["kernel_row"] and int(e.item()) == 0
    for mbs, kbs in g["rejected"]:
        with pytest.raises(kv.KVError) as ei:
            kv.kv_expand_kernel_blocks(cuda(np.array([[1]], np.int32)), mbs, kbs,
                                       kernel_table=torch.empty((1, 4), dtype=torch.int32,
                                                                device=dev()))
        assert ei.value.status == kv.KV_EUNSUPPORTED


# -------------------------------------------------------------- tiny config


@pytest.mark.parametrize("layout", ["P", "G"])
def test_tiny_whole_path(layout):
    w = wl.tiny()
    lay = w.layouts[layout]
    T, B, H, D = w.block_size, w.num_blocks, w.num_kv_heads, w.head_dim
    exp_s, exp_e = oracle.slot_mapping_paged(w.qsl, w.positions, lay.table, w.num_tokens,
                                             w.max_num_tokens, T, B)
    s, e = run_paged(w.qsl, w.positions, lay.table, w.num_tokens, w.max_num_tokens, T, B)
    assert e == exp_e and np.array_equal(s, exp_s)
    s2, e2 = run_range(w.qsl, w.positions, lay.range_start, lay.range_len, lay.num_ranges,
                       w.num_tokens, w.max_num_tokens, T, B)
    exp_s2, exp_e2 = oracle.slot_mapping_range(w.qsl, w.positions, lay.range_start, lay.range_len,
                                               lay.num_ranges, w.num_tokens, w.max_num_tokens, T,
                                               B)
    assert e2 == exp_e2 and np.array_equal(s2, exp_s2) and np.array_equal(s2, exp_s)

    L = 2
    key = wl.bf16_normal((L, w.num_tokens, H, D), 20)
    val = wl.bf16_normal((L, w.num_tokens, H, D), 21)
    kc = wl.bf16_normal((L, B, T, H, D), 22)
    vc = wl.bf16_normal((L, B, T, H, D), 23)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_we = oracle.cache_write(bits(key), bits(val), ek, ev, exp_s[:w.num_tokens], B, T)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    kv.kv_cache_write(key.to(dev()), val.to(dev()), kc_d, vc_d, cuda(s[:w.num_tokens]), err=e)
    assert int(e.item()) == exp_we
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)

    for layer in range(L):
        rows = int((w.gather_end - w.gather_start).sum())
        ko = np.zeros((rows, H, D), np.uint16)
        vo = np.zeros((rows, H, D), np.uint16)
        exp_ge = oracle.cache_gather(ek, ev, layer, B, T, lay.table, w.gather_start, w.gather_end,
                                     ko, vo)
        e = err_word()
        k_out, v_out = kv.kv_cache_gather(kc_d, vc_d, cuda(lay.table), cuda(w.gather_start),
                                          cuda(w.gather_end), layer=layer, out_rows=rows, err=e)
        assert int(e.item()) == exp_ge
        assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)
        # gather of what was written gives the written tokens back
        assert np.array_equal(bits(k_out), bits(key[layer]))


# --------------------------------------------------- adversarial slot maps


# Batches of up to a few hundred thousand tokens run one token per thread;
# padding max_num_tokens to 400k makes the same tokens run 4 per thread in
# both maps, with the range map's lane windows and warp descriptor cache
# carried across a thread's tokens.
PADS = [0, 400_000]


@pytest.mark.parametrize("pad", PADS)
@pytest.mark.parametrize("seed", range(40))
def test_paged_adversarial(seed, pad):
    rng = np.random.default_rng(1000 + seed)
    T, R, q, N, n_max, stride, B, table, pos = random_slot_case(rng)
    n_max += pad
    exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, n_max, T, B)
    s, e = run_paged(q, pos, table, N, n_max, T, B)
    assert e == exp_e
    assert np.array_equal(s, exp_s)


@pytest.mark.parametrize("pad", PADS)
@pytest.mark.parametrize("seed", range(40))
def test_range_adversarial(seed, pad):
    rng = np.random.default_rng(2000 + seed)
    T, R, q, N, n_max, stride, B, table, pos = random_slot_case(rng)
    n_max += pad
    rstride = int(rng.choice([1, 4, 40, 256]))
    rows = max(R, 1)
    rs = rng.integers(-2, B + 2, size=(rows, rstride)).astype(np.int32)
    rl = rng.integers(-1, 12, size=(rows, rstride)).astype(np.int32)
    if rng.random() < 0.5:
        rl = np.maximum(rl, 1)
    nr = rng.integers(0, rstride + 1, size=rows).astype(np.int32)
    if rng.random() < 0.3:
        nr[rng.integers(0, rows)] = rstride + 1
    exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, n_max, T, B)
    s, e = run_range(q, pos, rs, rl, nr, N, n_max, T, B)
    assert e == exp_e
    assert np.array_equal(s, exp_s)


@pytest.mark.parametrize("pad", PADS)
@pytest.mark.parametrize("seed", range(6))
def test_range_equals_paged_with_256_ranges(seed, pad):
    """Full descriptor rows (256 ranges, 8 warp chunks) agree with the table."""
    rng = np.random.default_rng(3000 + seed)
    T, R = 16, 3
    rs = np.zeros((R, 256), np.int32)
    rl = np.zeros((R, 256), np.int32)
    nr = np.full(R, 256, np.int32)
    lens = rng.integers(1, 6, size=(R, 256))
    cursor = 1
    for r in range(R):
        for i in range(256):
            rs[r, i] = cursor + int(rng.integers(0, 3))
            rl[r, i] = lens[r, i]
            cursor = rs[r, i] + lens[r, i]
    B = cursor + 1
    stride = wl.table_stride_for(int(lens.sum(axis=1).max()), T)
    table = oracle.table_from_ranges(rs, rl, nr, stride)
    tok = [int(rng.integers(1, 3000)) for _ in range(R)]
    q = np.concatenate([[0], np.cumsum(tok)]).astype(np.int32)
    pos = np.concatenate([rng.integers(0, int(lens[r].sum()) * T + 40, size=tok[r])
                          for r in range(R)]).astype(np.int64)
    N = int(q[-1])
    n_max = N + pad
    sp, ep = run_paged(q, pos, table, N, n_max, T, B)
    sr, er = run_range(q, pos, rs, rl, nr, N, n_max, T, B)
    exp, ee = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, n_max, T, B)
    assert ep == er == ee == 0
    assert np.array_equal(sr, exp) and np.array_equal(sp, exp)


# Tiles of 256, 1024 and 2048 tokens (one, four and eight tokens per thread)
# whose tokens belong to exactly 8 requests (descriptors staged per CTA) or
# to 9 (each lane walks its own request's ranges); some rows malformed.
# Rows of up to 40 ranges: those of more than 32 cannot be staged and their
# tiles take the general path.
@pytest.mark.parametrize("S", [12, 40])
@pytest.mark.parametrize("per_req,pad", [(32, 0), (31, 0), (128, 400_000), (127, 400_000),
                                         (256, 800_000), (255, 800_000)])
def test_range_staging_boundary(per_req, pad, S):
    rng = np.random.default_rng(3500 + per_req + S)
    T, R = 16, 40
    q = (np.arange(R + 1) * per_req).astype(np.int32)
    N = int(q[-1])
    rs = rng.integers(1, 5000, size=(R, S)).astype(np.int32)
    rl = rng.integers(1, 4, size=(R, S)).astype(np.int32)
    nr = rng.integers(1, S + 1, size=R).astype(np.int32)
    rl[3, 1] = 0          # an empty range inside a staged row
    nr[5] = S + 1         # a malformed count
    rl[11, 0] = -2        # a negative length
    pos = np.concatenate([rng.permutation(per_req) + int(rng.integers(0, 30)) * T
                          for _ in range(R)]).astype(np.int64)
    pos[7] = -4
    exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N + pad, T, 6000)
    s, e = run_range(q, pos, rs, rl, nr, N, N + pad, T, 6000)
    assert e == exp_e
    assert np.array_equal(s, exp_s)


def test_decode_batch_past_the_staging_limit():
    """10000 one-token requests: query_start_loc stays in global memory (more
    than the slot maps' 8191 and the fused calls' 2047 staged requests), and
    every thread's "request t owns token t" check hits there, the search
    never runs.  All four calls against the oracle."""
    rng = np.random.default_rng(7100)
    R, T, H, D, stride = 10000, 16, 1, 8, 4
    B = R * stride + 1
    q = np.arange(R + 1, dtype=np.int32)
    pos = rng.integers(0, stride * T, size=R).astype(np.int64)
    table = rng.permutation(np.arange(1, B)).astype(np.int32).reshape(R, stride)
    rs, rl = table.copy(), np.ones_like(table)
    nr = np.full(R, stride, np.int32)
    n_max = R + 100
    exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, R, n_max, T, B)
    assert exp_e == 0 and (exp_s[:R] >= 0).all()
    s, e = run_paged(q, pos, table, R, n_max, T, B)
    assert e == 0 and np.array_equal(s, exp_s)
    s, e = run_range(q, pos, rs, rl, nr, R, n_max, T, B)
    assert e == 0 and np.array_equal(s, exp_s)
    key = wl.bf16_normal((1, R, H, D), 711)
    for kind in ("paged", "range"):
        kc = torch.zeros((1, B, T, H, D), dtype=torch.bfloat16, device=dev())
        vc = torch.zeros_like(kc)
        e2 = err_word()
        if kind == "paged":
            sf = kv.kv_slot_mapping_paged_write(cuda(q), cuda(pos), cuda(table), T, B,
                                                key.to(dev()), key.to(dev()), kc, vc,
                                                max_num_tokens=n_max, err=e2)
        else:
            sf = kv.kv_slot_mapping_range_write(cuda(q), cuda(pos), cuda(rs), cuda(rl),
                                                cuda(nr), T, B, key.to(dev()), key.to(dev()),
                                                kc, vc, max_num_tokens=n_max, err=e2)
        assert int(e2.item()) == 0, kind
        assert np.array_equal(sf.cpu().numpy(), exp_s), kind
        ek = np.zeros((1, B, T, H, D), np.uint16)
        ev = ek.copy()
        assert oracle.cache_write(bits(key), bits(key), ek, ev, exp_s[:R], B, T) == 0
        assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev), kind


def test_many_requests_qsl_in_global_memory():
    rng = np.random.default_rng(7)
    R, T = 9000, 16
    lens = rng.integers(0, 3, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    table = rng.integers(0, 500, size=(R, 4)).astype(np.int32)
    pos = rng.integers(0, 64, size=N).astype(np.int64)
    exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, N + 7, T, 500)
    s, e = run_paged(q, pos, table, N, N + 7, T, 500)
    assert e == exp_e and np.array_equal(s, exp_s)
    rs = table.copy()
    rl = np.ones_like(rs)
    nr = np.full(R, 4, np.int32)
    exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N + 7, T, 500)
    s, e = run_range(q, pos, rs, rl, nr, N, N + 7, T, 500)
    assert e == exp_e and np.array_equal(s, exp_s)


def test_malformed_qsl_sets_error_and_stays_in_bounds():
    table = np.array([[1, 2], [3, 4]], np.int32)
    q = [0, 5, 2]
    pos = np.arange(5, dtype=np.int64)
    s, e = run_paged(q, pos, table, 5, 6, 16, 8)
    _, exp_e = oracle.slot_mapping_paged(q, pos, table, 5, 6, 16, 8)
    assert e == exp_e and e & kv.ERR_BITS["BAD_QSL"]
    assert s[5] == -1 and all(x == -1 or 16 <= x < 8 * 16 for x in s)


def test_empty_slot_mappings():
    s, e = run_paged([0], [], np.zeros((1, 4), np.int32), 0, 7, 16, 8)
    assert e == 0 and s.tolist() == [-1] * 7
    s, e = run_paged([0, 0, 0], [], np.zeros((2, 4), np.int32), 0, 0, 16, 8)
    assert e == 0 and len(s) == 0
    s, e = run_paged([0, 2, 1], [], np.zeros((2, 4), np.int32), 0, 0, 16, 8)
    assert e == kv.ERR_BITS["BAD_QSL"]
    z = np.zeros((1, 4), np.int32)
    s, e = run_range([0], [], z, z, [0], 0, 3, 16, 8)
    assert e == 0 and s.tolist() == [-1] * 3
    s, e = run_range([0, 0], [], z, z, [9], 0, 0, 16, 8)
    assert e == kv.ERR_BITS["BAD_RANGE"]


# ------------------------------------------------------------------- write


@pytest.mark.parametrize("H,D,L", [(8, 64, 1), (8, 128, 3), (1, 8, 2), (1, 128, 1), (16, 128, 2),
                                   (32, 128, 1), (2, 72, 1)])
def test_write_random_parity(H, D, L):
    rng = np.random.default_rng(H * 1000 + D + L)
    B, T, N = 37, 4, 61
    slots = rng.permutation(np.arange(0, B * T))[:N].astype(np.int64)
    slots[rng.random(N) < 0.15] = -1
    slots[rng.integers(0, N)] = B * T + 5
    slots[rng.integers(0, N)] = 1  # inside the null block
    key = wl.bf16_normal((L, N, H, D), 30)
    val = wl.bf16_normal((L, N, H, D), 31)
    kc = wl.bf16_normal((L, B, T, H, D), 32)
    vc = wl.bf16_normal((L, B, T, H, D), 33)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_e = oracle.cache_write(bits(key), bits(val), ek, ev, slots, B, T)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    kv.kv_cache_write(key.to(dev()), val.to(dev()), kc_d, vc_d, cuda(slots), err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)


def test_write_nothing_to_do():
    kc = torch.zeros((1, 4, 16, 8, 64), dtype=torch.bfloat16, device=dev())
    key = torch.zeros((1, 0, 8, 64), dtype=torch.bfloat16, device=dev())
    e = err_word()
    kv.kv_cache_write(key, key, kc, kc.clone(), torch.zeros(0, dtype=torch.int64, device=dev()),
                      err=e)
    assert int(e.item()) == 0 and int(kc.abs().sum().item()) == 0


# ------------------------------------------------------------------ gather


@pytest.mark.parametrize("bulk", [False, True])
# 4091-4095 requests: the offsets alone fit the 48 KiB of shared memory a
# launch gets by default, but not together with the kernel's static shared
# memory, so the launch must opt in to more
@pytest.mark.parametrize("seed,R,H,D", [(0, 1, 8, 128), (1, 5, 8, 64), (2, 300, 1, 8),
                                        (3, 4096, 1, 16), (4, 17, 16, 128), (5, 9, 2, 72),
                                        (6, 4093, 1, 8), (7, 4091, 1, 8), (8, 4095, 1, 8)])
def test_gather_random_parity(seed, R, H, D, bulk):
    if bulk and R > kv.MAX_GATHER_REQS // 2:
        pytest.skip("the bulk gather takes at most 2048 requests")
    rng = np.random.default_rng(4000 + seed)
    T, B, L, stride = 8, 50, 2, 6
    table = rng.integers(-1, B + 2, size=(R, stride)).astype(np.int32)
    table[rng.random(table.shape) < 0.2] = 0
    g0 = rng.integers(-1, stride * T, size=R).astype(np.int32)
    g1 = (g0 + rng.integers(-2, 20, size=R)).astype(np.int32)
    total = int(np.where((g0 >= 0) & (g1 >= g0), g1 - g0, 0).sum())
    out_rows = max(0, total - int(rng.integers(0, 3))) if seed % 2 else total + 3
    kc = wl.bf16_normal((L, B, T, H, D), 40 + seed)
    vc = wl.bf16_normal((L, B, T, H, D), 50 + seed)
    layer = seed % L
    ko = np.full((out_rows, H, D), 0x1234, np.uint16)
    vo = np.full((out_rows, H, D), 0x4321, np.uint16)
    exp_e = oracle.cache_gather(bits(kc), bits(vc), layer, B, T, table, g0, g1, ko, vo)
    k_out = torch.from_numpy(ko.view(np.int16).copy()).view(torch.bfloat16).to(dev())
    v_out = torch.from_numpy(vo.view(np.int16).copy()).view(torch.bfloat16).to(dev())
    e = err_word()
    kv.kv_cache_gather(kc.to(dev()), vc.to(dev()), cuda(table), cuda(g0), cuda(g1), layer=layer,
                       k_out=k_out, v_out=v_out, out_rows=out_rows, err=e, bulk=bulk)
    assert int(e.item()) == exp_e
    assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)


def test_gather_padding_rows_give_nothing():
    kc = wl.bf16_normal((1, 8, 16, 8, 128), 60).to(dev())
    table = torch.zeros((128, 64), dtype=torch.int32, device=dev())
    zeros = torch.zeros(128, dtype=torch.int32, device=dev())
    out = torch.empty((0, 8, 128), dtype=torch.bfloat16, device=dev())
    e = err_word()
    kv.kv_cache_gather(kc, kc, table, zeros, zeros, k_out=out, v_out=out, out_rows=0, err=e)
    assert int(e.item()) == 0


# ------------------------------------------------------------------ expand


@pytest.mark.parametrize("k,extra", [(1, 0), (2, 0), (2, 3), (3, 1), (4, 4), (8, 0)])
def test_expand_random_parity(k, extra):
    rng = np.random.default_rng(5000 + k * 10 + extra)
    R, Ms = 37, 19
    mgr = rng.integers(-2, 1 << 20, size=(R, Ms)).astype(np.int32)
    mgr[rng.random(mgr.shape) < 0.3] = 0
    mgr[0, 0] = (1 << 31) // k if k > 1 else mgr[0, 0]
    Ks = Ms * k + extra
    exp, exp_e = oracle.expand_kernel_blocks(mgr, 16 * k, 16, Ks)
    e = err_word()
    out = kv.kv_expand_kernel_blocks(cuda(mgr), 16 * k, 16,
                                     kernel_table=torch.full((R, Ks), 77, dtype=torch.int32,
                                                             device=dev()), err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(out.cpu().numpy(), exp)


@pytest.mark.parametrize("n_max", [1000, 150_000, 400_000, 700_000, 1_300_000, 2_600_000])
def test_slot_mapping_tile_variants(n_max):
    """Larger batches switch to 4 tokens per thread (paged) and 4, then 8
    (range); results are unchanged."""
    rng = np.random.default_rng(n_max)
    T, R = 16, 37
    lens = rng.multinomial(n_max - 5, np.ones(R) / R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    stride = wl.table_stride_for(int(lens.max()) // T + 2, T)
    B = R * stride + 1
    table = rng.permutation(np.arange(1, B)).astype(np.int32)[:R * stride].reshape(R, stride)
    pos = np.concatenate([np.arange(n, dtype=np.int64) for n in lens])
    exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, n_max, T, B)
    s, e = run_paged(q, pos, table, N, n_max, T, B)
    assert e == exp_e == 0 and np.array_equal(s, exp_s)
    # the same layout as one range per table row
    rs = table[:, :1].copy()
    rl = np.ones((R, 1), np.int32)
    nr = np.ones(R, np.int32)
    exp_r, exp_re = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, n_max, T, B)
    sr, er = run_range(q, pos, rs, rl, nr, N, n_max, T, B)
    assert er == exp_re and np.array_equal(sr, exp_r)


# ------------------------------------------- context-parallel slot mapping


@pytest.mark.parametrize("W,I,T", [(1, 1, 16), (2, 1, 16), (4, 4, 16), (8, 2, 16), (3, 2, 4),
                                   (2, 16, 16), (4, 1, 32)])
def test_cp_slot_mapping_parity_and_partition(W, I, T):
    rng = np.random.default_rng(12000 + W * 100 + I * 10 + T)
    R, stride = 6, 32
    B = 400
    table = rng.integers(-1, B + 2, size=(R, stride)).astype(np.int32)
    table[rng.random(table.shape) < 0.1] = 0
    lens = rng.integers(0, 300, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    pos = rng.integers(-1, stride * T * W + 50, size=N).astype(np.int64)
    owned = np.zeros(N, np.int64)
    for k in range(W):
        exp_s, exp_e = oracle.slot_mapping_paged_cp(q, pos, table, N, N + 9, T, B, W, k, I)
        e = err_word()
        s = kv.kv_slot_mapping_paged_cp(cuda(q), cuda(pos), cuda(table), T, B, W, k, I,
                                        max_num_tokens=N + 9, err=e)
        got = s.cpu().numpy()
        assert int(e.item()) == exp_e
        assert np.array_equal(got, exp_s)
        owned += got[:N] >= 0
    # every token with a valid table entry lives on exactly one rank
    ref, _ = oracle.slot_mapping_paged_cp(q, pos, table, N, N, T * W, B, 1, 0, 1)
    assert np.array_equal(owned, (ref >= 0).astype(np.int64))


@pytest.mark.parametrize("W,I", [(2, 1), (4, 16)])
def test_cp_slot_mapping_long_context(W, I):
    """The context-parallel map at the long-context size (1M positions, four
    tokens per thread), every rank, through the permuted table."""
    w = wl.long_context()
    table = w.layouts["P"].table
    T, B, N = w.block_size, w.num_blocks, w.num_tokens
    owned = np.zeros(N, np.int64)
    q, pos, tab = cuda(w.qsl), cuda(w.positions), cuda(table)
    for k in range(W):
        exp_s, exp_e = oracle.slot_mapping_paged_cp(w.qsl, w.positions, table, N, N, T, B, W,
                                                    k, I)
        e = err_word()
        s = kv.kv_slot_mapping_paged_cp(q, pos, tab, T, B, W, k, I, err=e)
        got = s.cpu().numpy()
        assert int(e.item()) == exp_e
        assert np.array_equal(got, exp_s)
        owned += got >= 0
    # every token of the (fully owned) contexts lives on exactly one rank
    assert (owned == 1).all()


@pytest.mark.parametrize("bulk", [False, True])
@pytest.mark.parametrize("T,H,D,R", [(16, 32, 128, 7), (32, 8, 128, 9), (16, 8, 128, 2048),
                                     (16, 8, 128, 2049), (4, 20, 1024, 5), (16, 1, 8, 33)])
def test_gather_chunking_and_fallback(T, H, D, R, bulk):
    """Bulk-copy chunks of several rows per block (8 KiB rows: 4-row chunks;
    2 KiB rows with 32-row blocks: 2 chunks per block) and the largest request
    count it takes; rows beyond a bulk stage (40 KiB) and 2049 requests are
    refused by the bulk gather and handled by the vector gather."""
    rng = np.random.default_rng(13000 + T * 7 + H + D + R)
    B, L, stride = 24, 1, 6
    table = rng.integers(-1, B + 2, size=(R, stride)).astype(np.int32)
    table[rng.random(table.shape) < 0.15] = 0
    g0 = rng.integers(0, stride * T, size=R).astype(np.int32)
    g1 = np.minimum(g0 + rng.integers(0, 3 * T, size=R), stride * T).astype(np.int32)
    total = int((g1 - g0).sum())
    out_rows = max(0, total - 5)
    kc = wl.bf16_normal((L, B, T, H, D), 77)
    vc = wl.bf16_normal((L, B, T, H, D), 78)
    ko = np.full((out_rows, H, D), 0x2222, np.uint16)
    vo = np.full((out_rows, H, D), 0x3333, np.uint16)
    exp_e = oracle.cache_gather(bits(kc), bits(vc), 0, B, T, table, g0, g1, ko, vo)
    k_out = torch.full((out_rows, H, D), 0x2222, dtype=torch.int16).view(torch.bfloat16).to(dev())
    v_out = torch.full((out_rows, H, D), 0x3333, dtype=torch.int16).view(torch.bfloat16).to(dev())
    e = err_word()
    args = (kc.to(dev()), vc.to(dev()), cuda(table), cuda(g0), cuda(g1))
    if bulk and (H * D * 2 > 32768 or R > 2048):
        with pytest.raises(kv.KVError) as ei:
            kv.kv_cache_gather(*args, k_out=k_out, v_out=v_out, out_rows=out_rows, err=e, bulk=True)
        assert ei.value.status == kv.KV_EUNSUPPORTED
        return
    kv.kv_cache_gather(*args, k_out=k_out, v_out=v_out, out_rows=out_rows, err=e, bulk=bulk)
    assert int(e.item()) == exp_e
    assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)


@pytest.mark.parametrize("T", [3, 12, 24])
def test_non_power_of_two_block_sizes_and_huge_positions(T):
    """Block sizes that are not powers of two take the division path, and
    positions past 2^31 its 64-bit branch (they fall past every table row)."""
    rng = np.random.default_rng(14000 + T)
    R, stride, B = 9, 40, 300
    table = rng.integers(0, B, size=(R, stride)).astype(np.int32)
    lens = rng.integers(0, 90, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    pos = rng.integers(0, stride * T + 30, size=N).astype(np.int64)
    big = rng.random(N) < 0.1
    pos[big] = rng.integers(1 << 31, 1 << 33, size=int(big.sum()))
    exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, N + 3, T, B)
    s, e = run_paged(q, pos, table, N, N + 3, T, B)
    assert e == exp_e and np.array_equal(s, exp_s)
    rs = rng.integers(1, B - 10, size=(R, 4)).astype(np.int32)
    rl = rng.integers(1, 10, size=(R, 4)).astype(np.int32)
    nr = rng.integers(0, 5, size=R).astype(np.int32)
    exp_r, exp_re = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N + 3, T, B)
    sr, er = run_range(q, pos, rs, rl, nr, N, N + 3, T, B)
    assert er == exp_re and np.array_equal(sr, exp_r)
    for W, I in ((2, 1), (3, T)):
        exp_c, exp_ce = oracle.slot_mapping_paged_cp(q, pos, table, N, N + 3, T, B, W, 1, I)
        e_ = err_word()
        sc = kv.kv_slot_mapping_paged_cp(cuda(q), cuda(pos), cuda(table), T, B, W, 1, I,
                                         max_num_tokens=N + 3, err=e_)
        assert int(e_.item()) == exp_ce and np.array_equal(sc.cpu().numpy(), exp_c)
    # write and gather with this block size
    H, D, L = 2, 64, 2
    live = exp_s[:N][exp_s[:N] >= 0]
    uniq, first = np.unique(live, return_index=True)
    slots = np.full(N, -1, np.int64)
    idx = np.nonzero(exp_s[:N] >= 0)[0][first]
    slots[idx] = uniq
    key = wl.bf16_normal((L, N, H, D), 140 + T)
    kc = wl.bf16_normal((L, B, T, H, D), 150 + T)
    ek, ev = bits(kc).copy(), bits(kc).copy()
    exp_we = oracle.cache_write(bits(key), bits(key), ek, ev, slots, B, T)
    kc_d, vc_d = kc.to(dev()), kc.clone().to(dev())
    e_ = err_word()
    kv.kv_cache_write(key.to(dev()), key.to(dev()), kc_d, vc_d, cuda(slots), err=e_)
    assert int(e_.item()) == exp_we
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)
    g0 = rng.integers(0, stride * T // 2, size=R).astype(np.int32)
    g1 = (g0 + rng.integers(0, stride * T // 2, size=R)).astype(np.int32)
    rows = int((g1 - g0).sum())
    for bulk in (False, True):
        ko = np.zeros((rows, H, D), np.uint16)
        vo = np.zeros((rows, H, D), np.uint16)
        exp_ge = oracle.cache_gather(ek, ev, 1, B, T, table, g0, g1, ko, vo)
        e_ = err_word()
        k_out, v_out = kv.kv_cache_gather(kc_d, vc_d, cuda(table), cuda(g0), cuda(g1), layer=1,
                                          out_rows=rows, err=e_, bulk=bulk)
        assert int(e_.item()) == exp_ge
        assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)


@pytest.mark.parametrize("T", [16, 24])
def test_slot_mapping_with_slots_past_int32(T):
    """A pool of 2^28 blocks gives slots past 2^31: the paged map takes its
    64-bit path (the 32-bit one needs num_blocks * block_size to fit int32),
    the range and context-parallel maps compute in 64 bits throughout."""
    rng = np.random.default_rng(15000 + T)
    B = 1 << 28
    R, stride = 6, 64
    table = rng.integers(0, B, size=(R, stride)).astype(np.int32)
    lens = rng.integers(1, 200, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    pos = rng.integers(0, stride * T, size=N).astype(np.int64)
    exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, N, T, B)
    assert exp_s.max() > (1 << 31)
    s, e = run_paged(q, pos, table, N, N, T, B)
    assert e == exp_e and np.array_equal(s, exp_s)
    rs = rng.integers(1 << 27, B - 100, size=(R, 3)).astype(np.int32)
    rl = rng.integers(1, 30, size=(R, 3)).astype(np.int32)
    nr = np.full(R, 3, np.int32)
    exp_r, exp_re = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N, T, B)
    sr, er = run_range(q, pos, rs, rl, nr, N, N, T, B)
    assert er == exp_re and np.array_equal(sr, exp_r)
    exp_c, exp_ce = oracle.slot_mapping_paged_cp(q, pos, table, N, N, T, B, 2, 0, 1)
    e_ = err_word()
    sc = kv.kv_slot_mapping_paged_cp(cuda(q), cuda(pos), cuda(table), T, B, 2, 0, 1, err=e_)
    assert int(e_.item()) == exp_ce and np.array_equal(sc.cpu().numpy(), exp_c)


@pytest.mark.parametrize("R,lo,hi,pad", [(5000, 20, 100, 0), (3000, 40, 160, 700_000),
                                         (12000, 1, 60, 0)])
def test_range_many_short_requests_past_one_wave(R, lo, hi, pad):
    """Batches beyond one wave of one token per thread made of many short
    requests (decode-like chunks): the range map that walks each request's
    ranges per lane, at four and eight tokens per thread, and the paged map
    through the expanded table."""
    rng = np.random.default_rng(17000 + R + pad)
    T, S = 16, 8
    lens = rng.integers(lo, hi, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    nr = rng.integers(1, S + 1, size=R).astype(np.int32)
    rl = rng.integers(1, 5, size=(R, S)).astype(np.int32)
    rs = np.zeros((R, S), np.int32)
    cursor = 1
    for r in range(R):
        for i in range(S):
            rs[r, i] = cursor
            cursor += int(rl[r, i]) + int(rng.integers(0, 3))
    B = cursor + 1
    rl[rng.random((R, S)) < 0.01] = 0      # a few empty ranges
    nr[rng.integers(0, R, size=3)] = S + 1  # a few malformed rows
    pos = np.concatenate([rng.integers(0, 40 * T, size=int(n)) for n in lens]).astype(np.int64)
    pos[rng.integers(0, N, size=5)] = -1
    n_max = N + pad
    exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, n_max, T, B)
    s, e = run_range(q, pos, rs, rl, nr, N, n_max, T, B)
    assert e == exp_e and np.array_equal(s, exp_s)
    stride = wl.table_stride_for(int(rl.sum(axis=1).max()), T)
    table = oracle.table_from_ranges(rs, rl, np.minimum(nr, S), stride)
    exp_p, exp_pe = oracle.slot_mapping_paged(q, pos, table, N, n_max, T, B)
    sp, ep = run_paged(q, pos, table, N, n_max, T, B)
    assert ep == exp_pe and np.array_equal(sp, exp_p)


def test_range_staged_with_qsl_in_global_memory():
    """More requests than query_start_loc entries fit in shared memory (9000)
    on a batch large enough for the staged range map (2.2M tokens, eight per
    thread): the tile's requests are found by searching global memory."""
    rng = np.random.default_rng(19000)
    T, R, S = 16, 9000, 6
    lens = rng.integers(150, 350, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    nr = rng.integers(1, S + 1, size=R).astype(np.int32)
    rl = rng.integers(1, 12, size=(R, S)).astype(np.int32)
    rs = rng.integers(1, 2_000_000, size=(R, S)).astype(np.int32)
    nr[rng.integers(0, R, size=4)] = S + 2
    pos = np.concatenate([int(rng.integers(0, 200)) + np.arange(int(n)) for n in lens])
    pos = pos.astype(np.int64)
    B = 2_000_020
    exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N, T, B)
    s, e = run_range(q, pos, rs, rl, nr, N, N, T, B)
    assert N > 2_000_000 and e == exp_e
    assert np.array_equal(s, exp_s)


def test_slot_maps_at_the_token_limit():
    """max_num_tokens = KV_MAX_TOKENS (2^31 - 65536, a 17 GB slot buffer):
    the largest launch every slot map accepts.  The last tiles' token indices
    come within one tile of 2^31, and the fused calls' grids (one CTA per 8
    tokens) pass 2^32 threads, so every grid-wide index must be 64-bit.  The
    real tokens match the oracle and every padded slot reads PAD (checked on
    the device)."""
    rng = np.random.default_rng(31000)
    T, B, H, D, R = 16, 512, 1, 8, 4
    lens = np.array([250, 1, 0, 300])
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(qsl[-1])
    pos = np.concatenate([np.arange(n) + int(rng.integers(0, 64)) for n in lens]).astype(np.int64)
    stride = 32
    perm = rng.permutation(np.arange(1, B))
    table = perm[:R * stride].reshape(R, stride).astype(np.int32)
    rs, rl = table.copy(), np.ones_like(table)  # one range per block
    nr = np.full(R, stride, np.int32)
    n_max = kv.MAX_TOKENS
    slot = torch.empty(n_max, dtype=torch.int64, device=dev())
    exp, exp_e = oracle.slot_mapping_paged(qsl, pos, table, N, N, T, B)
    exp_r, exp_re = oracle.slot_mapping_range(qsl, pos, rs, rl, nr, N, N, T, B)
    assert np.array_equal(exp, exp_r) and exp_e == exp_re == 0
    exp_cp, exp_cpe = oracle.slot_mapping_paged_cp(qsl, pos, table, N, N, T, B, 2, 1, 4)
    key = wl.bf16_normal((1, N, H, D), 310).to(dev())
    kc = torch.zeros((1, B, T, H, D), dtype=torch.bfloat16, device=dev())
    vc = torch.zeros_like(kc)
    calls = {
        "paged": (lambda e: kv.kv_slot_mapping_paged(cuda(qsl), cuda(pos), cuda(table), T, B,
                                                     max_num_tokens=n_max, slot_mapping=slot,
                                                     err=e), exp),
        "range": (lambda e: kv.kv_slot_mapping_range(cuda(qsl), cuda(pos), cuda(rs), cuda(rl),
                                                     cuda(nr), T, B, max_num_tokens=n_max,
                                                     slot_mapping=slot, err=e), exp),
        "cp": (lambda e: kv.kv_slot_mapping_paged_cp(cuda(qsl), cuda(pos), cuda(table), T, B, 2,
                                                     1, 4, max_num_tokens=n_max,
                                                     slot_mapping=slot, err=e), exp_cp),
        "paged_write": (lambda e: kv.kv_slot_mapping_paged_write(
            cuda(qsl), cuda(pos), cuda(table), T, B, key, key, kc, vc, max_num_tokens=n_max,
            slot_mapping=slot, err=e), exp),
        "range_write": (lambda e: kv.kv_slot_mapping_range_write(
            cuda(qsl), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B, key, key, kc, vc,
            max_num_tokens=n_max, slot_mapping=slot, err=e), exp),
    }
    for name, (call, want) in calls.items():
        slot[:N].fill_(12345)
        slot[-4096:].fill_(12345)
        e = err_word()
        call(e)
        torch.cuda.synchronize()
        assert int(e.item()) == 0, name
        assert np.array_equal(slot[:N].cpu().numpy(), want), name
        assert bool((slot[N:] == -1).all()), name
    ek = np.zeros((1, B, T, H, D), np.uint16)
    ev = ek.copy()
    assert oracle.cache_write(bits(key), bits(key), ek, ev, exp, B, T) == 0
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)
    del slot
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", ["paged_write", "range_write"])
def test_grid_wide_checks_on_grids_past_2_32_threads(kind):
    """The fused calls at max_num_tokens = 2^27: one CTA per 8 tokens is
    2^24 CTAs, 2^32 threads.  Their grid-wide checks (query_start_loc, and the
    range form's descriptor rows) must still visit the last requests: a
    decrease of query_start_loc near the end and a malformed last row are
    reported, exactly as the oracle reports them."""
    rng = np.random.default_rng(32000)
    T, B, H, D, R = 16, 8192, 1, 8, 5000
    n_max = 1 << 27
    qsl = np.arange(R + 1, dtype=np.int32)
    qsl[R - 2] = qsl[R - 1] + 1  # decreasing at R - 2
    pos = rng.integers(0, 4 * T, size=R).astype(np.int64)
    table = rng.integers(1, B, size=(R, 4)).astype(np.int32)
    rs, rl = table.copy(), np.ones_like(table)
    nr = np.full(R, 4, np.int32)
    nr[R - 1] = 5  # more ranges than the row holds
    if kind == "paged_write":
        _, exp_e = oracle.slot_mapping_paged(qsl, pos, table, R, R, T, B)
    else:
        _, exp_e = oracle.slot_mapping_range(qsl, pos, rs, rl, nr, R, R, T, B)
    assert exp_e & kv.ERR_BITS["BAD_QSL"]
    assert kind == "paged_write" or exp_e & kv.ERR_BITS["BAD_RANGE"]
    key = torch.zeros((1, R, H, D), dtype=torch.bfloat16, device=dev())
    kc = torch.zeros((1, B, T, H, D), dtype=torch.bfloat16, device=dev())
    vc = torch.zeros_like(kc)
    slot = torch.empty(n_max, dtype=torch.int64, device=dev())
    e = err_word()
    if kind == "paged_write":
        kv.kv_slot_mapping_paged_write(cuda(qsl), cuda(pos), cuda(table), T, B, key, key, kc, vc,
                                       max_num_tokens=n_max, slot_mapping=slot, err=e)
    else:
        kv.kv_slot_mapping_range_write(cuda(qsl), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B,
                                       key, key, kc, vc, max_num_tokens=n_max,
                                       slot_mapping=slot, err=e)
    torch.cuda.synchronize()
    got = int(e.item())
    check = kv.ERR_BITS["BAD_QSL"] | kv.ERR_BITS["BAD_RANGE"]
    assert got & check == exp_e & check
    assert bool((slot[R:] == -1).all())  # the padded tail, whatever the bad spans gave
    del slot
    torch.cuda.empty_cache()


@pytest.mark.parametrize("pad", [0, 700_000])
def test_range_lengths_past_int32(pad):
    """Ranges of 2^27 and 2^30 blocks (cumulative block counts past 2^31, so
    every scan of the lengths needs 64 bits): positions at the start of each
    range and one deep inside a huge range (its block is past the pool),
    through the range map (one token per thread, and the staged kernel on a
    long prefill), the fused range write and the range-addressed gather."""
    rng = np.random.default_rng(20000 + pad)
    T, H, D, R = 16, 1, 8, 4
    big = [(10, 5), (100, 1 << 27), (50, 3), (120, 1 << 30), (200, 1 << 30), (300, 7)]
    S = len(big)
    B = 400 * R  # request r's blocks lie in [400 r, 400 r + 400)
    rs = np.array([[st + 400 * r for st, _ in big] for r in range(R)], np.int32)
    rl = np.array([[ln for _, ln in big]] * R, np.int32)
    nr = np.full(R, S, np.int32)
    ends = np.cumsum([ln for _, ln in big])
    starts = ends - np.array([ln for _, ln in big])
    lbs = [int(starts[i]) + j for i in range(S) for j in range(6)]
    lbs += [int(starts[1]) + 5000, int(ends[-1]) + 2]  # past the pool; past every range
    pos1 = np.array([lb * T + int(rng.integers(0, T)) for lb in lbs], np.int64)
    reps = 6000 if pad else 1  # a long prefill of the same positions: the staged kernel
    q = np.concatenate([[0], np.cumsum([len(lbs) * reps] * R)]).astype(np.int32)
    pos = np.tile(pos1, reps * R)
    N = int(q[-1])
    exp_s, exp_e = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, N + pad, T, B)
    s, e = run_range(q, pos, rs, rl, nr, N, N + pad, T, B)
    assert e == exp_e and np.array_equal(s, exp_s)
    assert exp_e == kv.ERR_BITS["BAD_BLOCK"] and (exp_s[:N] >= 0).sum() == 6 * S * R * reps
    if pad:
        return
    assert len(np.unique(exp_s[exp_s >= 0])) == 6 * S * R  # the write below has no races
    # fused range write on a small cache
    key = wl.bf16_normal((1, N, H, D), 210)
    kc = wl.bf16_normal((1, B, T, H, D), 211)
    ek, ev = bits(kc).copy(), bits(kc).copy()
    exp_we = oracle.cache_write(bits(key), bits(key), ek, ev, exp_s[:N], B, T)
    kc_d, vc_d = kc.to(dev()), kc.clone().to(dev())
    e2 = err_word()
    sf = kv.kv_slot_mapping_range_write(cuda(q), cuda(pos), cuda(rs), cuda(rl), cuda(nr), T, B,
                                        key.to(dev()), key.to(dev()), kc_d, vc_d, err=e2)
    assert int(e2.item()) == exp_e | exp_we
    assert np.array_equal(sf.cpu().numpy(), exp_s[:N])
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)
    # range-addressed gather: spans at the start of the 2^27-block range
    # (rows), deep inside it (blocks past the pool: zero rows) and in range 0
    g0 = np.array([int(starts[1]) * T, 2_000_000_000, 0, int(starts[1]) * T + 3], np.int32)
    g1 = (g0 + np.array([40, 33, 90, 17])).astype(np.int32)
    rows = int((g1.astype(np.int64) - g0).sum())
    src, exp_ge = oracle.gather_rows_range(0, B, T, rs, rl, nr, g0, g1, rows)
    e3 = err_word()
    ko, vo = kv.kv_cache_gather_range(kc_d, vc_d, cuda(rs), cuda(rl), cuda(nr), cuda(g0),
                                      cuda(g1), out_rows=rows, err=e3)
    assert int(e3.item()) == exp_ge and exp_ge == kv.ERR_BITS["BAD_BLOCK"]
    kd = bits(kc_d).reshape(-1, H * D)
    exp_rows = np.where((src >= 0)[:, None], kd[np.maximum(src, 0)], 0)
    assert (src >= 0).sum() == 40 + 90 + 17
    assert np.array_equal(bits(ko).reshape(-1, H * D), exp_rows)


@pytest.mark.parametrize("T", [16, 24])
def test_paged_wide_slots_four_tokens_per_thread(T):
    """Slots past 2^31 on a batch beyond one wave (the paged map's 64-bit
    form at four tokens per thread)."""
    rng = np.random.default_rng(18000 + T)
    B = 1 << 28
    R, stride = 40, 128
    table = rng.integers(0, B, size=(R, stride)).astype(np.int32)
    table[rng.random(table.shape) < 0.05] = 0
    lens = rng.integers(8000, 12000, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])
    pos = rng.integers(-1, stride * T + 30, size=N).astype(np.int64)
    exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, N + 3, T, B)
    assert exp_s.max() > (1 << 31) and N > 320_000
    s, e = run_paged(q, pos, table, N, N + 3, T, B)
    assert e == exp_e and np.array_equal(s, exp_s)


@pytest.mark.parametrize("L,N", [(1, 40003), (3, 13333)])
def test_write_grouped_path(L, N):
    """Batches of tens of thousands of rows take the four-rows-per-warp write;
    token counts not a multiple of four, PAD, null-block and bad slots included."""
    rng = np.random.default_rng(16000 + N)
    T, H, D = 16, 1, 64
    B = -(-N // T) + 40
    slots = rng.permutation(np.arange(T, B * T))[:N].astype(np.int64)
    slots[rng.random(N) < 0.05] = -1
    slots[rng.integers(0, N, size=7)] = rng.integers(0, T, size=7)  # null block
    slots[rng.integers(0, N, size=5)] = B * T + 3                   # past the pool
    # keep the valid slots unique (the write races on duplicates)
    seen = set()
    for i in range(N):
        if slots[i] >= T and slots[i] < B * T:
            if slots[i] in seen:
                slots[i] = -1
            seen.add(int(slots[i]))
    key = wl.bf16_normal((L, N, H, D), 160 + L)
    val = wl.bf16_normal((L, N, H, D), 170 + L)
    kc = wl.bf16_normal((L, B, T, H, D), 180 + L)
    vc = wl.bf16_normal((L, B, T, H, D), 190 + L)
    ek, ev = bits(kc).copy(), bits(vc).copy()
    exp_e = oracle.cache_write(bits(key), bits(val), ek, ev, slots, B, T)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    e = err_word()
    kv.kv_cache_write(key.to(dev()), val.to(dev()), kc_d, vc_d, cuda(slots), err=e)
    assert int(e.item()) == exp_e
    assert np.array_equal(bits(kc_d), ek) and np.array_equal(bits(vc_d), ev)
