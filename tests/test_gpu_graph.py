"""The hot path under CUDA-graph capture.

The pages pad slot mappings and tables so that a captured decode step stays
valid while the batch changes ("Range-addressed KV cache blocks ...", The
Innovation: stable slot-mapping values under CUDA graph capture;
"Blocktabelle", CUDA-Graph-Padding).  Every launch here is sized by host
arguments only, so a step captured once is replayed on new inputs written in
place, and every replay must match the oracle bit for bit.  The binding's
prepared calls (validated once, relaunched with cached pointers) are the
uncaptured form of the same replay and are held to the same bar."""
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


def _batch(seed, R_pad, n_max, T, B, stride):
    """A padded decode batch: 1 token per live request, padding rows empty."""
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, R_pad + 1))
    ctx = rng.integers(1, stride * T + 1, size=R)
    perm = rng.permutation(np.arange(1, B))
    table = np.zeros((R_pad, stride), np.int32)
    k = 0
    for r in range(R):
        n = -(-int(ctx[r]) // T)
        table[r, :n] = perm[k:k + n]
        k += n
    qsl = np.zeros(R_pad + 1, np.int32)
    qsl[1:R + 1] = np.arange(1, R + 1)
    qsl[R + 1:] = R
    pos = np.zeros(n_max, np.int64)
    pos[:R] = ctx - 1
    g0 = np.zeros(R_pad, np.int32)
    g1 = np.zeros(R_pad, np.int32)
    g1[:R] = ctx
    return R, qsl, pos, table, g0, g1


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("mode", ["graph", "prepared"])
@pytest.mark.parametrize("bulk", [False, True])
def test_decode_step_captured_once_replayed_on_new_batches(bulk, mode, fused):
    T, B, H, D, stride, R_pad = 16, 512, 8, 128, 16, 32
    n_max = R_pad
    out_rows = R_pad * stride * T
    # device buffers written in place between replays
    d_qsl = torch.zeros(R_pad + 1, dtype=torch.int32, device=dev())
    d_pos = torch.zeros(n_max, dtype=torch.int64, device=dev())
    d_table = torch.zeros((R_pad, stride), dtype=torch.int32, device=dev())
    d_g0 = torch.zeros(R_pad, dtype=torch.int32, device=dev())
    d_g1 = torch.zeros(R_pad, dtype=torch.int32, device=dev())
    key = torch.zeros((1, n_max, H, D), dtype=torch.bfloat16, device=dev())
    val = torch.zeros_like(key)
    kc = wl.bf16_normal((1, B, T, H, D), 500, dev())
    vc = wl.bf16_normal((1, B, T, H, D), 501, dev())
    slot = torch.empty(n_max, dtype=torch.int64, device=dev())
    k_out = torch.zeros((out_rows, H, D), dtype=torch.bfloat16, device=dev())
    v_out = torch.zeros_like(k_out)
    err = err_word()

    def slot_and_write(prepare=False):
        if fused:
            return [kv.kv_slot_mapping_paged_write(d_qsl, d_pos, d_table, T, B, key, val, kc, vc,
                                                   max_num_tokens=n_max, slot_mapping=slot,
                                                   err=err, prepare=prepare)]
        return [kv.kv_slot_mapping_paged(d_qsl, d_pos, d_table, T, B, max_num_tokens=n_max,
                                         slot_mapping=slot, err=err, prepare=prepare),
                kv.kv_cache_write(key, val, kc, vc, slot, err=err, prepare=prepare)]

    def step():
        slot_and_write()
        kv.kv_cache_gather(kc, vc, d_table, d_g0, d_g1, k_out=k_out, v_out=v_out,
                           out_rows=out_rows, err=err, bulk=bulk)

    s = torch.cuda.Stream()
    if mode == "graph":
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()  # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        replay = graph.replay
    else:
        calls = slot_and_write(prepare=True) + [
            kv.kv_cache_gather(kc, vc, d_table, d_g0, d_g1, k_out=k_out, v_out=v_out,
                               out_rows=out_rows, err=err, bulk=bulk, prepare=True),
        ]
        assert all(isinstance(c, kv.Prepared) for c in calls)
        assert calls[0].result is slot
        assert calls[-1].result[0] is k_out and calls[-1].result[1] is v_out

        def replay():  # launches on the stream current at call time
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                for c in calls:
                    c()
            torch.cuda.current_stream().wait_stream(s)

    for it, seed in enumerate([11, 12, 13]):
        R, qsl, pos, table, g0, g1 = _batch(seed, R_pad, n_max, T, B, stride)
        new_k = wl.bf16_normal((1, n_max, H, D), 600 + it, dev())
        new_v = wl.bf16_normal((1, n_max, H, D), 700 + it, dev())
        kc_before, vc_before = bits(kc).copy(), bits(vc).copy()
        d_qsl.copy_(torch.from_numpy(qsl))
        d_pos.copy_(torch.from_numpy(pos))
        d_table.copy_(torch.from_numpy(table))
        d_g0.copy_(torch.from_numpy(g0))
        d_g1.copy_(torch.from_numpy(g1))
        key.copy_(new_k)
        val.copy_(new_v)
        err.zero_()
        replay()
        torch.cuda.synchronize()
        # oracle: the same step on the host
        exp_s, e1 = oracle.slot_mapping_paged(qsl, pos, table, R, n_max, T, B)
        assert np.array_equal(slot.cpu().numpy(), exp_s)
        assert (exp_s[R:] == -1).all()  # padding tokens stay PAD on every replay
        e2 = oracle.cache_write(bits(key), bits(val), kc_before, vc_before, exp_s, B, T)
        assert np.array_equal(bits(kc), kc_before) and np.array_equal(bits(vc), vc_before)
        ko = np.zeros((out_rows, H, D), np.uint16)
        vo = np.zeros((out_rows, H, D), np.uint16)
        ko[:] = bits(k_out)  # rows past this batch's total keep earlier contents
        vo[:] = bits(v_out)
        e3 = oracle.cache_gather(kc_before, vc_before, 0, B, T, table, g0, g1, ko, vo)
        assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)
        assert int(err.item()) == (e1 | e2 | e3) == 0


def _runs(table, R_pad, stride):
    """Each request's table row as contiguous range descriptors (runs of
    consecutive block ids), padded to `stride` descriptors per request."""
    rs = np.zeros((R_pad, stride), np.int32)
    rl = np.zeros((R_pad, stride), np.int32)
    nr = np.zeros(R_pad, np.int32)
    for r in range(R_pad):
        row = table[r][table[r] != 0]
        for b in row:
            k = nr[r]
            if k and rs[r, k - 1] + rl[r, k - 1] == b:
                rl[r, k - 1] += 1
            else:
                rs[r, k], rl[r, k] = b, 1
                nr[r] += 1
    return rs, rl, nr


def test_decode_step_with_the_range_map_on_a_second_graph_branch():
    """The decode step as the benchmark captures it: paged map -> write on the
    capturing stream and the range map, into its own slot buffer, on a forked
    stream joined back before the capture ends (two branches of one graph,
    both reporting into one error word).  Replayed on new batches, both slot
    mappings and the caches match the oracle."""
    T, B, H, D, stride, R_pad = 16, 512, 8, 128, 16, 32
    n_max = R_pad
    d_qsl = torch.zeros(R_pad + 1, dtype=torch.int32, device=dev())
    d_pos = torch.zeros(n_max, dtype=torch.int64, device=dev())
    d_table = torch.zeros((R_pad, stride), dtype=torch.int32, device=dev())
    d_rs = torch.zeros((R_pad, stride), dtype=torch.int32, device=dev())
    d_rl = torch.zeros((R_pad, stride), dtype=torch.int32, device=dev())
    d_nr = torch.zeros(R_pad, dtype=torch.int32, device=dev())
    key = torch.zeros((1, n_max, H, D), dtype=torch.bfloat16, device=dev())
    val = torch.zeros_like(key)
    kc = wl.bf16_normal((1, B, T, H, D), 510, dev())
    vc = wl.bf16_normal((1, B, T, H, D), 511, dev())
    slot_p = torch.empty(n_max, dtype=torch.int64, device=dev())
    slot_r = torch.empty(n_max, dtype=torch.int64, device=dev())
    err = err_word()
    side = torch.cuda.Stream()

    def step():
        cur = torch.cuda.current_stream()
        side.wait_stream(cur)
        kv.kv_slot_mapping_paged(d_qsl, d_pos, d_table, T, B, max_num_tokens=n_max,
                                 slot_mapping=slot_p, err=err)
        kv.kv_cache_write(key, val, kc, vc, slot_p, err=err)
        with torch.cuda.stream(side):
            kv.kv_slot_mapping_range(d_qsl, d_pos, d_rs, d_rl, d_nr, T, B, max_num_tokens=n_max,
                                     slot_mapping=slot_r, err=err)
        cur.wait_stream(side)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for it, seed in enumerate([21, 22, 23]):
        R, qsl, pos, table, _, _ = _batch(seed, R_pad, n_max, T, B, stride)
        rs, rl, nr = _runs(table, R_pad, stride)
        new_k = wl.bf16_normal((1, n_max, H, D), 610 + it, dev())
        new_v = wl.bf16_normal((1, n_max, H, D), 710 + it, dev())
        kc_before, vc_before = bits(kc).copy(), bits(vc).copy()
        for d, h in ((d_qsl, qsl), (d_pos, pos), (d_table, table), (d_rs, rs), (d_rl, rl),
                     (d_nr, nr)):
            d.copy_(torch.from_numpy(h))
        key.copy_(new_k)
        val.copy_(new_v)
        slot_r.fill_(12345)
        err.zero_()
        graph.replay()
        torch.cuda.synchronize()
        exp_p, e1 = oracle.slot_mapping_paged(qsl, pos, table, R, n_max, T, B)
        exp_r, e2 = oracle.slot_mapping_range(qsl, pos, rs, rl, nr, R, n_max, T, B)
        assert np.array_equal(exp_p, exp_r)  # one layout, two descriptions of it
        assert np.array_equal(slot_p.cpu().numpy(), exp_p)
        assert np.array_equal(slot_r.cpu().numpy(), exp_r)
        e3 = oracle.cache_write(bits(key), bits(val), kc_before, vc_before, exp_p, B, T)
        assert np.array_equal(bits(kc), kc_before) and np.array_equal(bits(vc), vc_before)
        assert int(err.item()) == (e1 | e2 | e3) == 0


def test_bounded_wait_times_out_and_context_survives():
    """The bounded wait used by the bulk-copy gather gives up on a barrier that
    nothing completes, reports KV_ERR_TIMEOUT, and the next kernels run."""
    lib = kv.load()
    e = err_word()
    rc = lib.kv_diag_bounded_wait(4096, e.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(e.item()) == kv.ERR_BITS["TIMEOUT"]
    # the context is still usable: a normal call right after gives correct slots
    q = torch.tensor([0, 3], dtype=torch.int32, device=dev())
    p = torch.tensor([0, 1, 17], dtype=torch.int64, device=dev())
    t = torch.tensor([[3, 4]], dtype=torch.int32, device=dev())
    e2 = err_word()
    s = kv.kv_slot_mapping_paged(q, p, t, 16, 8, max_num_tokens=5, err=e2)
    assert s.cpu().tolist() == [48, 49, 65, -1, -1] and int(e2.item()) == 0


def test_every_prepared_call_matches_its_direct_call():
    """prepare=True on each wrapper: the relaunched call reads the inputs as
    they are at launch time (contents changed after preparing) and gives the
    direct call's outputs and error word."""
    rng = np.random.default_rng(8100)
    T, B, H, D, R, S = 16, 64, 2, 64, 6, 4
    runs = rng.permutation(np.arange(1, B)).astype(np.int32)[:R * S].reshape(R, S)
    table = runs.copy()
    rs, rl, nr = runs.copy(), np.ones((R, S), np.int32), np.full(R, S, np.int32)
    lens = rng.integers(1, 5, size=R)
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(q[-1])

    def positions():
        return np.concatenate([rng.choice(S * T, size=n, replace=False)
                               for n in lens]).astype(np.int64)

    d = {"q": cuda(q), "pos": cuda(positions()), "table": cuda(table), "rs": cuda(rs),
         "rl": cuda(rl), "nr": cuda(nr), "g0": cuda(np.zeros(R, np.int32)),
         "g1": cuda(np.full(R, S * T, np.int32)), "mgr": cuda(table[:, :2]),
         "src": cuda(np.array([table[0, 0]], np.int32)),
         "dst": cuda(np.array([table[1, 0]], np.int32))}
    key = wl.bf16_normal((1, N, H, D), 8101, dev())
    caches = {n: wl.bf16_normal((1, B, T, H, D), 8102, dev()) for n in ("p", "d")}
    outs = {n: torch.zeros((R * S * T, H, D), dtype=torch.bfloat16, device=dev())
            for n in ("p", "d")}
    calls = {
        "paged": lambda o, **k: kv.kv_slot_mapping_paged(d["q"], d["pos"], d["table"], T, B,
                                                         slot_mapping=o, **k),
        "range": lambda o, **k: kv.kv_slot_mapping_range(d["q"], d["pos"], d["rs"], d["rl"],
                                                         d["nr"], T, B, slot_mapping=o, **k),
        "cp": lambda o, **k: kv.kv_slot_mapping_paged_cp(d["q"], d["pos"], d["table"], T, B, 2,
                                                         1, 1, slot_mapping=o, **k),
        "expand": lambda o, **k: kv.kv_expand_kernel_blocks(d["mgr"], 2 * T, T,
                                                            kernel_table=o, **k),
        "table": lambda o, **k: kv.kv_table_from_ranges(d["rs"], d["rl"], d["nr"],
                                                        block_table=o, **k),
    }
    shapes = {"paged": (N,), "range": (N,), "cp": (N,), "expand": (R, 4), "table": (R, S)}
    dtypes = {"paged": torch.int64, "range": torch.int64, "cp": torch.int64,
              "expand": torch.int32, "table": torch.int32}
    prepared = {}
    for name, fn in calls.items():
        o = torch.empty(shapes[name], dtype=dtypes[name], device=dev())
        e = err_word()
        prepared[name] = (fn(o, err=e, prepare=True), o, e)
    kc, vc = caches["p"], caches["p"].clone()
    sp = torch.empty(N, dtype=torch.int64, device=dev())
    ep = err_word()
    p_write = kv.kv_slot_mapping_paged_write(d["q"], d["pos"], d["table"], T, B, key, key, kc, vc,
                                             slot_mapping=sp, err=ep, prepare=True)
    p_gather = kv.kv_cache_gather_range(kc, vc, d["rs"], d["rl"], d["nr"], d["g0"], d["g1"],
                                        k_out=outs["p"], v_out=outs["p"].clone(),
                                        out_rows=R * S * T, err=ep, prepare=True)
    p_copy = kv.kv_copy_blocks(kc, vc, d["src"], d["dst"], err=ep, bulk=True, prepare=True)
    # new contents after preparing: the prepared calls must see them
    d["pos"].copy_(cuda(positions()))
    for name, (pc, o, e) in prepared.items():
        pc()
        o2 = torch.empty_like(o)
        e2 = err_word()
        calls[name](o2, err=e2)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and int(e.item()) == int(e2.item()), name
    p_write()
    p_copy()
    p_gather()
    kd, vd = caches["d"], caches["d"].clone()
    sd = torch.empty(N, dtype=torch.int64, device=dev())
    ed = err_word()
    kv.kv_slot_mapping_paged_write(d["q"], d["pos"], d["table"], T, B, key, key, kd, vd,
                                   slot_mapping=sd, err=ed)
    kv.kv_copy_blocks(kd, vd, d["src"], d["dst"], err=ed, bulk=True)
    ko = outs["d"]
    kv.kv_cache_gather_range(kd, vd, d["rs"], d["rl"], d["nr"], d["g0"], d["g1"], k_out=ko,
                             v_out=ko.clone(), out_rows=R * S * T, err=ed)
    torch.cuda.synchronize()
    assert torch.equal(sp, sd) and int(ep.item()) == int(ed.item()) == 0
    assert torch.equal(kc.view(torch.int16), kd.view(torch.int16))
    assert torch.equal(outs["p"].view(torch.int16), ko.view(torch.int16))
