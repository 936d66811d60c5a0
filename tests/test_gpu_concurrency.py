"""The library keeps no state between calls: host threads, each launching on
its own CUDA stream, run slot maps, writes and gathers at the same time
(ctypes releases the interpreter lock around every C call), and every result
still matches the oracle bit for bit."""
import threading

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_39_gb300 as kv
from paged_kv_cache_39_gb300 import workloads as wl
from gpu_helpers import bits, dev, random_slot_case

pytestmark = pytest.mark.gpu

THREADS, CASES = 4, 48


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    torch.cuda.set_device(dev())
    yield
    torch.cuda.synchronize()


def _cases():
    out = []
    for c in range(CASES):
        rng = np.random.default_rng(18000 + c)
        T, R, q, N, n_max, stride, B, table, pos = random_slot_case(rng)
        exp_s, exp_e = oracle.slot_mapping_paged(q, pos, table, N, n_max, T, B)
        # every table entry, null and bad ones included, as a range of one block
        rs = table.copy()
        rl = np.ones_like(table)
        nr = np.full(table.shape[0], table.shape[1], np.int32)
        exp_r, exp_re = oracle.slot_mapping_range(q, pos, rs, rl, nr, N, n_max, T, B)
        out.append(dict(T=T, B=B, q=q, pos=pos, table=table, rs=rs, rl=rl, nr=nr, N=N,
                        n_max=n_max, exp=(exp_s, exp_e, exp_r, exp_re)))
    return out


def test_threads_on_their_own_streams():
    cases = _cases()
    # a shared read-only cache for the gathers, and per-thread caches for writes
    L, Bc, Tc, H, D = 2, 64, 16, 2, 64
    kc = wl.bf16_normal((L, Bc, Tc, H, D), 180)
    vc = wl.bf16_normal((L, Bc, Tc, H, D), 181)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    g_rng = np.random.default_rng(181)
    g_table = g_rng.integers(0, Bc, size=(5, 8)).astype(np.int32)
    g0 = np.array([0, 3, 17, 40, 127], np.int32)
    g1 = np.array([128, 3, 60, 41, 128], np.int32)
    out_rows = int((g1 - g0).sum())
    ko = np.zeros((out_rows, H, D), np.uint16)
    vo = np.zeros((out_rows, H, D), np.uint16)
    exp_ge = oracle.cache_gather(bits(kc), bits(vc), 1, Bc, Tc, g_table, g0, g1, ko, vo)
    wkey = wl.bf16_normal((L, 40, H, D), 182)
    w_slots = np.random.default_rng(183).permutation(np.arange(Tc, Bc * Tc))[:40]
    wk, wv = bits(kc).copy(), bits(vc).copy()
    exp_we = oracle.cache_write(bits(wkey), bits(wkey), wk, wv, w_slots, Bc, Tc)

    torch.cuda.synchronize()  # shared inputs in place before any side stream reads them
    results, errors = {}, []

    def worker(w):
        try:
            torch.cuda.set_device(dev())
            s = torch.cuda.Stream(device=dev())
            with torch.cuda.stream(s):
                mine = {}
                kcw, vcw = kc_d.clone(), vc_d.clone()
                for i in range(w, CASES, THREADS):
                    c = cases[i]
                    t = {k: torch.from_numpy(np.ascontiguousarray(c[k])).to(dev())
                         for k in ("q", "pos", "table", "rs", "rl", "nr")}
                    e_p = torch.zeros(1, dtype=torch.int32, device=dev())
                    e_r = torch.zeros(1, dtype=torch.int32, device=dev())
                    sp = kv.kv_slot_mapping_paged(t["q"], t["pos"], t["table"], c["T"], c["B"],
                                                  max_num_tokens=c["n_max"], num_tokens=c["N"],
                                                  err=e_p)
                    sr = kv.kv_slot_mapping_range(t["q"], t["pos"], t["rs"], t["rl"], t["nr"],
                                                  c["T"], c["B"], max_num_tokens=c["n_max"],
                                                  num_tokens=c["N"], err=e_r)
                    e_g = torch.zeros(1, dtype=torch.int32, device=dev())
                    gk, gv = kv.kv_cache_gather(kc_d, vc_d, torch.from_numpy(g_table).to(dev()),
                                                torch.from_numpy(g0).to(dev()),
                                                torch.from_numpy(g1).to(dev()), layer=1,
                                                out_rows=out_rows, err=e_g, bulk=bool(i % 2))
                    mine[i] = (sp, e_p, sr, e_r, gk, gv, e_g)
                e_w = torch.zeros(1, dtype=torch.int32, device=dev())
                kv.kv_cache_write(wkey.to(dev()), wkey.to(dev()), kcw, vcw,
                                  torch.from_numpy(w_slots).to(dev()), err=e_w)
            s.synchronize()
            results[w] = (mine, (kcw, vcw, e_w))
        except Exception as exc:  # reported by the main thread
            errors.append(repr(exc))

    threads = [threading.Thread(target=worker, args=(w,)) for w in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for w in range(THREADS):
        mine, (kcw, vcw, e_w) = results[w]
        assert int(e_w.item()) == exp_we
        assert np.array_equal(bits(kcw), wk) and np.array_equal(bits(vcw), wv)
        for i, (sp, e_p, sr, e_r, gk, gv, e_g) in mine.items():
            exp_s, exp_e, exp_r, exp_re = cases[i]["exp"]
            assert np.array_equal(sp.cpu().numpy(), exp_s) and int(e_p.item()) == exp_e, i
            assert np.array_equal(sr.cpu().numpy(), exp_r) and int(e_r.item()) == exp_re, i
            assert int(e_g.item()) == exp_ge
            assert np.array_equal(bits(gk), ko) and np.array_equal(bits(gv), vo), i
