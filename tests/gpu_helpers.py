"""Helpers shared by the GPU parity tests (no method arithmetic here: the
expected rows come from the oracle)."""
import numpy as np
import torch

import oracle


def dev():
    return torch.device("cuda:0")


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a bf16 tensor as a host uint16 array."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def err_word():
    return torch.zeros(1, dtype=torch.int32, device=dev())


def free_bytes() -> int:
    free, _ = torch.cuda.mem_get_info(dev())
    return int(free)


def rows_view(t: torch.Tensor, row_elems: int) -> torch.Tensor:
    return t.view(-1, row_elems).view(torch.int16)


def device_rows_equal(out: torch.Tensor, cache: torch.Tensor, src_rows: np.ndarray,
                      row_elems: int, chunk: int = 1 << 18) -> bool:
    """Every output row o equals cache row src_rows[o] (or is zero when
    src_rows[o] == -1).  The source rows come from the oracle; torch only
    moves the bytes for the comparison."""
    o_rows = rows_view(out, row_elems)
    c_rows = rows_view(cache, row_elems)
    n = len(src_rows)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        idx = torch.from_numpy(src_rows[s:e]).to(out.device)
        zero = idx < 0
        exp = c_rows.index_select(0, idx.clamp_min(0))
        exp[zero] = 0
        if not torch.equal(o_rows[s:e], exp):
            return False
    return True


def sample_host_check(out: torch.Tensor, cache_host_rows, src_rows: np.ndarray, row_elems: int,
                      sample: np.ndarray) -> None:
    """Host-side check of sampled output rows against cache rows fetched one by one."""
    o_rows = rows_view(out, row_elems)
    got = o_rows[torch.from_numpy(sample).to(out.device)].cpu().numpy().view(np.uint16)
    for k, o in enumerate(sample):
        src = int(src_rows[o])
        exp = np.zeros(row_elems, np.uint16) if src < 0 else cache_host_rows(src)
        assert np.array_equal(got[k], exp), f"output row {o} (source {src}) differs"


FILL = 0x3C01  # bf16 bit pattern of the caches before the write (1.0078125)
SAMPLE = 2048


def filled_cache(shape):
    return torch.full(shape, FILL, dtype=torch.int16, device=dev()).view(torch.bfloat16)


def check_write(key, val, kc, vc, slots_host, L, N, B, T, E, rng):
    """Oracle destination rows; full device check; sampled host check; untouched rows."""
    dest, exp_e = oracle.write_rows(slots_host, N, L, B, T)
    flat_dest = dest.reshape(-1)
    valid = np.nonzero(flat_dest >= 0)[0]
    # every written row holds its token's K/V row
    src_k = rows_view(key, E)
    src_v = rows_view(val, E)
    kr, vr = rows_view(kc, E), rows_view(vc, E)
    for s in range(0, len(valid), 1 << 16):
        sel = torch.from_numpy(valid[s:s + (1 << 16)]).to(dev())
        drow = torch.from_numpy(flat_dest[valid[s:s + (1 << 16)]]).to(dev())
        assert torch.equal(kr.index_select(0, drow), src_k.index_select(0, sel))
        assert torch.equal(vr.index_select(0, drow), src_v.index_select(0, sel))
    # sampled host check through the oracle's per-row arithmetic
    pick = rng.choice(len(valid), size=min(SAMPLE, len(valid)), replace=False)
    for i in valid[pick][:256]:
        l, t = divmod(int(i), N)
        got = kr[int(flat_dest[i])].cpu().numpy().view(np.uint16)
        assert np.array_equal(got, src_k[l * N + t].cpu().numpy().view(np.uint16))
    # nothing else changed: rows differing from the fill pattern are exactly the written ones
    fill64 = torch.tensor([FILL], dtype=torch.int16).repeat(4).view(torch.int64).item()
    changed = 0
    for c in (kc, vc):
        per_layer = c.view(L, -1)
        for l in range(L):
            v64 = per_layer[l].view(torch.int16).view(-1, E).view(torch.int64)
            changed += int((v64 != fill64).any(dim=1).sum().item())
    assert changed == 2 * len(np.unique(flat_dest[valid]))
    return exp_e


# Seeded adversarial slot-map inputs: empty and zero-length requests, a
# shifted or truncated query_start_loc, untracked tokens, padding tails,
# negative and out-of-range positions, null and out-of-range table entries.
def random_slot_case(rng):
    T = int(rng.choice([1, 3, 4, 12, 16, 24, 32]))  # non-powers of two take the division paths
    R = int(rng.integers(0, 40))
    lens = rng.integers(0, 70, size=R)
    lens[rng.random(R) < 0.2] = 0
    q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    shift = int(rng.choice([0, 0, 0, 3]))
    q = q + shift
    N = int(q[-1]) + int(rng.choice([0, 0, 5]))
    if rng.random() < 0.1 and R > 0:
        q[-1] = max(q[-2], q[-1] - 2)
    n_max = N + int(rng.choice([0, 1, 300]))
    stride = int(rng.choice([0, 1, 8, 64]))
    B = int(rng.integers(1, 300))
    table = rng.integers(-1, B + 3, size=(max(R, 1), stride)).astype(np.int32)
    table[rng.random(table.shape) < 0.2] = 0
    pos = rng.integers(-2, max(stride, 1) * T + 20, size=N).astype(np.int64)
    return T, R, q.astype(np.int32), N, n_max, stride, B, table, pos


def check_write_vs_before(key, val, kc, vc, kc0, vc0, slots_host, L, N, B, T, E, rng):
    """check_write for caches of random contents.  kc0/vc0 are copies taken
    before the write (consumed here): the oracle's destination rows are set in
    them to their tokens' rows, after which the written caches must equal
    them whole, so every row the write must not touch is checked too."""
    dest, exp_e = oracle.write_rows(slots_host, N, L, B, T)
    flat_dest = dest.reshape(-1)
    valid = np.nonzero(flat_dest >= 0)[0]
    src_k, src_v = rows_view(key, E), rows_view(val, E)
    kr0, vr0 = rows_view(kc0, E), rows_view(vc0, E)
    for s in range(0, len(valid), 1 << 16):
        sel = torch.from_numpy(valid[s:s + (1 << 16)]).to(dev())
        drow = torch.from_numpy(flat_dest[valid[s:s + (1 << 16)]]).to(dev())
        kr0[drow] = src_k.index_select(0, sel)
        vr0[drow] = src_v.index_select(0, sel)
    assert torch.equal(rows_view(kc, E), kr0) and torch.equal(rows_view(vc, E), vr0)
    # sampled host check through the oracle's per-row arithmetic
    kr = rows_view(kc, E)
    pick = rng.choice(len(valid), size=min(256, len(valid)), replace=False)
    for i in valid[pick]:
        l, t = divmod(int(i), N)
        got = kr[int(flat_dest[i])].cpu().numpy().view(np.uint16)
        assert np.array_equal(got, src_k[l * N + t].cpu().numpy().view(np.uint16))
    return exp_e
