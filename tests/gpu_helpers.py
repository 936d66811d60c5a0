"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch


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
