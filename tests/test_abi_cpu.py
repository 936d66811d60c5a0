"""CPU-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects invalid host-visible arguments before launching
anything (these calls never reach the GPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvpaged.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_39_gb300 import _lib
    from paged_kv_cache_39_gb300 import build as kbuild
    variant = os.environ.get("KV_TEST_LIB")  # a sanitizer build of the same sources
    if variant:
        import ctypes
        l = ctypes.CDLL(variant)
        for name, (args, res) in _lib.SIGNATURES.items():
            getattr(l, name).argtypes = args
            getattr(l, name).restype = res
        return l
    if not os.path.exists(_lib.LIB_PATH):
        kbuild.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(kv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for fn in ["kv_slot_mapping_paged", "kv_slot_mapping_range", "kv_cache_write",
               "kv_cache_gather", "kv_expand_kernel_blocks"]:
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    from paged_kv_cache_39_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks a signature for {name}"


def test_status_strings_and_version(lib):
    assert lib.kv_abi_version() == 7
    assert lib.kv_status_string(0) == b"KV_OK"
    assert b"EINVAL" in lib.kv_status_string(-1)
    assert b"EUNSUPPORTED" in lib.kv_status_string(-2)


N = None


def test_slot_mapping_rejects_bad_arguments(lib):
    # negative sizes, num_tokens > max_num_tokens, block_size <= 0, missing pointers
    assert lib.kv_slot_mapping_paged(N, N, N, 0, -1, 0, 0, 16, 8, N, N, N) == -1
    assert lib.kv_slot_mapping_paged(N, N, N, 0, 0, 5, 4, 16, 8, N, N, N) == -1
    assert lib.kv_slot_mapping_paged(N, N, N, 0, 0, 0, 0, 0, 8, N, N, N) == -1
    assert lib.kv_slot_mapping_paged(N, N, N, 0, 0, 0, 0, 16, 0, N, N, N) == -1
    assert lib.kv_slot_mapping_paged(N, N, N, 0, 1, 0, 0, 16, 8, N, N, N) == -1  # qsl NULL
    assert lib.kv_slot_mapping_paged(N, N, N, 0, 0, 0, 4, 16, 8, N, N, N) == -1  # slots NULL
    # misaligned positions pointer
    assert lib.kv_slot_mapping_paged(N, 0x1004, N, 0, 0, 1, 1, 16, 8, 0x2000, N, N) == -1


def test_range_cap_fails_closed(lib):
    assert lib.kv_slot_mapping_range(N, N, N, N, N, 257, 0, 0, 0, 16, 8, N, N, N) == -2
    assert lib.kv_slot_mapping_range(N, N, N, N, N, -1, 0, 0, 0, 16, 8, N, N, N) == -1


def test_write_rejects_bad_arguments(lib):
    # row of 8x7 bf16 = 112 B is a multiple of 16: OK shape; 3x5 = 30 B is not
    assert lib.kv_cache_write(N, N, N, N, N, 1, 1, 8, 16, 3, 5, N, N) == -2
    assert lib.kv_cache_write(N, N, N, N, N, 1, 1, 8, 16, 8, 64, N, N) == -1  # NULL K/V
    assert lib.kv_cache_write(0x1008, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 8, 16, 8, 64, N,
                              N) == -1  # key not 16-byte aligned
    assert lib.kv_cache_write(N, N, N, N, N, 1, 1, 0, 16, 8, 64, N, N) == -1
    assert lib.kv_cache_write(N, N, N, N, N, 0, 1, 8, 16, 8, 64, N, N) == 0  # nothing to do


def test_gather_rejects_bad_arguments(lib):
    args = dict(kc=0x1000, vc=0x2000)
    assert lib.kv_cache_gather(args["kc"], args["vc"], 1, 1, 8, 16, 8, 64, N, 0, N, N, 0, N, N,
                               0, N, N) == -1  # layer out of range
    assert lib.kv_cache_gather(args["kc"], args["vc"], 0, 1, 8, 16, 8, 64, N, 0, N, N, 4097, N,
                               N, 0, N, N) == -2  # too many requests
    assert lib.kv_cache_gather(args["kc"], args["vc"], 0, 1, 8, 16, 8, 64, N, 0, N, N, 0, N, N,
                               0, N, N) == 0  # no requests
    assert lib.kv_cache_gather(args["kc"], args["vc"], 0, 1, 8, 16, 8, 64, N, 4, 0x3000, 0x4000,
                               2, N, N, 8, N, N) == -1  # table NULL with stride > 0


def test_expand_rejects_bad_arguments(lib):
    assert lib.kv_expand_kernel_blocks(N, 1, 4, 32, 12, N, 16, N, N) == -2  # non-divisor
    assert lib.kv_expand_kernel_blocks(N, 1, 4, 16, 32, N, 16, N, N) == -2
    assert lib.kv_expand_kernel_blocks(N, 1, 4, 32, 16, N, 7, N, N) == -1  # stride too small
    assert lib.kv_expand_kernel_blocks(N, 1, 4, 0, 16, N, 8, N, N) == -1
    assert lib.kv_expand_kernel_blocks(N, 0, 4, 32, 16, N, 8, N, N) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    import paged_kv_cache_39_gb300 as kv
    q = torch.zeros(2, dtype=torch.int32)
    p = torch.zeros(1, dtype=torch.int64)
    t = torch.zeros((1, 8), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        kv.kv_slot_mapping_paged(q, p, t, 16, 8)
    kc = torch.zeros((1, 4, 16, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        kv.kv_cache_gather(kc, kc, t, q[:1], q[:1])


def test_next_step_calls_reject_bad_arguments(lib):
    # kv_table_from_ranges
    assert lib.kv_table_from_ranges(N, N, N, 257, 1, N, 8, N, N) == -2
    assert lib.kv_table_from_ranges(N, N, N, 4, -1, N, 8, N, N) == -1
    assert lib.kv_table_from_ranges(N, N, N, 4, 1, N, 8, N, N) == -1  # num_ranges NULL
    assert lib.kv_table_from_ranges(N, N, N, 4, 0, N, 8, N, N) == 0
    # kv_cache_gather_range
    assert lib.kv_cache_gather_range(0x1000, 0x2000, 0, 1, 8, 16, 8, 64, N, N, N, 257, 0x3000,
                                     0x4000, 1, N, N, 0, N, N) == -2
    assert lib.kv_cache_gather_range(0x1000, 0x2000, 0, 1, 8, 16, 8, 64, N, N, N, 4, 0x3000,
                                     0x4000, 2, N, N, 0, N, N) == -1  # num_ranges NULL
    assert lib.kv_cache_gather_range(0x1000, 0x2000, 2, 1, 8, 16, 8, 64, N, N, N, 4, N, N, 0, N,
                                     N, 0, N, N) == -1  # layer out of range
    # kv_copy_blocks
    assert lib.kv_copy_blocks(N, N, 1, 8, 16, 3, 5, N, N, 1, N, N) == -2
    assert lib.kv_copy_blocks(N, N, 1, 8, 16, 8, 64, N, N, 1, N, N) == -1
    assert lib.kv_copy_blocks(N, N, 1, 8, 16, 8, 64, N, N, 0, N, N) == 0
    assert lib.kv_copy_blocks(N, N, 1, 8, 16, 8, 64, N, N, -1, N, N) == -1
    # kv_copy_blocks_bulk: the same checks
    assert lib.kv_copy_blocks_bulk(N, N, 1, 8, 16, 3, 5, N, N, 1, N, N) == -2
    assert lib.kv_copy_blocks_bulk(N, N, 1, 8, 16, 8, 64, N, N, 1, N, N) == -1
    assert lib.kv_copy_blocks_bulk(N, N, 1, 8, 16, 8, 64, N, N, 0, N, N) == 0
    assert lib.kv_copy_blocks_bulk(N, N, 1, 8, 16, 8, 64, N, N, -1, N, N) == -1
    assert lib.kv_copy_blocks_bulk(0x1008, 0x2000, 1, 8, 16, 8, 64, 0x3000, 0x4000, 1, N,
                                   N) == -1  # misaligned cache


def test_header_constants_match_the_binding():
    from paged_kv_cache_39_gb300 import _lib
    text = open(HEADER).read()
    defs = dict(re.findall(r"^#define\s+(KV_\w+)\s+\(?(-?\d+)\)?", text, flags=re.M))
    assert int(defs["KV_PAD_SLOT_ID"]) == _lib.PAD_SLOT_ID
    assert int(defs["KV_NULL_BLOCK_ID"]) == _lib.NULL_BLOCK_ID
    assert int(defs["KV_MAX_RANGES_PER_REQ"]) == _lib.MAX_RANGES_PER_REQ
    assert int(defs["KV_MAX_GATHER_REQS"]) == _lib.MAX_GATHER_REQS
    assert int(defs["KV_MAX_TOKENS"]) == _lib.MAX_TOKENS == (1 << 31) - 65536


def test_slot_maps_refuse_max_num_tokens_past_the_limit(lib):
    """Every slot-mapping entry point refuses max_num_tokens above
    KV_MAX_TOKENS on the host, before any launch (token indices of a whole
    last tile must stay in int32)."""
    from paged_kv_cache_39_gb300 import _lib
    over = _lib.MAX_TOKENS + 1
    big = (1 << 31) - 1
    for n_max in (over, big):
        assert lib.kv_slot_mapping_paged(0x1000, 0x2000, 0x3000, 8, 1, 0, n_max, 16, 8, 0x4000,
                                         N, N) == -1
        assert lib.kv_slot_mapping_range(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 4, 1, 0, n_max,
                                         16, 8, 0x6000, N, N) == -1
        assert lib.kv_slot_mapping_paged_cp(0x1000, 0x2000, 0x3000, 8, 1, 0, n_max, 16, 8, 2, 0,
                                            1, 0x4000, N, N) == -1
        assert lib.kv_slot_mapping_paged_write(0x1000, 0x2000, 0x3000, 8, 1, 0, n_max, 16, 8, N,
                                               N, N, N, 1, 8, 128, 0x4000, N, N) == -1
        assert lib.kv_slot_mapping_range_write(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 4, 1, 0,
                                               n_max, 16, 8, N, N, N, N, 1, 8, 128, 0x6000, N,
                                               N) == -1


def test_cp_slot_mapping_rejects_bad_arguments(lib):
    assert lib.kv_slot_mapping_paged_cp(N, N, N, 0, 0, 0, 0, 16, 8, 0, 0, 1, N, N, N) == -1
    assert lib.kv_slot_mapping_paged_cp(N, N, N, 0, 0, 0, 0, 16, 8, 2, 2, 1, N, N, N) == -1
    assert lib.kv_slot_mapping_paged_cp(N, N, N, 0, 0, 0, 0, 16, 8, 2, 0, 0, N, N, N) == -1
    assert lib.kv_slot_mapping_paged_cp(N, N, N, 0, 0, 0, 0, 16, 8, 2, 0, 3, N, N, N) == -2
    assert lib.kv_slot_mapping_paged_cp(N, N, N, 0, 0, 0, 0, 16, 8, 2, 1, 4, N, N, N) == 0


def test_bulk_gather_rejects_unsupported_shapes(lib):
    # rows of 40 KiB exceed a bulk stage; more than 2048 requests exceed its offsets
    assert lib.kv_cache_gather_bulk(0x1000, 0x2000, 0, 1, 8, 16, 20, 1024, N, 0, 0x3000, 0x4000,
                                    1, N, N, 0, N, N) == -2
    assert lib.kv_cache_gather_bulk(0x1000, 0x2000, 0, 1, 8, 16, 8, 128, N, 0, 0x3000, 0x4000,
                                    2049, N, N, 0, N, N) == -2
    assert lib.kv_cache_gather_bulk(0x1000, 0x2000, 0, 1, 8, 16, 8, 128, N, 0, N, N, 0, N, N, 0,
                                    N, N) == 0


def test_diag_bounded_wait_rejects_bad_arguments(lib):
    assert lib.kv_diag_bounded_wait(0, 0x1000, N) == -1
    assert lib.kv_diag_bounded_wait((1 << 20) + 1, 0x1000, N) == -1
    assert lib.kv_diag_bounded_wait(16, N, N) == -1


def test_fused_slot_write_rejects_bad_arguments(lib):
    # kv_slot_mapping_paged_write(qsl, pos, table, stride, R, N, N_max, T, B,
    #                             key, value, k_cache, v_cache, L, H, D, slots, err, stream)
    P = lib.kv_slot_mapping_paged_write
    assert P(N, N, N, 0, -1, 0, 0, 16, 8, N, N, N, N, 1, 8, 128, N, N, N) == -1
    assert P(N, N, N, 0, 0, 0, 0, 16, 8, N, N, N, N, -1, 8, 128, N, N, N) == -1
    assert P(N, N, N, 0, 0, 0, 0, 16, 8, N, N, N, N, 1, 3, 5, N, N, N) == -2  # 30-byte rows
    assert P(N, N, N, -1, 0, 0, 0, 16, 8, N, N, N, N, 1, 8, 128, N, N, N) == -1
    # one token to write but no key / a misaligned key
    assert P(N, 0x1000, N, 0, 0, 1, 1, 16, 8, N, 0x2000, 0x3000, 0x4000, 1, 8, 128, 0x5000, N,
             N) == -1
    assert P(N, 0x1000, N, 0, 0, 1, 1, 16, 8, 0x1008, 0x2000, 0x3000, 0x4000, 1, 8, 128, 0x5000,
             N, N) == -1
    assert P(N, N, N, 0, 0, 0, 0, 16, 8, N, N, N, N, 1, 8, 128, N, 0x1002, N) == -1  # err
    assert P(N, N, N, 0, 0, 0, 0, 16, 8, N, N, N, N, 1, 8, 128, N, N, N) == 0  # empty
    # kv_slot_mapping_range_write(qsl, pos, rs, rl, nr, rstride, R, N, N_max, T, B,
    #                             key, value, k_cache, v_cache, L, H, D, slots, err, stream)
    Q = lib.kv_slot_mapping_range_write
    assert Q(N, N, N, N, N, 257, 0, 0, 0, 16, 8, N, N, N, N, 1, 8, 128, N, N, N) == -2
    assert Q(N, N, N, N, N, -1, 0, 0, 0, 16, 8, N, N, N, N, 1, 8, 128, N, N, N) == -1
    assert Q(0x1000, N, N, N, N, 4, 1, 0, 0, 16, 8, N, N, N, N, 1, 8, 128, N, N, N) == -1
    assert Q(N, N, N, N, N, 4, 0, 0, 0, 16, 8, N, N, N, N, 1, 8, 64, N, N, N) == 0
