"""The boundary is a C ABI: a plain C11 program (and the same source as
C++17) includes `include/kvpaged.h`, links `libkvpaged.so` and calls it.  Only
calls that the host-side checks answer before any launch are made, so no GPU
is needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_39_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "kvpaged.h"

static int fails = 0;
#define EXPECT(cond) \
    do { if (!(cond)) { printf("FAILED: %s (line %d)\n", #cond, __LINE__); ++fails; } } while (0)

int main(void) {
    EXPECT(kv_abi_version() > 0);
    EXPECT(strcmp(kv_status_string(KV_OK), kv_status_string(KV_EINVAL)) != 0);
    EXPECT(kv_status_string(KV_EUNSUPPORTED) != NULL && kv_status_string(KV_ECUDA) != NULL);
    EXPECT(KV_PAD_SLOT_ID == -1 && KV_NULL_BLOCK_ID == 0);
    EXPECT(KV_MAX_TOKENS == 2147483647 - 65535);
    EXPECT(KV_ERR_BAD_BLOCK == 1 && KV_ERR_TIMEOUT == 128);

    int32_t qsl[2] = {0, 1};
    int64_t pos[1] = {5};
    int32_t table[4] = {1, 2, 3, 4};
    int64_t slots[1];
    kv_stream_t stream = NULL;
    /* a negative request count, a too-large max_num_tokens: refused on the host */
    EXPECT(kv_slot_mapping_paged(qsl, pos, table, 4, -1, 1, 1, 16, 8, slots, NULL, stream)
           == KV_EINVAL);
    EXPECT(kv_slot_mapping_paged(qsl, pos, table, 4, 1, 1, KV_MAX_TOKENS + 1, 16, 8, slots,
                                 NULL, stream) != KV_OK);
    /* more descriptors per request than the cap: fail closed */
    int32_t rs[1], rl[1], nr[1];
    EXPECT(kv_slot_mapping_range(qsl, pos, rs, rl, nr, KV_MAX_RANGES_PER_REQ + 1, 1, 1, 1, 16, 8,
                                 slots, NULL, stream) == KV_EUNSUPPORTED);
    /* nothing to write: no launch, KV_OK */
    EXPECT(kv_cache_write(NULL, NULL, NULL, NULL, NULL, 0, 1, 8, 16, 8, 128, NULL, stream)
           == KV_OK);
    /* a kernel block size that does not divide the manager block size */
    int32_t mgr[1] = {3}, kern[4];
    EXPECT(kv_expand_kernel_blocks(mgr, 1, 1, 32, 12, kern, 4, NULL, stream) == KV_EUNSUPPORTED);
    printf("%s\n", fails ? "C consumer: failures" : "C consumer: ok");
    return fails != 0;
}
"""


@pytest.fixture(scope="module")
def library():
    from paged_kv_cache_39_gb300 import _lib
    from paged_kv_cache_39_gb300 import build as kbuild
    if not os.path.exists(_lib.LIB_PATH):
        kbuild.build()
    return _lib.LIB_PATH


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_plain_c_program_links_and_calls(library, lang, tmp_path):
    compiler = "gcc" if lang == "c" else "g++"
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not available")
    src = tmp_path / ("consumer.c" if lang == "c" else "consumer.cpp")
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    std = "-std=c11" if lang == "c" else "-std=c++17"
    cmd = [compiler, std, "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           "-L", PKG, "-lkvpaged", f"-Wl,-rpath,{PKG}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C consumer: ok" in r.stdout
