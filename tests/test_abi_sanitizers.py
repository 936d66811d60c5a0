"""The library's host-side argument checks run clean under AddressSanitizer
and UBSan: the C ABI checks of `test_abi_cpu.py` (every call's invalid
arguments and empty work, none of which launches a kernel) against a build
of the same sources with the sanitizers in the host code."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_abi_checks_clean_under_asan_ubsan(tmp_path):
    asan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True,
                          text=True).stdout.strip()
    if not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("libasan not available")
    from paged_kv_cache_39_gb300 import build as kbuild
    lib = kbuild.build(host_flags=["-fsanitize=address", "-fsanitize=undefined",
                                   "-fno-sanitize-recover=all", "-fno-omit-frame-pointer"],
                       out=str(tmp_path / "libkvpaged_san.so"), build_dir=str(tmp_path / "obj"))
    env = dict(os.environ, KV_TEST_LIB=lib, LD_PRELOAD=asan,
               ASAN_OPTIONS="detect_leaks=0:protect_shadow_gap=0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_abi_cpu.py"), "-k", "not binding"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
