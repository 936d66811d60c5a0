"""The oracle runs its pin suite clean under AddressSanitizer and UBSan."""
import os
import subprocess
import sys

import pytest

from oracle.build import build_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_pins_clean_under_asan_ubsan(tmp_path):
    asan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True,
                          text=True).stdout.strip()
    if not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("libasan not available")
    lib = build_oracle(extra_flags=["-fsanitize=address,undefined", "-fno-sanitize-recover=all",
                                    "-g"], out=str(tmp_path / "libkvoracle_san.so"))
    env = dict(os.environ, KV_ORACLE_LIB=lib, LD_PRELOAD=asan, ASAN_OPTIONS="detect_leaks=0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
