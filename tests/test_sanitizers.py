"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer (no GPU).

compute-sanitizer is closed on the GPU pool, so the host side is checked this way instead: the
fp64 oracle (oracle/moe_oracle.c) and the library's host packer (csrc/moe_pack.cpp) are compiled
with -fsanitize=address,undefined next to small drivers (tests/sanitize/) that run every entry
point on seeded problems with buffers of exactly the needed size.  Any out-of-bounds access, use
after free, leak or undefined operation makes the run fail.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(ROOT, "_build", "sanitize")
FLAGS = ["-g", "-O1", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
         "-fno-omit-frame-pointer"]


def _run(cmd_build, exe):
    os.makedirs(OUT, exist_ok=True)
    r = subprocess.run(cmd_build, capture_output=True, text=True)
    if r.returncode != 0 and "sanitize" in (r.stderr or ""):
        pytest.skip("compiler without sanitizer runtimes: " + r.stderr.strip().splitlines()[-1])
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    env.pop("LD_PRELOAD", None)
    p = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=300)
    assert p.returncode == 0, p.stdout + p.stderr
    return p.stdout


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
def test_oracle_under_asan_ubsan():
    exe = os.path.join(OUT, "oracle_driver")
    out = _run(["gcc", "-std=c11", "-ffp-contract=off"] + FLAGS +
               [os.path.join(ROOT, "tests", "sanitize", "oracle_driver.c"),
                os.path.join(ROOT, "oracle", "moe_oracle.c"), "-lm", "-o", exe], exe)
    assert "oracle sanitizer run ok" in out


@pytest.mark.skipif(shutil.which("g++") is None, reason="g++ not found")
def test_host_packer_under_asan_ubsan():
    exe = os.path.join(OUT, "pack_driver")
    out = _run(["g++", "-std=c++17"] + FLAGS +
               ["-I", os.path.join(ROOT, "include"),
                os.path.join(ROOT, "tests", "sanitize", "pack_driver.cpp"),
                os.path.join(ROOT, "quantized_moe_expert_dequant_gb300", "csrc", "moe_pack.cpp"),
                "-o", exe], exe)
    assert "packer sanitizer run ok" in out
