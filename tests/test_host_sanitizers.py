"""The library's host-side managers (block manager with copy-on-write, and
the prefix cache with chained keys) under AddressSanitizer and
UndefinedBehaviorSanitizer: tests/host_managers_stress.cpp drives long
seeded random streams of their C ABI and checks the pool invariants after
every call; built here with g++ from the same sources the library compiles
(they hold no device code)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = [os.path.join(ROOT, "tests", "host_managers_stress.cpp"),
           os.path.join(ROOT, "paged_kv_cache_117_gb300", "csrc", "block_manager.cu"),
           os.path.join(ROOT, "paged_kv_cache_117_gb300", "csrc", "prefix_cache.cu")]


def _build(tmp_path, flags):
    exe = str(tmp_path / "stress")
    cmd = ["g++", "-std=c++17", "-O1", "-g", "-fno-omit-frame-pointer"] + flags
    for src in SOURCES:   # the .cu files are plain C++ (host code only)
        cmd += ["-x", "c++", src]
    cmd += ["-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return exe, r


@pytest.mark.timeout(600)
def test_host_managers_under_asan_and_ubsan(tmp_path):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    flags = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all"]
    exe, r = _build(tmp_path, flags)
    if r.returncode != 0 and "sanitize" in r.stderr:
        pytest.skip("this g++ has no sanitizer runtime: " + r.stderr.splitlines()[-1])
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1")
    p = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=500)
    out = p.stdout + p.stderr
    assert p.returncode == 0, out[-4000:]
    assert "all checks passed" in p.stdout
    assert "runtime error" not in out and "AddressSanitizer" not in out
