"""The host allocator under AddressSanitizer and UndefinedBehaviorSanitizer
(no GPU): tests/native/allocator_stress.c drives every host call of the C ABI
from a seeded random stream (refused appends, batches that repeat a
sequence, forks, frees, reused ids, preemption, admission, prefix-cache hits,
full and incremental batch tables) and checks the allocator's invariants
after every step; any out-of-bounds access, use after free, leak or
undefined behaviour aborts."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SAN = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-g",
       "-O1"]


@pytest.fixture(scope="module")
def stress(tmp_path_factory):
    cxx, cc = shutil.which("g++"), shutil.which("gcc")
    if cxx is None or cc is None:
        pytest.skip("no host C/C++ compiler")
    d = tmp_path_factory.mktemp("asan")
    inc = ["-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "paged_kv_cache_137_gb300", "csrc")]
    steps = [
        [cxx, "-std=c++17", *SAN, *inc, "-c", os.path.join(ROOT, "paged_kv_cache_137_gb300", "csrc",
                                                           "allocator.cpp"), "-o", str(d / "allocator.o")],
        [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", *SAN, *inc, "-c",
         os.path.join(HERE, "native", "allocator_stress.c"), "-o", str(d / "stress.o")],
        [cxx, *SAN, str(d / "stress.o"), str(d / "allocator.o"), "-o", str(d / "stress")],
    ]
    for cmd in steps:
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 and "asan" in (r.stderr or "").lower() and "cannot find" in r.stderr:
            pytest.skip("sanitizer runtime not installed")
        assert r.returncode == 0, r.stderr[-3000:]
    return str(d / "stress")


@pytest.mark.parametrize("caching", [0, 1])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_allocator_stress_under_sanitizers(stress, seed, caching):
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1")
    r = subprocess.run([stress, str(seed), "3000", str(caching)], capture_output=True, text=True,
                       timeout=300, env=env)
    assert r.returncode == 0, (r.returncode, r.stdout[-500:], r.stderr[-3000:])
    assert r.stdout.strip() == "ok 3000 steps"
