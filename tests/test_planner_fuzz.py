"""The host planners on random inputs under AddressSanitizer and UBSan (CPU only).

tests/fuzz_plan.cpp drives build_host_plan, build_host_plan_paged and
build_host_plan_multi with random layouts and options and checks every plan's
structure; the sanitizers catch any out-of-bounds access or undefined behaviour.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mla_decode_attention_09_gb300", "csrc")


def test_planner_fuzz_sanitized(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    exe = str(tmp_path / "fuzz_plan")
    cmd = [cxx, "-std=c++17", "-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-I", "/usr/local/cuda/include",
           os.path.join(ROOT, "tests", "fuzz_plan.cpp"), os.path.join(CSRC, "plan.cpp"), "-o", exe]
    b = subprocess.run(cmd, capture_output=True, text=True)
    if b.returncode != 0:
        if "asan" in b.stderr.lower() or "sanitizer" in b.stderr.lower():
            pytest.skip("sanitizer runtime not available: " + b.stderr[-200:])
        raise AssertionError(b.stderr[-2000:])
    for seed in (1, 2):
        r = subprocess.run([exe, str(seed), "4000"], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, (r.stdout[-1000:], r.stderr[-3000:])
        assert r.stdout.startswith("ok "), r.stdout
