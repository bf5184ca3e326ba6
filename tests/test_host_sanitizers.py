"""The C++ host layer (csrc/kvs_host.cpp: configuration checks, buffer
sizes, the decode work-item plan, failure injection, context creation that
fails before device work) under AddressSanitizer, LeakSanitizer and
UndefinedBehaviorSanitizer, on the CPU.  The kernel launchers are replaced
by stand-ins that report "no device" (tests/host_sanitize/stubs.cpp); the
driver (tests/host_sanitize/main.cpp) reaches none of them.  Any sanitizer
report, or a failed expectation, fails the test."""
import os
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HERE = Path(__file__).resolve().parent / "host_sanitize"
CUDA = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))


def test_host_layer_under_asan_ubsan(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None or not (CUDA / "include" / "cuda_runtime.h").exists():
        pytest.skip("g++ and the CUDA headers are needed")
    lib = next((p for p in (CUDA / "lib64", CUDA / "lib") if (p / "libcudart.so").exists()), None)
    if lib is None:
        pytest.skip("libcudart.so not found")
    flags = ["-std=c++17", "-O1", "-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
             "-fno-sanitize-recover=undefined", "-I", str(CUDA / "include"), "-I", str(ROOT / "include")]
    objs = []
    for src in (ROOT / "paged_kv_cache_flash_gb300" / "csrc" / "kvs_host.cpp", HERE / "stubs.cpp",
                HERE / "main.cpp"):
        obj = tmp_path / (src.stem + ".o")
        subprocess.run([gxx, *flags, "-c", str(src), "-o", str(obj)], check=True)
        objs.append(str(obj))
    exe = tmp_path / "host_sanitize"
    subprocess.run([gxx, "-fsanitize=address,undefined", *objs, "-L", str(lib), "-lcudart", "-ldl",
                    "-lpthread", f"-Wl,-rpath,{lib}", "-o", str(exe)], check=True)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:protect_shadow_gap=0:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=300)
    report = r.stdout + r.stderr
    assert r.returncode == 0, report
    assert "Sanitizer" not in report and "runtime error" not in report, report
    assert "all expectations hold" in r.stdout
