"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer (no GPU).

Two programs are built with gcc / g++ -fsanitize=address,undefined -fno-sanitize-recover=all
and run:
- tests/sanitize/host_check.cpp with the library's host sources (bsgemv_geometry.cpp,
  bsgemv_host.cpp, bsgemv_api.cu compiled as C++) and stand-ins for the device launchers: the
  launch geometry over thousands of random problems (every split, override, max_M and per-call
  row layout), the kernel parameters, and the C ABI's host-side error paths;
- tests/sanitize/oracle_check.c with the oracle (oracle/bsgemv_oracle.c, without OpenMP): every
  format on small random problems, NaN codes included, and the dense GEMV.
- tests/sanitize/plan_check.cpp with the same host sources linked against a fake CUDA runtime
  (tests/sanitize/fake_cuda.cpp) instead of libcudart: the planned entry points end to end on a
  fake device, failures of cudaMalloc and cudaMemset injected, every launch's pointers checked.
All must exit 0 and print "ok" with no sanitizer report.  ("[CUDA] Pin FP8 GEMV residency for
grids just past two blocks per SM", Tests: the host dispatch selectors are tested under UBSan.)
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-g", "-O1"]
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _run(exe, tmp_path):
    env = dict(os.environ)
    # the CUDA runtime keeps process-lifetime allocations; leaks are not what this test is for
    env["ASAN_OPTIONS"] = "detect_leaks=0:abort_on_error=0"
    env["UBSAN_OPTIONS"] = "print_stacktrace=1"
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=600, cwd=tmp_path)
    report = r.stdout + r.stderr
    assert r.returncode == 0, report[-4000:]
    assert "runtime error" not in report and "AddressSanitizer" not in report, report[-4000:]
    assert r.stdout.startswith("ok"), report[-2000:]
    return r.stdout


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_host_code_under_sanitizers(tmp_path):
    csrc = os.path.join(ROOT, "block_scaled_bit_gb300", "csrc")
    inc = ["-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include")]
    objs = []
    for src in ("bsgemv_geometry.cpp", "bsgemv_host.cpp", "bsgemv_api.cu"):
        obj = str(tmp_path / (src + ".o"))
        subprocess.run(["g++", "-std=c++17", "-x", "c++", *SAN, *inc, "-c", os.path.join(csrc, src),
                        "-o", obj], check=True, capture_output=True, text=True)
        objs.append(obj)
    exe = str(tmp_path / "host_check")
    r = subprocess.run(["g++", "-std=c++17", *SAN, *inc,
                        os.path.join(ROOT, "tests", "sanitize", "host_check.cpp"),
                        os.path.join(ROOT, "tests", "sanitize", "device_stubs.cpp"), *objs,
                        "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-ldl", "-lpthread",
                        f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = _run(exe, tmp_path)
    assert int(out.split()[1]) > 1000  # geometries checked


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_plans_on_a_fake_device_under_sanitizers(tmp_path):
    """The planned entry points' host code linked against a fake CUDA runtime
    (tests/sanitize/fake_cuda.cpp, no libcudart): plans, calls, a workspace allocation and a
    clear that fail, the autotuner's choice and its confirmation, the host-buffer paths."""
    csrc = os.path.join(ROOT, "block_scaled_bit_gb300", "csrc")
    inc = ["-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include")]
    objs = []
    for src in ("bsgemv_geometry.cpp", "bsgemv_host.cpp", "bsgemv_api.cu"):
        obj = str(tmp_path / (src + ".o"))
        subprocess.run(["g++", "-std=c++17", "-x", "c++", *SAN, *inc, "-c", os.path.join(csrc, src),
                        "-o", obj], check=True, capture_output=True, text=True)
        objs.append(obj)
    exe = str(tmp_path / "plan_check")
    r = subprocess.run(["g++", "-std=c++17", *SAN, *inc,
                        os.path.join(ROOT, "tests", "sanitize", "plan_check.cpp"),
                        os.path.join(ROOT, "tests", "sanitize", "fake_cuda.cpp"), *objs,
                        "-lpthread", "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = _run(exe, tmp_path)
    assert int(out.split()[1]) > 100  # kernel launches checked


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_oracle_under_sanitizers(tmp_path):
    exe = str(tmp_path / "oracle_check")
    r = subprocess.run(["gcc", "-std=c11", *SAN, os.path.join(ROOT, "oracle", "bsgemv_oracle.c"),
                        os.path.join(ROOT, "tests", "sanitize", "oracle_check.c"), "-lm", "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = _run(exe, tmp_path)
    assert int(out.split()[1]) == 500
