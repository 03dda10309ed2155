"""libdgt's host sources (packer, unpack, container reader and writer) built
with AddressSanitizer and UndefinedBehaviorSanitizer and driven by seeded
mutations of packed tensors and container files (tests/host_mutation_driver.cpp):
no out-of-bounds access and no undefined behaviour on damaged inputs."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "decode_gemv_tensor_gb300", "csrc")


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    gxx = shutil.which("g++")
    if not gxx:
        pytest.skip("g++ not found")
    exe = str(tmp_path_factory.mktemp("asan") / "host_mutation_driver")
    cmd = [gxx, "-O1", "-g", "-std=c++17", "-pthread", "-fsanitize=address,undefined",
           "-fno-sanitize-recover=undefined", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
           os.path.join(ROOT, "tests", "host_mutation_driver.cpp"), os.path.join(CSRC, "dgt_host.cpp"),
           os.path.join(CSRC, "dgt_io.cpp"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "sanitize" in r.stderr and "cannot find" in r.stderr:
        pytest.skip("the sanitizer runtimes are not installed")
    assert r.returncode == 0, r.stderr
    return exe


@pytest.mark.parametrize("seed", [1, 2])
def test_host_sources_clean_under_sanitizers(driver, seed, tmp_path):
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0", UBSAN_OPTIONS="print_stacktrace=1")
    r = subprocess.run([driver, "400", str(tmp_path), str(seed)], capture_output=True, text=True, timeout=600,
                       env=env)
    assert r.returncode == 0, r.stdout + r.stderr[-4000:]
    ok, err = (int(x) for x in r.stdout.split()[1::2])
    assert ok > 0 and err > 0     # damaged inputs were both accepted and rejected
