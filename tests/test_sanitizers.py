"""The oracle and the input generator under AddressSanitizer and UndefinedBehaviorSanitizer: a driver
compiled with both sources runs routing (selection and full sort), the permutation, the layer (dense and
permuted) and the hash route on a small seeded layer; any sanitizer report fails the run."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_and_generator_are_clean_under_sanitizers(tmp_path):
    cxx, cc = shutil.which("g++"), shutil.which("gcc")
    if not cxx or not cc:
        pytest.skip("no host compiler")
    flags = ["-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer"]
    synth_o = str(tmp_path / "synth.o")
    r = subprocess.run([cc, *flags, "-std=c11", "-c", os.path.join(ROOT, "synth", "synth.c"), "-o", synth_o],
                       capture_output=True, text=True)
    if r.returncode and "sanitize" in r.stderr:
        pytest.skip("the compiler has no sanitizer runtime")
    assert r.returncode == 0, r.stderr
    exe = str(tmp_path / "driver")
    r = subprocess.run([cxx, *flags, "-std=c++17", "-ffp-contract=off", "-pthread",
                        os.path.join(ROOT, "oracle", "moe_oracle.cpp"),
                        os.path.join(ROOT, "tests", "sanitize", "sanitize_driver.cpp"), synth_o, "-lm", "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0", UBSAN_OPTIONS="print_stacktrace=1")
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
