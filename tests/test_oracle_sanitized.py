"""The oracle under AddressSanitizer and UndefinedBehaviorSanitizer (no GPU).

oracle.c is rebuilt with -fsanitize=address,undefined (same -O2
-ffp-contract=off arithmetic) and every pin runs against that build in a
child process that preloads the sanitizer runtimes.  An out-of-bounds access,
a use of freed memory, a signed overflow, a bad shift or a misaligned load
in the oracle ends the child with the sanitizer's report, and the test
fails.  This is the host-side stand-in for a memory checker on the checker
itself.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

CHILD = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, pins
o = oracle.Oracle({lib!r})
for p in pins.ALL_PINS:
    p(o)
print("PINS_OK", len(pins.ALL_PINS))
"""


def runtime(name):
    p = subprocess.run(["gcc", "-print-file-name=" + name], capture_output=True, text=True).stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_pins_under_asan_ubsan(tmp_path):
    asan, ubsan = runtime("libasan.so"), runtime("libubsan.so")
    if asan is None or ubsan is None:
        pytest.skip("gcc sanitizer runtimes not installed")
    lib = str(tmp_path / "liboracle_san.so")
    oracle.compile_oracle(out=lib, extra=["-fsanitize=address,undefined", "-fno-sanitize-recover=all",
                                          "-fno-omit-frame-pointer", "-g"])
    env = dict(os.environ)
    env["LD_PRELOAD"] = asan + ":" + ubsan
    env["ASAN_OPTIONS"] = "detect_leaks=0:abort_on_error=0:halt_on_error=1"
    env["UBSAN_OPTIONS"] = "halt_on_error=1:print_stacktrace=1"
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, tests=TESTS, lib=lib)], env=env,
                       capture_output=True, text=True, timeout=900)
    report = r.stdout[-3000:] + r.stderr[-3000:]
    assert r.returncode == 0, report
    assert "PINS_OK" in r.stdout, report
    assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, report


def test_sanitizer_build_catches_a_planted_overrun(tmp_path):
    """The same harness on a copy of oracle.c whose weight quantizer writes
    one packed byte past each row (a planted out-of-bounds write on the last
    row): the child must fail with AddressSanitizer's report, so a clean run
    above means something."""
    asan, ubsan = runtime("libasan.so"), runtime("libubsan.so")
    if asan is None or ubsan is None:
        pytest.skip("gcc sanitizer runtimes not installed")
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    old = "        for (int64_t j = 0; j < K / 2; ++j) {\n            int q0 = quant_code(row[2 * j], s, 7);"
    assert src.count(old) == 1
    bad = src.replace(old, "        Wq[n * (K / 2) + K / 2] = 0;  /* planted: one byte past the row */\n" + old)
    path = tmp_path / "oracle_bad.c"
    path.write_text(bad)
    lib = str(tmp_path / "liboracle_bad.so")
    oracle.compile_oracle(src=str(path), out=lib, extra=["-fsanitize=address,undefined",
                                                        "-fno-sanitize-recover=all", "-g"])
    env = dict(os.environ)
    env["LD_PRELOAD"] = asan + ":" + ubsan
    env["ASAN_OPTIONS"] = "detect_leaks=0:halt_on_error=1"
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, tests=TESTS, lib=lib)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode != 0 and "AddressSanitizer" in r.stderr, (r.returncode, r.stderr[-2000:])
