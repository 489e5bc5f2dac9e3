"""The CPU oracle under AddressSanitizer and UndefinedBehaviorSanitizer.

The oracle's C source is built with -fsanitize=address,undefined into a
private library, and both pin suites run against it in a subprocess with the
sanitizer runtimes preloaded: an out-of-bounds access, a use after free or
undefined behaviour anywhere the pins reach ends that run with an error.
Skipped where gcc has no sanitizer runtimes.  The oracle itself is built and
used as usual everywhere else.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_pcg.c")


def _runtime(name):
    try:
        p = subprocess.run(["gcc", "-print-file-name=" + name], capture_output=True, text=True,
                           check=True).stdout.strip()
    except (OSError, subprocess.CalledProcessError):
        return None
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_pins_pass_under_sanitizers(tmp_path):
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not (asan and ubsan):
        pytest.skip("gcc has no sanitizer runtimes here")
    lib = tmp_path / "liboracle_sanitized.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-g", "-fsanitize=address,undefined",
                    "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer",
                    "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib), SRC, "-lm"],
                   check=True)
    logs = tmp_path / "report"  # the sanitizers write their reports to report.<pid>
    env = dict(os.environ, ORACLE_LIB=str(lib), LD_PRELOAD=asan + ":" + ubsan,
               ASAN_OPTIONS="detect_leaks=0:log_path=%s" % logs,
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1:log_path=%s" % logs)
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                          os.path.join(ROOT, "tests", "test_oracle_mg_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    reports = "".join(p.read_text()[:3000] for p in tmp_path.glob("report*"))
    assert res.returncode == 0 and not reports, reports + (res.stdout + res.stderr)[-2000:]
    assert " passed" in res.stdout
