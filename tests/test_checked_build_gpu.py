"""The checked debug build of the library (libgdn_checked.so, compiled with GDN_CHECKED).

Its chunked-prefill and projection kernels test every computed global and shared-memory range
against the region it belongs to before the access, and report a failed test in the device
status word (GDN_DEV_BOUNDS) instead of touching memory -- the stand-in for a device memory
checker.  The bounds tests (canaries around every output, untouched idle slots), the prefill
tests (ragged and empty sequences, partial chunks, GQA ratios, conv widths, both io dtypes, the
chunked d < 128 path), the pool tests (prefills run in pipelined segments among them), the mixed
steps, the edge cases and the projection tests run against it in a child process; every one of
them also asserts that the status word is clean, so no test passes with a skipped access."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_runs_the_bounds_prefill_and_projection_tests_clean():
    from gated_deltanet_linear_rule_gb300 import build

    lib = build.build(checked=True)
    env = dict(os.environ, GDN_LIBRARY_VARIANT="checked")
    probe = subprocess.run(
        [sys.executable, "-c", "from gated_deltanet_linear_rule_gb300 import binding; binding.lib(); "
                               "print(binding.lib_path())"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert probe.returncode == 0 and probe.stdout.strip() == lib, probe.stdout + probe.stderr
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider", "--timeout", "600",
         "tests/test_bounds_gpu.py", "tests/test_prefill_gpu.py", "tests/test_pool_gpu.py", "tests/test_mixed_gpu.py",
         "tests/test_edge_gpu.py", "tests/test_proj_gpu.py", "-k", "not 15998"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    import re

    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 70, r.stdout[-2000:]
    print(r.stdout.strip().splitlines()[-1])
