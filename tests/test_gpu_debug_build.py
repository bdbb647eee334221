"""The debug library (kernels compiled with PA_DEBUG) on the GPU: with shared
and tensor memory filled with NaN bytes before first use, every kernel family
still matches the fp64 oracle, and the work-item check turns an altered item
into PA_ERR_BAD_ITEM.  The cases (tests/debug_build_cases.py) run in a child
process that loads libpa_gb300_debug.so (PA_GB300_DEBUG=1)."""
import importlib.util
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_library_cases():
    spec = importlib.util.spec_from_file_location(
        "pa_build_for_debug_test", os.path.join(ROOT, "paged_quantized_kv_gqa_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert mod.build(debug=True).endswith("libpa_gb300_debug.so")
    env = dict(os.environ, PA_GB300_DEBUG="1")
    env.pop("PA_GB300_TRACE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_build_cases.py")],
                       env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert "library libpa_gb300_debug.so" in r.stdout
    assert "all cases passed" in r.stdout
