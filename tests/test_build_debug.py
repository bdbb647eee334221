"""The debug library (kernels compiled with PA_DEBUG: work-item bounds checks,
poisoned shared and tensor memory) builds, exports the same C ABI as the
default library, and the binding's PA_ERR_BAD_ITEM matches the header.
Host-side only."""
import ctypes
import importlib.util
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build_module():
    spec = importlib.util.spec_from_file_location(
        "pa_build_for_debug_cpu_test", os.path.join(ROOT, "paged_quantized_kv_gqa_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_debug_library_builds_and_exports_the_abi():
    path = _build_module().build(debug=True)
    assert path.endswith("libpa_gb300_debug.so") and os.path.exists(path)
    lib = ctypes.CDLL(path)
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "pa.h")).read(), flags=re.S)
    for name in sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", src))):
        assert hasattr(lib, name), name


def test_bad_item_status_matches_the_header():
    import paged_quantized_kv_gqa_gb300 as pa
    hdr = open(os.path.join(ROOT, "include", "pa.h")).read()
    m = re.search(r"PA_ERR_BAD_ITEM\s*=\s*(\d+)", hdr)
    assert m and int(m.group(1)) == pa.PA_ERR_BAD_ITEM


def test_trace_and_debug_are_separate_builds():
    import pytest
    with pytest.raises(ValueError):
        _build_module().build(trace=True, debug=True)
