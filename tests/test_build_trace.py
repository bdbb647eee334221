"""The diagnostic library with the pipeline trace (kernels compiled with
PA_TRACE) still builds, exports the same C ABI as the default library and,
unlike it, accepts a trace buffer.  Host-side only: the buffer pointer is
stored, never dereferenced, and tracing is switched off again at once."""
import ctypes
import importlib.util
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build_module():
    spec = importlib.util.spec_from_file_location(
        "pa_build_for_test", os.path.join(ROOT, "paged_quantized_kv_gqa_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traced_library_builds_and_takes_a_trace_buffer():
    path = _build_module().build(trace=True)
    assert path.endswith("libpa_gb300_trace.so") and os.path.exists(path)
    lib = ctypes.CDLL(path)
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "pa.h")).read(), flags=re.S)
    for name in sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", src))):
        assert hasattr(lib, name), name
    lib.pa_debug_set_trace.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]
    lib.pa_debug_set_trace.restype = ctypes.c_int32
    assert lib.pa_debug_set_trace(ctypes.c_void_p(256), 1, 1) == 0
    assert lib.pa_debug_set_trace(None, 0, 0) == 0
    # a non-null buffer still needs positive sizes
    assert lib.pa_debug_set_trace(ctypes.c_void_p(256), 0, 1) != 0
