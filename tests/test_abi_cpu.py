"""C ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every function include/trace_fp4.h declares; argument errors are
reported without touching a device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "trace_fp4.h")


@pytest.fixture(scope="module")
def lib():
    from fp4_rollout_guided_gb300 import build, trace
    build.build()
    return trace.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(trace_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_surveyed_entry_points():
    names = declared_functions()
    for need in ("trace_create", "trace_destroy", "trace_status_string", "trace_last_cuda_error",
                 "trace_rollout_quant", "trace_guide_pack", "trace_guide_unpack",
                 "trace_train_fakequant"):
        assert need in names


def test_every_declared_symbol_is_exported(lib):
    from fp4_rollout_guided_gb300 import trace
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
    assert set(names) == set(trace.SIGNATURES), "binding and header disagree"


def test_status_strings_and_version(lib):
    for code in range(7):
        s = lib.trace_status_string(code)
        assert isinstance(s, bytes) and s
    assert lib.trace_status_string(99) == b"unknown status"
    assert lib.trace_version() == 100


def test_create_rejects_bad_devices(lib):
    h = ctypes.c_void_p(1)
    assert lib.trace_create(ctypes.byref(h), -1) == 3 and not h.value
    assert lib.trace_create(ctypes.byref(h), 4096) == 3 and not h.value
    assert lib.trace_create(None, 0) == 1
    if not torch.cuda.is_available():
        assert lib.trace_create(ctypes.byref(h), 0) == 3 and not h.value


def test_null_handle_is_an_argument_error(lib):
    from fp4_rollout_guided_gb300.trace import Segments, KernelTime
    seg = Segments(None, 1)
    p = ctypes.c_void_p(256)
    assert lib.trace_rollout_quant(None, p, 1, 32, seg, p, p, p, None, None) == 1
    assert lib.trace_guide_pack(None, p, 1, 32, p, None) == 1
    assert lib.trace_guide_unpack(None, p, p, p, p, seg, 1, 32, p, None) == 1
    assert lib.trace_train_fakequant(None, p, 1, 32, seg, 0, None, None, None, seg, p, None,
                                     None, None, None) == 1
    assert lib.trace_profile_enable(None, 1) == 1
    arr = (KernelTime * 5)()
    assert lib.trace_profile_collect(None, arr) == 1
    assert lib.trace_destroy(None) == 0
    assert lib.trace_last_cuda_error(None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from fp4_rollout_guided_gb300 import trace
    monkeypatch.setattr(trace, "_lib", None)
    monkeypatch.setattr(trace, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(trace.TraceError):
        trace.lib()
