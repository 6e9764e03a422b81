"""C ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every function include/trace_fp4.h declares; argument errors are
reported without touching a device."""
import ctypes
import os
import re

import numpy as np
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


def test_header_declares_the_hot_path_entry_points():
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
    for code in range(8):
        s = lib.trace_status_string(code)
        assert isinstance(s, bytes) and s
    assert lib.trace_status_string(99) == b"unknown status"
    assert lib.trace_version() == 300


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


def test_segment_amax_and_scaled_fakequant_argument_errors(lib):
    from fp4_rollout_guided_gb300.trace import Segments
    seg = Segments(None, 1)
    p = ctypes.c_void_p(256)
    assert lib.trace_segment_amax(None, p, 1, 32, seg, p, None) == 1
    assert lib.trace_train_fakequant_gs(None, p, 1, 32, seg, p, 0, None, None, None, seg, p,
                                        None, None, None, None) == 1
    if not torch.cuda.is_available():
        return
    h = ctypes.c_void_p()
    assert lib.trace_create(ctypes.byref(h), 0) == 0
    try:
        # no scales, misaligned scales, bad shape: rejected before any work
        assert lib.trace_train_fakequant_gs(h, p, 1, 32, seg, None, 0, None, None, None, seg,
                                            p, None, None, None, None) == 1
        assert lib.trace_train_fakequant_gs(h, p, 1, 32, seg, ctypes.c_void_p(258), 0, None,
                                            None, None, seg, p, None, None, None, None) == 2
        assert lib.trace_segment_amax(h, p, 1, 48, seg, p, None) == 1
        assert lib.trace_segment_amax(h, p, 1, 32, seg, None, None) == 1
    finally:
        lib.trace_destroy(h)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from fp4_rollout_guided_gb300 import trace
    monkeypatch.setattr(trace, "_lib", None)
    monkeypatch.setattr(trace, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(trace.TraceError):
        trace.lib()


def _hand_record(kind, rows, cols, seg):
    """A guide record built here from its documented layout (64-byte header,
    256-byte-aligned sections: guide, block scales, global scales, offsets)."""
    a = lambda v: (v + 255) // 256 * 256
    n_seg = len(seg) - 1
    gbytes = rows * cols // 2 if kind == 1 else rows * (cols // 16) * 4
    goff = 256
    boff = a(goff + gbytes)
    soff = a(boff + rows * cols // 16)
    ooff = a(soff + 4 * n_seg)
    buf = np.zeros(ooff + 8 * (n_seg + 1), dtype=np.uint8)
    hdr = np.array([0x31475254, 1, kind, n_seg], dtype=np.uint32).view(np.uint8)
    buf[:16] = hdr
    buf[16:32] = np.array([rows, cols], dtype=np.int64).view(np.uint8)
    buf[32:64] = np.array([goff, boff, soff, ooff], dtype=np.uint64).view(np.uint8)
    buf[ooff:] = np.asarray(seg, dtype=np.int64).view(np.uint8)
    return buf


@pytest.mark.parametrize("kind,rows,cols,seg", [(1, 5, 64, [0, 2, 5]), (2, 7, 32, [0, 7]),
                                                (2, 0, 128, [0, 0]), (1, 33, 96, [0, 1, 1, 33])])
def test_record_layout_and_validation(lib, kind, rows, cols, seg):
    from fp4_rollout_guided_gb300 import trace
    buf = _hand_record(kind, rows, cols, seg)
    assert trace.record_size(kind, rows, cols, len(seg) - 1) == buf.size
    hd, offs = trace.record_info(buf)
    assert (hd.kind, hd.rows, hd.cols, hd.n_seg) == (kind, rows, cols, len(seg) - 1)
    assert offs.tolist() == seg
    # damaged records are rejected: truncated, bad magic, bad kind, moved
    # section, non-monotone or wrong-total segment table
    with pytest.raises(trace.TraceError):
        trace.record_info(buf[:-1])
    for byte, flip in ((0, 0x55), (4, 0x02), (8, 0x04), (40, 0x10), (56, 0x08)):
        bad = buf.copy()
        bad[byte] ^= flip
        with pytest.raises(trace.TraceError):
            trace.record_info(bad)
    if len(seg) > 2:
        bad = buf.copy()
        o = bad[hd.seg_offset:].view(np.int64)
        o[1] = rows + 1
        with pytest.raises(trace.TraceError):
            trace.record_info(bad)
    bad = buf.copy()
    bad[hd.seg_offset + 8 * (len(seg) - 1):].view(np.int64)[0] = rows + 1
    with pytest.raises(trace.TraceError):
        trace.record_info(bad)


def test_record_size_rejects_bad_shapes(lib):
    assert lib.trace_record_size(0, 4, 32, 1) == 0          # no guide kind
    assert lib.trace_record_size(1, 4, 48, 1) == 0          # cols % 32
    assert lib.trace_record_size(2, 4, 32, 0) == 0          # no segments
    assert lib.trace_record_size(2, 4, 32, 4001) == 0
    # sizes: header page + 256-aligned sections (compact 4 B per 16 elements)
    assert lib.trace_record_size(2, 16, 32, 1) == 256 + 256 + 256 + 256 + 16


def test_record_calls_without_handle(lib):
    from fp4_rollout_guided_gb300.trace import Segments
    p = ctypes.c_void_p(256)
    buf = ctypes.create_string_buffer(4096)
    assert lib.trace_record_export(None, 2, p, p, p, 1, 32, Segments(None, 1), buf, 4096,
                                   None) == 1
    assert lib.trace_record_import(None, buf, 4096, p, p, p, None) == 1
    assert lib.trace_record_info(buf, 4096, None) == 1


def test_options_and_device_status_without_handle(lib):
    assert lib.trace_set_option(None, 0, 1) == 1
    assert lib.trace_device_status(None, None) == 1


def test_mma_scale_bytes_match_the_oracle(lib):
    import oracle
    oracle.build()
    for rows, cols in ((1, 32), (130, 96), (256, 64), (4097, 4096)):
        assert lib.trace_block_scales_mma_bytes(rows, cols) == \
            oracle._load().orc_mma_scales_bytes(rows, cols)
    assert lib.trace_block_scales_mma_bytes(4, 48) == 0
    assert lib.trace_block_scales_mma_bytes(-1, 32) == 0


def test_gemm_calls_without_handle(lib):
    p = ctypes.c_void_p(256)
    assert lib.trace_block_scales_mma(None, p, 4, 32, p, None) == 1
    assert lib.trace_nvfp4_gemm(None, p, p, p, p, p, p, 16, 16, 64, p, 0, None) == 1
