"""The allocation-free rollout quantiser, checked against the regular one.

trace_rollout_quant_noalloc serves callers that must not call cudaMalloc
(code inside a device allocator or memory pool, runtimes that pre-reserve
all device memory, allocation-free real-time loops) and so cannot create a
handle.  Its scratch is a fixed array in the library.  This test calls it
through the C ABI twice in a row, on two different inputs, and requires
exactly the outputs of trace_rollout_quant (the same bit-exact standard as
every other parity test here), which also shows the shared scratch carries
nothing over from one call to the next.  The file name sorts last so that a
run stopping at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_noalloc_matches_handle_path_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from fp4_rollout_guided_gb300 import build, synth, trace
    build.build()
    lib = trace.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    cases = []
    for cfg, seed in ((2, 0), (5, 3)):
        w = synth.workload(cfg, small=True, seed=seed)
        x, r = synth.make_inputs(w, "cpu")
        cases.append((w, r.to(dev)))
    assert cases[1][0].n_seg_r <= lib_limit()

    with trace.Handle(0) as h:
        for w, r in cases:
            rows, cols = r.shape
            want = h.rollout_quant(r, w.seg_r)
            codes = torch.full((rows, cols // 2), 0xAB, dtype=torch.uint8, device=dev)
            bs = torch.full((rows, cols // 16), 0xCD, dtype=torch.uint8, device=dev)
            gs = torch.full((w.n_seg_r,), -1.0, dtype=torch.float32, device=dev)
            guide = torch.full((rows, cols // 16), -1, dtype=torch.int32, device=dev)
            seg = np.ascontiguousarray(w.seg_r, dtype=np.int64)
            st = lib.trace_rollout_quant_noalloc(
                ctypes.c_void_p(r.data_ptr()), rows, cols,
                trace.Segments(seg.ctypes.data, len(seg) - 1),
                ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(bs.data_ptr()),
                ctypes.c_void_p(gs.data_ptr()), ctypes.c_void_p(guide.data_ptr()), stream)
            assert st == 0, lib.trace_status_string(st)
            torch.cuda.synchronize()
            for name, got, exp in zip(("codes", "bs", "gs", "guide"), (codes, bs, gs, guide), want):
                assert torch.equal(got, exp), name


def _call(lib, trace, r, seg, codes, bs, gs, guide, stream):
    rows, cols = r.shape
    segs = trace.Segments(None, 1) if seg is None else trace.Segments(seg.ctypes.data,
                                                                       len(seg) - 1)
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.trace_rollout_quant_noalloc(vp(r), rows, cols, segs, vp(codes), vp(bs), vp(gs),
                                           vp(guide), stream)


@pytest.mark.parametrize("case", ["one_segment", "no_guide", "limit_segments", "empty"])
def test_noalloc_edge_cases_match_handle_path(case):
    """A missing segment table (one segment), no guide words, exactly the
    segment limit, and zero rows: the same outputs as trace_rollout_quant."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from fp4_rollout_guided_gb300 import build, trace
    build.build()
    lib = trace.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    g = torch.Generator().manual_seed(7)
    n = lib_limit()
    rows, cols, seg = {"one_segment": (300, 96, None), "no_guide": (257, 64, [0, 100, 257]),
                       "limit_segments": (n * 2 + 5, 32, None), "empty": (0, 64, [0, 0, 0])}[case]
    if case == "limit_segments":
        counts = np.full(n, 2)
        counts[-1] += 5
        seg = np.concatenate([[0], np.cumsum(counts)])
    seg = None if seg is None else np.ascontiguousarray(seg, dtype=np.int64)
    r = (torch.randn((rows, cols), generator=g) * 3.0).to(torch.bfloat16).to(dev)
    n_seg = 1 if seg is None else len(seg) - 1
    with trace.Handle(0) as h:
        want = h.rollout_quant(r, seg)
        codes = torch.full((rows, cols // 2), 0xAB, dtype=torch.uint8, device=dev)
        bs = torch.full((rows, cols // 16), 0xCD, dtype=torch.uint8, device=dev)
        gs = torch.full((n_seg,), -1.0, dtype=torch.float32, device=dev)
        guide = None if case == "no_guide" else torch.full((rows, cols // 16), -1,
                                                             dtype=torch.int32, device=dev)
        for _ in range(2):
            st = _call(lib, trace, r, seg, codes, bs, gs, guide, stream)
            assert st == 0, lib.trace_status_string(st)
            torch.cuda.synchronize()
            assert torch.equal(codes, want[0]) and torch.equal(bs, want[1])
            assert torch.equal(gs, want[2])
            if guide is not None:
                assert torch.equal(guide, want[3])
    if case == "empty":
        assert torch.all(gs == 0)


def test_noalloc_rejects_too_many_segments():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from fp4_rollout_guided_gb300 import build, trace
    build.build()
    lib = trace.lib()
    n = lib_limit() + 1
    rows, cols = n, 32
    dev = torch.device("cuda", 0)
    x = torch.zeros(rows, cols, dtype=torch.bfloat16, device=dev)
    out = torch.empty(rows * cols, dtype=torch.uint8, device=dev)
    gs = torch.empty(n, dtype=torch.float32, device=dev)
    seg = np.arange(n + 1, dtype=np.int64)
    p = ctypes.c_void_p(out.data_ptr())
    st = lib.trace_rollout_quant_noalloc(ctypes.c_void_p(x.data_ptr()), rows, cols,
                                         trace.Segments(seg.ctypes.data, n), p, p,
                                         ctypes.c_void_p(gs.data_ptr()), None, None)
    assert st == 1   # TRACE_ERR_INVALID_ARG, nothing enqueued
    # exactly the limit is accepted
    seg = np.arange(n, dtype=np.int64)
    seg[-1] = rows
    codes = torch.empty(rows * cols // 2, dtype=torch.uint8, device=dev)
    bs = torch.empty(rows * cols // 16, dtype=torch.uint8, device=dev)
    st = lib.trace_rollout_quant_noalloc(ctypes.c_void_p(x.data_ptr()), rows, cols,
                                         trace.Segments(seg.ctypes.data, n - 1),
                                         ctypes.c_void_p(codes.data_ptr()),
                                         ctypes.c_void_p(bs.data_ptr()),
                                         ctypes.c_void_p(gs.data_ptr()), None, None)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.all(gs[:n - 1] == 0) and torch.all(codes == 0)   # x is all zeros


def lib_limit():
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "trace_fp4.h")).read()
    return int(re.search(r"#define TRACE_NOALLOC_MAX_SEGMENTS (\d+)", text).group(1))
