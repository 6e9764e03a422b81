"""Argument errors with a live handle: every bad call returns its status
before anything is enqueued, and the handle keeps working afterwards."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from fp4_rollout_guided_gb300 import build, trace
    build.build()
    h = trace.Handle(0)
    yield trace, h
    h.close()


def test_status_codes(env):
    trace, h = env
    lib = trace.lib()
    dev = torch.device("cuda", 0)
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device=dev)
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    p = ctypes.c_void_p(buf.data_ptr())
    odd = ctypes.c_void_p(buf.data_ptr() + 8)
    xs = ctypes.c_void_p(x.data_ptr())
    one = trace.Segments(None, 1)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    H = h._h
    # shapes
    assert lib.trace_rollout_quant(H, xs, 4, 48, one, p, p, p, None, s) == 1
    assert lib.trace_rollout_quant(H, xs, -1, 64, one, p, p, p, None, s) == 1
    assert lib.trace_rollout_quant(H, xs, 4, 0, one, p, p, p, None, s) == 1
    assert lib.trace_rollout_quant(H, xs, 1 << 31, 64, one, p, p, p, None, s) == 1
    # alignment
    assert lib.trace_rollout_quant(H, odd, 4, 64, one, p, p, p, None, s) == 2
    assert lib.trace_rollout_quant(H, xs, 4, 64, one, odd, p, p, None, s) == 2
    assert lib.trace_guide_pack(H, odd, 4, 64, p, s) == 2
    # null pointers
    assert lib.trace_rollout_quant(H, None, 4, 64, one, p, p, p, None, s) == 1
    assert lib.trace_rollout_quant(H, xs, 4, 64, one, p, p, None, None, s) == 1
    # segment tables: wrong ends, decreasing, too many
    keep = []
    for bad in ([0, 3], [1, 4], [0, 3, 2, 4], list(range(0, 4)) + [4] * 3998):
        arr = np.asarray(bad, np.int64)
        keep.append(arr)
        seg = trace.Segments(arr.ctypes.data, len(arr) - 1)
        if len(arr) - 1 > trace.MAX_SEGMENTS:
            assert lib.trace_rollout_quant(H, xs, 4, 64, seg, p, p, p, None, s) == 1
        else:
            assert lib.trace_rollout_quant(H, xs, 4, 64, seg, p, p, p, None, s) == 1
    # guide kinds
    assert lib.trace_train_fakequant(H, xs, 4, 64, one, 7, p, p, p, one, p, None, None, None,
                                     s) == 1
    assert lib.trace_train_fakequant(H, xs, 4, 64, one, 2, None, p, p, one, p, None, None, None,
                                     s) == 1
    assert lib.trace_train_fakequant(H, xs, 4, 64, one, 2, p, p, None, one, p, None, None, None,
                                     s) == 1
    # the handle still works
    codes, bs, gs, guide = h.rollout_quant(x)
    torch.cuda.synchronize()
    assert torch.all(codes == 0) and gs.item() == 0.0
    assert lib.trace_last_cuda_error(H) == 0


def test_python_binding_checks(env):
    trace, h = env
    dev = torch.device("cuda", 0)
    with pytest.raises(ValueError):
        h.rollout_quant(torch.zeros(4, 64, dtype=torch.float32, device=dev))
    with pytest.raises(ValueError):
        h.rollout_quant(torch.zeros(4, 64, dtype=torch.bfloat16))       # host tensor
    with pytest.raises(trace.TraceError):
        h.rollout_quant(torch.zeros(4, 48, dtype=torch.bfloat16, device=dev))


def test_profiler_counts_launches(env):
    trace, h = env
    dev = torch.device("cuda", 0)
    x = torch.randn(512, 256, device=dev).to(torch.bfloat16)
    h.profile(True)
    codes, bs, gs, guide = h.rollout_quant(x)
    h.train_fakequant(x, None, "compact", guide, bs, gs)
    h.guide_pack(codes)
    t = h.collect()
    h.profile(False)
    # rollout side: one fused launch (the whole tensor fits a wave); training
    # side: amax + fake quant
    assert t["rollout_fused"][0] == 1 and t["rollout_quant"][0] == 0
    assert t["amax"][0] == 1 and t["fakequant"][0] == 1
    assert t["guide_pack"][0] == 1 and t["guide_unpack"][0] == 0
    assert all(ms >= 0 for _, ms in t.values())
    assert h.collect()["amax"][0] == 0
