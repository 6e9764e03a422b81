"""Page-locked, huge-page-backed host buffers (fp4_rollout_guided_gb300.hostmem)."""

import gc

import pytest
import torch

from fp4_rollout_guided_gb300 import hostmem

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.mark.parametrize("shape,dtype", [((0,), torch.float32), ((3, 5), torch.bfloat16),
                                         ((7,), torch.uint8), ((2, 3, 4), torch.int32)])
def test_host_empty_shapes_zero_filled(shape, dtype):
    t = hostmem.host_empty(shape, dtype)
    assert t.shape == shape and t.dtype == dtype and t.device.type == "cpu"
    assert t.is_contiguous()
    assert torch.count_nonzero(t).item() == 0


def test_host_empty_round_trip_beyond_a_huge_page():
    n = hostmem._HUGE + (3 << 20) + 6  # more than one huge page, not a multiple of one
    src = hostmem.host_empty((n,), torch.uint8)
    src.copy_(torch.randint(0, 256, (n,), dtype=torch.uint8, generator=torch.Generator().manual_seed(3)))
    back = hostmem.host_empty_like(src)
    s = torch.cuda.Stream(DEV)
    d = torch.empty(n, dtype=torch.uint8, device=DEV)
    with torch.cuda.stream(s):
        d.copy_(src, non_blocking=True)
        back.copy_(d, non_blocking=True)
    s.synchronize()
    assert torch.equal(back, src)


def test_host_empty_views_keep_the_buffer_and_release_it():
    t = hostmem.host_empty((1 << 20,), torch.float32)
    t[:] = 1.5
    view = t[10:20].view(2, 5)
    del t
    gc.collect()
    d = view.to(DEV, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.all(d == 1.5)
    del view, d
    gc.collect()
    # allocating and dropping many buffers leaves nothing registered behind
    for _ in range(20):
        b = hostmem.host_empty((64 << 20,), torch.uint8)
        b[-1] = 7
        del b
    gc.collect()
