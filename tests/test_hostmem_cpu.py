"""Host logic of the huge-page host allocator, on the CPU: a fake CUDA runtime
records the registrations (no GPU, no page locking)."""

import gc

import torch

from fp4_rollout_guided_gb300 import hostmem


class _FakeRuntime:
    def __init__(self):
        self.live = {}
        self.calls = []

    def cudaHostRegister(self, addr, size, flags):
        self.calls.append(("register", addr, size, flags))
        self.live[addr] = size
        return 0

    def cudaHostUnregister(self, addr):
        self.calls.append(("unregister", addr))
        assert addr in self.live
        del self.live[addr]
        return 0


def _with_fake(monkeypatch):
    fake = _FakeRuntime()
    monkeypatch.setattr(torch.cuda, "cudart", lambda: fake)
    return fake


def test_sizes_rounding_and_zero_fill(monkeypatch):
    fake = _with_fake(monkeypatch)
    small = hostmem.host_empty((3, 5), torch.bfloat16)
    assert small.shape == (3, 5) and small.dtype == torch.bfloat16
    assert torch.count_nonzero(small).item() == 0
    big = hostmem.host_empty((hostmem._HUGE + 10,), torch.uint8)
    sizes = [c[2] for c in fake.calls if c[0] == "register"]
    import mmap
    assert sizes[0] == mmap.PAGESIZE                     # below a huge page: page-rounded
    assert sizes[1] == 2 * hostmem._HUGE                 # whole huge pages
    assert all(c[3] == 0 for c in fake.calls if c[0] == "register")
    empty = hostmem.host_empty((0, 7), torch.float32)
    assert empty.shape == (0, 7)
    del small, big, empty
    gc.collect()
    assert fake.live == {}


def test_views_keep_the_registration_until_the_last_one_goes(monkeypatch):
    fake = _with_fake(monkeypatch)
    t = hostmem.host_empty((1024,), torch.float32)
    t[:] = 2.5
    v = t[100:110].view(2, 5)
    del t
    gc.collect()
    assert len(fake.live) == 1 and torch.all(v == 2.5)
    w = v[1]
    del v
    gc.collect()
    assert len(fake.live) == 1 and torch.all(w == 2.5)
    del w
    gc.collect()
    assert fake.live == {}
    assert [c[0] for c in fake.calls] == ["register", "unregister"]


def test_like_matches_shape_and_dtype(monkeypatch):
    _with_fake(monkeypatch)
    src = torch.zeros((4, 6), dtype=torch.int32)
    t = hostmem.host_empty_like(src)
    assert t.shape == src.shape and t.dtype == src.dtype
