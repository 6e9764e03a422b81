"""Guard bytes around every output, in place of a device-side memory checker.

compute-sanitizer is not available on the GPUs these tests run on, so every
output buffer is carved out of a larger allocation whose bytes before and
after it hold a fixed pattern; each entry point then runs on ragged shapes
(one row, rows that end inside a CTA step, columns that are not a multiple
of 64, segment tables with empty segments) with its outputs placed at
16-byte-only offsets, and the guards must come back unchanged.  Inputs get
the same treatment, so a kernel that reads past its input would also meet
the pattern (the results are checked against the ordinary call, which
would then differ).
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from fp4_rollout_guided_gb300 import build, trace
    build.build()
    hd = trace.Handle(0)
    yield hd
    hd.close()


class Guarded:
    """Tensors carved out of one allocation, each between guard regions."""

    def __init__(self):
        self.bufs = []

    def tensor(self, shape, dtype, offset=16, fill=None):
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        buf = torch.full((GUARD + offset + nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                         device=DEV)
        view = buf[GUARD + offset:GUARD + offset + nbytes].view(dtype).view(shape)
        if fill is not None:
            view.copy_(fill)
        self.bufs.append((buf, offset, nbytes))
        return view

    def check(self, label):
        torch.cuda.synchronize()
        for i, (buf, offset, nbytes) in enumerate(self.bufs):
            head = buf[:GUARD + offset]
            tail = buf[GUARD + offset + nbytes:]
            assert torch.all(head == PATTERN), f"{label}: bytes before buffer {i} overwritten"
            assert torch.all(tail == PATTERN), f"{label}: bytes after buffer {i} overwritten"


SHAPES = [(1, 32, None), (3, 96, [0, 0, 2, 3]), (257, 64, [0, 100, 100, 257]),
          (4099, 128, [0, 2048, 4099]), (130, 2048, [0, 1, 129, 130]), (17, 160, None)]


def rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("offset", [16, 48])
@pytest.mark.parametrize("rows,cols,seg", SHAPES)
def test_every_entry_point_stays_inside_its_buffers(h, rows, cols, seg, offset):
    from fp4_rollout_guided_gb300 import trace
    seg = None if seg is None else np.array(seg, np.int64)
    n_seg = 1 if seg is None else len(seg) - 1
    xr = rand((rows, cols), rows + cols, 2.0)
    rr = (xr.float() * (1 + 2.0 ** -6 * torch.randn(xr.shape, generator=torch.Generator()
                                                     .manual_seed(5)))).to(torch.bfloat16)
    g = Guarded()
    x = g.tensor((rows, cols), torch.bfloat16, offset, xr)
    r = g.tensor((rows, cols), torch.bfloat16, offset, rr)
    want = h.rollout_quant(rr.to(DEV), seg)
    label = f"{rows}x{cols} seg={None if seg is None else list(seg)} offset={offset}"

    for fused, wave in ((1, 4096), (1, 1 << 20), (0, 16 << 20)):
        h.set_option("fused_amax", fused)
        h.set_option("wave_bytes", wave)
        try:
            out = (g.tensor((rows, cols // 2), torch.uint8, offset),
                   g.tensor((rows, cols // 16), torch.uint8, offset),
                   g.tensor((n_seg,), torch.float32, offset),
                   g.tensor((rows, cols // 16), torch.int32, offset))
            h.rollout_quant(r, seg, out=out)
        finally:
            h.set_option("fused_amax", 1)
            h.set_option("wave_bytes", 32 << 20)
        g.check(f"rollout_quant fused={fused} wave={wave} {label}")
        for a, b in zip(out, want):
            assert torch.equal(a, b), label
    codes, bs, gs, guide = out
    packed = h.guide_pack(codes, out=g.tensor((rows, cols // 16), torch.int32, offset))
    unpacked = h.guide_unpack(x, guide, bs, gs, seg,
                              out=g.tensor((rows, cols // 2), torch.uint8, offset))
    g.check(f"pack / unpack {label}")
    assert torch.equal(packed, guide)
    for kind, gd in (("none", None), ("compact", guide), ("full", codes)):
        for want_codes, with_stats in ((False, False), (True, False), (True, True)):
            st = trace.new_stats(DEV) if with_stats else None
            o = (g.tensor((rows, cols), torch.bfloat16, offset),
                 g.tensor((rows, cols // 32), torch.int32, offset),
                 g.tensor((rows, cols // 2), torch.uint8, offset) if want_codes else None)
            args = (x, seg, kind) + (() if kind == "none" else (gd, bs, gs, seg))
            h.train_fakequant(*args, out=o, stats=st)
            ref = h.train_fakequant(*(tuple(a.clone() if torch.is_tensor(a) else a for a in args)),
                                    codes=want_codes)
            g.check(f"fakequant {kind} codes={want_codes} stats={with_stats} {label}")
            assert torch.equal(o[0], ref[0]) and torch.equal(o[1], ref[1]), label
    gin = h.ste_backward(x, o[1], out=g.tensor((rows, cols), torch.bfloat16, offset))
    gts = h.segment_amax(x, seg, out=g.tensor((n_seg,), torch.float32, offset))
    g.check(f"ste_backward / segment_amax {label}")
    assert gin.shape == x.shape and gts.shape == (n_seg,)
    nb = trace.lib().trace_block_scales_mma_bytes(rows, cols)
    mma = h.block_scales_mma(bs, rows, cols, out=g.tensor((nb,), torch.uint8, offset))
    o5 = (g.tensor((rows, cols // 2), torch.uint8, offset),
          g.tensor((rows, cols // 16), torch.uint8, offset),
          g.tensor((nb,), torch.uint8, offset), g.tensor((n_seg,), torch.float32, offset),
          g.tensor((rows, cols // 16), torch.int32, offset))
    h.rollout_quant_mma(r, seg, row_major=True, guide=True, out=o5)
    g.check(f"tile-layout scales {label}")
    assert torch.equal(o5[2], mma) and torch.equal(o5[0], codes)


def test_noalloc_entry_point_stays_inside_its_buffers():
    """The allocation-free rollout quantiser, including zero rows (it then
    only writes the global scales)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from fp4_rollout_guided_gb300 import build, trace
    build.build()
    lib = trace.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for rows, cols, seg in ((0, 64, [0, 0, 0]), (1, 32, None), (257, 96, [0, 0, 200, 257])):
        seg = None if seg is None else np.array(seg, np.int64)
        n_seg = 1 if seg is None else len(seg) - 1
        g = Guarded()
        x = g.tensor((rows, cols), torch.bfloat16, 16, rand((rows, cols), 3))
        codes = g.tensor((rows, cols // 2), torch.uint8, 48)
        bs = g.tensor((rows, cols // 16), torch.uint8, 16)
        gs = g.tensor((n_seg,), torch.float32, 48)
        guide = g.tensor((rows, cols // 16), torch.int32, 16)
        segs = trace.Segments(None, 1) if seg is None else trace.Segments(seg.ctypes.data, n_seg)
        st = lib.trace_rollout_quant_noalloc(
            ctypes.c_void_p(x.data_ptr()), rows, cols, segs, ctypes.c_void_p(codes.data_ptr()),
            ctypes.c_void_p(bs.data_ptr()), ctypes.c_void_p(gs.data_ptr()),
            ctypes.c_void_p(guide.data_ptr()), stream)
        assert st == 0, lib.trace_status_string(st)
        g.check(f"noalloc {rows}x{cols}")
        if rows == 0:
            assert torch.all(gs == 0)


@pytest.mark.parametrize("form", ["tc256", "tc128", "tc_pair"])
@pytest.mark.parametrize("m,n,k", [(130, 200, 96), (7, 36, 320), (257, 520, 544), (1, 8, 32)])
def test_nvfp4_gemm_stays_inside_its_output(h, form, m, n, k):
    """The tcgen05 GEMM's stores (tile tails in rows, columns and k; element
    stores when a row is not a multiple of 16 bytes) stay inside d, for fp32
    and bf16 outputs; inputs between guards too."""
    x, w = rand((m, k), m + k, 2.0), rand((n, k), n + 3, 2.0)
    ref_a, ref_b = h.nvfp4_operand(x.to(DEV)), h.nvfp4_operand(w.to(DEV))
    g = Guarded()
    a = tuple(g.tensor(t.shape, t.dtype, 16, t) for t in ref_a)
    b = tuple(g.tensor(t.shape, t.dtype, 48, t) for t in ref_b)
    h.set_option("gemm", form)
    try:
        for dt in (torch.float32, torch.bfloat16):
            want = h.nvfp4_gemm(ref_a, ref_b, out_dtype=dt)
            d = g.tensor((m, n), dt, 16)
            h.nvfp4_gemm(a, b, out=d)
            g.check(f"nvfp4_gemm {form} {m}x{n}x{k} {dt}")
            assert h.device_status() == 0
            assert torch.equal(d, want), (form, m, n, k, dt)
    finally:
        h.set_option("gemm", "tc256")
