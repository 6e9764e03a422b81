"""Thin ctypes binding over ``libtrace_fp4.so`` (include/trace_fp4.h).

Argument marshalling only: every step of the path runs in the library's
sm_103a kernels.  PyTorch supplies device memory and the current CUDA stream.
If the library has not been built, or no compute capability 10.3 GPU is
present, calls raise :class:`TraceError`; there is no fallback path.

Tensor dtypes: bf16 inputs are ``torch.bfloat16``; codes and block scales
are ``torch.uint8``; compact words and STE masks are ``torch.int32`` holding
the unsigned 32-bit patterns; global scales are ``torch.float32``; the
statistics block is ``torch.int64[11]`` (the layout of ``trace_stats_t``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

from . import build as _build
from . import hostmem

GUIDE_NONE, GUIDE_FULL, GUIDE_COMPACT = 0, 1, 2
_KINDS = {"none": GUIDE_NONE, "full": GUIDE_FULL, "compact": GUIDE_COMPACT}
KERNELS = ("amax", "rollout_quant", "guide_pack", "guide_unpack", "fakequant", "ste_backward",
           "rollout_fused", "mma_scales", "nvfp4_gemm", "rollout_delayed")
OPTIONS = {"fused_amax": 0, "wave_bytes": 1, "wait_limit_ns": 2, "wait_extra": 3,
           "debug_shrink": 4, "gemm": 5}
# values of the "gemm" option: the form of nvfp4_gemm
GEMM_FORMS = {"tc256": 0, "cublaslt": 1, "tc128": 2, "tc_pair": 3}
MAX_SEGMENTS = 4000
STATUS = {0: "ok", 1: "invalid argument", 2: "alignment", 3: "unsupported device",
          4: "CUDA error", 5: "out of memory", 6: "timeout", 7: "cuBLASLt missing or refused"}


class TraceError(RuntimeError):
    def __init__(self, where: str, status: int, cuda_error: int = 0):
        msg = f"{where}: {STATUS.get(status, status)}"
        if cuda_error:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)
        self.status = status
        self.cuda_error = cuda_error


class Segments(ctypes.Structure):
    _fields_ = [("row_offsets", ctypes.c_void_p), ("n_seg", ctypes.c_int32)]


class KernelTime(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_uint64), ("total_ms", ctypes.c_double)]


_lock = threading.Lock()
_lib = None

# name -> (restype, argtypes); every symbol the header declares
P, I64, I32, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
SIGNATURES = {
    "trace_create": (INT, [ctypes.POINTER(ctypes.c_void_p), INT]),
    "trace_destroy": (INT, [P]),
    "trace_status_string": (ctypes.c_char_p, [INT]),
    "trace_last_cuda_error": (INT, [P]),
    "trace_version": (INT, []),
    "trace_rollout_quant": (INT, [P, P, I64, I64, Segments, P, P, P, P, P]),
    "trace_guide_pack": (INT, [P, P, I64, I64, P, P]),
    "trace_guide_unpack": (INT, [P, P, P, P, P, Segments, I64, I64, P, P]),
    "trace_train_fakequant": (INT, [P, P, I64, I64, Segments, INT, P, P, P, Segments, P, P,
                                    P, P, P]),
    "trace_train_fakequant_gs": (INT, [P, P, I64, I64, Segments, P, INT, P, P, P, Segments, P,
                                       P, P, P, P]),
    "trace_train_fakequant_delayed": (INT, [P, P, I64, I64, Segments, P, INT, P, P, P,
                                             Segments, P, P, P, P]),
    "trace_segment_amax": (INT, [P, P, I64, I64, Segments, P, P]),
    "trace_ste_backward": (INT, [P, P, P, I64, I64, P, P]),
    "trace_set_option": (INT, [P, INT, I64]),
    "trace_device_status": (INT, [P, P]),
    "trace_debug_bounds": (INT, [P, ctypes.POINTER(ctypes.c_int),
                                 ctypes.POINTER(ctypes.c_uint64)]),
    "trace_rollout_quant_mma": (INT, [P, P, I64, I64, Segments, P, P, P, P, P, P]),
    "trace_rollout_quant_delayed": (INT, [P, P, I64, I64, Segments, P, P, P, P, P, P, P]),
    "trace_block_scales_mma_bytes": (ctypes.c_size_t, [I64, I64]),
    "trace_block_scales_mma": (INT, [P, P, I64, I64, P, P]),
    "trace_nvfp4_gemm": (INT, [P, P, P, P, P, P, P, I64, I64, I64, P, INT, P]),
    "trace_record_size": (ctypes.c_size_t, [INT, I64, I64, ctypes.c_int32]),
    "trace_record_export": (INT, [P, INT, P, P, P, I64, I64, Segments, P, ctypes.c_size_t, P]),
    "trace_record_info": (INT, [P, ctypes.c_size_t, P]),
    "trace_record_import": (INT, [P, P, ctypes.c_size_t, P, P, P, P]),
    "trace_rollout_quant_noalloc": (INT, [P, I64, I64, Segments, P, P, P, P, P]),
    "trace_profile_enable": (INT, [P, INT]),
    "trace_profile_collect": (INT, [P, ctypes.POINTER(KernelTime)]),
}


RECORD_MAGIC = 0x31475254


class RecordHeader(ctypes.Structure):
    """trace_record_header_t: the 64-byte header of a guide record."""
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32),
                ("kind", ctypes.c_uint32), ("n_seg", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("guide_offset", ctypes.c_uint64), ("bs_offset", ctypes.c_uint64),
                ("gs_offset", ctypes.c_uint64), ("seg_offset", ctypes.c_uint64)]


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded library; raises TraceError if it was never built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise TraceError(f"libtrace_fp4.so missing at {path}; build it with "
                                 "__graft_entry__.build()", 3)
            so = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(so, name)
                fn.restype = res
                fn.argtypes = args
            _lib = so
        return _lib


def _segments(seg, rows, keep: list) -> Segments:
    if seg is None:
        return Segments(None, 1)
    arr = np.ascontiguousarray(np.asarray(seg, dtype=np.int64))
    keep.append(arr)
    return Segments(arr.ctypes.data, len(arr) - 1)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t: torch.Tensor, dtype, shape, name, device):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)}, got "
                         f"{t.dtype} {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name}: expected a tensor on {device}, got {t.device}")


class Handle:
    """One library handle on one CUDA device (owns a small device scratch)."""

    def __init__(self, device: Optional[int] = None):
        if device is None:
            device = torch.cuda.current_device()
        self.device_index = int(device)
        self.device = torch.device("cuda", self.device_index)
        h = ctypes.c_void_p()
        st = lib().trace_create(ctypes.byref(h), self.device_index)
        if st != 0:
            raise TraceError("trace_create", st)
        self._h = h

    # -- life cycle ----------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            torch.cuda.synchronize(self.device)
            lib().trace_destroy(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            if getattr(self, "_h", None):
                lib().trace_destroy(self._h)
                self._h = None
        except Exception:
            pass

    def _check(self, where, st):
        if st != 0:
            raise TraceError(where, st, lib().trace_last_cuda_error(self._h))

    # -- a1 + a2 ---------------------------------------------------------------
    def rollout_quant(self, x: torch.Tensor, seg=None, *, guide: bool = True, out=None):
        """-> (codes uint8[rows, cols/2], bs uint8[rows, cols/16],
        gs float32[n_seg], guide int32[rows, cols/16] or None)."""
        rows, cols = x.shape
        n_seg = 1 if seg is None else len(seg) - 1
        if out is None:
            out = (torch.empty((rows, cols // 2), dtype=torch.uint8, device=self.device),
                   torch.empty((rows, cols // 16), dtype=torch.uint8, device=self.device),
                   torch.empty((n_seg,), dtype=torch.float32, device=self.device),
                   torch.empty((rows, cols // 16), dtype=torch.int32, device=self.device)
                   if guide else None)
        codes, bs, gs, gd = out
        _need(x, torch.bfloat16, (rows, cols), "x", self.device)
        _need(codes, torch.uint8, (rows, cols // 2), "codes", self.device)
        _need(bs, torch.uint8, (rows, cols // 16), "bs", self.device)
        _need(gs, torch.float32, (n_seg,), "gs", self.device)
        if gd is not None:
            _need(gd, torch.int32, (rows, cols // 16), "guide", self.device)
        keep = []
        st = lib().trace_rollout_quant(self._h, _ptr(x), rows, cols, _segments(seg, rows, keep),
                                       _ptr(codes), _ptr(bs), _ptr(gs), _ptr(gd), _stream())
        self._check("trace_rollout_quant", st)
        return codes, bs, gs, gd

    def rollout_quant_delayed(self, x: torch.Tensor, seg, amax_prev: torch.Tensor, *,
                              guide: bool = True, amax_out: bool = True, out=None):
        """Rollout quantisation scaled by given per-segment maxima (delayed
        scaling): -> (codes, bs, gs, guide or None, this tensor's maxima
        float32[n_seg] or None)."""
        rows, cols = x.shape
        n_seg = 1 if seg is None else len(seg) - 1
        if out is None:
            out = (torch.empty((rows, cols // 2), dtype=torch.uint8, device=self.device),
                   torch.empty((rows, cols // 16), dtype=torch.uint8, device=self.device),
                   torch.empty((n_seg,), dtype=torch.float32, device=self.device),
                   torch.empty((rows, cols // 16), dtype=torch.int32, device=self.device)
                   if guide else None,
                   torch.empty((n_seg,), dtype=torch.float32, device=self.device)
                   if amax_out else None)
        codes, bs, gs, gd, am = out
        _need(x, torch.bfloat16, (rows, cols), "x", self.device)
        _need(amax_prev, torch.float32, (n_seg,), "amax_prev", self.device)
        _need(codes, torch.uint8, (rows, cols // 2), "codes", self.device)
        _need(bs, torch.uint8, (rows, cols // 16), "bs", self.device)
        _need(gs, torch.float32, (n_seg,), "gs", self.device)
        if gd is not None:
            _need(gd, torch.int32, (rows, cols // 16), "guide", self.device)
        if am is not None:
            _need(am, torch.float32, (n_seg,), "amax_out", self.device)
        keep = []
        st = lib().trace_rollout_quant_delayed(self._h, _ptr(x), rows, cols,
                                               _segments(seg, rows, keep), _ptr(amax_prev),
                                               _ptr(codes), _ptr(bs), _ptr(gs), _ptr(gd),
                                               _ptr(am), _stream())
        self._check("trace_rollout_quant_delayed", st)
        return codes, bs, gs, gd, am

    # -- a3 ----------------------------------------------------------------------
    def guide_pack(self, codes: torch.Tensor, out: Optional[torch.Tensor] = None):
        rows, half = codes.shape
        cols = half * 2
        if out is None:
            out = torch.empty((rows, cols // 16), dtype=torch.int32, device=self.device)
        _need(codes, torch.uint8, (rows, half), "codes", self.device)
        _need(out, torch.int32, (rows, cols // 16), "guide", self.device)
        st = lib().trace_guide_pack(self._h, _ptr(codes), rows, cols, _ptr(out), _stream())
        self._check("trace_guide_pack", st)
        return out

    # -- a4 ----------------------------------------------------------------------
    def guide_unpack(self, x_ref, guide, bs_r, gs_r, seg_r=None, out=None):
        rows, cols = x_ref.shape
        if out is None:
            out = torch.empty((rows, cols // 2), dtype=torch.uint8, device=self.device)
        _need(x_ref, torch.bfloat16, (rows, cols), "x_ref", self.device)
        _need(guide, torch.int32, (rows, cols // 16), "guide", self.device)
        _need(bs_r, torch.uint8, (rows, cols // 16), "bs_r", self.device)
        _need(out, torch.uint8, (rows, cols // 2), "codes", self.device)
        keep = []
        st = lib().trace_guide_unpack(self._h, _ptr(x_ref), _ptr(guide), _ptr(bs_r), _ptr(gs_r),
                                      _segments(seg_r, rows, keep), rows, cols, _ptr(out),
                                      _stream())
        self._check("trace_guide_unpack", st)
        return out

    # -- a5 + a6 -----------------------------------------------------------------
    def segment_amax(self, x: torch.Tensor, seg=None, out: Optional[torch.Tensor] = None):
        """-> gs float32[n_seg]: per-segment amax / 2688 (one streaming kernel)."""
        rows, cols = x.shape
        _need(x, torch.bfloat16, (rows, cols), "x", self.device)
        keep = []
        sg = _segments(seg, rows, keep)
        if out is None:
            out = torch.empty(sg.n_seg, dtype=torch.float32, device=self.device)
        _need(out, torch.float32, (sg.n_seg,), "gs", self.device)
        self._check("trace_segment_amax",
                    lib().trace_segment_amax(self._h, _ptr(x), rows, cols, sg, _ptr(out),
                                             _stream()))
        return out

    def train_fakequant(self, x, seg_t=None, kind="none", guide=None, bs_r=None, gs_r=None,
                        seg_r=None, *, mask: bool = True, codes: bool = False,
                        stats: Optional[torch.Tensor] = None, out=None,
                        gs_t: Optional[torch.Tensor] = None):
        """-> (y bf16[rows, cols], mask int32[rows, cols/32] or None,
        codes uint8[rows, cols/2] or None, stats).  With gs_t (the training
        scales from segment_amax) the amax pass is skipped."""
        k = _KINDS[kind] if isinstance(kind, str) else int(kind)
        rows, cols = x.shape
        if out is None:
            out = (torch.empty((rows, cols), dtype=torch.bfloat16, device=self.device),
                   torch.empty((rows, cols // 32), dtype=torch.int32, device=self.device)
                   if mask else None,
                   torch.empty((rows, cols // 2), dtype=torch.uint8, device=self.device)
                   if codes else None)
        y, m, c = out
        _need(x, torch.bfloat16, (rows, cols), "x", self.device)
        _need(y, torch.bfloat16, (rows, cols), "y", self.device)
        if m is not None:
            _need(m, torch.int32, (rows, cols // 32), "mask", self.device)
        if c is not None:
            _need(c, torch.uint8, (rows, cols // 2), "codes_t", self.device)
        if stats is not None:
            _need(stats, torch.int64, (11,), "stats", self.device)
        if k != GUIDE_NONE:
            if k == GUIDE_FULL:
                _need(guide, torch.uint8, (rows, cols // 2), "guide", self.device)
            else:
                _need(guide, torch.int32, (rows, cols // 16), "guide", self.device)
            _need(bs_r, torch.uint8, (rows, cols // 16), "bs_r", self.device)
        keep = []
        sgt = _segments(seg_t, rows, keep)
        if gs_t is None:
            st = lib().trace_train_fakequant(
                self._h, _ptr(x), rows, cols, sgt, k, _ptr(guide), _ptr(bs_r), _ptr(gs_r),
                _segments(seg_r, rows, keep), _ptr(y), _ptr(m), _ptr(c), _ptr(stats), _stream())
            self._check("trace_train_fakequant", st)
        else:
            _need(gs_t, torch.float32, (sgt.n_seg,), "gs_t", self.device)
            st = lib().trace_train_fakequant_gs(
                self._h, _ptr(x), rows, cols, sgt, _ptr(gs_t), k, _ptr(guide), _ptr(bs_r),
                _ptr(gs_r), _segments(seg_r, rows, keep), _ptr(y), _ptr(m), _ptr(c), _ptr(stats),
                _stream())
            self._check("trace_train_fakequant_gs", st)
        return y, m, c, stats

    def train_fakequant_delayed(self, x, seg_t, amax_prev, kind="none", guide=None, bs_r=None,
                                gs_r=None, seg_r=None, *, mask: bool = True,
                                amax_out: bool = True, out=None):
        """Training-side fake quantisation scaled by given per-segment maxima
        (delayed scaling): -> (y, mask or None, x's own training-segment
        maxima float32[n_seg_t] or None)."""
        k = _KINDS[kind] if isinstance(kind, str) else int(kind)
        rows, cols = x.shape
        n_seg = 1 if seg_t is None else len(seg_t) - 1
        if out is None:
            out = (torch.empty((rows, cols), dtype=torch.bfloat16, device=self.device),
                   torch.empty((rows, cols // 32), dtype=torch.int32, device=self.device)
                   if mask else None,
                   torch.empty((n_seg,), dtype=torch.float32, device=self.device)
                   if amax_out else None)
        y, m, am = out
        _need(x, torch.bfloat16, (rows, cols), "x", self.device)
        _need(y, torch.bfloat16, (rows, cols), "y", self.device)
        _need(amax_prev, torch.float32, (n_seg,), "amax_prev", self.device)
        if m is not None:
            _need(m, torch.int32, (rows, cols // 32), "mask", self.device)
        if am is not None:
            _need(am, torch.float32, (n_seg,), "amax_out", self.device)
        if k != GUIDE_NONE:
            if k == GUIDE_FULL:
                _need(guide, torch.uint8, (rows, cols // 2), "guide", self.device)
            else:
                _need(guide, torch.int32, (rows, cols // 16), "guide", self.device)
            _need(bs_r, torch.uint8, (rows, cols // 16), "bs_r", self.device)
        keep = []
        st = lib().trace_train_fakequant_delayed(
            self._h, _ptr(x), rows, cols, _segments(seg_t, rows, keep), _ptr(amax_prev), k,
            _ptr(guide), _ptr(bs_r), _ptr(gs_r), _segments(seg_r, rows, keep), _ptr(y), _ptr(m),
            _ptr(am), _stream())
        self._check("trace_train_fakequant_delayed", st)
        return y, m, am

    # -- backward ---------------------------------------------------------------
    def ste_backward(self, grad_out: torch.Tensor, mask: torch.Tensor, out=None):
        """grad_in = grad_out where the STE mask bit is 1, +0 elsewhere."""
        rows, cols = grad_out.shape
        if out is None:
            out = torch.empty_like(grad_out)
        _need(grad_out, torch.bfloat16, (rows, cols), "grad_out", self.device)
        _need(mask, torch.int32, (rows, cols // 32), "mask", self.device)
        _need(out, torch.bfloat16, (rows, cols), "grad_in", self.device)
        st = lib().trace_ste_backward(self._h, _ptr(grad_out), _ptr(mask), rows, cols, _ptr(out),
                                      _stream())
        self._check("trace_ste_backward", st)
        return out

    # -- guide transport ---------------------------------------------------------
    def record_export(self, guide: torch.Tensor, bs: torch.Tensor, gs: torch.Tensor, seg=None,
                      out: Optional[torch.Tensor] = None, wait: bool = True) -> torch.Tensor:
        """Copies a rollout record (guide, block scales, global scales and the
        segment table) into one pinned host buffer.  The guide's dtype names
        the kind: uint8 [rows, cols/2] full codes, int32 [rows, cols/16]
        compact words.  With wait=False the device-to-host copies are still
        in flight on the current stream when this returns."""
        rows = guide.shape[0]
        if guide.dtype == torch.uint8:
            k, cols = GUIDE_FULL, guide.shape[1] * 2
        elif guide.dtype == torch.int32:
            k, cols = GUIDE_COMPACT, guide.shape[1] * 16
        else:
            raise ValueError("guide must be uint8 (full) or int32 (compact)")
        n_seg = 1 if seg is None else len(seg) - 1
        _need(guide, guide.dtype, tuple(guide.shape), "guide", self.device)
        _need(bs, torch.uint8, (rows, cols // 16), "bs", self.device)
        _need(gs, torch.float32, (n_seg,), "gs", self.device)
        size = record_size(k, rows, cols, n_seg)
        if out is None:
            out = hostmem.host_empty((size,), torch.uint8)
        p, n = _host_ptr(out)
        keep = []
        st = lib().trace_record_export(self._h, k, _ptr(guide), _ptr(bs), _ptr(gs), rows, cols,
                                       _segments(seg, rows, keep), p, n, _stream())
        self._check("trace_record_export", st)
        if wait:
            torch.cuda.current_stream(self.device).synchronize()
        return out

    def record_import(self, buf, out=None):
        """-> (guide, bs, gs, seg_offsets) on this device from a record in host
        memory (pinned memory makes the copies asynchronous)."""
        hd, seg = record_info(buf)
        rows, cols = hd.rows, hd.cols
        if out is None:
            gshape = (rows, cols // 2) if hd.kind == GUIDE_FULL else (rows, cols // 16)
            gdt = torch.uint8 if hd.kind == GUIDE_FULL else torch.int32
            out = (torch.empty(gshape, dtype=gdt, device=self.device),
                   torch.empty((rows, cols // 16), dtype=torch.uint8, device=self.device),
                   torch.empty((hd.n_seg,), dtype=torch.float32, device=self.device))
        g, bs, gs = out
        p, n = _host_ptr(buf)
        st = lib().trace_record_import(self._h, p, n, _ptr(g), _ptr(bs), _ptr(gs), _stream())
        self._check("trace_record_import", st)
        return g, bs, gs, seg

    # -- f4: NVFP4 GEMM over rollout codes --------------------------------------------
    def block_scales_mma(self, bs: torch.Tensor, rows: int, cols: int, out=None):
        """Row-major block scales uint8[rows, cols/16] -> tensor-core tile layout."""
        n = lib().trace_block_scales_mma_bytes(rows, cols)
        if n == 0:
            raise TraceError("trace_block_scales_mma_bytes", 1)
        if out is None:
            out = torch.empty(n, dtype=torch.uint8, device=self.device)
        _need(bs, torch.uint8, (rows, cols // 16), "bs", self.device)
        _need(out, torch.uint8, (n,), "scales_mma", self.device)
        self._check("trace_block_scales_mma",
                    lib().trace_block_scales_mma(self._h, _ptr(bs), rows, cols, _ptr(out),
                                                 _stream()))
        return out

    def rollout_quant_mma(self, x: torch.Tensor, seg=None, *, row_major: bool = False,
                          guide: bool = False, out=None):
        """rollout_quant writing the block scales in the tensor-core tile
        layout -> (codes, bs row-major or None, bs tile layout, gs, guide or None)."""
        rows, cols = x.shape
        n_seg = 1 if seg is None else len(seg) - 1
        nb = lib().trace_block_scales_mma_bytes(rows, cols)
        if nb == 0 and rows > 0:
            raise TraceError("trace_block_scales_mma_bytes", 1)
        dev = self.device
        if out is None:
            out = (torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev),
                   torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
                   if row_major else None,
                   torch.empty((nb,), dtype=torch.uint8, device=dev),
                   torch.empty((n_seg,), dtype=torch.float32, device=dev),
                   torch.empty((rows, cols // 16), dtype=torch.int32, device=dev)
                   if guide else None)
        codes, bs, mma, gs, gd = out
        _need(x, torch.bfloat16, (rows, cols), "x", dev)
        _need(codes, torch.uint8, (rows, cols // 2), "codes", dev)
        if bs is not None:
            _need(bs, torch.uint8, (rows, cols // 16), "bs", dev)
        _need(mma, torch.uint8, (nb,), "bs_mma", dev)
        _need(gs, torch.float32, (n_seg,), "gs", dev)
        if gd is not None:
            _need(gd, torch.int32, (rows, cols // 16), "guide", dev)
        keep = []
        st = lib().trace_rollout_quant_mma(self._h, _ptr(x), rows, cols,
                                           _segments(seg, rows, keep), _ptr(codes), _ptr(bs),
                                           _ptr(mma), _ptr(gs), _ptr(gd), _stream())
        self._check("trace_rollout_quant_mma", st)
        return codes, bs, mma, gs, gd

    def nvfp4_operand(self, x: torch.Tensor, out=None):
        """One NVFP4 GEMM operand from bf16 x [rows, k] through the rollout
        quantiser (one segment, scales written in the tile layout):
        -> (codes, scales in tile layout, gs)."""
        o = None if out is None else (out[0], None, out[1], out[2], None)
        codes, _, mma, gs, _ = self.rollout_quant_mma(x, None, out=o)
        return codes, mma, gs

    def nvfp4_gemm(self, a, b, out=None, out_dtype=torch.float32):
        """a, b: (codes [rows, k/2], scales_mma, gs [1]) -> d [m, n] =
        fl32(gs_a * gs_b) * sum_k A[i, k] B[j, k]."""
        a_codes, a_sc, a_gs = a
        b_codes, b_sc, b_gs = b
        m, k = a_codes.shape[0], a_codes.shape[1] * 2
        n = b_codes.shape[0]
        if out is None:
            out = torch.empty((m, n), dtype=out_dtype, device=self.device)
        kind = {torch.float32: 0, torch.bfloat16: 1}[out.dtype]
        _need(out, out.dtype, (m, n), "d", self.device)
        _need(b_codes, torch.uint8, (n, k // 2), "b_codes", self.device)
        for t, name in ((a_sc, "a_scales"), (b_sc, "b_scales"), (a_gs, "a_gs"), (b_gs, "b_gs")):
            if t.device != self.device:
                raise ValueError(f"{name}: expected a tensor on {self.device}")
        self._check("trace_nvfp4_gemm",
                    lib().trace_nvfp4_gemm(self._h, _ptr(a_codes), _ptr(a_sc), _ptr(a_gs),
                                           _ptr(b_codes), _ptr(b_sc), _ptr(b_gs), m, n, k,
                                           _ptr(out), kind, _stream()))
        return out

    # -- options and device status -----------------------------------------------
    def set_option(self, name: str, value: int):
        """fused_amax (0/1), wave_bytes, wait_limit_ns, gemm (a GEMM_FORMS
        name or value), wait_extra and debug_shrink (test hooks)."""
        if name == "gemm" and isinstance(value, str):
            value = GEMM_FORMS[value]
        self._check("trace_set_option", lib().trace_set_option(self._h, OPTIONS[name], int(value)))

    def device_status(self) -> int:
        """Synchronises the current stream; 0, or 6 (timeout) if an in-kernel
        wait of an earlier call ran out.  Clears the device error word."""
        st = lib().trace_device_status(self._h, _stream())
        if st not in (0, 6):
            self._check("trace_device_status", st)
        return st

    def debug_bounds(self):
        """-> (checked, violations): whether this build checks global accesses
        against the calls' registered buffers (TRACE_DEBUG_BOUNDS), and the
        out-of-range accesses counted since the last query (waits for the device)."""
        c, v = ctypes.c_int(0), ctypes.c_uint64(0)
        self._check("trace_debug_bounds",
                    lib().trace_debug_bounds(self._h, ctypes.byref(c), ctypes.byref(v)))
        return bool(c.value), int(v.value)

    # -- profiler ---------------------------------------------------------------
    def profile(self, enable: bool = True):
        self._check("trace_profile_enable", lib().trace_profile_enable(self._h, int(enable)))

    def collect(self) -> dict:
        arr = (KernelTime * len(KERNELS))()
        self._check("trace_profile_collect", lib().trace_profile_collect(self._h, arr))
        return {name: (int(arr[i].launches), float(arr[i].total_ms))
                for i, name in enumerate(KERNELS)}


def new_stats(device) -> torch.Tensor:
    return torch.zeros(11, dtype=torch.int64, device=device)


def stats_dict(stats: torch.Tensor) -> dict:
    v = stats.cpu().numpy().astype(np.uint64)
    return {"n_elems": int(v[0]), "mismatch_rtn": int(v[1]), "mismatch_guided": int(v[2]),
            "hist_rtn": [int(a) for a in v[3:7]], "hist_guided": [int(a) for a in v[7:11]]}


def record_size(kind, rows: int, cols: int, n_seg: int = 1) -> int:
    """Bytes of a guide record of this shape (host-only call)."""
    k = _KINDS[kind] if isinstance(kind, str) else int(kind)
    n = lib().trace_record_size(k, rows, cols, n_seg)
    if n == 0:
        raise TraceError("trace_record_size", 1)
    return int(n)


def _host_ptr(buf) -> Tuple[ctypes.c_void_p, int]:
    if isinstance(buf, torch.Tensor):
        if buf.device.type != "cpu" or buf.dtype != torch.uint8 or not buf.is_contiguous():
            raise ValueError("a record is a contiguous uint8 CPU tensor")
        return ctypes.c_void_p(buf.data_ptr()), buf.numel()
    arr = np.ascontiguousarray(buf, dtype=np.uint8)
    return ctypes.c_void_p(arr.ctypes.data), arr.size


def record_info(buf) -> Tuple[RecordHeader, np.ndarray]:
    """Validates a record and returns its header and row offsets (host-only)."""
    keep = buf if isinstance(buf, torch.Tensor) else np.ascontiguousarray(buf, dtype=np.uint8)
    p, n = _host_ptr(keep)
    hd = RecordHeader()
    st = lib().trace_record_info(p, n, ctypes.byref(hd))
    if st != 0:
        raise TraceError("trace_record_info", st)
    raw = keep.numpy() if isinstance(keep, torch.Tensor) else keep
    seg = raw[hd.seg_offset:hd.seg_offset + 8 * (hd.n_seg + 1)].view(np.int64).copy()
    return hd, seg


def save_record(buf, path: str) -> None:
    """Writes a record to disk as is (its bytes are the on-disk format)."""
    raw = buf.numpy() if isinstance(buf, torch.Tensor) else np.asarray(buf, dtype=np.uint8)
    with open(path, "wb") as f:
        f.write(memoryview(raw))


def load_record(path: str, pin: bool = True) -> torch.Tensor:
    """Reads a record file into a uint8 host tensor (page-locked, huge-page
    backed unless pin=False) and validates it."""
    size = os.path.getsize(path)
    buf = hostmem.host_empty((size,), torch.uint8) if pin else torch.empty(size, dtype=torch.uint8)
    with open(path, "rb") as f:
        got = f.readinto(memoryview(buf.numpy()))
    if got != size:
        raise TraceError("load_record: short read", 1)
    record_info(buf)
    return buf


__all__: Sequence[str] = ["Handle", "TraceError", "lib", "library_path", "new_stats",
                          "stats_dict", "GUIDE_NONE", "GUIDE_FULL", "GUIDE_COMPACT",
                          "KERNELS", "SIGNATURES", "MAX_SEGMENTS", "RecordHeader",
                          "record_size", "record_info", "save_record", "load_record",
                          "guided_fake_quant", "GuidedFakeQuant", "OPTIONS", "GEMM_FORMS"]


class GuidedFakeQuant(torch.autograd.Function):
    """Rollout-guided FP4 fake quantisation as an autograd function: the
    forward is trace_train_fakequant, the backward the straight-through
    estimator (trace_ste_backward) with the forward's mask."""

    @staticmethod
    def forward(ctx, x, handle, seg_t, kind, guide, bs_r, gs_r, seg_r):
        y, mask, _, _ = handle.train_fakequant(x.contiguous(), seg_t, kind, guide, bs_r, gs_r,
                                               seg_r, mask=True)
        ctx.handle = handle
        ctx.save_for_backward(mask)
        return y

    @staticmethod
    def backward(ctx, grad_y):
        (mask,) = ctx.saved_tensors
        g = grad_y.contiguous().to(torch.bfloat16)
        return ctx.handle.ste_backward(g, mask), None, None, None, None, None, None, None


def guided_fake_quant(x, handle, seg_t=None, kind="none", guide=None, bs_r=None, gs_r=None,
                      seg_r=None):
    return GuidedFakeQuant.apply(x, handle, seg_t, kind, guide, bs_r, gs_r, seg_r)
