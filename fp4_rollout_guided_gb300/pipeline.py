"""Host-streamed guided-NVFP4 step: inputs and outputs in pinned host memory,
processed in pieces of whole training segments so that the host->device copy
of piece k+1, the kernels of piece k and the device->host copy of piece k-1
overlap on CUDA streams.  The host-to-device copies of x and r share one
stream (two concurrent streams in the same direction only contend for the
link), the device-to-host copies run on another, so both directions of the
link work at once.  Pieces default to about a twelfth of the rows: enough to
overlap, few enough that enqueueing a step costs the host a few
milliseconds rather than as long as the step itself.

Training segments are independent (each has its own global scale, and the
rollout segments refine them), so running the step piece by piece gives the
same bits as one call over the whole tensors.  Only device buffers of the
full size are used (pieces are row ranges of them).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import hostmem, trace


@dataclass
class Piece:
    r0: int            # first row
    r1: int            # one past the last row
    s0: int            # first rollout segment
    s1: int            # one past the last rollout segment
    seg_t: np.ndarray  # training offsets rebased to r0
    seg_r: np.ndarray  # rollout offsets rebased to r0


def plan_pieces(seg_t: Sequence[int], seg_r: Sequence[int], min_rows: int = 1) -> List[Piece]:
    """Pieces of whole training segments (consecutive segments merged until a
    piece holds at least min_rows rows); every rollout boundary inside a
    piece must be a rollout boundary of the whole table, and every training
    boundary must be a rollout boundary (the rollout table refines it)."""
    seg_t = np.asarray(seg_t, dtype=np.int64)
    seg_r = np.asarray(seg_r, dtype=np.int64)
    if not set(seg_t.tolist()) <= set(seg_r.tolist()):
        raise ValueError("the rollout segments must refine the training segments")
    pieces: List[Piece] = []
    a = 0
    i = 0
    n = len(seg_t) - 1
    while i < n:
        j = i + 1
        while j < n and seg_t[j] - seg_t[i] < min_rows:
            j += 1
        r0, r1 = int(seg_t[i]), int(seg_t[j])
        s0 = int(np.searchsorted(seg_r, r0, side="left"))
        s1 = int(np.searchsorted(seg_r, r1, side="left"))
        pieces.append(Piece(r0, r1, s0, s1, (seg_t[i:j + 1] - r0).astype(np.int64),
                            (seg_r[s0:s1 + 1] - r0).astype(np.int64)))
        i = j
    return pieces


class HostStreamedStep:
    """The step of bench.py (rollout quantisation with the compact record,
    guide pack, guide unpack, guided fake quantisation with the STE mask)
    over host-resident x and r, streamed in pieces.

    Device buffers (all full size, on the handle's device) are allocated
    here; run() reads x_h, r_h (page-locked, bf16 [rows, cols]) and writes
    y_h, mask_h, guide_h, bs_h, gs_h (page-locked) and returns once everything
    is enqueued; synchronise the device (or the d2h stream) before reading.
    hostmem.host_empty gives host buffers whose copies keep the link's rate
    however fragmented the host's memory is."""

    def __init__(self, h: trace.Handle, rows: int, cols: int, seg_t, seg_r,
                 guide: str = "compact", min_piece_rows: Optional[int] = None):
        dev = h.device
        self.h = h
        self.guide = guide
        self.rows, self.cols = rows, cols
        if min_piece_rows is None:
            min_piece_rows = max(1, -(-rows // 12))
        self.pieces = plan_pieces(seg_t, seg_r, min_piece_rows)
        n_seg_r = len(seg_r) - 1
        self.x = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
        self.r = torch.empty_like(self.x)
        self.codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        self.bs = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
        self.gs = torch.empty((n_seg_r,), dtype=torch.float32, device=dev)
        self.guide_words = torch.empty((rows, cols // 16), dtype=torch.int32, device=dev)
        self.packed = torch.empty_like(self.guide_words)
        self.unpacked = torch.empty_like(self.codes)
        self.y = torch.empty_like(self.x)
        self.mask = torch.empty((rows, cols // 32), dtype=torch.int32, device=dev)
        self.s_in = torch.cuda.Stream(dev)
        self.s_run = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)
        self.done = torch.cuda.Event()

    def outputs(self):
        """Device outputs copied back by run(): y, mask, guide words, bs, gs."""
        return self.y, self.mask, self.guide_words, self.bs, self.gs

    def run(self, x_h: torch.Tensor, r_h: torch.Tensor, outs_h: Sequence[torch.Tensor]):
        y_h, mask_h, guide_h, bs_h, gs_h = outs_h
        h, kind = self.h, self.guide
        # a new run's copies into x / r wait for the previous run's kernels
        self.s_in.wait_event(self.done)
        for p in self.pieces:
            a, b = p.r0, p.r1
            with torch.cuda.stream(self.s_in):
                self.r[a:b].copy_(r_h[a:b], non_blocking=True)
                self.x[a:b].copy_(x_h[a:b], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(self.s_in)
            with torch.cuda.stream(self.s_run):
                self.s_run.wait_event(ev_in)
                xd, rd = self.x[a:b], self.r[a:b]
                out_r = (self.codes[a:b], self.bs[a:b], self.gs[p.s0:p.s1],
                         self.guide_words[a:b])
                h.rollout_quant(rd, p.seg_r, out=out_r)
                h.guide_pack(self.codes[a:b], out=self.packed[a:b])
                h.guide_unpack(rd, self.guide_words[a:b], self.bs[a:b], self.gs[p.s0:p.s1],
                               p.seg_r, out=self.unpacked[a:b])
                g = self.guide_words[a:b] if kind == "compact" else self.codes[a:b]
                h.train_fakequant(xd, p.seg_t, kind, g, self.bs[a:b], self.gs[p.s0:p.s1], p.seg_r,
                                  out=(self.y[a:b], self.mask[a:b], None))
                ev_run = torch.cuda.Event()
                ev_run.record(self.s_run)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_run)
                y_h[a:b].copy_(self.y[a:b], non_blocking=True)
                mask_h[a:b].copy_(self.mask[a:b], non_blocking=True)
                guide_h[a:b].copy_(self.guide_words[a:b], non_blocking=True)
                bs_h[a:b].copy_(self.bs[a:b], non_blocking=True)
                gs_h[p.s0:p.s1].copy_(self.gs[p.s0:p.s1], non_blocking=True)
        self.done.record(self.s_run)
        return self.s_out

    def host_outputs(self, pin: bool = True):
        """Host tensors matching outputs(): page-locked and backed by huge
        pages (hostmem.host_empty), or pageable with pin=False."""
        if not pin:
            return [torch.empty(t.shape, dtype=t.dtype) for t in self.outputs()]
        return [hostmem.host_empty(t.shape, t.dtype) for t in self.outputs()]


__all__ = ["Piece", "plan_pieces", "HostStreamedStep"]
