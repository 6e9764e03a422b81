"""Segment-parallel drivers around the oracle, for the large parity tests.

The oracle's functions are single-threaded; these helpers call them
unchanged on pieces of rows, on every host core.  A piece never crosses a
rollout segment (and the rollout segments refine the training segments in
every test that uses them), and each piece is given its segments' maxima,
which were taken first over the whole segments: segments are independent
once their maxima are known, so the concatenated pieces equal one
whole-tensor call (the oracle pins that segment independence).
"""
import numpy as np

import oracle


def pieces_of(seg, rows, target=256):
    """(first row, end row, segment) pieces inside the segments of ``seg``."""
    piece = max(64, rows // target)
    out = []
    for k in range(len(seg) - 1):
        a, b = int(seg[k]), int(seg[k + 1])
        for p in range(a, b, piece):
            out.append((p, min(p + piece, b), k))
    return out


def maxima(u, seg):
    """Per-segment max |x| of bf16 bit patterns (uint16), segment-parallel."""
    ps = pieces_of(seg, u.shape[0])
    part = oracle.parallel_map(lambda q: (q[2], float(oracle.segment_amax(u[q[0]:q[1]])[0])), ps)
    m = np.zeros(len(seg) - 1, dtype=np.float32)
    for k, v in part:
        m[k] = max(m[k], v)
    return m


def training_segment(seg_t, row):
    return int(np.searchsorted(seg_t, row, side="right") - 1)


def rollout_quant(ru, seg_r, amax=None):
    """Whole-tensor rollout record (codes, bs, gs, guide), piecewise; amax
    (float32[n_seg]) replaces the segments' own maxima (delayed scaling)."""
    if amax is None:
        amax = maxima(ru, seg_r)
    ps = pieces_of(seg_r, ru.shape[0])
    res = oracle.parallel_map(lambda q: oracle.rollout_quant(ru[q[0]:q[1]], None,
                                                             amax=amax[q[2]:q[2] + 1]), ps)
    codes = np.concatenate([r[0] for r in res])
    bs = np.concatenate([r[1] for r in res])
    guide = np.concatenate([r[3] for r in res])
    gs = np.array([oracle.global_scale(a) for a in amax], dtype=np.float32)
    return codes, bs, gs, guide


def train_fakequant(xu, seg_t, kind, guide, bs_r, gs_r, seg_r, amax_t=None):
    """Whole-tensor fake quantiser outputs (y, mask, codes_t, stats),
    piecewise."""
    if amax_t is None:
        amax_t = maxima(xu, seg_t)
    ps = pieces_of(seg_r, xu.shape[0])

    def one(q):
        a, b, k = q
        s = training_segment(seg_t, a)
        g = None if guide is None else guide[a:b]
        bs = None if bs_r is None else bs_r[a:b]
        gr = None if gs_r is None else gs_r[k:k + 1]
        return oracle.train_fakequant(xu[a:b], None, kind, g, bs, gr, None, amax_t=[amax_t[s]])

    res = oracle.parallel_map(one, ps)
    return (np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res]),
            np.concatenate([r[2] for r in res]), sum(r[3] for r in res))


def guide_unpack(xu, guide, bs_r, gs_r, seg_r):
    ps = pieces_of(seg_r, xu.shape[0])
    res = oracle.parallel_map(lambda q: oracle.guide_unpack(xu[q[0]:q[1]], guide[q[0]:q[1]],
                                                            bs_r[q[0]:q[1]],
                                                            gs_r[q[2]:q[2] + 1], None), ps)
    return np.concatenate(res)
