"""Every element of the workloads at their stated sizes against the oracle.

The GPU path runs each workload whole, in the launch configuration the
benchmark times (fused rollout kernel; guided fake quantiser with the STE
mask and nothing else), and again with the training codes and the mismatch
counters, for the compact and the full record.  The oracle then recomputes
the same outputs on the host, on every core: the segment maxima first, then
pieces of rows inside each rollout segment, each quantised with its
segment's maxima given (segments are independent once their maxima are
known).  Every byte of every output is compared, and the counters are
compared with the oracle's exact counts.

Workloads 1-4 are checked on every element.  The long-rollout KV stream
(6.44 G elements) is checked on every one of its 96 training segments, on
one whole 4096-token rollout chunk of each (chunk s mod 32 of segment s:
96 of the 3072 rollout segments, 201 M elements), with the training maxima
taken over the whole segments.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pieces as op
from oracle_pieces import maxima, pieces_of
from fp4_rollout_guided_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from fp4_rollout_guided_gb300 import build, trace
    build.build()
    oracle.build()
    hd = trace.Handle(0)
    yield hd
    hd.close()


def host(t):
    if t.dtype == torch.bfloat16:
        return synth.to_u16(t)
    a = t.detach().cpu().numpy()
    return a.view(np.uint32) if a.dtype == np.int32 else a


def gpu_outputs(h, x, r, w):
    from fp4_rollout_guided_gb300 import trace
    codes, bs, gs, guide = h.rollout_quant(r, w.seg_r)
    out = {"codes": codes, "bs": bs, "gs": gs, "guide": guide,
           "packed": h.guide_pack(codes),
           "unpack_r": h.guide_unpack(r, guide, bs, gs, w.seg_r),
           "unpack_x": h.guide_unpack(x, guide, bs, gs, w.seg_r)}
    for kind, g in (("compact", guide), ("full", codes)):
        y, m, _, _ = h.train_fakequant(x, w.seg_t, kind, g, bs, gs, w.seg_r)
        out[kind + "/y"], out[kind + "/mask"] = y, m
        st = trace.new_stats(DEV)
        y, m, c, _ = h.train_fakequant(x, w.seg_t, kind, g, bs, gs, w.seg_r, codes=True, stats=st)
        out[kind + "/y_c"], out[kind + "/mask_c"], out[kind + "/codes_t"] = y, m, c
        out[kind + "/stats"] = st
    torch.cuda.synchronize()
    return out


def compare_pieces(o, xu, ru, seg_t, amax_t, amax_r, pieces, gs_index):
    """Oracle on every piece, compared with the GPU outputs (host arrays in
    o); returns (list of mismatch messages, compact stats, full stats)."""

    def one(q):
        a, b, k = q
        s = int(np.searchsorted(seg_t, a, side="right") - 1)
        bad = []

        def same(name, got, want):
            if not np.array_equal(got, want):
                i = tuple(np.argwhere(got != want)[0])
                bad.append(f"{name} rows {a}:{b}: {int((got != want).sum())} differ, first {i}")

        codes, bs, gs, guide = oracle.rollout_quant(ru[a:b], None, amax=amax_r[k:k + 1])
        same("codes", o["codes"][a:b], codes)
        same("bs", o["bs"][a:b], bs)
        same("gs", o["gs"][gs_index(k):gs_index(k) + 1].view(np.uint32), gs.view(np.uint32))
        same("guide", o["guide"][a:b], guide)
        same("pack", o["packed"][a:b], guide)
        same("unpack(r)", o["unpack_r"][a:b], codes)
        same("unpack(x)", o["unpack_x"][a:b], oracle.guide_unpack(xu[a:b], guide, bs, gs, None))
        st = {}
        for kind, okind, g in (("compact", oracle.GUIDE_COMPACT, guide),
                               ("full", oracle.GUIDE_FULL, codes)):
            y, m, c, stats = oracle.train_fakequant(xu[a:b], None, okind, g, bs, gs, None,
                                                    amax_t=[amax_t[s]])
            same(kind + " y", o[kind + "/y"][a:b], y)
            same(kind + " mask", o[kind + "/mask"][a:b], m)
            same(kind + " y (codes, counters)", o[kind + "/y_c"][a:b], y)
            same(kind + " mask (codes, counters)", o[kind + "/mask_c"][a:b], m)
            same(kind + " codes_t", o[kind + "/codes_t"][a:b], c)
            st[kind] = stats
        return bad, st["compact"], st["full"]

    res = oracle.parallel_map(one, pieces)
    bad = [m for r in res for m in r[0]]
    return bad, sum(r[1] for r in res), sum(r[2] for r in res)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_every_element_at_full_size(h, cfg):
    w = synth.workload(cfg)
    x, r = synth.make_inputs(w, DEV)
    g = gpu_outputs(h, x, r, w)
    o = {k: host(v) for k, v in g.items() if not k.endswith("/stats")}
    stats_gpu = {k: g[k + "/stats"].cpu().numpy().astype(np.uint64) for k in ("compact", "full")}
    del g
    xu, ru = host(x), host(r)
    del x, r
    torch.cuda.empty_cache()
    amax_t = maxima(xu, w.seg_t)
    amax_r = maxima(ru, w.seg_r)
    bad, st_c, st_f = compare_pieces(o, xu, ru, w.seg_t, amax_t, amax_r,
                                     pieces_of(w.seg_r, w.rows), lambda k: k)
    assert not bad, f"{w.name}: " + "; ".join(bad[:8])
    assert st_c[0] == w.elems and st_f[0] == w.elems
    assert np.array_equal(stats_gpu["compact"], st_c), (stats_gpu["compact"], st_c)
    assert np.array_equal(stats_gpu["full"], st_f), (stats_gpu["full"], st_f)


def test_long_rollout_stream_every_segment(h):
    w = synth.workload(5)
    x, r = synth.make_inputs(w, DEV)
    g = gpu_outputs(h, x, r, w)
    # the training maxima over whole segments, on the host
    xu_all = host(x)
    amax_t = maxima(xu_all, w.seg_t)
    # one whole rollout chunk per training segment, rotating through the chunks
    rows_sel, picks = [], []
    for s in range(w.n_seg_t):
        inner, first = synth.rollout_segments_within(w, s)
        k = s % (len(inner) - 1)
        a, b = int(w.seg_t[s]) + int(inner[k]), int(w.seg_t[s]) + int(inner[k + 1])
        rows_sel.append((a, b))
        picks.append(first + k)
    idx = np.concatenate([np.arange(a, b) for a, b in rows_sel])
    sel = torch.from_numpy(idx).to(DEV)
    o = {}
    for k, v in g.items():
        if k.endswith("/stats") or k == "gs":
            continue
        o[k] = host(v.index_select(0, sel))
    o["gs"] = host(g["gs"])
    stats = {k: g[k + "/stats"].cpu().numpy().astype(np.uint64) for k in ("compact", "full")}
    xu = xu_all[idx]
    del xu_all
    ru = host(r.index_select(0, sel))
    del g, x, r, sel
    torch.cuda.empty_cache()
    # the selected rows laid end to end: one rollout segment per training segment
    seg_sel = np.concatenate([[0], np.cumsum([b - a for a, b in rows_sel])]).astype(np.int64)
    amax_r = maxima(ru, seg_sel)
    bad, st_c, st_f = compare_pieces(o, xu, ru, seg_sel, amax_t, amax_r,
                                     pieces_of(seg_sel, len(idx)), lambda k: picks[k])
    assert not bad, "; ".join(bad[:8])
    assert st_c[0] == len(idx) * w.cols
    # whole-tensor counters: every element counted once, guidance never
    # increases the mismatches
    for kind in ("compact", "full"):
        assert stats[kind][0] == w.elems
        assert stats[kind][2] <= stats[kind][1]


def test_delayed_scaling_every_element(h):
    """Both delayed forms on the KV-row workload (537 M elements), every
    element: the rollout side and the training side scaled by given maxima
    (90 % of the segments' own in alternate segments, so blocks saturate at
    scale, and 130 % in the others), and the maxima each call returns."""
    w = synth.workload(3)
    x, r = synth.make_inputs(w, DEV)
    xu, ru = host(x), host(r)
    own_r, own_t = maxima(ru, w.seg_r), maxima(xu, w.seg_t)
    f_r = np.where(np.arange(len(own_r)) % 2 == 0, 0.9, 1.3).astype(np.float32)
    f_t = np.where(np.arange(len(own_t)) % 2 == 0, 1.3, 0.9).astype(np.float32)
    prev_r, prev_t = (own_r * f_r).astype(np.float32), (own_t * f_t).astype(np.float32)
    codes, bs, gs, guide, am_r = h.rollout_quant_delayed(r, w.seg_r,
                                                         torch.from_numpy(prev_r).to(DEV))
    y, m, am_t = h.train_fakequant_delayed(x, w.seg_t, torch.from_numpy(prev_t).to(DEV),
                                           "compact", guide, bs, gs, w.seg_r)
    torch.cuda.synchronize()
    got = {"codes": host(codes), "bs": host(bs), "gs": host(gs), "guide": host(guide),
           "y": host(y), "mask": host(m)}
    am_r, am_t = host(am_r), host(am_t)
    del x, r, codes, bs, gs, guide, y, m
    torch.cuda.empty_cache()
    o_codes, o_bs, o_gs, o_guide = op.rollout_quant(ru, w.seg_r, amax=prev_r)
    for name, want in (("codes", o_codes), ("bs", o_bs), ("guide", o_guide)):
        assert np.array_equal(got[name], want), name
    assert np.array_equal(got["gs"].view(np.uint32), o_gs.view(np.uint32))
    assert np.array_equal(am_r.view(np.uint32), own_r.view(np.uint32))
    oy, om, _, _ = op.train_fakequant(xu, w.seg_t, oracle.GUIDE_COMPACT, o_guide, o_bs, o_gs,
                                      w.seg_r, amax_t=prev_t)
    assert np.array_equal(got["y"], oy)
    assert np.array_equal(got["mask"], om)
    assert np.array_equal(am_t.view(np.uint32), own_t.view(np.uint32))
