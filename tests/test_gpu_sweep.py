"""Exhaustive sweeps of the scalar steps, GPU against the oracle.

The kernels decide E2M1 codes with the hardware conversions and with exact
rounding-constant tricks, and E4M3 block scales with a reciprocal-multiply
shortcut that falls back to the division near a rounding boundary; these
sweeps drive every input those steps can see.

Sweep of magnitudes: a segment whose maximum A fixes its global scale
(gs = 1, a power of two, an awkward value, and one so small that the scales
of the lower codes flush) holds, for every E4M3 code k the segment can
produce, blocks whose maximum forces code k, filled with every finite bf16
magnitude up to that maximum and with each one's negative.  So every bf16
value is quantised, bracketed, decoded and fake-quantised at every block
scale below it.  Rollout records: the tensor's own (scale ratio 1), a copy
moved one bf16 step per element (codes change at every boundary), and the
own record read with its global scale times 0.9 and times 1.2 (the guided
choice on both sides of its fast form's window).

Sweep of block scales: segment and block maxima chosen so that
bamax / (gs * 6) lies within four binary32 ulps of every E4M3 rounding
midpoint (the reciprocal shortcut's bracket straddles the boundary, and the
division decides) and around them.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pieces as op
from fp4_rollout_guided_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
COLS = 256


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


def bits_to_bf16(b):
    return torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16)


def rows_of(blocks):
    """Blocks of 16 bf16 patterns -> [rows, COLS], zero blocks pad the tail."""
    per_row = COLS // 16
    n = -(-len(blocks) // per_row) * per_row
    out = np.zeros((n, 16), dtype=np.uint16)
    out[:len(blocks)] = blocks
    return out.reshape(-1, COLS)


def magnitude_sweep(a_bits):
    """One segment of the magnitude sweep for segment maximum A (bf16 bits)."""
    A = np.array([a_bits << 16], np.uint32).view(np.float32)[0]
    gs = oracle.global_scale(A)
    den = np.float32(np.float32(gs) * np.float32(6.0))
    mags = np.arange(0, a_bits + 1, dtype=np.uint32)            # every bf16 <= A
    q = ((mags << 16).view(np.float32) / den).astype(np.float32)
    code = oracle.e4m3_encode(q)
    blocks = [np.array([a_bits] + [0] * 15, np.uint16)]         # the segment maximum
    for k in range(1, 127):
        sel = np.nonzero(code == k)[0]
        if len(sel) == 0:
            continue
        m_bits = int(mags[sel[-1]])                               # largest maximum with code k
        vals = np.arange(0, m_bits + 1, dtype=np.uint16)
        vals = np.concatenate([vals, vals | 0x8000])              # and every negative
        pad = -len(vals) % 15
        vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, 15)
        lead = np.where(np.arange(len(vals)) % 2 == 0, m_bits, m_bits | 0x8000).astype(np.uint16)
        blocks.extend(np.concatenate([lead[:, None], vals], axis=1))
    return rows_of(np.stack(blocks))


def one_step_away(xu):
    """Every nonzero element moved one bf16 step, up and down alternately."""
    b = xu.astype(np.int32)
    mag = b & 0x7FFF
    step = np.where(np.arange(b.size).reshape(b.shape) % 2 == 0, 1, -1)
    mag2 = np.clip(mag + step, 1, 0x7F7F)
    out = np.where(mag == 0, b, (b & 0x8000) | mag2)
    return out.astype(np.uint16)


def check_all_paths(h, xu, seg, label):
    from fp4_rollout_guided_gb300 import trace

    def same(name, got, want):
        got, want = np.asarray(got), np.asarray(want)
        if not np.array_equal(got, want):
            i = tuple(np.argwhere(got != want)[0])
            raise AssertionError(f"{label} {name}: {int((got != want).sum())} differ, first at "
                                 f"{i}: gpu {got[i]!r} oracle {want[i]!r}")

    x = bits_to_bf16(xu).to(DEV)
    # rollout quantiser, fused and two-kernel forms
    o_codes, o_bs, o_gs, o_guide = op.rollout_quant(xu, seg)
    for fused in (1, 0):
        h.set_option("fused_amax", fused)
        try:
            codes, bs, gs, guide = h.rollout_quant(x, seg)
            torch.cuda.synchronize()
        finally:
            h.set_option("fused_amax", 1)
        same(f"codes (fused={fused})", codes.cpu().numpy(), o_codes)
        same(f"bs (fused={fused})", bs.cpu().numpy(), o_bs)
        same(f"gs (fused={fused})", gs.cpu().numpy().view(np.uint32), o_gs.view(np.uint32))
        same(f"guide (fused={fused})", guide.cpu().numpy().view(np.uint32), o_guide)
    # records: own, moved one step, own read at 0.9 and 1.2 of its scale
    yu = one_step_away(xu)
    y_codes, y_bs, y_gs, y_guide = op.rollout_quant(yu, seg)
    records = {"own": (o_codes, o_bs, o_gs, o_guide), "moved": (y_codes, y_bs, y_gs, y_guide),
               "own x0.9": (o_codes, o_bs, (o_gs * np.float32(0.9)).astype(np.float32), o_guide),
               "own x1.2": (o_codes, o_bs, (o_gs * np.float32(1.2)).astype(np.float32), o_guide)}
    # unpack of the own record against x itself and against the moved copy
    xg_moved = bits_to_bf16(yu).to(DEV)
    g_guide = torch.from_numpy(o_guide.view(np.int32)).to(DEV)
    g_bs, g_gs = torch.from_numpy(o_bs).to(DEV), torch.from_numpy(o_gs).to(DEV)
    for name, ref, refu in (("x", x, xu), ("moved", xg_moved, yu)):
        got = h.guide_unpack(ref, g_guide, g_bs, g_gs, seg)
        torch.cuda.synchronize()
        same(f"unpack({name})", got.cpu().numpy(), op.guide_unpack(refu, o_guide, o_bs, o_gs, seg))
    amax_t = op.maxima(xu, seg)
    want = {"none": op.train_fakequant(xu, seg, oracle.GUIDE_NONE, None, None, None, seg, amax_t)}
    y, m, c, _ = h.train_fakequant(x, seg, "none", codes=True)
    torch.cuda.synchronize()
    same("none y", synth.to_u16(y), want["none"][0])
    same("none mask", m.cpu().numpy().view(np.uint32), want["none"][1])
    same("none codes_t", c.cpu().numpy(), want["none"][2])
    for rname, (rc, rbs, rgs, rgd) in records.items():
        for kind, okind, gd in (("compact", oracle.GUIDE_COMPACT, rgd),
                                ("full", oracle.GUIDE_FULL, rc)):
            oy, om, oc, ost = op.train_fakequant(xu, seg, okind, gd, rbs, rgs, seg, amax_t)
            g_gd = torch.from_numpy(gd.view(np.int32) if kind == "compact" else gd).to(DEV)
            gb, gg = torch.from_numpy(rbs).to(DEV), torch.from_numpy(rgs).to(DEV)
            st = trace.new_stats(DEV)
            variants = {"counters": h.train_fakequant(x, seg, kind, g_gd, gb, gg, seg, codes=True,
                                                      stats=st),
                        "codes": h.train_fakequant(x, seg, kind, g_gd, gb, gg, seg, codes=True),
                        "mask": h.train_fakequant(x, seg, kind, g_gd, gb, gg, seg)}
            torch.cuda.synchronize()
            for vname, (y, m, c, _) in variants.items():
                lbl = f"{kind} record {rname} ({vname})"
                same(lbl + " y", synth.to_u16(y), oy)
                same(lbl + " mask", m.cpu().numpy().view(np.uint32), om)
                if c is not None:
                    same(lbl + " codes_t", c.cpu().numpy(), oc)
            same(f"{kind} record {rname} counters", st.cpu().numpy().astype(np.uint64), ost)


# segment maxima: gs = 1, gs = 2^-10, an awkward gs, and one whose lower
# codes' scales fall below 2^-128 (their reciprocal overflows: flushed)
@pytest.mark.parametrize("a_bits", [0x4528, 0x4028, 0x4479, 0x0880],
                         ids=["gs=1", "gs=2^-10", "gs=awkward", "gs=tiny"])
def test_every_bf16_magnitude_at_every_block_scale(h, a_bits):
    xu = magnitude_sweep(a_bits)
    seg = np.array([0, xu.shape[0]], np.int64)
    A = np.array([a_bits << 16], np.uint32).view(np.float32)[0]
    assert oracle.segment_amax(xu)[0] == A
    check_all_paths(h, xu, seg, f"A={A!r}")


def midpoint_pairs(per_midpoint=3):
    """(A, M) bf16 bit pairs with M / (fl(A / 2688) * 6) within four ulps of
    an E4M3 rounding midpoint, up to per_midpoint of them per midpoint."""
    vals = oracle.e4m3_decode(np.arange(127, dtype=np.uint8)).astype(np.float64)
    mids = np.concatenate([[2.0 ** -10], ((vals[:-1] + vals[1:]) / 2)[1:]])
    found = {}
    for ab in range(0x4500, 0x4580):
        A = np.array([ab << 16], np.uint32).view(np.float32)[0]
        den = np.float32(np.float32(oracle.global_scale(A)) * np.float32(6.0))
        mb = np.arange(1, ab + 1, dtype=np.uint32)
        q = ((mb << 16).view(np.float32) / den).astype(np.float32)
        idx = np.clip(np.searchsorted(mids, q.astype(np.float64)), 1, len(mids) - 1)
        for cand in (idx - 1, idx):
            mu = mids[cand].astype(np.float32)
            ulps = np.abs(q.view(np.int32).astype(np.int64) - mu.view(np.int32).astype(np.int64))
            for c, m in zip(cand[ulps <= 4], mb[ulps <= 4]):
                lst = found.setdefault(int(c), [])
                if len(lst) < per_midpoint:
                    lst.append((ab, int(m)))
    return found


def test_block_scales_at_every_e4m3_midpoint(h):
    pairs = midpoint_pairs()
    assert len(pairs) == 126, "every E4M3 rounding midpoint is reached"
    by_a = {}
    for lst in pairs.values():
        for ab, mb in lst:
            by_a.setdefault(ab, []).append(mb)
    segs, parts = [0], []
    for ab in sorted(by_a):
        blocks = [np.array([ab] + [0] * 15, np.uint16)]
        for mb in by_a[ab]:
            # the maximum, then the fifteen bf16 values just below it
            vals = np.clip(mb - np.arange(1, 16), 0, None).astype(np.uint16)
            blocks.append(np.concatenate([[mb], vals]).astype(np.uint16))
            blocks.append(np.concatenate([[mb | 0x8000], vals | 0x8000]).astype(np.uint16))
        part = rows_of(np.stack(blocks))
        parts.append(part)
        segs.append(segs[-1] + part.shape[0])
    xu = np.concatenate(parts)
    check_all_paths(h, xu, np.array(segs, np.int64), "midpoints")
