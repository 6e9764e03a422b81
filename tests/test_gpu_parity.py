"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
element by element and bit for bit, on the same seeded inputs.

Inputs come from the seeded generators or from hand-built edge cases; every
expected value comes from the oracle run on the host copy of those inputs.
Small workloads are checked on every element; the full-size workloads are
checked on sampled row windows (the oracle is given the segment maxima taken
from the whole segment on the host) plus whole-tensor invariants.
"""
import numpy as np
import pytest
import torch

import oracle
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


def u32(t):
    return t.cpu().numpy().view(np.uint32)


def u16(t):
    return synth.to_u16(t)


def bf16_from_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def assert_same(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} mismatches, first at {i}: "
                             f"gpu={got[i]!r} oracle={want[i]!r}")


def run_everything(h, x_cpu, r_cpu, seg_t, seg_r, stats=True):
    """All entry points on the GPU; returns numpy outputs."""
    from fp4_rollout_guided_gb300 import trace
    xg, rg = x_cpu.to(DEV), r_cpu.to(DEV)
    codes, bs, gs, guide = h.rollout_quant(rg, seg_r)
    packed = h.guide_pack(codes)
    unpack_r = h.guide_unpack(rg, guide, bs, gs, seg_r)
    unpack_x = h.guide_unpack(xg, guide, bs, gs, seg_r)
    out = {}
    for kind, g in (("none", None), ("full", codes), ("compact", guide)):
        st = trace.new_stats(DEV) if stats else None
        if kind == "none":
            y, m, c, _ = h.train_fakequant(xg, seg_t, "none", codes=True, stats=st)
        else:
            y, m, c, _ = h.train_fakequant(xg, seg_t, kind, g, bs, gs, seg_r, codes=True, stats=st)
        out[kind] = (u16(y), u32(m), c.cpu().numpy(),
                     None if st is None else st.cpu().numpy().astype(np.uint64))
        if kind != "none":
            # without counters the kernel takes the distance-free form of the
            # guided choice wherever the scale ratio allows it: once with the
            # training codes, once with the output and mask only
            y2, m2, c2, _ = h.train_fakequant(xg, seg_t, kind, g, bs, gs, seg_r, codes=True)
            y3, m3, _, _ = h.train_fakequant(xg, seg_t, kind, g, bs, gs, seg_r)
            out[kind + "/codes"] = (u16(y2), u32(m2), c2.cpu().numpy(), None)
            out[kind + "/mask"] = (u16(y3), u32(m3), None, None)
    torch.cuda.synchronize()
    return dict(codes=codes.cpu().numpy(), bs=bs.cpu().numpy(), gs=gs.cpu().numpy(),
                guide=u32(guide), packed=u32(packed), unpack_r=unpack_r.cpu().numpy(),
                unpack_x=unpack_x.cpu().numpy(), fq=out)


def oracle_everything(xu, ru, seg_t, seg_r):
    codes, bs, gs, guide = oracle.rollout_quant(ru, seg_r)
    fq = {"none": oracle.train_fakequant(xu, seg_t),
          "full": oracle.train_fakequant(xu, seg_t, oracle.GUIDE_FULL, codes, bs, gs, seg_r),
          "compact": oracle.train_fakequant(xu, seg_t, oracle.GUIDE_COMPACT, guide, bs, gs, seg_r)}
    return dict(codes=codes, bs=bs, gs=gs, guide=guide,
                unpack_x=oracle.guide_unpack(xu, guide, bs, gs, seg_r), fq=fq)


def check_all(h, x_cpu, r_cpu, seg_t, seg_r, label):
    # the contract covers finite inputs only
    assert torch.isfinite(x_cpu.float()).all() and torch.isfinite(r_cpu.float()).all(), label
    g = run_everything(h, x_cpu, r_cpu, seg_t, seg_r)
    o = oracle_everything(u16(x_cpu), u16(r_cpu), seg_t, seg_r)
    assert_same(f"{label} codes", g["codes"], o["codes"])
    assert_same(f"{label} bs", g["bs"], o["bs"])
    assert_same(f"{label} gs", g["gs"].view(np.uint32), o["gs"].view(np.uint32))
    assert_same(f"{label} guide", g["guide"], o["guide"])
    assert_same(f"{label} pack", g["packed"], o["guide"])
    assert_same(f"{label} unpack(r)", g["unpack_r"], o["codes"])
    assert_same(f"{label} unpack(x)", g["unpack_x"], o["unpack_x"])
    for kind in ("none", "full", "compact"):
        gy, gm, gc, gst = g["fq"][kind]
        oy, om, oc, ost = o["fq"][kind]
        assert_same(f"{label} {kind} y", gy, oy)
        assert_same(f"{label} {kind} mask", gm, om)
        assert_same(f"{label} {kind} codes_t", gc, oc)
        if kind == "none":
            assert gst[0] == ost[0]
        else:
            assert_same(f"{label} {kind} stats", gst, ost)
            for variant in ("/codes", "/mask"):
                vy, vm, vc, _ = g["fq"][kind + variant]
                assert_same(f"{label} {kind}{variant} y", vy, oy)
                assert_same(f"{label} {kind}{variant} mask", vm, om)
                if vc is not None:
                    assert_same(f"{label} {kind}{variant} codes_t", vc, oc)
    return g, o


# ---------------------------------------------------------------------------
# the five workloads, shrunk so the oracle checks every element
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_small_workloads_bit_exact(h, cfg):
    w = synth.workload(cfg, small=True)
    x, r = synth.make_inputs(w, "cpu")
    check_all(h, x, r, w.seg_t, w.seg_r, f"cfg{cfg}")


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def drift(x, seed, sigma):
    g = torch.Generator().manual_seed(seed + 1)
    return (x.float() * (1 + sigma * torch.randn(x.shape, generator=g))).to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (7, 160), (1000, 64), (517, 224),
                                        (2049, 32), (5, 4096),
                                        # smaller than one 128-row tensor-map box
                                        (1, 64), (3, 128), (100, 64)])
def test_ragged_shapes(h, rows, cols):
    x = rand_bf16((rows, cols), rows * 7 + cols)
    r = drift(x, rows, 2.0 ** -6)
    check_all(h, x, r, None, None, f"{rows}x{cols}")


def test_many_uneven_segments(h):
    rng = np.random.default_rng(5)
    counts = rng.integers(0, 9, 700)
    counts[::37] = 0                      # empty segments
    counts[5] = 300                       # one long segment spanning several steps
    rows = int(counts.sum())
    seg_t = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    # the rollout table cuts differently: finer, misaligned with training
    cuts = np.unique(np.concatenate([seg_t, rng.integers(0, rows, 500)]))
    seg_r = np.concatenate([cuts[cuts < rows], [rows]]).astype(np.int64)
    seg_r = np.unique(seg_r)
    x = rand_bf16((rows, 64), 11, scale=3.0)
    # per-row scale so segments differ widely
    x = (x.float() * torch.from_numpy(np.exp(rng.normal(0, 2, (rows, 1))).astype(np.float32))).to(torch.bfloat16)
    r = drift(x, 12, 2.0 ** -5)
    check_all(h, x, r, seg_t, seg_r, "segments")


def test_max_segments(h):
    from fp4_rollout_guided_gb300 import trace
    n = trace.MAX_SEGMENTS
    rows = n * 2 + 17
    counts = np.full(n, 2)
    counts[-1] += 17
    seg = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    x = rand_bf16((rows, 32), 21)
    r = drift(x, 22, 2.0 ** -7)
    check_all(h, x, r, seg, seg, "4000 segments")


def test_special_values(h):
    """Zeros, negative zeros, a block flushed by an overflowing reciprocal,
    values on E2M1 points and rounding ties (S = 1 exactly), values at the
    top of the bf16 range, and a zero segment."""
    rows, cols = 8, 64
    a = np.zeros((rows, cols), np.float32)
    a[0, 0] = 2688.0                                   # gs = 1 for segment 0
    a[0, 16:32] = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0,
                   -0.25, -5.0]                        # S = 1: exact ties and grid points
    a[0, 32:48] = -0.0
    a[0, 48] = 147.0                                   # clipped element
    a[1, :16] = 2.0 ** -118                            # tiny segment values
    a[1, 16] = 2.0 ** -118 / 1000.0                    # flushed block (1/S overflows)
    a[1, 17] = -(2.0 ** -118) / 3000.0
    a[2, :] = 1.0e38                                   # high in the bf16 range (the
    a[2, 1::2] = -5.0e37                               # drifted copy stays finite)
    a[3, :] = 1.0                                      # constant rows
    # rows 4..7: segment of zeros
    x = torch.from_numpy(a).to(torch.bfloat16)
    r = drift(x, 31, 2.0 ** -4)
    seg = np.array([0, 1, 2, 3, 4, 8], np.int64)
    check_all(h, x, r, seg, seg, "specials")
    # opposite-sign rollout record
    check_all(h, x, (-r.float()).to(torch.bfloat16), seg, seg, "specials negated")


def test_unrelated_rollout(h):
    """Independent rollout values: opposite signs and multi-entry mismatches
    exercise every branch of the guided choice and every histogram bucket."""
    x = rand_bf16((300, 256), 41)
    r = rand_bf16((300, 256), 42, scale=1.7)
    seg_t = np.array([0, 100, 300], np.int64)
    seg_r = np.array([0, 50, 51, 299, 300], np.int64)
    g, o = check_all(h, x, r, seg_t, seg_r, "unrelated")
    assert np.all(o["fq"]["full"][3][3:7] > 0)


def test_guided_choice_at_scale_ratio_window_edges(h):
    """The guided choice takes a distance-free form when the rollout/training
    scale ratio lies strictly inside (7/8, 7/6) (with a small margin) and the
    binary32 distance comparison elsewhere.  Rollout global scales swept
    finely across both edges of that window, and far outside it, must give
    the oracle's bytes either way; rows of one call mix both forms."""
    rows, cols = 512, 256
    x = rand_bf16((rows, cols), 51)
    r = drift(x, 52, 2.0 ** -7)
    xu, ru = u16(x), u16(r)
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(ru, None)
    factors = np.concatenate([np.linspace(0.86, 0.89, 13), np.linspace(1.15, 1.18, 13),
                              [0.5, 0.8, 1.0, 1.25, 2.0, 0.876, 1.165]]).astype(np.float32)
    n_seg = len(factors)
    seg = np.linspace(0, rows, n_seg + 1).astype(np.int64)
    seg[-1] = rows
    # the same rollout record, read with a different global scale per segment
    gs_r = (o_gs[0] * factors).astype(np.float32)
    xg = x.to(DEV)
    codes_g = torch.from_numpy(o_codes).to(DEV)
    bs_g = torch.from_numpy(o_bs).to(DEV)
    guide_g = torch.from_numpy(o_guide.view(np.int32)).to(DEV)
    gs_g = torch.from_numpy(gs_r).to(DEV)
    for kind, gd, od in (("compact", guide_g, o_guide), ("full", codes_g, o_codes)):
        okind = oracle.GUIDE_COMPACT if kind == "compact" else oracle.GUIDE_FULL
        oy, om, oc, _ = oracle.train_fakequant(xu, None, okind, od, o_bs, gs_r, seg,
                                               want_stats=False)
        for want_codes in (False, True):
            y, m, c, _ = h.train_fakequant(xg, None, kind, gd, bs_g, gs_g, seg, codes=want_codes)
            torch.cuda.synchronize()
            assert_same(f"ratio sweep {kind} y", u16(y), oy)
            assert_same(f"ratio sweep {kind} mask", u32(m), om)
            if want_codes:
                assert_same(f"ratio sweep {kind} codes_t", c.cpu().numpy(), oc)


def test_mixed_forms_in_one_warp(h):
    """Rows whose rollout copy is rescaled by 1.3 or 0.75 (outside the ratio
    window) interleaved with plain drifted rows, so warps hold both kinds of
    blocks and take the exact form, while neighbouring warps take the fast one."""
    rows, cols = 2048, 128
    x = rand_bf16((rows, cols), 61, scale=2.0)
    r = drift(x, 62, 2.0 ** -8).float()
    k = torch.arange(rows)
    r[k % 97 == 3] *= 1.3
    r[k % 89 == 5] *= 0.75
    r = r.to(torch.bfloat16)
    check_all(h, x, r, np.array([0, 700, 2048], np.int64), np.array([0, 1024, 2048], np.int64),
              "mixed")


def test_non_finite_inputs_leave_other_segments_exact(h):
    """NaN and infinities give unspecified results in their own segment but
    never fault, and the segments without them keep the oracle's bytes."""
    from fp4_rollout_guided_gb300 import trace
    rows, cols = 384, 128
    x = rand_bf16((rows, cols), 71, scale=2.0).float()
    x[200, 3] = float("nan")
    x[250, 0] = float("inf")
    x[300:310, :] = -float("inf")
    x[350, 64:96] = float("nan")
    x = x.to(torch.bfloat16)
    r = x.clone()
    r[:192] = drift(x[:192], 72, 2.0 ** -7)
    seg = np.array([0, 192, 384], np.int64)
    xg, rg = x.to(DEV), r.to(DEV)
    codes, bs, gs, guide = h.rollout_quant(rg, seg)
    outs = {}
    for kind, g in (("none", None), ("compact", guide), ("full", codes)):
        args = (xg, seg, kind) + (() if kind == "none" else (g, bs, gs, seg))
        outs[kind] = h.train_fakequant(*args, codes=True, stats=trace.new_stats(DEV))
        outs[kind + "/mask"] = h.train_fakequant(*args)
    unpacked = h.guide_unpack(xg, guide, bs, gs, seg)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    # the finite segment against the oracle
    xu, ru = u16(x[:192]), u16(r[:192])
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(ru, None)
    assert_same("codes", codes[:192].cpu().numpy(), o_codes)
    assert_same("guide", u32(guide[:192]), o_guide)
    assert_same("unpack", unpacked[:192].cpu().numpy(),
                oracle.guide_unpack(xu, o_guide, o_bs, o_gs, None))
    for kind, okind, og in (("none", oracle.GUIDE_NONE, None),
                            ("compact", oracle.GUIDE_COMPACT, o_guide),
                            ("full", oracle.GUIDE_FULL, o_codes)):
        oargs = (xu, None, okind) + (() if kind == "none" else (og, o_bs, o_gs, None))
        oy, om, oc, _ = oracle.train_fakequant(*oargs)
        assert_same(f"{kind} y", u16(outs[kind][0][:192]), oy)
        assert_same(f"{kind} mask", u32(outs[kind][1][:192]), om)
        assert_same(f"{kind} codes_t", outs[kind][2][:192].cpu().numpy(), oc)
        assert_same(f"{kind} y (mask only)", u16(outs[kind + "/mask"][0][:192]), oy)


# ---------------------------------------------------------------------------
# f1 (delayed form): rollout quantisation scaled by given maxima, one kernel
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols,seg", [(1, 32, None), (130, 96, [0, 0, 64, 130]),
                                           (4099, 128, [0, 2048, 2048, 4099]),
                                           (300, 2048, [0, 1, 299, 300]), (517, 224, None),
                                           (300, 64, [0, 50, 100, 150, 200, 300])])
def test_rollout_quant_delayed_matches_oracle(h, rows, cols, seg):
    """Codes, block scales, gs and compact words equal the oracle's with the
    given maxima (smaller than the segments' own: saturation; larger; equal;
    zero: the segment quantises to zero), and the maxima it returns are the
    segments' own."""
    seg = None if seg is None else np.array(seg, np.int64)
    x = rand_bf16((rows, cols), rows + 3 * cols, scale=2.0)
    xu = u16(x)
    own = oracle.segment_amax(xu, seg)
    factors = np.array([0.37, 1.0, 1.9, 0.0, 0.8], np.float32)
    prev = (own * factors[np.arange(len(own)) % len(factors)]).astype(np.float32)
    codes, bs, gs, gd, am = h.rollout_quant_delayed(x.to(DEV), seg,
                                                    torch.from_numpy(prev).to(DEV))
    torch.cuda.synchronize()
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(xu, seg, amax=prev)
    assert_same("codes", codes.cpu().numpy(), o_codes)
    assert_same("bs", bs.cpu().numpy(), o_bs)
    assert_same("gs", gs.cpu().numpy().view(np.uint32), o_gs.view(np.uint32))
    assert_same("guide", u32(gd), o_guide)
    assert_same("amax out", am.cpu().numpy().view(np.uint32), own.view(np.uint32))
    # the same without the maxima output, and without the compact words
    c2, b2, _, g2, a2 = h.rollout_quant_delayed(x.to(DEV), seg, torch.from_numpy(prev).to(DEV),
                                                guide=False, amax_out=False)
    torch.cuda.synchronize()
    assert g2 is None and a2 is None
    assert_same("codes (no maxima out)", c2.cpu().numpy(), o_codes)
    assert_same("bs (no maxima out)", b2.cpu().numpy(), o_bs)


@pytest.mark.parametrize("kind", ["compact", "full", "none"])
@pytest.mark.parametrize("rows,cols,seg_t,seg_r", [
    (1, 32, None, None), (300, 64, [0, 50, 100, 150, 200, 300], [0, 50, 100, 150, 200, 300]),
    (4099, 128, [0, 2048, 2048, 4099], [0, 1000, 2048, 2048, 3000, 4099]),
    (517, 224, None, [0, 100, 517])])
def test_train_fakequant_delayed_matches_oracle(h, kind, rows, cols, seg_t, seg_r):
    """y and the STE mask equal the oracle's with the training scales from
    the given maxima (smaller: saturated blocks; larger; equal; zero), with
    and without the mask, and the maxima returned are the segments' own."""
    seg_t = None if seg_t is None else np.array(seg_t, np.int64)
    seg_r = None if seg_r is None else np.array(seg_r, np.int64)
    x = rand_bf16((rows, cols), rows + 5 * cols, scale=2.0)
    r = drift(x, rows + 1, 2.0 ** -6)
    xu, ru = u16(x), u16(r)
    own = oracle.segment_amax(xu, seg_t)
    factors = np.array([0.37, 1.0, 1.9, 0.0, 0.8], np.float32)
    prev = (own * factors[np.arange(len(own)) % len(factors)]).astype(np.float32)
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(ru, seg_r)
    okind = {"none": oracle.GUIDE_NONE, "full": oracle.GUIDE_FULL,
             "compact": oracle.GUIDE_COMPACT}[kind]
    oargs = (xu, seg_t, okind) + (() if kind == "none" else (
        o_guide if kind == "compact" else o_codes, o_bs, o_gs, seg_r))
    oy, om, _, _ = oracle.train_fakequant(*oargs, amax_t=prev)
    g = {"compact": torch.from_numpy(o_guide.view(np.int32)), "full": torch.from_numpy(o_codes),
         "none": None}[kind]
    gargs = () if kind == "none" else (g.to(DEV), torch.from_numpy(o_bs).to(DEV),
                                       torch.from_numpy(o_gs).to(DEV), seg_r)
    y, m, am = h.train_fakequant_delayed(x.to(DEV), seg_t, torch.from_numpy(prev).to(DEV), kind,
                                         *gargs)
    y2, m2, am2 = h.train_fakequant_delayed(x.to(DEV), seg_t, torch.from_numpy(prev).to(DEV),
                                            kind, *gargs, mask=False, amax_out=False)
    torch.cuda.synchronize()
    assert m2 is None and am2 is None
    assert_same("y", u16(y), oy)
    assert_same("mask", u32(m), om)
    assert_same("y (no mask, no maxima)", u16(y2), oy)
    assert_same("amax out", am.cpu().numpy().view(np.uint32), own.view(np.uint32))


def test_rollout_quant_delayed_chain_and_empty(h):
    """Step t quantised with step t-1's maxima, as a loop would: each step's
    output maxima feed the next; a step of zero rows writes only gs and
    zeroes the maxima."""
    seg = np.array([0, 700, 700, 1500], np.int64)
    prev = torch.zeros(3, dtype=torch.float32, device=DEV)
    for t in range(3):
        x = rand_bf16((1500, 256), 40 + t, scale=1.0 + t)
        xu = u16(x)
        codes, bs, gs, gd, am = h.rollout_quant_delayed(x.to(DEV), seg, prev)
        torch.cuda.synchronize()
        o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(xu, seg, amax=prev.cpu().numpy())
        assert_same(f"codes step {t}", codes.cpu().numpy(), o_codes)
        assert_same(f"guide step {t}", u32(gd), o_guide)
        prev = am.clone()
    e = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    prev2 = torch.tensor([3.0, 0.5], dtype=torch.float32, device=DEV)
    _, _, gs, _, am = h.rollout_quant_delayed(e, np.array([0, 0, 0], np.int64), prev2)
    torch.cuda.synchronize()
    want = np.array([oracle.global_scale(np.float32(3.0)), oracle.global_scale(np.float32(0.5))],
                    np.float32)
    assert_same("gs (empty)", gs.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert torch.all(am == 0)


def test_empty_input(h):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    codes, bs, gs, guide = h.rollout_quant(x, np.array([0, 0, 0], np.int64))
    torch.cuda.synchronize()
    assert gs.shape == (2,) and torch.all(gs == 0)
    y, m, c, _ = h.train_fakequant(x, None, "compact", guide, bs, gs.new_zeros(1), None)
    assert y.numel() == 0


def test_repeated_calls_and_streams(h):
    """Scratch is reused call after call and across streams: results stay
    identical (the amax scratch re-zeroes itself)."""
    w = synth.workload(2, small=True)
    x, r = synth.make_inputs(w, "cpu")
    first = run_everything(h, x, r, w.seg_t, w.seg_r, stats=False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        second = run_everything(h, x, r, w.seg_t, w.seg_r, stats=False)
    s.synchronize()
    for k in ("codes", "bs", "gs", "guide", "unpack_x"):
        assert np.array_equal(first[k], second[k]), k
    for kind in ("none", "full", "compact"):
        for a, b in zip(first["fq"][kind][:3], second["fq"][kind][:3]):
            assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------

def sampled_check(h, cfg, windows_per_seg=2, window_rows=1536, seg_picks=3):
    from fp4_rollout_guided_gb300 import trace
    w = synth.workload(cfg)
    x, r = synth.make_inputs(w, DEV)
    codes, bs, gs, guide = h.rollout_quant(r, w.seg_r)
    packed = h.guide_pack(codes)
    unpacked = h.guide_unpack(r, guide, bs, gs, w.seg_r)
    st = trace.new_stats(DEV)
    y, m, _, _ = h.train_fakequant(x, w.seg_t, "compact", guide, bs, gs, w.seg_r, stats=st)
    torch.cuda.synchronize()
    # whole-tensor invariants that hold at any size
    assert torch.equal(packed, guide), "pack(codes) != rollout guide"
    assert torch.equal(unpacked, codes), "unpack(pack(codes), r) != codes"
    stats = st.cpu().numpy().astype(np.uint64)
    assert stats[0] == w.elems
    assert stats[2] <= stats[1]

    segs = np.unique(np.linspace(0, w.n_seg_t - 1, seg_picks).astype(int))
    for s in segs:
        t0, t1 = int(w.seg_t[s]), int(w.seg_t[s + 1])
        xs = u16(x[t0:t1])
        amax_t = np.abs(oracle.bf16_to_f32(xs)).max()
        # sample windows each inside one rollout segment
        inner, first = synth.rollout_segments_within(w, s)
        picks = np.unique(np.linspace(0, len(inner) - 2, windows_per_seg).astype(int))
        for k in picks:
            ra, rb = t0 + int(inner[k]), t0 + int(inner[k + 1])
            rs = u16(r[ra:rb])
            amax_r = np.abs(oracle.bf16_to_f32(rs)).max()
            a = ra + max(0, (rb - ra - window_rows) // 2)
            b = min(rb, a + window_rows)
            ru = u16(r[a:b])
            xu = u16(x[a:b])
            o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(ru, None, amax=[amax_r])
            lbl = f"cfg{cfg} seg{s} rows {a}:{b}"
            assert_same(lbl + " gs", gs[first + k:first + k + 1].cpu().numpy().view(np.uint32),
                        o_gs.view(np.uint32))
            assert_same(lbl + " codes", codes[a:b].cpu().numpy(), o_codes)
            assert_same(lbl + " bs", bs[a:b].cpu().numpy(), o_bs)
            assert_same(lbl + " guide", u32(guide[a:b]), o_guide)
            o_y, o_m, _, _ = oracle.train_fakequant(xu, None, oracle.GUIDE_COMPACT, o_guide, o_bs,
                                                    o_gs, None, amax_t=[amax_t],
                                                    want_codes=False, want_stats=False)
            assert_same(lbl + " y", u16(y[a:b]), o_y)
            assert_same(lbl + " mask", u32(m[a:b]), o_m)
    del x, r, codes, bs, gs, guide, packed, unpacked, y, m
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_full_size_sampled(h, cfg):
    sampled_check(h, cfg)


# ---------------------------------------------------------------------------
# straight-through backward and the autograd wrapper
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [1, 3, 5])
def test_ste_backward_bit_exact(h, cfg):
    w = synth.workload(cfg, small=True)
    x, r = synth.make_inputs(w, "cpu")
    xg = x.to(DEV)
    _, m, _, _ = h.train_fakequant(xg, w.seg_t, "none")
    g = rand_bf16(tuple(x.shape), 99 + cfg, scale=0.3)
    gi = h.ste_backward(g.to(DEV), m)
    # in place: the output may alias the incoming gradient
    gg = g.to(DEV)
    h.ste_backward(gg, m, out=gg)
    torch.cuda.synchronize()
    _, om, _, _ = oracle.train_fakequant(u16(x), w.seg_t)
    want = oracle.ste_backward(u16(g), om)
    assert_same(f"cfg{cfg} ste", u16(gi), want)
    assert_same(f"cfg{cfg} ste in place", u16(gg), want)


def test_autograd_guided_fake_quant(h):
    from fp4_rollout_guided_gb300 import trace
    w = synth.workload(2, small=True)
    x, r = synth.make_inputs(w, "cpu")
    xg, rg = x.to(DEV), r.to(DEV)
    codes, bs, gs, guide = h.rollout_quant(rg, w.seg_r)
    xr = xg.clone().requires_grad_(True)
    y = trace.guided_fake_quant(xr, h, w.seg_t, "compact", guide, bs, gs, w.seg_r)
    y.float().sum().backward()
    torch.cuda.synchronize()
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(u16(r), w.seg_r)
    o_y, o_m, _, _ = oracle.train_fakequant(u16(x), w.seg_t, oracle.GUIDE_COMPACT, o_guide, o_bs,
                                            o_gs, w.seg_r)
    assert_same("autograd y", u16(y.detach()), o_y)
    ones = np.full(u16(x).shape, 0x3F80, np.uint16)          # bf16 1.0
    assert_same("autograd grad", u16(xr.grad), oracle.ste_backward(ones, o_m))


# ---------------------------------------------------------------------------
# guide transport: device -> pinned host record -> disk -> host -> device
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["full", "compact"])
@pytest.mark.parametrize("cfg", [2, 5])
def test_record_round_trip(h, tmp_path, kind, cfg):
    from fp4_rollout_guided_gb300 import trace
    w = synth.workload(cfg, small=True)
    x, r = synth.make_inputs(w, "cpu")
    xg, rg = x.to(DEV), r.to(DEV)
    codes, bs, gs, guide = h.rollout_quant(rg, w.seg_r)
    g = codes if kind == "full" else guide
    rec = h.record_export(g, bs, gs, w.seg_r)
    assert rec.is_pinned() and rec.numel() == trace.record_size(kind, w.rows, w.cols, w.n_seg_r)
    path = str(tmp_path / f"guide_{kind}.trg")
    trace.save_record(rec, path)
    back = trace.load_record(path)
    g2, bs2, gs2, seg2 = h.record_import(back)
    torch.cuda.synchronize()
    assert seg2.tolist() == [int(v) for v in w.seg_r]
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(u16(r), w.seg_r)
    want = o_codes if kind == "full" else o_guide
    got = g2.cpu().numpy() if kind == "full" else u32(g2)
    assert_same(f"record {kind} guide", got, want)
    assert_same(f"record {kind} bs", bs2.cpu().numpy(), o_bs)
    assert_same(f"record {kind} gs", gs2.cpu().numpy().view(np.uint32), o_gs.view(np.uint32))
    # the imported record drives the training side to the oracle's result
    y, m, _, _ = h.train_fakequant(xg, w.seg_t, kind, g2, bs2, gs2, seg2)
    kk = oracle.GUIDE_FULL if kind == "full" else oracle.GUIDE_COMPACT
    o_y, o_m, _, _ = oracle.train_fakequant(u16(x), w.seg_t, kk, want, o_bs, o_gs, w.seg_r)
    assert_same(f"record {kind} y", u16(y), o_y)
    assert_same(f"record {kind} mask", u32(m), o_m)


def test_record_async_export_and_sizes(h):
    from fp4_rollout_guided_gb300 import trace
    w = synth.workload(3, small=True)
    _, r = synth.make_inputs(w, "cpu")
    codes, bs, gs, guide = h.rollout_quant(r.to(DEV), w.seg_r)
    full = h.record_export(codes, bs, gs, w.seg_r, wait=False)
    comp = h.record_export(guide, bs, gs, w.seg_r, wait=False)
    torch.cuda.current_stream().synchronize()
    hf, _ = trace.record_info(full)
    hc, _ = trace.record_info(comp)
    # guide sections: 4 bits per element (full) and 2 bits (compact), each
    # padded to 256 bytes
    pad = lambda v: (v + 255) // 256 * 256
    assert hf.bs_offset - hf.guide_offset == pad(w.rows * w.cols // 2)
    assert hc.bs_offset - hc.guide_offset == pad(w.rows * w.cols // 4)
    # a record that is too small is refused before any copy is queued
    small = torch.empty(full.numel() - 1, dtype=torch.uint8, pin_memory=True)
    with pytest.raises(trace.TraceError):
        h.record_export(codes, bs, gs, w.seg_r, out=small)


# ---------------------------------------------------------------------------
# fused amax + quantisation (one cooperative launch) against the oracle
# ---------------------------------------------------------------------------

def _rollout_vs_oracle(h, r_cpu, seg, label):
    codes, bs, gs, guide = h.rollout_quant(r_cpu.to(DEV), seg)
    torch.cuda.synchronize()
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(u16(r_cpu), seg)
    assert_same(f"{label} codes", codes.cpu().numpy(), o_codes)
    assert_same(f"{label} bs", bs.cpu().numpy(), o_bs)
    assert_same(f"{label} gs", gs.cpu().numpy().view(np.uint32), o_gs.view(np.uint32))
    assert_same(f"{label} guide", u32(guide), o_guide)


def _launched(h, fn):
    h.profile(True)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        t = h.collect()
        h.profile(False)
    return {k: n for k, (n, _) in t.items() if n}


@pytest.mark.parametrize("fused,wave_bytes", [(0, 16 << 20), (1, 4096), (1, 1 << 20),
                                              (1, 16 << 20), (1, 40 << 20)])
@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_rollout_fused_and_split_paths(h, cfg, fused, wave_bytes):
    w = synth.workload(cfg, small=True)
    _, r = synth.make_inputs(w, "cpu")
    h.set_option("fused_amax", fused)
    h.set_option("wave_bytes", wave_bytes)
    try:
        ran = _launched(h, lambda: _rollout_vs_oracle(h, r, w.seg_r, f"cfg{cfg}"))
    finally:
        h.set_option("fused_amax", 1)
        h.set_option("wave_bytes", 32 << 20)
    if fused:
        assert ran == {"rollout_fused": 1}, ran
    else:
        assert ran == {"amax": 1, "rollout_quant": 1}, ran
    assert h.device_status() == 0


def test_rollout_fused_uneven_and_empty_segments(h):
    rows, cols = 6000, 96
    x = rand_bf16((rows, cols), 71, scale=3.0)
    # empty segments first, in the middle and last; sizes from 1 row to 2400
    seg = [0, 0, 1, 1, 2401, 2401, 2413, 3000, 3000, 5999, 6000, 6000]
    h.set_option("wave_bytes", 4096)                # about one segment per wave
    try:
        ran = _launched(h, lambda: _rollout_vs_oracle(h, x, seg, "uneven fused"))
    finally:
        h.set_option("wave_bytes", 32 << 20)
    assert ran == {"rollout_fused": 1}
    _rollout_vs_oracle(h, x, seg, "uneven fused, default waves")
    assert h.device_status() == 0


@pytest.mark.parametrize("cols", [64, 96, 2048])
@pytest.mark.parametrize("offset_bytes", [16, 48, 112])
def test_rollout_input_16_byte_aligned_only(h, cols, offset_bytes):
    # x starts 16 bytes past a 128-byte boundary or more: the fused kernel's
    # tensor-map staging (cols % 64 == 0) and its bulk copies (cols = 96)
    # must not depend on more than the documented 16-byte alignment
    rows = 700
    x = rand_bf16((rows, cols), 73 + cols, scale=2.0)
    seg = [0, 5, 333, 640, rows]
    buf = torch.empty(rows * cols + 64, dtype=torch.bfloat16, device=DEV)
    off = offset_bytes // 2
    xv = buf[off:off + rows * cols].view(rows, cols)
    assert xv.data_ptr() % 16 == 0 and xv.data_ptr() % 128 != 0
    xv.copy_(x.to(DEV))
    ran = _launched(h, lambda: h.rollout_quant(xv, seg))
    assert ran == {"rollout_fused": 1}, ran
    codes, bs, gs, guide = h.rollout_quant(xv, seg)
    torch.cuda.synchronize()
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(u16(x), seg)
    label = f"offset {offset_bytes} cols {cols}"
    assert_same(f"{label} codes", codes.cpu().numpy(), o_codes)
    assert_same(f"{label} bs", bs.cpu().numpy(), o_bs)
    assert_same(f"{label} gs", gs.cpu().numpy().view(np.uint32), o_gs.view(np.uint32))
    assert_same(f"{label} guide", u32(guide), o_guide)
    assert h.device_status() == 0


@pytest.mark.parametrize("cfg", [1, 3, 5])
def test_segment_amax_and_scaled_fakequant(h, cfg):
    # the amax pass on its own, then the fake quantiser with those scales:
    # the same bytes as the one-call form and as the oracle
    from fp4_rollout_guided_gb300 import trace
    w = synth.workload(cfg, small=True)
    x, r = synth.make_inputs(w, "cpu")
    xg, rg = x.to(DEV), r.to(DEV)
    gs_t = h.segment_amax(xg, w.seg_t)
    torch.cuda.synchronize()
    _, _, o_gs, _ = oracle.rollout_quant(u16(x), w.seg_t)
    assert_same(f"cfg{cfg} gs_t", gs_t.cpu().numpy().view(np.uint32), o_gs.view(np.uint32))
    codes, bs, gs, guide = h.rollout_quant(rg, w.seg_r)
    for kind, g in (("none", None), ("full", codes), ("compact", guide)):
        st1, st2 = trace.new_stats(DEV), trace.new_stats(DEV)
        args = (xg, w.seg_t, kind) + (() if kind == "none" else (g, bs, gs, w.seg_r))
        one = h.train_fakequant(*args, codes=True, stats=st1)
        two = h.train_fakequant(*args, codes=True, stats=st2, gs_t=gs_t)
        torch.cuda.synchronize()
        for name, a, b in zip(("y", "mask", "codes_t", "stats"), one, two):
            assert torch.equal(a, b), f"cfg{cfg} {kind} {name}"


def test_segment_amax_empty_and_zero_segments(h):
    rows, cols = 300, 64
    x = rand_bf16((rows, cols), 81)
    x[100:200] = 0
    seg = [0, 0, 100, 200, 200, rows]
    gs = h.segment_amax(x.to(DEV), seg)
    torch.cuda.synchronize()
    _, _, o_gs, _ = oracle.rollout_quant(u16(x), seg)
    assert_same("gs", gs.cpu().numpy().view(np.uint32), o_gs.view(np.uint32))
    assert gs[0].item() == 0 and gs[2].item() == 0 and gs[3].item() == 0
    gs0 = h.segment_amax(torch.empty((0, cols), dtype=torch.bfloat16, device=DEV), [0, 0, 0])
    torch.cuda.synchronize()
    assert gs0.tolist() == [0.0, 0.0]


def test_two_handles_overlap_training_scales(h):
    # rollout side on one handle and stream, training scales on a second
    # handle and stream at the same time, then the scaled fake quantiser:
    # equal to the serial one-call path
    from fp4_rollout_guided_gb300 import trace
    w = synth.workload(3, small=True)
    x, r = synth.make_inputs(w, "cpu")
    xg, rg = x.to(DEV), r.to(DEV)
    h2 = trace.Handle(0)
    try:
        side = torch.cuda.Stream()
        start = torch.cuda.Event()
        start.record()
        with torch.cuda.stream(side):
            side.wait_event(start)
            gs_t = h2.segment_amax(xg, w.seg_t)
            done = torch.cuda.Event()
            done.record()
        codes, bs, gs, guide = h.rollout_quant(rg, w.seg_r)
        h.guide_pack(codes)
        h.guide_unpack(rg, guide, bs, gs, w.seg_r)
        torch.cuda.current_stream().wait_event(done)
        gs_t.record_stream(torch.cuda.current_stream())
        y, m, _, _ = h.train_fakequant(xg, w.seg_t, "compact", guide, bs, gs, w.seg_r, gs_t=gs_t)
        y1, m1, _, _ = h.train_fakequant(xg, w.seg_t, "compact", guide, bs, gs, w.seg_r)
        torch.cuda.synchronize()
        assert torch.equal(y, y1) and torch.equal(m, m1)
        assert h.device_status() == 0 and h2.device_status() == 0
    finally:
        h2.close()


def test_rollout_large_segment_takes_two_kernels(h):
    # one segment of 41 MiB of x is more than a fused wave may hold
    rows, cols = 10496, 2048
    x = rand_bf16((rows, cols), 72)
    seg = [0, 16, rows]
    ran = _launched(h, lambda: _rollout_vs_oracle(h, x, seg, "large segment"))
    assert ran == {"amax": 1, "rollout_quant": 1}, ran


def test_fused_wait_limit_reports_timeout(h):
    """The in-kernel waits are bounded: with the test hook on, every wait
    expects one arrival that never comes and gives up at its limit; the call
    finishes, the status says so, and the handle keeps working."""
    w = synth.workload(3, small=True)
    _, r = synth.make_inputs(w, "cpu")
    rg = r.to(DEV)
    assert h.device_status() == 0
    h.set_option("wait_limit_ns", 20_000_000)
    h.set_option("wait_extra", 1)
    try:
        h.rollout_quant(rg, w.seg_r)
        assert h.device_status() == 6
    finally:
        h.set_option("wait_extra", 0)
        h.set_option("wait_limit_ns", 1_000_000_000)
    assert h.device_status() == 0
    _rollout_vs_oracle(h, r, w.seg_r, "after timeout")
    assert h.device_status() == 0


@pytest.mark.parametrize("cfg", [3, 5])
def test_fused_equals_split_full_size(h, cfg):
    """At full size the fused kernel cycles its staging rings thousands of
    times; its outputs must equal the two-kernel path's bit for bit (that
    path is checked against the oracle on sampled windows above), for the
    default wave size and a large one, on repeated calls."""
    w = synth.workload(cfg)
    _, r = synth.make_inputs(w, DEV)
    h.set_option("fused_amax", 0)
    try:
        ref = [t.clone() for t in h.rollout_quant(r, w.seg_r)]
    finally:
        h.set_option("fused_amax", 1)
    try:
        for wave in (16 << 20, 32 << 20):
            h.set_option("wave_bytes", wave)
            out = h.rollout_quant(r, w.seg_r)
            for _ in range(2):
                ran = _launched(h, lambda: h.rollout_quant(r, w.seg_r, out=out))
                assert ran == {"rollout_fused": 1}, ran
                for name, a, b in zip(("codes", "bs", "gs", "guide"), out, ref):
                    assert torch.equal(a, b), f"cfg{cfg} wave {wave >> 20} MiB: {name} differs"
    finally:
        h.set_option("wave_bytes", 32 << 20)
    assert h.device_status() == 0


# ---------------------------------------------------------------------------
# f4: block scales in the tensor-core tile layout, NVFP4 GEMM over rollout
# codes (the library's tcgen05 kernel in its three tile forms, and cuBLASLt);
# a wrong tile layout or descriptor would put wrong scales on whole
# 16-element blocks or wrong codes in whole k-steps and miss the oracle by O(1)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(1, 32), (130, 96), (256, 64), (300, 2048), (4097, 128)])
def test_mma_scales_bit_exact(h, rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    bs = torch.randint(1, 255, (rows, cols // 16), generator=g, dtype=torch.int32).to(torch.uint8)
    got = h.block_scales_mma(bs.to(DEV), rows, cols)
    torch.cuda.synchronize()
    assert_same("mma scales", got.cpu().numpy(), oracle.mma_scales(bs.numpy(), rows, cols))


def _student_t(shape, seed):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(shape, generator=g)
    chi = (torch.randn((4,) + tuple(shape), generator=g) ** 2).sum(0) / 4
    return (2.0 * z / chi.sqrt()).to(torch.bfloat16)


GEMM_SHAPES = [(256, 256, 512), (128, 384, 1024), (512, 128, 256)]
# ragged: k not a multiple of the 256-element stage or of 64, n not a multiple
# of the tile (a B tile with one scale band), n % 8 != 0 (element stores),
# single rows and columns, one k-step
GEMM_RAGGED = [(1, 32, 32), (130, 200, 96), (300, 36, 320), (257, 520, 544), (64, 1000, 2048),
               (128, 1, 64), (7, 264, 4128)]


@pytest.fixture(params=["tc256", "tc128", "tc_pair", "cublaslt"])
def gemm_form(h, request):
    h.set_option("gemm", request.param)
    yield request.param
    h.set_option("gemm", "tc256")


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES + GEMM_RAGGED)
def test_nvfp4_gemm_against_oracle(h, gemm_form, m, n, k):
    if gemm_form == "cublaslt" and (m, n, k) in GEMM_RAGGED:
        pytest.skip("the library GEMM is checked on the aligned shapes")
    x = _student_t((m, k), 11 + m)
    w = _student_t((n, k), 13 + n)
    a = h.nvfp4_operand(x.to(DEV))
    b = h.nvfp4_operand(w.to(DEV))
    d = h.nvfp4_gemm(a, b)
    d16 = h.nvfp4_gemm(a, b, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    # the operands are the oracle's, bit for bit
    a_codes, a_bs, a_gs, _ = oracle.rollout_quant(u16(x), None)
    b_codes, b_bs, b_gs, _ = oracle.rollout_quant(u16(w), None)
    assert_same("A codes", a[0].cpu().numpy(), a_codes)
    assert_same("A scales", a[1].cpu().numpy(), oracle.mma_scales(a_bs, m, k))
    assert_same("B codes", b[0].cpu().numpy(), b_codes)
    ref = oracle.nvfp4_gemm(a_codes, a_bs, a_gs[0], b_codes, b_bs, b_gs[0])
    mag = oracle.nvfp4_gemm(a_codes & 0x77, a_bs, a_gs[0], b_codes & 0x77, b_bs, b_gs[0])
    # FP32 accumulation of exact products: |err| <= k * 2^-24 * sum |terms|
    # (plus the final scaling), a bound far below a misplaced block scale
    err = np.abs(d.cpu().double().numpy() - ref)
    bound = k * 2.0 ** -24 * mag + 2.0 ** -126
    assert np.all(err <= bound), float((err / bound).max())
    assert float(np.abs(ref).max()) > 0
    err16 = np.abs(d16.cpu().double().numpy() - ref)
    assert np.all(err16 <= bound + 2.0 ** -8 * np.abs(ref)), float(err16.max())


def test_nvfp4_gemm_full_size_sampled(h):
    """The GEMM at the size the benchmark times (16384 x 8192 x 8192, bf16 and
    fp32 out), every hand-written form; the oracle recomputes sampled rows
    (all 8192 columns each): the first and last rows of tiles, rows in the
    middle of the second tile pair, and seeded random rows."""
    m, n, k = 16384, 8192, 8192
    g = torch.Generator(device=DEV).manual_seed(5)
    x = (torch.randn((m, k), generator=g, device=DEV) * 2.0).to(torch.bfloat16)
    w = (torch.randn((n, k), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    a, b = h.nvfp4_operand(x), h.nvfp4_operand(w)
    rows = sorted(set([0, 127, 128, 255, 256, 383, 300, m - 129, m - 128, m - 1] +
                      np.random.default_rng(7).integers(0, m, 14).tolist()))
    sel = torch.tensor(rows, device=DEV)
    # the operands of the sampled rows and all of B, then the oracle
    a_codes = a[0].index_select(0, sel).cpu().numpy()
    b_codes = b[0].cpu().numpy()
    xs = x.index_select(0, sel).cpu()
    # (the sampled rows quantised with the whole tensor's maximum)
    o_codes, bs_a, _, _ = oracle.rollout_quant(u16(xs), None, amax=[float(x.abs().max())])
    assert_same("A codes (sampled rows)", a_codes, o_codes)
    wb = u16(w.cpu())
    bc, bbs, bgs, _ = oracle.rollout_quant(wb, None)
    assert_same("B codes", b_codes, bc)
    gs_a = np.float32(a[2].cpu().numpy()[0])
    ref = oracle.nvfp4_gemm(a_codes, bs_a, gs_a, bc, bbs, bgs[0])
    mag = oracle.nvfp4_gemm(a_codes & 0x77, bs_a, gs_a, bc & 0x77, bbs, bgs[0])
    bound = k * 2.0 ** -24 * mag + 2.0 ** -126
    try:
        for form in ("tc256", "tc_pair", "tc128"):
            h.set_option("gemm", form)
            for dt in (torch.bfloat16, torch.float32):
                d = h.nvfp4_gemm(a, b, out_dtype=dt)
                torch.cuda.synchronize()
                assert h.device_status() == 0
                got = d.index_select(0, sel).cpu().double().numpy()
                err = np.abs(got - ref)
                lim = bound + (2.0 ** -8 * np.abs(ref) if dt == torch.bfloat16 else 0.0)
                assert np.all(err <= lim), (form, dt, float((err / lim).max()))
    finally:
        h.set_option("gemm", "tc256")


def test_nvfp4_gemm_closed_form(h, gemm_form):
    m, n, k = 128, 128, 256
    x = torch.full((m, k), 1.5, dtype=torch.bfloat16, device=DEV)
    w = torch.full((n, k), -2.0, dtype=torch.bfloat16, device=DEV)
    d = h.nvfp4_gemm(h.nvfp4_operand(x), h.nvfp4_operand(w))
    torch.cuda.synchronize()
    # every element quantises to code 7 (6.0) with block scale 448 (E4M3 max):
    # the sum is exactly -k * 2688^2, scaled by fl32(gs_x * gs_w), gs = amax/2688
    gs_x = np.float32(1.5) / np.float32(2688.0)
    gs_w = np.float32(2.0) / np.float32(2688.0)
    want = np.float32(gs_x * gs_w) * np.float32(-k * 2688.0 * 2688.0)
    assert torch.all(d == float(want)), (float(d[0, 0]), float(want))


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("rows,cols,seg", [(130, 96, None), (256, 64, [0, 100, 256]),
                                           (300, 2048, [0, 1, 299, 300]), (1, 32, None),
                                           (4097, 128, [0, 2000, 4097])])
def test_rollout_quant_writes_tile_layout_scales(h, fused, rows, cols, seg):
    x = rand_bf16((rows, cols), rows * 3 + cols, scale=2.0)
    h.set_option("fused_amax", fused)
    try:
        codes, bs, mma, gs, gd = h.rollout_quant_mma(x.to(DEV), seg, row_major=True, guide=True)
        # the tile layout alone, with nothing else requested
        codes2, none_bs, mma2, _, _ = h.rollout_quant_mma(x.to(DEV), seg)
        torch.cuda.synchronize()
    finally:
        h.set_option("fused_amax", 1)
    assert none_bs is None
    o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(u16(x), seg)
    assert_same("codes", codes.cpu().numpy(), o_codes)
    assert_same("bs", bs.cpu().numpy(), o_bs)
    assert_same("guide", u32(gd), o_guide)
    want = oracle.mma_scales(o_bs, rows, cols)
    assert_same("tile scales", mma.cpu().numpy(), want)
    assert_same("tile scales alone", mma2.cpu().numpy(), want)
    assert_same("codes alone", codes2.cpu().numpy(), o_codes)


# ---------------------------------------------------------------------------
# the host-streamed step (pieces of training segments on three streams)
# equals the one-call step bit for bit
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg,min_rows", [(2, 1), (3, 1), (3, 5000), (5, 1), (5, None)])
def test_host_streamed_step_matches_one_call(h, cfg, min_rows):
    from fp4_rollout_guided_gb300 import pipeline
    w = synth.workload(cfg, small=True)
    x, r = synth.make_inputs(w, "cpu")
    g = run_everything(h, x, r, w.seg_t, w.seg_r, stats=False)
    streamer = pipeline.HostStreamedStep(h, w.rows, w.cols, w.seg_t, w.seg_r, "compact",
                                         min_piece_rows=min_rows)
    x_h, r_h = x.pin_memory(), r.pin_memory()
    outs = streamer.host_outputs()
    for _ in range(2):
        streamer.run(x_h, r_h, outs)
    torch.cuda.synchronize()
    y_h, m_h, gd_h, bs_h, gs_h = outs
    assert_same("streamed y", u16(y_h), g["fq"]["compact"][0])
    assert_same("streamed mask", m_h.numpy().view(np.uint32), g["fq"]["compact"][1])
    assert_same("streamed guide", gd_h.numpy().view(np.uint32), g["guide"])
    assert_same("streamed bs", bs_h.numpy(), g["bs"])
    assert_same("streamed gs", gs_h.numpy().view(np.uint32), g["gs"].view(np.uint32))


# ---------------------------------------------------------------------------
# seeded fuzz: random shapes, independent random segment tables (empty
# segments included), value scales over six decades, drift from tiny to
# unrelated, fused and split rollout paths, random wave sizes
# ---------------------------------------------------------------------------

def _random_table(rng, rows, n):
    cuts = np.sort(rng.integers(0, rows + 1, size=n - 1)) if n > 1 else np.array([], np.int64)
    return [0] + [int(c) for c in cuts] + [rows]


@pytest.mark.parametrize("case", range(16))
def test_fuzz_against_oracle(h, case):
    rng = np.random.default_rng(1000 + case)
    rows = int(rng.integers(1, 2500))
    cols = int(rng.choice([32, 64, 96, 128, 160, 2048]))
    seg_t = _random_table(rng, rows, int(rng.integers(1, 12)))
    seg_r = _random_table(rng, rows, int(rng.integers(1, 40)))
    scale = float(10.0 ** rng.uniform(-3, 3))
    g = torch.Generator().manual_seed(case)
    x = (torch.randn((rows, cols), generator=g) * scale).to(torch.bfloat16)
    sigma = float(rng.choice([2.0 ** -10, 2.0 ** -6, 0.25, 4.0]))
    r = (x.float() * (1 + sigma * torch.randn((rows, cols), generator=g))).to(torch.bfloat16)
    assert torch.isfinite(r.float()).all()
    h.set_option("fused_amax", int(rng.integers(0, 2)))
    h.set_option("wave_bytes", int(rng.choice([4096, 1 << 16, 1 << 20, 32 << 20])))
    try:
        check_all(h, x, r, seg_t, seg_r, f"fuzz{case}")
    finally:
        h.set_option("fused_amax", 1)
        h.set_option("wave_bytes", 32 << 20)
    assert h.device_status() == 0
