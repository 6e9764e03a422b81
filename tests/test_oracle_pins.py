"""Pins for the CPU oracle.

Each test fixes part of the oracle against something other than the oracle:
the worked example the pages print, the OCP format tables, PyTorch's own
float8/bfloat16 casts, brute force over the tiny E2M1 codebook, closed forms
of the guided rule, exact binary64 arithmetic, and invariants that hold at any
size.  A plausible slip anywhere in the oracle (a swapped operand, a wrong
tie rule, an inverted choice, a nibble or bit in the wrong place) fails one of
these.  None of them needs a GPU.

Sources: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
sections "Why Does FP4 Rollout 'Break' RL Training?" (worked example after
Fig. 1) and "TRACE Core Concept" (guided rounding; compact record after
Fig. 3).  OCP Microscaling Formats v1.0 for E2M1 and E4M3.
"""
import os

import numpy as np
import pytest
import torch

from fp4_rollout_guided_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# OCP MX v1.0, FP4 E2M1 table of magnitudes for codes 0..7 (the published
# table, not derived from the oracle's formula).
OCP_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                vals[k] = float(v)
    return vals


def f32_from_bits(u):
    return np.asarray(u, dtype=np.uint32).view(np.float32)


def bits_of(f):
    return np.asarray(f, dtype=np.float32).view(np.uint32)


def bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def neighbourhood(points, radius):
    """All binary32 patterns within +-radius ulps of each non-negative point."""
    out = []
    for p in points:
        b = int(bits_of(p))
        lo = max(0, b - radius)
        out.append(np.arange(lo, b + radius + 1, dtype=np.uint32))
    return f32_from_bits(np.concatenate(out))


# ---------------------------------------------------------------------------
# E2M1: codebook, bracket and round-to-nearest
# ---------------------------------------------------------------------------

def test_e2m1_codebook_matches_ocp_table(orc):
    assert [orc.e2m1_value(m) for m in range(8)] == list(OCP_E2M1)


def brute_rtn(t):
    t = np.asarray(t, dtype=np.float64)
    d = np.abs(t[:, None] - OCP_E2M1[None, :])
    best = d.min(axis=1, keepdims=True)
    tied = d == best
    # among tied indices (at most two adjacent ones) take the even index
    even = tied & (np.arange(8)[None, :] % 2 == 0)
    pick = np.where(tied.sum(1) > 1, even.argmax(1), tied.argmax(1))
    # binary64 distances lose the difference for huge t; mathematically the
    # nearest point above 6 is always 6 (index 7)
    pick[t > 6.0] = 7
    return pick.astype(np.uint8)


def brute_bracket(t):
    t = np.asarray(t, dtype=np.float64)
    lo = (OCP_E2M1[None, :] <= t[:, None]).sum(1) - 1
    hi = 8 - (OCP_E2M1[None, :] >= t[:, None]).sum(1)
    hi = np.minimum(hi, 7)           # above 6 saturates to the top code
    lo = np.where(t > 6.0, 7, lo)
    return lo.astype(np.uint8), hi.astype(np.uint8)


def e2m1_test_values():
    decisions = [0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0]
    near = neighbourhood(decisions, 4096)
    sweep = f32_from_bits(np.arange(0, int(bits_of(8.0)) + 1, 101, dtype=np.uint32))
    special = np.array([np.inf, np.finfo(np.float32).max, 1e30, 8.0, 7.0, 6.0000005],
                       dtype=np.float32)
    return np.concatenate([near, sweep, special]).astype(np.float32)


def test_e2m1_rtn_is_nearest_ties_even(orc):
    t = e2m1_test_values()
    np.testing.assert_array_equal(orc.e2m1_rtn(t), brute_rtn(t))
    # the tie points of the codebook, by hand: ties go to the even index
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    np.testing.assert_array_equal(orc.e2m1_rtn(ties), [0, 2, 2, 4, 4, 6, 6])


def test_e2m1_bracket_definition(orc):
    t = e2m1_test_values()
    lo, hi = orc.e2m1_bracket(t)
    blo, bhi = brute_bracket(t)
    np.testing.assert_array_equal(lo, blo)
    np.testing.assert_array_equal(hi, bhi)
    rtn = orc.e2m1_rtn(t)
    assert np.all((rtn == lo) | (rtn == hi))
    on_grid = np.isin(t.astype(np.float64), OCP_E2M1)
    assert np.all((lo == hi) == (on_grid | (t > 6)))
    assert np.all((hi - lo)[~(on_grid | (t > 6))] == 1)


# ---------------------------------------------------------------------------
# E4M3 and bfloat16 conversions against PyTorch's casts
# ---------------------------------------------------------------------------

def torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_in_range(orc):
    top = int(bits_of(464.0))
    sweep = f32_from_bits(np.arange(0, top, 37, dtype=np.uint32))
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    mids = (vals[:-1].astype(np.float64) + vals[1:]) / 2
    near = neighbourhood(np.concatenate([vals, mids.astype(np.float32)]), 300)
    near = near[near < 464.0]
    v = np.concatenate([sweep, near]).astype(np.float32)
    v = np.concatenate([v, -v[::7]])
    np.testing.assert_array_equal(orc.e4m3_encode(v), torch_e4m3(v))


def test_e4m3_saturation_and_specials(orc):
    # satfinite reading: everything at or above 448 (and infinity) -> 448
    big = np.array([448.0, 449.0, 463.99, 464.0, 500.0, 1e38, np.inf], dtype=np.float32)
    np.testing.assert_array_equal(orc.e4m3_encode(big), np.full(big.shape, 0x7E))
    np.testing.assert_array_equal(orc.e4m3_encode(-big), np.full(big.shape, 0xFE))
    assert orc.e4m3_encode([np.nan])[0] & 0x7F == 0x7F
    # below half the smallest subnormal -> 0; exactly half ties to even (0)
    tiny = np.array([2.0 ** -10, 2.0 ** -11, 1e-30, 0.0], dtype=np.float32)
    np.testing.assert_array_equal(orc.e4m3_encode(tiny), [0, 0, 0, 0])
    assert orc.e4m3_encode([2.0 ** -10 * 1.0000001])[0] == 1
    assert orc.e4m3_encode([3 * 2.0 ** -10])[0] == 2      # 1.5 subnormal steps -> even (2)


def test_e4m3_decode_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = orc.e4m3_decode(codes)
    finite = ~np.isnan(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]))
    assert orc.e4m3_decode([0x7E])[0] == 448.0


def test_bf16_rne_matches_torch(orc):
    rng = np.random.default_rng(0)
    sweep = np.arange(0, 2 ** 32, 251, dtype=np.uint64).astype(np.uint32)
    h = rng.integers(0, 2 ** 16, 200_000, dtype=np.uint64).astype(np.uint32) << 16
    halves = np.concatenate([h | 0x8000, h | 0x7FFF, h | 0x8001, h | 0x0001, h | 0xFFFF])
    u = np.concatenate([sweep, halves])
    f = f32_from_bits(u)
    f = f[~np.isnan(f)]
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(orc.f32_to_bf16(f), ref)
    assert np.isnan(orc.bf16_to_f32(orc.f32_to_bf16(np.array([np.nan], np.float32))))[0]


# ---------------------------------------------------------------------------
# Worked example printed on the pages
# ---------------------------------------------------------------------------

def worked_tensor(train, rollout, gap, shared_scale):
    """One row of two blocks.  Block 0 holds the segment maximum 6*448*gs with
    gs = 1, so the global scale is exactly 1; block 1 holds 6*S (fixing the
    block scale at S) and the example value."""
    seg_max = 6.0 * 448.0
    row_t = np.zeros(32, np.float32)
    row_r = np.zeros(32, np.float32)
    row_t[0] = row_r[0] = seg_max
    row_t[16] = row_r[16] = 6.0 * shared_scale
    row_t[17] = train
    row_r[17] = rollout
    return bf16_bits(row_t).reshape(1, 32), bf16_bits(row_r).reshape(1, 32)


def test_worked_example_from_pages(orc):
    g = read_golden("worked_example.txt")
    assert abs(g["train_value"] - g["rollout_value"] - g["value_gap"]) < 1e-9
    # the printed gap is (3 - 2) * S, so the shared scale is the gap itself
    S = g["amplified_gap"] / (g["train_rtn_value"] - g["rollout_rtn_value"])
    x_t, x_r = worked_tensor(g["train_value"], g["rollout_value"], g["value_gap"], S)

    codes_r, bs_r, gs_r, guide = orc.rollout_quant(x_r)
    codes_t, bs_t, gs_t, _ = orc.rollout_quant(x_t)
    assert gs_r[0] == 1.0 and gs_t[0] == 1.0                # the shared global scale
    assert bs_r[0, 1] == bs_t[0, 1] == 0x5C                  # E4M3 24.0: the shared block scale
    assert orc.e4m3_decode([0x5C])[0] == S

    Sv, inv = orc.scale_pair(bs_t[0, 1], gs_t[0])
    xt = float(orc.bf16_to_f32(x_t[:, 17])[0])
    xr = float(orc.bf16_to_f32(x_r[:, 17])[0])
    t_t = np.float32(xt) * np.float32(inv)
    t_r = np.float32(xr) * np.float32(inv)
    assert abs(t_t - g["train_normalised"]) < 0.005
    assert abs(t_r - g["rollout_normalised"]) < 0.005

    def nib(codes, e):
        b = codes[0, e // 2]
        return (b >> 4) if e & 1 else (b & 15)

    m_t, m_r = nib(codes_t, 17), nib(codes_r, 17)
    assert orc.e2m1_value(m_t) == g["train_rtn_value"]       # RTN: 2.51 -> 3
    assert orc.e2m1_value(m_r) == g["rollout_rtn_value"]     # RTN: 2.49 -> 2
    assert codes_t[0, 8] == 0x57 and codes_r[0, 8] == 0x47   # element 16 low nibble, 17 high

    # plain fake quant keeps the amplified gap; guidance removes it
    y_rtn, _, _, _ = orc.train_fakequant(x_t)
    y_full, _, c_full, st_full = orc.train_fakequant(x_t, kind=orc.GUIDE_FULL, guide=codes_r,
                                                     bs_r=bs_r, gs_r=gs_r)
    y_cmp, _, c_cmp, st_cmp = orc.train_fakequant(x_t, kind=orc.GUIDE_COMPACT, guide=guide,
                                                  bs_r=bs_r, gs_r=gs_r)
    y_rtn_v = orc.bf16_to_f32(y_rtn[0, 17])
    y_g_v = orc.bf16_to_f32(y_full[0, 17])
    roll_v = orc.e2m1_value(m_r) * S
    assert y_rtn_v - roll_v == g["amplified_gap"]
    assert y_g_v == roll_v
    np.testing.assert_array_equal(y_full, y_cmp)
    np.testing.assert_array_equal(c_full, c_cmp)
    assert st_full[orc.STAT_MISMATCH_RTN] == 1 and st_full[orc.STAT_MISMATCH_GUIDED] == 0
    # the compact word of block 1: all signs 0; LSB of element 16 (index 7)
    # is 1, of element 17 (index 4) is 0
    assert guide[0, 1] == 0x00010000


def test_clipped_element_mask_by_hand(orc):
    """gs = 1; a block whose max is 147: 147/6 = 24.5 lies between the E4M3
    values 24 and 26 and rounds (tie, even mantissa) to 24, so 6*S = 144 < 147
    and that element alone is clipped.  Placed at element 35 of the row, it is
    bit 3 of mask word 1."""
    row = np.zeros(64, np.float32)
    row[0] = 2688.0
    row[35] = 147.0
    row[36] = -100.0
    x = bf16_bits(row).reshape(1, 64)
    codes, bs, gs, _ = orc.rollout_quant(x)
    assert bs[0, 2] == 0x5C
    y, mask, codes_t, _ = orc.train_fakequant(x)
    assert mask[0, 0] == 0xFFFFFFFF
    assert mask[0, 1] == 0xFFFFFFFF & ~(1 << 3)
    # clipped element saturates to 6 * 24 = 144; -100/24 = 4.1667 -> 4 (-96)
    assert orc.bf16_to_f32(y[0, 35]) == 144.0
    assert orc.bf16_to_f32(y[0, 36]) == -96.0
    # element 35 is the high nibble of byte 17, element 36 the low nibble of 18
    assert codes_t[0, 17] == 0x70
    assert codes_t[0, 18] == 0x0E


# ---------------------------------------------------------------------------
# Guided rule: closed form at equal scales, exact-distance check elsewhere
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1.0, 0.375, 24.0, 0.3700000047683716, 1.2345e-3, 7.77e4])
def test_guided_rule_closed_form_equal_scales(orc, S):
    """With S_t == S_r: the answer is lo when the rollout sign differs or the
    rollout index is at most lo, else hi (opposite signs make the smaller
    magnitude the closer one)."""
    S = float(np.float32(S))
    inv = float(np.float32(1.0) / np.float32(S))
    for lo in range(7):
        a, b = OCP_E2M1[lo], OCP_E2M1[lo + 1]
        ts = np.linspace(a, b, 67)[1:-1].astype(np.float32)
        ts = np.concatenate([ts, f32_from_bits(bits_of(np.float32(a)) + np.arange(1, 4)),
                             f32_from_bits(bits_of(np.float32(b)) - np.arange(1, 4))])
        for t in ts:
            x_mag = np.float32(t) * np.float32(S)
            tt = np.float32(x_mag) * np.float32(inv)
            blo, bhi = brute_bracket(np.array([tt]))
            if blo[0] != lo or bhi[0] != lo + 1:
                continue   # the product moved t onto a neighbouring interval
            for s_t in (0, 1):
                x = -x_mag if s_t else x_mag
                for nib in range(16):
                    s_r, m_r = nib >> 3, nib & 7
                    expect = lo if (s_r != s_t or m_r <= lo) else lo + 1
                    got = orc.guided_index(x, S, inv, 1, nib, S)
                    assert got == expect, (S, lo, float(t), s_t, nib)


def test_guided_rule_agrees_with_exact_distances(orc):
    """Random scales on both sides: whenever the two candidates' exact
    (binary64) distances differ by more than a few binary32 ulps, the oracle's
    choice is the closer candidate; with no guide it is RTN."""
    rng = np.random.default_rng(1)
    n = 20000
    S_t = rng.uniform(0.01, 10, n).astype(np.float32)
    S_r = (S_t * rng.uniform(0.8, 1.25, n)).astype(np.float32)
    t = rng.uniform(0, 6, n).astype(np.float32)
    s_t = rng.integers(0, 2, n)
    nib = rng.integers(0, 16, n)
    checked = 0
    for i in range(n):
        inv = float(np.float32(1) / S_t[i])
        xm = np.float32(t[i]) * S_t[i]
        x = -xm if s_t[i] else xm
        tt = np.float32(abs(np.float32(x))) * np.float32(inv)
        lo, hi = (int(v[0]) for v in brute_bracket(np.array([tt])))
        got = orc.guided_index(x, S_t[i], inv, 1, int(nib[i]), S_r[i])
        assert got in (lo, hi)
        assert orc.guided_index(x, S_t[i], inv, 0, int(nib[i]), S_r[i]) == brute_rtn([tt])[0]
        if lo == hi:
            continue
        sgn_t = -1.0 if s_t[i] else 1.0
        sgn_r = -1.0 if nib[i] >> 3 else 1.0
        v_r = sgn_r * OCP_E2M1[nib[i] & 7] * float(S_r[i])
        d_lo = abs(sgn_t * OCP_E2M1[lo] * float(S_t[i]) - v_r)
        d_hi = abs(sgn_t * OCP_E2M1[hi] * float(S_t[i]) - v_r)
        if abs(d_lo - d_hi) > 1e-5 * (d_lo + d_hi + 1e-30):
            assert got == (lo if d_lo < d_hi else hi)
            checked += 1
    assert checked > n // 2


# ---------------------------------------------------------------------------
# Whole tensors: scales, outputs, mask and statistics against independent
# library arithmetic
# ---------------------------------------------------------------------------

def expand_rows(per_seg, seg, rows):
    idx = np.repeat(np.arange(len(seg) - 1), np.diff(seg))
    assert len(idx) == rows
    return per_seg[idx]


def block_real_scale(bs, gs, seg):
    """S = decode(bs) * gs per block, decode by PyTorch's float8 cast."""
    rows = bs.shape[0]
    dec = torch.from_numpy(np.ascontiguousarray(bs)).view(torch.float8_e4m3fn).float().numpy()
    g = expand_rows(gs.astype(np.float32), seg, rows)[:, None]
    return (dec * g).astype(np.float32)


def nibbles(codes):
    lo = codes & 15
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


SMALL = [1, 2, 3, 4, 5]


@pytest.fixture(scope="module")
def small_runs(orc):
    runs = {}
    for cfg in SMALL:
        w = synth.workload(cfg, small=True)
        x, r = synth.make_inputs(w, "cpu")
        xu, ru = synth.to_u16(x), synth.to_u16(r)
        codes_r, bs_r, gs_r, guide = orc.rollout_quant(ru, w.seg_r)
        runs[cfg] = dict(w=w, x=xu, r=ru, codes_r=codes_r, bs_r=bs_r, gs_r=gs_r, guide=guide)
    return runs


@pytest.mark.parametrize("cfg", SMALL)
def test_amax_and_global_scale_against_numpy(orc, small_runs, cfg):
    run = small_runs[cfg]
    w = run["w"]
    xf = orc.bf16_to_f32(run["r"])
    am = orc.segment_amax(run["r"], w.seg_r)
    for s in range(w.n_seg_r):
        part = xf[w.seg_r[s]:w.seg_r[s + 1]]
        ref = np.abs(part).max() if part.size else 0.0
        assert am[s] == ref
        expect_gs = np.float32(ref) / np.float32(2688.0) if ref > 0 else 0.0
        assert run["gs_r"][s] == expect_gs


@pytest.mark.parametrize("cfg", SMALL)
def test_block_scales_against_torch_e4m3(orc, small_runs, cfg):
    run = small_runs[cfg]
    w = run["w"]
    xf = np.abs(orc.bf16_to_f32(run["r"]))
    bamax = xf.reshape(w.rows, -1, 16).max(-1)
    g = expand_rows(run["gs_r"], w.seg_r, w.rows)[:, None]
    q = (bamax / (g * np.float32(6.0))).astype(np.float32)
    np.testing.assert_array_equal(run["bs_r"], torch_e4m3(np.minimum(q, 448.0)))


@pytest.mark.parametrize("cfg", SMALL)
def test_rtn_codes_and_outputs(orc, small_runs, cfg):
    """Unguided fake quant equals the rollout quantiser applied to the training
    tensor; each code is the nearest E2M1 point of |x| * (1/S) (brute force);
    y is PyTorch's bfloat16 cast of +-G[m] * S; the mask bit is 0 exactly when
    |x| exceeds 6*S, with 6*S rounded to binary32 from the exact binary64
    product."""
    run = small_runs[cfg]
    w = run["w"]
    codes_q, bs_t, gs_t, _ = orc.rollout_quant(run["x"], w.seg_t)
    y, mask, codes_t, stats = orc.train_fakequant(run["x"], w.seg_t)
    np.testing.assert_array_equal(codes_t, codes_q)
    S = np.repeat(block_real_scale(bs_t, gs_t, w.seg_t), 16, axis=1)
    with np.errstate(divide="ignore"):
        inv = np.where(S > 0, np.float32(1.0) / S, np.float32(0.0)).astype(np.float32)
    inv[np.isinf(inv)] = 0
    xf = orc.bf16_to_f32(run["x"])
    t = (np.abs(xf) * inv).astype(np.float32)
    nib = nibbles(codes_t)
    np.testing.assert_array_equal(nib & 7, brute_rtn(t.ravel()).reshape(t.shape))
    np.testing.assert_array_equal(nib >> 3, np.signbit(xf).astype(np.uint8))
    deq = (OCP_E2M1[nib & 7].astype(np.float32) * S).astype(np.float32)
    deq = np.where(np.signbit(xf), -deq, deq).astype(np.float32)
    ref_y = torch.from_numpy(deq).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(y, ref_y)
    six_s = (6.0 * S.astype(np.float64)).astype(np.float32)
    clipped = (S > 0) & (np.abs(xf) > six_s)
    bits = ((mask[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(w.rows, -1)
    np.testing.assert_array_equal(bits, (~clipped).astype(np.uint32))
    assert stats[orc.STAT_N] == w.elems


@pytest.mark.parametrize("cfg", SMALL)
def test_guided_invariants_and_statistics(orc, small_runs, cfg):
    """Guided index is always one of the two adjacent candidates (P4); the
    compact and full records give the same result wherever the rollout index
    lies in the training value's bracket in the rollout frame (P6); the
    statistics recount from the codes."""
    run = small_runs[cfg]
    w = run["w"]
    x = run["x"]
    _, bs_t, gs_t, _ = orc.rollout_quant(x, w.seg_t)
    y0, _, c_rtn, _ = orc.train_fakequant(x, w.seg_t)
    common = dict(bs_r=run["bs_r"], gs_r=run["gs_r"], seg_r=w.seg_r)
    y_f, m_f, c_f, st_f = orc.train_fakequant(x, w.seg_t, orc.GUIDE_FULL, run["codes_r"], **common)
    y_c, m_c, c_c, st_c = orc.train_fakequant(x, w.seg_t, orc.GUIDE_COMPACT, run["guide"], **common)

    xf = orc.bf16_to_f32(x)
    S_t = np.repeat(block_real_scale(bs_t, gs_t, w.seg_t), 16, axis=1)
    inv_t = np.where(S_t > 0, np.float32(1) / np.where(S_t > 0, S_t, 1), 0).astype(np.float32)
    lo, hi = orc.e2m1_bracket((np.abs(xf) * inv_t).astype(np.float32).ravel())
    lo, hi = lo.reshape(xf.shape), hi.reshape(xf.shape)
    for c in (c_f, c_c):
        m = nibbles(c) & 7
        assert np.all((m == lo) | (m == hi))
        single = lo == hi
        np.testing.assert_array_equal(nibbles(c)[single], nibbles(c_rtn)[single])

    # P6: compact == full where the rollout index is inside the bracket of
    # x_t measured in the rollout's scale frame (or that bracket is a point)
    S_r = np.repeat(block_real_scale(run["bs_r"], run["gs_r"], w.seg_r), 16, axis=1)
    inv_r = np.where(S_r > 0, np.float32(1) / np.where(S_r > 0, S_r, 1), 0).astype(np.float32)
    lo_r, hi_r = orc.e2m1_bracket((np.abs(xf) * inv_r).astype(np.float32).ravel())
    lo_r, hi_r = lo_r.reshape(xf.shape), hi_r.reshape(xf.shape)
    m_r = nibbles(run["codes_r"]) & 7
    inside = (m_r == lo_r) | (m_r == hi_r)
    agree = nibbles(c_f) == nibbles(c_c)
    assert np.all(agree[inside])
    np.testing.assert_array_equal(m_f, m_c)

    # statistics recount (signed index, +-0 equal)
    def k(n):
        m = (n & 7).astype(np.int64)
        return np.where(n >> 3, -m, m)
    k_r, k_rtn = k(nibbles(run["codes_r"])), k(nibbles(c_rtn))
    for c, st in ((c_f, st_f), (c_c, st_c)):
        assert st[orc.STAT_N] == w.elems
        assert sum(st[orc.STAT_HIST_RTN:orc.STAT_HIST_RTN + 4]) == w.elems
        assert sum(st[orc.STAT_HIST_GUIDED:orc.STAT_HIST_GUIDED + 4]) == w.elems
        assert st[orc.STAT_MISMATCH_GUIDED] <= st[orc.STAT_MISMATCH_RTN]
    assert st_f[orc.STAT_MISMATCH_RTN] == np.count_nonzero(k_rtn != k_r)
    assert st_f[orc.STAT_MISMATCH_GUIDED] == np.count_nonzero(k(nibbles(c_f)) != k_r)
    d = np.minimum(np.abs(k(nibbles(c_f)) - k_r), 3)
    np.testing.assert_array_equal(st_f[orc.STAT_HIST_GUIDED:orc.STAT_HIST_GUIDED + 4],
                                  np.bincount(d.ravel(), minlength=4))
    d = np.minimum(np.abs(k_rtn - k_r), 3)
    np.testing.assert_array_equal(st_f[orc.STAT_HIST_RTN:orc.STAT_HIST_RTN + 4],
                                  np.bincount(d.ravel(), minlength=4))
    # guidance never leaves more disagreements than RTN on these workloads
    assert st_f[orc.STAT_MISMATCH_GUIDED] <= st_f[orc.STAT_MISMATCH_RTN]


def test_idempotence_when_rollout_equals_training(orc, small_runs):
    """P4: a rollout record made from the training tensor itself changes
    nothing: guided == RTN, zero mismatches before and after."""
    run = small_runs[2]
    w = run["w"]
    codes, bs, gs, guide = orc.rollout_quant(run["x"], w.seg_t)
    y0, m0, c0, _ = orc.train_fakequant(run["x"], w.seg_t)
    for kind, g in ((orc.GUIDE_FULL, codes), (orc.GUIDE_COMPACT, guide)):
        y, m, c, st = orc.train_fakequant(run["x"], w.seg_t, kind, g, bs, gs, w.seg_t)
        np.testing.assert_array_equal(y, y0)
        np.testing.assert_array_equal(c, c0)
        assert st[orc.STAT_MISMATCH_RTN] == 0 and st[orc.STAT_MISMATCH_GUIDED] == 0


def test_equal_scale_tensor_closed_form(orc):
    """P3 at tensor level: the rollout copy keeps every block's largest
    element (so both sides have identical scales) and perturbs the rest; the
    guided code then follows the closed form of the equal-scale rule."""
    rng = np.random.default_rng(7)
    rows, cols = 64, 256
    xt = rng.standard_normal((rows, cols)).astype(np.float32)
    x = bf16_bits(xt).reshape(rows, cols)
    xf = orc.bf16_to_f32(x)
    pert = (xf * (1 + rng.standard_normal(xf.shape).astype(np.float32) * np.float32(0.05))).astype(np.float32)
    blocks = np.abs(xf).reshape(rows, -1, 16)
    is_max = (blocks == blocks.max(-1, keepdims=True)).reshape(rows, cols)
    pert = np.where(is_max, xf, np.clip(pert, -np.abs(xf).reshape(rows, -1, 16).max(-1).repeat(16, 1),
                                         np.abs(xf).reshape(rows, -1, 16).max(-1).repeat(16, 1)))
    r = bf16_bits(pert.ravel()).reshape(rows, cols)
    codes_r, bs_r, gs_r, guide = orc.rollout_quant(r)
    codes_t, bs_t, gs_t, _ = orc.rollout_quant(x)
    np.testing.assert_array_equal(bs_r, bs_t)
    assert gs_r[0] == gs_t[0]
    _, _, c_g, _ = orc.train_fakequant(x, None, orc.GUIDE_FULL, codes_r, bs_r, gs_r)
    S = np.repeat(block_real_scale(bs_t, gs_t, np.array([0, rows])), 16, axis=1)
    inv = (np.float32(1) / S).astype(np.float32)
    lo, hi = brute_bracket((np.abs(xf) * inv).astype(np.float32).ravel())
    lo, hi = lo.reshape(xf.shape), hi.reshape(xf.shape)
    nr = nibbles(codes_r)
    s_t = np.signbit(xf).astype(np.uint8)
    expect = np.where((nr >> 3 != s_t) | ((nr & 7) <= lo), lo, hi)
    expect = np.where(lo == hi, lo, expect)
    np.testing.assert_array_equal(nibbles(c_g) & 7, expect)


# ---------------------------------------------------------------------------
# Compact record: pack / unpack round trips (P7) and segment independence (P8)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", SMALL)
def test_pack_unpack_round_trip(orc, small_runs, cfg):
    run = small_runs[cfg]
    w = run["w"]
    g = orc.guide_pack(run["codes_r"])
    np.testing.assert_array_equal(g, run["guide"])
    back = orc.guide_unpack(run["r"], g, run["bs_r"], run["gs_r"], w.seg_r)
    np.testing.assert_array_equal(back, run["codes_r"])
    # unpack against the training values, then re-pack: signs always survive,
    # LSBs survive wherever the bracket is two points
    est = orc.guide_unpack(run["x"], g, run["bs_r"], run["gs_r"], w.seg_r)
    g2 = orc.guide_pack(est)
    np.testing.assert_array_equal(g2 & 0xFFFF, g & 0xFFFF)
    xf = orc.bf16_to_f32(run["x"])
    S_r = np.repeat(block_real_scale(run["bs_r"], run["gs_r"], w.seg_r), 16, axis=1)
    inv_r = np.where(S_r > 0, np.float32(1) / np.where(S_r > 0, S_r, 1), 0).astype(np.float32)
    lo, hi = brute_bracket((np.abs(xf) * inv_r).astype(np.float32).ravel())
    two = (lo != hi).reshape(w.rows, -1, 16)
    lsb1 = ((g[:, :, None] >> (16 + np.arange(16, dtype=np.uint32))) & 1).astype(bool)
    lsb2 = ((g2[:, :, None] >> (16 + np.arange(16, dtype=np.uint32))) & 1).astype(bool)
    assert np.all(lsb1[two] == lsb2[two])


def test_pack_bit_layout_by_hand(orc):
    codes = np.zeros((1, 16), np.uint8)            # one row of 32 elements
    codes[0, 0] = 0x9 | (0x3 << 4)                 # e0: -0.5 (sign, lsb 1); e1: 1.5 (lsb 1)
    codes[0, 9] = 0xE << 4                         # e19: -4 (sign, lsb 0)
    g = orc.guide_pack(codes)
    assert g[0, 0] == (1 << 0) | (1 << 16) | (1 << 17)
    assert g[0, 1] == (1 << 3)


def test_segment_independence(orc, small_runs):
    """P8: quantising one segment alone equals the same rows of a batched
    call; for the chunked KV stream, the batched record equals the
    concatenation of per-chunk calls."""
    for cfg in (2, 5):
        run = small_runs[cfg]
        w = run["w"]
        for s in range(0, w.n_seg_r, max(1, w.n_seg_r // 7)):
            a, b = int(w.seg_r[s]), int(w.seg_r[s + 1])
            c, bs, gs, g = orc.rollout_quant(run["r"][a:b])
            np.testing.assert_array_equal(c, run["codes_r"][a:b])
            np.testing.assert_array_equal(bs, run["bs_r"][a:b])
            np.testing.assert_array_equal(g, run["guide"][a:b])
            assert gs[0] == run["gs_r"][s]
    run = small_runs[5]
    w = run["w"]
    for s in (0, w.n_seg_t - 1):
        a, b = int(w.seg_t[s]), int(w.seg_t[s + 1])
        inner, first = synth.rollout_segments_within(w, s)
        y_part = orc.train_fakequant(run["x"][a:b], None, orc.GUIDE_COMPACT, run["guide"][a:b],
                                     run["bs_r"][a:b], run["gs_r"][first:first + len(inner) - 1],
                                     inner)[0]
        y_all = orc.train_fakequant(run["x"], w.seg_t, orc.GUIDE_COMPACT, run["guide"],
                                    run["bs_r"], run["gs_r"], w.seg_r)[0]
        np.testing.assert_array_equal(y_part, y_all[a:b])


def test_bad_arguments_rejected(orc):
    x = np.zeros((4, 32), np.uint16)
    with pytest.raises(ValueError):
        orc.rollout_quant(np.zeros((4, 48), np.uint16))
    with pytest.raises(ValueError):
        orc.rollout_quant(x, np.array([0, 3, 2, 4]))
    with pytest.raises(ValueError):
        orc.rollout_quant(x, np.array([0, 5]))
    with pytest.raises(ValueError):
        orc.train_fakequant(x, None, orc.GUIDE_COMPACT, None)


def test_empty_and_zero_inputs(orc):
    x = np.zeros((0, 64), np.uint16)
    c, bs, gs, g = orc.rollout_quant(x, np.array([0, 0, 0]))
    assert c.shape == (0, 32) and np.all(gs == 0)
    z = np.zeros((3, 64), np.uint16)
    c, bs, gs, g = orc.rollout_quant(z)
    assert gs[0] == 0 and np.all(bs == 0) and np.all(c == 0)
    y, m, ct, st = orc.train_fakequant(z)
    assert np.all(y == 0) and np.all(m == 0xFFFFFFFF)
    negz = np.full((1, 32), 0x8000, np.uint16)   # -0.0 keeps its sign bit in the code
    c, _, _, g = orc.rollout_quant(negz)
    assert np.all(c == 0x88) and g[0, 0] == 0xFFFF


def test_equal_distances_fall_back_to_rtn(orc):
    """Hand case: S_t = 1 and the rollout value 2.0 * 1.25 = 2.5 sits exactly
    halfway between the candidates 2 and 3, so the distances tie and the RTN
    choice stands: t = 2.3 -> index 4, t = 2.7 -> index 5."""
    S_t, inv_t, S_r = 1.0, 1.0, 1.25
    nib_r = 4                       # +2.0 in the rollout's frame -> 2.5
    assert orc.guided_index(2.3, S_t, inv_t, 1, nib_r, S_r) == 4
    assert orc.guided_index(2.7, S_t, inv_t, 1, nib_r, S_r) == 5
    assert orc.guided_index(-2.7, S_t, inv_t, 1, nib_r | 8, S_r) == 5
    # off the tie the closer candidate wins regardless of RTN
    assert orc.guided_index(2.7, S_t, inv_t, 1, nib_r, 1.2) == 4
    assert orc.guided_index(2.3, S_t, inv_t, 1, nib_r, 1.3) == 5


def test_tiny_block_is_flushed(orc):
    """A block whose real scale S is positive but below 2^-128 has a
    reciprocal that overflows binary32; by the flush reading its elements all
    normalise to 0 (code 0, output 0), while the mask still follows |x| > 6S.
    Checked with the exact binary64 reciprocal."""
    amax = 2.0 ** -118
    row = np.zeros(32, np.float32)
    row[0] = amax
    row[16] = amax / 1000.0         # block scale 0.448 -> E4M3 0.4375, S ~ 2^-130.6
    row[17] = -amax / 3000.0
    x = bf16_bits(row).reshape(1, 32)
    codes, bs, gs, _ = orc.rollout_quant(x)
    S, inv = orc.scale_pair(bs[0, 1], gs[0])
    assert S > 0 and 1.0 / float(S) > float(np.finfo(np.float32).max)   # overflows
    assert inv == 0.0
    assert codes[0, 8] == 0x80            # e16 -> +0, e17 -> -0 (sign kept)
    y, m, c, _ = orc.train_fakequant(x)
    assert y[0, 16] == 0 and y[0, 17] == 0x8000
    S0, inv0 = orc.scale_pair(bs[0, 0], gs[0])
    assert np.isfinite(inv0) and inv0 > 0


def test_unrelated_rollout_statistics(orc):
    """A rollout tensor drawn independently of the training tensor exercises
    opposite signs and far-apart codes: every histogram bucket fills, the
    compact record still agrees with the full one wherever the rollout index
    lies in the training value's rollout-frame bracket, and the counters
    recount exactly from codes (the compact run against its decoded codes)."""
    rng = np.random.default_rng(11)
    rows, cols = 96, 512
    seg = np.array([0, 40, 41, 96], np.int64)
    x = bf16_bits(rng.standard_normal(rows * cols).astype(np.float32)).reshape(rows, cols)
    r = bf16_bits((rng.standard_normal(rows * cols) * 1.7).astype(np.float32)).reshape(rows, cols)
    codes_r, bs_r, gs_r, guide = orc.rollout_quant(r, seg)
    _, _, c_rtn, _ = orc.train_fakequant(x, seg)
    kw = dict(bs_r=bs_r, gs_r=gs_r, seg_r=seg)
    _, _, c_f, st_f = orc.train_fakequant(x, seg, orc.GUIDE_FULL, codes_r, **kw)
    _, _, c_c, st_c = orc.train_fakequant(x, seg, orc.GUIDE_COMPACT, guide, **kw)
    dec = orc.guide_unpack(x, guide, bs_r, gs_r, seg)

    def k(n):
        m = (n & 7).astype(np.int64)
        return np.where(n >> 3, -m, m)

    for c, st, ref in ((c_f, st_f, codes_r), (c_c, st_c, dec)):
        k_r = k(nibbles(ref))
        for base, kk in ((orc.STAT_HIST_RTN, k(nibbles(c_rtn))), (orc.STAT_HIST_GUIDED, k(nibbles(c)))):
            d = np.minimum(np.abs(kk - k_r), 3)
            np.testing.assert_array_equal(st[base:base + 4], np.bincount(d.ravel(), minlength=4))
        assert st[orc.STAT_MISMATCH_RTN] == np.count_nonzero(k(nibbles(c_rtn)) != k_r)
        assert st[orc.STAT_MISMATCH_GUIDED] == np.count_nonzero(k(nibbles(c)) != k_r)
    assert np.all(st_f[orc.STAT_HIST_RTN:orc.STAT_HIST_RTN + 4] > 0)
    assert np.all(st_f[orc.STAT_HIST_GUIDED:orc.STAT_HIST_GUIDED + 4] > 0)

    xf = orc.bf16_to_f32(x)
    S_r = np.repeat(block_real_scale(bs_r, gs_r, seg), 16, axis=1)
    inv_r = (np.float32(1) / S_r).astype(np.float32)
    lo_r, hi_r = brute_bracket((np.abs(xf) * inv_r).astype(np.float32).ravel())
    lo_r, hi_r = lo_r.reshape(xf.shape), hi_r.reshape(xf.shape)
    n_r = nibbles(codes_r)
    inside = ((n_r & 7) == lo_r) | ((n_r & 7) == hi_r)
    assert np.count_nonzero(np.signbit(xf) != (n_r >> 3).astype(bool)) > 1000
    np.testing.assert_array_equal(nibbles(c_f)[inside], nibbles(c_c)[inside])
    np.testing.assert_array_equal(nibbles(dec)[inside], n_r[inside])


def test_ste_backward_against_numpy_unpackbits(orc):
    """The backward passes the gradient where numpy's little-endian unpacking
    of the mask words has a 1 and gives +0 elsewhere; with the fake
    quantiser's own mask, clipped elements (|x| > 6 S) get no gradient."""
    rng = np.random.default_rng(3)
    rows, cols = 37, 96
    g = rng.integers(0, 2 ** 16, (rows, cols), dtype=np.uint64).astype(np.uint16)
    m = rng.integers(0, 2 ** 32, (rows, cols // 32), dtype=np.uint64).astype(np.uint32)
    out = orc.ste_backward(g, m)
    bits = np.unpackbits(m.view(np.uint8), bitorder="little").reshape(rows, cols).astype(bool)
    np.testing.assert_array_equal(out, np.where(bits, g, 0))
    row = np.zeros(64, np.float32)
    row[0], row[35] = 2688.0, 147.0                      # element 35 is clipped (see above)
    x = bf16_bits(row).reshape(1, 64)
    _, mask, _, _ = orc.train_fakequant(x)
    grad = np.full((1, 64), 0x3F80, np.uint16)             # all ones
    gi = orc.ste_backward(grad, mask)
    assert gi[0, 35] == 0 and np.all(np.delete(gi[0], 35) == 0x3F80)


# ---------------------------------------------------------------------------
# tensor-core block-scale layout and the NVFP4 GEMM (the consumer of the
# rollout codes); the layout is NVIDIA's documented interface, not the
# article's, and is pinned against the hardware library by the GPU GEMM test
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(1, 32), (130, 80), (256, 64), (129, 2048), (300, 96)])
def test_mma_scales_as_tile_reshape(orc, rows, cols):
    """The tiled layout restated as a tensor reshape: pad to (R, C), split
    rows into (tile, 4 groups of 32) and columns into (tile, 4), order the
    axes (row tile, column tile, row in group, group, column in tile)."""
    g = np.random.default_rng(rows * 7 + cols)
    sc = cols // 16
    bs = g.integers(1, 256, size=(rows, sc), dtype=np.uint8)
    R, C = -(-rows // 128) * 128, -(-sc // 4) * 4
    pad = np.zeros((R, C), dtype=np.uint8)
    pad[:rows, :sc] = bs
    want = pad.reshape(R // 128, 4, 32, C // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    got = orc.mma_scales(bs, rows, cols)
    assert got.shape == want.shape and np.array_equal(got, want)


def test_mma_scales_places_every_scale_once(orc):
    rows, cols = 200, 112
    sc = cols // 16
    ids = np.arange(rows * sc, dtype=np.int64)
    # encode each position's identity in two layouts of distinct bytes
    lo = orc.mma_scales((ids % 251 + 1).astype(np.uint8), rows, cols)
    hi = orc.mma_scales((ids // 251 + 1).astype(np.uint8), rows, cols)
    filled = lo != 0
    assert filled.sum() == rows * sc and np.array_equal(filled, hi != 0)
    key = (hi[filled].astype(np.int64) - 1) * 251 + (lo[filled].astype(np.int64) - 1)
    assert np.array_equal(np.sort(key), ids)
    # row 33, scale column 2 of the first tile: 16 * 1 + 4 * 1 + 2
    assert (hi[22] - 1) * 251 + (lo[22] - 1) == 33 * sc + 2


def _dequant(codes, bs, rows, cols):
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(rows, cols)
    val = OCP_E2M1[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    s = torch.from_numpy(bs.copy()).view(torch.float8_e4m3fn).double().numpy()
    return val * np.repeat(s, 16, axis=1)


def test_nvfp4_gemm_matches_dequantised_matmul(orc):
    g = np.random.default_rng(5)
    m, n, k = 7, 5, 96
    a_codes = g.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    b_codes = g.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    a_bs = g.integers(0x20, 0x50, size=(m, k // 16), dtype=np.uint8)
    b_bs = g.integers(0x20, 0x50, size=(n, k // 16), dtype=np.uint8)
    a_gs, b_gs = np.float32(0.0123), np.float32(3.5e-3)
    d = orc.nvfp4_gemm(a_codes, a_bs, a_gs, b_codes, b_bs, b_gs)
    ref = _dequant(a_codes, a_bs, m, k) @ _dequant(b_codes, b_bs, n, k).T
    alpha = float(np.float32(a_gs * b_gs))
    np.testing.assert_allclose(d, alpha * ref, rtol=1e-12, atol=0)


def test_nvfp4_gemm_closed_form(orc):
    m, n, k = 3, 4, 64
    ones = np.full((m, k // 2), 0x22, dtype=np.uint8)       # E2M1 1.0 in both nibbles
    neg = np.full((n, k // 2), 0xAA, dtype=np.uint8)        # E2M1 -1.0
    s1 = np.full((m, k // 16), 0x38, dtype=np.uint8)        # E4M3 1.0
    s2 = np.full((n, k // 16), 0x40, dtype=np.uint8)        # E4M3 2.0
    d = orc.nvfp4_gemm(ones, s1, 0.5, neg, s2, 0.25)
    assert np.all(d == -k * 2.0 * 0.125)
