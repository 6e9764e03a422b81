"""The bounds-checking debug build (TRACE_DEBUG_BOUNDS).

The library is built a second time with -DTRACE_DEBUG_BOUNDS, into a
temporary directory, and loaded in a child process.  There every call
registers the byte ranges of its buffers and its scratch before it
launches, and the hot-path kernels count (and skip) any global access
outside them.  Every entry point runs on ragged shapes and segment tables
with empty segments: no access may fall outside, and the bytes must be the
oracle's.  With the test option that registers each output 16 bytes short,
the kernels' last stores must be counted and skipped (the bytes there keep
their fill pattern), which shows the checks are live.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import json, sys
import numpy as np, torch
sys.path.insert(0, ROOT)
sys.path.insert(0, ROOT + "/tests")
from fp4_rollout_guided_gb300 import build, synth, trace
import oracle
lib_path = build.build(extra_flags=["-DTRACE_DEBUG_BOUNDS"], out_dir=OUT)
trace.library_path = lambda: lib_path
oracle.build()
dev = torch.device("cuda", 0)
out = {"cases": []}
h = trace.Handle(0)
checked, v0 = h.debug_bounds()
out["checked"] = checked
def rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)
for rows, cols, seg in [(1, 32, None), (3, 96, [0, 0, 2, 3]), (257, 64, [0, 100, 100, 257]),
                        (4099, 128, [0, 2048, 4099]), (130, 2048, [0, 1, 129, 130])]:
    seg = None if seg is None else np.array(seg, np.int64)
    x = rand((rows, cols), rows + cols, 2.0)
    r = (x.float() * 1.01).to(torch.bfloat16)
    xg, rg = x.to(dev), r.to(dev)
    res = {"shape": [rows, cols]}
    ok = True
    for fused in (1, 0):
        h.set_option("fused_amax", fused)
        codes, bs, gs, guide = h.rollout_quant(rg, seg)
        torch.cuda.synchronize()
        o_codes, o_bs, o_gs, o_guide = oracle.rollout_quant(synth.to_u16(r), seg)
        ok &= bool(np.array_equal(codes.cpu().numpy(), o_codes))
        ok &= bool(np.array_equal(guide.cpu().numpy().view(np.uint32), o_guide))
    h.set_option("fused_amax", 1)
    h.guide_pack(codes)
    h.guide_unpack(xg, guide, bs, gs, seg)
    for kind, gd in (("none", None), ("compact", guide), ("full", codes)):
        st = trace.new_stats(dev)
        args = (xg, seg, kind) + (() if kind == "none" else (gd, bs, gs, seg))
        y, m, c, _ = h.train_fakequant(*args, codes=True, stats=st)
        y2, m2, _, _ = h.train_fakequant(*args)
        torch.cuda.synchronize()
        okind = {"none": oracle.GUIDE_NONE, "compact": oracle.GUIDE_COMPACT, "full": oracle.GUIDE_FULL}[kind]
        oargs = (synth.to_u16(x), seg, okind) + (() if kind == "none" else (
            o_guide if kind == "compact" else o_codes, o_bs, o_gs, seg))
        oy, om, oc, _ = oracle.train_fakequant(*oargs)
        ok &= bool(np.array_equal(synth.to_u16(y), oy) and np.array_equal(synth.to_u16(y2), oy))
        ok &= bool(np.array_equal(c.cpu().numpy(), oc))
    h.ste_backward(xg, m)
    h.segment_amax(xg, seg)
    _, v = h.debug_bounds()
    res["violations"] = v
    res["bit_exact"] = ok
    out["cases"].append(res)
# non-finite inputs (unspecified results, but every access stays in range)
rows, cols = 300, 96
xn = rand((rows, cols), 5, 2.0).float()
xn[3, 5] = float("nan"); xn[7, 0] = float("inf"); xn[7, 1] = -float("inf")
xn[100:110, :] = float("nan"); xn[200, 17] = 3.0e38; xn[250, :32] = float("inf")
xn = xn.to(torch.bfloat16).to(dev)
segn = np.array([0, 150, 150, 300], np.int64)
for fused in (1, 0):
    h.set_option("fused_amax", fused)
    codes, bs, gs, guide = h.rollout_quant(xn, segn)
h.set_option("fused_amax", 1)
h.guide_pack(codes)
h.guide_unpack(xn, guide, bs, gs, segn)
for kind, gd in (("none", None), ("compact", guide), ("full", codes)):
    args = (xn, segn, kind) + (() if kind == "none" else (gd, bs, gs, segn))
    y, m, c, _ = h.train_fakequant(*args, codes=True, stats=trace.new_stats(dev))
    h.train_fakequant(*args)
h.ste_backward(xn, m)
h.segment_amax(xn, segn)
_, v = h.debug_bounds()
out["nonfinite_violations"] = v
out["nonfinite_status"] = h.device_status()
# outputs registered 16 bytes short: the kernels' last stores are counted and skipped
h.set_option("debug_shrink", 1)
rows, cols = 257, 64
x = rand((rows, cols), 99, 3.0).to(dev)
codes = torch.full((rows, cols // 2), 0xAB, dtype=torch.uint8, device=dev)
bs = torch.full((rows, cols // 16), 0xCD, dtype=torch.uint8, device=dev)
gs = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
guide = torch.full((rows, cols // 16), -1, dtype=torch.int32, device=dev)
h.rollout_quant(x, None, out=(codes, bs, gs, guide))
y = torch.full((rows, cols), 7.0, dtype=torch.bfloat16, device=dev)
mask = torch.full((rows, cols // 32), -1, dtype=torch.int32, device=dev)
h.train_fakequant(x, None, "none", out=(y, mask, None))
_, v = h.debug_bounds()
h.set_option("debug_shrink", 0)
tail = lambda t: t.reshape(-1).view(torch.uint8)[-16:].cpu().numpy().tolist()
out["shrink"] = {"violations": v, "codes_tail": tail(codes), "y_tail_bf16": tail(y),
                 "guide_tail": tail(guide)}
h.close()
print("RESULT " + json.dumps(out))
'''


def test_debug_build_counts_no_violation_and_detects_one(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    code = CHILD.replace("ROOT", repr(ROOT)).replace("OUT", repr(str(tmp_path / "dbg")))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    assert res["checked"] is True
    for case in res["cases"]:
        assert case["violations"] == 0, case
        assert case["bit_exact"], case
    assert res["nonfinite_violations"] == 0 and res["nonfinite_status"] == 0
    shrink = res["shrink"]
    assert shrink["violations"] > 0
    # the last 16 bytes of each output kept their fill pattern
    assert shrink["codes_tail"] == [0xAB] * 16
    assert shrink["guide_tail"] == [0xFF] * 16
    assert shrink["y_tail_bf16"] == [0xE0, 0x40] * 8    # bf16 7.0 = 0x40E0, little-endian
