"""CPU oracle for the guided-NVFP4 hot path of TRACE (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``trace_oracle.c`` (plain,
single-threaded binary32 C) through ctypes and shares nothing with the CUDA
library in ``fp4_rollout_guided_gb300``.

Arrays follow the oracle's C header: bf16 tensors are ``uint16`` bit
patterns of shape ``[rows, cols]``; segment tables are ``int64`` row offsets
with ``n_seg + 1`` entries, or ``None`` for a single segment.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "trace_oracle.c")
_HDR = os.path.join(_HERE, "trace_oracle.h")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

GUIDE_NONE, GUIDE_FULL, GUIDE_COMPACT = 0, 1, 2
STAT_N, STAT_MISMATCH_RTN, STAT_MISMATCH_GUIDED = 0, 1, 2
STAT_HIST_RTN, STAT_HIST_GUIDED, STAT_COUNT = 3, 7, 11

# -ffp-contract=off: no fused multiply-add, so every binary32 operation
# rounds on its own exactly as written.  No fast-math of any kind.
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-fno-unsafe-math-optimizations", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc if the shared object is missing or stale."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(_HDR)))
    if force or stale:
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64, I32, F32, INT = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_int
        sig = {
            "orc_bf16_to_f32": (F32, [ctypes.c_uint16]),
            "orc_f32_to_bf16": (ctypes.c_uint16, [F32]),
            "orc_e4m3_encode": (ctypes.c_uint8, [F32]),
            "orc_e4m3_decode": (F32, [ctypes.c_uint8]),
            "orc_e2m1_value": (F32, [INT]),
            "orc_e2m1_rtn": (INT, [F32]),
            "orc_e2m1_bracket": (None, [F32, P, P]),
            "orc_global_scale": (F32, [F32]),
            "orc_block_scale": (ctypes.c_uint8, [F32, F32]),
            "orc_scale_pair": (None, [ctypes.c_uint8, F32, P, P]),
            "orc_unpack_index": (INT, [F32, INT]),
            "orc_guided_index": (INT, [F32, F32, F32, INT, INT, F32]),
            "orc_e2m1_rtn_array": (None, [P, I64, P]),
            "orc_e2m1_bracket_array": (None, [P, I64, P, P]),
            "orc_e4m3_encode_array": (None, [P, I64, P]),
            "orc_f32_to_bf16_array": (None, [P, I64, P]),
            "orc_segment_amax": (INT, [P, I64, I64, P, I32, P]),
            "orc_rollout_quant": (INT, [P, I64, I64, P, I32, P, P, P, P]),
            "orc_rollout_quant_given": (INT, [P, I64, I64, P, I32, P, P, P, P, P]),
            "orc_train_fakequant_given": (INT, [P, I64, I64, P, I32, P, INT, P, P, P, P,
                                                I32, P, P, P, P]),
            "orc_guide_pack": (INT, [P, I64, I64, P]),
            "orc_ste_backward": (INT, [P, P, I64, I64, P]),
            "orc_guide_unpack": (INT, [P, P, P, P, P, I32, I64, I64, P]),
            "orc_train_fakequant": (INT, [P, I64, I64, P, I32, INT, P, P, P, P,
                                          I32, P, P, P, P]),
            "orc_mma_scales_bytes": (I64, [I64, I64]),
            "orc_mma_scales": (INT, [P, I64, I64, P]),
            "orc_nvfp4_gemm": (INT, [P, P, F32, P, P, F32, I64, I64, I64, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def threads() -> int:
    """Host threads the segment-parallel helpers use: every core."""
    return max(1, os.cpu_count() or 1)


def parallel_map(fn, items, n_threads=None):
    """``[fn(item) for item in items]`` on a pool of host threads.

    The oracle's C functions are single-threaded and independent per call;
    ctypes releases the interpreter lock while one runs, so calls on
    disjoint segments proceed on all cores at once.  Results keep the
    order of ``items``."""
    from concurrent.futures import ThreadPoolExecutor
    items = list(items)
    n = min(n_threads or threads(), max(1, len(items)))
    if n == 1:
        return [fn(it) for it in items]
    with ThreadPoolExecutor(n) as ex:
        return list(ex.map(fn, items))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(x):
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        x = x.view(np.uint16)
    return x


def _seg(seg, rows):
    """(array or None, n_seg) for the C calls."""
    if seg is None:
        return None, 1
    s = np.ascontiguousarray(np.asarray(seg, dtype=np.int64))
    return s, len(s) - 1


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: bad arguments")


# ---- scalar and array forms of the number formats ------------------------

def bf16_to_f32(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(v):
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.empty(v.shape, dtype=np.uint16)
    _load().orc_f32_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode(v):
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.empty(v.shape, dtype=np.uint8)
    _load().orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(c):
    lib = _load()
    c = np.asarray(c, dtype=np.uint8)
    return np.array([lib.orc_e4m3_decode(int(b)) for b in c.ravel()],
                    dtype=np.float32).reshape(c.shape)


def e2m1_value(m):
    return _load().orc_e2m1_value(int(m))


def e2m1_rtn(t):
    t = np.ascontiguousarray(np.asarray(t, dtype=np.float32))
    out = np.empty(t.shape, dtype=np.uint8)
    _load().orc_e2m1_rtn_array(_ptr(t), t.size, _ptr(out))
    return out


def e2m1_bracket(t):
    t = np.ascontiguousarray(np.asarray(t, dtype=np.float32))
    lo = np.empty(t.shape, dtype=np.uint8)
    hi = np.empty(t.shape, dtype=np.uint8)
    _load().orc_e2m1_bracket_array(_ptr(t), t.size, _ptr(lo), _ptr(hi))
    return lo, hi


def global_scale(amax):
    return _load().orc_global_scale(float(amax))


def block_scale(bamax, gs):
    return _load().orc_block_scale(float(bamax), float(gs))


def scale_pair(bs, gs):
    S, inv = ctypes.c_float(), ctypes.c_float()
    _load().orc_scale_pair(int(bs), float(gs), ctypes.byref(S), ctypes.byref(inv))
    return S.value, inv.value


def unpack_index(t_ref, lsb):
    return _load().orc_unpack_index(float(t_ref), int(lsb))


def guided_index(x, S_t, inv_t, have_guide, nib_r, S_r):
    return _load().orc_guided_index(float(x), float(S_t), float(inv_t),
                                    int(have_guide), int(nib_r), float(S_r))


# ---- whole-tensor steps ---------------------------------------------------

def segment_amax(x, seg=None):
    x = _u16(x)
    rows, cols = x.shape
    s, n = _seg(seg, rows)
    out = np.zeros(n, dtype=np.float32)
    _check(_load().orc_segment_amax(_ptr(x), rows, cols, _ptr(s), n, _ptr(out)), "amax")
    return out


def rollout_quant(x, seg=None, want_guide=True, amax=None):
    """-> codes uint8[rows, cols/2], bs uint8[rows, cols/16], gs float32[n_seg],
    guide uint32[rows, cols/16] (or None).  ``amax`` (float32[n_seg]) replaces
    the segment maxima of the rows given (for sampled checks)."""
    x = _u16(x)
    rows, cols = x.shape
    s, n = _seg(seg, rows)
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    bs = np.zeros((rows, cols // 16), dtype=np.uint8)
    gs = np.zeros(n, dtype=np.float32)
    guide = np.zeros((rows, cols // 16), dtype=np.uint32) if want_guide else None
    am = None if amax is None else np.ascontiguousarray(amax, dtype=np.float32)
    _check(_load().orc_rollout_quant_given(_ptr(x), rows, cols, _ptr(s), n, _ptr(am),
                                           _ptr(codes), _ptr(bs), _ptr(gs), _ptr(guide)),
           "rollout_quant")
    return codes, bs, gs, guide


def guide_pack(codes):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    rows, half = codes.shape
    cols = half * 2
    guide = np.zeros((rows, cols // 16), dtype=np.uint32)
    _check(_load().orc_guide_pack(_ptr(codes), rows, cols, _ptr(guide)), "guide_pack")
    return guide


def guide_unpack(x_ref, guide, bs_r, gs_r, seg_r=None):
    x_ref = _u16(x_ref)
    rows, cols = x_ref.shape
    s, n = _seg(seg_r, rows)
    guide = np.ascontiguousarray(guide, dtype=np.uint32)
    bs_r = np.ascontiguousarray(bs_r, dtype=np.uint8)
    gs_r = np.ascontiguousarray(gs_r, dtype=np.float32)
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    _check(_load().orc_guide_unpack(_ptr(x_ref), _ptr(guide), _ptr(bs_r), _ptr(gs_r),
                                    _ptr(s), n, rows, cols, _ptr(codes)), "guide_unpack")
    return codes


def train_fakequant(x, seg_t=None, kind=GUIDE_NONE, guide=None, bs_r=None,
                    gs_r=None, seg_r=None, want_codes=True, want_stats=True,
                    want_mask=True, amax_t=None):
    """-> y uint16[rows, cols] (bf16 bits), mask uint32[rows, cols/32],
    codes_t uint8[rows, cols/2] (or None), stats uint64[11] (or None)."""
    x = _u16(x)
    rows, cols = x.shape
    st, nt = _seg(seg_t, rows)
    sr, nr = _seg(seg_r, rows)
    if guide is not None:
        guide = np.ascontiguousarray(guide)
    if bs_r is not None:
        bs_r = np.ascontiguousarray(bs_r, dtype=np.uint8)
    if gs_r is not None:
        gs_r = np.ascontiguousarray(gs_r, dtype=np.float32)
    y = np.zeros((rows, cols), dtype=np.uint16)
    mask = np.zeros((rows, cols // 32), dtype=np.uint32) if want_mask else None
    codes_t = np.zeros((rows, cols // 2), dtype=np.uint8) if want_codes else None
    stats = np.zeros(STAT_COUNT, dtype=np.uint64) if want_stats else None
    am = None if amax_t is None else np.ascontiguousarray(amax_t, dtype=np.float32)
    rc = _load().orc_train_fakequant_given(_ptr(x), rows, cols, _ptr(st), nt, _ptr(am),
                                           int(kind), _ptr(guide), _ptr(bs_r), _ptr(gs_r),
                                           _ptr(sr), nr, _ptr(y), _ptr(mask), _ptr(codes_t),
                                           _ptr(stats))
    _check(rc, "train_fakequant")
    return y, mask, codes_t, stats


def ste_backward(g, mask):
    """-> uint16[rows, cols]: g where the mask bit is 1, +0 elsewhere."""
    g = _u16(g)
    rows, cols = g.shape
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    out = np.zeros((rows, cols), dtype=np.uint16)
    _check(_load().orc_ste_backward(_ptr(g), _ptr(mask), rows, cols, _ptr(out)), "ste_backward")
    return out


def mma_scales(bs, rows, cols):
    """Row-major block scales uint8[rows, cols/16] -> the tensor-core tiled
    layout (uint8, zero-padded to 128-row x 4-column tiles)."""
    bs = np.ascontiguousarray(bs, dtype=np.uint8).reshape(rows, cols // 16)
    n = _load().orc_mma_scales_bytes(rows, cols)
    if n < 0:
        raise ValueError("mma_scales: bad shape")
    out = np.zeros(n, dtype=np.uint8)
    _check(_load().orc_mma_scales(_ptr(bs), rows, cols, _ptr(out)), "mma_scales")
    return out


def nvfp4_gemm(a_codes, a_bs, a_gs, b_codes, b_bs, b_gs):
    """d[m, n] = fl32(a_gs * b_gs) * sum_k A[i, k] B[j, k] in float64."""
    a_codes = np.ascontiguousarray(a_codes, dtype=np.uint8)
    b_codes = np.ascontiguousarray(b_codes, dtype=np.uint8)
    m, k = a_codes.shape[0], a_codes.shape[1] * 2
    n = b_codes.shape[0]
    a_bs = np.ascontiguousarray(a_bs, dtype=np.uint8)
    b_bs = np.ascontiguousarray(b_bs, dtype=np.uint8)
    d = np.zeros((m, n), dtype=np.float64)
    _check(_load().orc_nvfp4_gemm(_ptr(a_codes), _ptr(a_bs), float(a_gs), _ptr(b_codes),
                                  _ptr(b_bs), float(b_gs), m, n, k, _ptr(d)), "nvfp4_gemm")
    return d
