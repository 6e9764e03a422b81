"""Seeded synthetic workloads for the guided-NVFP4 path.

This module only draws input tensors; it holds none of the quantiser's
arithmetic.  The tests use it to feed both the CUDA library and the CPU
oracle, and the benchmark uses it to fill device memory.

The pages measure on routed-expert activations and KV caches of trained MoE
models, which are not available here.  These generators stand in for them
with the shapes and value structure described in the design notes:

  1  one tensor 256 x 2048, x = 2 * Student-t(4), drift sigma 2^-8
  2  routed-expert activations, 64 experts with Zipf(1.1) token counts
     summing to 32768 rows, hidden 2048, N(0,1) with 1% outlier channels
     scaled by 30, drift sigma 2^-8
  3  KV rows [32 layers][K,V][8192 tokens][8 heads][128], N(0,1) times a
     LogNormal(0, 0.5) scale per (layer, K/V, head), drift sigma 2^-7;
     one segment per (layer, K/V)
  4  routed-expert activations 262144 x 4096, 64 Zipf experts, 41 outlier
     channels, drift sigma 2^-6
  5  long-rollout KV stream [48][K,V][131072][4][128], N(0,1), drift sigma
     2^-8; training segments per (layer, K/V), rollout segments per
     (layer, K/V, 4096-token chunk)

The rollout tensor is r = bf16(x * (1 + eps)), eps ~ N(0, sigma^2), formed in
fp32 from the bf16 x.  Every tensor is drawn one training segment at a time
from a generator seeded by (config seed, segment index), so any segment can
be regenerated alone.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg: int
    rows: int
    cols: int
    seg_t: np.ndarray          # int64 [n_seg_t + 1] training segment rows
    seg_r: np.ndarray          # int64 [n_seg_r + 1] rollout segment rows
    sigma: float               # drift standard deviation
    seed: int = 0
    kind: str = "dense"        # "student", "moe", "kv"
    outliers: int = 0          # number of outlier channels (moe)
    kv_dims: Optional[tuple] = None   # (layers, tokens, heads, head_dim)
    head_lognormal: float = 0.0       # sigma of per-head LogNormal scale

    @property
    def elems(self) -> int:
        return self.rows * self.cols

    @property
    def n_seg_t(self) -> int:
        return len(self.seg_t) - 1

    @property
    def n_seg_r(self) -> int:
        return len(self.seg_r) - 1

    def describe(self) -> dict:
        d = {"workload": self.name, "rows": self.rows, "cols": self.cols,
             "elements": self.elems, "segments_train": self.n_seg_t,
             "segments_rollout": self.n_seg_r, "drift_sigma": self.sigma,
             "seed": self.seed}
        if self.kv_dims:
            d["kv_layout"] = "[layer][K,V][token][kv_head][head_dim]"
            d["layers"], d["tokens"], d["kv_heads"], d["head_dim"] = self.kv_dims
        return d


def zipf_counts(total: int, n: int, s: float = 1.1) -> np.ndarray:
    """Token counts n_i proportional to i^-s, largest-remainder rounded."""
    w = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    exact = w / w.sum() * total
    base = np.floor(exact).astype(np.int64)
    short = total - int(base.sum())
    order = np.argsort(-(exact - base), kind="stable")
    base[order[:short]] += 1
    return base


def _offsets(counts) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(counts, dtype=np.int64))]).astype(np.int64)


def workload(cfg: int, small: bool = False, seed: int = 0) -> Workload:
    """The five workloads; ``small`` shrinks rows so the oracle finishes in
    seconds while still spanning many tiles, segments and a ragged tail."""
    if cfg == 1:
        rows, cols = (256, 2048) if not small else (40, 2048)
        seg = _offsets([rows])
        return Workload("single tensor 256x2048 Student-t" if not small else
                        "single tensor 40x2048 Student-t", 1, rows, cols, seg, seg,
                        2.0 ** -8, seed, "student")
    if cfg in (2, 4):
        total, cols, out = ((32768, 2048, 20) if cfg == 2 else (262144, 4096, 41))
        sigma = 2.0 ** -8 if cfg == 2 else 2.0 ** -6
        if small:
            total = 3001 if cfg == 2 else 1537
        seg = _offsets(zipf_counts(total, 64))
        name = (f"moe routed-expert activations {total}x{cols}, 64 Zipf(1.1) experts, "
                f"{out} outlier channels x30")
        return Workload(name, cfg, total, cols, seg, seg, sigma, seed, "moe", outliers=out)
    if cfg == 3:
        layers, tokens, heads, hd = 32, 8192, 8, 128
        if small:
            tokens = 37
        rows = layers * 2 * tokens * heads
        seg = _offsets([tokens * heads] * (layers * 2))
        return Workload(f"fp4 kv rows [{layers}][K,V][{tokens}][{heads}][{hd}]", 3, rows, hd,
                        seg, seg, 2.0 ** -7, seed, "kv", kv_dims=(layers, tokens, heads, hd),
                        head_lognormal=0.5)
    if cfg == 5:
        layers, tokens, heads, hd, chunk = 48, 131072, 4, 128, 4096
        if small:
            layers, tokens, chunk = 3, 1000, 256   # last chunk ragged (232 tokens)
        rows = layers * 2 * tokens * heads
        seg_t = _offsets([tokens * heads] * (layers * 2))
        per = [min(chunk, tokens - c) * heads for c in range(0, tokens, chunk)]
        seg_r = _offsets(per * (layers * 2))
        return Workload(f"long-rollout kv stream [{layers}][K,V][{tokens}][{heads}][{hd}], "
                        f"{chunk}-token rollout chunks", 5, rows, hd, seg_t, seg_r,
                        2.0 ** -8, seed, "kv", kv_dims=(layers, tokens, heads, hd))
    raise ValueError(f"unknown workload {cfg}")


def _gen(work: Workload, salt: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((work.seed * 1_000_003 + work.cfg * 7919 + salt) & 0x7FFF_FFFF_FFFF)
    return g


def _outlier_channels(work: Workload) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(work.seed * 31 + work.cfg)
    return torch.randperm(work.cols, generator=g)[: work.outliers]


def _head_scales(work: Workload) -> torch.Tensor:
    layers, _, heads, _ = work.kv_dims
    g = torch.Generator(device="cpu")
    g.manual_seed(work.seed * 37 + work.cfg)
    z = torch.randn(layers * 2, heads, generator=g, dtype=torch.float64)
    return torch.exp(work.head_lognormal * z).to(torch.float32)


def segment_inputs(work: Workload, s: int, device="cpu"):
    """(x, r) bf16 tensors [rows_s, cols] for training segment ``s``."""
    r0, r1 = int(work.seg_t[s]), int(work.seg_t[s + 1])
    n = r1 - r0
    g = _gen(work, s, device)
    shape = (n, work.cols)
    if work.kind == "student":
        z = torch.randn(shape, generator=g, device=device)
        chi = torch.randn((4,) + shape, generator=g, device=device).square().sum(0)
        xf = 2.0 * z / torch.sqrt(chi / 4.0)
    elif work.kind == "moe":
        xf = torch.randn(shape, generator=g, device=device)
        ch = _outlier_channels(work).to(device)
        xf[:, ch] *= 30.0
    else:
        xf = torch.randn(shape, generator=g, device=device)
        if work.head_lognormal:
            _, tokens, heads, _ = work.kv_dims
            sc = _head_scales(work)[s].to(device)          # per head
            xf = (xf.view(tokens, heads, work.cols) * sc.view(1, heads, 1)).view(shape)
    x = xf.to(torch.bfloat16)
    eps = torch.randn(shape, generator=g, device=device) * work.sigma
    r = (x.float() * (1.0 + eps)).to(torch.bfloat16)
    return x, r


def make_inputs(work: Workload, device="cpu"):
    """Whole (x, r) bf16 tensors [rows, cols], drawn segment by segment."""
    x = torch.empty((work.rows, work.cols), dtype=torch.bfloat16, device=device)
    r = torch.empty_like(x)
    for s in range(work.n_seg_t):
        r0, r1 = int(work.seg_t[s]), int(work.seg_t[s + 1])
        if r1 > r0:
            xs, rs = segment_inputs(work, s, device)
            x[r0:r1].copy_(xs)
            r[r0:r1].copy_(rs)
    return x, r


def rollout_segments_within(work: Workload, s: int) -> np.ndarray:
    """Rollout segment offsets that fall inside training segment ``s``,
    rebased to the segment's first row (the rollout table refines the
    training table in every workload here)."""
    r0, r1 = int(work.seg_t[s]), int(work.seg_t[s + 1])
    inner = work.seg_r[(work.seg_r >= r0) & (work.seg_r <= r1)]
    return (inner - r0).astype(np.int64), int(np.searchsorted(work.seg_r, r0))


def to_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bytes_human(n: float) -> str:
    for u in ("B", "KiB", "MiB", "GiB"):
        if n < 1024 or u == "GiB":
            return f"{n:.1f} {u}"
        n /= 1024.0
    return f"{n:.1f} GiB"


__all__ = ["Workload", "workload", "segment_inputs", "make_inputs", "zipf_counts",
           "rollout_segments_within", "to_u16", "bytes_human"]

