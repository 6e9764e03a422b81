"""Host-side logic without a GPU: the workload generators, the work division
across ranks, and the multi-rank timing reduction of bench.py under a real
two-rank gloo process group on the CPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from fp4_rollout_guided_gb300 import shard, synth


def test_zipf_counts():
    c = synth.zipf_counts(32768, 64)
    assert c.sum() == 32768 and len(c) == 64
    assert np.all(np.diff(c) <= 0)
    assert abs(int(c[0]) - 8208) <= 3 and abs(int(c[-1]) - 85) <= 2
    c4 = synth.zipf_counts(262144, 64)
    assert c4.sum() == 262144 and abs(int(c4[0]) - 65667) <= 5


def test_workload_shapes():
    w5 = synth.workload(5)
    assert w5.rows == 48 * 2 * 131072 * 4 and w5.cols == 128
    assert w5.n_seg_t == 96 and w5.n_seg_r == 96 * 32
    assert np.all(np.diff(w5.seg_r) == 16384)
    assert set(w5.seg_t.tolist()) <= set(w5.seg_r.tolist())      # rollout refines training
    w3 = synth.workload(3)
    assert w3.rows == 4194304 and w3.n_seg_t == 64
    w2 = synth.workload(2)
    assert w2.rows == 32768 and w2.cols == 2048 and w2.n_seg_t == 64
    w4 = synth.workload(4)
    assert w4.elems == 262144 * 4096
    for cfg in (1, 2, 3, 4, 5):
        s = synth.workload(cfg, small=True)
        assert s.seg_t[-1] == s.rows and s.seg_r[-1] == s.rows and s.cols % 32 == 0


def test_generators_are_seeded_and_segment_addressable():
    w = synth.workload(2, small=True)
    x1, r1 = synth.make_inputs(w, "cpu")
    x2, r2 = synth.make_inputs(w, "cpu")
    assert torch.equal(x1.view(torch.int16), x2.view(torch.int16))
    s = 7
    xs, rs = synth.segment_inputs(w, s, "cpu")
    a, b = int(w.seg_t[s]), int(w.seg_t[s + 1])
    assert torch.equal(xs.view(torch.int16), x1[a:b].view(torch.int16))
    assert torch.isfinite(x1.float()).all() and torch.isfinite(r1.float()).all()
    # drift is relative and small: r = bf16(x (1 + eps)), sigma 2^-8
    rel = ((r1.float() - x1.float()).abs() / x1.float().abs().clamp_min(1e-30))
    assert float(rel[x1.float().abs() > 1e-3].median()) < 0.01
    other = synth.workload(2, small=True, seed=1)
    x3, _ = synth.make_inputs(other, "cpu")
    assert not torch.equal(x1.view(torch.int16), x3.view(torch.int16))


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_strong_plan_covers_whole_segments(world):
    w = synth.workload(2)
    plans = [shard.strong_plan(w.seg_t, world, r) for r in range(world)]
    assert plans[0].seg_lo == 0 and plans[-1].seg_hi == w.n_seg_t
    for p, q in zip(plans, plans[1:]):
        assert p.seg_hi == q.seg_lo                      # contiguous, no overlap
    rows = [int(w.seg_t[p.seg_hi] - w.seg_t[p.seg_lo]) for p in plans]
    assert sum(rows) == w.rows


def test_weak_plan_seeds_are_distinct():
    seeds = {shard.weak_plan(4, r, 10).seed for r in range(4)}
    assert seeds == {10, 11, 12, 13}
    with pytest.raises(ValueError):
        shard.weak_plan(2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.workload(2)
        plan = shard.strong_plan(w.seg_t, world, rank)
        t = torch.tensor([plan.seg_lo, plan.seg_hi], dtype=torch.int64)
        got = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(got, t)
        ms = bench.max_over_ranks(dist, 1.5 + rank, torch.device("cpu"))
        bench.barrier(dist)
        out.put((rank, [g.tolist() for g in got], ms, shard.weak_plan(world, rank).seed))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_plan_and_timing():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    gathered = res[0][1]
    assert gathered == res[1][1]
    assert gathered[0][0] == 0 and gathered[0][1] == gathered[1][0] and gathered[1][1] == 64
    assert all(r[2] == 2.5 for r in res)            # max over ranks of 1.5 and 2.5
    assert {r[3] for r in res} == {0, 1}            # weak scaling: one seed per rank


def test_pipeline_pieces_cover_the_rows():
    from fp4_rollout_guided_gb300 import pipeline
    for cfg in (1, 2, 3, 4, 5):
        w = synth.workload(cfg)
        for min_rows in (1, 100000):
            ps = pipeline.plan_pieces(w.seg_t, w.seg_r, min_rows)
            assert ps[0].r0 == 0 and ps[-1].r1 == w.rows
            assert all(p.r1 == q.r0 and p.s1 == q.s0 for p, q in zip(ps, ps[1:]))
            assert ps[0].s0 == 0 and ps[-1].s1 == w.n_seg_r
            for p in ps:
                assert p.seg_r[0] == 0 and p.seg_r[-1] == p.r1 - p.r0
                assert p.seg_t[0] == 0 and p.seg_t[-1] == p.r1 - p.r0
                assert len(p.seg_r) == p.s1 - p.s0 + 1
    with pytest.raises(ValueError):
        pipeline.plan_pieces([0, 5, 10], [0, 4, 10])
