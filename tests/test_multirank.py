"""The multi-GPU benchmark path, run as two gloo ranks on the CPU.

(b, h) heads are independent, so ranks shard by batch with no data-path
collective: each rank draws its own inputs (seed = rank), the step time is
the maximum over ranks and throughput counts the tokens of every rank. The
reference arm runs on rank 0 only.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench
    from linear_rnn_state_gb300 import inputs

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        ms = bench.reduce_max(local_ms, dist)
        value = bench.aggregate_tokens_per_s(world, 4, 4096, ms)
        d = inputs.generate(1, 8, 2, 16, "f32", seed=bench.shard_seed(rank))
        q.put((rank, ms, value, float(d["r"].sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    import multiprocessing as mp

    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    (_, ms0, v0, s0), (_, ms1, v1, s1) = res
    assert ms0 == ms1 == 15.0
    assert v0 == v1 == pytest.approx(2 * 4 * 4096 / 15e-3)
    assert s0 != s1  # each rank scans its own batch


def _shard_worker(rank, world, port, q):
    """Each rank runs the oracle's forward and backward on its own (b, h)
    heads of one shared batch; rank 0 gathers the pieces."""
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from linear_rnn_state_gb300 import inputs

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, T, H, N = 3, 40, 3, 16
        d = inputs.generate(B, T, H, N, "f32", 0.1, seed=5)  # one batch, the same on every rank
        mine = bench.head_shard(B, H, rank, world)
        o = {n: d[n].astype(np.float64) for n in ("r", "w", "k", "v", "a", "b", "dy")}
        y, sf, g = oracle.backward_heads(*(o[n] for n in ("r", "w", "k", "v", "a", "b", "dy")),
                                         d["s_init"].astype(np.float64), mine, nthreads=1)
        piece = {"heads": mine, "y": y, "s_final": sf, **g}
        pieces = [None] * world
        dist.all_gather_object(pieces, piece)
        if rank == 0:
            q.put(pieces)
    finally:
        dist.destroy_process_group()


def test_head_shards_concatenate_to_the_whole_batch_bit_for_bit():
    """Splitting one batch by (b, h) heads across two gloo ranks: the pieces
    cover every head once and, put together, equal the whole-batch oracle run
    bit for bit, so the split needs no exchange between ranks."""
    import multiprocessing as mp
    import socket

    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from linear_rnn_state_gb300 import inputs

    oracle.build()
    inputs.build()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    pieces = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    B, T, H, N = 3, 40, 3, 16
    heads = [hd for pc in pieces for hd in pc["heads"]]
    assert sorted(heads) == [(b, h) for b in range(B) for h in range(H)]
    assert len(pieces[0]["heads"]) and len(pieces[1]["heads"])
    d = inputs.generate(B, T, H, N, "f32", 0.1, seed=5)
    o = {n: d[n].astype(np.float64) for n in ("r", "w", "k", "v", "a", "b", "dy")}
    s0 = d["s_init"].astype(np.float64)
    y, sf = oracle.forward(*(o[n] for n in ("r", "w", "k", "v", "a", "b")), s0, nthreads=1)
    g = oracle.backward(*(o[n] for n in ("r", "w", "k", "v", "a", "b", "dy")), s0, nthreads=1)
    for pc in pieces:
        for p, (bi, hi) in enumerate(pc["heads"]):
            assert np.array_equal(pc["y"][p], y[bi, :, hi])
            assert np.array_equal(pc["s_final"][p], sf[bi, hi])
            assert np.array_equal(pc["dS_init"][p], g["dS_init"][bi, hi])
            for n in ("dr", "dw", "dk", "dv", "da", "db"):
                assert np.array_equal(pc[n][p], g[n][bi, :, hi]), (n, bi, hi)


def test_head_shard_is_a_partition():
    sys.path.insert(0, ROOT)
    import bench

    for B, H, world in ((4, 32, 8), (1, 40, 3), (3, 3, 2), (1, 1, 4)):
        got = [hd for r in range(world) for hd in bench.head_shard(B, H, r, world)]
        assert got == [(b, h) for b in range(B) for h in range(H)]


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0
    assert out.stdout.strip() == ""


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.aggregate_tokens_per_s(1, 4, 4096, 2.0) == pytest.approx(4 * 4096 / 2e-3)
    assert np.isfinite(bench.aggregate_tokens_per_s(8, 4, 4096, 1.0))


def _rwkv8_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench
    from tests.test_rwkv8_oracle import load_oracle
    from linear_rnn_state_gb300 import inputs

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        orc = load_oracle()
        shards = [inputs.generate_rwkv8(1, 12, 2, 2, 4, 3, "f64", seed=bench.shard_seed(r)) for r in range(world)]
        mine = shards[rank]
        # the decay is one parameter: every rank draws the same one (seed 0's)
        decay = shards[0]["decay"]
        g = orc.backward(mine["q"], mine["v"], decay, mine["dy"])
        t = torch.from_numpy(g["ddecay"].copy())
        bench.allreduce_param_grad(t, dist)
        full = {k: np.concatenate([sh[k] for sh in shards], axis=0) for k in ("q", "v", "dy")}
        ref = orc.backward(full["q"], full["v"], decay, full["dy"])["ddecay"]
        q.put((rank, float(np.abs(t.numpy() - ref).max()), float(np.abs(ref).max())))
    finally:
        dist.destroy_process_group()


def test_rwkv8_decay_gradient_is_summed_over_batch_shards():
    """Ranks that shard the batch add their ddecay; the sum equals the
    gradient of the whole batch (ddecay is additive over batch rows)."""
    import multiprocessing as mp
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rwkv8_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for _ in range(2):
        rank, err, scale = q.get(timeout=10)
        assert err <= 1e-12 * (1 + scale), (rank, err)
