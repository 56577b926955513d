"""The benchmark's multi-rank logic on CPU: world size 2 over gloo.

Ranks own disjoint, balanced shares of the independent (batch, kv-head)
units, exchange nothing on the data path, and agree on the maximum elapsed
time (the only collective besides the timing barrier).
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    r, w = bench.init_dist("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    mx = bench.max_over_ranks(10.0 + rank)
    lo, hi = bench.shard_units(64, r, w)
    out.put((rank, mx, lo, hi))
    dist.destroy_process_group()


def test_two_rank_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [m for _, m, _, _ in res] == [11.0, 11.0]
    assert [(lo, hi) for _, _, lo, hi in res] == [(0, 32), (32, 64)]


@pytest.mark.parametrize("n,world", [(64, 1), (64, 3), (8, 8), (5, 8), (1000, 7)])
def test_shard_units_partition(n, world):
    spans = [bench.shard_units(n, r, world) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    for (a, b), (c, _) in zip(spans, spans[1:]):
        assert b == c and a <= b
    sizes = [b - a for a, b in spans]
    assert max(sizes) - min(sizes) <= 1


def test_reference_arm_other_ranks_exit(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.parse_args(["--impl", "reference"])) == 0


def test_oracle_step_wraps_heads_within_batch_zero():
    # The reference arm samples batch 0 only; a step index past its heads
    # (long --steps runs) must wrap to another head of batch 0.
    import types
    import numpy as np
    rng = np.random.default_rng(5)
    w = types.SimpleNamespace(B=2, Hq=2, Hkv=1, N=64, d=16, scale=0.25, causal=True)
    t64 = {k: rng.standard_normal((1, w.Hq if k in ("Q", "dO") else w.Hkv, w.N, w.d)) for k in ("Q", "K", "V", "dO")}
    for head in (0, 1, 2, 5, 301):
        dt, fl = bench.oracle_step(w, t64, 64, head)
        assert dt >= 0 and fl == 3.5 * 4.0 * 64 * 64 * 16 / 2
