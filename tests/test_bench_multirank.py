"""Host logic of bench.py's multi-rank path on CPU (gloo, world size 2).

Each rank runs its own copy of the workload (the recurrence shards by sequence
with no exchange); the timed region ends in a barrier, the slowest rank's time
is taken and the throughput counts the units of all ranks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = 0.010 * (rank + 1)  # rank 1 is the slow one
    bench.barrier(world)
    m = bench.max_over_ranks(t, world, torch.device("cpu"))
    out[rank] = (m, bench.aggregate_throughput(16384, world, m))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        m, thr = res[rank]
        assert m == pytest.approx(0.020)
        assert thr == pytest.approx(16384 * 2 / 0.020)


def test_single_rank_defaults():
    assert bench.max_over_ranks(0.5, 1, torch.device("cpu")) == 0.5
    assert bench.aggregate_throughput(100, 1, 0.5) == 200


def test_algorithmic_counts_prefill():
    import gdn_inputs
    w = gdn_inputs.make_prefill(h_qk=16, h_v=32, d_k=128, d_v=128, batch=4, seqlen=64, g_shift=2.0)
    b, f = bench.prefill_algorithmic(w)
    T = 256
    per_tok = 2 * 16 * 128 * 2 + 32 * 128 * 2 + 2 * 32 * 4 + 32 * 128 * 2
    assert b == T * per_tok + 4 * 32 * 128 * 128 * 4
    assert f == pytest.approx(T * 32 * (6 * 128 * 128 + 2 * 64 * 384 + 4 * 64 * 128 / 2 + 2 * 64 * 64 / 3))


def test_traffic_summary_is_tied_to_kernel_sources(tmp_path, monkeypatch):
    f = tmp_path / "summary.txt"
    f.write_text(f"kernel_sha256: {bench.kernel_sha()}\ndram_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic() == 123.0
    f.write_text("kernel_sha256: 0000\ndram_bytes_per_launch: 123\n")
    assert bench.recorded_traffic() is None


def test_median_ci95_order_statistics():
    """The confidence interval of the median is the narrowest symmetric pair of
    order statistics that covers the median with probability >= 0.95 under
    the binomial law (n = 20: the 6th and 15th values, the textbook pair)."""
    import math
    r = bench.median_ci95(list(range(1, 21)))
    assert r["median"] == 10.5 and r["ci95"] == [6.0, 15.0] and r["n"] == 20
    for n in (5, 6, 10, 50, 101):
        xs = list(range(n))
        lo, hi = bench.median_ci95(xs)["ci95"]
        j, k = int(lo), int(hi)
        cover = sum(math.comb(n, i) for i in range(j + 1, k + 1)) / 2.0 ** n
        assert cover >= 0.95 or (j, k) == (0, n - 1)   # n < 6: the whole range is the widest there is
        if j + 1 <= n - 2 - j:  # one order statistic narrower on each side would not cover
            narrower = sum(math.comb(n, i) for i in range(j + 2, k)) / 2.0 ** n
            assert narrower < 0.95
    assert bench.median_ci95([3.0])["ci95"] == [3.0, 3.0]
