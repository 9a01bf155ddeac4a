"""The bench's multi-rank host logic on CPU: two gloo ranks, each timing a
different step, agree on the slowest rank's time and on the whole-job
throughput (independent replicas, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = [1.5, 2.25][rank]
    slow = bench.max_over_ranks(my_ms, world)
    gbs = bench.job_gbs(10 ** 9, slow, world)
    q.put((rank, slow, gbs))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
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
    for rank, slow, gbs in res:
        assert slow == 2.25
        assert gbs == pytest.approx(2 * 1e9 / 2.25e-3 / 1e9)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_gbs(2 * 10 ** 9, 1.0, 1) == pytest.approx(2000.0)


def test_algorithmic_bytes_of_the_step():
    import seeded_inputs as si
    b = [bench.alg_bytes(si.WORKLOADS[n]) for n in bench.STEP_WORKLOADS]
    # forward: read x, write y (bf16), gamma once, rstd per row
    assert b[0] == 16384 * 8192 * 4 + 8192 * 2 + 16384 * 4
    # fused add: read r and x, write h and y, gamma once
    assert b[1] == 32768 * 4096 * 8 + 4096 * 2
    # backward: read x and dy, write dx, read rstd, fp32 gamma and dgamma once
    assert b[2] == 16384 * 8192 * 6 + 16384 * 4 + 8192 * 4 + 8192 * 4


def test_traffic_record_applies_only_to_the_captured_sources_and_variants(tmp_path, monkeypatch):
    # a record taken on the current step-kernel sources and these variants
    import json
    os.makedirs(tmp_path / "profiles")
    variants = {"fwd": "fwd/cta/a", "fused_add": "fused_add/cta/b", "bwd": "bwd/staged/c"}
    rec = {"source_hash": bench.source_hash(), "variants": variants,
           "per_launch_bytes": {"fwd": 1, "fused_add": 2, "bwd": 3}}
    with open(tmp_path / "profiles" / "dram_traffic.json", "w") as f:
        json.dump(rec, f)
    real_hash = bench.source_hash()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda: real_hash)
    for op, n in (("fwd", 1), ("fused_add", 2), ("bwd", 3)):
        assert bench.ncu_traffic(op, variants[op]) == n
        # another variant picked by the dispatch: no traffic figure
        assert bench.ncu_traffic(op, variants[op] + "/other") is None
    # other kernel sources: no traffic figure for any op
    monkeypatch.setattr(bench, "source_hash", lambda: "0" * 16)
    for op in variants:
        assert bench.ncu_traffic(op, variants[op]) is None
    # no record at all
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "none"))
    assert bench.ncu_traffic("fwd", variants["fwd"]) is None


def test_threaded_oracle_step_covers_the_same_rows():
    # the all-cores baseline runs the same sample in row blocks: same bytes
    samples = bench._samples(1 / 4096)
    t1, b1 = bench._oracle_step(samples)
    t2, b2 = bench._oracle_step_threads(samples, 3)
    assert b1 == b2 > 0
