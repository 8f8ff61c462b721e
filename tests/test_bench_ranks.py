"""bench.py's multi-rank reduction, run as two gloo ranks on the CPU.

Every rank runs its own replica of the workload (channels are independent, so
the path shards with no data-path collective); the timed region is the maximum
over ranks and the job's throughput is world x per-rank bytes / that time.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    import torch
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t, e = bench.max_over_ranks(times[rank], dist, torch, "cpu")
        v, ve = bench.aggregate_gbs(world, 1.0e9, t, e)
        out_q.put((rank, t, e, v, ve))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_without_a_process_group():
    import torch
    import bench
    assert bench.max_over_ranks([1.5, 2.0], None, torch, "cpu") == [1.5, 2.0]
    v, ve = bench.aggregate_gbs(1, 2.0e9, 1.0, 4.0)
    assert v == pytest.approx(2000.0) and ve == pytest.approx(500.0)


def test_two_gloo_ranks_take_the_slowest_rank():
    import torch.multiprocessing as mp
    world = 2
    times = [[0.5, 3.0], [0.8, 2.0]]   # per rank: (kernel ms/step, end-to-end ms/step)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, e, v, ve in got:
        assert t == pytest.approx(0.8) and e == pytest.approx(3.0)
        assert v == pytest.approx(2 * 1.0e9 / 0.8e-3 / 1e9)      # 2 ranks x 1 GB per step / 0.8 ms
        assert ve == pytest.approx(2 * 1.0e9 / 3.0e-3 / 1e9)


def test_lean_form_choice_names_the_kernel_of_each_layer(monkeypatch):
    """bench.py names the kernel a direct bf16 scan runs on (its restatement of the library's rule): the
    regular form where it already fits in the fewest waves, the lean form at the narrowest width of fewest
    waves otherwise, and the MAMBA_TM_LEAN override."""
    import bench
    monkeypatch.delenv("MAMBA_TM_LEAN", raising=False)
    sms = 148
    assert bench.lean_warps(8, 1536, 4, sms) == 0        # 130M layer: one wave of 11-warp CTAs already
    assert bench.lean_warps(4, 5120, 4, sms) == 18       # 2.8B layer: one wave of 18-warp CTAs, not two
    assert bench.lean_warps(4, 5120, 16, sms) == 18      # N = 64, 16 lanes per channel: 4 waves, not 7
    assert bench.lean_warps(1, 21000, 4, sms) == 18      # the GPU test's widest-CTA shape
    assert bench.lean_warps(1, 10600, 8, sms) == 18
    monkeypatch.setenv("MAMBA_TM_LEAN", "0")
    assert bench.lean_warps(4, 5120, 4, sms) == 0
    monkeypatch.setenv("MAMBA_TM_LEAN", "1")
    assert bench.lean_warps(2, 300, 4, sms) == 12        # forced: the narrowest width of fewest waves


def test_traffic_records_apply_only_to_their_kernel_and_sources():
    """A stored ncu DRAM traffic record is reported only for the kernel instantiation and the source hash
    it was taken on (a flag or convolution variant of the same workload reports none)."""
    import json
    import bench
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    r = rec["mamba130m_b8_d1536_n16_l2048_bf16"]
    got = bench.traffic_record("mamba130m_b8_d1536_n16_l2048_bf16", kernel=r["kernel"])
    if r["source_sha"] == bench.kernel_source_sha():
        assert got == r["dram_bytes_per_launch"] == r["dram_read_bytes"] + r["dram_write_bytes"]
    else:
        assert got is None
    assert bench.traffic_record("mamba130m_b8_d1536_n16_l2048_bf16", kernel=r["kernel"][:-1] + ",flags>") is None
    assert bench.traffic_record("no_such_workload") is None
