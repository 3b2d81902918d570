"""The N > 1 host path of the benchmark, as world-size-2 gloo ranks on the
CPU: packs are independent problems, so every rank runs its own replica
(weak scaling, no collective on the data path); the job's step time is the
slowest rank's, and the job's rate counts the units of every rank.  Also:
every rank plans the same pack identically, only rank 0 runs the CPU
reference arm, and when one pack is split across the ranks (pk_plan_shard)
the shares each rank computes on its own partition the pack's work."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    import packed_varlen_masked_gb300 as pk
    import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # slowest rank's time, seen by every rank
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        # whole-job rate over that time
        v = bench.job_throughput(world, 100.0, 4, t)
        # the replica plan is identical on every rank
        pack = W.mixed_resolution(requests=2)
        plan = pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=152,
                       upload=False)
        items, offs = plan.items()
        digest = torch.tensor([float(np.int64(items.astype(np.int64).sum() * 31 + offs.sum())),
                               plan.useful_flops])
        gathered = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(gathered, digest.double())
        # the CPU reference arm works on rank 0 only
        class A:
            steps, warmup = 1, 3
        buf = io.StringIO()
        if rank != 0:
            with redirect_stdout(buf):
                r = bench.reference_arm(A, pack, rank, world)
            assert r is None and buf.getvalue() == ""
        np.save(os.path.join(out_dir, f"r{rank}.npy"),
                np.array([t, v] + [float(x) for g in gathered for x in g]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_whole_job_rate(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
        assert p.exitcode == 0, p.exitcode
    res = [np.load(tmp_path / f"r{r}.npy") for r in range(world)]
    for r in res:
        assert r[0] == 15.0                      # max over ranks
        assert r[1] == pytest.approx(2 * 100.0 * 4 / 0.015)
        assert r[2] == r[4] and r[3] == r[5]     # identical plans on both ranks
    assert (res[0] == res[1]).all()


def test_single_process_reduces_to_local_values():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_throughput(1, 10.0, 2, 1000.0) == 20.0


def test_peaks_file_is_read_with_burst_sustained_and_copy_figures(tmp_path):
    sys.path.insert(0, ROOT)
    import json
    import bench
    f = tmp_path / "peaks.json"
    f.write_text(json.dumps({"gpu": "GB300", "hbm_gbs": 6692.8, "bf16_tflops": 1878.4,
                             "bf16_tflops_sustained": 1724.6, "clocks": {"sm_mhz": 1477}}))
    p = bench.load_peaks(str(f))
    assert p == {"bf16_tflops": 1878.4, "hbm_gbs": 6692.8, "bf16_tflops_sustained": 1724.6,
                 "source": "measured"}
    assert bench.load_peaks(str(tmp_path / "missing.json"))["source"] == "fallback"


def _shard_rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import packed_varlen_masked_gb300 as pk
    import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        pack = W.mixed_resolution()
        full = pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=152,
                       upload=False)
        mine = full.shard(rank, world, num_ctas=152, upload=False)  # computed on this rank alone
        items, _ = mine.items()
        n = torch.tensor([len(items)], dtype=torch.int64)
        counts = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(counts, n)
        width = int(max(c.item() for c in counts))
        padded = torch.full((width, 8), -9, dtype=torch.int64)
        padded[:len(items)] = torch.as_tensor(items.astype(np.int64))
        gathered = [torch.zeros(width, 8, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(gathered, padded)
        flops = torch.tensor([mine.useful_flops], dtype=torch.float64)
        dist.all_reduce(flops)
        if rank == 0:
            f_items, _ = full.items()
            got = np.concatenate([g[:int(c.item())].numpy() for g, c in zip(gathered, counts)])
            np.save(os.path.join(out_dir, "shard_items.npy"), got)
            np.save(os.path.join(out_dir, "full_items.npy"), f_items.astype(np.int64))
            np.save(os.path.join(out_dir, "flops.npy"), np.array([float(flops.item()),
                                                                   full.useful_flops]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_one_pack_into_a_partition(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_shard_rank_main, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
        assert p.exitcode == 0, p.exitcode
    got = np.load(tmp_path / "shard_items.npy")
    full = np.load(tmp_path / "full_items.npy")
    assert sorted(map(tuple, got.tolist())) == sorted(map(tuple, full.tolist()))
    fl = np.load(tmp_path / "flops.npy")
    assert fl[0] == pytest.approx(fl[1], rel=1e-12)


def test_multi_gpu_runs_build_plans_for_the_one_cta_kernel():
    """TMA multicast stays in single-GPU runs: with more than one rank the
    bench takes every plan off the head-pair clusters."""
    import bench
    import packed_varlen_masked_gb300 as pk
    import workloads as W
    pack = W.cfg_pair()
    saved = bench.SINGLE_GPU
    try:
        for single, expect in ((True, True), (False, False)):
            bench.SINGLE_GPU = single
            plan = bench.cta_plan(pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                                          pack.d, num_ctas=152, upload=False))
            assert plan.kv_share == expect
            assert plan.share_schedule()[0].shape[0] > 0  # the schedule stays
    finally:
        bench.SINGLE_GPU = saved
