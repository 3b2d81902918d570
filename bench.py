"""Benchmark: packed mixed-mask attention, useful TFLOP/s on one GB300.

One step = one pk_attn_fwd over the whole pack (all heads, all sequences)
with inputs already resident in HBM: its two kernels, the conversion of the
values to fp16 and the attention, timed apart through the two calls that make
it up.  The plan is built once, outside the timed region (it is reused by
every layer and denoising step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  ``--impl reference`` times the fp64 CPU
oracle (the only reference that exists for this path) on a bounded row
sample of the same workload.  Under torchrun each rank runs its own replica
of the pack (independent packs: weak scaling, no collective on the data
path); the timed region is bracketed by barriers and the max over ranks is
reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "packed mixed-mask attention useful TFLOP/s & tokens/s; % of bf16 dense peak"
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
# The attention kernel's sources and the planner whose schedule sets its
# DRAM traffic: the committed traffic figure is valid only for these bytes.
KERNEL_SOURCES = ["packed_varlen_masked_gb300/csrc/pk_attn.cu",
                  "packed_varlen_masked_gb300/csrc/tmem_ops.cuh",
                  "packed_varlen_masked_gb300/csrc/sync.cuh",
                  "packed_varlen_masked_gb300/csrc/attn_common.cuh",
                  "packed_varlen_masked_gb300/csrc/pk_plan.cpp",
                  "packed_varlen_masked_gb300/csrc/pk_internal.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "pk_attn_fwd_d128_mixed_resolution_traffic.md")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _flatten(d, prefix=""):
    for k, v in d.items():
        key = f"{prefix}.{k}" if prefix else str(k)
        if isinstance(v, dict):
            yield from _flatten(v, key)
        elif isinstance(v, (int, float)) and not isinstance(v, bool):
            yield key.lower(), float(v)


def load_peaks(path=None):
    """Roofline denominators: the measured copy bandwidth and bf16 GEMM rate
    in MEASURED_PEAKS.json (burst and sustained), else the fallback."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                flat = dict(_flatten(json.load(f)))
            burst = [v for k, v in flat.items() if "bf16" in k and "tflop" in k
                     and "sustain" not in k]
            sus = [v for k, v in flat.items() if "bf16" in k and "tflop" in k and "sustain" in k]
            hbm = [v for k, v in flat.items() if ("hbm" in k or "copy" in k) and "gb" in k]
            if burst and hbm:
                return {"bf16_tflops": burst[0], "hbm_gbs": hbm[0],
                        "bf16_tflops_sustained": sus[0] if sus else None, "source": "measured"}
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0, source="fallback")


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, valid only while
    the kernel source is unchanged since the capture."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    text = open(TRAFFIC_FILE).read()
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != kernel_source_sha():
        return None
    return float(m_b.group(1))


# TMA multicast (the head-pair clusters' shared key/value copies) runs only in
# single-GPU runs: on more than one GPU every plan here takes the one-CTA
# kernel.
SINGLE_GPU = True


def cta_plan(plan):
    """The plan as this run may launch it (see SINGLE_GPU)."""
    if not SINGLE_GPU and plan.kv_share:
        plan.set_kv_share(False)
    return plan


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            # nvidia-smi takes a moment to start: let its first sample arrive
            # so that the samples cover the whole timed region
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.02)
            self.lines.clear()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and "WORLD_SIZE" in os.environ:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    return world, rank, local


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time: every rank's timed region is bracketed by
    barriers, so the job's step time is the maximum."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: float, steps: int, total_ms: float) -> float:
    """Whole-job rate: the units every rank processed over the max time."""
    return world * units_per_rank * steps / (total_ms * 1e-3)


def workload_config(pack, world: int, useful_flops: float, split: bool = False) -> dict:
    """The bench line's config, identical for both arms: the workload, its
    per-step useful FLOPs (each arm counts them its own way: the planner
    here, the oracle's visible keys in the reference arm) and the L2 rule."""
    T = pack.total_tokens
    q_mb = T * pack.hq * pack.d * 2 / 1e6
    kv_mb = 2 * T * pack.hkv * pack.d * 2 / 1e6
    return dict(pack.describe(), parallelism=f"split{world}" if split else f"replicas{world}",
                l2="inputs larger than L2 (q %.0f MB, k+v %.0f MB)" % (q_mb, kv_mb),
                useful_flops_per_step=float(useful_flops),
                padded_dense_mask_flops_per_step=4.0 * pack.d * pack.hq * len(pack.seqs)
                * pack.max_seqlen ** 2)


def reference_arm(args, pack, rank, world):
    """fp64 CPU oracle, as it stands, on bounded row samples of the pack."""
    if rank != 0:
        return
    import oracle
    import torch
    q, k, v = W.make_qkv(pack)
    cu = pack.cu_seqlens
    keys = oracle.row_keys(cu, pack.segments).astype(np.float64)  # FLOP count per row
    rng = np.random.default_rng(0)
    # calibrate: rows per ~2 s step
    probe = rng.integers(0, pack.total_tokens, size=32).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, cu, pack.segments, pack.hq, pack.hkv, pack.d, pack.scale, rows=probe)
    dt = time.perf_counter() - t0
    n_rows = int(max(16, min(4096, 32 * 2.0 / max(dt, 1e-6))))
    times, flops = [], []
    for step in range(args.warmup + args.steps):
        rows = rng.integers(0, pack.total_tokens, size=n_rows).astype(np.int32)
        t0 = time.perf_counter()
        oracle.attention(q, k, v, cu, pack.segments, pack.hq, pack.hkv, pack.d, pack.scale, rows=rows)
        t = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(t)
            flops.append(4.0 * pack.d * pack.hq * keys[rows].sum())
    total_t = sum(times)
    tflops = sum(flops) / total_t / 1e12
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_t / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(pack, world, 4.0 * pack.d * pack.hq * keys.sum()),
        "tokens_per_s": (n_rows * len(times)) / total_t,
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_rows} uniformly drawn query rows (all {pack.hq} heads) per step"},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def _oracle_rate(pack, seconds: float, seed: int = 1):
    """Useful TFLOP/s of the oracle on uniformly drawn rows of ``pack``,
    about ``seconds`` of CPU work; returns (TFLOP/s, seconds, rows)."""
    import oracle
    q, k, v = W.make_qkv(pack)
    cu = pack.cu_seqlens
    keys = oracle.row_keys(cu, pack.segments).astype(np.float64)  # FLOP count per row
    rng = np.random.default_rng(seed)
    probe = rng.integers(0, pack.total_tokens, size=16).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, cu, pack.segments, pack.hq, pack.hkv, pack.d, pack.scale, rows=probe)
    dt = time.perf_counter() - t0
    n_rows = int(max(16, min(20000, 16 * seconds / max(dt, 1e-6))))
    rows = rng.integers(0, pack.total_tokens, size=n_rows).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, cu, pack.segments, pack.hq, pack.hkv, pack.d, pack.scale, rows=rows)
    t = time.perf_counter() - t0
    return 4.0 * pack.d * pack.hq * keys[rows].sum() / t / 1e12, t, n_rows


def cpu_baseline(pack, seconds: float = 10.0, per_config_seconds: float = 1.5):
    """The oracle as it stands, on a bounded sample of the same workload, and
    on a short sample of every other configuration."""
    import oracle
    value, t, n_rows = _oracle_rate(pack, seconds)
    per = {}
    for name, fn in W.CONFIGS.items():
        rate, tc, nc = _oracle_rate(fn(), per_config_seconds)
        per[name] = {"tflops": rate, "rows": nc, "seconds": round(tc, 2)}
    return {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": t,
            "sample": f"{n_rows} uniformly drawn query rows x {pack.hq} heads of the workload",
            "per_config": per}


def replaced_path(torch, pack, q, k, v, ours_out, steps=3):
    """Time the path the pages replace: every sequence padded to the longest
    one, an explicit (bsz, 1, L, L) bool mask, torch SDPA.  Measurement
    only: its output is compared with ours on valid rows, never used."""
    import torch.nn.functional as F
    cu = pack.cu_seqlens
    S, L = len(pack.seqs), pack.max_seqlen
    dev = q.device
    group = pack.hq // pack.hkv
    qp = torch.zeros(S, pack.hq, L, pack.d, dtype=q.dtype, device=dev)
    kp = torch.zeros(S, pack.hq, L, pack.d, dtype=q.dtype, device=dev)  # KV heads repeated
    vp = torch.zeros_like(kp)
    mask = torch.zeros(S, 1, L, L, dtype=torch.bool, device=dev)
    for s_idx, seq in enumerate(pack.seqs):
        b, e = int(cu[s_idx]), int(cu[s_idx + 1])
        n = e - b
        qp[s_idx, :, :n] = q[b:e].transpose(0, 1)
        kp[s_idx, :, :n] = k[b:e].repeat_interleave(group, dim=1).transpose(0, 1)
        vp[s_idx, :, :n] = v[b:e].repeat_interleave(group, dim=1).transpose(0, 1)
        # the model's mask: causal, plus each image segment sees itself
        pos = torch.arange(L, device=dev)
        m = pos[None, :] <= pos[:, None]
        start = 0
        for typ, ln in seq:
            if typ == W.IMAGE:
                m[start:start + ln, start:start + ln] = True
            start += ln
        m[n:, :] = False
        m[:, n:] = False
        m[torch.arange(n, L, device=dev), torch.arange(n, L, device=dev)] = True  # padded rows: no NaN
        mask[s_idx, 0] = m
    from torch.nn.attention import SDPBackend, sdpa_kernel

    def run():
        # the memory-efficient kernel takes an arbitrary mask; never the
        # math fallback, which would materialise every score
        with sdpa_kernel([SDPBackend.EFFICIENT_ATTENTION]):
            return F.scaled_dot_product_attention(qp, kp, vp, attn_mask=mask, scale=pack.scale)
    try:
        o = run()
    except RuntimeError as exc:
        del qp, kp, vp, mask
        torch.cuda.empty_cache()
        return {"impl": "torch SDPA (memory-efficient backend), padded", "unavailable": str(exc)[:200]}
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        o = run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # agreement with our output on the valid rows
    err = 0.0
    for s_idx in range(S):
        b, e = int(cu[s_idx]), int(cu[s_idx + 1])
        err = max(err, float((o[s_idx, :, :e - b].transpose(0, 1).float() - ours_out[b:e].float())
                             .abs().max()))
    res = {"impl": "torch SDPA, padded to the longest sequence, explicit (bsz,1,L,L) bool mask",
           "ms": round(ms, 3), "max_abs_diff_vs_ours": round(err, 5),
           "mask_bytes": int(mask.numel()), "padded_tokens": int(S * L)}
    del qp, kp, vp, mask, o
    torch.cuda.empty_cache()
    return res


def merge_bench(pk, torch, stream, pack, out, lse, parts=2, reps=20):
    """The LSE merge (ring attention's per-step fold) at the workload's full
    output size: ``parts`` bf16 partial outputs [T, Hq, d] with their LSEs
    merged into a bf16 output.  HBM-bound; inputs exceed L2."""
    peaks = load_peaks()
    T, H, d = out.shape
    ps = [(out, lse)] + [(out.clone(), (lse - 0.5).contiguous()) for _ in range(parts - 1)]
    res_o = torch.empty_like(out)
    res_l = torch.empty_like(lse)
    for _ in range(3):
        pk.lse_merge(ps, out=res_o, lse_out=res_l)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        pk.lse_merge(ps, out=res_o, lse_out=res_l)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    nbytes = (parts + 1) * (T * H * d * out.element_size() + H * T * 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    # a ring step's fold: a bf16 block result into an fp32 running accumulator, in place
    acc = out.float()
    acc_l = lse.clone()
    for _ in range(3):
        pk.lse_merge([(acc, acc_l), (out, lse)], out=acc, lse_out=acc_l)
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        pk.lse_merge([(acc, acc_l), (out, lse)], out=acc, lse_out=acc_l)
        b.record(stream)
    torch.cuda.synchronize()
    ring_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    ring_bytes = T * H * d * (4 + 2 + 4) + 3 * H * T * 4
    ring_gbs = ring_bytes / (ring_ms * 1e-3) / 1e9
    del ps, res_o, res_l, acc, acc_l
    return {"kernel": "lse_merge_kernel", "parts": parts, "ms": round(ms, 4),
            "bytes_per_launch": nbytes,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "peak_source": peaks["source"]},
            "ring_fold_fp32_acc": {"ms": round(ring_ms, 4), "bytes_per_launch": ring_bytes,
                                   "achieved_gbs": round(ring_gbs, 1),
                                   "frac": round(ring_gbs / peaks["hbm_gbs"], 4)}}


def layouts_bench(pk, torch, stream, dev, pack, q, k, v, reps=10):
    """The workload's image tokens as queries over the whole sequence's keys
    (text prefix handed over from the autoregressive stage), with contiguous
    and with paged keys (shuffled 128-row block pool)."""
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    sg = W.seq_segments(pack)
    qs = q[torch.as_tensor(rows, device=dev)].contiguous()
    table, pool_rows = W.paged_layout(pack, np.random.default_rng(0))
    src = torch.as_tensor(np.maximum(pool_rows, 0), device=dev)
    kp, vp = k[src].contiguous(), v[src].contiguous()
    res = {}
    for name, kk, vv, kw in (("prefix", k, v, {}),
                             ("prefix_paged", kp, vp,
                              {"block_table": table, "num_kv_rows": kp.shape[0]})):
        pl = cta_plan(pk.plan_layout(cu_q, cu, sg, pack.hq, pack.hkv, pack.d, q_pos0=q_pos0,
                                     k_pos0=z, device=dev, **kw))
        out = torch.empty_like(qs)
        lse = torch.empty(pack.hq, qs.shape[0], dtype=torch.float32, device=dev)
        ws = torch.empty(pl.workspace_bytes, dtype=torch.uint8, device=dev)
        for _ in range(3):
            pk.attn_fwd(qs, kk, vv, pl, pack.scale, out=out, lse=lse, workspace=ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            pk.attn_fwd(qs, kk, vv, pl, pack.scale, out=out, lse=lse, workspace=ws)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[name] = {"ms": round(ms, 4), "useful_tflops": round(pl.useful_flops / ms / 1e9, 1),
                     "query_tokens": int(qs.shape[0]), "key_rows": int(kk.shape[0])}
        del pl, out, lse, ws
    del qs, kp, vp
    torch.cuda.empty_cache()
    return res


def fp8_bench(pk, torch, stream, dev, pack, q, k, v, reps=10):
    """The workload with FP8 E4M3 queries and keys (per-tensor scales) and
    bf16 values."""
    q8, qs = W.quantize_e4m3(q)
    k8, ks = W.quantize_e4m3(k)
    plan = cta_plan(pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, device=dev))
    out = torch.empty_like(q)
    lse = torch.empty(pack.hq, pack.total_tokens, dtype=torch.float32, device=dev)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    for _ in range(3):
        pk.attn_fwd_fp8(q8, qs, k8, ks, v, plan, pack.scale, out=out, lse=lse, workspace=ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        pk.attn_fwd_fp8(q8, qs, k8, ks, v, plan, pack.scale, out=out, lse=lse, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    res = {"kernel": "pk_attn_fwd_kernel<128, fp8 q/k>", "ms": round(ms, 4),
           "useful_tflops": round(plan.useful_flops / ms / 1e9, 1),
           "qk_bytes_saved": int(q.numel() + k.numel())}
    del q8, k8, out, lse, plan, ws
    torch.cuda.empty_cache()
    return res


def fp8_pv_bench(pk, torch, stream, dev, pack, q, k, v, reps=10):
    """The workload with FP8 E4M3 queries, keys and values and E4M3 softmax
    weights (one launch: the value transpose, then the attention)."""
    q8, qs = W.quantize_e4m3(q)
    k8, ks = W.quantize_e4m3(k)
    v8, vs = W.quantize_e4m3(v)
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(pack.hq, pack.total_tokens, dtype=torch.float32, device=dev)
    ws = torch.empty(plan.workspace_bytes_fp8_pv, dtype=torch.uint8, device=dev)

    def call():
        pk.attn_fwd_fp8_pv(q8, qs, k8, ks, v8, vs, plan, pack.scale, out=out, lse=lse,
                           workspace=ws)
    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    res = {"kernels": ["pk_v8_transpose_kernel", "pk_attn_fwd_kernel<128, fp8 q/k/v/p>"],
           "ms": round(ms, 4), "useful_tflops": round(plan.useful_flops / ms / 1e9, 1),
           "parity": "output error above the 1e-2 bound (E4M3 softmax weights); lse within "
                     "1e-3: recorded by the GPU tests"}
    del q8, k8, v8, out, lse, plan, ws
    torch.cuda.empty_cache()
    return res


def sweep(pk, torch, stream, dev):
    """Timing-only pass over every workload (device-generated inputs)."""
    res = {}
    for name, fn in W.CONFIGS.items():
        pack = fn()
        g = torch.Generator(device=dev).manual_seed(0)
        T = pack.total_tokens
        q = torch.randn(T, pack.hq, pack.d, device=dev, generator=g).bfloat16() * pack.q_mult
        k = torch.randn(T, pack.hkv, pack.d, device=dev, generator=g).bfloat16()
        v = torch.randn(T, pack.hkv, pack.d, device=dev, generator=g).bfloat16()
        plan = cta_plan(pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d,
                                device=dev))
        out = torch.empty_like(q)
        lse = torch.empty(pack.hq, T, dtype=torch.float32, device=dev)
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
        def timed(pl):
            for _ in range(3):
                pk.attn_fwd(q, k, v, pl, pack.scale, out=out, lse=lse, workspace=ws)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            n = 10
            torch.cuda.synchronize()
            ev[0].record(stream)
            for _ in range(n):
                pk.attn_fwd(q, k, v, pl, pack.scale, out=out, lse=lse, workspace=ws)
            ev[1].record(stream)
            torch.cuda.synchronize()
            return ev[0].elapsed_time(ev[1]) / n
        ms = timed(plan)
        fl = plan.useful_flops
        res[name] = {"ms": round(ms, 4), "useful_tflops": round(fl / ms / 1e9, 1),
                     "tokens_per_s": round(T / ms * 1e3), "total_tokens": T}
        if pack.d == 128:  # the opt-in SM-pair kernel on the same inputs
            pair = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d,
                           device=dev).set_sm_pairs(True)
            ms2 = timed(pair)
            res[name]["sm_pairs"] = {"ms": round(ms2, 4), "useful_tflops": round(fl / ms2 / 1e9, 1)}
            del pair
            if plan.kv_share:  # the same inputs on one CTA per SM, without the sharing
                one = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d,
                              device=dev).set_kv_share(False)
                ms4 = timed(one)
                res[name]["one_cta"] = {"ms": round(ms4, 4),
                                        "useful_tflops": round(fl / ms4 / 1e9, 1)}
                del one
            # FP8 E4M3 queries and keys (per-tensor scales) on the same inputs
            q8, qs = W.quantize_e4m3(q)
            k8, ks = W.quantize_e4m3(k)
            for _ in range(3):
                pk.attn_fwd_fp8(q8, qs, k8, ks, v, plan, pack.scale, out=out, lse=lse, workspace=ws)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            torch.cuda.synchronize()
            ev[0].record(stream)
            for _ in range(10):
                pk.attn_fwd_fp8(q8, qs, k8, ks, v, plan, pack.scale, out=out, lse=lse, workspace=ws)
            ev[1].record(stream)
            torch.cuda.synchronize()
            ms3 = ev[0].elapsed_time(ev[1]) / 10
            res[name]["fp8_qk"] = {"ms": round(ms3, 4), "useful_tflops": round(fl / ms3 / 1e9, 1)}
            del q8, k8
        del q, k, v, out, lse, plan, ws
        torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed_resolution", choices=sorted(W.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-replaced", action="store_true",
                    help="skip timing the replaced padded + explicit-mask SDPA path")
    ap.add_argument("--no-merge", action="store_true",
                    help="skip timing the LSE merge at the workload's output size")
    ap.add_argument("--merge-only", action="store_true",
                    help="time only the LSE merge (for profiling it alone)")
    ap.add_argument("--split", action="store_true",
                    help="under torchrun, split the one pack across the ranks (pk_plan_shard: "
                         "whole (sequence, kv head) units per rank, no exchange; strong scaling) "
                         "instead of running one replica per rank")
    ap.add_argument("--one-cta", action="store_true",
                    help="run the step on the one-CTA kernel (pk_plan_set_kv_share off)")
    ap.add_argument("--sm-pairs", action="store_true",
                    help="run the step on the opt-in SM-pair kernel (pk_plan_set_sm_pairs)")
    ap.add_argument("--requests", type=int, default=8,
                    help="requests in the mixed-resolution pack (x2 CFG branches)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup(args)
    global SINGLE_GPU
    SINGLE_GPU = world == 1
    pack = (W.mixed_resolution(requests=args.requests) if args.workload == "mixed_resolution"
            else W.CONFIGS[args.workload]())

    if args.impl == "reference":
        return reference_arm(args, pack, rank, world)

    import torch
    import packed_varlen_masked_gb300 as pk
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=dev)
        dist = dist_mod

    def barrier():
        if dist is not None:
            dist.barrier()

    q, k, v = W.make_qkv(pack)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    plan = cta_plan(pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, device=dev))
    split = args.split and world > 1
    full_plan = plan
    if split:  # this rank's share of the one pack, on the full tensors
        plan = cta_plan(full_plan.shard(rank, world, device=dev))
    if args.sm_pairs:
        plan.set_sm_pairs(True)
    elif args.one_cta and plan.kv_share:
        plan.set_kv_share(False)
    shared_kv = plan.kv_share and not args.sm_pairs
    out = torch.empty_like(q)
    lse = torch.empty(pack.hq, pack.total_tokens, dtype=torch.float32, device=dev)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        pk.convert_values(v, plan, workspace=ws, status=status)
        pk.attn_fwd_converted(q, k, ws, plan, pack.scale, out=out, lse=lse, status=status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")
    if args.merge_only:
        if rank == 0:
            print(json.dumps({"merge": merge_bench(pk, torch, stream, pack, out, lse)}), flush=True)
        return

    # timed region: K steps, events before, between and after each step's two
    # launches on the launching stream (per-launch durations for the rooflines)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
           for _ in range(args.steps)]
    t_all = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                      else local) as clk:
        barrier()
        torch.cuda.synchronize()
        t_all[0].record(stream)
        for i in range(args.steps):
            evs[i][0].record(stream)
            pk.convert_values(v, plan, workspace=ws, status=status)
            evs[i][1].record(stream)
            pk.attn_fwd_converted(q, k, ws, plan, pack.scale, out=out, lse=lse, status=status)
            evs[i][2].record(stream)
        t_all[1].record(stream)
        torch.cuda.synchronize()
        barrier()
    total_ms = t_all[0].elapsed_time(t_all[1])
    conv_ms = [a.elapsed_time(b) for a, b, _ in evs]
    launch_ms = [b.elapsed_time(c) for _, b, c in evs]
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")
    total_ms = max_over_ranks(total_ms, dist, dev)

    flops = plan.useful_flops  # this rank's launches
    ms_step = total_ms / args.steps
    # the job's units per step: one pack split across the ranks, or one
    # replica per rank
    job_ranks, job_flops = (1, full_plan.useful_flops) if split else (world, flops)
    value = job_throughput(job_ranks, job_flops, args.steps, total_ms) / 1e12
    tokens_per_s = job_throughput(job_ranks, pack.total_tokens, args.steps, total_ms)

    # end to end through the public host-buffer API: every step copies its
    # inputs from pinned host memory and its outputs back.  HostPipeline runs
    # each step's copy-in, kernel and copy-out on three streams over three
    # device slots, so one step's copies overlap its neighbours' kernels; the
    # single-stream call (copy, kernel, copy back in series) is timed too.
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()
        qh, kh, vh = pin(q), pin(k), pin(v)
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        # the call's own device staging (its v is converted to fp16 in place)
        bufs = {"q": torch.empty_like(q), "k": torch.empty_like(k), "v": torch.empty_like(v),
                "out": torch.empty_like(out), "lse": torch.empty_like(lse)}
        for _ in range(args.warmup):
            pk.attn_fwd_host(qh, kh, vh, plan, pack.scale, bufs, oh, lh)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            pk.attn_fwd_host(qh, kh, vh, plan, pack.scale, bufs, oh, lh)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        serial_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)

        pipe = pk.HostPipeline(plan, num_slots=3, device=dev)
        for _ in range(args.warmup):
            pipe.submit(qh, kh, vh, oh, lh, pack.scale)
        pipe.sync()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        p0.record(pipe.stream(0))
        for _ in range(args.steps):
            pipe.submit(qh, kh, vh, oh, lh, pack.scale)
        p1.record(pipe.stream(2))
        pipe.sync()
        torch.cuda.synchronize()
        barrier()
        e_ms = max_over_ranks(p0.elapsed_time(p1), dist, dev)
        pipe.close()
        del bufs
        e2e = {"value": job_throughput(job_ranks, job_flops, args.steps, e_ms) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e_ms / args.steps,
               "h2d_bytes_per_step": int((q.numel() + k.numel() + v.numel()) * 2),
               "d2h_bytes_per_step": int(out.numel() * 2 + lse.numel() * 4),
               "api": "HostPipeline (3 device slots; copy-in, compute, copy-out streams)",
               "serial_ms_per_step": serial_ms / args.steps,
               "serial_value": job_throughput(job_ranks, job_flops, args.steps, serial_ms) / 1e12}

    per_workload = None
    if not args.no_sweep and rank == 0:
        per_workload = sweep(pk, torch, stream, dev)
    layouts = fp8 = fp8_pv = None
    if not args.no_sweep and rank == 0:
        layouts = layouts_bench(pk, torch, stream, dev, pack, q, k, v)
        fp8 = fp8_bench(pk, torch, stream, dev, pack, q, k, v)
        fp8_pv = fp8_pv_bench(pk, torch, stream, dev, pack, q, k, v)
    merge = None
    if not args.no_merge and rank == 0:
        merge = merge_bench(pk, torch, stream, pack, out, lse)
    replaced = None
    if not args.no_replaced and rank == 0:
        step()
        torch.cuda.synchronize()
        replaced = replaced_path(torch, pack, q, k, v, out)
        replaced["speedup_of_packed"] = round(replaced["ms"] / ms_step, 2)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peaks = load_peaks()
    avg_launch_ms = statistics.mean(launch_ms)
    achieved = flops / (avg_launch_ms * 1e-3) / 1e12
    avg_conv_ms = statistics.mean(conv_ms)
    conv_bytes = 2 * plan.workspace_bytes  # read bf16 v, write fp16 v
    conv_gbs = conv_bytes / (avg_conv_ms * 1e-3) / 1e9
    # the committed capture is of the default kernel (head-pair clusters)
    traffic = load_traffic() if shared_kv else None
    info = plan.info
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(pack)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "strong" if split else "weak", "vs_baseline": None,
        "dtype": "bf16", "pv_dtype": "fp16", "data": "synthetic",
        "config": workload_config(pack, world, full_plan.useful_flops, split),
        "tokens_per_s": round(tokens_per_s),
        "pct_of_nominal_bf16_peak": round(100 * value / world / NOMINAL_BF16_TFLOPS, 2),
        "pct_of_measured_bf16_peak": round(100 * value / world / peaks["bf16_tflops"], 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
                     "frac_of_sustained": (round(achieved / peaks["bf16_tflops_sustained"], 4)
                                           if peaks.get("bf16_tflops_sustained") else None),
                     "peak_source": peaks["source"] + " (bf16 burst)",
                     "kernel": ("pk_attn_fwd_kernel<128> on SM pairs" if args.sm_pairs
                                else "pk_attn_fwd_kernel<128> on head-pair clusters "
                                     "(key/value tiles multicast)" if shared_kv
                                else "pk_attn_fwd_kernel<128>, one CTA per SM"),
                     "launch_ms_mean": round(avg_launch_ms, 4),
                     "launch_ms_median": round(statistics.median(launch_ms), 4),
                     "launch_ms_min": round(min(launch_ms), 4)},
        "value_conversion": {"kernel": "pk_v_to_f16_kernel", "bound": "hbm",
                             "ms_mean": round(avg_conv_ms, 4), "bytes_per_launch": conv_bytes,
                             "achieved": round(conv_gbs, 1), "peak": peaks["hbm_gbs"],
                             "unit": "GB/s", "frac": round(conv_gbs / peaks["hbm_gbs"], 4),
                             "share_of_step": round(avg_conv_ms / ms_step, 4)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
        "plan": dict({k2: info[k2] for k2 in ("num_items", "num_ctas", "num_full_tiles",
                                               "num_partial_tiles")},
                     head_pair_clusters=int(len(plan.share_schedule()[1]) - 1) if shared_kv else 0),
        "per_workload": per_workload,
        "replaced_path": replaced,
        "layouts": layouts,
        "fp8_qk": fp8,
        "fp8_qkvp": fp8_pv,
        "lse_merge": merge,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
