"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, under the rule of parity_tol.py: max-abs 1e-2 on the
bf16 outputs (plus half a bf16 ulp only where |o| >= 4, where no bf16 value
can do better) and 1e-3 on the fp32 LSE, on every workload, the q x4 pack
included."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import packed_varlen_masked_gb300 as pk
import workloads as W
from parity_tol import check

pytestmark = pytest.mark.gpu


def _gpu(pack, q, k, v, plan=None):
    if plan is None:
        plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    out, lse = pk.attn_fwd(q.cuda(), k.cuda(), v.cuda(), plan, pack.scale, check_status=True)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _compare(pack, out_g, lse_g, out_o, lse_o, rows=None, tag=""):
    if rows is not None:
        out_g, lse_g = out_g[rows], lse_g[:, rows]
    check(pack.name + tag, out_g, lse_g, out_o, lse_o)


def _full(pack, q=None, k=None, v=None):
    if q is None:
        q, k, v = W.make_qkv(pack)
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq,
                                    pack.hkv, pack.d, pack.scale)
    out_g, lse_g = _gpu(pack, q, k, v)
    _compare(pack, out_g, lse_g, out_o, lse_o)


def _small_packs():
    rng = np.random.default_rng(2024)
    packs = []
    for i, (hq, hkv, d) in enumerate([(8, 2, 128), (8, 2, 64), (6, 2, 128), (4, 4, 64),
                                      (2, 1, 128), (3, 3, 64)]):
        packs.append(W.random_pack(rng, 4, 700, hq=hq, hkv=hkv, d=d, name=f"rand{i}-h{hq}-{hkv}-d{d}"))
    packs.append(W.Pack("ragged-tails", [[(W.TEXT, 1)], [], [(W.IMAGE, 1)], [(W.IMAGE, 129)],
                                         [(W.TEXT, 128), (W.IMAGE, 129), (W.TEXT, 3)],
                                         [(W.IMAGE, 255), (W.TEXT, 1)], [(W.TEXT, 383)]],
                        hq=4, hkv=2, d=128, seed=5))
    packs.append(W.Pack("adjacent-images", [[(W.TEXT, 40), (W.IMAGE, 200), (W.IMAGE, 200),
                                             (W.IMAGE, 300), (W.TEXT, 7)]],
                        hq=8, hkv=2, d=128, seed=6))
    packs.append(W.Pack("all-text-causal", [[(W.TEXT, 513)], [(W.TEXT, 77)]], hq=4, hkv=2, d=128, seed=7))
    packs.append(W.Pack("all-image-full", [[(W.IMAGE, 513)], [(W.IMAGE, 77)]], hq=4, hkv=2, d=64, seed=8))
    packs.append(W.Pack("sharp-q8", [[(W.TEXT, 100), (W.IMAGE, 400)], [(W.TEXT, 30), (W.IMAGE, 256)]],
                        hq=8, hkv=2, d=128, seed=9, q_mult=8.0))
    return packs


@pytest.mark.parametrize("pack", _small_packs(), ids=lambda p: p.name)
def test_small_packs_full(pack):
    _full(pack)


def test_tiny_config_full():
    _full(W.tiny_pack())


def test_cfg_pair_config_full():
    _full(W.cfg_pair())


@pytest.mark.parametrize("name,budget", [("mixed_resolution", 384), ("highres_edit", 192),
                                         ("skewed", 384)])
def test_full_size_configs_sampled(name, budget):
    """Full-size packs in the benchmark's launch configuration (one CTA per
    SM), compared on a deterministic row sample that includes every sequence
    and segment edge and rows on both sides of 128-row tile edges."""
    pack = W.CONFIGS[name]()
    q, k, v = W.make_qkv(pack)
    rows = W.sample_rows(pack, budget)
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq,
                                    pack.hkv, pack.d, pack.scale, rows=rows)
    out_g, lse_g = _gpu(pack, q, k, v)
    _compare(pack, out_g, lse_g, out_o, lse_o, rows=rows, tag="/sampled")


@pytest.mark.parametrize("name,budget", [("mixed_resolution", 1536), ("highres_edit", 512),
                                         ("skewed", 1536)])
def test_full_size_boundary_tiles(name, budget):
    """Full-size packs, every row of the query tiles where the mask changes
    shape (segment starts and ends, ragged sequence tails): the rows whose
    key tiles are partial."""
    pack = W.CONFIGS[name]()
    q, k, v = W.make_qkv(pack)
    rows = W.boundary_tile_rows(pack, budget)
    assert len(rows) >= 256
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq,
                                    pack.hkv, pack.d, pack.scale, rows=rows)
    out_g, lse_g = _gpu(pack, q, k, v)
    _compare(pack, out_g, lse_g, out_o, lse_o, rows=rows, tag="/boundary-tiles")


def test_growing_maximum_rescales_output():
    """Scores that grow key tile after key tile force the running maximum to
    move by more than the lazy-rescale threshold many times."""
    pack = W.Pack("growing", [[(W.IMAGE, 1024)], [(W.TEXT, 640)]], hq=2, hkv=1, d=64, seed=3)
    q, k, v = W.make_qkv(pack)
    T = pack.total_tokens
    ramp = torch.linspace(0.0, 6.0, T).view(T, 1, 1)
    k = (k.float() * 0.1 + ramp).bfloat16()
    q = torch.ones_like(q) * 0.5
    _full(pack, q, k, v)


def test_every_row_written_and_guard_bands_untouched():
    pack = W.Pack("guard", [[(W.TEXT, 50), (W.IMAGE, 200)], [(W.TEXT, 3)], [(W.IMAGE, 130)]],
                  hq=4, hkv=2, d=128, seed=11)
    q, k, v = W.make_qkv(pack)
    T, G = pack.total_tokens, 4096
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    out_buf = torch.full((T * pack.hq * pack.d + 2 * G,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_buf = torch.full((T * pack.hq + 2 * G,), float("nan"), dtype=torch.float32, device="cuda")
    out = out_buf[G:G + T * pack.hq * pack.d].view(T, pack.hq, pack.d)
    lse = lse_buf[G:G + T * pack.hq].view(pack.hq, T)
    pk.attn_fwd(q.cuda(), k.cuda(), v.cuda(), plan, pack.scale, out=out, lse=lse, check_status=True)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    assert torch.isnan(out_buf[:G]).all() and torch.isnan(out_buf[-G:]).all()
    assert torch.isnan(lse_buf[:G]).all() and torch.isnan(lse_buf[-G:]).all()


def test_deterministic_and_plan_reusable():
    pack = W.mixed_resolution(seed=3, requests=2)
    q, k, v = W.make_qkv(pack, device="cuda")
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    o1, l1 = pk.attn_fwd(q, k, v, plan, pack.scale, check_status=True)
    o2, l2 = pk.attn_fwd(q, k, v, plan, pack.scale, check_status=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # same plan, other inputs
    q2 = torch.randn_like(q, dtype=torch.float32).bfloat16()
    o3, _ = pk.attn_fwd(q2, k, v, plan, pack.scale, check_status=True)
    assert not torch.equal(o1, o3)


def test_single_token_and_empty_pack():
    pack = W.Pack("one", [[(W.TEXT, 1)]], hq=2, hkv=1, d=64, seed=1)
    _full(pack)
    empty = pk.plan([0, 0], [], 2, 1, 64)
    z = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    zk = torch.zeros(0, 1, 64, dtype=torch.bfloat16, device="cuda")
    out, lse = pk.attn_fwd(z, zk, zk, empty, 0.125, check_status=True)
    assert out.shape == (0, 2, 64) and lse.shape == (2, 0)


def test_misaligned_tensor_rejected_before_launch():
    pack = W.Pack("mis", [[(W.TEXT, 64)]], hq=2, hkv=2, d=64, seed=1)
    plan = pk.plan(pack.cu_seqlens, pack.segments, 2, 2, 64)
    lib = pk.load()
    base = torch.zeros(64 * 2 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    good = base[:64 * 2 * 64]
    lse = torch.zeros(2, 64, dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    st = lib.pk_attn_fwd(plan.handle, ctypes.c_void_p(base.data_ptr() + 2), ctypes.c_void_p(good.data_ptr()),
                         ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(good.data_ptr()),
                         ctypes.c_void_p(lse.data_ptr()), 0.125, ctypes.c_void_p(ws.data_ptr()),
                         plan.workspace_bytes, None, None)
    assert st == pk.PK_ERR_ALIGNMENT
    # a workspace one byte short, or misaligned, is rejected before any launch
    st = lib.pk_attn_fwd(plan.handle, ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(good.data_ptr()),
                         ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(good.data_ptr()),
                         ctypes.c_void_p(lse.data_ptr()), 0.125, ctypes.c_void_p(ws.data_ptr()),
                         plan.workspace_bytes - 1, None, None)
    assert st == pk.PK_ERR_INVALID_ARG
    st = lib.pk_attn_fwd(plan.handle, ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(good.data_ptr()),
                         ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(good.data_ptr()),
                         ctypes.c_void_p(lse.data_ptr()), 0.125, ctypes.c_void_p(ws.data_ptr() + 8),
                         plan.workspace_bytes, None, None)
    assert st == pk.PK_ERR_ALIGNMENT


def test_bounded_wait_reports_timeout_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.debug_wait_timeout(status, 2_000_000)  # 2 ms
    torch.cuda.synchronize()
    assert int(status.item()) == pk.PK_ERR_TIMEOUT
    _full(W.Pack("after-timeout", [[(W.TEXT, 20), (W.IMAGE, 150)]], hq=2, hkv=1, d=64, seed=2))


def test_short_wait_limit_aborts_real_launches_and_the_context_survives():
    """Wait limits of a few microseconds or less make the attention kernel's
    own waits run out: the launch must report PK_ERR_TIMEOUT, leave through
    its abort path (drains bounded independently of the limit) and keep the
    context usable; with the default limit restored the next launch is
    exact again."""
    pack = W.mixed_resolution(seed=5, requests=2)
    q, k, v = W.make_qkv(pack, device="cuda")
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    seen = []
    try:
        for limit in (2000, 300, 1):
            pk.set_wait_timeout_ns(limit)
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            pk.attn_fwd(q, k, v, plan, pack.scale, status=status)
            torch.cuda.synchronize()
            seen.append(int(status.item()))
    finally:
        pk.set_wait_timeout_ns(4_000_000_000)
    assert set(seen) <= {pk.PK_OK, pk.PK_ERR_TIMEOUT}, seen
    assert pk.PK_ERR_TIMEOUT in seen, seen
    rows = W.sample_rows(pack, 128)
    out_o, lse_o = oracle.attention(q.cpu(), k.cpu(), v.cpu(), pack.cu_seqlens, pack.segments,
                                    pack.hq, pack.hkv, pack.d, pack.scale, rows=rows)
    out_g, lse_g = _gpu(pack, q, k, v, plan)
    _compare(pack, out_g, lse_g, out_o, lse_o, rows=rows, tag="/after-abort")


@pytest.mark.parametrize("world", [2, 3])
def test_pack_split_across_ranks_assembles_to_the_single_launch(world):
    """The shares of pk_plan_shard, run one after another on this GPU (they
    do not wait on one another), each write only their units' rows and
    heads; put together they equal the one-launch result bit for bit."""
    pack = W.mixed_resolution(seed=7, requests=2)
    q, k, v = W.make_qkv(pack, device="cuda")
    full = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    ref_o, ref_l = pk.attn_fwd(q, k, v, full, pack.scale, check_status=True)
    owner = torch.full((pack.total_tokens, pack.hq), -1, dtype=torch.int32, device="cuda")
    asm_o = torch.zeros_like(ref_o)
    asm_l = torch.zeros_like(ref_l)
    for r in range(world):
        sh = full.shard(r, world)
        o = torch.full_like(ref_o, float("nan"))
        l = torch.full_like(ref_l, float("nan"))
        pk.attn_fwd(q, k, v, sh, pack.scale, out=o, lse=l, check_status=True)
        written = ~torch.isnan(l).T  # [T, hq]
        assert bool((owner[written] == -1).all()), "a row/head written by two ranks"
        assert bool((~torch.isnan(o)).all(-1).eq(written).all())
        owner[written] = r
        asm_o[written] = o[written]
        asm_l.T[written] = l.T[written]
    assert bool((owner >= 0).all())
    assert torch.equal(asm_o, ref_o) and torch.equal(asm_l, ref_l)


def test_one_64k_token_sequence_sampled():
    """A single 65,536-token sequence (1,024 text + 64,512 image): 512 key
    tiles per query tile, the longest rows any workload here has."""
    pack = W.Pack("64k", [[(W.TEXT, 1024), (W.IMAGE, 64512)]], hq=8, hkv=2, d=128, seed=21)
    q, k, v = W.make_qkv(pack)
    rows = np.array([0, 1, 127, 128, 1023, 1024, 1025, 30000, 65407, 65535], np.int32)
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                                    pack.d, pack.scale, rows=rows)
    out_g, lse_g = _gpu(pack, q, k, v)
    _compare(pack, out_g, lse_g, out_o, lse_o, rows=rows)


@pytest.mark.parametrize("hq,hkv,d", [(64, 8, 128), (16, 1, 64), (1, 1, 128)])
def test_head_layouts(hq, hkv, d):
    """Wide GQA groups (8 and 16 query heads per key/value head) and a single
    head."""
    pack = W.Pack(f"heads-{hq}-{hkv}-{d}", [[(W.TEXT, 77), (W.IMAGE, 300)], [(W.IMAGE, 129)]],
                  hq=hq, hkv=hkv, d=d, seed=hq + hkv + d)
    _full(pack)


def test_workspace_may_be_v_itself():
    """Passing v as the workspace converts it in place: same results, and v
    holds the fp16 values afterwards."""
    pack = W.Pack("inplace", [[(W.TEXT, 60), (W.IMAGE, 300)], [(W.IMAGE, 129)]], hq=4, hkv=2,
                  d=128, seed=12)
    q, k, v = W.make_qkv(pack, device="cuda")
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    o1, l1 = pk.attn_fwd(q, k, v, plan, pack.scale, check_status=True)
    v2 = v.clone()
    o2, l2 = pk.attn_fwd(q, k, v2, plan, pack.scale, check_status=True, workspace=v2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(v2.view(torch.float16), v.to(torch.float16))


def test_values_outside_fp16_range_are_reported():
    """A value of magnitude 2^16 cannot enter the fp16 P V product: the launch
    reports PK_ERR_RANGE (and the outputs stay finite: it saturates)."""
    pack = W.Pack("range", [[(W.TEXT, 40), (W.IMAGE, 200)]], hq=2, hkv=1, d=64, seed=13)
    q, k, v = W.make_qkv(pack, device="cuda")
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.attn_fwd(q, k, v, plan, pack.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == pk.PK_OK
    v[17, 0, 5] = 65536.0
    out, _ = pk.attn_fwd(q, k, v, plan, pack.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == pk.PK_ERR_RANGE
    assert torch.isfinite(out).all()
