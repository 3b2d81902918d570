"""GPU parity of the head-pair clusters (pk_plan_set_kv_share: the default
at head_dim 128 wherever every work item holds two query heads, opt-in at
64).  Each CTA of
a cluster runs the one-CTA kernel's arithmetic, in the same order, on its
query head; only the copies of the key and value tiles are shared.  So the
outputs must equal the one-CTA kernel's bit for bit (the default path is
also held to the oracle by every other parity test); one case is compared
with the oracle directly."""
import numpy as np
import pytest
import torch

import oracle
import packed_varlen_masked_gb300 as pk
import workloads as W
from parity_tol import check

pytestmark = pytest.mark.gpu


def _both(pack, q, k, v, plan_args=None, plan_kw=None, fp8=None):
    """(one-CTA out, lse), (head-pair cluster out, lse) for the same inputs."""
    if plan_args is None:
        plan_args = (pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    mk = (lambda: pk.plan_layout(*plan_args, **plan_kw)) if plan_kw is not None else \
        (lambda: pk.plan(*plan_args))
    one = mk().set_kv_share(False)
    share = mk().set_kv_share(True)  # the default at d = 128, opt-in at 64
    assert share.kv_share
    res = []
    for plan in (one, share):
        if fp8 is None:
            res.append(pk.attn_fwd(q, k, v, plan, pack.scale, check_status=True))
        else:
            q8, qs, k8, ks = fp8
            res.append(pk.attn_fwd_fp8(q8, qs, k8, ks, v, plan, pack.scale, check_status=True))
    return res


def _assert_identical(a, b):
    (o1, l1), (o2, l2) = a, b
    assert torch.equal(o1, o2), float((o1.float() - o2.float()).abs().max())
    assert torch.equal(l1.nan_to_num(), l2.nan_to_num()) and \
        torch.equal(torch.isneginf(l1), torch.isneginf(l2))


def _packs():
    rng = np.random.default_rng(91)
    packs = [W.random_pack(rng, 5, 900, hq=hq, hkv=hkv, d=d, name=f"rnd{i}-h{hq}-{hkv}-d{d}")
             for i, (hq, hkv, d) in enumerate([(8, 2, 128), (4, 2, 128), (2, 1, 128), (16, 2, 128),
                                               (8, 4, 128), (8, 2, 64), (4, 2, 64)])]
    packs += [
        W.Pack("odd-tiles", [[(W.TEXT, 1)], [], [(W.IMAGE, 129)], [(W.TEXT, 128), (W.IMAGE, 257)],
                             [(W.IMAGE, 383), (W.TEXT, 1)]], hq=4, hkv=2, d=128, seed=41),
        W.Pack("one-item", [[(W.TEXT, 17)]], hq=2, hkv=1, d=128, seed=42),
        W.Pack("sharp-q8", [[(W.TEXT, 100), (W.IMAGE, 400)], [(W.TEXT, 30), (W.IMAGE, 256)]],
               hq=8, hkv=2, d=128, seed=43, q_mult=8.0),
    ]
    return packs


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
def test_share_equals_the_one_cta_kernel(pack):
    q, k, v = W.make_qkv(pack, device="cuda")
    _assert_identical(*_both(pack, q, k, v))


@pytest.mark.parametrize("name", ["cfg_pair", "mixed_resolution", "highres_edit", "skewed"])
def test_share_equals_the_one_cta_kernel_on_the_configurations(name):
    pack = W.CONFIGS[name]()
    q, k, v = W.make_qkv(pack, device="cuda")
    _assert_identical(*_both(pack, q, k, v))


@pytest.mark.parametrize("name", ["cfg_pair", "mixed_resolution"])
def test_share_fp8_equals_the_one_cta_kernel(name):
    """FP8 queries and keys: one-box key tiles, which the two CTAs split by
    rows (64 each)."""
    pack = W.CONFIGS[name]()
    q, k, v = W.make_qkv(pack)
    q8, qs = W.quantize_e4m3(q)
    k8, ks = W.quantize_e4m3(k)
    _assert_identical(*_both(pack, None, None, v.cuda(), fp8=(q8.cuda(), qs, k8.cuda(), ks)))


@pytest.mark.parametrize("ctas", [2, 7, 24])
def test_share_with_few_clusters(ctas):
    """Plans built for few CTAs: one to twelve clusters, each running many
    items back to back (and an odd CTA count, whose last CTA the clusters
    leave out)."""
    pack = W.CONFIGS["cfg_pair"]()
    q, k, v = W.make_qkv(pack, device="cuda")
    args = (pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    one = pk.plan(*args, num_ctas=ctas).set_kv_share(False)
    share = pk.plan(*args, num_ctas=ctas)
    assert share.kv_share and len(share.share_schedule()[1]) - 1 == ctas // 2
    _assert_identical(pk.attn_fwd(q, k, v, one, pack.scale, check_status=True),
                      pk.attn_fwd(q, k, v, share, pack.scale, check_status=True))


def _sweep_packs():
    rng = np.random.default_rng(2024)
    out = []
    for i in range(24):
        hkv = int(rng.choice([1, 2, 4]))
        group = int(rng.choice([2, 4, 8]))
        d = int(rng.choice([64, 128]))
        out.append(W.random_pack(rng, int(rng.integers(1, 7)), int(rng.integers(40, 1600)),
                                 hq=hkv * group, hkv=hkv, d=d,
                                 name=f"sweep{i}-h{hkv * group}-{hkv}-d{d}"))
    return out


@pytest.mark.parametrize("pack", _sweep_packs(), ids=lambda p: p.name)
def test_share_random_sweep(pack):
    """Seeded random packs over group sizes 2 to 8, one to four key/value
    heads and both head dimensions; FP8 queries and keys too at d = 128."""
    q, k, v = W.make_qkv(pack, device="cuda")
    _assert_identical(*_both(pack, q, k, v))
    if pack.d == 128:
        q8, qs = W.quantize_e4m3(q)
        k8, ks = W.quantize_e4m3(k)
        _assert_identical(*_both(pack, None, None, v, fp8=(q8, qs, k8, ks)))


def test_share_d64_against_the_oracle():
    pack = W.Pack("share-d64", [[(W.TEXT, 70), (W.IMAGE, 300)], [(W.IMAGE, 129), (W.TEXT, 5)]],
                  hq=8, hkv=2, d=64, seed=46)
    q, k, v = W.make_qkv(pack)
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                                    pack.d, pack.scale)
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    assert not plan.kv_share  # opt-in at d = 64
    plan.set_kv_share(True)
    out, lse = pk.attn_fwd(q.cuda(), k.cuda(), v.cuda(), plan, pack.scale, check_status=True)
    check(pack.name, out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)


def test_share_against_the_oracle():
    pack = _packs()[-1]
    q, k, v = W.make_qkv(pack)
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                                    pack.d, pack.scale)
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    assert plan.kv_share  # the default at d = 128
    out, lse = pk.attn_fwd(q.cuda(), k.cuda(), v.cuda(), plan, pack.scale, check_status=True)
    check(pack.name + "/share", out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)


def test_share_on_a_cached_prefix_with_paged_keys_and_on_key_chunks():
    pack = W.Pack("share-layouts", [[(W.TEXT, 70), (W.IMAGE, 900)], [(W.TEXT, 33), (W.IMAGE, 600)]],
                  hq=8, hkv=2, d=128, seed=44)
    q, k, v = W.make_qkv(pack, device="cuda")
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    table, pool_rows = W.paged_layout(pack, np.random.default_rng(5))
    src = torch.as_tensor(np.maximum(pool_rows, 0), device="cuda")
    kp, vp = k[src].contiguous(), v[src].contiguous()
    qr = q[torch.as_tensor(rows, device="cuda")].contiguous()
    args = (cu_q, cu, W.seq_segments(pack), pack.hq, pack.hkv, pack.d)
    kw = dict(q_pos0=q_pos0, k_pos0=z, block_table=table, num_kv_rows=kp.shape[0])
    _assert_identical(*_both(pack, qr, kp, vp, plan_args=args, plan_kw=kw))
    for cu_k, k_pos0, krows in W.key_chunks(pack, 384):
        kr = torch.as_tensor(krows, device="cuda")
        args = (cu, cu_k, W.seq_segments(pack), pack.hq, pack.hkv, pack.d)
        kw = dict(q_pos0=z, k_pos0=k_pos0)
        _assert_identical(*_both(pack, q, k[kr].contiguous(), v[kr].contiguous(), plan_args=args,
                                 plan_kw=kw))


def test_share_short_wait_limit_aborts_and_the_context_survives():
    """Waits of a few microseconds or less run out in the clusters too: the
    launch reports PK_ERR_TIMEOUT, both CTAs of every cluster leave through
    the abort path (bounded drains of the shared rings), and with the
    default limit restored the next launch equals the one-CTA kernel."""
    pack = W.mixed_resolution(seed=6, requests=2)
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
    _assert_identical(*_both(pack, q, k, v))


def test_plans_without_the_schedule_run_the_one_cta_kernel():
    """An odd number of query heads per key/value head: no head-pair
    schedule; the default launch is the one-CTA kernel, held to the oracle."""
    pack = W.Pack("odd-group", [[(W.TEXT, 50), (W.IMAGE, 300)], [(W.IMAGE, 200)]], hq=6, hkv=2,
                  d=128, seed=45)
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    assert plan.share_schedule()[0].shape[0] == 0
    q, k, v = W.make_qkv(pack)
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                                    pack.d, pack.scale)
    out, lse = pk.attn_fwd(q.cuda(), k.cuda(), v.cuda(), plan, pack.scale, check_status=True)
    check(pack.name, out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)
