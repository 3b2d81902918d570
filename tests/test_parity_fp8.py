"""GPU parity of the FP8 path (E4M3 queries and keys, bf16 values) against
the fp64 oracle's E4M3 entry on the same codes and scales.  The quantisation
is part of the inputs, not of the kernel: both sides read the same E4M3
values, so the rule is the bf16 path's (parity_tol.py)."""
import numpy as np
import pytest
import torch

import oracle
import packed_varlen_masked_gb300 as pk
import workloads as W
from parity_tol import check

pytestmark = pytest.mark.gpu


def _compare(name, out_g, lse_g, out_o, lse_o):
    check(name, out_g, lse_g, out_o, lse_o)


def _quantised(pack):
    q, k, v = W.make_qkv(pack)
    q8, qs = W.quantize_e4m3(q)
    k8, ks = W.quantize_e4m3(k)
    return q8, qs, k8, ks, v


@pytest.mark.parametrize("pack", [
    W.Pack("fp8-mixed", [[(W.TEXT, 40), (W.IMAGE, 600), (W.TEXT, 9)], [(W.IMAGE, 300), (W.IMAGE, 130)],
                         [(W.TEXT, 1)], [], [(W.TEXT, 77), (W.IMAGE, 513)]], hq=8, hkv=2, d=128, seed=51),
    W.Pack("fp8-mha-odd", [[(W.TEXT, 129), (W.IMAGE, 256)], [(W.IMAGE, 383)]], hq=3, hkv=3, d=128, seed=52),
    W.Pack("fp8-sharp", [[(W.TEXT, 100), (W.IMAGE, 400)]], hq=4, hkv=1, d=128, seed=53, q_mult=4.0),
], ids=lambda p: p.name)
def test_fp8_small_packs_full(pack):
    q8, qs, k8, ks, v = _quantised(pack)
    out_o, lse_o = oracle.attention_e4m3(q8, qs, k8, ks, v, pack.cu_seqlens, pack.segments,
                                         pack.hq, pack.hkv, pack.d, pack.scale)
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    out, lse = pk.attn_fwd_fp8(q8.cuda(), qs, k8.cuda(), ks, v.cuda(), plan, pack.scale,
                               check_status=True)
    _compare(pack.name, out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)


def test_fp8_full_size_sampled():
    pack = W.mixed_resolution()
    q8, qs, k8, ks, v = _quantised(pack)
    rows = W.sample_rows(pack, 256)
    out_o, lse_o = oracle.attention_e4m3(q8, qs, k8, ks, v, pack.cu_seqlens, pack.segments,
                                         pack.hq, pack.hkv, pack.d, pack.scale, rows=rows)
    plan = pk.plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d)
    out, lse = pk.attn_fwd_fp8(q8.cuda(), qs, k8.cuda(), ks, v.cuda(), plan, pack.scale,
                               check_status=True)
    _compare("mixed_resolution/fp8", out.float().cpu().numpy()[rows], lse.cpu().numpy()[:, rows],
             out_o, lse_o)


def test_fp8_cached_prefix_paged_keys():
    """FP8 on the general layout: image queries over a paged key pool; the
    oracle side is the E4M3 attention's image rows."""
    pack = W.Pack("fp8-prefix", [[(W.TEXT, 70), (W.IMAGE, 400)], [(W.TEXT, 33), (W.IMAGE, 260)]],
                  hq=8, hkv=2, d=128, seed=54)
    q8, qs, k8, ks, v = _quantised(pack)
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    table, pool_rows = W.paged_layout(pack, np.random.default_rng(9))
    src = torch.as_tensor(np.maximum(pool_rows, 0))
    kp8, vp = k8[src].clone(), v[src].clone()
    kp8[torch.as_tensor(pool_rows < 0)] = 0x7E  # junk (448) in unowned rows
    pl = pk.plan_layout(cu_q, cu, W.seq_segments(pack), pack.hq, pack.hkv, pack.d, q_pos0=q_pos0,
                        k_pos0=z, block_table=table, num_kv_rows=kp8.shape[0])
    out, lse = pk.attn_fwd_fp8(q8[torch.as_tensor(rows)].contiguous().cuda(), qs, kp8.cuda(), ks,
                               vp.cuda(), pl, pack.scale, check_status=True)
    out_o, lse_o = oracle.attention_e4m3(q8, qs, k8, ks, v, cu, pack.segments, pack.hq, pack.hkv,
                                         pack.d, pack.scale, rows=rows.astype(np.int32))
    _compare("fp8-prefix-paged", out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)
