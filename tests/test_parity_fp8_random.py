"""Seeded random sweep of the FP8 path (E4M3 queries and keys, bf16 values)
against the fp64 oracle, on the same kinds of random packs as the bf16
sweep: whole sequences against the oracle's E4M3 entry, and the cached
prefix with paged keys and key chunks against its general-layout entry on
the exactly decoded tensors (power-of-two scales make every E4M3 value
exact in bf16).  The quantisation is part of the inputs, so the bf16 rule
holds (parity_tol.py)."""
import numpy as np
import pytest
import torch

import oracle
import packed_varlen_masked_gb300 as pk
import workloads as W
from parity_tol import check

pytestmark = pytest.mark.gpu


def _pow2_quantised(x):
    amax = float(x.float().abs().max())
    scale = float(2.0 ** np.ceil(np.log2(amax / 448.0))) if amax > 0 else 1.0
    return (x.float() / scale).to(torch.float8_e4m3fn).view(torch.uint8), scale


def _decoded(codes, scale):
    return (codes.view(torch.float8_e4m3fn).float() * scale).to(torch.bfloat16)


def _packs():
    rng = np.random.default_rng(8088)
    out = []
    for i in range(8):
        group = int(rng.choice([1, 2, 4, 8]))
        hkv = int(rng.choice([1, 2]))
        out.append(W.random_pack(rng, int(rng.integers(1, 5)), int(rng.choice([50, 300, 700])),
                                 hq=group * hkv, hkv=hkv, d=128, name=f"fp8rnd{i}-g{group}-kv{hkv}"))
    return out


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
def test_fp8_random_pack_all_layouts(pack):
    if pack.total_tokens == 0:
        pytest.skip("empty pack")
    q, k, v = W.make_qkv(pack)
    q8, qs = _pow2_quantised(q)
    k8, ks = _pow2_quantised(k)
    qd, kd = _decoded(q8, qs), _decoded(k8, ks)
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    sg = W.seq_segments(pack)
    out_o, lse_o = oracle.attention_e4m3(q8, qs, k8, ks, v, cu, pack.segments, pack.hq, pack.hkv,
                                         pack.d, pack.scale)
    plan = pk.plan(cu, pack.segments, pack.hq, pack.hkv, pack.d)
    o, l = pk.attn_fwd_fp8(q8.cuda(), qs, k8.cuda(), ks, v.cuda(), plan, pack.scale,
                           check_status=True)
    check(pack.name, o.float().cpu().numpy(), l.cpu().numpy(), out_o, lse_o)
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    if len(rows):
        table, pool_rows = W.paged_layout(pack, np.random.default_rng(pack.seed % 1000))
        src = torch.as_tensor(np.maximum(pool_rows, 0))
        kp8, vp = k8[src].clone(), v[src].clone()
        pl = pk.plan_layout(cu_q, cu, sg, pack.hq, pack.hkv, pack.d, q_pos0=q_pos0, k_pos0=z,
                            block_table=table, num_kv_rows=kp8.shape[0])
        o, l = pk.attn_fwd_fp8(q8[torch.as_tensor(rows)].contiguous().cuda(), qs, kp8.cuda(), ks,
                               vp.cuda(), pl, pack.scale, check_status=True)
        check(pack.name + "/prefix-paged", o.float().cpu().numpy(), l.cpu().numpy(),
              out_o[rows], lse_o[:, rows])
    chunk = int(np.random.default_rng(pack.seed).choice([128, 200, 384]))
    for cu_k, k_pos0, krows in W.key_chunks(pack, chunk):
        idx = torch.as_tensor(krows)
        if idx.numel() == 0:
            continue
        oo, lo = oracle.attention_general(qd, kd[idx].contiguous(), v[idx].contiguous(), cu, cu_k, z,
                                          k_pos0, sg, pack.hq, pack.hkv, pack.d, pack.scale)
        pl = pk.plan_layout(cu, cu_k, sg, pack.hq, pack.hkv, pack.d, q_pos0=z, k_pos0=k_pos0)
        o, l = pk.attn_fwd_fp8(q8.cuda(), qs, k8[idx].contiguous().cuda(), ks,
                               v[idx].contiguous().cuda(), pl, pack.scale, check_status=True)
        check(pack.name + "/key-chunk", o.float().cpu().numpy(), l.cpu().numpy(), oo, lo)
