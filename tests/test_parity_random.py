"""Seeded random sweep of the CUDA path against the fp64 oracle: random
segment structures (text/image runs, adjacent images, one-token segments,
empty sequences), GQA groups 1-8, head dims 64 and 128, each pack also run
as a cached prefix, in key chunks and with paged keys."""
import numpy as np
import pytest
import torch

import oracle
import packed_varlen_masked_gb300 as pk
import workloads as W
from parity_tol import check

pytestmark = pytest.mark.gpu


def _check(out_g, lse_g, out_o, lse_o, case="random"):
    check(case, out_g, lse_g, out_o, lse_o)


def _packs():
    rng = np.random.default_rng(12345)
    out = []
    for i in range(30):
        group = int(rng.choice([1, 2, 3, 4, 8]))
        hkv = int(rng.choice([1, 2]))
        d = int(rng.choice([64, 128]))
        out.append(W.random_pack(rng, int(rng.integers(1, 5)), int(rng.choice([50, 300, 700])),
                                 hq=group * hkv, hkv=hkv, d=d, name=f"rnd{i}-g{group}-kv{hkv}-d{d}"))
    return out


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
def test_random_pack_all_layouts(pack):
    if pack.total_tokens == 0:
        pytest.skip("empty pack")
    q, k, v = W.make_qkv(pack)
    cu = pack.cu_seqlens
    S = len(cu) - 1
    z = np.zeros(S, np.int32)
    sg = W.seq_segments(pack)
    # whole sequences
    out_o, lse_o = oracle.attention(q, k, v, cu, pack.segments, pack.hq, pack.hkv, pack.d,
                                    pack.scale)
    plan = pk.plan(cu, pack.segments, pack.hq, pack.hkv, pack.d)
    o, l = pk.attn_fwd(q.cuda(), k.cuda(), v.cuda(), plan, pack.scale, check_status=True)
    _check(o.float().cpu().numpy(), l.cpu().numpy(), out_o, lse_o, pack.name)
    # cached prefix with paged keys: rows of the full result
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    if len(rows):
        table, pool_rows = W.paged_layout(pack, np.random.default_rng(pack.seed % 1000))
        src = torch.as_tensor(np.maximum(pool_rows, 0))
        kp, vp = k[src].clone(), v[src].clone()
        pl = pk.plan_layout(cu_q, cu, sg, pack.hq, pack.hkv, pack.d, q_pos0=q_pos0, k_pos0=z,
                            block_table=table, num_kv_rows=kp.shape[0])
        o, l = pk.attn_fwd(q[torch.as_tensor(rows)].contiguous().cuda(), kp.cuda(), vp.cuda(), pl,
                           pack.scale, check_status=True)
        _check(o.float().cpu().numpy(), l.cpu().numpy(), out_o[rows], lse_o[:, rows],
               pack.name + "/prefix-paged")
    # key chunks against the oracle's general entry
    for cu_k, k_pos0, krows in W.key_chunks(pack, int(np.random.default_rng(pack.seed).choice([64, 128, 200]))):
        idx = torch.as_tensor(krows)
        kc, vc = k[idx].contiguous(), v[idx].contiguous()
        if kc.shape[0] == 0:
            continue
        oo, lo = oracle.attention_general(q, kc, vc, cu, cu_k, z, k_pos0, sg, pack.hq, pack.hkv,
                                          pack.d, pack.scale)
        pl = pk.plan_layout(cu, cu_k, sg, pack.hq, pack.hkv, pack.d, q_pos0=z, k_pos0=k_pos0)
        o, l = pk.attn_fwd(q.cuda(), kc.cuda(), vc.cuda(), pl, pack.scale, check_status=True)
        _check(o.float().cpu().numpy(), l.cpu().numpy(), oo, lo, pack.name + "/key-chunk")
