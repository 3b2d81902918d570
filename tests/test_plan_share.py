"""The head-pair cluster schedule (pk_plan_set_kv_share), checked on the
host: it holds exactly the plan's work items, the clusters' offsets cover
them, the loads follow the longest-first rule of the one-CTA schedule, and
plans whose items do not all carry two query heads (or built for a single
CTA) have none and refuse to enable it."""
import numpy as np
import pytest

import packed_varlen_masked_gb300 as pk
import workloads as W

# item columns: q_start, q_rows, kv_start, n_kt, n_full, hq0, hq1, hkv
NKT, NF, H1 = 3, 4, 6


def _cost(it):
    """The planner's relative item cost: per query head one per full key
    tile, 1.3 per partial tile and 3 per unit."""
    per_head = it[NF] + 1.3 * (it[NKT] - it[NF]) + 3.0
    return per_head * (2 if it[H1] >= 0 else 1)


def _plans():
    out = []
    for name in ("cfg_pair", "mixed_resolution", "skewed", "highres_edit"):
        pack = W.CONFIGS[name]()
        plan = pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=152,
                       upload=False)
        plan.requested_ctas = 152
        out.append((name, plan))
    for seed in range(6):
        hq, hkv = [(8, 2), (4, 2), (16, 8), (2, 1)][seed % 4]
        pack = W.random_pack(np.random.default_rng(500 + seed), num_seqs=1 + seed % 5,
                             max_len=2000, hq=hq, hkv=hkv, d=[128, 64][seed % 2],
                             name=f"rnd{seed}")
        ctas = [2, 7, 16, 152, 3, 60][seed]
        plan = pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=ctas,
                       upload=False)
        plan.requested_ctas = ctas
        out.append((pack.name, plan))
    return out


@pytest.mark.parametrize("name,plan", _plans(), ids=lambda x: x if isinstance(x, str) else "")
def test_share_schedule_holds_every_item_once(name, plan):
    # on by default at head_dim 128 wherever the schedule exists, opt-in at 64
    assert plan.kv_share == (plan.head_dim == 128)
    plan.set_kv_share(True)
    assert plan.kv_share
    plan.set_kv_share(False)
    assert not plan.kv_share
    items, _ = plan.items()
    sitems, soffs = plan.share_schedule()
    assert sitems.shape == items.shape
    assert sorted(map(tuple, sitems.tolist())) == sorted(map(tuple, items.tolist()))
    # num_ctas / 2 clusters of the CTAs asked for, at most one per item
    assert len(soffs) - 1 == min(plan.requested_ctas // 2, items.shape[0])
    assert soffs[0] == 0 and soffs[-1] == items.shape[0] and np.all(np.diff(soffs) >= 1)
    assert np.all(sitems[:, H1] >= 0)


@pytest.mark.parametrize("name,plan", _plans(), ids=lambda x: x if isinstance(x, str) else "")
def test_share_schedule_is_longest_first(name, plan):
    sitems, soffs = plan.share_schedule()
    loads = [sum(_cost(it) for it in sitems[a:b]) for a, b in zip(soffs[:-1], soffs[1:])]
    biggest = max(_cost(it) for it in sitems)
    # greedy least-loaded placement: no cluster ends above the lightest by
    # more than one item
    assert max(loads) <= min(loads) + biggest + 1e-9
    for a, b in zip(soffs[:-1], soffs[1:]):  # each cluster takes its items longest first
        c = [_cost(it) for it in sitems[a:b]]
        assert all(x >= y - 1e-9 for x, y in zip(c, c[1:]))


@pytest.mark.parametrize("hq,hkv,d,ctas", [(4, 4, 64, 152), (6, 2, 128, 152), (3, 3, 128, 152),
                                           (6, 2, 64, 152), (8, 2, 128, 1)])
def test_no_share_schedule_without_two_heads_per_item(hq, hkv, d, ctas):
    pack = W.Pack("no-share", [[(W.TEXT, 40), (W.IMAGE, 300)], [(W.IMAGE, 129)]], hq=hq, hkv=hkv,
                  d=d, seed=1)
    plan = pk.Plan(pack.cu_seqlens, pack.segments, hq, hkv, d, num_ctas=ctas, upload=False)
    sitems, soffs = plan.share_schedule()
    assert sitems.shape[0] == 0 and len(soffs) == 1
    assert not plan.kv_share
    with pytest.raises(pk.PKError) as e:
        plan.set_kv_share(True)
    assert e.value.status == pk.PK_ERR_UNSUPPORTED
    plan.set_kv_share(False)  # the one-CTA kernel: always allowed
    assert not plan.kv_share


def test_shards_have_their_own_share_schedule():
    pack = W.mixed_resolution()
    full = pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=152,
                   upload=False)
    seen = []
    for r in range(3):
        sh = full.shard(r, 3, num_ctas=152, upload=False)
        items, _ = sh.items()
        sitems, soffs = sh.share_schedule()
        assert sorted(map(tuple, sitems.tolist())) == sorted(map(tuple, items.tolist()))
        seen += list(map(tuple, sitems.tolist()))
    assert sorted(seen) == sorted(map(tuple, full.items()[0].tolist()))
