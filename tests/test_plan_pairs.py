"""The SM-pair schedule (pk_plan_set_sm_pairs), checked on the host: every
work item's query heads appear once each as a rank of a pair, partners read the same key and
value tiles, a pair visits the larger key-tile count and masks by the
smaller full-tile count, items pair with their neighbours by key-tile count,
and the clusters' offsets cover the pairs."""
from collections import defaultdict

import numpy as np
import pytest

import packed_varlen_masked_gb300 as pk
import workloads as W

# item columns: q_start, q_rows, kv_start, n_kt, n_full, hq0, hq1, hkv
Q0, QR, KV, NKT, NF, H0, H1, HK = range(8)


def _plans():
    out = []
    for name in ("cfg_pair", "mixed_resolution", "skewed"):
        pack = W.CONFIGS[name]()
        out.append((name, pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d,
                                  num_ctas=152, upload=False)))
    for seed in range(6):
        pack = W.random_pack(np.random.default_rng(300 + seed), num_seqs=1 + seed % 5,
                             max_len=2000, hq=8, hkv=2, d=128, name=f"rnd{seed}")
        out.append((pack.name, pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d,
                                       num_ctas=[2, 7, 16, 152][seed % 4], upload=False)))
    return out


def _key(it):
    return (int(it[KV]), int(it[HK]), int(it[H0]), int(it[H1]))


def _one_head_items(items):
    """The plan's items taken one query head at a time, as the pair schedule
    takes them."""
    out = []
    for it in items:
        for h in (it[H0], it[H1]):
            if h < 0:
                continue
            x = it.copy()
            x[H0], x[H1] = h, -1
            out.append(x)
    return np.array(out, dtype=np.int32).reshape(-1, 8)


@pytest.mark.parametrize("name,plan", _plans(), ids=lambda x: x if isinstance(x, str) else "")
def test_pairs_cover_every_item_once(name, plan):
    items = _one_head_items(plan.items()[0])
    pitems, poffs = plan.pairs()
    npairs = pitems.shape[0] // 2
    assert npairs > 0
    assert poffs[0] == 0 and poffs[-1] == npairs and np.all(np.diff(poffs) >= 0)
    assert len(poffs) - 1 == min(plan.info["num_ctas"] // 2, npairs)
    singles = {tuple(int(x) for x in it) for it in items}
    assert len(singles) == items.shape[0]
    seen = set()
    by_key = defaultdict(list)
    for it in items:
        by_key[_key(it)].append(it)
    for i in range(npairs):
        a, b = pitems[2 * i], pitems[2 * i + 1]
        assert _key(a) == _key(b) and a[H1] == -1
        assert a[NKT] == b[NKT] and a[NF] == b[NF]
        assert a[QR] > 0
        for r in (a, b):
            if r[QR] == 0:  # no partner: loads the leader's rows, writes none
                assert r[Q0] == a[Q0]
                continue
            orig = [it for it in by_key[_key(r)] if it[Q0] == r[Q0]]
            assert len(orig) == 1
            o = orig[0]
            assert o[QR] == r[QR] and o[NKT] <= r[NKT] and o[NF] >= r[NF]
            t = (int(o[Q0]), int(o[HK]), int(o[H0]), int(o[H1]))
            assert t not in seen
            seen.add(t)
        if b[QR] > 0:
            oa = [it for it in by_key[_key(a)] if it[Q0] == a[Q0]][0]
            ob = [it for it in by_key[_key(b)] if it[Q0] == b[Q0]][0]
            assert a[NKT] == max(oa[NKT], ob[NKT]) and a[NF] == min(oa[NF], ob[NF])
    assert len(seen) == items.shape[0]


@pytest.mark.parametrize("name,plan", _plans()[:3], ids=lambda x: x if isinstance(x, str) else "")
def test_pairing_by_key_tile_count_keeps_the_masked_waste_small(name, plan):
    """Neighbours by key-tile count: the extra (fully masked) tiles a pair
    visits are those of sorted neighbours, a few percent of the work."""
    items = _one_head_items(plan.items()[0])
    pitems, _ = plan.pairs()
    by_key = defaultdict(list)
    for it in items:
        by_key[_key(it)].append(int(it[NKT]))
    best = 0
    for ks in by_key.values():
        ks.sort()
        for i in range(0, len(ks), 2):
            best += (2 * ks[i + 1] - ks[i] - ks[i + 1]) if i + 1 < len(ks) else ks[i]
    # the pair schedule's waste, rebuilt from the originals, equals the sorted pairing's
    orig = {(int(it[Q0]), _key(it)): int(it[NKT]) for it in items}
    waste = 0
    for i in range(pitems.shape[0] // 2):
        a, b = pitems[2 * i], pitems[2 * i + 1]
        na = orig[(int(a[Q0]), _key(a))]
        if b[QR] == 0:
            waste += int(a[NKT])
            continue
        nb = orig[(int(b[Q0]), _key(b))]
        waste += 2 * int(a[NKT]) - na - nb
    assert waste == best
    assert waste <= 0.06 * sum(int(it[NKT]) for it in items) + 1


def test_plans_without_a_pair_schedule():
    lib = pk.load()
    assert lib.pk_plan_set_sm_pairs(None, 1) == pk.PK_ERR_INVALID_ARG
    p64 = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 64, num_ctas=8, upload=False)
    assert p64.pairs()[0].shape[0] == 0
    assert lib.pk_plan_set_sm_pairs(p64.handle, 1) == pk.PK_ERR_UNSUPPORTED
    assert lib.pk_plan_set_sm_pairs(p64.handle, 0) == pk.PK_OK
    one = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 128, num_ctas=1, upload=False)
    assert one.pairs()[0].shape[0] == 0
    with pytest.raises(pk.PKError):
        one.set_sm_pairs(True)
    two = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 128, num_ctas=2, upload=False)
    assert two.set_sm_pairs(True) is two
    assert lib.pk_plan_get_pairs(None, None, None, None, 0, None, 0) == pk.PK_ERR_INVALID_ARG


def test_shards_have_pair_schedules_of_their_own_items():
    pack = W.CONFIGS["mixed_resolution"]()
    full = pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=152,
                   upload=False)
    total = 0
    for r in range(3):
        sh = full.shard(r, 3, num_ctas=152, upload=False)
        items = _one_head_items(sh.items()[0])
        pitems, _ = sh.pairs()
        rows = {(int(it[Q0]), int(it[H0])) for it in items}
        prow = {(int(it[Q0]), int(it[H0])) for it in pitems if it[QR] > 0}
        assert rows == prow
        total += items.shape[0]
    assert total == _one_head_items(full.items()[0]).shape[0]
