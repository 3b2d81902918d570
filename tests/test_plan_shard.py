"""Splitting one pack across ranks (pk_plan_shard), on the host: the ranks'
shares partition the full plan's work items exactly, never split a
(sequence, key/value head) unit, cover every (query row, query head) of the
output exactly once between them, add up to the full plan's useful FLOPs, and
are balanced as longest-first assignment guarantees."""
import collections

import numpy as np
import pytest

import packed_varlen_masked_gb300 as pk
import workloads as W


def _packs():
    rng = np.random.default_rng(77)
    out = [W.tiny_pack(), W.cfg_pair(), W.mixed_resolution(), W.skewed(),
           W.Pack("one-seq", [[(W.TEXT, 300), (W.IMAGE, 1000)]], hq=8, hkv=2, d=128)]
    out += [W.random_pack(rng, int(rng.integers(1, 7)), 900, hq=8, hkv=int(rng.choice([1, 2, 4])),
                          d=128, name=f"rnd{i}") for i in range(6)]
    return out


def _units(plan, items):
    cu = plan._cu_q
    seq = np.searchsorted(cu, items[:, 0], side="right") - 1
    return seq * plan.hkv + items[:, 7]


def _cost(items):
    per_head = items[:, 4] * 1.0 + (items[:, 3] - items[:, 4]) * 1.3 + 3.0
    return np.where(items[:, 6] >= 0, 2.0, 1.0) * per_head


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shards_partition_the_plan(pack, world):
    full = pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=152,
                   upload=False)
    full._cu_q = pack.cu_seqlens
    f_items, _ = full.items()
    key = lambda a: sorted(map(tuple, a.tolist()))
    shards = [full.shard(r, world, num_ctas=152, upload=False) for r in range(world)]
    all_items, owner_units, flops, loads = [], {}, 0.0, []
    cover = collections.Counter()
    for r, sh in enumerate(shards):
        it, offs = sh.items()
        assert offs[-1] == len(it)
        all_items.append(it)
        for u in set(_units(full, it).tolist()) if len(it) else []:
            assert u not in owner_units, "a (sequence, kv head) unit was split"
            owner_units[u] = r
        for row in it.tolist():
            for h in (row[5], row[6]):
                if h >= 0:
                    for t in range(row[0], row[0] + row[1]):
                        cover[(t, h)] += 1
        flops += sh.useful_flops
        loads.append(_cost(it).sum() if len(it) else 0.0)
        assert (sh.kv_limit() == full.kv_limit()).all()
    merged = np.concatenate(all_items) if all_items else np.zeros((0, 8), np.int32)
    assert key(merged) == key(f_items)                       # exact partition
    assert len(cover) == pack.total_tokens * pack.hq and set(cover.values()) == {1}
    assert flops == pytest.approx(full.useful_flops, rel=1e-12)
    # longest-first bound: no rank exceeds the mean load by more than one unit
    unit_cost = collections.defaultdict(float)
    for u, c in zip(_units(full, f_items).tolist(), _cost(f_items).tolist()):
        unit_cost[u] += c
    assert max(loads) <= sum(loads) / world + max(unit_cost.values()) + 1e-9


def test_shard_arguments_are_checked():
    pack = W.tiny_pack()
    full = pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=4,
                   upload=False)
    lib = pk.load()
    import ctypes
    out = ctypes.c_void_p()
    for rank, world in ((0, 0), (2, 2), (-1, 2)):
        assert lib.pk_plan_shard(full.handle, rank, world, 4, ctypes.byref(out)) == pk.PK_ERR_INVALID_ARG
        assert out.value is None
    assert lib.pk_plan_shard(None, 0, 1, 4, ctypes.byref(out)) == pk.PK_ERR_INVALID_ARG
    # more ranks than units: the spare ranks get empty plans
    units = len(pack.seqs) * pack.hkv
    empty = full.shard(units, units + 1, num_ctas=4, upload=False)
    assert empty.info["num_items"] == 0 and empty.useful_flops == 0.0
