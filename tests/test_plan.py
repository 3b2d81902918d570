"""Host planner (CPU only): the per-token key limit and the tile classes
against the oracle's dense mask, work coverage, schedule balance and
argument validation."""
import numpy as np
import pytest

import oracle
import packed_varlen_masked_gb300 as pk
from packed_varlen_masked_gb300 import PKError
import workloads as W


def _plan(pack, num_ctas=16):
    return pk.Plan(pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d,
                   num_ctas=num_ctas, upload=False)


def _packs():
    rng = np.random.default_rng(7)
    packs = [W.tiny_pack()]
    for i in range(12):
        packs.append(W.random_pack(rng, int(rng.integers(1, 6)), int(rng.choice([40, 300, 700])),
                                   hq=int(rng.choice([2, 6, 8])), hkv=2, d=64, name=f"r{i}"))
    packs.append(W.Pack("edges", [[(W.TEXT, 1)], [], [(W.IMAGE, 1)], [(W.IMAGE, 128)],
                                  [(W.TEXT, 128), (W.IMAGE, 129)], [(W.IMAGE, 255), (W.TEXT, 1)]],
                        hq=4, hkv=4, d=128))
    return packs


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
def test_kv_limit_is_the_dense_mask_prefix(pack):
    """Every row of the dense mask is exactly the key prefix [0, kv_limit]
    (the limit is an index into the row's own key range)."""
    lim = _plan(pack).kv_limit()
    cu = pack.cu_seqlens
    for s in range(len(cu) - 1):
        b, e = int(cu[s]), int(cu[s + 1])
        if e == b:
            continue
        M = oracle.dense_mask(cu, pack.segments, s)
        L = e - b
        want = np.arange(L)[None, :] <= lim[b:e][:, None]
        np.testing.assert_array_equal(M, want)


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
def test_tile_classes_against_dense_mask(pack):
    pl = _plan(pack)
    items, offs = pl.items()
    cu = pack.cu_seqlens
    masks = {}
    seen = set()
    for q_start, q_rows, kv_start, n_kt, n_full, hq0, hq1, hkv in items.tolist():
        s = int(np.searchsorted(cu, kv_start, side="right") - 1)
        while cu[s + 1] == cu[s]:
            s += 1
        assert cu[s] == kv_start
        if s not in masks:
            masks[s] = oracle.dense_mask(cu, pack.segments, s)
        M = masks[s]
        L = M.shape[0]
        r0 = q_start - kv_start
        assert 1 <= q_rows <= 128 and r0 % 128 == 0 and r0 + q_rows == min(r0 + 128, L)
        rows = M[r0:r0 + q_rows]
        n_tiles_total = (L + 127) // 128
        for kt in range(n_tiles_total):
            blk = rows[:, kt * 128:(kt + 1) * 128]
            full_width = blk.shape[1] == 128
            if kt < n_full:
                assert full_width and blk.all(), "full tile must be entirely visible"
            elif kt < n_kt:
                assert blk.any() and not (full_width and blk.all()), "partial tile"
            else:
                assert not blk.any(), "skipped tile must be entirely masked"
        group = pack.hq // pack.hkv
        for h in (hq0, hq1):
            if h < 0:
                continue
            assert h // group == hkv
            key = (q_start, h)
            assert key not in seen
            seen.add(key)
    # every (query tile, query head) exactly once
    n_tiles = sum((int(cu[s + 1] - cu[s]) + 127) // 128 for s in range(len(cu) - 1))
    assert len(seen) == n_tiles * pack.hq
    assert offs[0] == 0 and offs[-1] == len(items) and np.all(np.diff(offs) >= 0)


def test_pair_slots_share_kv_head_and_odd_groups_leave_slot_empty():
    pack = W.Pack("g3", [[(W.TEXT, 10), (W.IMAGE, 300)]], hq=6, hkv=2, d=64)
    items, _ = _plan(pack).items()
    single = items[items[:, 6] < 0]
    assert len(single) > 0 and (single[:, 5] % 3 == 2).all()
    paired = items[items[:, 6] >= 0]
    assert (paired[:, 6] == paired[:, 5] + 1).all()


def test_visible_pairs_and_flops_match_oracle():
    for name in ["tiny", "cfg_pair", "skewed"]:
        pack = W.CONFIGS[name]()
        info = _plan(pack, 152).info
        vp = oracle.visible_pairs(pack.cu_seqlens, pack.segments)
        assert info["visible_pairs"] == vp
        assert info["useful_flops"] == 4.0 * pack.d * pack.hq * vp


def test_schedule_balance_and_longest_first():
    pack = W.skewed()
    pl = _plan(pack, 152)
    items, offs = pl.items()
    cost = np.where(items[:, 6] >= 0, 2.0, 1.0) * (items[:, 4] + 1.3 * (items[:, 3] - items[:, 4]) + 3.0)
    loads = np.array([cost[offs[c]:offs[c + 1]].sum() for c in range(len(offs) - 1)])
    # greedy LPT bound: max load <= mean + largest item
    assert loads.max() <= loads.mean() + cost.max() + 1e-9
    for c in range(len(offs) - 1):
        seg = cost[offs[c]:offs[c + 1]]
        assert np.all(np.diff(seg) <= 1e-9), "each CTA runs its items longest first"


def test_grid_is_capped_by_items():
    pack = W.Pack("one", [[(W.TEXT, 5)]], hq=2, hkv=1, d=64)
    info = _plan(pack, 152).info
    assert info["num_items"] == 1 and info["num_ctas"] == 1


def test_empty_pack():
    pack = W.Pack("empty", [[], []], hq=2, hkv=1, d=64)
    pl = _plan(pack, 152)
    assert pl.info["num_items"] == 0 and pl.info["total_tokens"] == 0


@pytest.mark.parametrize("cu,segs,hq,hkv,d,code", [
    ([0, 4], [(0, 4, 0)], 4, 3, 64, pk.PK_ERR_INVALID_ARG),        # hq % hkv
    ([0, 4], [(0, 4, 0)], 4, 2, 96, pk.PK_ERR_UNSUPPORTED),        # head_dim
    ([1, 4], [(1, 3, 0)], 4, 2, 64, pk.PK_ERR_INVALID_ARG),        # cu[0] != 0
    ([0, 4, 2], [(0, 4, 0)], 4, 2, 64, pk.PK_ERR_INVALID_ARG),     # decreasing
    ([0, 4], [(0, 3, 0)], 4, 2, 64, pk.PK_ERR_INVALID_ARG),        # segments short
    ([0, 4], [(0, 2, 0), (2, 3, 1)], 4, 2, 64, pk.PK_ERR_INVALID_ARG),  # crosses end
    ([0, 4], [(0, 4, 2)], 4, 2, 64, pk.PK_ERR_INVALID_ARG),        # bad type
    ([0, 4], [(0, 2, 0), (3, 2, 1)], 4, 2, 64, pk.PK_ERR_INVALID_ARG),  # gap
    ([0, 4], [(0, 4, 0), (4, 1, 0)], 4, 2, 64, pk.PK_ERR_INVALID_ARG),  # extra segment
    ([0, 4], [(0, 0, 0), (0, 4, 0)], 4, 2, 64, pk.PK_ERR_INVALID_ARG),  # empty segment
])
def test_invalid_descriptors(cu, segs, hq, hkv, d, code):
    with pytest.raises(PKError) as ei:
        pk.Plan(cu, segs, hq, hkv, d, num_ctas=4, upload=False)
    assert ei.value.status == code


def test_boundary_tile_rows_are_whole_mask_boundary_tiles():
    """The full-size parity sample of mask-boundary tiles: whole 128-row
    query tiles, each holding a segment's first or last row or a sequence's
    last row, and the tiles in which a row's key limit changes shape."""
    for name in ["mixed_resolution", "skewed", "cfg_pair"]:
        pack = W.CONFIGS[name]()
        rows = W.boundary_tile_rows(pack, 1536)
        cu = pack.cu_seqlens
        assert 0 < len(rows) <= 1536 and np.all(np.diff(rows) > 0)
        seq = np.searchsorted(cu, rows, side="right") - 1
        edges = set()
        for s in range(len(cu) - 1):
            edges.add(int(cu[s + 1]) - 1)
        for st, n, _ in pack.segments:
            edges.update((int(st), int(st + n - 1)))
        tiles = {}
        for r, s in zip(rows.tolist(), seq.tolist()):
            t0 = int(cu[s]) + (r - int(cu[s])) // 128 * 128
            tiles.setdefault((s, t0), []).append(r)
        for (s, t0), rs in tiles.items():
            t1 = min(t0 + 128, int(cu[s + 1]))
            assert rs == list(range(t0, t1)), "a sampled tile is whole"
            assert any(t0 <= e < t1 for e in edges), "it holds a segment or sequence edge"
