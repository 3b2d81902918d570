"""Host planner on general layouts (CPU only): queries and keys as position
ranges of their sequences (cached prefix, key chunks) and paged keys.  The
per-row key limit is checked against the oracle's dense mask of the whole
sequence, the work list against the contiguous plan, and malformed layouts
against their error codes."""
import numpy as np
import pytest

import oracle
import packed_varlen_masked_gb300 as pk
from packed_varlen_masked_gb300 import PKError
import workloads as W


def _pack():
    return W.Pack("g", [[(W.TEXT, 40), (W.IMAGE, 150), (W.TEXT, 9)],
                        [(W.IMAGE, 60), (W.IMAGE, 70)],
                        [(W.TEXT, 33)],
                        [],
                        [(W.TEXT, 20), (W.IMAGE, 300)]], hq=4, hkv=2, d=64)


def _layout_plan(pack, cu_q, cu_k, q_pos0, k_pos0, **kw):
    return pk.plan_layout(cu_q, cu_k, W.seq_segments(pack), pack.hq, pack.hkv, pack.d,
                          q_pos0=q_pos0, k_pos0=k_pos0, num_ctas=16, upload=False, **kw)


def _check_limits(pack, pl, cu_q, cu_k, q_pos0, k_pos0):
    lim = pl.kv_limit()
    cu = pack.cu_seqlens
    pairs = 0
    for s in range(len(cu) - 1):
        nq, nk = int(cu_q[s + 1] - cu_q[s]), int(cu_k[s + 1] - cu_k[s])
        if nq == 0:
            continue
        M = oracle.dense_mask(cu, pack.segments, s)
        rows = M[q_pos0[s]:q_pos0[s] + nq, k_pos0[s]:k_pos0[s] + nk]
        want = np.arange(nk)[None, :] <= lim[cu_q[s]:cu_q[s + 1]][:, None]
        np.testing.assert_array_equal(rows, want)
        pairs += int(rows.sum())
    assert pl.info["visible_pairs"] == pairs


def test_whole_sequences_layout_equals_packed_plan():
    pack = _pack()
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    a = _layout_plan(pack, cu, cu, z, z)
    b = pk.Plan(cu, pack.segments, pack.hq, pack.hkv, pack.d, num_ctas=16, upload=False)
    np.testing.assert_array_equal(a.kv_limit(), b.kv_limit())
    ia, oa = a.items()
    ib, ob = b.items()
    np.testing.assert_array_equal(ia, ib)
    np.testing.assert_array_equal(oa, ob)
    assert a.info == b.info


def test_cached_prefix_limits():
    pack = _pack()
    cu = pack.cu_seqlens
    _, cu_q, q_pos0 = W.prefix_split(pack)
    k_pos0 = np.zeros(len(cu) - 1, np.int32)
    pl = _layout_plan(pack, cu_q, cu, q_pos0, k_pos0)
    assert pl.total_tokens == int(cu_q[-1]) and pl.kv_rows == int(cu[-1])
    _check_limits(pack, pl, cu_q, cu, q_pos0, k_pos0)


@pytest.mark.parametrize("chunk", [32, 97, 128, 256])
def test_key_chunk_limits_and_empty_rows(chunk):
    pack = _pack()
    cu = pack.cu_seqlens
    q_pos0 = np.zeros(len(cu) - 1, np.int32)
    saw_empty = False
    for cu_k, k_pos0, _ in W.key_chunks(pack, chunk):
        pl = _layout_plan(pack, cu, cu_k, q_pos0, k_pos0)
        _check_limits(pack, pl, cu, cu_k, q_pos0, k_pos0)
        lim = pl.kv_limit()
        saw_empty |= bool((lim < 0).any())
        items, _ = pl.items()
        for q_start, q_rows, kv_start, n_kt, n_full, *_ in items.tolist():
            rl = lim[q_start:q_start + q_rows]
            assert n_kt == (1 if rl[-1] < 0 else rl[-1] // 128 + 1)
            assert n_full == min(n_kt, 0 if rl[0] < 0 else (rl[0] + 1) // 128)
            assert (rl[:-1] <= rl[1:]).all(), "limits are monotone inside a tile"
    assert saw_empty


def test_paged_items_address_the_block_table():
    pack = _pack()
    cu = pack.cu_seqlens
    S = len(cu) - 1
    z = np.zeros(S, np.int32)
    table, pool_rows = W.paged_layout(pack, np.random.default_rng(3))
    pg = _layout_plan(pack, cu, cu, z, z, block_table=table, num_kv_rows=len(pool_rows))
    ct = _layout_plan(pack, cu, cu, z, z)
    np.testing.assert_array_equal(pg.kv_limit(), ct.kv_limit())
    ip, _ = pg.items()
    ic, _ = ct.items()
    np.testing.assert_array_equal(np.delete(ip, 2, axis=1), np.delete(ic, 2, axis=1))
    bps = table.shape[1]
    for row_p, row_c in zip(ip.tolist(), ic.tolist()):
        s = int(np.searchsorted(cu, row_c[2], side="right") - 1)
        while cu[s + 1] == cu[s]:
            s += 1
        assert row_p[2] == s * bps
    assert pg.kv_rows == len(pool_rows)
    assert pg.device_bytes >= ct.device_bytes + table.size * 4


def test_paged_prefix_chunk_offsets():
    """Paged keys starting at a block boundary inside the sequence."""
    pack = _pack()
    cu = pack.cu_seqlens
    S = len(cu) - 1
    table, pool_rows = W.paged_layout(pack, np.random.default_rng(4))
    L = np.diff(cu)
    k_pos0 = np.where(L > 128, 128, 0).astype(np.int32)
    nk = L - k_pos0
    cu_k = np.concatenate([[0], np.cumsum(nk)]).astype(np.int32)
    q_pos0 = np.zeros(S, np.int32)
    pl = _layout_plan(pack, cu, cu_k, q_pos0, k_pos0, block_table=table,
                      num_kv_rows=len(pool_rows))
    _check_limits(pack, pl, cu, cu_k, q_pos0, k_pos0)
    items, _ = pl.items()
    starts = {s * table.shape[1] + k_pos0[s] // 128 for s in range(S) if nk[s] > 0}
    assert set(items[:, 2].tolist()) <= starts | {0}


def _err(pack, cu_q, cu_k, q_pos0, k_pos0, segs=None, **kw):
    with pytest.raises(PKError) as ei:
        pk.plan_layout(cu_q, cu_k, W.seq_segments(pack) if segs is None else segs,
                       pack.hq, pack.hkv, pack.d, q_pos0=q_pos0, k_pos0=k_pos0,
                       num_ctas=4, upload=False, **kw)
    return ei.value.status


def test_invalid_layouts():
    pack = W.Pack("v", [[(W.TEXT, 10), (W.IMAGE, 300)], [(W.TEXT, 50)]], hq=2, hkv=1, d=64)
    cu = pack.cu_seqlens  # [0, 310, 360]
    z = np.zeros(2, np.int32)
    E = pk.PK_ERR_INVALID_ARG
    # query range beyond the sequence
    assert _err(pack, cu, cu, np.array([1, 0], np.int32), z) == E
    # key range beyond the sequence
    assert _err(pack, cu, cu, z, np.array([0, 5], np.int32)) == E
    # negative offsets
    assert _err(pack, cu, cu, np.array([-1, 0], np.int32), z) == E
    # segments out of sequence order / not tiling from position 0
    sg = W.seq_segments(pack)
    assert _err(pack, cu, cu, z, z, segs=sg[[1, 0, 2]]) == E
    bad = sg.copy(); bad[1, 1] += 1
    assert _err(pack, cu, cu, z, z, segs=bad) == E
    # contiguous keys: fewer key rows than cu_seqlens_k covers
    assert _err(pack, cu, cu, z, z, num_kv_rows=300) == E
    table, pool_rows = W.paged_layout(pack, np.random.default_rng(0))
    # paged: pool rows not a multiple of the block, block id out of the pool,
    # key range not starting on a block boundary, table too narrow
    assert _err(pack, cu, cu, z, z, block_table=table, num_kv_rows=len(pool_rows) - 1) == E
    t2 = table.copy(); t2[0, 0] = len(pool_rows) // 128
    assert _err(pack, cu, cu, z, z, block_table=t2, num_kv_rows=len(pool_rows)) == E
    cu_k = np.array([0, 300, 350], np.int32)
    assert _err(pack, cu, cu_k, z, np.array([10, 0], np.int32), block_table=table,
                num_kv_rows=len(pool_rows)) == E
    assert _err(pack, cu, cu, z, z, block_table=table[:, :1],
                num_kv_rows=len(pool_rows)) == E
    # queries but no key tensor at all
    assert _err(pack, cu, np.zeros(3, np.int32), z, z, num_kv_rows=0) == E


def test_empty_key_ranges_are_planned_as_masked_rows():
    pack = W.Pack("nk", [[(W.TEXT, 70)], [(W.IMAGE, 200)]], hq=2, hkv=1, d=128)
    cu = pack.cu_seqlens
    cu_k = np.array([0, 0, 200], np.int32)
    z = np.zeros(2, np.int32)
    pl = _layout_plan(pack, cu, cu_k, z, z)
    lim = pl.kv_limit()
    assert (lim[:70] == -1).all() and (lim[70:] == 199).all()
    items, _ = pl.items()
    first = items[items[:, 0] < 70]
    assert (first[:, 3] == 1).all() and (first[:, 4] == 0).all()
