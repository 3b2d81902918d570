"""Pins for the oracle's general entry (queries and keys as position ranges
of their sequences, contiguous or paged keys) and for the LSE merge.  Each is
checked against the pinned packed-attention oracle or a closed form."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _pack():
    return W.Pack("g", [[(W.TEXT, 40), (W.IMAGE, 150), (W.TEXT, 9)],
                        [(W.IMAGE, 60), (W.IMAGE, 70)],
                        [(W.TEXT, 33)],
                        [(W.TEXT, 20), (W.IMAGE, 200)]], hq=4, hkv=2, d=32, seed=21)


def _full(pack, q, k, v):
    return oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                            pack.d, pack.scale)


def test_general_with_whole_sequences_is_packed_attention():
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    cu = pack.cu_seqlens
    S = len(cu) - 1
    zeros = np.zeros(S, np.int32)
    o1, l1 = oracle.attention_general(q, k, v, cu, cu, zeros, zeros, W.seq_segments(pack),
                                      pack.hq, pack.hkv, pack.d, pack.scale)
    o0, l0 = _full(pack, q, k, v)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_cached_prefix_queries_equal_rows_of_full_attention():
    """Image queries over the whole sequence's keys (text prefix handed over)
    give exactly the image rows of the packed attention."""
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    cu = pack.cu_seqlens
    o, l = oracle.attention_general(q[rows], k, v, cu_q, cu, q_pos0, np.zeros(len(cu) - 1, np.int32),
                                    W.seq_segments(pack), pack.hq, pack.hkv, pack.d, pack.scale)
    o0, l0 = _full(pack, q, k, v)
    np.testing.assert_array_equal(o, o0[rows])
    np.testing.assert_array_equal(l, l0[:, rows])


def test_paged_keys_equal_contiguous_keys():
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    table, pool_rows = W.paged_layout(pack, np.random.default_rng(5))
    kp = torch.zeros(len(pool_rows), pack.hkv, pack.d, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    src = torch.as_tensor(np.maximum(pool_rows, 0))
    kp[:] = k[src]
    vp[:] = v[src]
    kp[torch.as_tensor(pool_rows < 0)] = 77.0  # unused pool rows hold junk
    cu = pack.cu_seqlens
    zeros = np.zeros(len(cu) - 1, np.int32)
    o, l = oracle.attention_general(q, kp, vp, cu, cu, zeros, zeros, W.seq_segments(pack),
                                    pack.hq, pack.hkv, pack.d, pack.scale, block_table=table)
    o0, l0 = _full(pack, q, k, v)
    np.testing.assert_array_equal(o, o0)
    np.testing.assert_array_equal(l, l0)


def _chunked(pack, q, k, v, chunk):
    """Attention over key chunks [c*chunk, (c+1)*chunk) of every sequence,
    one general call per chunk index; returns the stacked parts."""
    cu = pack.cu_seqlens
    S = len(cu) - 1
    o_parts, l_parts = [], []
    for cu_k, k_pos0, rows in W.key_chunks(pack, chunk):
        idx = torch.as_tensor(rows)
        o, l = oracle.attention_general(q, k[idx], v[idx], cu, cu_k, np.zeros(S, np.int32), k_pos0,
                                        W.seq_segments(pack), pack.hq, pack.hkv, pack.d, pack.scale)
        o_parts.append(o)
        l_parts.append(l)
    return np.stack(o_parts), np.stack(l_parts)


@pytest.mark.parametrize("chunk", [32, 97, 128])
def test_key_chunks_merged_by_lse_equal_full_attention(chunk):
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    o_parts, l_parts = _chunked(pack, q, k, v, chunk)
    assert np.isneginf(l_parts).any(), "some rows see no key of some chunk"
    o_empty = o_parts[np.broadcast_to(np.isneginf(l_parts).transpose(0, 2, 1)[..., None], o_parts.shape)]
    assert (o_empty == 0).all()
    o, l = oracle.lse_merge(o_parts, l_parts)
    o0, l0 = _full(pack, q, k, v)
    np.testing.assert_allclose(o, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, l0, rtol=0, atol=1e-12)


def test_lse_merge_closed_forms():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((1, 5, 3, 4))
    l = rng.standard_normal((1, 3, 5))
    om, lm = oracle.lse_merge(o, l)
    np.testing.assert_array_equal(om, o[0])
    np.testing.assert_array_equal(lm, l[0])
    # two identical parts: same output, lse + ln 2
    om, lm = oracle.lse_merge(np.concatenate([o, o]), np.concatenate([l, l]))
    np.testing.assert_allclose(om, o[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lm, l[0] + math.log(2.0), rtol=0, atol=1e-15)
    # a -inf part contributes nothing; all -inf gives zeros and -inf
    l2 = np.concatenate([l, np.full_like(l, -np.inf)])
    om, lm = oracle.lse_merge(np.concatenate([o, 5 + o]), l2)
    np.testing.assert_array_equal(om, o[0])
    om, lm = oracle.lse_merge(o, np.full_like(l, -np.inf))
    assert (om == 0).all() and np.isneginf(lm).all()
    # two parts, written out
    o2 = rng.standard_normal((2, 1, 1, 2))
    l2 = np.array([[[0.3]], [[-1.1]]])
    om, lm = oracle.lse_merge(o2, l2)
    z = math.exp(0.3) + math.exp(-1.1)
    want = (math.exp(0.3) * o2[0, 0, 0] + math.exp(-1.1) * o2[1, 0, 0]) / z
    np.testing.assert_allclose(om[0, 0], want, rtol=0, atol=1e-15)
    assert abs(lm[0, 0] - math.log(z)) < 1e-15
