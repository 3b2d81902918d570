"""Pins for the fp64 oracle, each against something other than the oracle:
library special cases (textbook causal / full attention), closed forms, a
hand-derived mask fixture and invariants of the method."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pack(seqs, hq=2, hkv=2, d=16, seed=0, q_mult=1.0):
    return W.Pack("t", seqs, hq=hq, hkv=hkv, d=d, seed=seed, q_mult=q_mult)


def _run(pack, q=None, k=None, v=None, rows=None):
    if q is None:
        q, k, v = W.make_qkv(pack)
    return oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq,
                            pack.hkv, pack.d, pack.scale, rows=rows)


def _sdpa(q, k, v, scale, causal):
    """torch SDPA in fp64 on [L,H,d] slices (MHA); returns out [L,H,d] and the
    per-row log-sum-exp from torch.logsumexp of the (masked) score matrix."""
    qd = q.double().permute(1, 0, 2)
    kd = k.double().permute(1, 0, 2)
    vd = v.double().permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(
        qd, kd, vd, is_causal=causal, scale=scale)
    s = torch.matmul(qd, kd.transpose(1, 2)) * scale
    if causal:
        L = s.shape[-1]
        s = s.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
    return o.permute(1, 0, 2).numpy(), torch.logsumexp(s, dim=-1).numpy()


def test_bf16_decoding():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x3F81) == 1.0078125
    assert oracle.bf16_to_double(0x0000) == 0.0
    assert oracle.bf16_to_double(0x4049) == 3.140625


def test_validate_rejects_bad_descriptors():
    ok_cu, ok_sg = [0, 3, 5], [(0, 2, 0), (2, 1, 1), (3, 2, 1)]
    assert oracle.validate(ok_cu, ok_sg) == 0
    assert oracle.validate([1, 3, 5], ok_sg) != 0          # cu[0] != 0
    assert oracle.validate([0, 5, 3], ok_sg) != 0          # decreasing
    assert oracle.validate(ok_cu, [(0, 2, 0), (2, 1, 1)]) != 0           # gap
    assert oracle.validate(ok_cu, [(0, 2, 0), (2, 2, 1), (4, 1, 1)]) != 0  # crosses seq
    assert oracle.validate(ok_cu, [(0, 2, 0), (2, 1, 7), (3, 2, 1)]) != 0  # bad type
    assert oracle.validate([0, 0, 2], [(0, 2, 1)]) == 0    # empty sequence


def _read_golden_masks():
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "mask_small.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("seq"):
                segs = []
                for tok in line.split()[1:]:
                    segs.append((W.TEXT if tok[0] == "T" else W.IMAGE, int(tok[1:])))
                cur = (segs, [])
                blocks.append(cur)
            else:
                cur[1].append([c == "1" for c in line])
    return blocks


def test_dense_mask_matches_hand_derived_fixture():
    blocks = _read_golden_masks()
    pack = _pack([b[0] for b in blocks])
    for s, (_, rows) in enumerate(blocks):
        M = oracle.dense_mask(pack.cu_seqlens, pack.segments, s)
        assert M.tolist() == rows


def test_all_text_equals_textbook_causal_attention():
    pack = _pack([[(W.TEXT, 7)], [(W.TEXT, 3), (W.TEXT, 20)], [(W.TEXT, 1)]],
                 hq=3, hkv=3, d=32, seed=5)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    cu = pack.cu_seqlens
    for s in range(len(cu) - 1):
        b, e = cu[s], cu[s + 1]
        o_ref, lse_ref = _sdpa(q[b:e], k[b:e], v[b:e], pack.scale, causal=True)
        np.testing.assert_allclose(out[b:e], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, b:e], lse_ref, rtol=0, atol=1e-12)


def test_single_image_segment_equals_full_attention():
    pack = _pack([[(W.IMAGE, 19)], [(W.IMAGE, 5)]], hq=2, hkv=2, d=16, seed=9)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    cu = pack.cu_seqlens
    for s in range(2):
        b, e = cu[s], cu[s + 1]
        o_ref, lse_ref = _sdpa(q[b:e], k[b:e], v[b:e], pack.scale, causal=False)
        np.testing.assert_allclose(out[b:e], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, b:e], lse_ref, rtol=0, atol=1e-12)


def test_mixed_rows_equal_prefix_attention():
    """Text row i attends exactly keys [0, i]; an image row of segment
    [a, b) attends exactly keys [0, b): each is full attention (SDPA, no
    mask) over that key prefix."""
    seqs = [[(W.TEXT, 5), (W.IMAGE, 9), (W.TEXT, 3), (W.IMAGE, 4), (W.IMAGE, 6)]]
    pack = _pack(seqs, hq=2, hkv=2, d=16, seed=11)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    pos = 0
    for typ, n in seqs[0]:
        for i in range(pos, pos + n):
            lim = i if typ == W.TEXT else pos + n - 1
            o_ref, lse_ref = _sdpa(q[i:i + 1], k[:lim + 1], v[:lim + 1], pack.scale, False)
            np.testing.assert_allclose(out[i], o_ref[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[:, i], lse_ref[:, 0], rtol=0, atol=1e-12)
        pos += n


def test_first_text_row_closed_form():
    pack = _pack([[(W.TEXT, 4), (W.IMAGE, 4)]], hq=2, hkv=1, d=8, seed=3)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    for h in range(2):
        np.testing.assert_array_equal(out[0, h], vd[0, 0])
        assert abs(lse[h, 0] - pack.scale * float(qd[0, h] @ kd[0, 0])) < 1e-14


def test_two_key_closed_form():
    """Row 1 of a text sequence: softmax over two scores, written out."""
    pack = _pack([[(W.TEXT, 2)]], hq=1, hkv=1, d=4, seed=0)
    q = torch.tensor([[[1.0, 0.0, 0.5, 0.0]], [[0.0, 2.0, 0.0, -1.0]]]).bfloat16()
    k = torch.tensor([[[1.0, 1.0, 0.0, 0.0]], [[0.0, 1.0, 2.0, 1.0]]]).bfloat16()
    v = torch.tensor([[[1.0, 2.0, 3.0, 4.0]], [[-1.0, 0.0, 1.0, 0.5]]]).bfloat16()
    out, lse = _run(pack, q, k, v)
    s0 = 0.5 * (0 * 1 + 2 * 1 + 0 * 0 + -1 * 0)   # scale = 1/sqrt(4)
    s1 = 0.5 * (0 * 0 + 2 * 1 + 0 * 2 + -1 * 1)
    z = math.exp(s0) + math.exp(s1)
    p0, p1 = math.exp(s0) / z, math.exp(s1) / z
    want = [p0 * 1 + p1 * -1, p0 * 2 + p1 * 0, p0 * 3 + p1 * 1, p0 * 4 + p1 * 0.5]
    np.testing.assert_allclose(out[1, 0], want, rtol=0, atol=1e-14)
    assert abs(lse[0, 1] - math.log(z)) < 1e-14


def test_constant_v_returns_v():
    pack = _pack([[(W.TEXT, 6), (W.IMAGE, 10), (W.TEXT, 2)], [(W.IMAGE, 7)]],
                 hq=4, hkv=2, d=8, seed=2)
    q, k, v = W.make_qkv(pack)
    v = torch.full_like(v, 0.375)
    out, _ = _run(pack, q, k, v)
    np.testing.assert_allclose(out, 0.375, rtol=0, atol=1e-14)


def test_packed_equals_each_sequence_alone():
    seqs = [[(W.TEXT, 5), (W.IMAGE, 7)], [(W.IMAGE, 4), (W.TEXT, 3)], [(W.TEXT, 9)]]
    pack = _pack(seqs, hq=4, hkv=2, d=16, seed=4)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    cu = pack.cu_seqlens
    for s in range(3):
        b, e = cu[s], cu[s + 1]
        alone = _pack([seqs[s]], hq=4, hkv=2, d=16)
        o1, l1 = _run(alone, q[b:e], k[b:e], v[b:e])
        np.testing.assert_array_equal(out[b:e], o1)
        np.testing.assert_array_equal(lse[:, b:e], l1)


def test_permuting_sequences_permutes_outputs():
    seqs = [[(W.TEXT, 5), (W.IMAGE, 7)], [(W.IMAGE, 4), (W.TEXT, 3)], [(W.TEXT, 9)]]
    pack = _pack(seqs, hq=2, hkv=1, d=16, seed=6)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    perm = [2, 0, 1]
    cu = pack.cu_seqlens
    idx = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in perm])
    packp = _pack([seqs[s] for s in perm], hq=2, hkv=1, d=16)
    op, lp = _run(packp, q[idx], k[idx], v[idx])
    np.testing.assert_array_equal(op, out[idx])
    np.testing.assert_array_equal(lp, lse[:, idx])


def test_gqa_equals_mha_with_repeated_kv_heads():
    seqs = [[(W.TEXT, 6), (W.IMAGE, 8), (W.TEXT, 2)], [(W.IMAGE, 5), (W.IMAGE, 3)]]
    pack = _pack(seqs, hq=6, hkv=2, d=16, seed=8)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    mha = _pack(seqs, hq=6, hkv=6, d=16)
    o2, l2 = _run(mha, q, k.repeat_interleave(3, dim=1), v.repeat_interleave(3, dim=1))
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(lse, l2)


def test_softmax_weights_sum_to_one_on_the_mask():
    """With v[j] = e_j the output row is the softmax row itself: it sums to
    one, is zero exactly where the dense mask is zero, and each weight is
    exp(s_ij - lse_i)."""
    seqs = [[(W.TEXT, 3), (W.IMAGE, 5), (W.TEXT, 2), (W.IMAGE, 3)]]
    pack = _pack(seqs, hq=1, hkv=1, d=16, seed=12)
    L = 13
    q, k, _ = W.make_qkv(pack)
    v = torch.zeros(L, 1, 16)
    v[torch.arange(L), 0, torch.arange(L)] = 1.0
    out, lse = _run(pack, q, k, v.bfloat16())
    P = out[:, 0, :L]
    M = oracle.dense_mask(pack.cu_seqlens, pack.segments, 0)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-14)
    assert ((P > 0) == M).all()
    s = (q.double()[:, 0] @ k.double()[:, 0].T).numpy() * pack.scale
    np.testing.assert_allclose(P[M], np.exp(s - lse[0][:, None])[M], rtol=1e-13, atol=0)


def test_permuting_kv_inside_an_image_segment():
    """Rows that see a whole image segment are invariant to permuting the
    keys/values inside it; the causal text rows inside it are not."""
    seqs = [[(W.TEXT, 4), (W.IMAGE, 12), (W.TEXT, 3)]]
    pack = _pack(seqs, hq=2, hkv=2, d=16, seed=13)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    perm = np.arange(19)
    perm[4:16] = np.random.default_rng(0).permutation(np.arange(4, 16))
    k2, v2 = k.clone(), v.clone()
    k2[4:16], v2[4:16] = k[perm[4:16]], v[perm[4:16]]
    q2 = q.clone()  # the queries stay put; only the keys/values move
    o2, l2 = _run(pack, q2, k2, v2)
    np.testing.assert_allclose(o2[4:], out[4:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2[:, 4:], lse[:, 4:], rtol=0, atol=1e-12)


def _closed_form_pairs(pack):
    """sum over text rows of (i + 1) plus, over image rows, the end of their
    own segment (both sequence-relative)."""
    total = 0
    for seq in pack.seqs:
        pos = 0
        for typ, n in seq:
            if typ == W.TEXT:
                total += sum(i + 1 for i in range(pos, pos + n))
            else:
                total += n * (pos + n)
            pos += n
    return total


@pytest.mark.parametrize("name", ["tiny", "cfg_pair", "highres_edit", "skewed",
                                  "mixed_resolution"])
def test_visible_pairs_closed_form(name):
    pack = W.CONFIGS[name]()
    assert oracle.visible_pairs(pack.cu_seqlens, pack.segments) == _closed_form_pairs(pack)


def test_visible_pairs_printed_values():
    assert oracle.visible_pairs(W.tiny_pack().cu_seqlens, W.tiny_pack().segments) == 79512
    p = W.cfg_pair()
    assert oracle.visible_pairs(p.cu_seqlens, p.segments) == 34653332
    p = W.highres_edit()
    assert oracle.visible_pairs(p.cu_seqlens, p.segments) == 918618368


def test_row_sampled_call_equals_full_call():
    pack = W.random_pack(np.random.default_rng(3), 5, 40, hq=4, hkv=2, d=16)
    q, k, v = W.make_qkv(pack)
    out, lse = _run(pack, q, k, v)
    rows = np.array([0, 7, pack.total_tokens - 1, 13, 7], dtype=np.int32)
    o2, l2 = _run(pack, q, k, v, rows=rows)
    np.testing.assert_array_equal(o2, out[rows])
    np.testing.assert_array_equal(l2, lse[:, rows])


@pytest.mark.parametrize("name", ["tiny", "cfg_pair"])
def test_row_keys_are_mask_row_sums_and_closed_form(name):
    """Per-row visible keys: a text row at position x of its sequence sees
    x + 1 keys, an image row sees every key up to its segment's end; they sum
    to the pinned pair count."""
    pack = W.CONFIGS[name]()
    n = oracle.row_keys(pack.cu_seqlens, pack.segments)
    want = np.zeros(pack.total_tokens, np.int64)
    cu = pack.cu_seqlens
    for s, seq in enumerate(pack.seqs):
        pos = 0
        for typ, ln in seq:
            for x in range(pos, pos + ln):
                want[cu[s] + x] = (pos + ln) if typ == W.IMAGE else x + 1
            pos += ln
    np.testing.assert_array_equal(n, want)
    assert int(n.sum()) == oracle.visible_pairs(cu, pack.segments)
    if name == "tiny":
        for s in range(len(cu) - 1):
            M = oracle.dense_mask(cu, pack.segments, s)
            np.testing.assert_array_equal(n[cu[s]:cu[s + 1]], M.sum(axis=1))


def test_brute_force_python_loops_on_a_tiny_pack():
    """A second, independent implementation: plain Python loops over the
    mask rule as stated (text causal; an image token also sees its whole own
    segment; nothing across sequences), fp64 math.exp, on a tiny pack with
    adjacent image segments and GQA.  The oracle must agree to 1e-12."""
    import math
    seqs = [[(W.TEXT, 5), (W.IMAGE, 7), (W.IMAGE, 4), (W.TEXT, 3)], [(W.IMAGE, 6)], [(W.TEXT, 9)]]
    pack = W.Pack("brute", seqs, hq=4, hkv=2, d=8, seed=77)
    q, k, v = W.make_qkv(pack)
    qf, kf, vf = q.double().numpy(), k.double().numpy(), v.double().numpy()
    T, group = pack.total_tokens, pack.hq // pack.hkv
    # (sequence, segment index, type, segment start, segment end) per token
    info = []
    for s, seq in enumerate(pack.seqs):
        pos = 0
        for gi, (typ, n) in enumerate(seq):
            for _ in range(n):
                info.append((s, gi, typ, pos, pos + n))
            pos += n
    start_of = {}
    t0 = 0
    for s, seq in enumerate(pack.seqs):
        start_of[s] = t0
        t0 += sum(n for _, n in seq)
    out = np.zeros((T, pack.hq, pack.d))
    lse = np.zeros((pack.hq, T))
    for i in range(T):
        si, gi, ti, _, _ = info[i]
        for h in range(pack.hq):
            g = h // group
            keys = []
            for j in range(T):
                sj, gj, _, _, _ = info[j]
                if sj != si:
                    continue
                if j <= i or (ti == W.IMAGE and gj == gi):
                    keys.append(j)
            sc = [pack.scale * sum(qf[i, h, c] * kf[j, g, c] for c in range(pack.d)) for j in keys]
            mx = max(sc)
            z = sum(math.exp(x - mx) for x in sc)
            lse[h, i] = mx + math.log(z)
            for c in range(pack.d):
                out[i, h, c] = sum(math.exp(x - lse[h, i]) * vf[j, g, c] for x, j in zip(sc, keys))
    o, l = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv, pack.d,
                            pack.scale)
    np.testing.assert_allclose(o, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, lse, rtol=0, atol=1e-12)
