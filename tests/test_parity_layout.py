"""GPU parity on general layouts: queries and keys as position ranges of
their sequences (cached text prefix, ring-style key chunks) and paged keys,
through the C ABI, against the fp64 oracle's general entry on the same
seeded inputs, under the rule of parity_tol.py; rows that see no key of
their range must come back as out = 0 and lse = -inf exactly."""
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


def _run(pl, q, k, v, scale):
    out, lse = pk.attn_fwd(q.cuda(), k.cuda(), v.cuda(), pl, scale, check_status=True)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _packs():
    return [
        W.Pack("mixed", [[(W.TEXT, 40), (W.IMAGE, 300), (W.TEXT, 9)],
                         [(W.IMAGE, 200), (W.IMAGE, 130)],
                         [(W.TEXT, 33)],
                         [],
                         [(W.TEXT, 77), (W.IMAGE, 513)]], hq=8, hkv=2, d=128, seed=31),
        W.Pack("d64-g3", [[(W.TEXT, 129), (W.IMAGE, 256)], [(W.TEXT, 1), (W.IMAGE, 700)]],
               hq=6, hkv=2, d=64, seed=32),
    ]


def _pool(pack, k, v, seed):
    """Keys/values scattered into a shuffled 128-row block pool; pool rows no
    sequence owns hold large junk that must never be read."""
    table, pool_rows = W.paged_layout(pack, np.random.default_rng(seed))
    src = torch.as_tensor(np.maximum(pool_rows, 0))
    kp, vp = k[src].clone(), v[src].clone()
    junk = torch.as_tensor(pool_rows < 0)
    kp[junk] = 50.0
    vp[junk] = -300.0
    return table, kp, vp


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
def test_cached_prefix(pack):
    """Image-token queries over the whole sequence's keys, the text prefix
    handed over from the autoregressive stage."""
    q, k, v = W.make_qkv(pack)
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    sg = W.seq_segments(pack)
    qs = q[torch.as_tensor(rows)].contiguous()
    out_o, lse_o = oracle.attention_general(qs, k, v, cu_q, cu, q_pos0, z, sg,
                                            pack.hq, pack.hkv, pack.d, pack.scale)
    pl = pk.plan_layout(cu_q, cu, sg, pack.hq, pack.hkv, pack.d, q_pos0=q_pos0, k_pos0=z)
    _compare(pack.name + "/prefix", *_run(pl, qs, k, v, pack.scale), out_o, lse_o)


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
def test_paged_keys(pack):
    q, k, v = W.make_qkv(pack)
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    sg = W.seq_segments(pack)
    table, kp, vp = _pool(pack, k, v, 5)
    out_o, lse_o = oracle.attention_general(q, kp, vp, cu, cu, z, z, sg, pack.hq, pack.hkv,
                                            pack.d, pack.scale, block_table=table)
    pl = pk.plan_layout(cu, cu, sg, pack.hq, pack.hkv, pack.d, q_pos0=z, k_pos0=z,
                        block_table=table, num_kv_rows=kp.shape[0])
    _compare(pack.name + "/paged", *_run(pl, q, kp, vp, pack.scale), out_o, lse_o)


@pytest.mark.parametrize("pack", _packs(), ids=lambda p: p.name)
def test_paged_cached_prefix(pack):
    """Both at once: image queries, paged keys holding the whole sequence."""
    q, k, v = W.make_qkv(pack)
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    sg = W.seq_segments(pack)
    table, kp, vp = _pool(pack, k, v, 6)
    qs = q[torch.as_tensor(rows)].contiguous()
    out_o, lse_o = oracle.attention_general(qs, kp, vp, cu_q, cu, q_pos0, z, sg, pack.hq,
                                            pack.hkv, pack.d, pack.scale, block_table=table)
    pl = pk.plan_layout(cu_q, cu, sg, pack.hq, pack.hkv, pack.d, q_pos0=q_pos0, k_pos0=z,
                        block_table=table, num_kv_rows=kp.shape[0])
    _compare(pack.name + "/paged-prefix", *_run(pl, qs, kp, vp, pack.scale), out_o, lse_o)


@pytest.mark.parametrize("chunk", [97, 128, 256])
def test_key_chunks_with_empty_rows(chunk):
    """Every query against one key chunk of its sequence at a time: rows
    before the chunk see nothing, rows inside it see a prefix of it."""
    pack = _packs()[0]
    q, k, v = W.make_qkv(pack)
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    sg = W.seq_segments(pack)
    n_empty = 0
    for cu_k, k_pos0, krows in W.key_chunks(pack, chunk):
        kc = k[torch.as_tensor(krows)].contiguous()
        vc = v[torch.as_tensor(krows)].contiguous()
        out_o, lse_o = oracle.attention_general(q, kc, vc, cu, cu_k, z, k_pos0, sg, pack.hq,
                                                pack.hkv, pack.d, pack.scale)
        pl = pk.plan_layout(cu, cu_k, sg, pack.hq, pack.hkv, pack.d, q_pos0=z, k_pos0=k_pos0)
        _compare(f"chunk{chunk}@{k_pos0.tolist()}", *_run(pl, q, kc, vc, pack.scale), out_o, lse_o)
        n_empty += int(np.isneginf(lse_o).sum())
    assert n_empty > 0


def test_rescale_with_empty_rows_in_the_same_warp():
    """Rows that see none of the key chunk share a warp with image rows whose
    scores grow key tile after key tile, so the rare rescale path recomputes
    a tile that also holds rows without keys."""
    pack = W.Pack("grow-empty", [[(W.TEXT, 140), (W.IMAGE, 460)]], hq=2, hkv=1, d=64, seed=4)
    q, k, v = W.make_qkv(pack)
    T = pack.total_tokens
    ramp = torch.linspace(0.0, 6.0, T).view(T, 1, 1)
    k = (k.float() * 0.1 + ramp).bfloat16()
    q = torch.ones_like(q) * 0.5
    sg = W.seq_segments(pack)
    cu = pack.cu_seqlens
    k_pos0 = np.array([130], np.int32)
    cu_k = np.array([0, T - 130], np.int32)
    kc, vc = k[130:].contiguous(), v[130:].contiguous()
    z = np.zeros(1, np.int32)
    out_o, lse_o = oracle.attention_general(q, kc, vc, cu, cu_k, z, k_pos0, sg, pack.hq,
                                            pack.hkv, pack.d, pack.scale)
    assert np.isneginf(lse_o[:, 128:130]).all() and np.isfinite(lse_o[:, 130:160]).all()
    pl = pk.plan_layout(cu, cu_k, sg, pack.hq, pack.hkv, pack.d, q_pos0=z, k_pos0=k_pos0)
    _compare("grow-empty", *_run(pl, q, kc, vc, pack.scale), out_o, lse_o)


def test_full_size_prefix_paged_sampled():
    """The full mixed-resolution pack with a cached text prefix and paged
    keys, in the benchmark's launch configuration, on a row sample.  The
    oracle side is the packed attention's rows (the general entry equals
    them exactly for these layouts)."""
    pack = W.mixed_resolution()
    q, k, v = W.make_qkv(pack)
    rows, cu_q, q_pos0 = W.prefix_split(pack)
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    sg = W.seq_segments(pack)
    table, kp, vp = _pool(pack, k, v, 7)
    qs = q[torch.as_tensor(rows)].contiguous()
    pl = pk.plan_layout(cu_q, cu, sg, pack.hq, pack.hkv, pack.d, q_pos0=q_pos0, k_pos0=z,
                        block_table=table, num_kv_rows=kp.shape[0])
    out_g, lse_g = _run(pl, qs, kp, vp, pack.scale)
    sample = W.sample_rows(pack, 256)
    pos = np.full(pack.total_tokens, -1, np.int64)
    pos[rows] = np.arange(len(rows))
    sample = sample[pos[sample] >= 0]
    out_o, lse_o = oracle.attention(q, k, v, cu, pack.segments, pack.hq, pack.hkv, pack.d,
                                    pack.scale, rows=sample)
    _compare("mixed_resolution/paged-prefix", out_g[pos[sample]], lse_g[:, pos[sample]],
             out_o, lse_o)
