"""GPU parity of the LSE merge (pk_lse_merge) against the oracle's merge on
the same inputs, and of the compositions it serves: attention over key
chunks merged by LSE, and a ring-style running merge into an fp32
accumulator, both against the fp64 oracle's full attention.  Also the
head split behind Ulysses sequence parallelism: heads are independent, so
running head groups separately is bit-identical to one launch.

Tolerances.  The merge alone is fp32 arithmetic on the given parts: fp32
outputs within 1e-5 (1 + |o|), bf16 outputs within that plus half a bf16 ulp
(the rounding of the result), LSE within 1e-5 (1 + |lse|).  A composition
from bf16 parts inherits each part's error: the merged output is a convex
combination of the parts, so its error is at most the largest part error,
1e-2 plus half a bf16 ulp of that part, plus the final rounding."""
import numpy as np
import pytest
import torch

import oracle
import packed_varlen_masked_gb300 as pk
import workloads as W

pytestmark = pytest.mark.gpu


def _half_ulp_bf16(x):
    a = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 0.5 * np.exp2(np.floor(np.log2(a)) - 7)


def _random_parts(C, T, H, d, dtype, seed, empty_frac=0.2):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(C, T, H, d, generator=g) * 2.0
    lse = torch.randn(C, H, T, generator=g) * 4.0 + 3.0
    drop = torch.rand(C, H, T, generator=g) < empty_frac
    lse[drop] = -float("inf")
    lse[:, 0, :3] = -float("inf")  # rows no part saw
    o = o.to(dtype)
    return o, lse


def _merge_gpu(o, lse, out_dtype, inplace=False):
    parts = [(o[c].cuda().contiguous(), lse[c].cuda().contiguous()) for c in range(o.shape[0])]
    if inplace:
        out, l = pk.lse_merge(parts, out=parts[0][0], lse_out=parts[0][1])
        assert out.data_ptr() == parts[0][0].data_ptr()
    else:
        out, l = pk.lse_merge(parts, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), l.cpu().numpy()


def _check_merge(o, lse, out_g, lse_g, out_bf16):
    om, lm = oracle.lse_merge(o.double().numpy(), lse.double().numpy())
    empty = np.isneginf(lm)
    assert (np.isneginf(lse_g) == empty).all()
    assert (out_g[np.broadcast_to(empty.T[..., None], out_g.shape)] == 0).all()
    tol = 1e-5 * (1 + np.abs(om)) + (_half_ulp_bf16(om) if out_bf16 else 0)
    assert (np.abs(out_g - om) <= tol).all(), float(np.abs(out_g - om).max())
    f = ~empty
    assert (np.abs(lse_g[f] - lm[f]) <= 1e-5 * (1 + np.abs(lm[f]))).all()


@pytest.mark.parametrize("C,d,pdt,odt", [
    (1, 128, torch.bfloat16, torch.bfloat16), (2, 128, torch.bfloat16, torch.bfloat16),
    (3, 64, torch.bfloat16, torch.float32), (5, 128, torch.float32, torch.float32),
    (16, 32, torch.float32, torch.bfloat16), (2, 256, torch.bfloat16, torch.float32),
    (4, 8, torch.float32, torch.float32)])
def test_merge_matches_oracle(C, d, pdt, odt):
    T, H = 333, 6
    o, lse = _random_parts(C, T, H, d, pdt, seed=C * 1000 + d)
    out_g, lse_g = _merge_gpu(o, lse, odt)
    _check_merge(o.float(), lse, out_g, lse_g, odt == torch.bfloat16)


@pytest.mark.parametrize("pdt", [torch.bfloat16, torch.float32])
def test_merge_in_place(pdt):
    o, lse = _random_parts(3, 257, 4, 128, pdt, seed=7)
    out_g, lse_g = _merge_gpu(o, lse, None, inplace=True)
    _check_merge(o.float(), lse, out_g, lse_g, pdt == torch.bfloat16)


def test_merge_nan_lse_poisons_only_its_row():
    o, lse = _random_parts(2, 64, 2, 64, torch.float32, seed=3, empty_frac=0.0)
    lse[1, 1, 10] = float("nan")
    out_g, lse_g = _merge_gpu(o, lse, torch.float32)
    assert np.isnan(lse_g[1, 10]) and np.isnan(out_g[10, 1]).all()
    lse_g[1, 10] = 0.0
    assert np.isneginf(lse_g[0, :3]).all()  # rows no part saw
    lse_g[0, :3] = 0.0
    assert np.isfinite(lse_g).all()


def _layout_parts(pack, q, k, v, chunk, out_f32=False):
    cu = pack.cu_seqlens
    z = np.zeros(len(cu) - 1, np.int32)
    sg = W.seq_segments(pack)
    parts = []
    for cu_k, k_pos0, krows in W.key_chunks(pack, chunk):
        idx = torch.as_tensor(krows)
        kc, vc = k[idx].contiguous().cuda(), v[idx].contiguous().cuda()
        pl = pk.plan_layout(cu, cu_k, sg, pack.hq, pack.hkv, pack.d, q_pos0=z, k_pos0=k_pos0)
        parts.append(pk.attn_fwd(q.cuda(), kc, vc, pl, pack.scale, check_status=True))
    return parts


def _pack():
    return W.Pack("ring", [[(W.TEXT, 40), (W.IMAGE, 600), (W.TEXT, 9)],
                           [(W.IMAGE, 300), (W.IMAGE, 130)],
                           [(W.TEXT, 77), (W.IMAGE, 513)]], hq=8, hkv=2, d=128, seed=41)


@pytest.mark.parametrize("chunk", [128, 200, 384])
def test_key_chunks_merged_equal_full_attention(chunk):
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    parts = _layout_parts(pack, q, k, v, chunk)
    out, lse = pk.lse_merge(parts)
    torch.cuda.synchronize()
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                                    pack.d, pack.scale)
    out_g, lse_g = out.float().cpu().numpy(), lse.cpu().numpy()
    part_ulp = np.max(np.stack([_half_ulp_bf16(p[0].float().cpu().numpy()) for p in parts]), axis=0)
    err = np.abs(out_g - out_o)
    print(f"chunk {chunk}: {len(parts)} parts, max|dout|={err.max():.3e}, "
          f"max|dlse|={np.abs(lse_g - lse_o).max():.3e}")
    assert (err <= 1e-2 + _half_ulp_bf16(out_o) + part_ulp).all()
    assert np.abs(lse_g - lse_o).max() <= 1e-3


def test_ring_running_merge_into_fp32_accumulator():
    """Ring order: the accumulator starts as the first key block's result and
    every later block is merged into it in place (fp32 output)."""
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    parts = _layout_parts(pack, q, k, v, 256)
    acc_o, acc_l = pk.lse_merge(parts[:1], out_dtype=torch.float32)
    for p in parts[1:]:
        pk.lse_merge([(acc_o, acc_l), p], out=acc_o, lse_out=acc_l)
    torch.cuda.synchronize()
    out_o, lse_o = oracle.attention(q, k, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                                    pack.d, pack.scale)
    part_ulp = np.max(np.stack([_half_ulp_bf16(p[0].float().cpu().numpy()) for p in parts]), axis=0)
    err = np.abs(acc_o.cpu().numpy() - out_o)
    assert (err <= 1e-2 + part_ulp).all(), float(err.max())
    assert np.abs(acc_l.cpu().numpy() - lse_o).max() <= 1e-3


def test_head_groups_run_separately_are_bit_identical():
    """Ulysses hands each rank all tokens of a subset of heads: attention on
    a KV-head group and its query heads alone equals those heads of the full
    launch exactly."""
    pack = _pack()
    q, k, v = W.make_qkv(pack, device="cuda")
    full_o, full_l = pk.attn_fwd(q, k, v, pk.plan(pack.cu_seqlens, pack.segments, pack.hq,
                                                  pack.hkv, pack.d), pack.scale, check_status=True)
    group = pack.hq // pack.hkv
    for g0 in range(0, pack.hkv, 1):
        hs = slice(g0 * group, (g0 + 1) * group)
        pl = pk.plan(pack.cu_seqlens, pack.segments, group, 1, pack.d)
        o, l = pk.attn_fwd(q[:, hs].contiguous(), k[:, g0:g0 + 1].contiguous(),
                           v[:, g0:g0 + 1].contiguous(), pl, pack.scale, check_status=True)
        assert torch.equal(o, full_o[:, hs]) and torch.equal(l, full_l[hs])
