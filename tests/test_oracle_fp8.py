"""Pins for the oracle's FP8 entry (E4M3 queries and keys, bf16 values):
the E4M3 decoder against torch's float8_e4m3fn for every code, and the
attention against the pinned bf16 oracle where the two must agree."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W


def test_e4m3_decoder_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2  # S.1111.111
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_to_double(0x7E) == 448.0 and oracle.e4m3_to_double(0x01) == 2.0 ** -9


def _pack():
    return W.Pack("fp8", [[(W.TEXT, 30), (W.IMAGE, 90), (W.TEXT, 5)], [(W.IMAGE, 70)],
                          [(W.TEXT, 41)]], hq=4, hkv=2, d=32, seed=13)


def test_e4m3_attention_equals_bf16_attention_on_the_decoded_values():
    """Every E4M3 value times a power-of-two scale is exact in bf16, so the
    FP8 entry must reproduce the bf16 oracle on those bf16 tensors."""
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    q8, _ = W.quantize_e4m3(q)
    k8, _ = W.quantize_e4m3(k)
    qs, ks = 2.0 ** -5, 2.0 ** -4
    qd = (q8.view(torch.float8_e4m3fn).float() * qs).to(torch.bfloat16)
    kd = (k8.view(torch.float8_e4m3fn).float() * ks).to(torch.bfloat16)
    assert torch.equal(qd.float(), q8.view(torch.float8_e4m3fn).float() * qs)  # exact
    o8, l8 = oracle.attention_e4m3(q8, qs, k8, ks, v, pack.cu_seqlens, pack.segments, pack.hq,
                                   pack.hkv, pack.d, pack.scale)
    o, l = oracle.attention(qd, kd, v, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                            pack.d, pack.scale)
    np.testing.assert_allclose(o8, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, l, rtol=0, atol=1e-12)


def test_e4m3_scales_fold_into_the_softmax_scale_and_rows_sample():
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    q8, qs = W.quantize_e4m3(q)
    k8, ks = W.quantize_e4m3(k)
    o1, l1 = oracle.attention_e4m3(q8, qs, k8, ks, v, pack.cu_seqlens, pack.segments, pack.hq,
                                   pack.hkv, pack.d, pack.scale)
    o2, l2 = oracle.attention_e4m3(q8, 1.0, k8, 1.0, v, pack.cu_seqlens, pack.segments, pack.hq,
                                   pack.hkv, pack.d, pack.scale * qs * ks)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)
    rows = np.array([0, 29, 30, 119, 120, 124, 125, 194, 195, 235], np.int32)
    o3, l3 = oracle.attention_e4m3(q8, qs, k8, ks, v, pack.cu_seqlens, pack.segments, pack.hq,
                                   pack.hkv, pack.d, pack.scale, rows=rows)
    np.testing.assert_array_equal(o3, o1[rows])
    np.testing.assert_array_equal(l3, l1[:, rows])


def test_quantizer_uses_the_full_e4m3_range():
    x = torch.randn(1000, dtype=torch.float32).to(torch.bfloat16)
    codes, s = W.quantize_e4m3(x)
    deq = codes.view(torch.float8_e4m3fn).float() * s
    assert float(deq.abs().max()) == pytest.approx(float(x.float().abs().max()), rel=1e-6)
    assert float((deq - x.float()).abs().max()) <= float(x.float().abs().max()) * 2.0 ** -4


def test_e4m3_value_attention_equals_bf16_attention_on_the_decoded_values():
    """E4M3 values too (codes and a power-of-two scale, exact in bf16): the
    all-E4M3 entry must reproduce the pinned bf16 oracle on the decoded
    q, k and v, and the value scale must act as a plain factor."""
    pack = _pack()
    q, k, v = W.make_qkv(pack)
    q8, _ = W.quantize_e4m3(q)
    k8, _ = W.quantize_e4m3(k)
    v8, _ = W.quantize_e4m3(v)
    qs, ks, vs = 2.0 ** -5, 2.0 ** -4, 2.0 ** -3
    dec = lambda c, s: (c.view(torch.float8_e4m3fn).float() * s).to(torch.bfloat16)
    qd, kd, vd = dec(q8, qs), dec(k8, ks), dec(v8, vs)
    assert torch.equal(vd.float(), v8.view(torch.float8_e4m3fn).float() * vs)  # exact
    o8, l8 = oracle.attention_e4m3_v8(q8, qs, k8, ks, v8, vs, pack.cu_seqlens, pack.segments,
                                      pack.hq, pack.hkv, pack.d, pack.scale)
    o, l = oracle.attention(qd, kd, vd, pack.cu_seqlens, pack.segments, pack.hq, pack.hkv,
                            pack.d, pack.scale)
    np.testing.assert_allclose(o8, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, l, rtol=0, atol=1e-12)
    o2, l2 = oracle.attention_e4m3_v8(q8, qs, k8, ks, v8, 2 * vs, pack.cu_seqlens, pack.segments,
                                      pack.hq, pack.hkv, pack.d, pack.scale)
    np.testing.assert_allclose(o2, 2 * o8, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(l2, l8)
