"""pk_attn_fwd_noalloc, the attention entry point for callers that cannot
allocate device memory at the call: code inside a host framework that owns
all device memory through its own pool and forbids other allocations, or a
latency-critical loop that must not make a call that can synchronise the
device, as cudaMalloc and cudaFree can.  It keeps the fp16 copy of the values
in a 64 MiB static device array of the library instead of a caller's
workspace.

Its results must match pk_attn_fwd's (the entry point that takes a
workspace) under the rule every parity test uses (parity_tol.py), on two
calls in a row: the second call, on another pack, reads an array the first
one left full of other values, so a part of it the second call failed to
rewrite would show.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import packed_varlen_masked_gb300 as pk
import workloads as W
from parity_tol import check

pytestmark = pytest.mark.gpu


def _noalloc(plan, q, k, v, scale):
    out = torch.empty(plan.total_tokens, plan.hq, plan.head_dim, dtype=torch.bfloat16,
                      device="cuda")
    lse = torch.empty(plan.hq, plan.total_tokens, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = pk.load().pk_attn_fwd_noalloc(
        plan.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), float(scale), ctypes.c_void_p(stream),
        ctypes.c_void_p(status.data_ptr()))
    assert st == pk.PK_OK, pk.PKError(st, "pk_attn_fwd_noalloc")
    torch.cuda.synchronize()
    assert int(status.item()) == pk.PK_OK
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_the_workspace_entry_on_two_calls_in_a_row():
    # First call: a pack whose values fill ~17 MB of the array.
    a = W.cfg_pair(seed=3)
    q, k, v = W.make_qkv(a, device="cuda")
    plan_a = pk.plan(a.cu_seqlens, a.segments, a.hq, a.hkv, a.d)
    ref_o, ref_l = pk.attn_fwd(q, k, v, plan_a, a.scale, check_status=True)
    o, l = _noalloc(plan_a, q, k, v, a.scale)
    check("noalloc/call1", o, l, ref_o.float().cpu().numpy(), ref_l.cpu().numpy())

    # Second call: key chunks of a smaller pack over a key tensor with rows no
    # sequence owns (holding large values): the kernel reads some of those rows
    # as masked keys, from array rows the first call left holding its values.
    b = W.Pack("noalloc-chunks", [[(W.TEXT, 50), (W.IMAGE, 700)], [(W.TEXT, 9), (W.IMAGE, 300)]],
               hq=8, hkv=2, d=128, seed=4)
    q, k, v = W.make_qkv(b, device="cuda")
    cu = b.cu_seqlens
    cu_k, k_pos0, krows = next(iter(W.key_chunks(b, 384)))
    idx = torch.as_tensor(krows, device="cuda")
    spare = 200
    kc = torch.cat([k[idx], torch.full((spare, b.hkv, b.d), 30.0, dtype=k.dtype, device="cuda")])
    vc = torch.cat([v[idx], torch.full((spare, b.hkv, b.d), -500.0, dtype=v.dtype, device="cuda")])
    plan_b = pk.plan_layout(cu, cu_k, W.seq_segments(b), b.hq, b.hkv, b.d,
                            q_pos0=np.zeros(len(cu) - 1, np.int32), k_pos0=k_pos0,
                            num_kv_rows=kc.shape[0])
    ref_o, ref_l = pk.attn_fwd(q, kc, vc, plan_b, b.scale, check_status=True)
    o, l = _noalloc(plan_b, q, kc, vc, b.scale)
    check("noalloc/call2", o, l, ref_o.float().cpu().numpy(), ref_l.cpu().numpy())


def test_noalloc_rejects_plans_beyond_its_scratch():
    big = W.Pack("noalloc-big", [[(W.IMAGE, 32768 + 128)]], hq=8, hkv=8, d=128)
    plan = pk.Plan(big.cu_seqlens, big.segments, big.hq, big.hkv, big.d, upload=False)
    assert plan.workspace_bytes > 64 << 20
    st = pk.load().pk_attn_fwd_noalloc(plan.handle, 16, 16, 16, 16, 16, 0.1, None, None)
    assert st == pk.PK_ERR_TOO_LARGE
