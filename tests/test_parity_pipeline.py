"""The host-buffer pipeline (three streams, caller-owned device slots) gives
exactly the single-call results, step after step, with distinct inputs per
step and more steps than slots."""
import numpy as np
import pytest
import torch

import packed_varlen_masked_gb300 as pk
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("num_slots", [1, 2, 3])
def test_pipeline_steps_equal_single_calls(num_slots):
    base = W.Pack("pipe", [[(W.TEXT, 70), (W.IMAGE, 500)], [(W.TEXT, 9), (W.IMAGE, 300)]],
                  hq=8, hkv=2, d=128)
    plan = pk.plan(base.cu_seqlens, base.segments, base.hq, base.hkv, base.d)
    pipe = pk.HostPipeline(plan, num_slots=num_slots)
    steps = []
    for s in range(5):
        pack = W.Pack("pipe", base.seqs, hq=8, hkv=2, d=128, seed=100 + s)
        q, k, v = W.make_qkv(pack)
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        oh = torch.empty_like(q).pin_memory()
        lh = torch.empty(pack.hq, pack.total_tokens, dtype=torch.float32).pin_memory()
        pipe.submit(qh, kh, vh, oh, lh, pack.scale)
        steps.append((q, k, v, oh, lh))
    pipe.sync()
    for q, k, v, oh, lh in steps:
        o_ref, l_ref = pk.attn_fwd(q.cuda(), k.cuda(), v.cuda(), plan, base.scale, check_status=True)
        assert torch.equal(oh, o_ref.cpu()) and torch.equal(lh, l_ref.cpu())
    s0, s1, s2 = pipe.stream(0), pipe.stream(1), pipe.stream(2)
    assert len({s0.cuda_stream, s1.cuda_stream, s2.cuda_stream}) == 3
    pipe.close()
