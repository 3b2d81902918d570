"""Packed mixed-mask variable-length attention for GB300 (sm_103a).

Thin ctypes binding over the C ABI declared in ``include/pk.h``: argument
marshalling only.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and importing this package
fails loudly when the compiled library is missing.

    plan = pk.plan(cu_seqlens, segments, hq, hkv, head_dim)   # host planner
    out, lse = pk.attn_fwd(q, k, v, plan, scale)               # fp16 values, attention
    out, lse = pk.attn_fwd_fp8(q8, qs, k8, ks, v, plan, scale) # E4M3 queries/keys
    out, lse = pk.attn_fwd_fp8_pv(q8, qs, k8, ks, v8, vs, plan) # E4M3 values and P too
    out, lse = pk.lse_merge([(o1, l1), (o2, l2)])              # key blocks -> union
    plan = pk.plan_layout(cu_q, cu_k, seq_segments, hq, hkv, head_dim,
                          q_pos0=..., k_pos0=..., block_table=...)  # prefix / paged / chunks
    pipe = pk.HostPipeline(plan); pipe.submit(qh, kh, vh, oh, lh)   # host buffers

``segments`` is a sequence of (start, length, type) triples in token order,
type 0 = text (causal), 1 = image (sees its whole own segment).  PyTorch
provides device memory and the current stream.
"""
from __future__ import annotations

from ._native import (PK_ERR_ALIGNMENT, PK_ERR_CUDA, PK_ERR_DEVICE_CHECK,  # noqa: F401
                      PK_ERR_INVALID_ARG, PK_ERR_NOT_UPLOADED, PK_ERR_OUT_OF_MEMORY, PK_ERR_RANGE,
                      PK_ERR_TIMEOUT, PK_ERR_TOO_LARGE,
                      PK_ERR_UNSUPPORTED, PK_OK, PKError, lib_path, load)
from .api import (IMAGE, TEXT, HostPipeline, Plan, attn_fwd, attn_fwd_converted,  # noqa: F401
                  attn_fwd_fp8, attn_fwd_fp8_pv, attn_fwd_host, convert_values, debug_wait_timeout, lse_merge,
                  plan, plan_layout, set_wait_timeout_ns)

__all__ = ["plan", "plan_layout", "Plan", "attn_fwd", "convert_values", "attn_fwd_converted",
           "attn_fwd_fp8", "attn_fwd_fp8_pv", "attn_fwd_host",
           "lse_merge", "HostPipeline", "PKError", "TEXT", "IMAGE", "set_wait_timeout_ns",
           "debug_wait_timeout", "load", "lib_path"]
