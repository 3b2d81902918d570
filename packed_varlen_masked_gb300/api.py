"""User-facing calls (argument marshalling around the C ABI; all computation
happens in the library): ``plan`` / ``plan_layout`` / ``Plan``, ``attn_fwd``,
``attn_fwd_fp8``, ``attn_fwd_host``, ``HostPipeline`` and ``lse_merge``."""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence, Tuple

import numpy as np

from ._native import (PK_DTYPE_BF16, PK_DTYPE_F32, DevSlot, Layout, MergePart, PlanInfo,
                      Segment, SeqSegment, WorkItem, check, load)

TEXT = 0
IMAGE = 1


def _segments_struct(segments) -> Tuple[ctypes.Array, int]:
    arr = np.asarray(segments, dtype=np.int64).reshape(-1, 3)
    n = arr.shape[0]
    segs = (Segment * max(n, 1))()
    for i, (st, ln, ty) in enumerate(arr.tolist()):
        segs[i] = Segment(int(st), int(ln), int(ty))
    return segs, n


class Plan:
    """A host plan (tile classes + longest-work-first schedule) and, once
    uploaded, its device image in a PyTorch-allocated buffer.

    Build it once per pack composition and reuse it for every layer and
    denoising step: it is read-only after upload.
    """

    def __init__(self, cu_seqlens, segments, hq: int, hkv: int, head_dim: int,
                 num_ctas: int = 0, device=None, upload: bool = True, _layout=None, _shard=None):
        self._lib = load()
        self._h = ctypes.c_void_p()
        self.hq, self.hkv, self.head_dim = int(hq), int(hkv), int(head_dim)
        self._buf = None
        if _shard is not None:
            full, rank, world = _shard
            check(self._lib.pk_plan_shard(full.handle, int(rank), int(world), int(num_ctas),
                                          ctypes.byref(self._h)), "pk_plan_shard")
        elif _layout is not None:
            lay, keep = _layout
            check(self._lib.pk_plan_create_layout(ctypes.byref(lay), self.hq, self.hkv,
                                                  self.head_dim, int(num_ctas),
                                                  ctypes.byref(self._h)), "pk_plan_create_layout")
            del keep
        else:
            cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
            if cu.ndim != 1 or cu.size < 1:
                raise ValueError("cu_seqlens must be a 1-D array with at least one entry")
            segs, n = _segments_struct(segments)
            check(self._lib.pk_plan_create(cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                           cu.size - 1, segs, n, self.hq, self.hkv,
                                           self.head_dim, int(num_ctas), ctypes.byref(self._h)),
                  "pk_plan_create")
        info = self.info
        self.total_tokens = int(info["total_tokens"])
        self.kv_rows = int(info["kv_rows"])
        if upload:
            self.upload(device)

    def shard(self, rank: int, num_ranks: int, num_ctas: int = 0, device=None,
              upload: bool = True) -> "Plan":
        """Rank ``rank``'s share of this plan (pk_plan_shard): whole
        (sequence, key/value head) units, longest first to the least-loaded
        rank; launched on the full tensors, it writes only its units' rows
        and heads."""
        return Plan(None, None, self.hq, self.hkv, self.head_dim, num_ctas=num_ctas,
                    device=device, upload=upload, _shard=(self, rank, num_ranks))

    # -- lifetime -----------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.pk_plan_destroy(self._h)
            self._h = ctypes.c_void_p()
        self._buf = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    # -- device image -------------------------------------------------------
    @property
    def device_bytes(self) -> int:
        return int(self._lib.pk_plan_device_bytes(self._h))

    def upload(self, device=None) -> None:
        import torch
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        nbytes = self.device_bytes
        buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        check(self._lib.pk_plan_upload(self._h, ctypes.c_void_p(buf.data_ptr()), nbytes,
                                       ctypes.c_void_p(stream)), "pk_plan_upload")
        self._buf = buf

    @property
    def device_buffer(self):
        return self._buf

    # -- introspection --------------------------------------------------------
    @property
    def info(self) -> dict:
        pi = PlanInfo()
        check(self._lib.pk_plan_get_info(self._h, ctypes.byref(pi)), "pk_plan_get_info")
        return {name: getattr(pi, name) for name, _ in PlanInfo._fields_}

    @property
    def useful_flops(self) -> float:
        return float(self._lib.pk_plan_useful_flops(self._h))

    @property
    def workspace_bytes(self) -> int:
        """Bytes of the per-launch workspace (the fp16 copy of the values)."""
        return int(self._lib.pk_attn_workspace_bytes(self._h))

    @property
    def workspace_bytes_fp8_pv(self) -> int:
        """Bytes of attn_fwd_fp8_pv's workspace (the transposed E4M3 values)."""
        return int(self._lib.pk_attn_workspace_bytes_fp8_pv(self._h))

    def set_sm_pairs(self, enable: bool = True) -> "Plan":
        """Run this plan on SM pairs (pk_plan_set_sm_pairs; head_dim 128):
        against the one-CTA kernel faster on packs of long sequences and
        slower on short ones; slower than the default head-pair clusters on
        every pack measured, off by default.  Returns the plan."""
        check(self._lib.pk_plan_set_sm_pairs(self._h, 1 if enable else 0), "pk_plan_set_sm_pairs")
        return self

    def set_kv_share(self, enable: bool = True) -> "Plan":
        """Head-pair clusters sharing each key/value tile (pk_plan_set_kv_share):
        on by default at head_dim 128 where the plan has their schedule (an
        even number of query heads per key/value head), opt-in at 64;
        ``False`` selects the
        one-CTA kernel.  Bit-identical results either way.  Returns the plan."""
        check(self._lib.pk_plan_set_kv_share(self._h, 1 if enable else 0), "pk_plan_set_kv_share")
        return self

    @property
    def kv_share(self) -> bool:
        """Whether launches of this plan run on head-pair clusters
        (pk_plan_kv_share; ``set_sm_pairs(True)`` takes precedence)."""
        return bool(self._lib.pk_plan_kv_share(self._h))

    def share_schedule(self) -> Tuple[np.ndarray, np.ndarray]:
        """(items int32 [num_items, 8], cluster-ordered; cluster offsets int32
        [num_clusters + 1]) of the head-pair cluster schedule; empty when the
        plan has none.  Columns as ``items``."""
        ncl = ctypes.c_int32()
        check(self._lib.pk_plan_get_share(self._h, ctypes.byref(ncl), None, 0, None, 0),
              "pk_plan_get_share")
        if ncl.value == 0:
            return np.zeros((0, 8), dtype=np.int32), np.zeros(1, dtype=np.int32)
        n = int(self.info["num_items"])
        items = (WorkItem * max(n, 1))()
        offs = np.zeros(ncl.value + 1, dtype=np.int32)
        check(self._lib.pk_plan_get_share(self._h, ctypes.byref(ncl), items, n,
                                          offs.ctypes.data_as(ctypes.c_void_p), offs.size),
              "pk_plan_get_share")
        arr = np.frombuffer(bytes(items), dtype=np.int32).reshape(-1, 8)[:n].copy()
        return arr, offs

    def pairs(self) -> Tuple[np.ndarray, np.ndarray]:
        """(pair items int32 [2 * num_pairs, 8], rank 0 then rank 1 of each
        pair, cluster-ordered; cluster offsets int32 [num_clusters + 1], in
        pairs).  Columns as ``items``."""
        npairs, ncl = ctypes.c_int32(), ctypes.c_int32()
        check(self._lib.pk_plan_get_pairs(self._h, ctypes.byref(npairs), ctypes.byref(ncl), None, 0,
                                          None, 0), "pk_plan_get_pairs")
        n = 2 * npairs.value
        items = (WorkItem * max(n, 1))()
        offs = np.zeros(ncl.value + 1, dtype=np.int32)
        if ncl.value > 0:
            check(self._lib.pk_plan_get_pairs(self._h, ctypes.byref(npairs), ctypes.byref(ncl),
                                              items, n, offs.ctypes.data_as(ctypes.c_void_p),
                                              offs.size), "pk_plan_get_pairs")
        arr = np.frombuffer(bytes(items), dtype=np.int32).reshape(-1, 8)[:n].copy()
        return arr, offs

    def kv_limit(self) -> np.ndarray:
        out = np.zeros(max(self.total_tokens, 1), dtype=np.int32)
        check(self._lib.pk_plan_get_kv_limit(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                              out.size), "pk_plan_get_kv_limit")
        return out[: self.total_tokens]

    def items(self) -> Tuple[np.ndarray, np.ndarray]:
        """(items int32 [n, 8] in CTA order, cta_offsets int32 [num_ctas + 1]).
        Columns: q_start, q_rows, kv_start, n_kt, n_full, hq0, hq1, hkv."""
        info = self.info
        n, g = info["num_items"], info["num_ctas"]
        items = (WorkItem * max(n, 1))()
        offs = np.zeros(g + 1, dtype=np.int32)
        check(self._lib.pk_plan_get_items(self._h, items, n,
                                           offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                           g + 1), "pk_plan_get_items")
        arr = np.frombuffer(bytes(items), dtype=np.int32).reshape(-1, 8)[:n].copy()
        return arr, offs


def plan(cu_seqlens, segments, hq: int, hkv: int, head_dim: int, num_ctas: int = 0,
         device=None) -> Plan:
    return Plan(cu_seqlens, segments, hq, hkv, head_dim, num_ctas=num_ctas, device=device)


def plan_layout(cu_seqlens_q, cu_seqlens_k, seq_segments, hq: int, hkv: int, head_dim: int,
                q_pos0=None, k_pos0=None, block_table=None, num_kv_rows: Optional[int] = None,
                num_ctas: int = 0, device=None, upload: bool = True) -> Plan:
    """Plan for queries and keys that are position ranges of their sequences
    (cached prefix, key chunks) and optionally paged keys (see pk_layout in
    include/pk.h).  ``seq_segments``: (seq, start, len, type) rows in each
    sequence's position space; ``block_table`` [num_seqs, blocks_per_seq]
    of 128-row pool blocks."""
    i32 = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    p32 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if a is not None else None
    cq, ck = i32(cu_seqlens_q), i32(cu_seqlens_k)
    S = cq.size - 1
    qp = i32(q_pos0) if q_pos0 is not None else None
    kp = i32(k_pos0) if k_pos0 is not None else None
    sg = np.asarray(seq_segments, dtype=np.int64).reshape(-1, 4)
    segs = (SeqSegment * max(sg.shape[0], 1))()
    for i, (a, b, c, d) in enumerate(sg.tolist()):
        segs[i] = SeqSegment(int(a), int(b), int(c), int(d))
    bt = i32(block_table).reshape(S, -1) if block_table is not None else None
    if num_kv_rows is None:
        if bt is not None:
            raise ValueError("num_kv_rows (pool rows) is required with a block table")
        num_kv_rows = int(ck[-1])
    lay = Layout(S, p32(cq), p32(qp), p32(ck), p32(kp), segs, sg.shape[0],
                 p32(bt) if bt is not None else None, bt.shape[1] if bt is not None else 0,
                 int(num_kv_rows))
    keep = (cq, ck, qp, kp, segs, bt)
    return Plan(None, None, hq, hkv, head_dim, num_ctas=num_ctas, device=device, upload=upload,
                _layout=(lay, keep))


def _check_tensor(t, name, shape):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _workspace(plan: "Plan", workspace, device, nbytes: Optional[int] = None):
    """The launch's workspace: the caller's tensor (checked), else a fresh
    one from PyTorch's caching allocator on the current stream."""
    import torch
    if nbytes is None:
        nbytes = plan.workspace_bytes
    if workspace is None:
        return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or \
            not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} bytes, "
                         f"the plan needs {nbytes}")
    return workspace


def attn_fwd(q, k, v, plan: Plan, scale: Optional[float] = None, out=None, lse=None,
             status=None, check_status: bool = False, workspace=None):
    """Packed mixed-mask attention forward on the current CUDA stream.

    q [T, hq, d], k and v [Tk, hkv, d] bf16 CUDA tensors (Tk = T for a
    plan from ``plan``; the key rows or pool rows for ``plan_layout``).
    Returns (out bf16 [T, hq, d], lse fp32 [hq, T]).  ``workspace``: a CUDA
    tensor of at least ``plan.workspace_bytes`` bytes for the fp16 copy of
    the values (allocated here when omitted; passing ``v`` converts v in
    place).  With ``check_status`` the call synchronises and raises if the
    kernels reported a device-side failure.
    """
    import torch
    T, hq, hkv, d = plan.total_tokens, plan.hq, plan.hkv, plan.head_dim
    Tk = plan.kv_rows
    _check_tensor(q, "q", (T, hq, d))
    _check_tensor(k, "k", (Tk, hkv, d))
    _check_tensor(v, "v", (Tk, hkv, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_tensor(out, "out", (T, hq, d))
    if lse is None:
        lse = torch.empty(hq, T, dtype=torch.float32, device=q.device)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (hq, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor of shape [hq, T]")
    ws = _workspace(plan, workspace, q.device)
    if check_status and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    check(plan._lib.pk_attn_fwd(plan.handle, ctypes.c_void_p(q.data_ptr()),
                                ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                float(scale), ctypes.c_void_p(ws.data_ptr()),
                                ws.numel() * ws.element_size(), ctypes.c_void_p(stream),
                                ctypes.c_void_p(status.data_ptr() if status is not None else 0)),
          "pk_attn_fwd")
    if check_status:
        torch.cuda.current_stream(q.device).synchronize()
        check(int(status.item()), "pk_attn_fwd (device)")
    return out, lse


def convert_values(v, plan: Plan, workspace=None, status=None):
    """pk_attn_convert_values: the fp16 copy of the value rows ``plan`` reads,
    into ``workspace`` (allocated when omitted; ``v`` itself converts in
    place).  Returns the workspace, for ``attn_fwd_converted``."""
    import torch
    _check_tensor(v, "v", (plan.kv_rows, plan.hkv, plan.head_dim))
    ws = _workspace(plan, workspace, v.device)
    stream = torch.cuda.current_stream(v.device).cuda_stream
    check(plan._lib.pk_attn_convert_values(
        plan.handle, ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
        ws.numel() * ws.element_size(), ctypes.c_void_p(stream),
        ctypes.c_void_p(status.data_ptr() if status is not None else 0)), "pk_attn_convert_values")
    return ws


def attn_fwd_converted(q, k, v16, plan: Plan, scale: Optional[float] = None, out=None, lse=None,
                       status=None, check_status: bool = False):
    """pk_attn_fwd_converted: the attention on values ``convert_values``
    prepared (``v16``: its workspace, only read)."""
    import torch
    T, hq, hkv, d = plan.total_tokens, plan.hq, plan.hkv, plan.head_dim
    _check_tensor(q, "q", (T, hq, d))
    _check_tensor(k, "k", (plan.kv_rows, hkv, d))
    if not isinstance(v16, torch.Tensor) or not v16.is_cuda or \
            v16.numel() * v16.element_size() < plan.workspace_bytes:
        raise ValueError("v16 must be a CUDA tensor of at least plan.workspace_bytes bytes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty(hq, T, dtype=torch.float32, device=q.device)
    _check_tensor(out, "out", (T, hq, d))
    if check_status and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    check(plan._lib.pk_attn_fwd_converted(
        plan.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v16.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), float(scale), ctypes.c_void_p(stream),
        ctypes.c_void_p(status.data_ptr() if status is not None else 0)), "pk_attn_fwd_converted")
    if check_status:
        torch.cuda.current_stream(q.device).synchronize()
        check(int(status.item()), "pk_attn_fwd_converted (device)")
    return out, lse


def attn_fwd_fp8(q8, q_scale: float, k8, k_scale: float, v, plan: Plan,
                 scale: Optional[float] = None, out=None, lse=None, status=None,
                 check_status: bool = False, workspace=None):
    """Attention with FP8 E4M3 queries and keys (pk_attn_fwd_fp8).

    q8 [T, hq, 128] and k8 [Tk, hkv, 128]: CUDA uint8 or float8_e4m3fn
    tensors of E4M3 codes, dequantised by q_scale / k_scale; v bf16
    [Tk, hkv, 128].  Returns (out bf16 [T, hq, 128], lse fp32 [hq, T]).
    ``workspace`` as for ``attn_fwd``."""
    import torch
    T, hq, hkv, d = plan.total_tokens, plan.hq, plan.hkv, plan.head_dim
    Tk = plan.kv_rows
    for name, t, shape in (("q8", q8, (T, hq, d)), ("k8", k8, (Tk, hkv, d))):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.element_size() != 1:
            raise TypeError(f"{name} must be a CUDA tensor of 1-byte E4M3 codes")
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous with shape {shape}")
    _check_tensor(v, "v", (Tk, hkv, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(T, hq, d, dtype=torch.bfloat16, device=v.device)
    else:
        _check_tensor(out, "out", (T, hq, d))
    if lse is None:
        lse = torch.empty(hq, T, dtype=torch.float32, device=v.device)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (hq, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor of shape [hq, T]")
    ws = _workspace(plan, workspace, v.device)
    if check_status and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=v.device)
    stream = torch.cuda.current_stream(v.device).cuda_stream
    check(plan._lib.pk_attn_fwd_fp8(plan.handle, ctypes.c_void_p(q8.data_ptr()), float(q_scale),
                                    ctypes.c_void_p(k8.data_ptr()), float(k_scale),
                                    ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(lse.data_ptr()), float(scale),
                                    ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
                                    ctypes.c_void_p(stream),
                                    ctypes.c_void_p(status.data_ptr() if status is not None else 0)),
          "pk_attn_fwd_fp8")
    if check_status:
        torch.cuda.current_stream(v.device).synchronize()
        check(int(status.item()), "pk_attn_fwd_fp8 (device)")
    return out, lse


def attn_fwd_fp8_pv(q8, q_scale: float, k8, k_scale: float, v8, v_scale: float, plan: Plan,
                    scale: Optional[float] = None, out=None, lse=None, status=None,
                    check_status: bool = False, workspace=None):
    """Attention with FP8 E4M3 queries, keys and values, the softmax weights
    rounded to E4M3 for an FP8 P V product (pk_attn_fwd_fp8_pv).

    q8 [T, hq, 128], k8 and v8 [Tk, hkv, 128]: CUDA uint8 or float8_e4m3fn
    tensors of E4M3 codes, dequantised by q_scale / k_scale / v_scale.
    Returns (out bf16 [T, hq, 128], lse fp32 [hq, T]).  ``workspace``: at
    least ``plan.workspace_bytes_fp8_pv`` bytes, else one is taken from
    PyTorch's allocator."""
    import torch
    T, hq, hkv, d = plan.total_tokens, plan.hq, plan.hkv, plan.head_dim
    Tk = plan.kv_rows
    for name, t, shape in (("q8", q8, (T, hq, d)), ("k8", k8, (Tk, hkv, d)),
                           ("v8", v8, (Tk, hkv, d))):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.element_size() != 1:
            raise TypeError(f"{name} must be a CUDA tensor of 1-byte E4M3 codes")
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous with shape {shape}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(T, hq, d, dtype=torch.bfloat16, device=v8.device)
    else:
        _check_tensor(out, "out", (T, hq, d))
    if lse is None:
        lse = torch.empty(hq, T, dtype=torch.float32, device=v8.device)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (hq, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor of shape [hq, T]")
    ws = _workspace(plan, workspace, v8.device, plan.workspace_bytes_fp8_pv)
    if check_status and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=v8.device)
    stream = torch.cuda.current_stream(v8.device).cuda_stream
    check(plan._lib.pk_attn_fwd_fp8_pv(
        plan.handle, ctypes.c_void_p(q8.data_ptr()), float(q_scale),
        ctypes.c_void_p(k8.data_ptr()), float(k_scale), ctypes.c_void_p(v8.data_ptr()),
        float(v_scale), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        float(scale), ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
        ctypes.c_void_p(stream), ctypes.c_void_p(status.data_ptr() if status is not None else 0)),
        "pk_attn_fwd_fp8_pv")
    if check_status:
        torch.cuda.current_stream(v8.device).synchronize()
        check(int(status.item()), "pk_attn_fwd_fp8_pv (device)")
    return out, lse


def attn_fwd_host(q_host, k_host, v_host, plan: Plan, scale: float, dev_buffers: dict,
                  out_host, lse_host, status=None):
    """End-to-end call from host buffers (ideally pinned): copies q/k/v to the
    caller's device buffers, runs the attention and copies out/lse back, all
    on the current stream.  ``dev_buffers`` holds CUDA tensors 'q', 'k', 'v',
    'out', 'lse' of the pk_attn_fwd shapes ('v' also serves as the workspace:
    its values are converted to fp16 in place)."""
    import torch
    for name, t in (("q_host", q_host), ("k_host", k_host), ("v_host", v_host),
                    ("out_host", out_host), ("lse_host", lse_host)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    db = dev_buffers
    stream = torch.cuda.current_stream(db["q"].device).cuda_stream
    check(plan._lib.pk_attn_fwd_host(
        plan.handle, ctypes.c_void_p(q_host.data_ptr()), ctypes.c_void_p(k_host.data_ptr()),
        ctypes.c_void_p(v_host.data_ptr()), ctypes.c_void_p(out_host.data_ptr()),
        ctypes.c_void_p(lse_host.data_ptr()), ctypes.c_void_p(db["q"].data_ptr()),
        ctypes.c_void_p(db["k"].data_ptr()), ctypes.c_void_p(db["v"].data_ptr()),
        ctypes.c_void_p(db["out"].data_ptr()), ctypes.c_void_p(db["lse"].data_ptr()),
        float(scale), ctypes.c_void_p(stream),
        ctypes.c_void_p(status.data_ptr() if status is not None else 0)), "pk_attn_fwd_host")
    return out_host, lse_host


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return PK_DTYPE_BF16
    if t.dtype == torch.float32:
        return PK_DTYPE_F32
    raise TypeError("partial outputs must be bfloat16 or float32")


def lse_merge(parts, out=None, lse_out=None, out_dtype=None, status=None,
              check_status: bool = False):
    """Merge partial attentions over disjoint key sets (pk_lse_merge).

    ``parts``: sequence of (o [T, H, d], lse [H, T] fp32) CUDA tensors, o bf16
    or fp32.  Returns (out [T, H, d], lse [H, T]); ``out`` / ``lse_out`` may
    be a part's own tensors (in-place accumulation).  Runs on the current
    stream; with ``check_status`` it synchronises and raises on a device-side
    failure."""
    import torch
    parts = list(parts)
    if not parts:
        raise ValueError("lse_merge needs at least one part")
    o0, l0 = parts[0]
    if o0.dim() != 3:
        raise ValueError("partial outputs must be [T, H, d]")
    T, H, d = o0.shape
    arr = (MergePart * len(parts))()
    for i, (o, l) in enumerate(parts):
        if not (o.is_cuda and l.is_cuda) or tuple(o.shape) != (T, H, d) or not o.is_contiguous():
            raise ValueError(f"part {i}: o must be a contiguous CUDA tensor of shape {(T, H, d)}")
        if l.dtype != torch.float32 or tuple(l.shape) != (H, T) or not l.is_contiguous():
            raise ValueError(f"part {i}: lse must be a contiguous float32 CUDA tensor [H, T]")
        arr[i] = MergePart(o.data_ptr(), l.data_ptr(), _dtype_code(o))
    if out is None:
        out = torch.empty(T, H, d, dtype=out_dtype or o0.dtype, device=o0.device)
    elif tuple(out.shape) != (T, H, d) or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor [T, H, d]")
    if lse_out is None:
        lse_out = torch.empty(H, T, dtype=torch.float32, device=o0.device)
    elif lse_out.dtype != torch.float32 or tuple(lse_out.shape) != (H, T) or not lse_out.is_contiguous():
        raise ValueError("lse_out must be a contiguous float32 CUDA tensor [H, T]")
    if check_status and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=o0.device)
    stream = torch.cuda.current_stream(o0.device).cuda_stream
    check(load().pk_lse_merge(arr, len(parts), T, H, d, ctypes.c_void_p(out.data_ptr()),
                              _dtype_code(out), ctypes.c_void_p(lse_out.data_ptr()),
                              ctypes.c_void_p(stream),
                              ctypes.c_void_p(status.data_ptr() if status is not None else 0)),
          "pk_lse_merge")
    if check_status:
        torch.cuda.current_stream(o0.device).synchronize()
        check(int(status.item()), "pk_lse_merge (device)")
    return out, lse_out


class HostPipeline:
    """Successive steps from host buffers with the copies of one step
    overlapping the kernels of its neighbours (pk_pipeline_*).

    ``slots`` device buffer sets (dicts of CUDA tensors 'q', 'k', 'v', 'out',
    'lse' of the pk_attn_fwd shapes; allocated here when omitted) are used
    round robin; a slot's 'v' is its launch's workspace (converted to fp16
    in place).  ``submit`` enqueues one step; ``sync`` waits for all."""

    def __init__(self, plan: Plan, num_slots: int = 2, slots=None, device=None):
        import torch
        self._lib = plan._lib
        self.plan = plan
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        if slots is None:
            T, Tk, hq, hkv, d = plan.total_tokens, plan.kv_rows, plan.hq, plan.hkv, plan.head_dim
            e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device=dev)
            slots = [{"q": e(T, hq, d), "k": e(Tk, hkv, d), "v": e(Tk, hkv, d), "out": e(T, hq, d),
                      "lse": torch.empty(hq, T, dtype=torch.float32, device=dev)}
                     for _ in range(num_slots)]
        self.slots = slots
        arr = (DevSlot * len(slots))()
        for i, sl in enumerate(slots):
            arr[i] = DevSlot(sl["q"].data_ptr(), sl["k"].data_ptr(), sl["v"].data_ptr(),
                             sl["out"].data_ptr(), sl["lse"].data_ptr())
        self._h = ctypes.c_void_p()
        check(self._lib.pk_pipeline_create(plan.handle, arr, len(slots), ctypes.byref(self._h)),
              "pk_pipeline_create")
        self._inflight = []  # host tensors of submitted steps, kept alive until sync

    def submit(self, q_host, k_host, v_host, out_host, lse_host, scale: Optional[float] = None,
               status=None) -> None:
        if scale is None:
            scale = 1.0 / math.sqrt(self.plan.head_dim)
        for name, t in (("q_host", q_host), ("k_host", k_host), ("v_host", v_host),
                        ("out_host", out_host), ("lse_host", lse_host)):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host tensor")
        check(self._lib.pk_pipeline_submit(
            self._h, ctypes.c_void_p(q_host.data_ptr()), ctypes.c_void_p(k_host.data_ptr()),
            ctypes.c_void_p(v_host.data_ptr()), ctypes.c_void_p(out_host.data_ptr()),
            ctypes.c_void_p(lse_host.data_ptr()), float(scale),
            ctypes.c_void_p(status.data_ptr() if status is not None else 0)), "pk_pipeline_submit")
        self._inflight.append((q_host, k_host, v_host, out_host, lse_host, status))

    def sync(self) -> None:
        check(self._lib.pk_pipeline_sync(self._h), "pk_pipeline_sync")
        self._inflight.clear()

    def stream(self, which: int):
        """torch view of the pipeline's stream: 0 copy-in, 1 compute, 2 copy-out."""
        import torch
        return torch.cuda.ExternalStream(self._lib.pk_pipeline_stream(self._h, which))

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.pk_pipeline_destroy(self._h)  # waits for outstanding steps
            self._h = ctypes.c_void_p()
            self._inflight = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def set_wait_timeout_ns(ns: int) -> None:
    load().pk_set_wait_timeout_ns(int(ns))


def debug_wait_timeout(status, timeout_ns: int) -> None:
    """Launch the bounded-wait self-test kernel (see pk.h)."""
    import torch
    stream = torch.cuda.current_stream(status.device).cuda_stream
    check(load().pk_debug_wait_timeout(ctypes.c_void_p(status.data_ptr()), int(timeout_ns),
                                       ctypes.c_void_p(stream)), "pk_debug_wait_timeout")
