"""fp64 CPU oracle for packed mixed-mask variable-length attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never imports, links or calls it, and it imports
nothing from the CUDA library.

The arithmetic lives in ``pk_oracle.c`` (plain C, fp64, OpenMP over rows);
this module only compiles it with gcc and marshals numpy arrays through
ctypes.  What it computes, with the passages it follows, is stated at the top
of ``pk_oracle.c``:

* packing over ``cu_seqlens`` with no cross-sequence attention
  ("[RFC]: HunyuanImage 3.0 deployment", Proposed Change, P0 "Packed
  Attention for Multi-Request Batching");
* the generalized causal mask, text causal and image tokens seeing their
  whole own segment (same page, P0 "Attention mask challenge"; "Model
  structure", item 1), materialised densely per sequence;
* grouped-query heads, query head h reading key/value head h // (Hq // Hkv);
* fp64 scores, a max-subtracted natural-log LSE and the softmax-weighted
  sum of V.

Every function here is pinned by ``tests/test_oracle.py`` against closed
forms, library special cases (textbook causal and full attention), a
hand-derived mask fixture and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pk_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libpk_oracle.so")
_lock = threading.Lock()
_lib = None

TEXT = 0
IMAGE = 1


def _fingerprint() -> str:
    """Host architecture + source bytes: a library built on another machine
    type or from another source is rebuilt, whatever the file times say."""
    import hashlib
    import platform
    h = hashlib.sha256(platform.machine().encode())
    with open(_SRC, "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile ``pk_oracle.c`` into ``_build/libpk_oracle.so`` with gcc."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    stamp = _LIB + ".stamp"
    if not force and os.path.exists(_LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == _fingerprint():
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    with open(stamp, "w") as f:
        f.write(_fingerprint())
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32p = ctypes.POINTER(ctypes.c_int32)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.pko_validate.argtypes = [i32p, ctypes.c_int32, i32p, ctypes.c_int32]
        lib.pko_validate.restype = ctypes.c_int
        lib.pko_mask_dense.argtypes = [i32p, ctypes.c_int32, i32p, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.POINTER(ctypes.c_uint8)]
        lib.pko_mask_dense.restype = ctypes.c_int
        lib.pko_visible_pairs.argtypes = [i32p, ctypes.c_int32, i32p, ctypes.c_int32]
        lib.pko_visible_pairs.restype = ctypes.c_int64
        lib.pko_row_keys.argtypes = [i32p, ctypes.c_int32, i32p, ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_int64)]
        lib.pko_row_keys.restype = ctypes.c_int
        lib.pko_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.pko_e4m3_to_double.restype = ctypes.c_double
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.pko_attention_e4m3.argtypes = [u8p, ctypes.c_double, u8p, ctypes.c_double, u16p,
                                           i32p, ctypes.c_int32, i32p, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_double, i32p, ctypes.c_int32, f64p, f64p,
                                           ctypes.c_int32]
        lib.pko_attention_e4m3.restype = ctypes.c_int
        lib.pko_attention_e4m3_v8.argtypes = [u8p, ctypes.c_double, u8p, ctypes.c_double, u8p,
                                              ctypes.c_double, i32p, ctypes.c_int32, i32p,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_double, i32p,
                                              ctypes.c_int32, f64p, f64p, ctypes.c_int32]
        lib.pko_attention_e4m3_v8.restype = ctypes.c_int
        lib.pko_attention.argtypes = [u16p, u16p, u16p, i32p, ctypes.c_int32, i32p,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_double, i32p,
                                      ctypes.c_int32, f64p, f64p, ctypes.c_int32]
        lib.pko_attention.restype = ctypes.c_int
        lib.pko_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.pko_bf16_to_double.restype = ctypes.c_double
        lib.pko_max_threads.argtypes = []
        lib.pko_max_threads.restype = ctypes.c_int32
        _lib = lib
        return lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _segs_array(segments) -> np.ndarray:
    arr = _i32(segments).reshape(-1, 3) if len(segments) else np.zeros((0, 3), np.int32)
    return np.ascontiguousarray(arr)


def _bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 bit patterns."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # local: only for tensors handed in by tests
    assert x.dtype == torch.bfloat16 and x.device.type == "cpu"
    return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))


def bf16_to_double(bits: int) -> float:
    return float(_load().pko_bf16_to_double(ctypes.c_uint16(bits)))


def validate(cu_seqlens, segments) -> int:
    cu = _i32(cu_seqlens)
    sg = _segs_array(segments)
    return int(_load().pko_validate(_ptr(cu, ctypes.c_int32), len(cu) - 1,
                                    _ptr(sg, ctypes.c_int32), sg.shape[0]))


def dense_mask(cu_seqlens, segments, s: int) -> np.ndarray:
    """The explicit L x L bool mask of sequence ``s`` (row = query)."""
    cu = _i32(cu_seqlens)
    sg = _segs_array(segments)
    L = int(cu[s + 1] - cu[s])
    M = np.zeros((L, L), dtype=np.uint8)
    rc = _load().pko_mask_dense(_ptr(cu, ctypes.c_int32), len(cu) - 1,
                                _ptr(sg, ctypes.c_int32), sg.shape[0], s,
                                _ptr(M, ctypes.c_uint8))
    if rc:
        raise ValueError(f"oracle: invalid descriptors (code {rc})")
    return M.astype(bool)


def visible_pairs(cu_seqlens, segments) -> int:
    """Visible (query, key) pairs of the pack for one head."""
    cu = _i32(cu_seqlens)
    sg = _segs_array(segments)
    n = int(_load().pko_visible_pairs(_ptr(cu, ctypes.c_int32), len(cu) - 1,
                                      _ptr(sg, ctypes.c_int32), sg.shape[0]))
    if n < 0:
        raise ValueError("oracle: invalid descriptors")
    return n


def row_keys(cu_seqlens, segments) -> np.ndarray:
    """Visible keys of every query row (int64 [T]): row sums of the mask."""
    cu = _i32(cu_seqlens)
    sg = _segs_array(segments)
    out = np.zeros(max(int(cu[-1]), 1), dtype=np.int64)
    rc = _load().pko_row_keys(_ptr(cu, ctypes.c_int32), len(cu) - 1, _ptr(sg, ctypes.c_int32),
                              sg.shape[0], _ptr(out, ctypes.c_int64))
    if rc:
        raise ValueError("oracle: invalid descriptors")
    return out[: int(cu[-1])]


def e4m3_to_double(code: int) -> float:
    """Value of an FP8 E4M3 code (OCP 8-bit format, decoded by definition)."""
    return float(_load().pko_e4m3_to_double(ctypes.c_uint8(int(code))))


def _codes(x) -> np.ndarray:
    """FP8 codes as a contiguous uint8 array (torch float8/uint8 tensor or array)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.contiguous().view(torch.uint8).cpu().numpy())
    except ImportError:
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint8))


def attention_e4m3(q8, q_scale: float, k8, k_scale: float, v, cu_seqlens, segments, hq: int,
                   hkv: int, d: int, scale: float, rows=None, nthreads: int = 0):
    """fp64 packed masked attention with E4M3 q and k (codes + one scale each)
    and bf16 v.  Returns (out [R, hq, d], lse [hq, R]) like ``attention``."""
    qb, kb, vb = _codes(q8), _codes(k8), _bits(v)
    cu = _i32(cu_seqlens)
    sg = _segs_array(segments)
    T = int(cu[-1])
    if rows is None:
        R, rp = T, None
    else:
        rr = _i32(rows)
        R, rp = rr.size, _ptr(rr, ctypes.c_int32)
    out = np.zeros((R, hq, d), dtype=np.float64)
    lse = np.zeros((hq, R), dtype=np.float64)
    rc = _load().pko_attention_e4m3(
        _ptr(qb, ctypes.c_uint8), float(q_scale), _ptr(kb, ctypes.c_uint8), float(k_scale),
        _ptr(vb, ctypes.c_uint16), _ptr(cu, ctypes.c_int32), len(cu) - 1,
        _ptr(sg, ctypes.c_int32), sg.shape[0], hq, hkv, d, float(scale), rp, R,
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), int(nthreads))
    if rc:
        raise ValueError(f"oracle: invalid arguments (code {rc})")
    return out, lse


def attention_e4m3_v8(q8, q_scale: float, k8, k_scale: float, v8, v_scale: float, cu_seqlens,
                      segments, hq: int, hkv: int, d: int, scale: float, rows=None,
                      nthreads: int = 0):
    """fp64 packed masked attention with E4M3 q, k and v (codes + one scale
    each).  Returns (out [R, hq, d], lse [hq, R]) like ``attention``."""
    qb, kb, vb = _codes(q8), _codes(k8), _codes(v8)
    cu = _i32(cu_seqlens)
    sg = _segs_array(segments)
    T = int(cu[-1])
    if rows is None:
        R, rp = T, None
    else:
        rr = _i32(rows)
        R, rp = rr.size, _ptr(rr, ctypes.c_int32)
    out = np.zeros((R, hq, d), dtype=np.float64)
    lse = np.zeros((hq, R), dtype=np.float64)
    rc = _load().pko_attention_e4m3_v8(
        _ptr(qb, ctypes.c_uint8), float(q_scale), _ptr(kb, ctypes.c_uint8), float(k_scale),
        _ptr(vb, ctypes.c_uint8), float(v_scale), _ptr(cu, ctypes.c_int32), len(cu) - 1,
        _ptr(sg, ctypes.c_int32), sg.shape[0], hq, hkv, d, float(scale), rp, R,
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), int(nthreads))
    if rc:
        raise ValueError(f"oracle: invalid arguments (code {rc})")
    return out, lse


def attention(q, k, v, cu_seqlens, segments, hq: int, hkv: int, d: int,
              scale: float, rows=None, nthreads: int = 0):
    """fp64 packed masked attention.

    q: bf16 [T, hq, d]; k, v: bf16 [T, hkv, d] (torch CPU tensors or uint16
    bit arrays).  Returns (out fp64 [R, hq, d], lse fp64 [hq, R]) with R = T,
    or R = len(rows) when ``rows`` lists global token indices.
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cu = _i32(cu_seqlens)
    sg = _segs_array(segments)
    T = int(cu[-1])
    assert qb.size == T * hq * d and kb.size == T * hkv * d and vb.size == T * hkv * d
    if rows is None:
        R, rp, nr = T, None, 0
    else:
        rr = _i32(rows)
        R, rp, nr = rr.size, _ptr(rr, ctypes.c_int32), rr.size
    out = np.zeros((R, hq, d), dtype=np.float64)
    lse = np.zeros((hq, R), dtype=np.float64)
    rc = _load().pko_attention(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                               _ptr(vb, ctypes.c_uint16), _ptr(cu, ctypes.c_int32),
                               len(cu) - 1, _ptr(sg, ctypes.c_int32), sg.shape[0],
                               hq, hkv, d, float(scale), rp, nr,
                               _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
                               int(nthreads))
    if rc:
        raise ValueError(f"oracle: invalid arguments (code {rc})")
    return out, lse


def max_threads() -> int:
    return int(_load().pko_max_threads())


def _load_general():
    lib = _load()
    if not hasattr(lib, "_general_ready"):
        i32p = ctypes.POINTER(ctypes.c_int32)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.pko_attention_general.argtypes = [
            u16p, u16p, u16p, i32p, i32p, i32p, i32p, ctypes.c_int32, i32p, i32p, i32p, i32p,
            ctypes.c_int32, i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_double, f64p, f64p, ctypes.c_int32]
        lib.pko_attention_general.restype = ctypes.c_int
        lib.pko_lse_merge.argtypes = [f64p, f64p, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, f64p, f64p]
        lib.pko_lse_merge.restype = None
        lib._general_ready = True
    return lib


def attention_general(q, k, v, cu_seqlens_q, cu_seqlens_k, q_pos0, k_pos0, seq_segments,
                      hq: int, hkv: int, d: int, scale: float, block_table=None,
                      block: int = 128, nthreads: int = 0):
    """fp64 attention of queries over keys that are position ranges of their
    sequences (see pk_oracle.c).  ``seq_segments``: (seq, start, len, type)
    rows in sequence-position space.  ``block_table`` [S, blocks_per_seq]
    places key position p of sequence s at pool row table[s, p // block] *
    block + p % block.  Returns (out [Tq, hq, d], lse [hq, Tq]); rows that
    see no key get out 0 and lse -inf."""
    lib = _load_general()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    qp, kp = _i32(q_pos0), _i32(k_pos0)
    sg = _i32(seq_segments).reshape(-1, 4)
    cols = [np.ascontiguousarray(sg[:, i]) for i in range(4)]
    S = len(cq) - 1
    Tq = int(cq[-1])
    if block_table is None:
        bt, bps, bp = None, 0, None
    else:
        bt = _i32(block_table).reshape(S, -1)
        bps = bt.shape[1]
        bp = _ptr(np.ascontiguousarray(bt), ctypes.c_int32)
    out = np.zeros((Tq, hq, d), dtype=np.float64)
    lse = np.zeros((hq, Tq), dtype=np.float64)
    rc = lib.pko_attention_general(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        _ptr(cq, ctypes.c_int32), _ptr(ck, ctypes.c_int32), _ptr(qp, ctypes.c_int32),
        _ptr(kp, ctypes.c_int32), S, *[_ptr(c, ctypes.c_int32) for c in cols], sg.shape[0],
        bp, bps, block, hq, hkv, d, float(scale), _ptr(out, ctypes.c_double),
        _ptr(lse, ctypes.c_double), int(nthreads))
    if rc:
        raise ValueError(f"oracle: invalid arguments (code {rc})")
    return out, lse


def lse_merge(o_parts, lse_parts):
    """Merge partial attentions over disjoint key sets: o_parts [C, T, H, d],
    lse_parts [C, H, T] (fp64) -> (out [T, H, d], lse [H, T])."""
    lib = _load_general()
    o = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    C, T, H, d = o.shape
    out = np.zeros((T, H, d), dtype=np.float64)
    lse = np.zeros((H, T), dtype=np.float64)
    lib.pko_lse_merge(_ptr(o, ctypes.c_double), _ptr(l, ctypes.c_double), C, T, H, d,
                      _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    return out, lse
