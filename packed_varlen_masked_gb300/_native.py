"""ctypes declarations of the C ABI in ``include/pk.h``."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libpk.so")
_lock = threading.Lock()
_lib = None

PK_OK = 0
PK_ERR_INVALID_ARG = 1
PK_ERR_UNSUPPORTED = 2
PK_ERR_ALIGNMENT = 3
PK_ERR_CUDA = 4
PK_ERR_TIMEOUT = 5
PK_ERR_DEVICE_CHECK = 6
PK_ERR_NOT_UPLOADED = 7
PK_ERR_OUT_OF_MEMORY = 8
PK_ERR_RANGE = 9
PK_ERR_TOO_LARGE = 10


class PKError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {status_string(status)} (pk_status {status})")


class Segment(ctypes.Structure):
    _fields_ = [("start", ctypes.c_int32), ("len", ctypes.c_int32), ("type", ctypes.c_int32)]


class SeqSegment(ctypes.Structure):
    _fields_ = [("seq", ctypes.c_int32), ("start", ctypes.c_int32), ("len", ctypes.c_int32),
                ("type", ctypes.c_int32)]


_I32P = ctypes.POINTER(ctypes.c_int32)


class Layout(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("cu_seqlens_q", _I32P), ("q_pos0", _I32P),
                ("cu_seqlens_k", _I32P), ("k_pos0", _I32P),
                ("segs", ctypes.POINTER(SeqSegment)), ("num_segs", ctypes.c_int32),
                ("block_table", _I32P), ("blocks_per_seq", ctypes.c_int32),
                ("num_kv_rows", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("num_items", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("num_full_tiles", ctypes.c_int32), ("num_partial_tiles", ctypes.c_int32),
                ("kv_rows", ctypes.c_int32), ("visible_pairs", ctypes.c_int64),
                ("useful_flops", ctypes.c_double)]


class MergePart(ctypes.Structure):
    _fields_ = [("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("dtype", ctypes.c_int32)]


PK_DTYPE_BF16 = 0
PK_DTYPE_F32 = 1


class DevSlot(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


class WorkItem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("q_start", "q_rows", "kv_start", "n_kt", "n_full", "hq0", "hq1", "hkv")]


# Every function the header declares, with its ctypes signature.
_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p
SIGNATURES = {
    "pk_plan_create": (ctypes.c_int, [_i32p, ctypes.c_int32, ctypes.POINTER(Segment),
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_vp)]),
    "pk_plan_create_layout": (ctypes.c_int, [ctypes.POINTER(Layout), ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.POINTER(_vp)]),
    "pk_plan_shard": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.POINTER(_vp)]),
    "pk_plan_set_sm_pairs": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "pk_plan_set_kv_share": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "pk_plan_kv_share": (ctypes.c_int32, [_vp]),
    "pk_plan_get_share": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int32), _vp, ctypes.c_int64,
                                         _vp, ctypes.c_int64]),
    "pk_plan_get_pairs": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int32),
                                         ctypes.POINTER(ctypes.c_int32), _vp, ctypes.c_int64,
                                         _vp, ctypes.c_int64]),
    "pk_plan_device_bytes": (ctypes.c_size_t, [_vp]),
    "pk_plan_upload": (ctypes.c_int, [_vp, _vp, ctypes.c_size_t, _vp]),
    "pk_attn_workspace_bytes": (ctypes.c_size_t, [_vp]),
    "pk_attn_workspace_bytes_fp8_pv": (ctypes.c_size_t, [_vp]),
    "pk_attn_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp,
                                   ctypes.c_size_t, _vp, _vp]),
    "pk_attn_convert_values": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]),
    "pk_attn_fwd_converted": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp,
                                             _vp]),
    "pk_attn_fwd_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp,
                                           _vp]),
    "pk_attn_fwd_fp8": (ctypes.c_int, [_vp, _vp, ctypes.c_float, _vp, ctypes.c_float, _vp, _vp,
                                       _vp, ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp]),
    "pk_attn_fwd_fp8_pv": (ctypes.c_int, [_vp, _vp, ctypes.c_float, _vp, ctypes.c_float, _vp,
                                          ctypes.c_float, _vp, _vp, ctypes.c_float, _vp,
                                          ctypes.c_size_t, _vp, _vp]),
    "pk_attn_fwd_host": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _vp, ctypes.c_float, _vp, _vp]),
    "pk_plan_destroy": (None, [_vp]),
    "pk_pipeline_create": (ctypes.c_int, [_vp, ctypes.POINTER(DevSlot), ctypes.c_int32,
                                          ctypes.POINTER(_vp)]),
    "pk_pipeline_submit": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp]),
    "pk_pipeline_sync": (ctypes.c_int, [_vp]),
    "pk_pipeline_stream": (_vp, [_vp, ctypes.c_int32]),
    "pk_pipeline_destroy": (None, [_vp]),
    "pk_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pk_plan_useful_flops": (ctypes.c_double, [_vp]),
    "pk_plan_get_info": (ctypes.c_int, [_vp, ctypes.POINTER(PlanInfo)]),
    "pk_plan_get_kv_limit": (ctypes.c_int, [_vp, _i32p, ctypes.c_int64]),
    "pk_plan_get_items": (ctypes.c_int, [_vp, ctypes.POINTER(WorkItem), ctypes.c_int64,
                                         _i32p, ctypes.c_int64]),
    "pk_lse_merge": (ctypes.c_int, [ctypes.POINTER(MergePart), ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp,
                                    _vp]),
    "pk_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "pk_debug_wait_timeout": (ctypes.c_int, [_vp, ctypes.c_uint64, _vp]),
}


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load ``_build/libpk.so``; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"packed_varlen_masked_gb300: compiled library missing at {_LIB_PATH}; "
                "run packed_varlen_masked_gb300/build.py (nvcc, sm_103a)")
        try:  # share PyTorch's CUDA runtime when it is importable
            import torch  # noqa: F401
        except Exception:
            pass
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().pk_status_string(int(status)).decode()
    except Exception:
        return "unknown"


def check(status: int, what: str) -> None:
    if status != PK_OK:
        raise PKError(status, what)
