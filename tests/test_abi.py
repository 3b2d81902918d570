"""The C-ABI library loads and exports every symbol ``include/pk.h``
declares; host-side argument checks (no device work)."""
import ctypes
import os
import re

import pytest

import packed_varlen_masked_gb300 as pk
from packed_varlen_masked_gb300 import _native

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "pk.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pk_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["pk_plan_create", "pk_plan_upload", "pk_attn_fwd", "pk_plan_destroy",
                     "pk_plan_device_bytes", "pk_status_string", "pk_plan_useful_flops",
                     "pk_attn_workspace_bytes"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(pk.lib_path())
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert set(_declared_functions()) <= set(_native.SIGNATURES)


def test_status_strings():
    lib = pk.load()
    for code in range(11):
        assert lib.pk_status_string(code).decode() != "unknown status"
    assert lib.pk_status_string(pk.PK_ERR_TIMEOUT).decode() == "device wait timed out"


def test_null_and_bad_arguments_are_rejected_without_a_device():
    lib = pk.load()
    out = ctypes.c_void_p()
    assert lib.pk_plan_create(None, 1, None, 0, 4, 4, 64, 4, ctypes.byref(out)) == pk.PK_ERR_INVALID_ARG
    assert lib.pk_plan_device_bytes(None) == 0
    assert lib.pk_attn_fwd(None, None, None, None, None, None, 0.125, None, 0, None, None) \
        == pk.PK_ERR_INVALID_ARG
    plan = pk.Plan([0, 3], [(0, 3, 0)], 2, 2, 64, num_ctas=2, upload=False)
    # scale must be finite and positive
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert lib.pk_attn_fwd(plan.handle, None, None, None, None, None, bad, None, 0, None,
                               None) == pk.PK_ERR_INVALID_ARG
    # not uploaded yet
    assert lib.pk_attn_fwd(plan.handle, 16, 16, 16, 16, 16, 0.125, 16, 1 << 20, None, None) \
        == pk.PK_ERR_NOT_UPLOADED
    assert lib.pk_plan_upload(plan.handle, None, 0, None) == pk.PK_ERR_INVALID_ARG


def test_workspace_bytes_is_the_fp16_copy_of_the_value_rows():
    lib = pk.load()
    assert lib.pk_attn_workspace_bytes(None) == 0
    plan = pk.Plan([0, 300, 1000], [(0, 300, 1), (300, 700, 0)], 8, 2, 128, num_ctas=4,
                   upload=False)
    assert plan.workspace_bytes == 1000 * 2 * 128 * 2
    lay = pk.plan_layout([0, 5], [0, 300], [(0, 0, 300, 1)], 4, 1, 64, k_pos0=[0],
                         block_table=[[3, 0, 1]], num_kv_rows=512, num_ctas=2, upload=False)
    assert lay.workspace_bytes == 512 * 1 * 64 * 2  # the whole pool


def test_fp8_pv_workspace_is_the_transposed_copy_with_16_row_sequences():
    lib = pk.load()
    assert lib.pk_attn_workspace_bytes_fp8_pv(None) == 0
    # contiguous keys: every sequence's key rows rounded up to 16
    plan = pk.Plan([0, 300, 300, 1000, 1001], [(0, 300, 1), (300, 700, 0), (1000, 1, 0)], 8, 2,
                   128, num_ctas=4, upload=False)
    assert plan.workspace_bytes_fp8_pv == (304 + 704 + 16) * 2 * 128
    # paged keys: the pool's rows
    lay = pk.plan_layout([0, 5], [0, 300], [(0, 0, 300, 1)], 4, 1, 128, k_pos0=[0],
                         block_table=[[3, 0, 1]], num_kv_rows=512, num_ctas=2, upload=False)
    assert lay.workspace_bytes_fp8_pv == 512 * 1 * 128
    # no key at all: one zeroed tile for the masked reads
    nokeys = pk.plan_layout([0, 5], [0, 0], [(0, 0, 8, 0)], 4, 1, 128, q_pos0=[3], k_pos0=[0],
                            num_kv_rows=16, num_ctas=2, upload=False)
    assert nokeys.workspace_bytes_fp8_pv == 128 * 1 * 128


def test_fp8_pv_entry_argument_checks_without_a_device():
    lib = pk.load()
    plan = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 128, num_ctas=4, upload=False)
    f = lib.pk_attn_fwd_fp8_pv
    W = (16, 1 << 20)
    assert f(None, 16, 1.0, 16, 1.0, 16, 1.0, 16, 16, 0.1, *W, None, None) == pk.PK_ERR_INVALID_ARG
    for qs, ks, vs, sc in ((0.0, 1.0, 1.0, 0.1), (1.0, 1.0, -1.0, 0.1),
                           (1.0, 1.0, float("inf"), 0.1), (1.0, 1.0, float("nan"), 0.1),
                           (1.0, 1.0, 1.0, 0.0)):
        assert f(plan.handle, 16, qs, 16, ks, 16, vs, 16, 16, sc, *W, None, None) \
            == pk.PK_ERR_INVALID_ARG
    assert f(plan.handle, 16, 1.0, 16, 1.0, 16, 1.0, 16, 16, 0.1, *W, None, None) \
        == pk.PK_ERR_NOT_UPLOADED
    p64 = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 64, num_ctas=4, upload=False)
    assert f(p64.handle, 16, 1.0, 16, 1.0, 16, 1.0, 16, 16, 0.1, *W, None, None) \
        == pk.PK_ERR_UNSUPPORTED


def test_upload_rejects_small_or_misaligned_buffers_before_touching_memory():
    lib = pk.load()
    plan = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 128, num_ctas=4, upload=False)
    n = plan.device_bytes
    assert n > 0 and n % 256 == 0
    assert lib.pk_plan_upload(plan.handle, 4096, n - 1, None) == pk.PK_ERR_INVALID_ARG
    assert lib.pk_plan_upload(plan.handle, 4096 + 16, n, None) == pk.PK_ERR_ALIGNMENT


def test_lse_merge_argument_checks_without_a_device():
    lib = pk.load()
    MP = _native.MergePart
    good = (MP * 17)(*[MP(4096 * (i + 1), 8192 * (i + 1), 0) for i in range(17)])
    f = lib.pk_lse_merge
    assert f(None, 1, 4, 2, 64, 4096, 0, 4096, None, None) == pk.PK_ERR_INVALID_ARG
    assert f(good, 0, 4, 2, 64, 4096, 0, 4096, None, None) == pk.PK_ERR_INVALID_ARG
    assert f(good, 17, 4, 2, 64, 4096, 0, 4096, None, None) == pk.PK_ERR_UNSUPPORTED
    for d in (0, 12, 96, 512):
        assert f(good, 2, 4, 2, d, 4096, 0, 4096, None, None) == pk.PK_ERR_UNSUPPORTED
    assert f(good, 2, 4, 2, 64, 4096, 2, 4096, None, None) == pk.PK_ERR_INVALID_ARG   # out dtype
    assert f(good, 2, 4, 2, 64, 4096 + 8, 0, 4096, None, None) == pk.PK_ERR_ALIGNMENT
    assert f(good, 2, 4, 2, 64, 4096, 0, 4096 + 2, None, None) == pk.PK_ERR_ALIGNMENT
    bad = (MP * 2)(MP(4096, 8192, 0), MP(4096 + 4, 8192, 0))
    assert f(bad, 2, 4, 2, 64, 4096, 0, 4096, None, None) == pk.PK_ERR_ALIGNMENT
    bad = (MP * 2)(MP(4096, 8192, 0), MP(4096, 8192, 7))
    assert f(bad, 2, 4, 2, 64, 4096, 0, 4096, None, None) == pk.PK_ERR_INVALID_ARG
    bad = (MP * 2)(MP(4096, 8192, 0), MP(0, 8192, 0))
    assert f(bad, 2, 4, 2, 64, 4096, 0, 4096, None, None) == pk.PK_ERR_INVALID_ARG
    # zero rows: nothing to launch
    assert f(good, 2, 0, 2, 64, 4096, 0, 4096, None, None) == pk.PK_OK


def test_fp8_entry_argument_checks_without_a_device():
    lib = pk.load()
    plan = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 128, num_ctas=4, upload=False)
    f = lib.pk_attn_fwd_fp8
    W = (16, 1 << 20)  # workspace pointer and bytes
    assert f(None, 16, 1.0, 16, 1.0, 16, 16, 16, 0.1, *W, None, None) == pk.PK_ERR_INVALID_ARG
    for qs, ks, sc in ((0.0, 1.0, 0.1), (1.0, -1.0, 0.1), (1.0, 1.0, float("nan")),
                       (1e30, 1e30, 1e30)):
        assert f(plan.handle, 16, qs, 16, ks, 16, 16, 16, sc, *W, None, None) == pk.PK_ERR_INVALID_ARG
    assert f(plan.handle, 16, 1.0, 16, 1.0, 16, 16, 16, 0.1, *W, None, None) == pk.PK_ERR_NOT_UPLOADED
    p64 = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 64, num_ctas=4, upload=False)
    assert f(p64.handle, 16, 1.0, 16, 1.0, 16, 16, 16, 0.1, *W, None, None) == pk.PK_ERR_UNSUPPORTED


def test_pipeline_argument_checks_without_a_device():
    lib = pk.load()
    out = ctypes.c_void_p()
    plan = pk.Plan([0, 300], [(0, 300, 1)], 4, 2, 128, num_ctas=4, upload=False)
    S = _native.DevSlot
    good = (S * 2)(S(16, 16, 16, 16, 16), S(16, 16, 16, 16, 16))
    assert lib.pk_pipeline_create(None, good, 2, ctypes.byref(out)) == pk.PK_ERR_INVALID_ARG
    assert lib.pk_pipeline_create(plan.handle, None, 2, ctypes.byref(out)) == pk.PK_ERR_INVALID_ARG
    assert lib.pk_pipeline_create(plan.handle, good, 0, ctypes.byref(out)) == pk.PK_ERR_INVALID_ARG
    assert lib.pk_pipeline_create(plan.handle, good, 9, ctypes.byref(out)) == pk.PK_ERR_INVALID_ARG
    bad = (S * 1)(S(16, 16, 0, 16, 16))
    assert lib.pk_pipeline_create(plan.handle, bad, 1, ctypes.byref(out)) == pk.PK_ERR_INVALID_ARG
    assert out.value is None
    assert lib.pk_pipeline_submit(None, 16, 16, 16, 16, 16, 0.1, None) == pk.PK_ERR_INVALID_ARG
    assert lib.pk_pipeline_sync(None) == pk.PK_ERR_INVALID_ARG
    assert lib.pk_pipeline_stream(None, 0) is None
    lib.pk_pipeline_destroy(None)
