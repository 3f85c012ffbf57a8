"""C-ABI checks that need no GPU: the library loads, exports every entry point the
header declares, and rejects bad host-side arguments before launching anything."""
import ctypes
import math
import os
import re

import pytest

from ragged_paged_attention_gb300 import api
from ragged_paged_attention_gb300 import build as rpa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    rpa_build.build()
    return api.load_library()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names.update(re.findall(r"^RPA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M))
    return names


def test_header_declares_the_four_operations():
    names = declared_symbols()
    for n in ("rpa_forward", "rpa_update_kv_cache", "mla_rpa_forward", "sparse_mla_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert names, "no declarations found"
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(api.EXPORTS) <= names
    assert lib.rpa_version() == api.ABI_VERSION


def good_rpa():
    return api.rpa_params(struct_size=ctypes.sizeof(api.rpa_params), version=1, max_num_tokens=16, num_q_heads=8,
                          num_combined_kv_heads=4, head_dim=128, total_num_pages=8, page_size=16, max_num_seqs=2,
                          pages_per_seq=4, q_dtype=1, kv_dtype=1, sm_scale=0.1, sliding_window=0, soft_cap=0.0,
                          mask_value=math.nan, k_scale=0.0, v_scale=0.0)


@pytest.mark.parametrize("field,value,code", [
    ("num_combined_kv_heads", 3, -2), ("num_q_heads", 5, -2), ("head_dim", 80, -5), ("q_dtype", 2, -3),
    ("kv_dtype", 3, -3), ("sliding_window", -1, -4), ("soft_cap", math.inf, -4), ("mask_value", math.inf, -4),
    ("version", 7, -4), ("struct_size", 4, -4), ("page_size", 0, -2), ("sm_scale", math.nan, -4),
])
def test_rpa_host_validation(lib, field, value, code):
    p = good_rpa()
    setattr(p, field, value)
    n = ctypes.c_size_t(0)
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == code
    rc = lib.rpa_forward(ctypes.byref(p), *([ctypes.c_void_p(16)] * 7), ctypes.c_void_p(256), 1 << 30, None)
    assert rc == code
    assert lib.rpa_last_error()


def test_rpa_rejects_null_and_small_workspace(lib):
    p = good_rpa()
    n = ctypes.c_size_t(0)
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value > 256
    ptrs = [ctypes.c_void_p(256 * (i + 1)) for i in range(7)]
    one = ctypes.c_void_p(256)
    assert lib.rpa_forward(ctypes.byref(p), None, *ptrs[1:], one, 1 << 30, None) == -1
    assert lib.rpa_forward(ctypes.byref(p), *ptrs, ctypes.c_void_p(4096), 16, None) == -8
    assert lib.rpa_forward(ctypes.byref(p), *ptrs, ctypes.c_void_p(4096 + 8), n.value, None) == -8
    assert lib.rpa_forward(ctypes.byref(p), *ptrs, None, n.value, None) == -8
    assert lib.rpa_forward(ctypes.byref(p), *ptrs[:6], ptrs[0], one, n.value, None) == -4  # out aliases q
    assert lib.rpa_forward(None, *ptrs, one, 1, None) == -1


def test_mla_and_sparse_host_validation(lib):
    m = api.mla_params(struct_size=ctypes.sizeof(api.mla_params), version=1, max_num_tokens=8, num_q_heads=128,
                       lkv_dim=512, r_dim=64, lkv_dim_pad=512, r_dim_pad=128, total_num_pages=4, page_size=64,
                       kv_packing=2, max_num_seqs=2, pages_per_seq=2, sm_scale=0.07, sliding_window=0,
                       soft_cap=0.0, mask_value=math.nan)
    n = ctypes.c_size_t(0)
    assert lib.mla_workspace_size(ctypes.byref(m), ctypes.byref(n)) == 0
    m.r_dim_pad = 64
    assert lib.mla_workspace_size(ctypes.byref(m), ctypes.byref(n)) == -2
    m.r_dim_pad, m.kv_packing = 128, 4
    assert lib.mla_workspace_size(ctypes.byref(m), ctypes.byref(n)) == -3
    s = api.sparse_params(struct_size=ctypes.sizeof(api.sparse_params), version=1, batch=1, num_queries=4,
                          num_heads=128, dk=576, dv=512, row_stride=640, topk=32, read_block=64, page_size=64,
                          max_pages=4, total_num_pages=4, seq_len=256, sm_scale=0.07)
    assert lib.sparse_mla_workspace_size(ctypes.byref(s), ctypes.byref(n)) == 0
    s.sm_scale = 0.0
    assert lib.sparse_mla_workspace_size(ctypes.byref(s), ctypes.byref(n)) == -4
    s.sm_scale, s.read_block = 0.07, 48
    assert lib.sparse_mla_workspace_size(ctypes.byref(s), ctypes.byref(n)) == -2
    s.read_block, s.num_heads = 64, 100
    assert lib.sparse_mla_workspace_size(ctypes.byref(s), ctypes.byref(n)) == -5


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(4, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.rpa_forward(q, q, q, q, q, q)


def test_batch_kind_is_optional_and_checked(lib):
    p = good_rpa()
    n = ctypes.c_size_t(0)
    p.batch_kind = 3
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == -4
    p.batch_kind = 2
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    # a caller built against the struct without the field: its struct_size ends before it
    p.batch_kind = 99
    p.struct_size = api.rpa_params.batch_kind.offset
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    p.struct_size = api.rpa_params.batch_kind.offset - 4
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == -4


def test_mla_query_dtype_is_optional_and_checked(lib):
    m = api.mla_params(struct_size=ctypes.sizeof(api.mla_params), version=1, max_num_tokens=8, num_q_heads=128,
                       lkv_dim=512, r_dim=64, lkv_dim_pad=512, r_dim_pad=128, total_num_pages=4, page_size=64,
                       kv_packing=2, max_num_seqs=2, pages_per_seq=2, sm_scale=0.07, sliding_window=0,
                       soft_cap=0.0, mask_value=math.nan)
    n = ctypes.c_size_t(0)
    ws = lambda: lib.mla_workspace_size(ctypes.byref(m), ctypes.byref(n))  # noqa: E731
    assert ws() == 0  # q_dtype 0 reads as bf16
    for qd, qs, code in ((api.FP8_E4M3, 0.0, 0), (api.FP8_E4M3, 0.25, 0), (api.BF16, 0.25, -4),
                         (api.FP8_E4M3, -1.0, -4), (api.FP8_E4M3, math.nan, -4), (api.INT8, 0.0, -3),
                         (api.F32, 0.0, -3)):
        m.q_dtype, m.q_scale = qd, qs
        assert ws() == code, (qd, qs)
    # a caller built against the struct without the two fields gets bf16 queries
    m.q_dtype, m.q_scale = 77, -1.0
    m.struct_size = api.mla_params.q_dtype.offset
    assert ws() == 0
    m.struct_size = api.mla_params.q_dtype.offset - 4
    assert ws() == -4


def test_head_dim_96_attention_is_bf16_only(lib):
    # 96 and 192 pass the parameter check (the cache write takes any dtype) but attention at
    # those widths needs a bf16 cache without scales: refused before anything launches
    p = good_rpa()
    p.head_dim = 96
    n = ctypes.c_size_t(0)
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    ptrs = [ctypes.c_void_p(256 * (i + 1)) for i in range(7)]
    ws = ctypes.c_void_p(1 << 20)
    for field, value in (("kv_dtype", 2), ("k_scale", 0.5), ("page_size", 12), ("mask_value", -1.5)):
        q = good_rpa()
        q.head_dim = 96
        setattr(q, field, value)
        assert lib.rpa_forward(ctypes.byref(q), *ptrs, ws, 1 << 30, None) == -5, field
        assert b"head_dim 96" in lib.rpa_last_error()
