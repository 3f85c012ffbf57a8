"""Python binding of ``librpa_gb300.so`` (the C ABI in ``include/rpa.h``).

Argument marshalling only: each function checks dtypes/shapes, turns torch CUDA
tensors into pointers and sizes, and calls the C entry point of the same name on
the current torch stream.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback.  When the library or a CUDA device is missing
the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librpa_gb300.so")
ABI_VERSION = 1

BF16, FP8_E4M3, F32, INT8, INT4 = 1, 2, 3, 4, 5

STATUS = {0: "RPA_OK", -1: "RPA_ERR_NULL", -2: "RPA_ERR_SHAPE", -3: "RPA_ERR_DTYPE", -4: "RPA_ERR_VALUE",
          -5: "RPA_ERR_UNSUPPORTED", -6: "RPA_ERR_CUDA", -7: "RPA_ERR_DEVICE_CHECK", -8: "RPA_ERR_WORKSPACE"}

EXPORTS = ("rpa_workspace_size", "rpa_forward", "rpa_update_kv_cache", "mla_workspace_size",
           "mla_update_kv_cache", "mla_rpa_forward", "sparse_mla_workspace_size", "sparse_mla_forward",
           "rpa_check_device_status", "rpa_last_error", "rpa_version", "rpa_profile_enable",
           "rpa_profile_reset", "rpa_profile_read", "rpa_forward_noalloc", "rpa_launch_count",
           "rpa_forward_update", "sparse_mla_ragged_workspace_size", "sparse_mla_write_and_attend_ragged",
           "rpa_selftest_bounded_wait")


class RpaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class rpa_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


class rpa_params(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("version", ctypes.c_uint32),
                ("max_num_tokens", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_combined_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("total_num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_num_seqs", ctypes.c_int32), ("pages_per_seq", ctypes.c_int32),
                ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("sliding_window", ctypes.c_int32), ("soft_cap", ctypes.c_float), ("mask_value", ctypes.c_float),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float), ("batch_kind", ctypes.c_int32)]


BATCH_MIXED, BATCH_DECODE_ONLY, BATCH_PREFILL_ONLY = 0, 1, 2


class mla_params(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("version", ctypes.c_uint32),
                ("max_num_tokens", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("lkv_dim", ctypes.c_int32), ("r_dim", ctypes.c_int32), ("lkv_dim_pad", ctypes.c_int32),
                ("r_dim_pad", ctypes.c_int32), ("total_num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("kv_packing", ctypes.c_int32), ("max_num_seqs", ctypes.c_int32),
                ("pages_per_seq", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("sliding_window", ctypes.c_int32), ("soft_cap", ctypes.c_float), ("mask_value", ctypes.c_float),
                ("q_dtype", ctypes.c_int32), ("q_scale", ctypes.c_float)]


class sparse_params(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("version", ctypes.c_uint32), ("batch", ctypes.c_int32),
                ("num_queries", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("row_stride", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("read_block", ctypes.c_int32), ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("total_num_pages", ctypes.c_int32), ("seq_len", ctypes.c_int32), ("sm_scale", ctypes.c_float)]


class sparse_ragged_params(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("version", ctypes.c_uint32), ("num_tokens", ctypes.c_int32),
                ("num_seqs", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("rope", ctypes.c_int32), ("row_stride", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("read_block", ctypes.c_int32), ("page_size", ctypes.c_int32), ("num_page_ids", ctypes.c_int32),
                ("total_num_pages", ctypes.c_int32), ("sm_scale", ctypes.c_float)]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (raises when it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with ragged_paged_attention_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        szp = ctypes.POINTER(ctypes.c_size_t)
        lib.rpa_version.restype = ctypes.c_int
        lib.rpa_last_error.restype = ctypes.c_char_p
        lib.rpa_workspace_size.argtypes = [ctypes.POINTER(rpa_params), szp]
        lib.rpa_forward.argtypes = [ctypes.POINTER(rpa_params), P, P, P, P, P, P, P, P, sz, P]
        lib.rpa_forward_noalloc.argtypes = [ctypes.POINTER(rpa_params), P, P, P, P, P, P, P, P]
        lib.rpa_update_kv_cache.argtypes = [ctypes.POINTER(rpa_params), P, P, P, P, P, P, P, P, sz, P]
        lib.rpa_forward_update.argtypes = [ctypes.POINTER(rpa_params), P, P, P, P, P, P, P, P, P, P, sz, P]
        lib.mla_workspace_size.argtypes = [ctypes.POINTER(mla_params), szp]
        lib.mla_update_kv_cache.argtypes = [ctypes.POINTER(mla_params), P, P, P, P, P, P, P, P, P, sz, P]
        lib.mla_rpa_forward.argtypes = [ctypes.POINTER(mla_params), P, P, P, P, P, P, P, P, P, P, P, P, sz, P]
        lib.sparse_mla_workspace_size.argtypes = [ctypes.POINTER(sparse_params), szp]
        lib.sparse_mla_forward.argtypes = [ctypes.POINTER(sparse_params), P, P, P, P, P, P, P, sz, P]
        lib.sparse_mla_ragged_workspace_size.argtypes = [ctypes.POINTER(sparse_ragged_params), szp]
        lib.sparse_mla_write_and_attend_ragged.argtypes = [ctypes.POINTER(sparse_ragged_params)] + [P] * 14 + [sz, P]
        lib.rpa_check_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
        lib.rpa_selftest_bounded_wait.argtypes = [P, sz, P]
        lib.rpa_profile_enable.argtypes = [ctypes.c_int]
        lib.rpa_profile_reset.argtypes = []
        lib.rpa_profile_read.argtypes = [ctypes.POINTER(rpa_kernel_time), ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        lib.rpa_launch_count.argtypes = []
        lib.rpa_launch_count.restype = ctypes.c_int64
        for name in EXPORTS:
            if name not in ("rpa_last_error",):
                getattr(lib, name).restype = ctypes.c_int
        if lib.rpa_version() != ABI_VERSION:
            raise RuntimeError(f"library ABI {lib.rpa_version()} != binding ABI {ABI_VERSION}")
        _lib = lib
        return lib


def _check(rc: int):
    if rc != 0:
        msg = _lib.rpa_last_error().decode() if _lib is not None else ""
        raise RpaError(rc, msg)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _opt(x, default=0.0):
    return default if x is None else x


class Workspace:
    """A zero-initialised device buffer reused across calls (one per device and purpose)."""

    _cache: dict = {}

    @classmethod
    def get(cls, nbytes: int, device, tag: str = "default") -> torch.Tensor:
        key = (str(device), tag)
        buf = cls._cache.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            cls._cache[key] = buf
        return buf


def _kv_code(dtype) -> int:
    if dtype == torch.bfloat16:
        return BF16
    if dtype == torch.float8_e4m3fn:
        return FP8_E4M3
    if dtype == torch.int8:
        return INT8
    if dtype == torch.uint8:  # int4 values packed two a byte (element 2i in the low nibble of byte i)
        return INT4
    raise ValueError(f"unsupported KV dtype {dtype}")


def kv_head_dim(kv_pages) -> int:
    """Head dim of a cache tensor: its last dim, twice that for a packed int4 (uint8) cache."""
    return kv_pages.shape[-1] * (2 if kv_pages.dtype == torch.uint8 else 1)


def make_rpa_params(q, kv_pages, page_indices, *, sm_scale=1.0, sliding_window=None, soft_cap=None,
                    mask_value=None, k_scale=None, v_scale=None, batch_kind=BATCH_MIXED) -> rpa_params:
    P, ps, C, _ = kv_pages.shape
    D = kv_head_dim(kv_pages)
    max_num_seqs, pps = page_indices.shape
    return rpa_params(
        struct_size=ctypes.sizeof(rpa_params), version=ABI_VERSION, max_num_tokens=q.shape[0],
        num_q_heads=q.shape[1], num_combined_kv_heads=C, head_dim=D, total_num_pages=P, page_size=ps,
        max_num_seqs=max_num_seqs, pages_per_seq=pps, q_dtype=BF16, kv_dtype=_kv_code(kv_pages.dtype),
        sm_scale=float(sm_scale), sliding_window=int(_opt(sliding_window, 0)), soft_cap=float(_opt(soft_cap)),
        mask_value=math.nan if mask_value is None else float(mask_value), k_scale=float(_opt(k_scale)),
        v_scale=float(_opt(v_scale)), batch_kind=int(batch_kind))


def rpa_workspace_size(params: rpa_params) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib.rpa_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def rpa_forward(q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, *, sm_scale=1.0, sliding_window=None,
                soft_cap=None, mask_value=None, k_scale=None, v_scale=None, out=None, workspace=None,
                batch_kind=BATCH_MIXED):
    """Ragged paged attention; returns ``out`` [max_num_tokens, Hq, D] bf16.  ``batch_kind``
    (BATCH_DECODE_ONLY / BATCH_PREFILL_ONLY) lets the library skip the other class's launches."""
    lib = load_library()
    _dev(q, "q", torch.bfloat16)
    _dev(kv_pages, "kv_pages")
    for n, t in (("kv_lens", kv_lens), ("page_indices", page_indices), ("cu_q_lens", cu_q_lens),
                 ("num_seqs", num_seqs)):
        _dev(t, n, torch.int32)
    prm = make_rpa_params(q, kv_pages, page_indices, sm_scale=sm_scale, sliding_window=sliding_window,
                          soft_cap=soft_cap, mask_value=mask_value, k_scale=k_scale, v_scale=v_scale,
                          batch_kind=batch_kind)
    if kv_lens.numel() != prm.max_num_seqs or cu_q_lens.numel() != prm.max_num_seqs + 1 or num_seqs.numel() != 1:
        raise ValueError("kv_lens must be [max_num_seqs], cu_q_lens [max_num_seqs + 1], num_seqs [1]")
    if kv_head_dim(kv_pages) != q.shape[-1]:
        raise ValueError("q and kv_pages head_dim differ")
    if out is None:
        out = torch.empty_like(q)
    elif tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out must have q's shape {tuple(q.shape)}, got {tuple(out.shape)}")
    _dev(out, "out", torch.bfloat16)
    if workspace is None:
        workspace = Workspace.get(rpa_workspace_size(prm), q.device, "rpa")
    _check(lib.rpa_forward(ctypes.byref(prm), _ptr(q), _ptr(kv_pages), _ptr(kv_lens), _ptr(page_indices),
                           _ptr(cu_q_lens), _ptr(num_seqs), _ptr(out), _ptr(workspace), workspace.numel(),
                           _stream()))
    return out


def _header_noalloc_bytes() -> int:
    """RPA_NOALLOC_SCRATCH_BYTES as ``include/rpa.h`` defines it (the one definition of the
    size; the binding reads it instead of restating it)."""
    path = os.path.join(os.path.dirname(_HERE), "include", "rpa.h")
    with open(path) as f:
        m = re.search(r"#define\s+RPA_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", f.read())
    if m is None:
        raise RuntimeError(f"RPA_NOALLOC_SCRATCH_BYTES not found in {path}")
    return int(m.group(1)) << int(m.group(2))


NOALLOC_SCRATCH_BYTES = _header_noalloc_bytes()


def rpa_forward_noalloc(q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, *, out, sm_scale=1.0,
                        sliding_window=None, soft_cap=None, mask_value=None, k_scale=None, v_scale=None):
    """rpa_forward through the entry point that allocates nothing.

    For callers that cannot allocate device memory (their host application's memory
    manager owns the GPU, or allocation is not allowed once serving has started): the
    library uses its own fixed scratch array instead of a workspace, so ``out`` must be
    given.  Overlapping calls race on that array; problems needing more than
    ``NOALLOC_SCRATCH_BYTES`` of scratch raise ``RpaError`` (RPA_ERR_WORKSPACE).
    """
    # shapes first: the C call sees only pointers, so a q narrower than the cache or an
    # out smaller than q would be read or written past its end
    if kv_head_dim(kv_pages) != q.shape[-1]:
        raise ValueError("q and kv_pages head_dim differ")
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out must have q's shape {tuple(q.shape)}, got {tuple(out.shape)}")
    lib = load_library()
    _dev(q, "q", torch.bfloat16)
    _dev(kv_pages, "kv_pages")
    _dev(out, "out", torch.bfloat16)
    for n, t in (("kv_lens", kv_lens), ("page_indices", page_indices), ("cu_q_lens", cu_q_lens),
                 ("num_seqs", num_seqs)):
        _dev(t, n, torch.int32)
    prm = make_rpa_params(q, kv_pages, page_indices, sm_scale=sm_scale, sliding_window=sliding_window,
                          soft_cap=soft_cap, mask_value=mask_value, k_scale=k_scale, v_scale=v_scale)
    if kv_lens.numel() != prm.max_num_seqs or cu_q_lens.numel() != prm.max_num_seqs + 1 or num_seqs.numel() != 1:
        raise ValueError("kv_lens must be [max_num_seqs], cu_q_lens [max_num_seqs + 1], num_seqs [1]")
    _check(lib.rpa_forward_noalloc(ctypes.byref(prm), _ptr(q), _ptr(kv_pages), _ptr(kv_lens), _ptr(page_indices),
                                   _ptr(cu_q_lens), _ptr(num_seqs), _ptr(out), _stream()))
    return out


def rpa_update_kv_cache(new_k, new_v, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, *, workspace=None):
    """Scatter new K/V [max_num_tokens, Hkv, D] into ``kv_pages`` in place; returns ``kv_pages``."""
    lib = load_library()
    _dev(kv_pages, "kv_pages")
    _dev(new_k, "new_k", kv_pages.dtype)
    _dev(new_v, "new_v", kv_pages.dtype)
    for n, t in (("kv_lens", kv_lens), ("page_indices", page_indices), ("cu_q_lens", cu_q_lens),
                 ("num_seqs", num_seqs)):
        _dev(t, n, torch.int32)
    if new_k.shape != new_v.shape or new_k.shape[1] * 2 != kv_pages.shape[2] or new_k.shape[2] != kv_pages.shape[3]:
        raise ValueError("new_k/new_v must be [max_num_tokens, num_kv_heads, head_dim]")
    fake_q = torch.empty((new_k.shape[0], new_k.shape[1]), device="meta")
    prm = make_rpa_params(fake_q, kv_pages, page_indices)
    if workspace is None:
        workspace = Workspace.get(256, kv_pages.device, "update")
    _check(lib.rpa_update_kv_cache(ctypes.byref(prm), _ptr(new_k), _ptr(new_v), _ptr(kv_pages), _ptr(kv_lens),
                                   _ptr(page_indices), _ptr(cu_q_lens), _ptr(num_seqs), _ptr(workspace),
                                   workspace.numel(), _stream()))
    return kv_pages


def rpa_forward_update(q, new_k, new_v, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, *, sm_scale=1.0,
                       sliding_window=None, soft_cap=None, mask_value=None, k_scale=None, v_scale=None, out=None,
                       workspace=None, batch_kind=BATCH_MIXED):
    """rpa_update_kv_cache then rpa_forward in one call (the cache write shares the plan's
    launch); writes ``kv_pages`` in place and returns ``out``."""
    lib = load_library()
    _dev(q, "q", torch.bfloat16)
    _dev(kv_pages, "kv_pages")
    _dev(new_k, "new_k", kv_pages.dtype)
    _dev(new_v, "new_v", kv_pages.dtype)
    for n, t in (("kv_lens", kv_lens), ("page_indices", page_indices), ("cu_q_lens", cu_q_lens),
                 ("num_seqs", num_seqs)):
        _dev(t, n, torch.int32)
    prm = make_rpa_params(q, kv_pages, page_indices, sm_scale=sm_scale, sliding_window=sliding_window,
                          soft_cap=soft_cap, mask_value=mask_value, k_scale=k_scale, v_scale=v_scale,
                          batch_kind=batch_kind)
    if kv_lens.numel() != prm.max_num_seqs or cu_q_lens.numel() != prm.max_num_seqs + 1 or num_seqs.numel() != 1:
        raise ValueError("kv_lens must be [max_num_seqs], cu_q_lens [max_num_seqs + 1], num_seqs [1]")
    if kv_head_dim(kv_pages) != q.shape[-1]:
        raise ValueError("q and kv_pages head_dim differ")
    if (new_k.shape != new_v.shape or new_k.shape[0] != q.shape[0] or new_k.shape[1] * 2 != kv_pages.shape[2]
            or new_k.shape[2] != kv_pages.shape[3]):
        raise ValueError("new_k/new_v must be [max_num_tokens, num_kv_heads, head_dim]")
    if out is None:
        out = torch.empty_like(q)
    elif tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out must have q's shape {tuple(q.shape)}, got {tuple(out.shape)}")
    _dev(out, "out", torch.bfloat16)
    if workspace is None:
        workspace = Workspace.get(rpa_workspace_size(prm), q.device, "rpa")
    _check(lib.rpa_forward_update(ctypes.byref(prm), _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(kv_pages),
                                  _ptr(kv_lens), _ptr(page_indices), _ptr(cu_q_lens), _ptr(num_seqs), _ptr(out),
                                  _ptr(workspace), workspace.numel(), _stream()))
    return out


def make_mla_params(ql_nope, q_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, *, sm_scale=1.0,
                    sliding_window=None, soft_cap=None, mask_value=None, q_scale=None) -> mla_params:
    P, ps_pk, pk, lkv_pad = cache_kv_c.shape
    max_num_seqs = kv_lens.numel()
    fp8 = ql_nope.dtype == torch.float8_e4m3fn
    return mla_params(
        struct_size=ctypes.sizeof(mla_params), version=ABI_VERSION, max_num_tokens=ql_nope.shape[0],
        num_q_heads=ql_nope.shape[1], lkv_dim=ql_nope.shape[2], r_dim=q_pe.shape[2], lkv_dim_pad=lkv_pad,
        r_dim_pad=cache_k_pe.shape[-1], total_num_pages=P, page_size=ps_pk * pk, kv_packing=pk,
        max_num_seqs=max_num_seqs, pages_per_seq=page_indices.numel() // max_num_seqs, sm_scale=float(sm_scale),
        sliding_window=int(_opt(sliding_window, 0)), soft_cap=float(_opt(soft_cap)),
        mask_value=math.nan if mask_value is None else float(mask_value),
        q_dtype=FP8_E4M3 if fp8 else BF16, q_scale=float(_opt(q_scale)) if fp8 else 0.0)


def mla_workspace_size(params: mla_params) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib.mla_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def _check_mla(ql_nope, q_pe, new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, cu_q_lens,
               distribution):
    qdt = torch.float8_e4m3fn if ql_nope.dtype == torch.float8_e4m3fn else torch.bfloat16
    for n, t in (("ql_nope", ql_nope), ("q_pe", q_pe)):
        _dev(t, n, qdt)
    for n, t in (("new_kv_c", new_kv_c), ("new_k_pe", new_k_pe), ("cache_kv_c", cache_kv_c),
                 ("cache_k_pe", cache_k_pe)):
        _dev(t, n, torch.bfloat16)
    for n, t in (("kv_lens", kv_lens), ("page_indices", page_indices), ("cu_q_lens", cu_q_lens),
                 ("distribution", distribution)):
        _dev(t, n, torch.int32)
    if cu_q_lens.numel() != kv_lens.numel() + 1 or distribution.numel() != 3:
        raise ValueError("cu_q_lens must be [max_num_seqs + 1] and distribution [3]")
    if page_indices.numel() % kv_lens.numel():
        raise ValueError("page_indices must hold max_num_seqs * pages_per_seq entries")


def mla_update_kv_cache(new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, cu_q_lens,
                        distribution, *, workspace=None):
    """MLA cache scatter, in place; returns ``(cache_kv_c, cache_k_pe)``."""
    lib = load_library()
    T = new_kv_c.shape[0]
    fake_ql = torch.empty((T, 1, new_kv_c.shape[1]), device="meta")
    fake_qr = torch.empty((T, 1, new_k_pe.shape[1]), device="meta")
    _check_mla(new_kv_c.unsqueeze(1), new_k_pe.unsqueeze(1), new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens,
               page_indices, cu_q_lens, distribution)
    prm = make_mla_params(fake_ql, fake_qr, cache_kv_c, cache_k_pe, kv_lens, page_indices)
    if workspace is None:
        workspace = Workspace.get(256, cache_kv_c.device, "update")
    _check(lib.mla_update_kv_cache(ctypes.byref(prm), _ptr(new_kv_c), _ptr(new_k_pe), _ptr(cache_kv_c),
                                   _ptr(cache_k_pe), _ptr(kv_lens), _ptr(page_indices), _ptr(cu_q_lens),
                                   _ptr(distribution), _ptr(workspace), workspace.numel(), _stream()))
    return cache_kv_c, cache_k_pe


def mla_rpa_forward(ql_nope, q_pe, new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, cu_q_lens,
                    distribution, *, sm_scale=1.0, sliding_window=None, soft_cap=None, mask_value=None, q_scale=None,
                    out=None, workspace=None):
    """MLA update_kv_cache + attention; returns ``out`` [max_num_tokens, H, lkv] bf16 (caches updated in place).

    ``ql_nope`` and ``q_pe`` are bf16, or both float8_e4m3fn with ``q_scale`` multiplying the
    scores after ``sm_scale``."""
    lib = load_library()
    _check_mla(ql_nope, q_pe, new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, cu_q_lens,
               distribution)
    if q_scale is not None and ql_nope.dtype != torch.float8_e4m3fn:
        raise ValueError("q_scale applies to float8_e4m3fn queries only")
    prm = make_mla_params(ql_nope, q_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, sm_scale=sm_scale,
                          sliding_window=sliding_window, soft_cap=soft_cap, mask_value=mask_value, q_scale=q_scale)
    if out is None:
        out = torch.empty(ql_nope.shape, dtype=torch.bfloat16, device=ql_nope.device)
    _dev(out, "out", torch.bfloat16)
    if workspace is None:
        workspace = Workspace.get(mla_workspace_size(prm), ql_nope.device, "mla")
    _check(lib.mla_rpa_forward(ctypes.byref(prm), _ptr(ql_nope), _ptr(q_pe), _ptr(new_kv_c), _ptr(new_k_pe),
                               _ptr(cache_kv_c), _ptr(cache_k_pe), _ptr(kv_lens), _ptr(page_indices),
                               _ptr(cu_q_lens), _ptr(distribution), _ptr(out), _ptr(workspace), workspace.numel(),
                               _stream()))
    return out


def make_sparse_params(q, cache, indices, page_table, *, read_block, page_size, seq_len, sm_scale,
                       dv=512) -> sparse_params:
    B, S, H, Dk = q.shape
    row_stride = cache.shape[-1]
    P = cache.numel() // (page_size * row_stride)
    return sparse_params(
        struct_size=ctypes.sizeof(sparse_params), version=ABI_VERSION, batch=B, num_queries=S, num_heads=H, dk=Dk,
        dv=dv, row_stride=row_stride, topk=indices.shape[-1], read_block=read_block, page_size=page_size,
        max_pages=page_table.shape[-1], total_num_pages=P, seq_len=seq_len, sm_scale=float(sm_scale))


def sparse_mla_workspace_size(params: sparse_params) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib.sparse_mla_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def sparse_mla_forward(q, cache, indices, positions, page_table, *, read_block, page_size, seq_len, sm_scale,
                       dv=512, out=None, workspace=None):
    """DSA sparse MLA; returns ``out`` [B, S, H, dv] float32."""
    lib = load_library()
    _dev(q, "q", torch.bfloat16)
    _dev(cache, "cache", torch.bfloat16)
    for n, t in (("indices", indices), ("positions", positions), ("page_table", page_table)):
        _dev(t, n, torch.int32)
    B, S, H, _ = q.shape
    if indices.shape[:2] != (B, S) or positions.shape != (B, S) or page_table.shape[0] != B:
        raise ValueError("indices [B, S, K], positions [B, S] and page_table [B, max_pages] must match q")
    if sm_scale is None:
        raise ValueError("sm_scale is required")
    prm = make_sparse_params(q, cache, indices, page_table, read_block=read_block, page_size=page_size,
                             seq_len=seq_len, sm_scale=sm_scale, dv=dv)
    if out is None:
        out = torch.empty((B, S, H, dv), dtype=torch.float32, device=q.device)
    _dev(out, "out", torch.float32)
    if workspace is None:
        workspace = Workspace.get(sparse_mla_workspace_size(prm), q.device, "sparse")
    _check(lib.sparse_mla_forward(ctypes.byref(prm), _ptr(q), _ptr(cache), _ptr(indices), _ptr(positions),
                                  _ptr(page_table), _ptr(out), _ptr(workspace), workspace.numel(), _stream()))
    return out


def make_sparse_ragged_params(ql, qpe, cache, topk, seq_lens, page_indices, *, read_block, page_size,
                              sm_scale) -> sparse_ragged_params:
    T, H, dv = ql.shape
    row_stride = cache.shape[-1]
    return sparse_ragged_params(
        struct_size=ctypes.sizeof(sparse_ragged_params), version=ABI_VERSION, num_tokens=T, num_seqs=seq_lens.numel(),
        num_heads=H, dv=dv, rope=qpe.shape[-1], row_stride=row_stride, topk=topk.shape[-1], read_block=read_block,
        page_size=page_size, num_page_ids=page_indices.numel(),
        total_num_pages=cache.numel() // (page_size * row_stride), sm_scale=float(sm_scale))


def sparse_mla_ragged_workspace_size(params: sparse_ragged_params) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib.sparse_mla_ragged_workspace_size(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def sparse_mla_write_and_attend_ragged(ql, qpe, kvc, kpe, cache, topk, positions, loc, seq_lens, cu_q_lens,
                                       cu_kv_lens, page_indices, *, read_block, page_size, sm_scale, out=None,
                                       workspace=None):
    """Packed-ragged sparse MLA with the self-write: writes ``kvc``/``kpe`` rows (may be None,
    with ``loc``) into ``cache`` in place, then attends; returns ``out`` [T, H, dv] float32."""
    lib = load_library()
    for n, t in (("ql", ql), ("qpe", qpe), ("cache", cache)):
        _dev(t, n, torch.bfloat16)
    for n, t in (("topk", topk), ("positions", positions), ("seq_lens", seq_lens), ("cu_q_lens", cu_q_lens),
                 ("cu_kv_lens", cu_kv_lens), ("page_indices", page_indices)):
        _dev(t, n, torch.int32)
    T, H, dv = ql.shape
    if qpe.shape[:2] != (T, H) or topk.shape[0] != T or positions.numel() != T:
        raise ValueError("qpe [T, H, rope], topk [T, K] and positions [T] must match ql [T, H, dv]")
    if cu_q_lens.numel() != seq_lens.numel() + 1 or cu_kv_lens.numel() != seq_lens.numel() + 1:
        raise ValueError("cu_q_lens and cu_kv_lens must have num_seqs + 1 entries")
    if (kvc is None) != (kpe is None) or (kvc is None) != (loc is None):
        raise ValueError("kvc, kpe and loc go together")
    if kvc is not None:
        _dev(kvc, "kvc", torch.bfloat16)
        _dev(kpe, "kpe", torch.bfloat16)
        _dev(loc, "loc", torch.int32)
        if kvc.shape != (T, dv) or kpe.shape != (T, qpe.shape[-1]) or loc.numel() != T:
            raise ValueError("kvc [T, dv], kpe [T, rope] and loc [T] must match ql")
    if sm_scale is None:
        raise ValueError("sm_scale is required")
    prm = make_sparse_ragged_params(ql, qpe, cache, topk, seq_lens, page_indices, read_block=read_block,
                                    page_size=page_size, sm_scale=sm_scale)
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.float32, device=ql.device)
    _dev(out, "out", torch.float32)
    if workspace is None:
        workspace = Workspace.get(sparse_mla_ragged_workspace_size(prm), ql.device, "sparse_ragged")
    _check(lib.sparse_mla_write_and_attend_ragged(
        ctypes.byref(prm), _ptr(ql), _ptr(qpe), _ptr(kvc), _ptr(kpe), _ptr(cache), _ptr(topk), _ptr(positions),
        _ptr(loc), _ptr(seq_lens), _ptr(cu_q_lens), _ptr(cu_kv_lens), _ptr(page_indices), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream()))
    return out


def selftest_bounded_wait(workspace: torch.Tensor) -> None:
    """Launch the failure-path check (a bounded wait that runs out after 2 s and records
    RPA_DEV_ERR_TIMEOUT in ``workspace``'s error word)."""
    _check(load_library().rpa_selftest_bounded_wait(_ptr(workspace), workspace.numel(), _stream()))


def check_device_status(workspace: torch.Tensor) -> int:
    """Synchronise, read and clear the workspace error word; returns its bits (0 = fine)."""
    lib = load_library()
    bits = ctypes.c_uint32(0)
    rc = lib.rpa_check_device_status(_ptr(workspace), ctypes.byref(bits), _stream())
    if rc not in (0, -7):
        _check(rc)
    return bits.value


def launch_count() -> int:
    """Kernels the library has launched since it was loaded (``rpa_launch_count``)."""
    return int(load_library().rpa_launch_count())


class KernelTimer:
    """Per-kernel CUDA-event timing of the library's own launches (``rpa_profile_*``).

    ``with KernelTimer() as kt: ...`` then ``kt.result`` maps kernel name to
    ``(launches, total_ms)``.
    """

    def __enter__(self):
        lib = load_library()
        _check(lib.rpa_profile_reset())
        _check(lib.rpa_profile_enable(1))
        self.result = {}
        return self

    def __exit__(self, *exc):
        lib = load_library()
        _check(lib.rpa_profile_enable(0))
        n = ctypes.c_int(0)
        buf = (rpa_kernel_time * 64)()
        _check(lib.rpa_profile_read(buf, 64, ctypes.byref(n)))
        self.result = {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
                       for i in range(min(n.value, 64))}
        _check(lib.rpa_profile_reset())
        return False
