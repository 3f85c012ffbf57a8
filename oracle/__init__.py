"""Float64 CPU oracle for ragged paged attention, MLA and DSA sparse MLA.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package.  The GPU library never imports, links or calls it, and the two share
no code: the only thing both sides see is the seeded input generator
(``ragged_paged_attention_gb300.workloads``), which holds none of the
method's arithmetic.

The arithmetic lives in ``rpa_oracle.c`` (plain C, binary64, OpenMP over
output rows).  This module compiles it with gcc on first use and marshals
torch CPU tensors into it.  Passages followed, per function:

* :func:`rpa` -- tpu-inference ``ragged_paged_attention/v2/kernel.py``,
  ``ref_ragged_paged_attention`` (GQA repeat, sm_scale, soft cap, additive
  mask, optional fp8 k/v scale rounded to the query dtype).
* :func:`rpa_update_kv_cache` -- not on the pages (the v2 wrapper only has a
  TODO for a cache-write kernel); defined by analogy with MLA ``update_kv_cache``.
* :func:`mla_update_kv_cache`, :func:`mla` -- tpu-inference ``mla/v1/kernel.py``,
  ``update_kv_cache`` and ``ref_mla_ragged_paged_attention`` (masked logits
  replaced by ``mask_value``).
* :func:`sparse_mla` -- sglang-jax ``dsa/sparse_mla_prefill.py``,
  ``_sparse_mla_kernel_chunked_hminor`` validity rule and -inf-safe softmax,
  with units expanded as in ``units_to_token_ids``.

Parity pins: every function here is checked by ``tests/test_oracle_pins.py``
against brute force, closed forms and invariants (none is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rpa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 1
E4M3 = 2
INT8 = 3
INT4 = 4  # packed two to a byte: a uint8 cache tensor [P, ps, C, D / 2]
DEFAULT_MASK_VALUE = -0.7 * 3.4028234663852886e38  # -0.7 * float32 max


class RpaParams(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_combined_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("total_num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_num_seqs", ctypes.c_int32),
        ("pages_per_seq", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("sm_scale", ctypes.c_double),
        ("sliding_window", ctypes.c_int32),
        ("soft_cap", ctypes.c_double),
        ("mask_value", ctypes.c_double),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
    ]


class MlaParams(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("lkv_dim", ctypes.c_int32),
        ("lkv_dim_pad", ctypes.c_int32),
        ("r_dim", ctypes.c_int32),
        ("r_dim_pad", ctypes.c_int32),
        ("total_num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_num_seqs", ctypes.c_int32),
        ("pages_per_seq", ctypes.c_int32),
        ("sm_scale", ctypes.c_double),
        ("sliding_window", ctypes.c_int32),
        ("soft_cap", ctypes.c_double),
        ("mask_value", ctypes.c_double),
        ("q_dtype", ctypes.c_int32),
        ("q_scale", ctypes.c_double),
    ]


class SparseParams(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_queries", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32),
        ("row_stride", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("read_block", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("total_num_pages", ctypes.c_int32),
        ("seq_len", ctypes.c_int32),
        ("sm_scale", ctypes.c_double),
    ]


class RaggedParams(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("dv", ctypes.c_int32),
        ("rope", ctypes.c_int32),
        ("row_stride", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("read_block", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_page_ids", ctypes.c_int32),
        ("total_num_pages", ctypes.c_int32),
        ("sm_scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile ``rpa_oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        lib.oracle_rpa.argtypes = [ctypes.POINTER(RpaParams), P, P, P, P, P, i32, P, i32, P, ctypes.c_int]
        lib.oracle_rpa_update_kv_cache.argtypes = [ctypes.POINTER(RpaParams), P, P, P, P, P, P, i32]
        lib.oracle_mla_update_kv_cache.argtypes = [ctypes.POINTER(MlaParams), P, P, P, P, P, P, P, i32]
        lib.oracle_mla.argtypes = [ctypes.POINTER(MlaParams), P, P, P, P, P, P, P, i32, P, i32, P,
                                   ctypes.c_int]
        lib.oracle_sparse_mla.argtypes = [ctypes.POINTER(SparseParams), P, P, P, P, P, P, i32, P,
                                          ctypes.c_int]
        lib.oracle_sparse_ragged_write.argtypes = [ctypes.POINTER(RaggedParams), P, P, P, P]
        lib.oracle_sparse_mla_ragged.argtypes = [ctypes.POINTER(RaggedParams), P, P, P, P, P, P, P, P, P, P, i32,
                                                 P, ctypes.c_int]
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e4m3.restype = ctypes.c_double
        lib.oracle_decode_int8.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_int8.restype = ctypes.c_double
        lib.oracle_decode_int4.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_int4.restype = ctypes.c_double
        lib.oracle_round_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_round_f32_to_bf16.restype = ctypes.c_double
        for f in ("oracle_rpa", "oracle_rpa_update_kv_cache", "oracle_mla_update_kv_cache",
                  "oracle_mla", "oracle_sparse_mla", "oracle_sparse_ragged_write", "oracle_sparse_mla_ragged"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    assert t.device.type == "cpu", "oracle inputs live on the host"
    assert t.is_contiguous(), "oracle inputs must be contiguous"
    return ctypes.c_void_p(t.data_ptr())


def _i32(t) -> torch.Tensor:
    return torch.as_tensor(t, dtype=torch.int32).contiguous()


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc}")


def _kv_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return BF16
    if dtype == torch.float8_e4m3fn:
        return E4M3
    if dtype == torch.int8:
        return INT8
    if dtype == torch.uint8:  # int4 values, two per byte (element 2i in the low nibble of byte i)
        return INT4
    raise ValueError(f"unsupported kv dtype {dtype}")


def _nthreads(n):
    return 0 if n is None else int(n)


def rpa_params(q, kv_pages, page_indices, *, sm_scale=1.0, sliding_window=None, soft_cap=None,
               mask_value=None, k_scale=None, v_scale=None) -> RpaParams:
    P, ps, C, D = kv_pages.shape
    if kv_pages.dtype == torch.uint8:  # int4: two values per byte along the head dimension
        D *= 2
    max_num_seqs, pps = page_indices.shape
    return RpaParams(
        num_q_heads=q.shape[1], num_combined_kv_heads=C, head_dim=D, total_num_pages=P,
        page_size=ps, max_num_seqs=max_num_seqs, pages_per_seq=pps,
        kv_dtype=_kv_code(kv_pages.dtype), sm_scale=float(sm_scale),
        sliding_window=int(sliding_window or 0), soft_cap=float(soft_cap or 0.0),
        mask_value=DEFAULT_MASK_VALUE if mask_value is None else float(mask_value),
        k_scale=float(k_scale or 0.0), v_scale=float(v_scale or 0.0))


def rpa(q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, *, tokens=None, nthreads=None,
        **kw) -> torch.Tensor:
    """Ragged paged attention; returns float64 ``[max_tokens, Hq, D]``.

    Rows of tokens that were not computed (padding, or not in ``tokens``) are NaN.
    """
    lib = _load()
    q = q.contiguous()
    assert q.dtype == torch.bfloat16
    kv_pages = kv_pages.contiguous()
    page_indices = _i32(page_indices)
    prm = rpa_params(q, kv_pages, page_indices, **kw)
    out = torch.full(q.shape, math.nan, dtype=torch.float64)
    kv_lens, cu_q_lens = _i32(kv_lens), _i32(cu_q_lens)
    tok = None if tokens is None else _i32(tokens)
    rc = lib.oracle_rpa(ctypes.byref(prm), _ptr(q), _ptr(kv_pages), _ptr(kv_lens), _ptr(page_indices),
                        _ptr(cu_q_lens), int(num_seqs), _ptr(tok), 0 if tok is None else tok.numel(),
                        _ptr(out), _nthreads(nthreads))
    _check(rc, "oracle_rpa")
    return out


def rpa_update_kv_cache(new_k, new_v, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs):
    """Scatter new K/V ``[T, Hkv, D]`` into a copy of ``kv_pages``; returns the copy."""
    lib = _load()
    pages = kv_pages.clone().contiguous()
    page_indices = _i32(page_indices)
    prm = rpa_params(torch.empty(1, 1), pages, page_indices)
    new_k, new_v = new_k.contiguous(), new_v.contiguous()
    assert new_k.dtype == pages.dtype and new_v.dtype == pages.dtype
    kv_lens, cu_q_lens = _i32(kv_lens), _i32(cu_q_lens)
    rc = lib.oracle_rpa_update_kv_cache(ctypes.byref(prm), _ptr(new_k), _ptr(new_v), _ptr(pages),
                                        _ptr(kv_lens), _ptr(page_indices), _ptr(cu_q_lens), int(num_seqs))
    _check(rc, "oracle_rpa_update_kv_cache")
    return pages


def mla_params(ql_nope, q_pe, cache_kv_c, cache_k_pe, page_indices, max_num_seqs, *, sm_scale=1.0,
               sliding_window=None, soft_cap=None, mask_value=None, q_scale=None) -> MlaParams:
    P = cache_kv_c.shape[0]
    ps = cache_kv_c.shape[1] * cache_kv_c.shape[2]
    return MlaParams(
        num_q_heads=ql_nope.shape[1], lkv_dim=ql_nope.shape[2], lkv_dim_pad=cache_kv_c.shape[-1],
        r_dim=q_pe.shape[2], r_dim_pad=cache_k_pe.shape[-1], total_num_pages=P, page_size=ps,
        max_num_seqs=max_num_seqs, pages_per_seq=page_indices.numel() // max_num_seqs,
        sm_scale=float(sm_scale), sliding_window=int(sliding_window or 0),
        soft_cap=float(soft_cap or 0.0),
        mask_value=DEFAULT_MASK_VALUE if mask_value is None else float(mask_value),
        q_dtype=E4M3 if ql_nope.dtype == torch.float8_e4m3fn else BF16, q_scale=float(q_scale or 0.0))


def mla_update_kv_cache(new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, cu_q_lens,
                        distribution):
    """MLA cache scatter on copies of the caches; returns ``(cache_kv_c, cache_k_pe)``."""
    lib = _load()
    ckv, ckpe = cache_kv_c.clone().contiguous(), cache_k_pe.clone().contiguous()
    kv_lens, cu_q_lens, page_indices = _i32(kv_lens), _i32(cu_q_lens), _i32(page_indices).reshape(-1)
    qn = torch.empty(1, 1, new_kv_c.shape[1])
    qr = torch.empty(1, 1, new_k_pe.shape[1])
    prm = mla_params(qn, qr, ckv, ckpe, page_indices, kv_lens.numel())
    num_seqs = int(_i32(distribution)[2])
    rc = lib.oracle_mla_update_kv_cache(ctypes.byref(prm), _ptr(new_kv_c.contiguous()),
                                        _ptr(new_k_pe.contiguous()), _ptr(ckv), _ptr(ckpe), _ptr(kv_lens),
                                        _ptr(page_indices), _ptr(cu_q_lens), num_seqs)
    _check(rc, "oracle_mla_update_kv_cache")
    return ckv, ckpe


def mla(ql_nope, q_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, cu_q_lens, distribution, *,
        tokens=None, nthreads=None, **kw) -> torch.Tensor:
    """MLA attention over already-updated caches; returns float64 ``[T, H, lkv]``."""
    lib = _load()
    kv_lens, cu_q_lens, page_indices = _i32(kv_lens), _i32(cu_q_lens), _i32(page_indices).reshape(-1)
    ql_nope, q_pe = ql_nope.contiguous(), q_pe.contiguous()
    prm = mla_params(ql_nope, q_pe, cache_kv_c, cache_k_pe, page_indices, kv_lens.numel(), **kw)
    num_seqs = int(_i32(distribution)[2])
    out = torch.full(ql_nope.shape, math.nan, dtype=torch.float64)
    tok = None if tokens is None else _i32(tokens)
    rc = lib.oracle_mla(ctypes.byref(prm), _ptr(ql_nope), _ptr(q_pe), _ptr(cache_kv_c.contiguous()),
                        _ptr(cache_k_pe.contiguous()), _ptr(kv_lens), _ptr(page_indices), _ptr(cu_q_lens),
                        num_seqs, _ptr(tok), 0 if tok is None else tok.numel(), _ptr(out),
                        _nthreads(nthreads))
    _check(rc, "oracle_mla")
    return out


def mla_forward(ql_nope, q_pe, new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices,
                cu_q_lens, distribution, **kw):
    """update_kv_cache followed by attention, as the MLA reference does."""
    ckv, ckpe = mla_update_kv_cache(new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices,
                                    cu_q_lens, distribution)
    return mla(ql_nope, q_pe, ckv, ckpe, kv_lens, page_indices, cu_q_lens, distribution, **kw), ckv, ckpe


def sparse_mla(q, cache, indices, positions, page_table, *, read_block, page_size, seq_len, sm_scale,
               dv=512, queries=None, nthreads=None) -> torch.Tensor:
    """DSA sparse MLA; returns float64 ``[B, S, H, dv]``.

    ``cache`` is the paged latent cache in any shape whose row-major bytes are
    ``[P * page_size, row_stride]``; ``queries`` lists flat ``b * S + s`` ids.
    """
    lib = _load()
    B, S, H, Dk = q.shape
    K = indices.shape[-1]
    row_stride = cache.shape[-1]
    P = cache.numel() // (page_size * row_stride)
    prm = SparseParams(batch=B, num_queries=S, num_heads=H, dk=Dk, dv=dv, row_stride=row_stride, topk=K,
                       read_block=read_block, page_size=page_size, max_pages=page_table.shape[-1],
                       total_num_pages=P, seq_len=seq_len, sm_scale=float(sm_scale))
    out = torch.full((B, S, H, dv), math.nan, dtype=torch.float64)
    qs = None if queries is None else _i32(queries)
    rc = lib.oracle_sparse_mla(ctypes.byref(prm), _ptr(q.contiguous()), _ptr(cache.contiguous()),
                               _ptr(_i32(indices)), _ptr(_i32(positions)), _ptr(_i32(page_table)), _ptr(qs),
                               0 if qs is None else qs.numel(), _ptr(out), _nthreads(nthreads))
    _check(rc, "oracle_sparse_mla")
    return out


def _ragged_params(ql, qpe, cache, topk, seq_lens, page_indices, *, read_block, page_size, sm_scale):
    T, H, dv = ql.shape
    row_stride = cache.shape[-1]
    return RaggedParams(num_tokens=T, num_seqs=seq_lens.numel(), num_heads=H, dv=dv, rope=qpe.shape[-1],
                        row_stride=row_stride, topk=topk.shape[-1], read_block=read_block, page_size=page_size,
                        num_page_ids=page_indices.numel(),
                        total_num_pages=cache.numel() // (page_size * row_stride), sm_scale=float(sm_scale))


def sparse_ragged_write(kvc, kpe, cache, loc, *, page_size) -> torch.Tensor:
    """The packed-ragged self-write; returns a written copy of ``cache`` (any shape whose
    row-major bytes are ``[P * page_size, row_stride]``)."""
    lib = _load()
    T, dv = kvc.shape
    row_stride = cache.shape[-1]
    prm = RaggedParams(num_tokens=T, num_seqs=1, num_heads=1, dv=dv, rope=kpe.shape[-1], row_stride=row_stride,
                       topk=1, read_block=1, page_size=page_size, num_page_ids=1,
                       total_num_pages=cache.numel() // (page_size * row_stride), sm_scale=1.0)
    out = cache.contiguous().clone()
    _check(lib.oracle_sparse_ragged_write(ctypes.byref(prm), _ptr(kvc.contiguous()), _ptr(kpe.contiguous()),
                                          _ptr(out), _ptr(_i32(loc))), "oracle_sparse_ragged_write")
    return out


def sparse_mla_ragged(ql, qpe, cache, topk, positions, seq_lens, cu_q_lens, cu_kv_lens, page_indices, *,
                      read_block, page_size, sm_scale, queries=None, nthreads=None) -> torch.Tensor:
    """DSA sparse MLA in the packed-ragged mode over an already written cache; returns
    float64 ``[T, H, dv]`` (rows of unlisted tokens are NaN)."""
    lib = _load()
    prm = _ragged_params(ql, qpe, cache, topk, seq_lens, page_indices, read_block=read_block, page_size=page_size,
                         sm_scale=sm_scale)
    T, H, dv = ql.shape
    out = torch.full((T, H, dv), math.nan, dtype=torch.float64)
    qs = None if queries is None else _i32(queries)
    rc = lib.oracle_sparse_mla_ragged(ctypes.byref(prm), _ptr(ql.contiguous()), _ptr(qpe.contiguous()),
                                      _ptr(cache.contiguous()), _ptr(_i32(topk)), _ptr(_i32(positions)),
                                      _ptr(_i32(seq_lens)), _ptr(_i32(cu_q_lens)), _ptr(_i32(cu_kv_lens)),
                                      _ptr(_i32(page_indices)), _ptr(qs), 0 if qs is None else qs.numel(), _ptr(out),
                                      _nthreads(nthreads))
    _check(rc, "oracle_sparse_mla_ragged")
    return out


def decode_bf16(bits: int) -> float:
    return _load().oracle_decode_bf16(bits)


def decode_e4m3(bits: int) -> float:
    return _load().oracle_decode_e4m3(bits)


def decode_int8(bits: int) -> float:
    return _load().oracle_decode_int8(bits)


def decode_int4(nibble: int) -> float:
    return _load().oracle_decode_int4(nibble)


def round_f32_to_bf16(x: float) -> float:
    return _load().oracle_round_f32_to_bf16(x)
