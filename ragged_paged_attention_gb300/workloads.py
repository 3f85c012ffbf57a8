"""Seeded synthetic inputs for ragged paged attention, MLA and DSA sparse MLA.

This module is the only code that both the GPU library's tests/benchmark and
the float64 oracle see.  It draws random numbers and lays them out in the
paged formats; it holds none of the attention arithmetic.

Recipe (the shapes follow the workloads the source pages describe):

* values are N(0, 1) drawn in float32 from numpy PCG64 and rounded to the
  storage dtype (bf16, or fp8 e4m3 for quantised KV caches);
* metadata uses the same generator: ``seed = 1000 + config index``;
* decode sequences come first, prefill chunks after; a chunk's queries are the
  last ``q_len`` positions of its ``kv_len``;
* physical pages are one random permutation of ``range(total_num_pages)``;
* every byte the kernels must not read is poisoned: page slots past
  ``kv_len`` and unused pages hold NaN, unused page-table entries hold
  ``INT32_MAX``, padded query rows hold NaN, metadata of sequences past
  ``num_seqs`` is garbage.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np
import torch

POISON_PAGE = 2**31 - 1
BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F


_CHUNK = 1 << 22  # values per independently seeded block (fixed: results do not depend on threads)


def _randn(rng: np.random.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    """N(0, 1) float32 values rounded to ``dtype``.  Large draws are split into fixed
    blocks, each from its own PCG64 stream spawned from one seed taken from ``rng``,
    and filled by a thread pool."""
    if dtype == torch.int8:  # integer caches: uniform over the whole byte
        return torch.from_numpy(rng.integers(-128, 128, size=tuple(shape)).astype(np.int8))
    if dtype == torch.uint8:  # int4 caches: two uniform nibbles per byte (the last dim is halved)
        shape = tuple(shape[:-1]) + (shape[-1] // 2,)
        return torch.from_numpy(rng.integers(0, 256, size=shape).astype(np.uint8))
    n = int(np.prod(shape))
    if n <= _CHUNK:
        x = rng.standard_normal(size=n, dtype=np.float32)
    else:
        x = np.empty(n, dtype=np.float32)
        blocks = (n + _CHUNK - 1) // _CHUNK
        seeds = np.random.SeedSequence(int(rng.integers(0, 2**63))).spawn(blocks)

        def fill(i):
            g = np.random.Generator(np.random.PCG64(seeds[i]))
            g.standard_normal(out=x[i * _CHUNK:(i + 1) * _CHUNK], dtype=np.float32)

        with concurrent.futures.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(blocks)))
    return torch.from_numpy(x).reshape(shape).to(dtype)


def _fill_nan(t: torch.Tensor) -> None:
    if t.numel() == 0:
        return
    if t.dtype == torch.bfloat16:
        t.view(torch.int16).fill_(BF16_NAN)
    elif t.dtype == torch.float8_e4m3fn:
        t.view(torch.uint8).fill_(E4M3_NAN)
    elif t.dtype == torch.int8:  # no NaN: the extreme value, which would show in any output
        t.fill_(127)
    elif t.dtype == torch.uint8:  # int4 pairs: the largest value in both nibbles
        t.fill_(0x77)
    else:
        t.fill_(float("nan"))


def _assign_pages(rng, kv_lens, page_size, pages_per_seq, max_num_seqs, extra_pages):
    """Random physical pages for each sequence; unused entries are poisoned."""
    need = [math.ceil(k / page_size) for k in kv_lens]
    total = sum(need) + extra_pages
    perm = rng.permutation(max(total, 1)).astype(np.int32)
    table = np.full((max_num_seqs, pages_per_seq), POISON_PAGE, dtype=np.int32)
    off = 0
    for s, n in enumerate(need):
        table[s, :n] = perm[off:off + n]
        off += n
    return table, max(total, 1), need


@dataclasses.dataclass
class RpaInputs:
    """One ragged batch for ``rpa_forward`` / ``rpa_update_kv_cache``."""
    q: torch.Tensor             # [max_num_tokens, Hq, D] bf16
    kv_pages: torch.Tensor      # [P, ps, 2*Hkv, D] bf16 or fp8 e4m3
    kv_lens: torch.Tensor       # [max_num_seqs] int32
    page_indices: torch.Tensor  # [max_num_seqs, pages_per_seq] int32
    cu_q_lens: torch.Tensor     # [max_num_seqs + 1] int32
    num_seqs: torch.Tensor      # [1] int32
    new_k: torch.Tensor         # [max_num_tokens, Hkv, D] cache dtype
    new_v: torch.Tensor         # [max_num_tokens, Hkv, D] cache dtype
    q_lens: list
    kv_lens_list: list
    sm_scale: float
    sliding_window: int | None = None
    soft_cap: float | None = None
    k_scale: float | None = None
    v_scale: float | None = None
    mask_value: float | None = None

    @property
    def num_tokens(self) -> int:
        return int(sum(self.q_lens))

    def options(self) -> dict:
        return dict(sm_scale=self.sm_scale, sliding_window=self.sliding_window, soft_cap=self.soft_cap,
                    k_scale=self.k_scale, v_scale=self.v_scale, mask_value=self.mask_value)

    def tensors(self) -> dict:
        return {f.name: getattr(self, f.name) for f in dataclasses.fields(self)
                if isinstance(getattr(self, f.name), torch.Tensor)}

    def to(self, device) -> "RpaInputs":
        kw = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
              for k, v in dataclasses.asdict(self).items()}
        return RpaInputs(**kw)


def make_rpa(q_lens, kv_lens, *, num_q_heads, num_kv_heads, head_dim, page_size, seed,
             kv_dtype=torch.bfloat16, pages_per_seq=None, max_num_seqs=None, max_num_tokens=None,
             extra_pages=0, sm_scale=None, sliding_window=None, soft_cap=None, k_scale=None,
             v_scale=None, mask_value=None, poison=True) -> RpaInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    q_lens, kv_lens = [int(x) for x in q_lens], [int(x) for x in kv_lens]
    num_seqs = len(q_lens)
    assert num_seqs == len(kv_lens)
    max_num_seqs = max_num_seqs or max(num_seqs, 1)
    T = sum(q_lens)
    max_num_tokens = max_num_tokens or max(T, 1)
    pps = pages_per_seq or max(1, max((math.ceil(k / page_size) for k in kv_lens), default=1))
    table, P, need = _assign_pages(rng, kv_lens, page_size, pps, max_num_seqs, extra_pages)
    C = 2 * num_kv_heads
    q = _randn(rng, (max_num_tokens, num_q_heads, head_dim), torch.bfloat16)
    kv = _randn(rng, (P, page_size, C, head_dim), kv_dtype)
    new_k = _randn(rng, (max_num_tokens, num_kv_heads, head_dim), kv_dtype)
    new_v = _randn(rng, (max_num_tokens, num_kv_heads, head_dim), kv_dtype)
    if poison:
        _fill_nan(q[T:])
        used = set()
        for s in range(num_seqs):
            pages = table[s, :need[s]]
            used.update(int(p) for p in pages)
            if need[s] and kv_lens[s] % page_size:
                _fill_nan(kv[int(pages[-1]), kv_lens[s] % page_size:])
        for p in range(P):
            if p not in used:
                _fill_nan(kv[p])
    kvl = np.full(max_num_seqs, 10**9 if poison else 0, dtype=np.int32)
    kvl[:num_seqs] = kv_lens
    cu = np.full(max_num_seqs + 1, -5 if poison else T, dtype=np.int32)
    cu[:num_seqs + 1] = np.concatenate([[0], np.cumsum(q_lens, dtype=np.int64)]).astype(np.int32)
    return RpaInputs(
        q=q, kv_pages=kv, kv_lens=torch.from_numpy(kvl), page_indices=torch.from_numpy(table),
        cu_q_lens=torch.from_numpy(cu), num_seqs=torch.tensor([num_seqs], dtype=torch.int32),
        new_k=new_k, new_v=new_v, q_lens=q_lens, kv_lens_list=kv_lens,
        sm_scale=(1.0 / math.sqrt(head_dim)) if sm_scale is None else float(sm_scale),
        sliding_window=sliding_window, soft_cap=soft_cap, k_scale=k_scale, v_scale=v_scale,
        mask_value=mask_value)


@dataclasses.dataclass
class MlaInputs:
    """One ragged batch for ``mla_rpa_forward``."""
    ql_nope: torch.Tensor       # [max_num_tokens, H, lkv] bf16
    q_pe: torch.Tensor          # [max_num_tokens, H, r] bf16
    new_kv_c: torch.Tensor      # [max_num_tokens, lkv] bf16
    new_k_pe: torch.Tensor      # [max_num_tokens, r] bf16
    cache_kv_c: torch.Tensor    # [P, ps/pk, pk, lkv_pad] bf16
    cache_k_pe: torch.Tensor    # [P, ps/pk, pk, r_pad] bf16
    kv_lens: torch.Tensor       # [max_num_seqs] int32
    page_indices: torch.Tensor  # [max_num_seqs * pages_per_seq] int32
    cu_q_lens: torch.Tensor     # [max_num_seqs + 1] int32
    distribution: torch.Tensor  # [3] int32
    q_lens: list
    kv_lens_list: list
    sm_scale: float
    sliding_window: int | None = None
    soft_cap: float | None = None
    mask_value: float | None = None
    q_scale: float | None = None

    @property
    def num_tokens(self) -> int:
        return int(sum(self.q_lens))

    def options(self) -> dict:
        opts = dict(sm_scale=self.sm_scale, sliding_window=self.sliding_window, soft_cap=self.soft_cap,
                    mask_value=self.mask_value)
        if self.q_scale is not None:
            opts["q_scale"] = self.q_scale
        return opts

    def to(self, device) -> "MlaInputs":
        kw = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
              for k, v in dataclasses.asdict(self).items()}
        return MlaInputs(**kw)


def make_mla(q_lens, kv_lens, *, num_q_heads=128, lkv_dim=512, r_dim=64, page_size=64, kv_packing=2,
             seed, num_decode=None, pages_per_seq=None, max_num_seqs=None, max_num_tokens=None,
             extra_pages=0, sm_scale=None, sliding_window=None, soft_cap=None, mask_value=None,
             q_dtype=torch.bfloat16, q_scale=None, poison=True) -> MlaInputs:
    """``q_dtype=torch.float8_e4m3fn`` draws the queries as N(0, 1) / q_scale (default 1/8)
    rounded to e4m3: the per-tensor quantised queries whose scores carry q_scale."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q_lens, kv_lens = [int(x) for x in q_lens], [int(x) for x in kv_lens]
    num_seqs = len(q_lens)
    max_num_seqs = max_num_seqs or max(num_seqs, 1)
    T = sum(q_lens)
    max_num_tokens = max_num_tokens or max(T, 1)
    pps = pages_per_seq or max(1, max((math.ceil(k / page_size) for k in kv_lens), default=1))
    table, P, need = _assign_pages(rng, kv_lens, page_size, pps, max_num_seqs, extra_pages)
    lkv_pad = -(-lkv_dim // 128) * 128
    r_pad = -(-r_dim // 128) * 128
    ql = _randn(rng, (max_num_tokens, num_q_heads, lkv_dim), torch.bfloat16)
    qpe = _randn(rng, (max_num_tokens, num_q_heads, r_dim), torch.bfloat16)
    nkv = _randn(rng, (max_num_tokens, lkv_dim), torch.bfloat16)
    nkpe = _randn(rng, (max_num_tokens, r_dim), torch.bfloat16)
    ckv = torch.zeros((P, page_size, lkv_pad), dtype=torch.bfloat16)
    ckv[..., :lkv_dim] = _randn(rng, (P, page_size, lkv_dim), torch.bfloat16)
    ckpe = torch.zeros((P, page_size, r_pad), dtype=torch.bfloat16)
    ckpe[..., :r_dim] = _randn(rng, (P, page_size, r_dim), torch.bfloat16)
    if q_dtype == torch.float8_e4m3fn:
        q_scale = 0.125 if q_scale is None else float(q_scale)
        ql = (ql.float() / q_scale).to(q_dtype)
        qpe = (qpe.float() / q_scale).to(q_dtype)
    elif q_dtype != torch.bfloat16 or q_scale is not None:
        raise ValueError("MLA queries are bf16, or float8_e4m3fn with a q_scale")
    if poison:
        _fill_nan(ql[T:])
        _fill_nan(qpe[T:])
        _fill_nan(nkv[T:])
        _fill_nan(nkpe[T:])
        used = set()
        for s in range(num_seqs):
            pages = table[s, :need[s]]
            used.update(int(p) for p in pages)
            # the slots the update will write, and the tail past kv_len
            for pos in range(kv_lens[s] - q_lens[s], need[s] * page_size):
                pg, sl = int(pages[pos // page_size]), pos % page_size
                _fill_nan(ckv[pg, sl])
                _fill_nan(ckpe[pg, sl])
        for p in range(P):
            if p not in used:
                _fill_nan(ckv[p])
                _fill_nan(ckpe[p])
    kvl = np.full(max_num_seqs, 10**9 if poison else 0, dtype=np.int32)
    kvl[:num_seqs] = kv_lens
    cu = np.full(max_num_seqs + 1, -5 if poison else T, dtype=np.int32)
    cu[:num_seqs + 1] = np.concatenate([[0], np.cumsum(q_lens, dtype=np.int64)]).astype(np.int32)
    if num_decode is None:
        num_decode = sum(1 for x in q_lens if x == 1)
    dist = torch.tensor([num_decode, num_seqs, num_seqs], dtype=torch.int32)
    return MlaInputs(
        ql_nope=ql, q_pe=qpe, new_kv_c=nkv, new_k_pe=nkpe,
        cache_kv_c=ckv.reshape(P, page_size // kv_packing, kv_packing, lkv_pad),
        cache_k_pe=ckpe.reshape(P, page_size // kv_packing, kv_packing, r_pad),
        kv_lens=torch.from_numpy(kvl), page_indices=torch.from_numpy(table.reshape(-1).copy()),
        cu_q_lens=torch.from_numpy(cu), distribution=dist, q_lens=q_lens, kv_lens_list=kv_lens,
        sm_scale=(1.0 / math.sqrt(192.0)) if sm_scale is None else float(sm_scale),
        sliding_window=sliding_window, soft_cap=soft_cap, mask_value=mask_value, q_scale=q_scale)


@dataclasses.dataclass
class SparseInputs:
    """One batch for ``sparse_mla_forward`` (paged latent cache, per-batch table)."""
    q: torch.Tensor           # [B, S, H, 576] bf16
    cache: torch.Tensor       # [P, ps/2, 2, 640] bf16 (cols 576.. are zero pad)
    indices: torch.Tensor     # [B, S, K] int32 unit ids, -1 padded
    positions: torch.Tensor   # [B, S] int32
    page_table: torch.Tensor  # [B, max_pages] int32
    read_block: int
    page_size: int
    seq_len: int
    sm_scale: float
    dv: int = 512

    def options(self) -> dict:
        return dict(read_block=self.read_block, page_size=self.page_size, seq_len=self.seq_len,
                    sm_scale=self.sm_scale, dv=self.dv)

    def to(self, device) -> "SparseInputs":
        kw = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
              for k, v in dataclasses.asdict(self).items()}
        return SparseInputs(**kw)


def sorted_causal_subsets(rng, positions: np.ndarray, topk: int, read_block: int) -> np.ndarray:
    """For each query: ``topk`` distinct unit ids drawn uniformly from the units
    whose first token is at or before the query position, sorted ascending and
    padded with -1 when fewer exist."""
    flat = positions.reshape(-1)
    n_units = flat // read_block + 1
    umax = int(n_units.max())
    out = np.full((flat.size, topk), -1, dtype=np.int32)
    chunk = max(1, (1 << 24) // max(umax, 1))
    for a in range(0, flat.size, chunk):
        b = min(flat.size, a + chunk)
        keys = rng.random((b - a, umax), dtype=np.float32)
        keys[np.arange(umax)[None, :] >= n_units[a:b, None]] = np.inf
        k = min(topk, umax)
        pick = np.argpartition(keys, k - 1, axis=1)[:, :k] if k < umax else np.argsort(keys, axis=1)[:, :k]
        valid = np.take_along_axis(keys, pick, axis=1) < np.inf
        pick = np.where(valid, pick, np.iinfo(np.int32).max)
        pick.sort(axis=1)
        pick = np.where(pick == np.iinfo(np.int32).max, -1, pick)
        out[a:b, :k] = pick
    return out.reshape(positions.shape + (topk,))


def make_sparse(*, batch, num_queries, seq_len, positions, topk, read_block, seed, num_heads=128,
                dk=576, dv=512, page_size=64, kv_packing=2, row_stride=640, sm_scale=None,
                indices=None, extra_pages=0) -> SparseInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    max_pages = -(-seq_len // page_size)
    P = batch * max_pages + extra_pages
    perm = rng.permutation(P).astype(np.int32)
    table = perm[:batch * max_pages].reshape(batch, max_pages).copy()
    q = _randn(rng, (batch, num_queries, num_heads, dk), torch.bfloat16)
    cache = torch.zeros((P, page_size, row_stride), dtype=torch.bfloat16)
    cache[..., :dk] = _randn(rng, (P, page_size, dk), torch.bfloat16)
    # slots past seq_len in each sequence's last page, and spare pages: NaN
    for b in range(batch):
        if seq_len % page_size:
            _fill_nan(cache[int(table[b, -1]), seq_len % page_size:])
    for p in perm[batch * max_pages:]:
        _fill_nan(cache[int(p)])
    pos = np.asarray(positions, dtype=np.int32).reshape(batch, num_queries)
    if indices is None:
        indices = sorted_causal_subsets(rng, pos, topk, read_block)
    return SparseInputs(
        q=q, cache=cache.reshape(P, page_size // kv_packing, kv_packing, row_stride),
        indices=torch.from_numpy(np.ascontiguousarray(indices, dtype=np.int32)),
        positions=torch.from_numpy(pos.copy()), page_table=torch.from_numpy(table),
        read_block=read_block, page_size=page_size, seq_len=seq_len,
        sm_scale=(1.0 / math.sqrt(192.0)) if sm_scale is None else float(sm_scale), dv=dv)


@dataclasses.dataclass
class SparseRaggedInputs:
    """One packed-ragged batch for ``sparse_mla_write_and_attend_ragged``."""
    ql: torch.Tensor           # [T, H, 512] bf16
    qpe: torch.Tensor          # [T, H, 64] bf16
    kvc: torch.Tensor          # [T, 512] bf16 new latent rows
    kpe: torch.Tensor          # [T, 64] bf16
    cache: torch.Tensor        # [P, ps/2, 2, 640] bf16 (cols 576.. zero; rows to be written: NaN)
    topk: torch.Tensor         # [T, K] int32 request-local unit ids, -1 padded
    positions: torch.Tensor    # [T] int32
    loc: torch.Tensor          # [T] int32 flat cache row of each token's new row (-1: padding)
    seq_lens: torch.Tensor     # [S] int32
    cu_q_lens: torch.Tensor    # [S + 1] int32
    cu_kv_lens: torch.Tensor   # [S + 1] int32 page-aligned
    page_indices: torch.Tensor  # [sum of pages] int32
    read_block: int
    page_size: int
    sm_scale: float
    q_lens: list

    def options(self) -> dict:
        return dict(read_block=self.read_block, page_size=self.page_size, sm_scale=self.sm_scale)

    def to(self, device) -> "SparseRaggedInputs":
        kw = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in dataclasses.asdict(self).items()}
        return SparseRaggedInputs(**kw)


def make_sparse_ragged(q_lens, seq_lens, *, topk, read_block, seed, num_heads=128, dv=512, rope=64, page_size=64,
                       kv_packing=2, row_stride=640, extra_pages=0, pad_tokens=0, sm_scale=None) -> SparseRaggedInputs:
    """Requests extending their sequences: request r's q_lens[r] new tokens sit at the end of its
    seq_lens[r] keys; its pages are a random run of the packed page list starting at
    cu_kv_lens[r] / page_size; each token writes its new row to the slot of its own position
    (those rows hold NaN until written) and selects ``topk`` units drawn causally within its
    request. ``pad_tokens`` padding tokens follow with loc = -1."""
    rng = np.random.Generator(np.random.PCG64(seed))
    S = len(q_lens)
    pages = [-(-int(L) // page_size) for L in seq_lens]
    cu_kv = np.concatenate([[0], np.cumsum([n * page_size for n in pages])]).astype(np.int32)
    n_ids = int(sum(pages))
    P = n_ids + extra_pages
    perm = rng.permutation(P).astype(np.int32)
    page_ids = perm[:n_ids].copy()
    cache = torch.zeros((P, page_size, row_stride), dtype=torch.bfloat16)
    cache[..., :dv + rope] = _randn(rng, (P, page_size, dv + rope), torch.bfloat16)
    for p in perm[n_ids:]:
        _fill_nan(cache[int(p)])
    flat = cache.view(P * page_size, row_stride)
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(cu_q[-1]) + pad_tokens
    positions = np.zeros(T, np.int32)
    loc = np.full(T, -1, np.int32)
    for r in range(S):
        L, base = int(seq_lens[r]), int(cu_kv[r]) // page_size
        if L % page_size:  # slots past the request's keys in its last page
            _fill_nan(cache[int(page_ids[base + pages[r] - 1]), L % page_size:])
        for j, t in enumerate(range(cu_q[r], cu_q[r + 1])):
            pos = L - q_lens[r] + j
            positions[t] = pos
            loc[t] = int(page_ids[base + pos // page_size]) * page_size + pos % page_size
            _fill_nan(flat[int(loc[t])])
    topk_ids = np.full((T, topk), -1, np.int32)
    for r in range(S):
        toks = np.arange(cu_q[r], cu_q[r + 1])
        if len(toks):
            topk_ids[toks] = sorted_causal_subsets(rng, positions[toks], topk, read_block)
    for t in range(int(cu_q[-1]), T):
        positions[t] = int(seq_lens[-1]) - 1
        topk_ids[t, 0] = 0
    return SparseRaggedInputs(
        ql=_randn(rng, (T, num_heads, dv), torch.bfloat16), qpe=_randn(rng, (T, num_heads, rope), torch.bfloat16),
        kvc=_randn(rng, (T, dv), torch.bfloat16), kpe=_randn(rng, (T, rope), torch.bfloat16),
        cache=cache.reshape(P, page_size // kv_packing, kv_packing, row_stride),
        topk=torch.from_numpy(topk_ids), positions=torch.from_numpy(positions), loc=torch.from_numpy(loc),
        seq_lens=torch.tensor(list(seq_lens), dtype=torch.int32), cu_q_lens=torch.from_numpy(cu_q),
        cu_kv_lens=torch.from_numpy(cu_kv), page_indices=torch.from_numpy(page_ids), read_block=read_block,
        page_size=page_size, sm_scale=(1.0 / math.sqrt(192.0)) if sm_scale is None else float(sm_scale),
        q_lens=list(q_lens))


def dsa_sparse_ragged(*, mode="token", scale=1.0, seed=1005) -> SparseRaggedInputs:
    """DSA multi-request extend, packed: 4 requests of 256 new tokens each at the end of
    seq_lens U[2048, 8192]; token mode RB 1, K 2048; page mode RB 64, K 32."""
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    ql = max(1, int(256 * scale))
    seq = rng.integers(max(ql, int(2048 * scale)), max(ql, int(8192 * scale)) + 1, size=4)
    RB, K = (1, max(16, int(2048 * scale))) if mode == "token" else (64, max(2, int(32 * scale)))
    return make_sparse_ragged([ql] * 4, list(seq), topk=K, read_block=RB, seed=seed)


# ---------------------------------------------------------------------------
# The five named workloads.  ``scale`` < 1 shrinks lengths and counts for
# parity runs the oracle finishes in seconds; 1.0 is the benchmark size.
# ---------------------------------------------------------------------------

def tiny_rpa(seed=1000) -> RpaInputs:
    """4 q / 2 kv heads, D 128, ps 16, q_lens [1,1,5], kv_lens [17,40,64], 16 pages."""
    return make_rpa([1, 1, 5], [17, 40, 64], num_q_heads=4, num_kv_heads=2, head_dim=128, page_size=16,
                    seed=seed, pages_per_seq=4, extra_pages=16 - 9)


def llama_mixed(scale=1.0, seed=1001, num_decode=128, num_prefill=4) -> RpaInputs:
    """Llama-3-8B shape: 32 q / 8 kv heads, D 128, ps 16; decodes kv U[512,4096],
    prefill chunks q 512 with kv U[512,2048]."""
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    nd = max(1, int(round(num_decode * scale)))
    npf = max(1, int(round(num_prefill * min(1.0, scale * 4))))
    qp = max(8, int(512 * scale))
    dec = rng.integers(max(1, int(512 * scale)), int(4096 * scale) + 1, size=nd)
    pre = rng.integers(max(qp, int(512 * scale)), max(qp, int(2048 * scale)) + 1, size=npf)
    return make_rpa([1] * nd + [qp] * npf, list(dec) + list(pre), num_q_heads=32, num_kv_heads=8,
                    head_dim=128, page_size=16, seed=seed, pages_per_seq=max(1, int(4096 * scale) // 16 + 1))


def gemma_options(scale=1.0, seed=1002, num_decode=64, num_prefill=2) -> RpaInputs:
    """Gemma-2-style: 16 q / 8 kv heads, D 256, ps 32, fp8 e4m3 KV (scale 0.5),
    sliding window 4096, soft cap 50; decodes kv U[1024,8192], 2 prefill chunks
    of 1024."""
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    nd = max(1, int(round(num_decode * scale)))
    qp = max(8, int(1024 * scale))
    dec = rng.integers(max(1, int(1024 * scale)), int(8192 * scale) + 1, size=nd)
    pre = rng.integers(qp, max(qp, int(8192 * scale)) + 1, size=num_prefill)
    sw = max(1, int(4096 * scale))
    return make_rpa([1] * nd + [qp] * num_prefill, list(dec) + list(pre), num_q_heads=16, num_kv_heads=8,
                    head_dim=256, page_size=32, seed=seed, kv_dtype=torch.float8_e4m3fn,
                    pages_per_seq=max(1, int(8192 * scale) // 32 + 1), k_scale=0.5, v_scale=0.5,
                    sliding_window=sw, soft_cap=50.0)


def mla_deepseek(scale=1.0, seed=1003, num_decode=64, num_prefill=2) -> MlaInputs:
    """DeepSeek-V3 MLA: 128 heads, lkv 512, rope 64 (padded to 128), ps 64, pk 2;
    decodes kv U[1024,8192], 2 prefill chunks of q 256; sm_scale 1/sqrt(192)."""
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    nd = max(1, int(round(num_decode * scale)))
    qp = max(4, int(256 * scale))
    dec = rng.integers(max(1, int(1024 * scale)), int(8192 * scale) + 1, size=nd)
    pre = rng.integers(max(qp, int(1024 * scale)), max(qp, int(8192 * scale)) + 1, size=num_prefill)
    return make_mla([1] * nd + [qp] * num_prefill, list(dec) + list(pre), seed=seed, num_decode=nd,
                    pages_per_seq=max(1, int(8192 * scale) // 64 + 1))


def dsa_sparse(*, mode="token", phase="prefill", scale=1.0, seed=1004) -> SparseInputs:
    """DSA sparse MLA: 128 heads, Dk 576, Dv 512, paged latent ps 64, T 8192.

    mode "token": RB 1, K 2048; mode "page": RB 64, K 32.  phase "prefill":
    4 sequences x 1024 queries at positions T-1024..T-1; "decode": 64
    sequences x 1 query at T-1.
    """
    T = max(128, int(8192 * scale))
    if phase == "prefill":
        B, S = 4, max(1, int(1024 * scale))
        pos = np.tile(np.arange(T - S, T, dtype=np.int32), (B, 1))
    else:
        B, S = max(1, int(64 * scale)), 1
        pos = np.full((B, 1), T - 1, dtype=np.int32)
    if mode == "token":
        RB, K = 1, max(16, int(2048 * scale))
    else:
        RB, K = 64, max(2, int(32 * scale))
    return make_sparse(batch=B, num_queries=S, seq_len=T, positions=pos, topk=K, read_block=RB, seed=seed)
