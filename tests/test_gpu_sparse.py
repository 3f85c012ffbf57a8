"""GPU parity of sparse_mla_forward against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_gb300 import api, workloads
from parity import TOL_BF16, max_abs

pytestmark = pytest.mark.gpu


def run_and_check(s, queries=None):
    ref = oracle.sparse_mla(s.q, s.cache, s.indices, s.positions, s.page_table, queries=queries, **s.options())
    g = s.to("cuda")
    prm = api.make_sparse_params(g.q, g.cache, g.indices, g.page_table, read_block=s.read_block,
                                 page_size=s.page_size, seq_len=s.seq_len, sm_scale=s.sm_scale)
    ws = torch.zeros(api.sparse_mla_workspace_size(prm), dtype=torch.uint8, device="cuda")
    out = api.sparse_mla_forward(g.q, g.cache, g.indices, g.positions, g.page_table, workspace=ws, **s.options())
    assert api.check_device_status(ws) == 0
    B, S = s.positions.shape
    flat_out = out.reshape(B * S, *out.shape[2:])
    flat_ref = ref.reshape(B * S, *ref.shape[2:])
    rows = list(range(B * S)) if queries is None else list(queries)
    err = max_abs(flat_out[rows], flat_ref[rows])
    assert err <= TOL_BF16, f"max-abs {err}"


@pytest.mark.parametrize("mode", ["token", "page"])
@pytest.mark.parametrize("phase", ["prefill", "decode"])
def test_sparse_small(mode, phase):
    run_and_check(workloads.dsa_sparse(mode=mode, phase=phase, scale=1 / 16))


def test_sparse_early_positions_pad_with_minus_one():
    # queries near position 0 have fewer causal units than K: their slots are -1 padded
    pos = np.array([[0, 1, 5, 63, 64, 200]], dtype=np.int32)
    for rb, k in [(1, 32), (16, 4)]:
        s = workloads.make_sparse(batch=1, num_queries=6, seq_len=256, positions=pos, topk=k, read_block=rb, seed=31)
        assert (s.indices == -1).any()
        run_and_check(s)


def test_sparse_duplicates_and_future_units():
    pos = np.array([[100, 100]], dtype=np.int32)
    idx = np.array([[[3, 3, 50, 120, 200, -1, 7, 7], [0, 1, 2, 3, 99, 100, 101, -1]]], dtype=np.int32)
    s = workloads.make_sparse(batch=1, num_queries=2, seq_len=256, positions=pos, topk=8, read_block=1, seed=32,
                              indices=idx)
    run_and_check(s)


@pytest.mark.parametrize("mode", ["token", "page"])
def test_sparse_prefill_full_size_sampled(mode):
    s = workloads.dsa_sparse(mode=mode, phase="prefill")
    # 48 queries: the first and the last, and one drawn from each of 46 equal strata between
    n = s.positions.numel()
    rng = np.random.default_rng(5)
    edges = np.linspace(1, n - 1, 47).astype(int)
    mid = [int(rng.integers(lo, max(lo + 1, hi))) for lo, hi in zip(edges[:-1], edges[1:])]
    run_and_check(s, queries=sorted({0, n - 1, *mid}))


@pytest.mark.parametrize("mode", ["token", "page"])
def test_sparse_decode_full_size_sampled(mode):
    s = workloads.dsa_sparse(mode=mode, phase="decode")
    run_and_check(s, queries=list(range(s.positions.numel())))  # every query of the batch


def test_sparse_split_merge():
    # two queries x 4096 selected tokens: far above one item per two-CTA cluster, so each
    # query's keys are split (8 ways) and the partials merged by the log-sum-exp rule
    pos = np.array([[8191, 5000]], dtype=np.int32)
    s = workloads.make_sparse(batch=1, num_queries=2, seq_len=8192, positions=pos, topk=4096, read_block=1, seed=33)
    # the library's rule: chunk = max(512, ceil(2 * 4096 / 38)) rounded to 64 keys -> 8 splits
    assert s.indices.shape[-1] * s.read_block > 512
    run_and_check(s)


# ---------------------------------------------------------------------------
# packed-ragged mode with the self-write
# ---------------------------------------------------------------------------
def run_ragged(s, *, write=True, tokens=None):
    """GPU call against the oracle: cache bytes after the self-write (bit exact) and the
    output rows of ``tokens`` (all by default) within the bf16 tolerance."""
    flat = s.cache.reshape(-1, s.cache.shape[-1])
    ref_cache = oracle.sparse_ragged_write(s.kvc, s.kpe, flat, s.loc, page_size=s.page_size)
    ref = oracle.sparse_mla_ragged(s.ql, s.qpe, ref_cache, s.topk, s.positions, s.seq_lens, s.cu_q_lens,
                                   s.cu_kv_lens, s.page_indices, queries=tokens, **s.options())
    g = s.to("cuda")
    if not write:  # attend only, over a cache already holding the rows
        g.cache.copy_(ref_cache.reshape(g.cache.shape).to("cuda"))
    prm = api.make_sparse_ragged_params(g.ql, g.qpe, g.cache, g.topk, g.seq_lens, g.page_indices, **s.options())
    ws = torch.zeros(api.sparse_mla_ragged_workspace_size(prm), dtype=torch.uint8, device="cuda")
    out = api.sparse_mla_write_and_attend_ragged(
        g.ql, g.qpe, g.kvc if write else None, g.kpe if write else None, g.cache, g.topk, g.positions,
        g.loc if write else None, g.seq_lens, g.cu_q_lens, g.cu_kv_lens, g.page_indices, workspace=ws, **s.options())
    assert api.check_device_status(ws) == 0
    torch.cuda.synchronize()
    got_cache = g.cache.reshape(-1, g.cache.shape[-1]).cpu()
    assert torch.equal(got_cache.view(torch.int16), ref_cache.view(torch.int16))
    rows = list(range(s.ql.shape[0])) if tokens is None else list(tokens)
    err = max_abs(out[rows], ref[rows])
    assert err <= TOL_BF16, f"max-abs {err}"
    return out


@pytest.mark.parametrize("rb,k", [(1, 24), (16, 6), (64, 3)])
def test_sparse_ragged_small(rb, k):
    # three requests (one a single decode token), padding tokens with loc -1, spare pages
    s = workloads.make_sparse_ragged([3, 5, 1], [200, 333, 90], topk=k, read_block=rb, seed=40 + rb, extra_pages=3,
                                     pad_tokens=2)
    run_ragged(s)


def test_sparse_ragged_attend_only():
    s = workloads.make_sparse_ragged([4, 2], [150, 70], topk=16, read_block=1, seed=47, extra_pages=1)
    run_ragged(s, write=False)


def test_sparse_ragged_full_size_sampled():
    for mode in ("token", "page"):
        s = workloads.dsa_sparse_ragged(mode=mode)
        rng = np.random.default_rng(3)
        tokens = sorted(rng.choice(s.ql.shape[0], size=48, replace=False).tolist())
        run_ragged(s, tokens=tokens)
