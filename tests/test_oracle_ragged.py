"""Pins of the packed-ragged sparse-MLA oracle (sglang-jax "dsa/sparse_mla_prefill.py",
prefill_write_and_attend_ragged and the ragged branch of sparse_mla_attention) against things
other than itself: a dense brute force in numpy/scipy over every cache row, the already pinned
per-batch paged oracle (one request), plain causal attention (every key selected), and the
bytes of the self-write."""
import numpy as np
import pytest
import torch

import oracle

scipy_special = pytest.importorskip("scipy.special")


def _bf16(rng, shape, scale=1.0):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)


def make_case(seed, *, q_lens, seq_lens, page_size=4, read_block=2, topk=3, heads=2, dv=8, rope=4, row_stride=16,
              pad_tokens=0, extra_pages=3):
    """Tiny packed-ragged batch: request r owns tokens cu_q_lens[r]..; its pages are a random
    run of the packed page list starting at cu_kv_lens[r] / page_size."""
    rng = np.random.default_rng(seed)
    S = len(q_lens)
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(cu_q[-1]) + pad_tokens
    pages_per = [-(-int(L) // page_size) for L in seq_lens]
    cu_kv = np.concatenate([[0], np.cumsum([n * page_size for n in pages_per])]).astype(np.int32)
    ptw = int(sum(pages_per))
    P = ptw + extra_pages
    page_indices = rng.permutation(P)[:ptw].astype(np.int32)
    cache = _bf16(rng, (P * page_size, row_stride))
    ql, qpe = _bf16(rng, (T, heads, dv)), _bf16(rng, (T, heads, rope))
    positions = np.zeros(T, np.int32)
    topk_ids = np.full((T, topk), -1, np.int32)
    for r in range(S):
        L = int(seq_lens[r])
        for j, t in enumerate(range(cu_q[r], cu_q[r + 1])):
            positions[t] = L - q_lens[r] + j
            n_units = -(-L // read_block)
            k = min(topk, n_units)
            topk_ids[t, :k] = rng.choice(n_units, size=k, replace=False)
    for t in range(cu_q[-1], T):  # padding tokens: any position, units of the last request
        positions[t] = int(seq_lens[-1]) - 1
        topk_ids[t, 0] = 0
    return dict(ql=ql, qpe=qpe, cache=cache, topk=torch.from_numpy(topk_ids), positions=torch.from_numpy(positions),
                seq_lens=torch.tensor(seq_lens, dtype=torch.int32), cu_q_lens=torch.from_numpy(cu_q),
                cu_kv_lens=torch.from_numpy(cu_kv), page_indices=torch.from_numpy(page_indices),
                read_block=read_block, page_size=page_size, sm_scale=0.3)


def numpy_ragged(c):
    """Dense brute force: the score of every query against every cache row, masked to the rows
    the query's selected units name (request from np.searchsorted, bound, packed page base)."""
    ql = c["ql"].float().numpy().astype(np.float64)
    qpe = c["qpe"].float().numpy().astype(np.float64)
    cache = c["cache"].float().numpy().astype(np.float64)
    q = np.concatenate([ql, qpe], axis=-1)  # [T, H, dk]
    T, H, dk = q.shape
    dv = ql.shape[-1]
    ps, rb = c["page_size"], c["read_block"]
    cu_q, seq_lens, cu_kv = c["cu_q_lens"].numpy(), c["seq_lens"].numpy(), c["cu_kv_lens"].numpy()
    pages = c["page_indices"].numpy()
    S = len(seq_lens)
    rid = np.clip(np.searchsorted(cu_q[1:], np.arange(T), side="right"), 0, S - 1)
    scores = np.einsum("thd,rd->thr", q, cache[:, :dk]) * c["sm_scale"]  # every row
    count = np.zeros((T, cache.shape[0]))  # how many selected keys name each row
    for t in range(T):
        r = rid[t]
        for u in c["topk"][t].numpy():
            if u < 0:
                continue
            for kp in range(u * rb, u * rb + rb):
                if kp <= c["positions"][t] and kp < seq_lens[r]:
                    pidx = min(cu_kv[r] // ps + kp // ps, len(pages) - 1)
                    count[t, pages[pidx] * ps + kp % ps] += 1
    out = np.zeros((T, H, dv))
    for t in range(T):
        rows = np.nonzero(count[t])[0]
        if len(rows) == 0:
            continue
        # a row named twice counts twice: log-weights carry the multiplicity
        logits = scores[t][:, rows] + np.log(count[t, rows])[None, :]
        w = scipy_special.softmax(logits, axis=-1)
        out[t] = w @ cache[rows][:, :dv]
    return out


def run_oracle(c, **kw):
    return oracle.sparse_mla_ragged(c["ql"], c["qpe"], c["cache"], c["topk"], c["positions"], c["seq_lens"],
                                    c["cu_q_lens"], c["cu_kv_lens"], c["page_indices"], read_block=c["read_block"],
                                    page_size=c["page_size"], sm_scale=c["sm_scale"], **kw).numpy()


@pytest.mark.parametrize("seed,rb,pad", [(0, 1, 0), (1, 2, 0), (2, 4, 2), (3, 2, 3)])
def test_ragged_oracle_matches_dense_brute_force(seed, rb, pad):
    c = make_case(seed, q_lens=[3, 1, 4], seq_lens=[9, 5, 13], read_block=rb, pad_tokens=pad)
    np.testing.assert_allclose(run_oracle(c), numpy_ragged(c), rtol=1e-12, atol=1e-12)


def test_ragged_oracle_one_request_is_the_paged_oracle():
    # one request: the packed list is its page table, bound = seq_len, base 0
    c = make_case(7, q_lens=[6], seq_lens=[14], read_block=2, topk=4)
    T = c["ql"].shape[0]
    q = torch.cat([c["ql"], c["qpe"]], dim=-1).reshape(1, T, *c["ql"].shape[1:2], -1)
    ref = oracle.sparse_mla(q, c["cache"], c["topk"].reshape(1, T, -1), c["positions"].reshape(1, T),
                            c["page_indices"].reshape(1, -1), read_block=2, page_size=c["page_size"], seq_len=14,
                            sm_scale=c["sm_scale"], dv=c["ql"].shape[-1])
    np.testing.assert_allclose(run_oracle(c), ref.reshape(T, *ref.shape[2:]).numpy(), rtol=1e-13, atol=1e-13)


def test_ragged_oracle_all_keys_selected_is_causal_attention():
    # read_block 1 and every key of the request selected: plain causal attention (torch SDPA)
    c = make_case(11, q_lens=[5, 3], seq_lens=[12, 7], read_block=1, topk=12)
    cu_q = c["cu_q_lens"].numpy()
    for r, L in enumerate([12, 7]):
        for t in range(cu_q[r], cu_q[r + 1]):
            ids = np.full(12, -1, np.int32)
            ids[:L] = np.arange(L)
            c["topk"][t] = torch.from_numpy(ids)
    got = run_oracle(c)
    ps, pages = c["page_size"], c["page_indices"].numpy()
    cache = c["cache"].double()
    for r, L in enumerate([12, 7]):
        base = int(c["cu_kv_lens"][r]) // ps
        rows = [pages[base + kp // ps] * ps + kp % ps for kp in range(L)]
        k = cache[rows][:, :12]                       # [L, dk]
        v = cache[rows][:, :8]                        # [L, dv]
        toks = list(range(cu_q[r], cu_q[r + 1]))
        q = torch.cat([c["ql"][toks], c["qpe"][toks]], dim=-1).double().transpose(0, 1)  # [H, n, dk]
        pos = c["positions"][toks]
        mask = torch.arange(L)[None, :] <= pos[:, None]   # [n, L]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k[None].expand(q.shape[0], -1, -1), v[None].expand(q.shape[0], -1, -1), attn_mask=mask,
            scale=c["sm_scale"])
        np.testing.assert_allclose(got[toks], ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_ragged_self_write_bytes():
    rng = np.random.default_rng(5)
    P, ps, stride, dv, rope = 6, 4, 16, 8, 4
    cache = _bf16(rng, (P * ps, stride))
    T = 7
    kvc, kpe = _bf16(rng, (T, dv)), _bf16(rng, (T, rope))
    loc = torch.tensor([3, -1, 20, P * ps, 0, 23, -5], dtype=torch.int32)  # -1, -5 and 24 are dropped
    out = oracle.sparse_ragged_write(kvc, kpe, cache, loc, page_size=ps)
    want = cache.clone()
    for t, slot in enumerate(loc.tolist()):
        if 0 <= slot < P * ps:
            want[slot] = torch.cat([kvc[t], kpe[t], torch.zeros(stride - dv - rope, dtype=torch.bfloat16)])
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    untouched = [s for s in range(P * ps) if s not in {3, 20, 0, 23}]
    assert torch.equal(out[untouched].view(torch.int16), cache[untouched].view(torch.int16))


def test_ragged_padding_tokens_belong_to_the_last_request():
    # tokens past cu_q_lens[S] take the last request's bound and page base (the page's clip)
    c = make_case(13, q_lens=[2, 2], seq_lens=[6, 10], read_block=2, pad_tokens=2)
    got = run_oracle(c)
    c2 = dict(c)
    c2["cu_q_lens"] = torch.tensor([0, 2, 6], dtype=torch.int32)  # the padding made part of request 1
    np.testing.assert_allclose(got[4:], run_oracle(c2)[4:], rtol=0, atol=0)
