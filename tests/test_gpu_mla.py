"""GPU parity of mla_rpa_forward / mla_update_kv_cache against the float64 oracle."""
import pytest
import torch

import oracle
from ragged_paged_attention_gb300 import api, workloads
from parity import TOL_BF16, max_abs, sample_tokens

pytestmark = pytest.mark.gpu


def run_and_check(m, tokens=None, **over):
    opts = m.options()
    opts.update(over)
    ref, ckv, ckpe = oracle.mla_forward(m.ql_nope, m.q_pe, m.new_kv_c, m.new_k_pe, m.cache_kv_c, m.cache_k_pe,
                                        m.kv_lens, m.page_indices, m.cu_q_lens, m.distribution, tokens=tokens, **opts)
    g = m.to("cuda")
    out = torch.full(g.ql_nope.shape, 7.0, dtype=torch.bfloat16, device="cuda")
    prm = api.make_mla_params(g.ql_nope, g.q_pe, g.cache_kv_c, g.cache_k_pe, g.kv_lens, g.page_indices, **opts)
    ws = torch.zeros(api.mla_workspace_size(prm), dtype=torch.uint8, device="cuda")
    api.mla_rpa_forward(g.ql_nope, g.q_pe, g.new_kv_c, g.new_k_pe, g.cache_kv_c, g.cache_k_pe, g.kv_lens,
                        g.page_indices, g.cu_q_lens, g.distribution, out=out, workspace=ws, **opts)
    assert api.check_device_status(ws) == 0
    assert torch.equal(g.cache_kv_c.cpu().view(torch.int16), ckv.view(torch.int16))
    assert torch.equal(g.cache_k_pe.cpu().view(torch.int16), ckpe.view(torch.int16))
    T = m.num_tokens
    rows = list(range(T)) if tokens is None else list(tokens)
    err = max_abs(out[rows], ref[rows])
    assert err <= TOL_BF16, f"max-abs {err}"
    assert (out[T:].float() == 7.0).all()


def test_mla_small():
    run_and_check(workloads.mla_deepseek(scale=1 / 16))


def test_mla_window_and_cap():
    m = workloads.make_mla([1, 1, 40], [700, 65, 300], seed=21, max_num_tokens=48)
    run_and_check(m, sliding_window=100, soft_cap=20.0)


def test_mla_prefill_from_zero_and_short_keys():
    m = workloads.make_mla([1, 64, 3], [1, 64, 3], seed=22, extra_pages=2, max_num_seqs=5)
    run_and_check(m)


@pytest.mark.parametrize("page_size", [64, 16])
def test_mla_short_items_after_split_items(page_size):
    # a long decode row (split items: fp32 partials, merged) beside a causal prefill whose rows
    # see 1..256 keys: short items follow long ones on the same CTAs, and a block that is not
    # full must hold zeros, never stale shared-memory bytes, past its keys
    m = workloads.make_mla([1, 256], [24000, 256], seed=27, page_size=page_size)
    run_and_check(m)


@pytest.mark.parametrize("page_size", [12, 4])
def test_mla_register_gather_page_sizes(page_size):
    # page sizes that no TMA box fits (not a power of two, or under 8 rows): the key rows come
    # through the register-gather instantiation
    m = workloads.make_mla([1, 1, 40], [700, 65, 300], seed=28, page_size=page_size, max_num_tokens=48)
    run_and_check(m)


def test_mla_full_size_sampled():
    m = workloads.mla_deepseek()
    run_and_check(m, tokens=sample_tokens(m.q_lens, per_chunk=4))


def test_mla_update_only_bit_exact():
    m = workloads.make_mla([2, 1, 9], [10, 64, 70], seed=23, extra_pages=3, max_num_seqs=4, max_num_tokens=16)
    ckv, ckpe = oracle.mla_update_kv_cache(m.new_kv_c, m.new_k_pe, m.cache_kv_c, m.cache_k_pe, m.kv_lens,
                                           m.page_indices, m.cu_q_lens, m.distribution)
    g = m.to("cuda")
    api.mla_update_kv_cache(g.new_kv_c, g.new_k_pe, g.cache_kv_c, g.cache_k_pe, g.kv_lens, g.page_indices,
                            g.cu_q_lens, g.distribution)
    torch.cuda.synchronize()
    assert torch.equal(g.cache_kv_c.cpu().view(torch.int16), ckv.view(torch.int16))
    assert torch.equal(g.cache_k_pe.cpu().view(torch.int16), ckpe.view(torch.int16))


@pytest.mark.parametrize("mask,sw", [(-1.5, None), (-3.0, 100), (0.25, 40)])
def test_mla_mild_mask_value_replaces(mask, sw):
    # The MLA reference replaces a masked logit by mask_value; with a value that leaves masked
    # keys real weight, each query sees every key of its sequence: its future keys (prefill)
    # and the keys outside the window at mask_value.
    m = workloads.make_mla([1, 1, 40, 3], [700, 65, 300, 9], seed=24, max_num_tokens=48)
    run_and_check(m, mask_value=mask, sliding_window=sw)


@pytest.mark.parametrize("q_scale,sw,cap", [(0.125, None, None), (0.03, 100, 25.0), (0.5, None, None)])
def test_mla_fp8_queries(q_scale, sw, cap):
    # per-tensor fp8 e4m3 queries: widened exactly in the kernel, scores carry q_scale
    m = workloads.make_mla([1, 1, 40, 3, 70], [700, 65, 300, 9, 70], seed=25, max_num_tokens=128,
                           q_dtype=torch.float8_e4m3fn, q_scale=q_scale)
    assert m.ql_nope.dtype == torch.float8_e4m3fn
    run_and_check(m, sliding_window=sw, soft_cap=cap)


def test_mla_fp8_queries_full_size_sampled():
    m0 = workloads.mla_deepseek()
    m = workloads.make_mla(m0.q_lens, m0.kv_lens_list, seed=26, q_dtype=torch.float8_e4m3fn)
    run_and_check(m, tokens=sample_tokens(m.q_lens, per_chunk=2))
