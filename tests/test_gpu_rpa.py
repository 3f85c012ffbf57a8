"""GPU parity of rpa_forward / rpa_update_kv_cache against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from ragged_paged_attention_gb300 import api, workloads
from parity import TOL_BF16, TOL_FP8, gpu, max_abs, sample_tokens

pytestmark = pytest.mark.gpu


def run_gpu(b, **over):
    g = b.to("cuda")
    opts = b.options()
    opts.update(over)
    ws = torch.zeros(api.rpa_workspace_size(api.make_rpa_params(g.q, g.kv_pages, g.page_indices, **opts)),
                     dtype=torch.uint8, device="cuda")
    out = torch.full_like(g.q, 7.0)
    api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, out=out, workspace=ws, **opts)
    bits = api.check_device_status(ws)
    return out, bits, ws


def check(b, tol, tokens=None, **over):
    out, bits, _ = run_gpu(b, **over)
    assert bits == 0, f"device error bits {bits:#x}"
    opts = b.options()
    opts.update(over)
    ref = oracle.rpa(b.q, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens), tokens=tokens, **opts)
    T = b.num_tokens
    rows = list(range(T)) if tokens is None else list(tokens)
    err = max_abs(out[rows], ref[rows])
    assert err <= tol, f"max-abs {err} > {tol}"
    # rows of padding tokens are never written
    assert (out[T:].float() == 7.0).all()
    return out


def test_tiny_batch():
    check(workloads.tiny_rpa(), TOL_BF16)


def test_llama_mixed_small():
    check(workloads.llama_mixed(scale=1 / 8), TOL_BF16)


def test_gemma_options_small():
    check(workloads.gemma_options(scale=1 / 8), TOL_FP8)


def test_llama_mixed_full_size_sampled():
    b = workloads.llama_mixed()
    check(b, TOL_BF16, tokens=sample_tokens(b.q_lens))


def test_gemma_options_full_size_sampled():
    b = workloads.gemma_options()
    check(b, TOL_FP8, tokens=sample_tokens(b.q_lens))


@pytest.mark.parametrize("hq,hkv,d,ps", [(8, 1, 64, 8), (16, 2, 128, 4), (4, 4, 256, 16), (32, 2, 128, 32)])
def test_head_layouts(hq, hkv, d, ps):
    b = workloads.make_rpa([1, 3, 17, 70, 2], [1, 40, 17, 150, 9], num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                           page_size=ps, seed=hq * d + ps, max_num_seqs=7, max_num_tokens=100, extra_pages=3)
    check(b, TOL_BF16)


@pytest.mark.parametrize("sw,cap", [(1, None), (5, 30.0), (64, None), (None, 2.0)])
def test_window_and_cap(sw, cap):
    b = workloads.make_rpa([1, 4, 40, 1], [300, 33, 120, 1], num_q_heads=8, num_kv_heads=2, head_dim=128,
                           page_size=16, seed=11, sliding_window=sw, soft_cap=cap)
    check(b, TOL_BF16)


def test_fp8_without_scale_and_bf16_with_scale():
    b = workloads.make_rpa([1, 9], [77, 30], num_q_heads=8, num_kv_heads=4, head_dim=128, page_size=16, seed=12,
                           kv_dtype=torch.float8_e4m3fn)
    check(b, TOL_FP8)
    b2 = workloads.make_rpa([1, 9], [77, 30], num_q_heads=8, num_kv_heads=4, head_dim=128, page_size=16, seed=13,
                            k_scale=0.37, v_scale=1.7)
    check(b2, TOL_BF16)


@pytest.mark.parametrize("ks,vs", [(0.5, 4.0), (0.37, 1.7)])
def test_fp8_scales_and_query_magnitudes(ks, vs):
    # power-of-two scales take the f16 tensor-core paths of decode and prefill (exact fp8 ->
    # f16, scales applied to S and O); other scales dequantise to bf16. Query rows far from
    # unit size exercise the per-row power-of-two range factor in both directions (the 9- and
    # 5-token sequences are prefill tiles, the others decode).
    b = workloads.make_rpa([1, 9, 1, 5], [77, 30, 200, 64], num_q_heads=8, num_kv_heads=2, head_dim=128,
                           page_size=16, seed=17, kv_dtype=torch.float8_e4m3fn, k_scale=ks, v_scale=vs)
    for (lo, hi), f in zip([(0, 1), (1, 10), (10, 11), (11, 16)], [2e4, 1e-3, 64.0, 300.0]):
        b.q[lo:hi] = (b.q[lo:hi].float() * f).to(b.q.dtype)
    check(b, TOL_FP8 * vs)


@pytest.mark.parametrize("q_lens,kv_lens,hq,hkv", [
    ([1, 1] + [256] * 4, [40, 70] + [1024] * 4, 16, 4),        # prefill-heavy: decode ends first
    ([1] * 60 + [40], [3000] * 60 + [300], 16, 4),             # decode-heavy, one small prefill
    ([1] * 30, list(range(100, 3100, 100)), 16, 4),            # decode only
    ([200, 300], [900, 300], 16, 4),                           # prefill only
    ([1, 1, 1, 1, 24], [5000, 17, 2000, 1, 600], 32, 2),       # 16 query rows: two 8-row halves
])
def test_prefill_beside_decode_regimes(q_lens, kv_lens, hq, hkv):
    # the SM split between the two kernels, the prefill left for the launch after decode and
    # the equal decode shares depend on the batch's mix of work
    b = workloads.make_rpa(q_lens, kv_lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, page_size=16,
                           seed=sum(kv_lens) % 1000)
    check(b, TOL_BF16, tokens=sample_tokens(b.q_lens))


@pytest.mark.parametrize("kv_dtype,d,ps,ks", [(torch.bfloat16, 128, 16, None), (torch.float8_e4m3fn, 256, 32, 0.5),
                                              (torch.float8_e4m3fn, 128, 16, 0.37)],
                         ids=["bf16-tma", "fp8-f16", "fp8-dequant"])
def test_many_short_prefill_items(kv_dtype, d, ps, ks):
    # 1200 one-block prefill tiles: every CTA runs several items back to back, its producers
    # and QK issuer already on the next item while the softmax warps finish the current one.
    # Queries of alternate sequences differ in size by 2^6, so a Q tile or a per-row factor
    # taken from the wrong item would show at once.
    rng = np.random.default_rng(31)
    n = 600
    kv_lens = [int(x) for x in rng.integers(8, 61, size=n)]
    extra = {} if ks is None else dict(k_scale=ks, v_scale=ks)
    b = workloads.make_rpa([8] * n, kv_lens, num_q_heads=8, num_kv_heads=2, head_dim=d, page_size=ps, seed=31,
                           kv_dtype=kv_dtype, **extra)
    for s in range(n):
        f = 8.0 if s % 2 else 0.125
        b.q[8 * s:8 * s + 8] = (b.q[8 * s:8 * s + 8].float() * f).to(b.q.dtype)
    check(b, TOL_BF16 if kv_dtype == torch.bfloat16 else TOL_FP8)


def test_serialised_launches():
    # with per-kernel timing on, the kernels run one after another (prefill on every SM,
    # decode after it): the same results within tolerance
    b = workloads.llama_mixed(scale=1 / 8)
    with api.KernelTimer() as kt:
        check(b, TOL_BF16)
    assert {"rpa_plan", "rpa_prefill_attn", "rpa_decode_attn"} <= set(kt.result)


def test_empty_batch_and_zero_length_sequences():
    b = workloads.make_rpa([0, 2, 0], [5, 2, 0], num_q_heads=4, num_kv_heads=2, head_dim=128, page_size=16, seed=14,
                           max_num_tokens=8)
    check(b, TOL_BF16)
    g = b.to("cuda")
    g.num_seqs.zero_()
    out = torch.full_like(g.q, 7.0)
    api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, out=out, **b.options())
    torch.cuda.synchronize()
    assert (out.float() == 7.0).all()


def test_long_prefill_from_position_zero():
    b = workloads.make_rpa([300, 1], [300, 600], num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                           seed=15)
    check(b, TOL_BF16)


def test_page_permutation_is_bit_exact():
    b = workloads.make_rpa([1, 1, 33], [900, 20, 200], num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                           seed=16, extra_pages=5)
    out1, bits, _ = run_gpu(b)
    P = b.kv_pages.shape[0]
    perm = torch.from_numpy(np.random.default_rng(3).permutation(P))
    pages = torch.empty_like(b.kv_pages)
    pages[perm] = b.kv_pages
    table = b.page_indices.clone()
    ok = table < P
    table[ok] = perm[table[ok].long()].to(torch.int32)
    b.kv_pages, b.page_indices = pages, table
    out2, bits2, _ = run_gpu(b)
    T = b.num_tokens
    assert bits == bits2 == 0
    assert torch.equal(out1[:T].view(torch.int16), out2[:T].view(torch.int16))


def test_bad_page_index_sets_device_error():
    b = workloads.make_rpa([1, 5], [40, 50], num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, seed=17)
    b.page_indices[1, 1] = b.kv_pages.shape[0] + 3   # out of range: the kernels skip it and report
    out, bits, _ = run_gpu(b)
    assert bits & 0x08
    b.page_indices[1, 1] = 0
    b.kv_lens[0] = 10**6                             # more pages than pages_per_seq
    out, bits, _ = run_gpu(b)
    assert bits & 0x04


@pytest.mark.parametrize("d", [128, 96, 192])
@pytest.mark.parametrize("kv_dtype", [torch.bfloat16, torch.float8_e4m3fn, torch.int8, torch.uint8])
def test_update_kv_cache_bit_exact(kv_dtype, d):
    # (uint8: packed int4; the cache write moves any of the dtypes at any of the head sizes)
    b = workloads.make_rpa([1, 1, 6, 19], [33, 1, 6, 40], num_q_heads=8, num_kv_heads=4, head_dim=d, page_size=16,
                           seed=18, kv_dtype=kv_dtype, max_num_seqs=6, max_num_tokens=32, extra_pages=4)
    ref = oracle.rpa_update_kv_cache(b.new_k[:b.num_tokens].contiguous(), b.new_v[:b.num_tokens].contiguous(),
                                     b.kv_pages, b.kv_lens[:4], b.page_indices[:4], b.cu_q_lens[:5], 4)
    g = b.to("cuda")
    api.rpa_update_kv_cache(g.new_k, g.new_v, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs)
    torch.cuda.synchronize()
    assert torch.equal(g.kv_pages.cpu().view(torch.uint8), ref.view(torch.uint8))


def test_update_then_attend_full_size():
    b = workloads.llama_mixed(scale=1 / 4)
    g = b.to("cuda")
    api.rpa_update_kv_cache(g.new_k, g.new_v, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs)
    ref_pages = oracle.rpa_update_kv_cache(b.new_k[:b.num_tokens].contiguous(), b.new_v[:b.num_tokens].contiguous(),
                                           b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens))
    torch.cuda.synchronize()
    assert torch.equal(g.kv_pages.cpu().view(torch.int16), ref_pages.view(torch.int16))
    out = api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, **b.options())
    toks = sample_tokens(b.q_lens)
    ref = oracle.rpa(b.q, ref_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens), tokens=toks,
                     **b.options())
    assert max_abs(out[toks], ref[toks]) <= TOL_BF16


@pytest.mark.parametrize("make", [
    lambda: workloads.llama_mixed(scale=1 / 8),
    lambda: workloads.gemma_options(scale=1 / 8),
    lambda: workloads.make_rpa([1, 1, 6, 19, 1], [33, 1, 6, 40, 300], num_q_heads=8, num_kv_heads=4, head_dim=64,
                               page_size=8, seed=19, kv_dtype=torch.float8_e4m3fn, k_scale=0.37, v_scale=1.7,
                               max_num_seqs=7, max_num_tokens=40, extra_pages=4),
], ids=["llama", "gemma_fp8", "fp8_scaled_d64"])
def test_forward_update_matches_update_then_forward(make):
    # the fused call writes the same cache bytes as rpa_update_kv_cache and attends over them
    b = make()
    n = len(b.q_lens)
    ref_pages = oracle.rpa_update_kv_cache(b.new_k[:b.num_tokens].contiguous(), b.new_v[:b.num_tokens].contiguous(),
                                           b.kv_pages, b.kv_lens[:n], b.page_indices[:n], b.cu_q_lens[:n + 1], n)
    g1, g2 = b.to("cuda"), b.to("cuda")
    opts = b.options()
    api.rpa_update_kv_cache(g1.new_k, g1.new_v, g1.kv_pages, g1.kv_lens, g1.page_indices, g1.cu_q_lens, g1.num_seqs)
    out1 = api.rpa_forward(g1.q, g1.kv_pages, g1.kv_lens, g1.page_indices, g1.cu_q_lens, g1.num_seqs, **opts)
    ws = torch.zeros(api.rpa_workspace_size(api.make_rpa_params(g2.q, g2.kv_pages, g2.page_indices, **opts)),
                     dtype=torch.uint8, device="cuda")
    out2 = torch.full_like(g2.q, 7.0)
    api.rpa_forward_update(g2.q, g2.new_k, g2.new_v, g2.kv_pages, g2.kv_lens, g2.page_indices, g2.cu_q_lens,
                           g2.num_seqs, out=out2, workspace=ws, **opts)
    assert api.check_device_status(ws) == 0
    torch.cuda.synchronize()
    assert torch.equal(g2.kv_pages.cpu().view(torch.uint8), ref_pages.view(torch.uint8))
    T = b.num_tokens
    assert torch.equal(out2[:T], out1[:T])  # same plan, same kernels: the same bits
    assert (out2[T:].float() == 7.0).all()
    tokens = sample_tokens(b.q_lens)
    ref = oracle.rpa(b.q, ref_pages, b.kv_lens, b.page_indices, b.cu_q_lens, n, tokens=tokens, **opts)
    tol = TOL_FP8 * (opts["v_scale"] or 1.0) if b.kv_pages.dtype == torch.float8_e4m3fn else TOL_BF16
    assert max_abs(out2[tokens], ref[tokens]) <= tol


@pytest.mark.parametrize("ks,vs", [(None, None), (1 / 32, 1 / 64), (0.0123, 0.021)],
                         ids=["exact", "pow2_f16", "scaled_bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_int8_kv(ks, vs, d):
    # int8 caches: exact integers without scales and with power-of-two scales (the f16
    # tensor-core path), bf16(float(x) * scale) otherwise; decode and prefill sequences
    hq, hkv = (8, 2) if d < 256 else (4, 2)
    b = workloads.make_rpa([1, 9, 1, 40], [77, 30, 300, 200], num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                           page_size=16, seed=60 + d, kv_dtype=torch.int8, k_scale=ks, v_scale=vs,
                           sm_scale=2.0 / (74.0 * (ks or 1.0) * math.sqrt(d)))  # logits' spread ~2
    out, bits, _ = run_gpu(b)
    assert bits == 0
    ref = oracle.rpa(b.q, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens), **b.options())
    T = b.num_tokens
    scale = float(ref[:T].abs().max())
    assert max_abs(out[:T], ref[:T]) <= 2e-2 * scale


@pytest.mark.parametrize("mask", [-1.5, -4.0, 0.5])
@pytest.mark.parametrize("kind", ["bf16_tma", "fp8_raw", "window_cap", "int8_decode_rows"])
def test_mild_mask_value_is_added(mask, kind):
    # The RPA reference adds mask_value to a masked logit. With a value that leaves masked keys
    # real weight, every key of a sequence takes part: the future keys of a chunk's queries and
    # the keys outside the window, each with mask_value added after the scale and the soft cap.
    # Decode rows (q_len * G <= 16, including two-row decode items) and prefill tiles; the bf16
    # TMA path, the fp8 raw-staging path and the int8 register path.
    if kind == "bf16_tma":
        b = workloads.make_rpa([1, 1, 9, 40], [300, 33, 120, 200], num_q_heads=8, num_kv_heads=2, head_dim=128,
                               page_size=16, seed=41)
        tol = TOL_BF16
    elif kind == "fp8_raw":
        b = workloads.make_rpa([1, 70, 1, 130], [500, 300, 90, 260], num_q_heads=16, num_kv_heads=8, head_dim=256,
                               page_size=32, seed=42, kv_dtype=torch.float8_e4m3fn, k_scale=0.5, v_scale=0.5)
        tol = TOL_FP8
    elif kind == "window_cap":
        b = workloads.make_rpa([1, 5, 33, 1], [400, 64, 150, 7], num_q_heads=8, num_kv_heads=4, head_dim=128,
                               page_size=16, seed=43, sliding_window=50, soft_cap=30.0)
        tol = TOL_BF16
    else:
        b = workloads.make_rpa([2, 3, 1, 20], [40, 90, 700, 64], num_q_heads=16, num_kv_heads=4, head_dim=128,
                               page_size=16, seed=44, kv_dtype=torch.int8, k_scale=1 / 64, v_scale=1 / 64,
                               sliding_window=30)
        tol = TOL_BF16
    check(b, tol, mask_value=mask)


def _launches(fn):
    n0 = api.launch_count()
    fn()
    torch.cuda.synchronize()
    return api.launch_count() - n0


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_batch_kind_hint_skips_the_other_launches(kind):
    # a batch of one class with the matching hint: the same bits, with the other class's
    # launches (decode: both prefill grids; prefill: decode and the prefill tail) not made
    if kind == "decode":
        b = workloads.make_rpa([1] * 30 + [2], list(range(100, 3100, 100)) + [40], num_q_heads=16, num_kv_heads=4,
                               head_dim=128, page_size=16, seed=51)
        hint = api.BATCH_DECODE_ONLY
    else:
        b = workloads.make_rpa([200, 37], [900, 300], num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=16,
                               seed=52)
        hint = api.BATCH_PREFILL_ONLY
    g = b.to("cuda")
    opts = b.options()
    ref = torch.full_like(g.q, 7.0)
    n_plain = _launches(lambda: api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens,
                                                g.num_seqs, out=ref, **opts))
    out = torch.full_like(g.q, 7.0)
    ws = torch.zeros(api.rpa_workspace_size(api.make_rpa_params(g.q, g.kv_pages, g.page_indices, **opts)),
                     dtype=torch.uint8, device="cuda")
    n_hint = _launches(lambda: api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs,
                                               out=out, workspace=ws, batch_kind=hint, **opts))
    assert api.check_device_status(ws) == 0
    assert n_hint == 2 and n_plain == 4
    T = b.num_tokens
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    tokens = sample_tokens(b.q_lens)
    ref64 = oracle.rpa(b.q, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens), tokens=tokens, **opts)
    assert max_abs(out[tokens], ref64[tokens]) <= TOL_BF16
    assert (out[T:].float() == 7.0).all()


def test_batch_kind_hint_violation_is_reported():
    # a decode-only hint on a mixed batch: the prefill-class sequence is skipped (its rows stay
    # unwritten) and reported; the decode rows are computed
    b = workloads.make_rpa([1, 40, 1], [300, 200, 77], num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                           seed=53)
    g = b.to("cuda")
    opts = b.options()
    ws = torch.zeros(api.rpa_workspace_size(api.make_rpa_params(g.q, g.kv_pages, g.page_indices, **opts)),
                     dtype=torch.uint8, device="cuda")
    out = torch.full_like(g.q, 7.0)
    api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, out=out, workspace=ws,
                    batch_kind=api.BATCH_DECODE_ONLY, **opts)
    assert api.check_device_status(ws) & 0x80
    assert (out[1:41].float() == 7.0).all()
    ref = oracle.rpa(b.q, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, 3, tokens=[0, 41], **opts)
    assert max_abs(out[[0, 41]], ref[[0, 41]]) <= TOL_BF16


@pytest.mark.parametrize("ks,vs", [(None, None), (1 / 4, 1 / 8), (0.0123, 0.021)],
                         ids=["exact", "pow2", "scaled"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_int4_kv(ks, vs, d):
    # int4 caches (two's-complement nibbles, element 2i in the low nibble of byte i): exact
    # integers without scales, bf16(float(x) * scale) with them; decode rows (two-row items too)
    # and prefill tiles, windowed and not
    hq, hkv = (8, 2) if d < 256 else (4, 2)
    b = workloads.make_rpa([1, 9, 2, 40], [77, 30, 300, 200], num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                           page_size=16, seed=70 + d, kv_dtype=torch.uint8, k_scale=ks, v_scale=vs,
                           sliding_window=150 if d == 128 else None,
                           sm_scale=2.0 / (4.6 * (ks or 1.0) * math.sqrt(d)))  # logits' spread ~2
    out, bits, _ = run_gpu(b)
    assert bits == 0
    ref = oracle.rpa(b.q, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens), **b.options())
    T = b.num_tokens
    scale = float(ref[:T].abs().max())
    assert max_abs(out[:T], ref[:T]) <= 2e-2 * scale
    assert (out[T:].float() == 7.0).all()


def test_int4_update_then_attend():
    # the cache write moves packed bytes unchanged; the fused call attends over them
    b = workloads.make_rpa([1, 1, 6, 19], [33, 1, 6, 40], num_q_heads=8, num_kv_heads=4, head_dim=128, page_size=16,
                           seed=18, kv_dtype=torch.uint8, max_num_seqs=6, max_num_tokens=32, extra_pages=4,
                           k_scale=0.5, v_scale=0.5)
    n = len(b.q_lens)
    ref_pages = oracle.rpa_update_kv_cache(b.new_k[:b.num_tokens].contiguous(), b.new_v[:b.num_tokens].contiguous(),
                                           b.kv_pages, b.kv_lens[:n], b.page_indices[:n], b.cu_q_lens[:n + 1], n)
    g = b.to("cuda")
    out = api.rpa_forward_update(g.q, g.new_k, g.new_v, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens,
                                 g.num_seqs, **b.options())
    torch.cuda.synchronize()
    assert torch.equal(g.kv_pages.cpu(), ref_pages)
    ref = oracle.rpa(b.q, ref_pages, b.kv_lens, b.page_indices, b.cu_q_lens, n, **b.options())
    T = b.num_tokens
    assert max_abs(out[:T], ref[:T]) <= 2e-2 * float(ref[:T].abs().max())


@pytest.mark.parametrize("d", [96, 192])
@pytest.mark.parametrize("hq,hkv,ps,sw,cap", [(8, 2, 16, None, None), (16, 4, 32, 40, 30.0), (12, 4, 8, None, None),
                                              (4, 4, 64, 100, None)])
def test_head_dim_96_and_192(d, hq, hkv, ps, sw, cap):
    # head_dim that is not a multiple of 64: decode at its own width, prefill at the next multiple
    # of 128 with the tensor maps' zero fill past the row (G = 3 takes the per-thread Q rows)
    b = workloads.make_rpa([1, 1, 3, 40, 130, 2], [1, 700, 64, 40, 300, 77], num_q_heads=hq, num_kv_heads=hkv,
                           head_dim=d, page_size=ps, seed=d + hq + ps, max_num_seqs=8, max_num_tokens=200,
                           extra_pages=2, sliding_window=sw, soft_cap=cap)
    check(b, TOL_BF16)


def test_head_dim_96_update_then_attend():
    b = workloads.make_rpa([1, 5, 33], [90, 5, 200], num_q_heads=8, num_kv_heads=2, head_dim=96, page_size=16,
                           seed=97, extra_pages=2)
    T = b.num_tokens
    rng = np.random.default_rng(98)
    nk = torch.from_numpy(rng.standard_normal((b.q.shape[0], 2, 96), dtype=np.float32)).to(torch.bfloat16)
    nv = torch.from_numpy(rng.standard_normal((b.q.shape[0], 2, 96), dtype=np.float32)).to(torch.bfloat16)
    kv_ref = oracle.rpa_update_kv_cache(nk, nv, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens))
    g = b.to("cuda")
    out = api.rpa_forward_update(g.q, nk.cuda(), nv.cuda(), g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens,
                                 g.num_seqs, **b.options())
    torch.cuda.synchronize()
    assert torch.equal(g.kv_pages.cpu().view(torch.int16), kv_ref.view(torch.int16))
    ref = oracle.rpa(b.q, kv_ref, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens), **b.options())
    assert max_abs(out[:T], ref[:T]) <= TOL_BF16


def test_head_dim_96_refuses_what_its_prefill_cannot_run():
    b = workloads.make_rpa([1, 9], [40, 30], num_q_heads=8, num_kv_heads=2, head_dim=96, page_size=16, seed=99,
                           kv_dtype=torch.float8_e4m3fn)
    g = b.to("cuda")
    with pytest.raises(api.RpaError, match="RPA_ERR_UNSUPPORTED"):
        api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, **b.options())
