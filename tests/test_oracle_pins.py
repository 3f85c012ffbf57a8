"""Pins for the float64 oracle: brute force, closed forms, invariants, goldens.

Each check ties the oracle to something other than itself: dense unpaged
attention built with numpy matrix ops from contiguous K/V (the tests page the
data themselves with their own permutation), values the number formats fix,
hand-worked examples under ``tests/golden/``, and identities the method must
satisfy.  A plausible mistake in the oracle -- a dropped rope term, a wrong
page or slot index, GQA mapping, mask sign or window bound, add-vs-replace of
the mask value, an un-rounded dequant -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
MASK = oracle.DEFAULT_MASK_VALUE


# ---------------------------------------------------------------------------
# test-side paging and dense attention (independent of the oracle)
# ---------------------------------------------------------------------------

def page_rpa(K_list, V_list, page_size, rng, extra_pages=3, dtype=torch.bfloat16):
    """Dense per-sequence K/V [kv_len, Hkv, D] -> kv_pages [P, ps, 2Hkv, D] + table."""
    Hkv, D = K_list[0].shape[1:]
    need = [-(-k.shape[0] // page_size) for k in K_list]
    P = sum(need) + extra_pages
    perm = rng.permutation(P)
    pps = max(need)
    table = np.full((len(K_list), pps), 2**31 - 1, dtype=np.int32)
    pages = torch.full((P, page_size, 2 * Hkv, D), float("nan")).to(dtype)
    off = 0
    for s, (K, V) in enumerate(zip(K_list, V_list)):
        for lp in range(need[s]):
            phys = int(perm[off + lp])
            table[s, lp] = phys
            lo, hi = lp * page_size, min(K.shape[0], (lp + 1) * page_size)
            for g in range(Hkv):
                pages[phys, :hi - lo, 2 * g] = K[lo:hi, g]
                pages[phys, :hi - lo, 2 * g + 1] = V[lo:hi, g]
        off += need[s]
    return pages, torch.from_numpy(table)


def dense_attention(q, K, V, q_pos, sm_scale, soft_cap=None, sw=None, mask_value=MASK, mode="add"):
    """q [n, H, D]; K, V [kv, H, D] float64 (heads already repeated)."""
    s = np.einsum("qhd,khd->hqk", q, K) * sm_scale
    if soft_cap:
        s = soft_cap * np.tanh(s / soft_cap)
    kpos = np.arange(K.shape[0])
    mask = q_pos[:, None] < kpos[None, :]
    if sw:
        mask |= (q_pos[:, None] - sw) >= kpos[None, :]
    if mode == "add":
        s = s + np.where(mask, mask_value, 0.0)[None]
    else:
        s = np.where(mask[None], mask_value, s)
    p = scipy.special.softmax(s, axis=-1)
    return np.einsum("hqk,khd->qhd", p, V)


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def rand_bf16(rng, shape):
    return bf16(rng.standard_normal(shape))


def pack_int4(x):
    """int values in [-8, 7] [..., D] -> uint8 [..., D / 2]: element 2i in the low nibble of
    byte i, element 2i+1 in the high nibble (two's complement in each nibble)."""
    u = (x.to(torch.int16) & 15).to(torch.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).contiguous()


def ragged_case(rng, q_lens, kv_lens, Hq, Hkv, D, ps, sm_scale=None, sw=None, soft_cap=None,
                dtype=torch.bfloat16, scale=None, mask_value=MASK):
    if dtype == torch.int8:  # the full two's-complement range
        K_list = [torch.from_numpy(rng.integers(-128, 128, size=(k, Hkv, D)).astype(np.int8)) for k in kv_lens]
        V_list = [torch.from_numpy(rng.integers(-128, 128, size=(k, Hkv, D)).astype(np.int8)) for k in kv_lens]
    elif dtype == "int4":  # the full 4-bit range, held as int8 values on the dense side
        K_list = [torch.from_numpy(rng.integers(-8, 8, size=(k, Hkv, D)).astype(np.int8)) for k in kv_lens]
        V_list = [torch.from_numpy(rng.integers(-8, 8, size=(k, Hkv, D)).astype(np.int8)) for k in kv_lens]
    else:
        K_list = [rand_bf16(rng, (k, Hkv, D)).to(dtype) for k in kv_lens]
        V_list = [rand_bf16(rng, (k, Hkv, D)).to(dtype) for k in kv_lens]
    T = sum(q_lens)
    q = rand_bf16(rng, (T, Hq, D))
    if dtype == "int4":
        pages, table = page_rpa(K_list, V_list, ps, rng, dtype=torch.int8)
        pages = pack_int4(pages)  # the oracle reads the packed bytes
    else:
        pages, table = page_rpa(K_list, V_list, ps, rng, dtype=dtype)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    kvl = torch.tensor(kv_lens, dtype=torch.int32)
    sm_scale = 1 / math.sqrt(D) if sm_scale is None else sm_scale
    out = oracle.rpa(q, pages, kvl, table, cu, len(q_lens), sm_scale=sm_scale, sliding_window=sw,
                     soft_cap=soft_cap, k_scale=scale, v_scale=scale, mask_value=mask_value)
    # dense side
    expect = []
    G = Hq // Hkv
    for s in range(len(q_lens)):
        Kd = K_list[s].to(torch.float64)
        Vd = V_list[s].to(torch.float64)
        if scale is not None:  # the reference: float32 product rounded to bf16
            Kd = (K_list[s].to(torch.float32) * scale).to(torch.bfloat16).to(torch.float64)
            Vd = (V_list[s].to(torch.float32) * scale).to(torch.bfloat16).to(torch.float64)
        Kd = np.repeat(Kd.numpy(), G, axis=1)
        Vd = np.repeat(Vd.numpy(), G, axis=1)
        qs = q[cu[s]:cu[s + 1]].to(torch.float64).numpy()
        q_pos = kv_lens[s] - q_lens[s] + np.arange(q_lens[s])
        expect.append(dense_attention(qs, Kd, Vd, q_pos, sm_scale, soft_cap, sw, mask_value))
    return out.numpy(), np.concatenate(expect, axis=0), (q, pages, kvl, table, cu, K_list, V_list)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_bf16_decode_all_codes():
    codes = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_bf16(c) for c in range(0, 65536, 1)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_e4m3_decode_all_codes_and_golden():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.decode_e4m3(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    gold = json.load(open(os.path.join(GOLD, "e4m3_values.json")))
    for code, val in gold["values"]:
        v = oracle.decode_e4m3(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == val and math.copysign(1, v) == math.copysign(1, val)


def test_f32_to_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                         np.float32([1 + 2**-8, 1 + 3 * 2**-8, -1 - 2**-8, 3.0e38, 1e-40, 0.0])])
    ref = torch.from_numpy(xs).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_f32_to_bf16(float(x)) for x in xs])
    np.testing.assert_array_equal(got, ref)
    assert oracle.round_f32_to_bf16(1 + 2**-8) == 1.0           # tie to even (down)
    assert oracle.round_f32_to_bf16(1 + 3 * 2**-8) == 1 + 2**-6  # tie to even (up)


# ---------------------------------------------------------------------------
# standard RPA
# ---------------------------------------------------------------------------

def test_rpa_golden_two_keys():
    g = json.load(open(os.path.join(GOLD, "rpa_two_keys.json")))
    ps, P = g["page_size"], g["total_num_pages"]
    K, V = np.array(g["K"], dtype=np.float32), np.array(g["V"], dtype=np.float32)
    pages = torch.full((P, ps, 2, 4), float("nan")).to(torch.bfloat16)
    table = g["page_table"]
    for k in range(3):
        pages[table[0][k // ps], k % ps, 0] = bf16(K[k])
        pages[table[0][k // ps], k % ps, 1] = bf16(V[k])
    out = oracle.rpa(bf16(g["q"]), pages, [3], torch.tensor(table, dtype=torch.int32), [0, 2], 1,
                     sm_scale=g["sm_scale"])
    np.testing.assert_allclose(out.numpy(), np.array(g["expected"]), rtol=0, atol=1e-15)


@pytest.mark.parametrize("ps", [1, 2, 16])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (4, 4), (8, 1)])
def test_rpa_matches_dense_bruteforce(ps, Hq, Hkv):
    rng = np.random.default_rng(ps * 100 + Hq * 10 + Hkv)
    out, exp, _ = ragged_case(rng, [1, 1, 5, 0, 3], [17, 40, 64, 3, 3], Hq, Hkv, 32, ps)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-12)


def test_rpa_window_softcap_bruteforce():
    rng = np.random.default_rng(7)
    out, exp, _ = ragged_case(rng, [1, 6, 4], [30, 25, 9], 4, 2, 16, 4, sw=5, soft_cap=0.7)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-12)


def test_int8_decode_all_codes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.int8).to(torch.float64).numpy()
    got = np.array([oracle.decode_int8(c) for c in range(256)])
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("scale,sm_scale", [(None, 0.002), (1 / 64, None), (0.0123, None)])
def test_rpa_int8_bruteforce(scale, sm_scale):
    # int8 K/V: promoted exactly without a scale, else bf16(float32(x) * scale) (torch's casts)
    rng = np.random.default_rng(21)
    out, exp, _ = ragged_case(rng, [1, 3], [20, 11], 4, 2, 16, 8, dtype=torch.int8, scale=scale, sm_scale=sm_scale)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-10)


def test_int4_decode_all_codes():
    # two's complement in four bits, decoded from the definition
    assert [oracle.decode_int4(n) for n in range(16)] == [float(n if n < 8 else n - 16) for n in range(16)]


@pytest.mark.parametrize("scale,sm_scale", [(None, 0.02), (1 / 8, None), (0.0123, 0.9)])
def test_rpa_int4_bruteforce(scale, sm_scale):
    # int4 K/V unpacked on the dense side by the test's own nibble order: promoted exactly
    # without a scale, else bf16(float32(x) * scale)
    rng = np.random.default_rng(23)
    out, exp, _ = ragged_case(rng, [1, 3, 2], [20, 11, 40], 4, 2, 16, 8, dtype="int4", scale=scale, sm_scale=sm_scale)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-10)


def test_int4_one_key_returns_its_value_in_element_order():
    # a single key returns its value row exactly; the value's nibbles all differ, so a swapped
    # nibble order or byte order shows in the output's element order
    D = 16
    v = torch.tensor([[-8, 7, 1, -1, 2, -2, 3, -3, 4, -4, 5, -5, 6, -6, 0, -7]], dtype=torch.int8)
    k = torch.zeros(1, D, dtype=torch.int8)
    pages = torch.zeros(2, 4, 2, D // 2, dtype=torch.uint8)
    pages[1, 0, 0] = pack_int4(k)[0]
    pages[1, 0, 1] = pack_int4(v)[0]
    q = bf16(np.ones((1, 1, D)))
    out = oracle.rpa(q, pages, torch.tensor([1], dtype=torch.int32), torch.tensor([[1]], dtype=torch.int32),
                     torch.tensor([0, 1], dtype=torch.int32), 1, sm_scale=0.5)
    np.testing.assert_array_equal(out[0, 0].numpy(), v[0].double().numpy())


def test_rpa_fp8_scaled_bruteforce():
    rng = np.random.default_rng(8)
    out, exp, _ = ragged_case(rng, [1, 3], [20, 11], 4, 2, 16, 8, dtype=torch.float8_e4m3fn, scale=0.37)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-12)


def test_rpa_mask_value_is_added():
    # a mild mask value leaks weight onto masked keys; the reference adds it
    rng = np.random.default_rng(9)
    out, exp, _ = ragged_case(rng, [3], [6], 2, 1, 8, 2, mask_value=-1.5)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-12)
    # and the default mask value gives zero weight to masked keys
    out2, exp2, _ = ragged_case(np.random.default_rng(9), [3], [6], 2, 1, 8, 2)
    assert np.abs(out - out2).max() > 1e-3


def test_rpa_single_key_returns_value():
    rng = np.random.default_rng(10)
    out, _, (q, pages, kvl, table, cu, K_list, V_list) = ragged_case(rng, [1], [1], 4, 2, 32, 16)
    V = V_list[0].to(torch.float64).numpy()  # [1, Hkv, D]
    np.testing.assert_array_equal(out[0], np.repeat(V[0], 2, axis=0))


@pytest.mark.parametrize("sw", [None, 7])
def test_rpa_zero_query_is_mean_of_visible_values(sw):
    rng = np.random.default_rng(11)
    q_lens, kv_lens = [1, 4], [30, 20]
    _, _, (q, pages, kvl, table, cu, K_list, V_list) = ragged_case(rng, q_lens, kv_lens, 4, 2, 16, 4)
    q0 = torch.zeros_like(q)
    out = oracle.rpa(q0, pages, kvl, table, cu, 2, sm_scale=0.25, sliding_window=sw).numpy()
    row = 0
    for s in range(2):
        V = V_list[s].to(torch.float64).numpy()
        for j in range(q_lens[s]):
            qp = kv_lens[s] - q_lens[s] + j
            lo = 0 if sw is None else max(0, qp - sw + 1)
            mean = V[lo:qp + 1].mean(axis=0)  # [Hkv, D]
            np.testing.assert_allclose(out[row], np.repeat(mean, 2, axis=0), rtol=0, atol=1e-14)
            row += 1


def test_rpa_zero_scale_is_mean():
    rng = np.random.default_rng(12)
    _, _, (q, pages, kvl, table, cu, K_list, V_list) = ragged_case(rng, [2], [9], 2, 1, 8, 4)
    out = oracle.rpa(q, pages, kvl, table, cu, 1, sm_scale=0.0).numpy()
    V = V_list[0].to(torch.float64).numpy()
    np.testing.assert_allclose(out[1], np.repeat(V.mean(axis=0), 2, axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(out[0], np.repeat(V[:8].mean(axis=0), 2, axis=0), rtol=0, atol=1e-14)


def test_rpa_huge_cap_and_wide_window_are_no_ops():
    rng = np.random.default_rng(13)
    _, _, (q, pages, kvl, table, cu, _, _) = ragged_case(rng, [1, 5], [33, 12], 4, 2, 16, 4)
    base = oracle.rpa(q, pages, kvl, table, cu, 2, sm_scale=0.3).numpy()
    cap = oracle.rpa(q, pages, kvl, table, cu, 2, sm_scale=0.3, soft_cap=1e30).numpy()
    win = oracle.rpa(q, pages, kvl, table, cu, 2, sm_scale=0.3, sliding_window=33).numpy()
    np.testing.assert_allclose(cap, base, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(win, base)


def test_rpa_page_permutation_invariance_is_exact():
    rng = np.random.default_rng(14)
    _, _, (q, pages, kvl, table, cu, _, _) = ragged_case(rng, [1, 4, 2], [19, 23, 5], 4, 2, 16, 4)
    base = oracle.rpa(q, pages, kvl, table, cu, 3, sm_scale=0.2).numpy()
    P = pages.shape[0]
    perm = torch.from_numpy(rng.permutation(P))          # new slot of each old page
    new_pages = torch.empty_like(pages)
    new_pages[perm] = pages
    t = table.clone()
    ok = t < P
    t[ok] = perm[t[ok].long()].to(torch.int32)
    got = oracle.rpa(q, new_pages, kvl, t, cu, 3, sm_scale=0.2).numpy()
    np.testing.assert_array_equal(got, base)


def test_rpa_gqa_equals_mha_with_repeated_heads():
    rng = np.random.default_rng(15)
    Hq, Hkv, D, ps = 8, 2, 16, 4
    _, _, (q, pages, kvl, table, cu, K_list, V_list) = ragged_case(rng, [2, 1], [10, 7], Hq, Hkv, D, ps)
    gqa = oracle.rpa(q, pages, kvl, table, cu, 2, sm_scale=0.3).numpy()
    G = Hq // Hkv
    Kr = [k.repeat_interleave(G, dim=1) for k in K_list]
    Vr = [v.repeat_interleave(G, dim=1) for v in V_list]
    pages2, table2 = page_rpa(Kr, Vr, ps, rng)
    mha = oracle.rpa(q, pages2, kvl, table2, cu, 2, sm_scale=0.3).numpy()
    np.testing.assert_array_equal(gqa, mha)


def test_rpa_batch_equals_per_sequence_calls():
    rng = np.random.default_rng(16)
    q_lens, kv_lens = [1, 3, 2], [12, 9, 30]
    _, _, (q, pages, kvl, table, cu, _, _) = ragged_case(rng, q_lens, kv_lens, 4, 2, 8, 4)
    whole = oracle.rpa(q, pages, kvl, table, cu, 3, sm_scale=0.5).numpy()
    for s in range(3):
        qs = q[cu[s]:cu[s + 1]].contiguous()
        one = oracle.rpa(qs, pages, kvl[s:s + 1], table[s:s + 1], [0, q_lens[s]], 1, sm_scale=0.5).numpy()
        np.testing.assert_array_equal(one, whole[cu[s]:cu[s + 1]])


def test_rpa_padding_rows_and_unused_metadata_untouched():
    rng = np.random.default_rng(17)
    _, _, (q, pages, kvl, table, cu, _, _) = ragged_case(rng, [1, 2], [5, 6], 2, 1, 8, 4)
    qpad = torch.cat([q, torch.full((3, 2, 8), float("nan")).to(torch.bfloat16)])
    kvl2 = torch.cat([kvl, torch.tensor([10**9], dtype=torch.int32)])
    table2 = torch.cat([table, torch.full((1, table.shape[1]), 2**31 - 1, dtype=torch.int32)])
    cu2 = torch.cat([cu, torch.tensor([-5], dtype=torch.int32)])
    out = oracle.rpa(qpad, pages, kvl2, table2, cu2, 2, sm_scale=0.4).numpy()
    base = oracle.rpa(q, pages, kvl, table, cu, 2, sm_scale=0.4).numpy()
    np.testing.assert_array_equal(out[:3], base)
    assert np.isnan(out[3:]).all()


def test_rpa_rejects_bad_metadata():
    rng = np.random.default_rng(18)
    _, _, (q, pages, kvl, table, cu, _, _) = ragged_case(rng, [2], [5], 2, 1, 8, 4)
    with pytest.raises(oracle.OracleError):
        oracle.rpa(q, pages, torch.tensor([1], dtype=torch.int32), table, cu, 1)  # q_len > kv_len
    bad = table.clone()
    bad[0, 0] = pages.shape[0]
    with pytest.raises(oracle.OracleError):
        oracle.rpa(q, pages, kvl, bad, cu, 1)


# ---------------------------------------------------------------------------
# RPA cache update
# ---------------------------------------------------------------------------

def test_rpa_update_then_attend_equals_dense():
    rng = np.random.default_rng(20)
    Hq, Hkv, D, ps = 4, 2, 16, 4
    q_lens, kv_lens = [1, 5, 3], [9, 5, 14]
    full_K = [rand_bf16(rng, (k, Hkv, D)) for k in kv_lens]
    full_V = [rand_bf16(rng, (k, Hkv, D)) for k in kv_lens]
    # the cache holds only the old prefix; the new tokens arrive as new_k/new_v
    old_K = [torch.cat([k[:k.shape[0] - ql], torch.full((ql, Hkv, D), float("nan")).to(torch.bfloat16)])
             for k, ql in zip(full_K, q_lens)]
    old_V = [torch.cat([v[:v.shape[0] - ql], torch.full((ql, Hkv, D), float("nan")).to(torch.bfloat16)])
             for v, ql in zip(full_V, q_lens)]
    pages, table = page_rpa(old_K, old_V, ps, rng)
    new_k = torch.cat([k[k.shape[0] - ql:] for k, ql in zip(full_K, q_lens)])
    new_v = torch.cat([v[v.shape[0] - ql:] for v, ql in zip(full_V, q_lens)])
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    kvl = torch.tensor(kv_lens, dtype=torch.int32)
    upd = oracle.rpa_update_kv_cache(new_k, new_v, pages, kvl, table, cu, 3)
    ref_pages, ref_table = page_rpa(full_K, full_V, ps, np.random.default_rng(20 + 1))
    q = rand_bf16(rng, (sum(q_lens), Hq, D))
    a = oracle.rpa(q, upd, kvl, table, cu, 3, sm_scale=0.25).numpy()
    b = oracle.rpa(q, ref_pages, kvl, ref_table, cu, 3, sm_scale=0.25).numpy()
    np.testing.assert_array_equal(a, b)
    # every byte outside the written slots is unchanged
    changed = (upd.view(torch.int16) != pages.view(torch.int16)).any(dim=-1)  # [P, ps, C]
    written = torch.zeros_like(changed)
    for s in range(3):
        for j in range(q_lens[s]):
            pos = kv_lens[s] - q_lens[s] + j
            written[table[s, pos // ps], pos % ps] = True
    assert not (changed & ~written).any()


# ---------------------------------------------------------------------------
# MLA
# ---------------------------------------------------------------------------

def page_mla(C_list, R_list, ps, pk, rng, lkv_pad, r_pad, extra_pages=2):
    need = [-(-c.shape[0] // ps) for c in C_list]
    P = sum(need) + extra_pages
    perm = rng.permutation(P)
    pps = max(need)
    table = np.full(len(C_list) * pps, 2**31 - 1, dtype=np.int32)
    ckv = torch.full((P, ps, lkv_pad), float("nan")).to(torch.bfloat16)
    ckpe = torch.full((P, ps, r_pad), float("nan")).to(torch.bfloat16)
    off = 0
    for s, (c, r) in enumerate(zip(C_list, R_list)):
        for lp in range(need[s]):
            phys = int(perm[off + lp])
            table[s * pps + lp] = phys
            lo, hi = lp * ps, min(c.shape[0], (lp + 1) * ps)
            ckv[phys, :hi - lo] = 0
            ckpe[phys, :hi - lo] = 0
            ckv[phys, :hi - lo, :c.shape[1]] = c[lo:hi]
            ckpe[phys, :hi - lo, :r.shape[1]] = r[lo:hi]
        off += need[s]
    return (ckv.reshape(P, ps // pk, pk, lkv_pad), ckpe.reshape(P, ps // pk, pk, r_pad),
            torch.from_numpy(table))


def mla_case(rng, q_lens, kv_lens, H=4, L=32, R=8, ps=8, pk=2, zero_rope=False):
    C_list = [rand_bf16(rng, (k, L)) for k in kv_lens]
    R_list = [rand_bf16(rng, (k, R)) for k in kv_lens]
    ckv, ckpe, table = page_mla(C_list, R_list, ps, pk, rng, -(-L // 128) * 128, -(-R // 128) * 128)
    T = sum(q_lens)
    ql = rand_bf16(rng, (T, H, L))
    qpe = torch.zeros((T, H, R), dtype=torch.bfloat16) if zero_rope else rand_bf16(rng, (T, H, R))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    kvl = torch.tensor(kv_lens, dtype=torch.int32)
    dist = torch.tensor([0, 0, len(q_lens)], dtype=torch.int32)
    return ql, qpe, ckv, ckpe, kvl, table, cu, dist, C_list, R_list


def test_mla_matches_dense_bruteforce():
    rng = np.random.default_rng(30)
    q_lens, kv_lens = [1, 4, 2], [20, 9, 13]
    ql, qpe, ckv, ckpe, kvl, table, cu, dist, C_list, R_list = mla_case(rng, q_lens, kv_lens)
    sm = 1 / math.sqrt(40)
    out = oracle.mla(ql, qpe, ckv, ckpe, kvl, table, cu, dist, sm_scale=sm).numpy()
    for s in range(3):
        K = torch.cat([C_list[s], R_list[s]], dim=1).to(torch.float64).numpy()[:, None, :]
        V = C_list[s].to(torch.float64).numpy()[:, None, :]
        qs = torch.cat([ql, qpe], dim=2)[cu[s]:cu[s + 1]].to(torch.float64).numpy()
        q_pos = kv_lens[s] - q_lens[s] + np.arange(q_lens[s])
        exp = dense_attention(qs, np.repeat(K, 4, axis=1), np.repeat(V, 4, axis=1), q_pos, sm, mode="replace")
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], exp, rtol=0, atol=1e-12)


@pytest.mark.parametrize("q_scale", [None, 0.5, 0.037])
def test_mla_fp8_queries_match_dense_bruteforce(q_scale):
    # fp8 e4m3 queries (torch's decode of the bytes, on the dense side) with the MLA kernel's
    # q_scale multiplying the scores after sm_scale
    rng = np.random.default_rng(33)
    q_lens, kv_lens = [1, 4], [20, 9]
    ql, qpe, ckv, ckpe, kvl, table, cu, dist, C_list, R_list = mla_case(rng, q_lens, kv_lens)
    ql8 = (ql.float() * 3).to(torch.float8_e4m3fn)
    qpe8 = (qpe.float() * 3).to(torch.float8_e4m3fn)
    sm = 1 / math.sqrt(40)
    out = oracle.mla(ql8, qpe8, ckv, ckpe, kvl, table, cu, dist, sm_scale=sm, q_scale=q_scale).numpy()
    for s in range(2):
        K = torch.cat([C_list[s], R_list[s]], dim=1).to(torch.float64).numpy()[:, None, :]
        V = C_list[s].to(torch.float64).numpy()[:, None, :]
        qs = torch.cat([ql8, qpe8], dim=2)[cu[s]:cu[s + 1]].to(torch.float64).numpy()
        q_pos = kv_lens[s] - q_lens[s] + np.arange(q_lens[s])
        exp = dense_attention(qs, np.repeat(K, 4, axis=1), np.repeat(V, 4, axis=1), q_pos, sm * (q_scale or 1.0),
                              mode="replace")
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], exp, rtol=0, atol=1e-12)


def test_mla_mask_value_replaces_logit():
    rng = np.random.default_rng(31)
    ql, qpe, ckv, ckpe, kvl, table, cu, dist, C_list, R_list = mla_case(rng, [3], [5], H=2)
    out = oracle.mla(ql, qpe, ckv, ckpe, kvl, table, cu, dist, sm_scale=0.3, mask_value=-0.5,
                     sliding_window=2, soft_cap=3.0).numpy()
    K = torch.cat([C_list[0], R_list[0]], dim=1).to(torch.float64).numpy()[:, None, :]
    V = C_list[0].to(torch.float64).numpy()[:, None, :]
    qs = torch.cat([ql, qpe], dim=2).to(torch.float64).numpy()
    exp = dense_attention(qs, np.repeat(K, 2, 1), np.repeat(V, 2, 1), np.array([2, 3, 4]), 0.3,
                          soft_cap=3.0, sw=2, mask_value=-0.5, mode="replace")
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-12)


def test_mla_zero_rope_reduces_to_mqa_rpa():
    rng = np.random.default_rng(32)
    q_lens, kv_lens = [1, 3], [17, 6]
    ql, qpe, ckv, ckpe, kvl, table, cu, dist, C_list, _ = mla_case(rng, q_lens, kv_lens, zero_rope=True)
    a = oracle.mla(ql, qpe, ckv, ckpe, kvl, table, cu, dist, sm_scale=0.2).numpy()
    # standard RPA with a single kv head whose key and value are both kv_c
    pages, t2 = page_rpa([c[:, None, :] for c in C_list], [c[:, None, :] for c in C_list], 4, rng)
    b = oracle.rpa(ql, pages, kvl, t2, cu, 2, sm_scale=0.2).numpy()
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_mla_update_golden_slots():
    g = json.load(open(os.path.join(GOLD, "mla_update_slots.json")))
    ps, pk, P = g["page_size"], g["kv_packing"], g["total_num_pages"]
    L, R = 128, 64
    ckv = torch.zeros((P, ps // pk, pk, L), dtype=torch.bfloat16)
    ckpe = torch.full((P, ps // pk, pk, 128), 7.0).to(torch.bfloat16)
    T = 4
    nkv = torch.arange(T * L, dtype=torch.float32).reshape(T, L).to(torch.bfloat16) + 1
    nkpe = -torch.arange(T * R, dtype=torch.float32).reshape(T, R).to(torch.bfloat16) - 1
    c, r = oracle.mla_update_kv_cache(nkv, nkpe, ckv, ckpe, g["kv_lens"], g["page_indices"], g["cu_q_lens"],
                                      [0, 0, 2])
    seen = torch.zeros((P, ps // pk, pk), dtype=torch.bool)
    for t, (pg, row, col) in enumerate(g["expected_page_row_col"]):
        assert torch.equal(c[pg, row, col], nkv[t])
        assert torch.equal(r[pg, row, col, :R], nkpe[t])
        assert (r[pg, row, col, R:] == 0).all()
        seen[pg, row, col] = True
    assert torch.equal(c[~seen], ckv[~seen]) and torch.equal(r[~seen], ckpe[~seen])


def test_mla_update_then_attend_equals_dense():
    rng = np.random.default_rng(33)
    q_lens, kv_lens, H, L, R, ps = [1, 3], [10, 7], 2, 32, 8, 4
    C_full = [rand_bf16(rng, (k, L)) for k in kv_lens]
    R_full = [rand_bf16(rng, (k, R)) for k in kv_lens]
    nan = lambda n, w: torch.full((n, w), float("nan")).to(torch.bfloat16)  # noqa: E731
    C_old = [torch.cat([c[:-ql], nan(ql, L)]) for c, ql in zip(C_full, q_lens)]
    R_old = [torch.cat([r[:-ql], nan(ql, R)]) for r, ql in zip(R_full, q_lens)]
    ckv, ckpe, table = page_mla(C_old, R_old, ps, 2, rng, 128, 128)
    nkv = torch.cat([c[-ql:] for c, ql in zip(C_full, q_lens)])
    nkpe = torch.cat([r[-ql:] for r, ql in zip(R_full, q_lens)])
    cu = torch.tensor([0, 1, 4], dtype=torch.int32)
    kvl = torch.tensor(kv_lens, dtype=torch.int32)
    dist = torch.tensor([1, 2, 2], dtype=torch.int32)
    ql_, qpe = rand_bf16(rng, (4, H, L)), rand_bf16(rng, (4, H, R))
    out, c2, r2 = oracle.mla_forward(ql_, qpe, nkv, nkpe, ckv, ckpe, kvl, table, cu, dist, sm_scale=0.3)
    ckv_ref, ckpe_ref, table_ref = page_mla(C_full, R_full, ps, 2, np.random.default_rng(5), 128, 128)
    ref = oracle.mla(ql_, qpe, ckv_ref, ckpe_ref, kvl, table_ref, cu, dist, sm_scale=0.3)
    np.testing.assert_array_equal(out.numpy(), ref.numpy())


# ---------------------------------------------------------------------------
# DSA sparse MLA
# ---------------------------------------------------------------------------

def sparse_case(rng, B, S, T, H=4, Dk=40, Dv=32, ps=16, stride=48, extra_pages=2):
    lat = rand_bf16(rng, (B, T, Dk))
    max_pages = -(-T // ps)
    P = B * max_pages + extra_pages
    perm = rng.permutation(P)
    table = perm[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    cache = torch.full((P, ps, stride), float("nan")).to(torch.bfloat16)
    for b in range(B):
        for lp in range(max_pages):
            lo, hi = lp * ps, min(T, (lp + 1) * ps)
            cache[table[b, lp], :hi - lo] = 0
            cache[table[b, lp], :hi - lo, :Dk] = lat[b, lo:hi]
    q = rand_bf16(rng, (B, S, H, Dk))
    return lat, cache, torch.from_numpy(table), q


def sparse_dense(q, lat, keys_per_query, positions, T, sm, Dv):
    """Brute force: explicit token lists -> dense softmax per (b, s)."""
    B, S, H, _ = q.shape
    out = np.zeros((B, S, H, Dv))
    for b in range(B):
        for s in range(S):
            ks = [k for k in keys_per_query[b][s] if k <= positions[b, s] and k < T]
            if not ks:
                continue
            Kb = lat[b, ks].to(torch.float64).numpy()
            logits = q[b, s].to(torch.float64).numpy() @ Kb.T * sm
            p = scipy.special.softmax(logits, axis=-1)
            out[b, s] = p @ Kb[:, :Dv]
    return out


@pytest.mark.parametrize("RB", [1, 4, 16])
def test_sparse_matches_bruteforce(RB):
    rng = np.random.default_rng(40 + RB)
    B, S, T, K = 2, 3, 64, 6
    lat, cache, table, q = sparse_case(rng, B, S, T)
    pos = np.array([[10, 40, 63], [0, 5, 33]], dtype=np.int32)
    idx = rng.integers(-1, T // RB, size=(B, S, K)).astype(np.int32)
    keys = [[[u * RB + r for u in idx[b, s] if u >= 0 for r in range(RB)] for s in range(S)] for b in range(B)]
    out = oracle.sparse_mla(q, cache, idx, pos, table, read_block=RB, page_size=16, seq_len=T, sm_scale=0.2,
                            dv=32).numpy()
    np.testing.assert_allclose(out, sparse_dense(q, lat, keys, pos, T, 0.2, 32), rtol=0, atol=1e-12)


def test_sparse_all_units_equals_dense_mla():
    rng = np.random.default_rng(50)
    B, S, T, H, Dk, Dv, ps = 1, 4, 48, 4, 40, 32, 16
    lat, cache, table, q = sparse_case(rng, B, S, T, H=H, Dk=Dk, Dv=Dv, ps=ps)
    pos = np.array([[0, 17, 30, 47]], dtype=np.int32)
    for RB, K in [(1, T), (16, T // 16)]:
        idx = np.tile(np.arange(K, dtype=np.int32), (B, S, 1))
        out = oracle.sparse_mla(q, cache, idx, pos, table, read_block=RB, page_size=ps, seq_len=T,
                                sm_scale=0.15, dv=Dv).numpy()
        # dense MLA over the same latent: kv_c = first Dv cols, k_pe = the rest
        c = lat[0, :, :Dv].contiguous()
        r = lat[0, :, Dv:].contiguous()
        ckv, ckpe, t2 = page_mla([c], [r], ps, 2, rng, 128, 128)
        for s in range(S):
            qs = q[0, s:s + 1]
            m = oracle.mla(qs[:, :, :Dv].contiguous(), qs[:, :, Dv:].contiguous(), ckv, ckpe,
                           [int(pos[0, s]) + 1], t2, [0, 1], [0, 0, 1], sm_scale=0.15).numpy()
            np.testing.assert_allclose(out[0, s], m[0], rtol=0, atol=1e-12)


def test_sparse_empty_selection_is_zero_and_duplicates_count_twice():
    rng = np.random.default_rng(51)
    lat, cache, table, q = sparse_case(rng, 1, 2, 32)
    idx = np.array([[[-1, -1, -1], [3, 3, 9]]], dtype=np.int32)
    pos = np.array([[31, 31]], dtype=np.int32)
    out = oracle.sparse_mla(q, cache, idx, pos, table, read_block=1, page_size=16, seq_len=32,
                            sm_scale=0.3, dv=32).numpy()
    assert (out[0, 0] == 0).all()
    np.testing.assert_allclose(out, sparse_dense(q, lat, [[[], [3, 3, 9]]], pos, 32, 0.3, 32), atol=1e-12,
                               rtol=0)
    single = oracle.sparse_mla(q, cache, np.array([[[-1, -1, -1], [3, 9, -1]]], dtype=np.int32), pos, table,
                               read_block=1, page_size=16, seq_len=32, sm_scale=0.3, dv=32).numpy()
    assert np.abs(single[0, 1] - out[0, 1]).max() > 1e-6


def test_sparse_slot_permutation_and_future_units():
    rng = np.random.default_rng(52)
    lat, cache, table, q = sparse_case(rng, 1, 1, 64)
    pos = np.array([[20]], dtype=np.int32)
    idx = np.array([[[1, 4, 7, 30, 50]]], dtype=np.int32)  # 30 and 50 are in the future
    a = oracle.sparse_mla(q, cache, idx, pos, table, read_block=1, page_size=16, seq_len=64, sm_scale=0.3,
                          dv=32).numpy()
    b = oracle.sparse_mla(q, cache, idx[..., ::-1].copy(), pos, table, read_block=1, page_size=16, seq_len=64,
                          sm_scale=0.3, dv=32).numpy()
    c = oracle.sparse_mla(q, cache, np.array([[[1, 4, 7, -1, -1]]], dtype=np.int32), pos, table, read_block=1,
                          page_size=16, seq_len=64, sm_scale=0.3, dv=32).numpy()
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(a, c)


def test_sparse_unit_row_resolution_golden():
    # RB 16 in pages of 64: unit 5 = tokens 80..95 = logical page 1, offset 16
    rng = np.random.default_rng(53)
    lat, cache, table, q = sparse_case(rng, 1, 1, 128, ps=64)
    idx = np.array([[[5]]], dtype=np.int32)
    pos = np.array([[127]], dtype=np.int32)
    out = oracle.sparse_mla(q, cache, idx, pos, table, read_block=16, page_size=64, seq_len=128, sm_scale=0.1,
                            dv=32).numpy()
    flat = cache.reshape(-1, cache.shape[-1])
    rows = flat[int(table[0, 1]) * 64 + 16: int(table[0, 1]) * 64 + 32, :40].to(torch.float64).numpy()
    logits = q[0, 0].to(torch.float64).numpy() @ rows.T * 0.1
    exp = scipy.special.softmax(logits, axis=-1) @ rows[:, :32]
    np.testing.assert_allclose(out[0, 0], exp, rtol=0, atol=1e-12)
