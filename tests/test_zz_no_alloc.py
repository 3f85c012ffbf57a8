"""rpa_forward_noalloc: the entry point for callers that cannot allocate device memory.

Such callers (a plugin inside an application whose memory manager owns the GPU, or a
serving loop that may not call cudaMalloc once it runs) get rpa_forward without a
workspace: the library's fixed scratch array stands in for it.  These tests call it
through the C ABI and check that it returns exactly what rpa_forward returns on the
same inputs (the same plan and the same kernels run, only the scratch differs), on two
calls in a row (the second reuses the scratch the first left behind), and that a
problem too large for the array is refused before anything launches.
This file is collected last on purpose.
"""
import ctypes
import math
import re

import pytest
import torch

from ragged_paged_attention_gb300 import api, workloads


def _batches():
    return [
        workloads.llama_mixed(scale=1 / 4),
        # bf16 with a window and a soft cap, GQA 4
        workloads.make_rpa([1, 1, 7, 40], [900, 35, 64, 300], num_q_heads=16, num_kv_heads=4, head_dim=128,
                           page_size=16, seed=77, sliding_window=128, soft_cap=30.0),
        # the Gemma-2 options scaled down: fp8 e4m3 cache at head_dim 256, scales, window, cap
        workloads.gemma_options(scale=1 / 4),
        # int8 cache with power-of-two scales
        workloads.make_rpa([1, 3, 1, 33], [500, 77, 1300, 200], num_q_heads=8, num_kv_heads=2, head_dim=128,
                           page_size=16, seed=78, kv_dtype=torch.int8, k_scale=0.25, v_scale=0.5),
    ]


@pytest.mark.gpu
def test_noalloc_matches_rpa_forward_on_two_calls():
    for b in _batches():
        g = b.to("cuda")
        prm = api.make_rpa_params(g.q, g.kv_pages, g.page_indices, **b.options())
        # the problem fits the fixed array (else the call would be refused)
        assert api.rpa_workspace_size(prm) <= api.NOALLOC_SCRATCH_BYTES
        ref = api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, **b.options())
        T = b.num_tokens
        for _ in range(2):
            out = torch.full_like(g.q, 7.0)
            api.rpa_forward_noalloc(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, out=out,
                                    **b.options())
            torch.cuda.synchronize()
            assert torch.equal(out[:T].view(torch.int16), ref[:T].view(torch.int16))
            assert (out[T:].float() == 7.0).all()


def test_noalloc_rejects_problems_larger_than_its_scratch():
    lib = api.load_library()
    p = api.rpa_params(struct_size=ctypes.sizeof(api.rpa_params), version=1, max_num_tokens=1 << 20,
                       num_q_heads=64, num_combined_kv_heads=16, head_dim=256, total_num_pages=1 << 16,
                       page_size=16, max_num_seqs=1 << 14, pages_per_seq=64, q_dtype=1, kv_dtype=1, sm_scale=0.1,
                       sliding_window=0, soft_cap=0.0, mask_value=math.nan, k_scale=0.0, v_scale=0.0)
    n = ctypes.c_size_t(0)
    assert lib.rpa_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value > api.NOALLOC_SCRATCH_BYTES
    ptrs = [ctypes.c_void_p(256 * (i + 1)) for i in range(7)]
    assert lib.rpa_forward_noalloc(ctypes.byref(p), *ptrs, None) == -8
    msg = lib.rpa_last_error().decode()
    assert "static scratch" in msg
    # the size the library enforces is the one the binding reads from include/rpa.h
    need, have = (int(x) for x in re.search(r"need (\d+) bytes.*holds (\d+)", msg).groups())
    assert need == n.value and have == api.NOALLOC_SCRATCH_BYTES


def test_noalloc_binding_checks_shapes_before_calling():
    q = torch.zeros(8, 4, 128, dtype=torch.bfloat16)
    kv = torch.zeros(2, 16, 4, 128, dtype=torch.bfloat16)
    i32 = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="head_dim"):
        api.rpa_forward_noalloc(q[..., :64].contiguous(), kv, i32, i32, i32, i32, out=q[..., :64].contiguous())
    with pytest.raises(ValueError, match="shape"):
        api.rpa_forward_noalloc(q, kv, i32, i32, i32, i32, out=q[:4].contiguous())
