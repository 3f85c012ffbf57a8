"""Failure detection without a GPU fault: a bounded wait that runs out reports
RPA_DEV_ERR_TIMEOUT through the workspace's error word, and the context stays usable."""
import time

import pytest
import torch

import oracle
from ragged_paged_attention_gb300 import api, workloads
from parity import TOL_BF16, max_abs

pytestmark = pytest.mark.gpu

RPA_DEV_ERR_TIMEOUT = 0x40


def test_bounded_wait_reports_timeout_and_the_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.time()
    api.selftest_bounded_wait(ws)
    bits = api.check_device_status(ws)  # synchronises, reads and clears the word
    elapsed = time.time() - t0
    assert bits == RPA_DEV_ERR_TIMEOUT
    assert 1.5 < elapsed < 60  # the wait's 2 s limit, then the kernel returned
    assert api.check_device_status(ws) == 0  # cleared by the read
    # the same context still runs attention correctly
    b = workloads.tiny_rpa()
    g = b.to("cuda")
    out = api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, **b.options())
    torch.cuda.synchronize()
    ref = oracle.rpa(b.q, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens), **b.options())
    T = b.num_tokens
    assert max_abs(out[:T], ref[:T]) <= TOL_BF16
