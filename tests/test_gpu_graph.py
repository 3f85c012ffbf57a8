"""The library's calls captured in a CUDA graph: replays give the eager results bit for bit,
including after the inputs change in place (the RPA launches chain programmatically; the
capture keeps those dependencies)."""
import pytest
import torch

from ragged_paged_attention_gb300 import api, workloads

pytestmark = pytest.mark.gpu


def capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture (attributes, tensor maps)
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


@pytest.mark.parametrize("fused", [True, False], ids=["rpa_forward_update", "rpa_forward"])
def test_rpa_in_cuda_graph(fused):
    b = workloads.llama_mixed(scale=1 / 4)
    g = b.to("cuda")
    opts = b.options()
    ws = torch.zeros(api.rpa_workspace_size(api.make_rpa_params(g.q, g.kv_pages, g.page_indices, **opts)),
                     dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(g.q)

    def call():
        if fused:
            api.rpa_forward_update(g.q, g.new_k, g.new_v, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens,
                                   g.num_seqs, out=out, workspace=ws, **opts)
        else:
            api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, out=out,
                            workspace=ws, **opts)

    graph = capture(call)
    T = b.num_tokens
    for step in range(2):
        if step:  # new queries in place (a power-of-two factor: exact in bf16)
            g.q.mul_(0.5)
        call()
        torch.cuda.synchronize()
        eager = out[:T].clone()
        pages = g.kv_pages.clone()
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out[:T], eager)
        assert torch.equal(g.kv_pages.view(torch.uint8), pages.view(torch.uint8))
    assert api.check_device_status(ws) == 0


def test_mla_in_cuda_graph():
    m = workloads.mla_deepseek(scale=1 / 8)
    g = m.to("cuda")
    opts = m.options()
    prm = api.make_mla_params(g.ql_nope, g.q_pe, g.cache_kv_c, g.cache_k_pe, g.kv_lens, g.page_indices, **opts)
    ws = torch.zeros(api.mla_workspace_size(prm), dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(g.ql_nope)

    def call():
        api.mla_rpa_forward(g.ql_nope, g.q_pe, g.new_kv_c, g.new_k_pe, g.cache_kv_c, g.cache_k_pe, g.kv_lens,
                            g.page_indices, g.cu_q_lens, g.distribution, out=out, workspace=ws, **opts)

    graph = capture(call)
    call()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    T = int(m.cu_q_lens[int(m.distribution[2])])
    assert torch.equal(out[:T], eager[:T])
    assert api.check_device_status(ws) == 0


def test_sparse_in_cuda_graph():
    s = workloads.dsa_sparse(mode="token", phase="prefill", scale=1 / 16)
    g = s.to("cuda")
    prm = api.make_sparse_params(g.q, g.cache, g.indices, g.page_table, read_block=s.read_block,
                                 page_size=s.page_size, seq_len=s.seq_len, sm_scale=s.sm_scale)
    ws = torch.zeros(api.sparse_mla_workspace_size(prm), dtype=torch.uint8, device="cuda")
    out = torch.zeros(s.q.shape[:3] + (512,), dtype=torch.float32, device="cuda")

    def call():
        api.sparse_mla_forward(g.q, g.cache, g.indices, g.positions, g.page_table, out=out, workspace=ws,
                               **s.options())

    graph = capture(call)
    call()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert api.check_device_status(ws) == 0
