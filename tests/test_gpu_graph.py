"""GPU: the entry points are CUDA-graph capturable (their host arguments and
tensor maps are consumed at capture time) and a replayed graph gives bitwise
the eager result, also after the inputs were overwritten in place."""
import pytest
import torch

import packed_sequence_attention_gb300 as h3
from packed_sequence_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu
SCALE = 128 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    h3.lib()
    yield
    assert h3.status_word() == 0


def _eager(g, q, k):
    qq, kk = q.clone(), k.clone()
    return h3.attention_block(qq, kk, g["v"], g["wq"], g["wk"], g["pos_thw"], g["cu_seqlens_q"],
                              g["valid_len"], scale=SCALE)


@pytest.mark.parametrize("name", ["medium", "stage1_batch2"])
def test_block_step_graph_replay_is_bitwise_eager(name):
    w = W.workload(name)
    g = W.make_inputs(w, device="cuda")
    q0, k0 = g["q"].clone(), g["k"].clone()
    ref = _eager(g, q0, k0)
    q, k = q0.clone(), k0.clone()
    out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture (sets kernel attributes once)
        h3.attention_block(q, k, g["v"], g["wq"], g["wk"], g["pos_thw"], g["cu_seqlens_q"],
                           g["valid_len"], scale=SCALE, out=out)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        h3.attention_block(q, k, g["v"], g["wq"], g["wk"], g["pos_thw"], g["cu_seqlens_q"],
                           g["valid_len"], scale=SCALE, out=out)
    for trial in range(2):  # fresh inputs copied in place, then replay
        gen = torch.Generator(device="cuda").manual_seed(100 + trial)
        q0 = torch.randn(q0.shape, generator=gen, device="cuda").to(torch.bfloat16)
        k0 = torch.randn(k0.shape, generator=gen, device="cuda").to(torch.bfloat16)
        q.copy_(q0)
        k.copy_(k0)
        out.fill_(float("nan"))
        graph.replay()
        ref = _eager(g, q0, k0)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_sparse_stages_graph_replay():
    g = W.make_inputs("medium", device="cuda")
    n = 4000
    ref, _, _ = h3.sol_attention(g["q"], g["k"], g["v"], n, 1.0, 300, SCALE)
    out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        h3.sol_attention(g["q"], g["k"], g["v"], n, 1.0, 300, SCALE, out=out)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        h3.sol_attention(g["q"], g["k"], g["v"], n, 1.0, 300, SCALE, out=out)
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out[:n].view(torch.int16), ref[:n].view(torch.int16))
