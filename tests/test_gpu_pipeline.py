"""GPU: the host-memory pipeline (head groups copied in, computed and copied
out on overlapping streams) gives bitwise the result of the same kernels on
whole device tensors; its 2-D copy helper moves head slices exactly."""
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


def test_copy_2d_head_slices():
    gen = torch.Generator().manual_seed(3)
    host = torch.randn((300, 7, 128), generator=gen).to(torch.bfloat16).pin_memory()
    dev = torch.full((300, 7, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    h3.copy_2d(dev[:, 2:5], host[:, 2:5])
    back = torch.zeros_like(host).pin_memory()
    h3.copy_2d(back[:, 2:5], dev[:, 2:5])
    torch.cuda.synchronize()
    assert torch.equal(dev[:, 2:5].cpu().view(torch.int16), host[:, 2:5].view(torch.int16))
    assert torch.isnan(dev[:, :2].float()).all() and torch.isnan(dev[:, 5:].float()).all()
    assert torch.equal(back[:, 2:5].view(torch.int16), host[:, 2:5].view(torch.int16))
    assert (back[:, :2] == 0).all() and (back[:, 5:] == 0).all()


PIPE_CASES = [
    ("medium", 6), ("medium", 5), ("medium", 42), ("medium", 1),
    (W.custom("two_seq", 9, [W.Segment(700, 700, 650, (2, 10, 15), 250, 100),
                             W.Segment(520, 520, 520, (1, 20, 20), 100, 20)]), 4),
]


@pytest.mark.parametrize("wl,group", PIPE_CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_host_pipeline_is_bitwise_the_device_path(wl, group):
    w = W.workload(wl) if isinstance(wl, str) else wl
    g = W.make_inputs(w, device="cuda", fill="B")
    host = {n: g[n].cpu().pin_memory() for n in ("q", "k", "v", "wq", "wk", "pos_thw")}
    ref = h3.attention_block(g["q"].clone(), g["k"].clone(), g["v"], g["wq"], g["wk"], g["pos_thw"],
                             g["cu_seqlens_q"], g["valid_len"], scale=SCALE)
    pipe = h3.HostPipeline(w.q_rows, w.n_heads, heads_per_group=group)
    out = torch.full(ref.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    for _ in range(2):  # the second run reuses the device buffers
        pipe.run(host["q"], host["k"], host["v"], host["wq"], host["wk"], host["pos_thw"],
                 g["cu_seqlens_q"], g["valid_len"], out, scale=SCALE)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16))
    # the host inputs are untouched (the prologue works on the device copies)
    assert torch.equal(host["q"].view(torch.int16), g["q"].cpu().view(torch.int16))


def test_host_pipeline_explicit_group_sizes():
    w = W.workload("medium")
    g = W.make_inputs(w, device="cuda")
    host = {n: g[n].cpu().pin_memory() for n in ("q", "k", "v", "wq", "wk", "pos_thw")}
    ref = h3.attention_block(g["q"].clone(), g["k"].clone(), g["v"], g["wq"], g["wk"], g["pos_thw"],
                             g["cu_seqlens_q"], g["valid_len"], scale=SCALE)
    pipe = h3.HostPipeline(w.q_rows, w.n_heads, group_sizes=[1, 20, 2, 19])
    assert pipe.groups == [(0, 1), (1, 21), (21, 23), (23, 42)]
    out = torch.full(ref.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    pipe.run(host["q"], host["k"], host["v"], host["wq"], host["wk"], host["pos_thw"],
             g["cu_seqlens_q"], g["valid_len"], out, scale=SCALE)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16))


def test_host_pipeline_attention_only_grouped():
    w = W.custom("grp", 5, [W.Segment(64, 64), W.Segment(200, 900), W.Segment(333, 1500)],
                 self_attention=False)
    g = W.make_inputs(w, device="cuda")
    ref = h3.attention(g["q"], g["k"], g["v"], g["cu_seqlens_q"], g["cu_seqlens_kv"], None, SCALE)
    host = {n: g[n].cpu().pin_memory() for n in ("q", "k", "v")}
    pipe = h3.HostPipeline(w.q_rows, w.n_heads, heads_per_group=2, kv_rows=w.kv_rows)
    out = torch.full(ref.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    pipe.run_attention(host["q"], host["k"], host["v"], g["cu_seqlens_q"], g["cu_seqlens_kv"], None,
                       out, scale=SCALE)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16))
