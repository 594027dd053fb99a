"""GPU: row addressing beyond 2^31 elements (a regression category the
Sol-H3 page lists, section 6).  A 42-head tensor of 400,300 rows puts its
second sequence at row 400,000, element offset 400,000 x 5,376 > 2^31, and
both the prologue (called on the whole tensor) and attention address it
with in-kernel row arithmetic."""
import numpy as np
import pytest
import torch

import packed_sequence_attention_gb300 as h3
from oracle import oracle as O

pytestmark = pytest.mark.gpu
SCALE = 128 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    h3.lib()
    yield
    assert h3.status_word() == 0


def test_rows_past_2_pow_31_elements():
    H, r0, n = 42, 400_000, 300
    R = r0 + n
    assert r0 * H * 128 > 2 ** 31
    gen = torch.Generator(device="cuda").manual_seed(31)
    q, k, v = (torch.zeros((R, H, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    for t in (q, k, v):
        t[r0:] = torch.randn((n, H, 128), generator=gen, device="cuda").to(torch.bfloat16)
    wq = (1 + 0.1 * torch.randn((H, 128), generator=gen, device="cuda")).to(torch.bfloat16)
    wk = (1 + 0.1 * torch.randn((H, 128), generator=gen, device="cuda")).to(torch.bfloat16)
    pos = torch.zeros((R, 3), dtype=torch.int32, device="cuda")
    pos[r0:, 0] = torch.arange(n, dtype=torch.int32, device="cuda")
    q_in, k_in = q[r0:].cpu(), k[r0:].cpu()
    h3.qk_norm_rope(q, k, wq, wk, pos, n_rows=R)
    out = torch.full((R, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    h3.attention(q, k, v, [0, r0, R], [0, r0, R], [0, n], SCALE, out=out)
    torch.cuda.synchronize()
    p = pos[r0:].cpu().numpy()
    for x_in, x_gpu, w in ((q_in, q[r0:], wq), (k_in, k[r0:], wk)):
        ref = O.qk_norm_rope(O.widen(x_in), O.widen(w), p)
        assert np.abs(O.widen(x_gpu) - ref).max() <= 2e-2
    ref = O.attention(O.widen(q[r0:]), O.widen(k[r0:]), O.widen(v[r0:]), [0, n], [0, n], None, SCALE)
    got = O.widen(out[r0:])
    assert np.abs(got - ref).max() <= 2e-2
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3
    assert bool((out[:r0] == 0).all())  # the empty first sequence's rows are written as 0


def test_varlen_prologue_rows_past_2_pow_31_elements():
    # The same layout through the packed-sequence prologue: the second
    # sequence's first buffer row comes from the launch's sequence table.
    H, r0, n = 42, 400_000, 300
    R = r0 + n + 16
    gen = torch.Generator(device="cuda").manual_seed(32)
    q, k = (torch.full((R, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(2))
    for t in (q, k):
        t[r0:r0 + n] = torch.randn((n, H, 128), generator=gen, device="cuda").to(torch.bfloat16)
    wq = (1 + 0.1 * torch.randn((H, 128), generator=gen, device="cuda")).to(torch.bfloat16)
    wk = (1 + 0.1 * torch.randn((H, 128), generator=gen, device="cuda")).to(torch.bfloat16)
    pos = torch.randint(0, 1800, (R, 3), generator=gen, device="cuda", dtype=torch.int32)
    q_ref, k_ref = q[r0:r0 + n].clone(), k[r0:r0 + n].clone()
    h3.qk_norm_rope(q_ref, k_ref, wq, wk, pos[r0:], n_rows=n)
    h3.qk_norm_rope_varlen(q, k, wq, wk, pos, [0, r0, R], [0, n])
    torch.cuda.synchronize()
    fill = torch.full((1,), float("nan"), dtype=torch.bfloat16).view(torch.int16).item()
    for got, ref in ((q, q_ref), (k, k_ref)):
        assert torch.equal(got[r0:r0 + n].view(torch.int16), ref.view(torch.int16))
        bits = got.view(torch.int16)
        assert bool((bits[:r0] == fill).all())       # the empty sequence: untouched
        assert bool((bits[r0 + n:] == fill).all())   # past the valid rows: untouched
