"""GPU parity of the wire-format kernels: layout records bit-identical to the
torch permutations they replace, INT8 / FP8 records byte-identical to the
oracle's encoding, and decodes bit-identical to the oracle's decode."""
import numpy as np
import pytest
import torch

import packed_sequence_attention_gb300 as h3
from oracle import oracle as O
from packed_sequence_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    h3.lib()
    yield
    assert h3.status_word() == 0


def qkv(rows=300, H=6, packed=True, seed=0):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    if packed:
        buf = torch.randn((rows, 3, H, 128), generator=gen, device="cuda").to(torch.bfloat16)
        return buf[:, 0], buf[:, 1], buf[:, 2]
    return [torch.randn((rows, H, 128), generator=gen, device="cuda").to(torch.bfloat16)
            for _ in range(3)]


def as_bytes(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("n_dest", [1, 2, 3, 6])
def test_pack_qkv_bf16_is_the_permutation(n_dest):
    q, k, v = qkv()
    wire = h3.pack_qkv(q, k, v, n_dest, h3.WIRE_BF16)
    rows, H = q.shape[0], q.shape[1]
    ref = torch.stack([q, k, v], 2).reshape(rows, n_dest, H // n_dest, 3, 128) \
        .permute(1, 0, 2, 3, 4).contiguous()
    torch.cuda.synchronize()
    assert torch.equal(wire.view(torch.int16).view(ref.shape), ref.view(torch.int16))
    for d in range(n_dest):
        uq, uk, uv = h3.unpack_qkv(wire[d], h3.WIRE_BF16)
        hs = slice(d * H // n_dest, (d + 1) * H // n_dest)
        for a, b in ((uq, q), (uk, k), (uv, v)):
            assert torch.equal(a.view(torch.int16), b[:, hs].contiguous().view(torch.int16))


@pytest.mark.parametrize("n_dest", [1, 2])
def test_pack_qkv_int8_records_and_decode(n_dest):
    q, k, v = qkv(packed=False, seed=1)
    q[0, 0] = 0.0                     # an all-zero group
    k[1, 2, :32] *= 1000.0            # a wide group
    wire = h3.pack_qkv(q, k, v, n_dest, h3.WIRE_INT8)
    torch.cuda.synchronize()
    H = q.shape[1]
    hl = H // n_dest
    qq, kk, vv = O.widen(q), O.widen(k), O.widen(v)
    for d in range(n_dest):
        hs = slice(d * hl, (d + 1) * hl)
        ref = O.qkv_int8_records(qq[:, hs], kk[:, hs], vv[:, hs])
        assert np.array_equal(as_bytes(wire[d]), ref)
        uq, uk, uv = h3.unpack_qkv(wire[d], h3.WIRE_INT8)
        torch.cuda.synchronize()
        for t, got in enumerate((uq, uk, uv)):
            vals = ref[..., t * 128:(t + 1) * 128].view(np.int8)
            codes = ref[..., 384 + 4 * t:388 + 4 * t]
            dec = O.round_bf16(O.int8_group32_decode(vals, codes))
            assert np.array_equal(O.widen(got), dec)


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("n_src", [1, 3])
def test_output_records_and_head_merge(fmt, n_src):
    g = W.make_inputs("tiny", device="cuda")
    rows, H = 200, 6
    gen = torch.Generator(device="cuda").manual_seed(fmt * 10 + n_src)
    o = (torch.randn((rows, H, 128), generator=gen, device="cuda") * 3).to(torch.bfloat16)
    o[5, 1, 7] = 1000.0               # saturates in FP8
    hl = H // n_src
    parts = torch.stack([h3.pack_out(o[:, s * hl:(s + 1) * hl].contiguous(), fmt)
                         for s in range(n_src)])
    merged = h3.merge_heads(parts, fmt)
    torch.cuda.synchronize()
    oo = O.widen(o)
    if fmt == h3.WIRE_BF16:
        assert torch.equal(merged.view(torch.int16), o.view(torch.int16))
        return
    for s in range(n_src):
        x = oo[:, s * hl:(s + 1) * hl]
        ref = O.out_int8_records(x) if fmt == h3.WIRE_INT8 else O.out_fp8_records(x)
        assert np.array_equal(as_bytes(parts[s]), ref)
    if fmt == h3.WIRE_INT8:
        vals = np.stack([O.out_int8_records(oo[:, s * hl:(s + 1) * hl]) for s in range(n_src)])
        dec = np.concatenate([O.int8_group32_decode(vals[s, ..., :128].view(np.int8),
                                                    vals[s, ..., 128:132]) for s in range(n_src)], 1)
    else:
        dec = O.e4m3_round(oo)
    assert np.array_equal(O.widen(merged), O.round_bf16(dec))


def test_wire_record_sizes():
    assert [h3.wire_record_bytes("qkv", f) for f in (0, 1)] == [768, 400]
    assert [h3.wire_record_bytes("out", f) for f in (0, 1, 2)] == [256, 144, 128]
