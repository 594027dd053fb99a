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


@pytest.mark.parametrize("n_dest,rows,H", [(1, 300, 6), (2, 300, 6), (3, 301, 6), (1, 301, 5),
                                           (5, 77, 5)])
def test_pack_qkv_int8_records_and_decode(n_dest, rows, H):
    # odd rows x heads leaves the last warp pass half full; hl odd makes a
    # warp's two units straddle destinations
    q, k, v = qkv(rows=rows, H=H, packed=False, seed=1)
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


def hard_int8_values(rows, H, seed):
    """bf16 [rows, H, 128] whose 32-value groups stress the INT8 encoder:
    exact half-integer quotients x / value(c) (rounding ties) at every scale
    code, groups whose max sits exactly on 127 * value(c), values past the
    largest code (saturation), subnormal and all-zero groups."""
    rng = np.random.default_rng(seed)
    n_groups = rows * H * 4
    codes = rng.integers(0, 256, n_groups)
    s = O.ue5m3_value(codes)[:, None]
    kind = rng.integers(0, 5, n_groups)[:, None]
    j = rng.integers(-127, 127, (n_groups, 32)).astype(np.float64)
    x = np.where(kind == 0, (j + 0.5) * s, j * s)                       # ties / grid points
    x = np.where(kind == 2, x * 3.0e4, x)                                # saturation
    x = np.where(kind == 3, rng.standard_normal((n_groups, 32)) * 1e-39, x)  # subnormal bf16
    x = np.where((kind == 4) & (rng.random((n_groups, 1)) < 0.2), 0.0, x)
    edge = (kind == 1)[:, 0] & (codes % 8 == 0)
    x[edge, 0] = 127.0 * s[edge, 0]                                      # amax on a boundary
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).reshape(rows, H, 128)
    return t


def test_int8_encoder_hard_values():
    rows, H = 160, 6
    q, k, v = (hard_int8_values(rows, H, seed).cuda() for seed in (11, 12, 13))
    qq, kk, vv = O.widen(q), O.widen(k), O.widen(v)
    ties = np.abs(qq.reshape(-1, 32)) / O.ue5m3_value(
        O.ue5m3_scale_code(np.abs(qq.reshape(-1, 32)).max(-1)))[:, None]
    assert np.any(ties % 1.0 == 0.5) and np.any(ties > 127)  # the cases above survive bf16
    wire = h3.pack_qkv(q, k, v, 2, h3.WIRE_INT8)
    out = h3.pack_out(q, h3.WIRE_INT8)
    torch.cuda.synchronize()
    for d in range(2):
        hs = slice(d * 3, d * 3 + 3)
        assert np.array_equal(as_bytes(wire[d]), O.qkv_int8_records(qq[:, hs], kk[:, hs], vv[:, hs]))
    assert np.array_equal(as_bytes(out), O.out_int8_records(qq))
