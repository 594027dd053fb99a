"""GPU: no entry point writes outside its outputs.

Every output (and every in-place tensor) lives inside a device byte buffer
framed by canary margins; row-strided tensors also carry canary pad columns
and rows past the extent the call may touch.  After each call every canary
byte must be intact.  compute-sanitizer is not available, so these guard
regions stand in for an out-of-bounds store detector."""
import ctypes

import numpy as np
import pytest
import torch

import packed_sequence_attention_gb300 as h3
from packed_sequence_attention_gb300 import _binding
from packed_sequence_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu
CANARY = 0xA5
MARGIN = 4096
SCALE = 128 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    h3.lib()
    yield
    assert h3.status_word() == 0


class Guarded:
    """nbytes of payload framed by MARGIN canary bytes on both sides."""

    def __init__(self, nbytes):
        self.n = nbytes
        self.buf = torch.full((2 * MARGIN + nbytes,), CANARY, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        return self.buf[MARGIN:MARGIN + self.n].view(dtype).view(shape)

    def ptr(self):
        return self.buf.data_ptr() + MARGIN

    def margins_intact(self):
        return bool((self.buf[:MARGIN] == CANARY).all() and (self.buf[MARGIN + self.n:] == CANARY).all())


def guarded_rows(rows, H, pad=8, extra_rows=0, fill=None):
    """bf16 [rows, H, 128] view with row stride H*128 + pad inside a guarded
    buffer of rows + extra_rows rows; returns (guard, view, canary_mask_fn)."""
    stride = H * 128 + pad
    g = Guarded((rows + extra_rows) * stride * 2)
    full = g.view(torch.bfloat16, (rows + extra_rows, stride))
    view = full[:rows, :H * 128].view(rows, H, 128)
    if fill is not None:
        view.copy_(fill)

    def untouched_outside():
        b = full.view(torch.uint8).view(rows + extra_rows, stride * 2)
        pads = (b[:, H * 256:] == CANARY).all()
        tail = (b[rows:] == CANARY).all() if extra_rows else torch.tensor(True)
        return bool(pads and tail) and g.margins_intact()
    return g, view, untouched_outside


def rnd(shape, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)


def test_prologue_and_lora_stay_in_their_rows():
    H, rows, n = 6, 300, 250
    _, q, q_ok = guarded_rows(rows, H, extra_rows=5, fill=rnd((rows, H, 128), 1))
    _, k, k_ok = guarded_rows(rows, H, extra_rows=5, fill=rnd((rows, H, 128), 2))
    q_tail, k_tail = q[n:].clone(), k[n:].clone()
    w = rnd((H, 128), 3)
    pos = torch.zeros((rows, 3), dtype=torch.int32, device="cuda")
    h3.qk_norm_rope(q, k, w, w, pos, n_rows=n)
    torch.cuda.synchronize()
    assert q_ok() and k_ok()
    assert torch.equal(q[n:].view(torch.int16), q_tail.view(torch.int16))  # rows >= n untouched
    assert torch.equal(k[n:].view(torch.int16), k_tail.view(torch.int16))
    dq, dk = rnd((rows, H, 128), 4), rnd((rows, H, 128), 5)
    h3.qk_norm_rope_lora(q, dq, k, dk, w, w, pos, n_rows=n)
    torch.cuda.synchronize()
    assert q_ok() and k_ok()
    assert torch.equal(q[n:].view(torch.int16), q_tail.view(torch.int16))


def test_attention_and_groups_outputs():
    H, rows = 3, 700
    q, k, v = rnd((rows, H, 128), 6), rnd((rows, H, 128), 7), rnd((rows, H, 128), 8)
    _, out, ok = guarded_rows(rows, H, extra_rows=3)
    h3.attention(q, k, v, [0, 300, 650], [0, 300, 650], [290, 350], SCALE, out=out)
    torch.cuda.synchronize()
    assert ok()
    assert (out[650:].view(torch.uint8) == CANARY).all()  # rows past the last segment
    _, out2, ok2 = guarded_rows(rows, H, extra_rows=3)
    h3.attention_groups(q, k, v, [(10, 100, 0, 300, 0, 0), (400, 77, 100, 500, 0, 0)], None, None,
                        SCALE, out=out2)
    torch.cuda.synchronize()
    assert ok2()
    b = out2.view(torch.uint8)
    assert (b[:10] == CANARY).all() and (b[110:400] == CANARY).all() and (b[477:] == CANARY).all()


def test_block_sparse_stages():
    lib = h3.lib()
    H, rows = 2, 1000
    nb = -(-rows // 128)
    q, k, v = rnd((rows, H, 128), 9), rnd((rows, H, 128), 10), rnd((rows, H, 128), 11)
    gm = [Guarded(nb * H * 128 * 4) for _ in range(2)]
    for g, x in zip(gm, (q, k)):
        assert lib.h3_block_means(x.data_ptr(), H * 128, rows, H, 128, g.ptr(), None) == 0
    gqk = [Guarded(nb * H * 128 * 4) for _ in range(2)]
    assert lib.h3_block_means_qk(q.data_ptr(), H * 128, k.data_ptr(), H * 128, rows, H, 128,
                                 gqk[0].ptr(), gqk[1].ptr(), None) == 0
    gl, gc, gs = Guarded(H * nb * nb * 4), Guarded(H * nb * 4), Guarded(H * nb * nb * 4)
    assert lib.h3_block_select(gm[0].ptr(), gm[1].ptr(), nb, nb, H, SCALE, 0.5, 1, gs.ptr(),
                               gl.ptr(), gc.ptr(), None) == 0
    _, out, ok = guarded_rows(rows, H, extra_rows=2)
    assert lib.h3_sparse_attention(q.data_ptr(), H * 128, k.data_ptr(), H * 128, v.data_ptr(),
                                   H * 128, out.data_ptr(), out.stride(0), rows, H, 128, gl.ptr(),
                                   gc.ptr(), 1, SCALE, None) == 0
    torch.cuda.synchronize()
    assert all(g.margins_intact() for g in (*gm, *gqk, gl, gc, gs)) and ok()


@pytest.mark.parametrize("fmt", [h3.WIRE_BF16, h3.WIRE_INT8])
def test_qkv_wire_kernels(fmt):
    lib = h3.lib()
    H, rows, nd = 6, 250, 3
    q, k, v = rnd((rows, H, 128), 12), rnd((rows, H, 128), 13), rnd((rows, H, 128), 14)
    rec = h3.wire_record_bytes("qkv", fmt)
    gw = Guarded(nd * rows * (H // nd) * rec)
    assert lib.h3_pack_qkv(q.data_ptr(), H * 128, k.data_ptr(), H * 128, v.data_ptr(), H * 128,
                           rows, H, nd, fmt, gw.ptr(), None) == 0
    outs = [guarded_rows(rows, H // nd, extra_rows=1) for _ in range(3)]
    assert lib.h3_unpack_qkv(gw.ptr(), rows, H // nd, fmt, outs[0][1].data_ptr(), outs[0][1].stride(0),
                             outs[1][1].data_ptr(), outs[1][1].stride(0), outs[2][1].data_ptr(),
                             outs[2][1].stride(0), None) == 0
    torch.cuda.synchronize()
    assert gw.margins_intact() and all(o[2]() for o in outs)


@pytest.mark.parametrize("fmt", [h3.WIRE_BF16, h3.WIRE_INT8, h3.WIRE_FP8])
def test_output_wire_kernels(fmt):
    lib = h3.lib()
    H, rows, ns = 6, 250, 2
    o = rnd((rows, H, 128), 15)
    rec = h3.wire_record_bytes("out", fmt)
    gw = Guarded(ns * rows * (H // ns) * rec)
    for s in range(ns):
        part = o[:, s * (H // ns):(s + 1) * (H // ns)]
        assert lib.h3_pack_out(part.data_ptr(), H * 128, rows, H // ns, fmt,
                               gw.ptr() + s * rows * (H // ns) * rec, None) == 0
    _, merged, ok = guarded_rows(rows, H, extra_rows=1)
    assert lib.h3_merge_heads(gw.ptr(), rows, H, ns, fmt, merged.data_ptr(), merged.stride(0), None) == 0
    torch.cuda.synchronize()
    assert gw.margins_intact() and ok()
