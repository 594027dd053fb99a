"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Gate (both bf16 outputs): max |gpu - ref| <= 2e-2 and
||gpu - ref||_2 / ||ref||_2 <= 5e-3 over valid rows.  The prologue also has
an elementwise bound derived from its arithmetic: one bf16 rounding
(<= 2^-8 relative, a flipped rounding included) plus fp32 angle error
(pos * inv_freq rounded in fp32: <= ~2e-4 rad at pos 1,800).

Small and ragged cases are compared on every output element; the full-size
workloads are compared on sampled rows that always include every modality
boundary, tile edges and the last 128 valid rows, and on properties that
hold at any size (padded rows are 0, padded-row contents do not matter,
repeat runs are bitwise identical).
"""
import math
import zlib

import numpy as np
import pytest
import torch

import packed_sequence_attention_gb300 as h3
from oracle import oracle as O
from packed_sequence_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GATE_ABS, GATE_REL = 2e-2, 5e-3
SCALE = 1.0 / math.sqrt(128.0)
ROT = (32, 48, 48)


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    major, minor = torch.cuda.get_device_capability(0)
    assert (major, minor) == (10, 3), "these kernels are built for sm_103a"
    h3.lib()
    torch.cuda.set_device(0)
    yield
    assert h3.status_word() == 0


def gate(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert err.max() <= GATE_ABS and rel <= GATE_REL, \
        f"{what}: max_abs={err.max():.3e} rel_l2={rel:.3e}"
    return err.max(), rel


def prologue_bound(got, ref):
    """Elementwise bound: 2^-8 |ref| + 3e-4 * rms of the (row, head) vector."""
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bad = np.abs(got - ref) > (2.0 ** -8) * np.abs(ref) + 3e-4 * rms + 1e-12
    assert not bad.any(), f"{int(bad.sum())} elements outside the prologue bound"


def to_dev(inp):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


def run_prologue(g):
    w = g["workload"]
    for b, s in enumerate(w.segments):
        r0 = g["cu_seqlens_q"][b]
        h3.qk_norm_rope(g["q"][r0:], g["k"][r0:], g["wq"], g["wk"], g["pos_thw"][r0:],
                        n_rows=s.n_valid_q(), rot=ROT)


def run_attention(g, out=None):
    return h3.attention(g["q"], g["k"], g["v"], g["cu_seqlens_q"], g["cu_seqlens_kv"],
                        g["valid_len"], SCALE, out=g["out"] if out is None else out)


# ------------------------------------------------------------------ prologue
@pytest.mark.parametrize("name", ["tiny", "medium", "stage1_batch2"])
def test_prologue_full_compare(name):
    inp = W.make_inputs(name)
    g = to_dev(inp)
    run_prologue(g)
    # the one-launch form the bench step and attention_block use: the same bits
    qv, kv = inp["q"].cuda(), inp["k"].cuda()
    h3.qk_norm_rope_varlen(qv, kv, g["wq"], g["wk"], g["pos_thw"], g["cu_seqlens_q"],
                           g["valid_len"], rot=ROT)
    torch.cuda.synchronize()
    assert torch.equal(qv.view(torch.int16), g["q"].view(torch.int16))
    assert torch.equal(kv.view(torch.int16), g["k"].view(torch.int16))
    w = inp["workload"]
    pos = inp["pos_thw"].numpy()
    for t, wn in (("q", "wq"), ("k", "wk")):
        got = O.widen(g[t])
        for b, s in enumerate(w.segments):
            r0, n = inp["cu_seqlens_q"][b], s.n_valid_q()
            ref = O.qk_norm_rope(O.widen(inp[t][r0:r0 + n]), O.widen(inp[wn]), pos[r0:r0 + n])
            gate(got[r0:r0 + n], ref, f"{name} {t} seg{b}")
            prologue_bound(got[r0:r0 + n], ref)
            # rows past the valid length are not touched
            pad = slice(r0 + n, r0 + s.q_rows)
            assert torch.equal(g[t][pad].view(torch.int16).cpu(), inp[t][pad].view(torch.int16))


@pytest.mark.parametrize("rot", [(16, 16, 16), (0, 0, 0), (128, 0, 0), (0, 2, 126), (30, 2, 8)])
def test_prologue_rotary_splits(rot):
    w = W.custom("rot", 3, [W.Segment(300, 300, 293, (3, 7, 9), 80, 24)])
    inp = W.make_inputs(w, seed=11)
    g = to_dev(inp)
    h3.qk_norm_rope(g["q"], g["k"], g["wq"], g["wk"], g["pos_thw"], n_rows=293, rot=rot)
    torch.cuda.synchronize()
    pos = inp["pos_thw"].numpy()[:293]
    for t, wn in (("q", "wq"), ("k", "wk")):
        ref = O.qk_norm_rope(O.widen(inp[t][:293]), O.widen(inp[wn]), pos, sections=rot)
        got = O.widen(g[t])[:293]
        gate(got, ref, f"rot {rot} {t}")
        prologue_bound(got, ref)


@pytest.mark.parametrize("H,rows", [(1, 1), (7, 5), (42, 33), (200, 9), (448, 3)])
def test_prologue_head_counts(H, rows):
    w = W.custom(f"h{H}", H, [W.Segment(rows, rows, None, None, rows, 0)])
    inp = W.make_inputs(w, seed=H)
    g = to_dev(inp)
    h3.qk_norm_rope(g["q"], g["k"], g["wq"], g["wk"], g["pos_thw"], rot=ROT)
    torch.cuda.synchronize()
    pos = inp["pos_thw"].numpy()
    for t, wn in (("q", "wq"), ("k", "wk")):
        ref = O.qk_norm_rope(O.widen(inp[t]), O.widen(inp[wn]), pos)
        got = O.widen(g[t])
        gate(got, ref, f"H={H} {t}")
        prologue_bound(got, ref)


VARLEN = {
    # name: (heads, cu_seqlens, valid_len)
    "two_ragged": (42, [0, 640, 1280], [611, 640]),
    "empty_and_full": (5, [0, 384, 448, 576, 1216], [300, 0, 77, 640]),
    "all_valid": (3, [0, 100, 357], None),
    "sixteen_short": (2, list(range(0, 16 * 40 + 1, 40)), [40 - 2 * i for i in range(16)]),
    "one_row_each": (7, [0, 1, 2, 3], [1, 1, 1]),
}


@pytest.mark.parametrize("case", sorted(VARLEN))
def test_prologue_varlen(case):
    """One launch over several packed sequences: bitwise the per-sequence
    launches, within the prologue bound of the oracle, and no other row
    (padding, or the rows past the last sequence) touched."""
    H, cu, valid = VARLEN[case]
    gen = torch.Generator().manual_seed(zlib.crc32(case.encode()))
    R = cu[-1] + 64  # rows past the last sequence
    q = torch.randn((R, H, 128), generator=gen).to(torch.bfloat16)
    k = torch.randn((R, H, 128), generator=gen).to(torch.bfloat16)
    wq = (1.0 + 0.1 * torch.randn((H, 128), generator=gen)).to(torch.bfloat16)
    wk = (1.0 + 0.1 * torch.randn((H, 128), generator=gen)).to(torch.bfloat16)
    pos = torch.randint(0, 1800, (R, 3), generator=gen, dtype=torch.int32)
    n_valid = [valid[b] if valid is not None else cu[b + 1] - cu[b] for b in range(len(cu) - 1)]
    for b, n in enumerate(n_valid):
        q[cu[b] + n:cu[b + 1]] = float("nan")
        k[cu[b] + n:cu[b + 1]] = float("inf")
    q[cu[-1]:], k[cu[-1]:] = float("nan"), float("-inf")
    dev = {n: t.cuda() for n, t in (("wq", wq), ("wk", wk), ("pos", pos))}
    gq, gk = q.cuda(), k.cuda()
    h3.qk_norm_rope_varlen(gq, gk, dev["wq"], dev["wk"], dev["pos"], cu, valid, rot=ROT)
    sq, sk = q.cuda(), k.cuda()
    for b, n in enumerate(n_valid):
        if n:
            h3.qk_norm_rope(sq[cu[b]:], sk[cu[b]:], dev["wq"], dev["wk"], dev["pos"][cu[b]:],
                            n_rows=n, rot=ROT)
    torch.cuda.synchronize()
    for got, per_seq, src, w, t in ((gq, sq, q, wq, "q"), (gk, sk, k, wk, "k")):
        got_bits = got.view(torch.int16).cpu()
        assert torch.equal(got_bits, per_seq.view(torch.int16).cpu()), f"{t}: != per-sequence"
        got64 = O.widen(got.cpu())
        for b, n in enumerate(n_valid):
            r0 = cu[b]
            if n:
                ref = O.qk_norm_rope(O.widen(src[r0:r0 + n]), O.widen(w), pos.numpy()[r0:r0 + n])
                gate(got64[r0:r0 + n], ref, f"{case} {t} seq{b}")
                prologue_bound(got64[r0:r0 + n], ref)
            untouched = slice(r0 + n, cu[b + 1])
            assert torch.equal(got_bits[untouched], src[untouched].view(torch.int16))
        assert torch.equal(got_bits[cu[-1]:], src[cu[-1]:].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "medium"])
def test_lora_prologue_matches_separate_branches_bitwise(name):
    # The pages' claim for the fused LoRA consumer: byte-exact against the
    # native path that adds the branches into a bf16 tensor first.
    inp = W.make_inputs(name, device="cuda")
    w = inp["workload"]
    n = w.segments[0].n_valid_q()
    gen = torch.Generator(device="cuda").manual_seed(123)
    dq = (0.05 * torch.randn(inp["q"].shape, generator=gen, device="cuda")).to(torch.bfloat16)
    dk = (0.05 * torch.randn(inp["k"].shape, generator=gen, device="cuda")).to(torch.bfloat16)
    q0, k0 = inp["q"].clone(), inp["k"].clone()
    qf, kf = inp["q"].clone(), inp["k"].clone()
    h3.qk_norm_rope_lora(qf, dq, kf, dk, inp["wq"], inp["wk"], inp["pos_thw"], n_rows=n, rot=ROT)
    qs, ks = q0 + dq, k0 + dk  # the separate branches: bf16 sum stored, then the prologue
    h3.qk_norm_rope(qs, ks, inp["wq"], inp["wk"], inp["pos_thw"], n_rows=n, rot=ROT)
    torch.cuda.synchronize()
    assert torch.equal(qf[:n].view(torch.int16), qs[:n].view(torch.int16))
    assert torch.equal(kf[:n].view(torch.int16), ks[:n].view(torch.int16))
    assert torch.equal(qf[n:].view(torch.int16), q0[n:].view(torch.int16))  # rows past n untouched
    pos = inp["pos_thw"].cpu().numpy()[:n]
    for base, delta, wn, got in ((q0, dq, "wq", qf), (k0, dk, "wk", kf)):
        ref = O.qk_norm_rope_lora(O.widen(base[:n]), O.widen(delta[:n]), O.widen(inp[wn]), pos)
        gate(O.widen(got[:n]), ref, f"lora {name}")
        prologue_bound(O.widen(got[:n]), ref)


def test_lora_prologue_strided_views():
    inp = W.make_inputs("medium", device="cuda", packed_qkv=True)
    n = 4000
    gen = torch.Generator(device="cuda").manual_seed(5)
    dbuf = (0.1 * torch.randn((4096, 2, 42, 128), generator=gen, device="cuda")).to(torch.bfloat16)
    dq, dk = dbuf[:, 0], dbuf[:, 1]
    q0, k0 = inp["q"].clone(), inp["k"].clone()
    h3.qk_norm_rope_lora(inp["q"], dq, inp["k"], dk, inp["wq"], inp["wk"], inp["pos_thw"], n_rows=n)
    torch.cuda.synchronize()
    pos = inp["pos_thw"].cpu().numpy()[:n]
    for base, delta, wn, got in ((q0, dq, "wq", inp["q"]), (k0, dk, "wk", inp["k"])):
        ref = O.qk_norm_rope_lora(O.widen(base[:n]), O.widen(delta[:n]), O.widen(inp[wn]), pos)
        gate(O.widen(got[:n]), ref, "lora strided")


def test_prologue_full_size_sampled():
    inp = W.make_inputs("full", device="cuda")
    q0, k0 = inp["q"].cpu(), inp["k"].cpu()
    run_prologue(inp)
    torch.cuda.synchronize()
    rows = sample_rows(inp["workload"].segments[0], 0)
    pos = inp["pos_thw"].cpu().numpy()[rows]
    for t, src, wn in (("q", q0, "wq"), ("k", k0, "wk")):
        ref = O.qk_norm_rope(O.widen(src[rows]), O.widen(inp[wn]), pos)
        got = O.widen(inp[t][torch.as_tensor(rows, device="cuda")])
        gate(got, ref, f"full {t}")
        prologue_bound(got, ref)


# ----------------------------------------------------------------- attention
def sample_rows(seg, r0, n_random=96, seed=0):
    """Row sample: modality boundaries, tile edges, the last 128 valid rows."""
    n = seg.n_valid_q()
    picks = {0, 1, 127, 128, 129, 255, 256, 257, n - 1}
    if seg.video is not None:
        nv = seg.video[0] * seg.video[1] * seg.video[2]
        picks |= {nv - 1, nv, nv + seg.audio - 1, nv + seg.audio}
    picks |= set(range(max(0, n - 128), n))
    picks |= set(np.random.default_rng(seed).integers(0, n, n_random).tolist())
    return np.array(sorted(p + r0 for p in picks if 0 <= p < n))


def check_sampled(inp_cpu, g_after, out, chain_inputs=None):
    """Stage-wise: oracle attention on the GPU prologue's bf16 output.
    End-to-end (chain_inputs given): oracle prologue (fp64, unrounded) ->
    oracle attention, against GPU prologue -> GPU attention."""
    w = inp_cpu["workload"]
    H = w.n_heads
    qg, kg, vg = g_after["q"].cpu(), g_after["k"].cpu(), g_after["v"].cpu()
    outc = out.cpu()
    for b, s in enumerate(w.segments):
        q0, kv0 = inp_cpu["cu_seqlens_q"][b], inp_cpu["cu_seqlens_kv"][b]
        nq, nkv = s.n_valid_q(), s.n_valid_kv()
        if nq == 0:
            continue
        rows = sample_rows(s, q0)
        got = O.widen(outc[torch.as_tensor(rows)])
        ref = np.zeros_like(got)
        ref_e2e = np.zeros_like(got) if chain_inputs is not None else None
        rows_t = torch.as_tensor(rows)
        for h in range(H):
            qs = O.widen(qg[rows_t, h])
            kh, vh = O.widen(kg[kv0:kv0 + nkv, h]), O.widen(vg[kv0:kv0 + nkv, h])
            ref[:, h] = O.attention(qs[:, None], kh[:, None], vh[:, None], [0, len(rows)],
                                    [0, nkv], None, SCALE)[:, 0]
            if chain_inputs is not None:
                q_src, k_src, pos = chain_inputs
                pq = O.qk_norm_rope(O.widen(q_src[torch.as_tensor(rows), h:h + 1]),
                                    O.widen(inp_cpu["wq"][h:h + 1]), pos[rows])[:, 0]
                pk = O.qk_norm_rope(O.widen(k_src[kv0:kv0 + nkv, h:h + 1]),
                                    O.widen(inp_cpu["wk"][h:h + 1]), pos[kv0:kv0 + nkv])[:, 0]
                ref_e2e[:, h] = O.attention(pq[:, None], pk[:, None], vh[:, None],
                                            [0, len(rows)], [0, nkv], None, SCALE)[:, 0]
        gate(got, ref, f"{w.name} seg{b} stage-wise")
        if ref_e2e is not None:
            gate(got, ref_e2e, f"{w.name} seg{b} end-to-end")
        pad = outc[q0 + nq:q0 + s.q_rows]
        assert (pad.float() == 0).all(), "padded output rows must be 0"


@pytest.mark.parametrize("name", ["tiny", "medium"])
def test_attention_full_compare(name):
    inp = W.make_inputs(name, fill="B")
    g = to_dev(inp)
    run_prologue(g)
    out = run_attention(g)
    torch.cuda.synchronize()
    n = inp["valid_len"][0]
    qg, kg, vg = O.widen(g["q"][:n]), O.widen(g["k"][:n]), O.widen(g["v"][:n])
    ref = O.attention(qg, kg, vg, [0, n], [0, n], None, SCALE)
    got = O.widen(out)
    gate(got[:n], ref, f"{name} stage-wise")
    assert (got[n:] == 0).all()
    # end to end from the fp64 prologue
    pos = inp["pos_thw"].numpy()[:n]
    pq = O.qk_norm_rope(O.widen(inp["q"][:n]), O.widen(inp["wq"]), pos)
    pk = O.qk_norm_rope(O.widen(inp["k"][:n]), O.widen(inp["wk"]), pos)
    gate(got[:n], O.attention(pq, pk, O.widen(inp["v"][:n]), [0, n], [0, n], None, SCALE),
         f"{name} end-to-end")


RAGGED = {
    # name: (heads, cu_q, cu_kv, valid_len)
    "one_key": (2, [0, 8], [0, 8], [1]),
    "kv129": (3, [0, 200], [0, 200], [129]),
    "q257": (1, [0, 300], [0, 300], [257]),
    "multi_seg_with_empty": (4, [0, 384, 448, 576, 1216], [0, 384, 448, 576, 1216],
                             [300, 0, 77, 513]),
    "grouped": (3, [0, 5, 200, 201], [0, 700, 701, 1000], None),
    "grouped_empty_kv": (2, [0, 10, 20], [0, 0, 50], None),
    "many_segments": (2, list(range(0, 16 * 40 + 1, 40)), list(range(0, 16 * 40 + 1, 40)),
                      [40 - i for i in range(16)]),
    "long_kv_short_q": (2, [0, 3], [0, 2000], None),
}


@pytest.mark.parametrize("case", sorted(RAGGED))
def test_attention_ragged_cases(case):
    H, cu_q, cu_kv, valid = RAGGED[case]
    gen = torch.Generator().manual_seed(zlib.crc32(case.encode()))
    Rq, Rkv = cu_q[-1], cu_kv[-1]
    q = torch.randn((Rq, H, 128), generator=gen).to(torch.bfloat16)
    k = torch.randn((Rkv, H, 128), generator=gen).to(torch.bfloat16)
    v = torch.randn((Rkv, H, 128), generator=gen).to(torch.bfloat16)
    if valid is not None:  # garbage in padded rows
        for b in range(len(valid)):
            for t in (q, k, v):
                t[cu_q[b] + valid[b]:cu_q[b + 1]] = float("nan")
    out = torch.full((Rq, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    h3.attention(q.cuda(), k.cuda(), v.cuda(), cu_q, cu_kv, valid, SCALE, out=out)
    torch.cuda.synchronize()
    ref = O.attention(O.widen(q), O.widen(k), O.widen(v), cu_q, cu_kv, valid, SCALE)
    got = O.widen(out)
    assert np.isfinite(got).all()
    if np.linalg.norm(ref) > 0:
        gate(got, ref, case)
    zero = np.linalg.norm(ref.reshape(Rq, -1), axis=1) == 0
    assert (got[zero] == 0).all()


def test_attention_full_size_sampled():
    inp = W.make_inputs("full", device="cuda", fill="B")
    q_src, k_src = inp["q"].cpu(), inp["k"].cpu()
    run_prologue(inp)
    out = run_attention(inp)
    torch.cuda.synchronize()
    cpu = dict(inp, wq=inp["wq"].cpu(), wk=inp["wk"].cpu())
    check_sampled(cpu, inp, out, (q_src, k_src, inp["pos_thw"].cpu().numpy()))


def test_attention_stage1_batch2_sampled():
    inp = W.make_inputs("stage1_batch2", device="cuda", fill="B")
    run_prologue(inp)
    out = run_attention(inp)
    torch.cuda.synchronize()
    check_sampled(dict(inp), inp, out)


def test_attention_grouped_chunk_sampled():
    inp = W.make_inputs("grouped_chunk", device="cuda")
    out = run_attention(inp)
    torch.cuda.synchronize()
    check_sampled(dict(inp), inp, out)


# ----------------------------------------------------------- properties
def test_padded_rows_do_not_matter_bitwise():
    outs = []
    for fill in ("A", "B"):
        g = to_dev(W.make_inputs("medium", fill=fill))
        run_prologue(g)
        outs.append(run_attention(g).clone())
    torch.cuda.synchronize()
    n = 4000
    assert torch.equal(outs[0][:n].view(torch.int16), outs[1][:n].view(torch.int16))
    assert (outs[0][n:].float() == 0).all() and (outs[1][n:].float() == 0).all()


def test_repeat_runs_bitwise_identical():
    g = to_dev(W.make_inputs("stage1_batch2"))
    run_prologue(g)
    a = run_attention(g).clone()
    b = run_attention(g, out=torch.empty_like(g["out"])).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("layout", ["packed_qkv", "row_pad"])
def test_strided_views_match_contiguous_bitwise(layout):
    base = W.make_inputs("medium", device="cuda")
    run_prologue(base)
    ref = run_attention(base).clone()
    kw = {"packed_qkv": True} if layout == "packed_qkv" else {"row_pad": 24}
    g = W.make_inputs("medium", device="cuda", **kw)
    assert g["q"].stride(0) != g["q"].shape[1] * 128
    run_prologue(g)
    out_buf = torch.full((4096, 42 * 128 + 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = run_attention(g, out=out_buf[:, :42 * 128].view(4096, 42, 128))
    torch.cuda.synchronize()
    assert torch.equal(out[:4000].view(torch.int16), ref[:4000].view(torch.int16))


def test_key_permutation_equivariance():
    g = to_dev(W.make_inputs("medium"))
    run_prologue(g)
    a = run_attention(g).clone()
    perm = torch.randperm(4000, generator=torch.Generator().manual_seed(3)).cuda()
    g["k"][:4000] = g["k"][:4000][perm]
    g["v"][:4000] = g["v"][:4000][perm]
    b = run_attention(g, out=torch.empty_like(g["out"]))
    torch.cuda.synchronize()
    gate(O.widen(b[:4000]), O.widen(a[:4000]), "permuted keys")


@pytest.mark.parametrize("boost", [1.5, 6.0, 40.0])
def test_attention_row_max_jumps(boost):
    # Keys past row 300 are scaled up, so the row max of later KV tiles jumps
    # by up to ~2^(boost * 12) over the first tile's: the softmax's exact
    # rescaling path (and, for small boosts, the no-rescale path) must agree
    # with the oracle.
    H, L = 2, 700
    gen = torch.Generator().manual_seed(int(boost * 10))
    q = torch.randn((L, H, 128), generator=gen)
    k = torch.randn((L, H, 128), generator=gen)
    k[300:] *= boost
    v = torch.randn((L, H, 128), generator=gen)
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    out = h3.attention(q.cuda(), k.cuda(), v.cuda(), [0, L], [0, L], None, SCALE)
    torch.cuda.synchronize()
    ref = O.attention(O.widen(q), O.widen(k), O.widen(v), [0, L], [0, L], None, SCALE)
    gate(O.widen(out), ref, f"boost {boost}")


def _rand(shape, gen):
    return torch.randn(shape, generator=gen).to(torch.bfloat16)


GROUP_CASES = {
    # name: (heads, q rows, kv rows, cache rows, groups)
    "ref_cache": (3, 300, 300, 500, [(0, 260, 0, 260, 0, 500)]),
    "overlapping_views": (2, 200, 400, 0, [(0, 50, 0, 300, 0, 0), (50, 130, 100, 300, 0, 0),
                                          (180, 20, 399, 1, 0, 0)]),
    "cache_only_and_empty": (2, 160, 64, 333, [(0, 40, 0, 0, 17, 300), (40, 60, 0, 0, 0, 0),
                                             (100, 50, 10, 54, 1, 129)]),
    "skipped_rows": (2, 400, 400, 256, [(100, 150, 0, 400, 0, 256), (300, 77, 300, 100, 128, 128)]),
}


@pytest.mark.parametrize("case", sorted(GROUP_CASES))
def test_attention_groups_cases(case):
    H, nq, nkv, nc, groups = GROUP_CASES[case]
    gen = torch.Generator().manual_seed(zlib.crc32(case.encode()))
    q, k, v = _rand((nq, H, 128), gen), _rand((nkv, H, 128), gen), _rand((nkv, H, 128), gen)
    kc = _rand((max(nc, 1), H, 128), gen)
    vc = _rand((max(nc, 1), H, 128), gen)
    out = torch.full((nq, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    h3.attention_groups(q.cuda(), k.cuda(), v.cuda(), groups, kc.cuda(), vc.cuda(), SCALE, out=out)
    torch.cuda.synchronize()
    rows, ref = O.attention_groups(O.widen(q), O.widen(k), O.widen(v), O.widen(kc), O.widen(vc),
                                   groups, SCALE)
    got = O.widen(out)
    if np.linalg.norm(ref) > 0:
        gate(got[rows], ref, case)
    assert (got[rows][np.linalg.norm(ref.reshape(len(rows), -1), axis=1) == 0] == 0).all()
    untouched = np.setdiff1d(np.arange(nq), rows)
    assert np.isnan(got[untouched]).all(), "rows outside every group must not be written"


def test_attention_groups_equal_cu_seqlens_bitwise():
    g = to_dev(W.make_inputs("stage1_batch2"))
    run_prologue(g)
    a = run_attention(g).clone()
    groups = [(0, 16422, 0, 16422, 0, 0), (16448, 16422, 16448, 16422, 0, 0)]
    b = torch.full_like(a, float("nan"))
    h3.attention_groups(g["q"], g["k"], g["v"], groups, scale=SCALE, out=b)
    torch.cuda.synchronize()
    for r0 in (0, 16448):
        assert torch.equal(a[r0:r0 + 16422].view(torch.int16), b[r0:r0 + 16422].view(torch.int16))


def test_attention_groups_ref_cached_full_size_sampled():
    inp = W.ref_cached_inputs(device="cuda")
    out = h3.attention_groups(inp["q"], inp["k"], inp["v"], inp["groups"], inp["k_cache"],
                              inp["v_cache"], SCALE, out=inp["out"])
    torch.cuda.synchronize()
    n, nc = 16422, inp["k_cache"].shape[0]
    rows = sample_rows(W.Segment(16448, 16448, n, (21, 24, 28), 1800, 510), 0)
    rows_t = torch.as_tensor(rows)
    qc, kc, vc = inp["q"].cpu(), inp["k"].cpu(), inp["v"].cpu()
    kcc, vcc = inp["k_cache"].cpu(), inp["v_cache"].cpu()
    got = O.widen(out.cpu()[rows_t])
    ref = np.zeros_like(got)
    for h in range(42):
        _, r = O.attention_groups(O.widen(qc[rows_t, h:h + 1]), O.widen(kc[:n, h:h + 1]),
                                  O.widen(vc[:n, h:h + 1]), O.widen(kcc[:, h:h + 1]),
                                  O.widen(vcc[:, h:h + 1]), [(0, len(rows), 0, n, 0, nc)], SCALE)
        ref[:, h] = r[:, 0]
    gate(got, ref, "ref-cached full size")
    assert torch.isnan(out[n:].float()).all()  # padded rows belong to no group


def test_closed_forms_on_gpu():
    # all V rows equal -> out = that row; single valid key -> out = v_0
    H, L = 2, 300
    gen = torch.Generator().manual_seed(5)
    q = torch.randn((L, H, 128), generator=gen).to(torch.bfloat16).cuda()
    k = torch.randn((L, H, 128), generator=gen).to(torch.bfloat16).cuda()
    row = torch.randn((1, H, 128), generator=gen).to(torch.bfloat16).cuda()
    v = row.repeat(L, 1, 1)
    out = h3.attention(q, k, v, [0, L], [0, L], None, SCALE)
    torch.cuda.synchronize()
    got, exp = O.widen(out), O.widen(v)
    assert (np.abs(got - exp) <= 2.0 ** -8 * np.abs(exp)).all()
    v2 = torch.randn((L, H, 128), generator=gen).to(torch.bfloat16).cuda()
    out = h3.attention(q, k, v2, [0, L], [0, L], [1], SCALE)
    torch.cuda.synchronize()
    assert torch.equal(out[:1].view(torch.int16), v2[:1].view(torch.int16))
    assert (out[1:].float() == 0).all()
