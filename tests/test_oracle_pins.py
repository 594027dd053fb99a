"""Pins of the fp64 oracle against facts fixed outside itself.

Each check ties one part of the oracle to a closed form, an invariant, the
independent pure-Python brute force, or a library routine (torch SDPA in
float64 on the CPU), so that a plausible slip -- a dropped term, a wrong
sign, a swapped index, a transposed operand, another rotary pairing -- fails
at least one of them.  ``test_planted_mistakes_are_caught`` plants such
slips in copies of the oracle and checks that the pins reject every one.
"""
import json
import math
import os
import types

import numpy as np
import pytest
import torch

from oracle import brute
from oracle import oracle as O
from packed_sequence_attention_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
SECTIONS = (32, 48, 48)
THETA = 10000.0
EPS = 1e-6
SCALE = 1.0 / math.sqrt(128.0)


def _tiny_inputs(fill="A"):
    inp = W.make_inputs("tiny", fill=fill)
    return inp, {k: O.widen(inp[k]) for k in ("q", "k", "v", "wq", "wk")}


def _prologued_tiny(Ox=O, fill="A"):
    inp, f = _tiny_inputs(fill)
    pos = inp["pos_thw"].numpy()
    q = Ox.qk_norm_rope(f["q"], f["wq"], pos, SECTIONS, THETA, EPS)
    k = Ox.qk_norm_rope(f["k"], f["wk"], pos, SECTIONS, THETA, EPS)
    return inp, q, k, f["v"]


# ------------------------------------------------------------ pin checks
# Each returns the worst deviation found; a pin holds when it is <= its bound.

def pin_norm_closed_form(Ox):
    """Unit weights: output mean square = ms / (ms + eps); explicit vector."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 128)) * np.array([1e-3, 1.0, 30.0])[None, :, None]
    y = Ox.rms_norm(x, np.ones(128), EPS)
    ms = np.mean(x * x, -1)
    dev = np.max(np.abs(np.mean(y * y, -1) - ms / (ms + EPS)) / (ms / (ms + EPS)))
    # x = (3, 4, 0, ...): mean square 25/128, y = x / sqrt(25/128 + eps) * w
    x1 = np.zeros(128); x1[0], x1[1] = 3.0, 4.0
    w1 = np.linspace(0.5, 1.5, 128)
    y1 = Ox.rms_norm(x1, w1, EPS)
    r = 1.0 / math.sqrt(25.0 / 128.0 + EPS)
    exp1 = np.zeros(128); exp1[0], exp1[1] = 3.0 * r * w1[0], 4.0 * r * w1[1]
    return max(dev, float(np.max(np.abs(y1 - exp1))))


def pin_norm_scale_invariance(Ox):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 2, 128))
    w = rng.standard_normal(128)
    return float(np.max(np.abs(Ox.rms_norm(37.5 * x, w, 0.0) - Ox.rms_norm(x, w, 0.0))))


def pin_rope_closed_forms(Ox):
    """Single nonzero pair -> the 2x2 rotation by pos * theta^(-2j/d) of its
    own axis; pairs are adjacent channels; other channels untouched."""
    worst = 0.0
    cases = [  # (channel c0, pos (t,h,w), expected angle)
        (0, (1, 0, 0), 1.0),                                   # t, j=0
        (2, (1, 0, 0), THETA ** (-2.0 / 32)),                  # t, j=1
        (30, (3, 0, 0), 3 * THETA ** (-30.0 / 32)),            # t, last pair
        (32, (0, 1, 0), 1.0),                                  # h, j=0
        (32, (5, 0, 7), 0.0),                                  # h ignores t, w
        (78, (0, 2, 0), 2 * THETA ** (-46.0 / 48)),            # h, last pair
        (80, (0, 0, 1), 1.0),                                  # w, j=0
        (126, (0, 0, 3), 3 * THETA ** (-46.0 / 48)),           # w, last pair
        (100, (9, 9, 0), 0.0),                                 # w ignores t, h
    ]
    for c0, p, ang in cases:
        y = np.zeros((1, 1, 128)); y[0, 0, c0] = 0.6; y[0, 0, c0 + 1] = -0.8
        out = Ox.rope_axial(y, np.array([p]), SECTIONS, THETA)[0, 0]
        exp = np.zeros(128)
        exp[c0] = 0.6 * math.cos(ang) + 0.8 * math.sin(ang)
        exp[c0 + 1] = 0.6 * math.sin(ang) - 0.8 * math.cos(ang)
        worst = max(worst, float(np.max(np.abs(out - exp))))
    return worst


def pin_rope_invariants(Ox):
    """|R(p) y| = |y| per pair; R(0) = I; <R(p+s)q, R(p'+s)k> = <R(p)q, R(p')k>
    for a shift s along each axis separately."""
    rng = np.random.default_rng(3)
    y = rng.standard_normal((6, 2, 128))
    pos = rng.integers(0, 60, size=(6, 3))
    r = Ox.rope_axial(y, pos, SECTIONS, THETA)
    pair_norm = lambda a: a[..., 0::2] ** 2 + a[..., 1::2] ** 2
    worst = float(np.max(np.abs(pair_norm(r) - pair_norm(y))))
    worst = max(worst, float(np.max(np.abs(
        Ox.rope_axial(y, np.zeros((6, 3), int), SECTIONS, THETA) - y))))
    q = rng.standard_normal((1, 1, 128)); k = rng.standard_normal((1, 1, 128))
    p, pp = np.array([[4, 7, 2]]), np.array([[11, 3, 19]])
    base = float(np.sum(Ox.rope_axial(q, p, SECTIONS, THETA) *
                        Ox.rope_axial(k, pp, SECTIONS, THETA)))
    for axis in range(3):
        s = np.zeros((1, 3), int); s[0, axis] = 13
        sh = float(np.sum(Ox.rope_axial(q, p + s, SECTIONS, THETA) *
                          Ox.rope_axial(k, pp + s, SECTIONS, THETA)))
        worst = max(worst, abs(sh - base))
    return worst


def pin_prologue_brute(Ox):
    """NumPy prologue == pure-Python brute force on tiny rows of each kind."""
    inp, f = _tiny_inputs()
    pos = inp["pos_thw"].numpy()
    rows = [0, 1, 63, 64, 127, 128, 150, 191, 192, 220, 249]
    worst = 0.0
    for name, wname in (("q", "wq"), ("k", "wk")):
        got = Ox.qk_norm_rope(f[name], f[wname], pos, SECTIONS, THETA, EPS)
        for r in rows:
            for h in range(2):
                exp = brute.norm_rope_row(list(f[name][r, h]), list(f[wname][h]),
                                          tuple(int(v) for v in pos[r]),
                                          SECTIONS, THETA, EPS)
                worst = max(worst, float(np.max(np.abs(got[r, h] - np.array(exp)))))
    return worst


def pin_attention_brute(Ox):
    """NumPy attention == pure-Python brute force (tiny, sampled rows)."""
    inp, q, k, v = _prologued_tiny(Ox)
    cu, vl = inp["cu_seqlens_q"], inp["valid_len"]
    rows = [0, 5, 64, 127, 128, 191, 192, 249]
    got = Ox.attention(q, k, v, cu, cu, vl, SCALE, rows=rows)
    worst = 0.0
    n = vl[0]
    for i, r in enumerate(rows):
        for h in range(2):
            exp = brute.attention_row(list(q[r, h]), [list(k[j, h]) for j in range(n)],
                                      [list(v[j, h]) for j in range(n)], SCALE)
            worst = max(worst, float(np.max(np.abs(got[i, h] - np.array(exp)))))
    return worst


def pin_attention_closed_forms(Ox):
    rng = np.random.default_rng(4)
    L, H, D = 37, 2, 128
    q = rng.standard_normal((L, H, D)); k = rng.standard_normal((L, H, D))
    v = rng.standard_normal((L, H, D))
    cu = [0, L]
    worst = 0.0
    # one valid key -> o = v_0 on valid rows (valid_len 1 -> only row 0 valid)
    o = Ox.attention(q, k, v, cu, cu, [1], SCALE)
    worst = max(worst, float(np.max(np.abs(o[0] - v[0]))), float(np.max(np.abs(o[1:]))))
    # all V rows equal c -> o = c
    c = rng.standard_normal((1, H, D))
    o = Ox.attention(q, k, np.repeat(c, L, 0), cu, cu, None, SCALE)
    worst = max(worst, float(np.max(np.abs(o - c))))
    # all K rows equal -> uniform weights -> o = mean(V)
    o = Ox.attention(q, np.repeat(k[:1], L, 0), v, cu, cu, None, SCALE)
    worst = max(worst, float(np.max(np.abs(o - v.mean(0, keepdims=True)))))
    # Q = 0 -> o = mean(V over valid keys)
    o = Ox.attention(np.zeros_like(q), k, v, cu, cu, [20], SCALE)
    worst = max(worst, float(np.max(np.abs(o[:20] - v[:20].mean(0, keepdims=True)))))
    # two keys with score gap g -> weights (1, e^-g)/(1 + e^-g), exact closed form
    qq = np.zeros((1, 1, D)); qq[0, 0, 0] = 1.0
    kk = np.zeros((2, 1, D)); kk[0, 0, 0] = 3.0 / SCALE; kk[1, 0, 0] = 1.0 / SCALE
    vv = np.zeros((2, 1, D)); vv[0, 0, 5] = 1.0; vv[1, 0, 5] = -2.0
    o = Ox.attention(qq, kk, vv, [0, 1], [0, 2], None, SCALE)
    p0 = 1.0 / (1.0 + math.exp(-2.0))
    worst = max(worst, abs(o[0, 0, 5] - (p0 - 2.0 * (1.0 - p0))))
    return worst


def pin_attention_sdpa(Ox):
    """Library cross-check: torch SDPA in float64 on the CPU, per segment."""
    inp, q, k, v = _prologued_tiny(Ox)
    n = inp["valid_len"][0]
    got = Ox.attention(q, k, v, inp["cu_seqlens_q"], inp["cu_seqlens_kv"],
                       inp["valid_len"], SCALE)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a[:n].transpose(1, 0, 2)))[None]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v))
    ref = ref[0].numpy().transpose(1, 0, 2)
    return float(np.max(np.abs(got[:n] - ref)))


def pin_attention_grouped_sdpa(Ox):
    """Grouped query ranges with unequal KV extents vs SDPA per group."""
    rng = np.random.default_rng(5)
    H, D = 2, 128
    cu_q, cu_kv = [0, 9, 40, 41], [0, 30, 33, 100]
    q = rng.standard_normal((41, H, D)); k = rng.standard_normal((100, H, D))
    v = rng.standard_normal((100, H, D))
    got = Ox.attention(q, k, v, cu_q, cu_kv, None, 0.3)
    worst = 0.0
    for b in range(3):
        t = lambda a, lo, hi: torch.from_numpy(np.ascontiguousarray(
            a[lo:hi].transpose(1, 0, 2)))[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            t(q, cu_q[b], cu_q[b + 1]), t(k, cu_kv[b], cu_kv[b + 1]),
            t(v, cu_kv[b], cu_kv[b + 1]), scale=0.3)[0].numpy().transpose(1, 0, 2)
        worst = max(worst, float(np.max(np.abs(got[cu_q[b]:cu_q[b + 1]] - ref))))
    return worst


def pin_attention_invariants(Ox):
    """Joint permutation of valid K/V rows changes nothing; padded-row
    contents (including NaN / Inf) change nothing on valid rows; padded
    output rows are 0."""
    inp, q, k, v = _prologued_tiny(Ox)
    cu, vl = inp["cu_seqlens_q"], inp["valid_len"]
    n = vl[0]
    base = Ox.attention(q, k, v, cu, cu, vl, SCALE)
    perm = np.random.default_rng(6).permutation(n)
    k2, v2 = k.copy(), v.copy()
    k2[:n], v2[:n] = k[perm], v[perm]
    worst = float(np.max(np.abs(Ox.attention(q, k2, v2, cu, cu, vl, SCALE) - base)))
    k3, v3, q3 = k.copy(), v.copy(), q.copy()
    for a in (q3, k3, v3):
        a[n:] = np.nan
        a[n::3] = np.inf
    o3 = Ox.attention(q3, k3, v3, cu, cu, vl, SCALE)
    diff = np.abs(o3[:n] - base[:n])
    worst = max(worst, float(np.max(np.where(np.isfinite(diff), diff, np.inf))))
    worst = max(worst, float(np.max(np.abs(base[n:]))))
    return worst


def pin_attention_groups(Ox):
    """Groups over KV views: (i) disjoint views without a cache reproduce
    ``attention`` over cu_seqlens; (ii) splitting a view between the current
    and the cache tensors changes nothing; (iii) key order is irrelevant;
    (iv) torch SDPA in float64 on the concatenated keys; (v) a group with no
    key outputs zeros."""
    rng = np.random.default_rng(10)
    H, D = 2, 128
    q = rng.standard_normal((60, H, D)); k = rng.standard_normal((90, H, D))
    v = rng.standard_normal((90, H, D))
    kc = rng.standard_normal((40, H, D)); vc = rng.standard_normal((40, H, D))
    groups = [(0, 20, 0, 30, 0, 0), (20, 40, 30, 60, 0, 0)]
    rows, got = Ox.attention_groups(q, k, v, kc, vc, groups, 0.2)
    ref = Ox.attention(q, k, v, [0, 20, 60], [0, 30, 90], None, 0.2)
    worst = float(np.max(np.abs(got - ref[rows])))
    # (ii) keys 50..89 moved to the cache tensors
    kc2 = np.concatenate([k[50:90], kc]); vc2 = np.concatenate([v[50:90], vc])
    rows2, got2 = Ox.attention_groups(q, k, v, kc2, vc2, [(20, 40, 30, 20, 0, 40)], 0.2)
    worst = max(worst, float(np.max(np.abs(got2 - got[20:]))))
    # (iii) + (iv) overlapping views with a cache range against SDPA
    g = [(5, 30, 10, 50, 7, 33), (30, 25, 0, 70, 0, 0)]
    rows3, got3 = Ox.attention_groups(q, k, v, kc, vc, g, 0.15)
    for (q0, nq, k0, nk, c0, nc), lo in zip(g, (0, 30)):
        kk = np.concatenate([kc[c0:c0 + nc], k[k0:k0 + nk]])   # other key order
        vv = np.concatenate([vc[c0:c0 + nc], v[k0:k0 + nk]])
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a.transpose(1, 0, 2)))[None]
        sd = torch.nn.functional.scaled_dot_product_attention(
            t(q[q0:q0 + nq]), t(kk), t(vv), scale=0.15)[0].numpy().transpose(1, 0, 2)
        worst = max(worst, float(np.max(np.abs(got3[lo:lo + nq] - sd))))
    # (v) no key
    rows4, got4 = Ox.attention_groups(q, k, v, kc, vc, [(0, 4, 0, 0, 0, 0)], 0.2)
    worst = max(worst, float(np.max(np.abs(got4))), 0.0 if list(rows4) == [0, 1, 2, 3] else 1.0)
    return worst


def pin_block_means(Ox):
    """Rows holding their own index: a full block's mean is b*B + (B-1)/2, the
    partial last block's mean is the mean of its valid row indices."""
    B, n = 8, 29
    x = np.repeat(np.arange(32, dtype=np.float64)[:, None, None], 2, axis=1).repeat(3, axis=2)
    m = Ox.block_means(x, n, B)
    exp = np.array([b * B + (B - 1) / 2 for b in range(3)] + [(24 + 28) / 2])
    return float(np.max(np.abs(m[:, 0, 0] - exp))) + (0.0 if m.shape == (4, 2, 3) else 1.0)


def pin_block_selection(Ox):
    """Hand-worked rows (tau = 0.9): scores (0, 0, 0, 3, 4) have mean 1.4 and
    population std sqrt(3.04) = 1.7436, threshold 2.969 -> blocks 3 and 4
    (a sample std would give 3.154 and drop block 3).  A constant row keeps
    nothing above its mean: only the sinks.  Prefix query blocks keep all."""
    s = np.array([[[0.0, 0, 0, 3, 4], [2.0, 2, 2, 2, 2], [0.0, 0, 0, 3, 4]]])
    keep = Ox.select_blocks(s, 0.9, 0)
    worst = 0.0 if (keep[0, 0].tolist() == [False, False, False, True, True] and
                    not keep[0, 1].any()) else 1.0
    keep1 = Ox.select_blocks(s, 0.9, 1)
    worst += 0.0 if (keep1[0, 0].all() and keep1[0, 1].tolist() == [True, False, False, False, False]
                     and keep1[0, 2].tolist() == [True, False, False, True, True]) else 1.0
    # larger tau keeps a subset
    r = np.random.default_rng(11).standard_normal((2, 6, 40))
    a, b = Ox.select_blocks(r, 1.0, 2), Ox.select_blocks(r, 1.5, 2)
    worst += 0.0 if (b <= a).all() and a.sum() > b.sum() else 1.0
    return worst


def pin_block_sparse_attention(Ox):
    """All blocks kept = dense attention; one block kept = SDPA over exactly
    that block's keys; scores are the scaled dot of the block means."""
    rng = np.random.default_rng(12)
    B, n, H = 16, 70, 2
    q = rng.standard_normal((80, H, 128)); k = rng.standard_normal((80, H, 128))
    v = rng.standard_normal((80, H, 128))
    nb = 5
    keep = np.ones((H, nb, nb), bool)
    got = Ox.block_sparse_attention(q, k, v, n, keep, B, 0.1)
    dense = Ox.attention(q, k, v, [0, 80], [0, 80], [n], 0.1)
    worst = float(np.max(np.abs(got - dense)))
    keep = np.zeros((H, nb, nb), bool)
    keep[:, :, 4] = True                       # only the partial last block (rows 64..69)
    got = Ox.block_sparse_attention(q, k, v, n, keep, B, 0.1)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.transpose(1, 0, 2)))[None]
    sd = torch.nn.functional.scaled_dot_product_attention(
        t(q[:n]), t(k[64:n]), t(v[64:n]), scale=0.1)[0].numpy().transpose(1, 0, 2)
    worst = max(worst, float(np.max(np.abs(got[:n] - sd))), float(np.max(np.abs(got[n:]))))
    qm, km = np.zeros((2, 1, 128)), np.zeros((3, 1, 128))
    qm[0, 0, 0], qm[1, 0, 1], km[2, 0, 0], km[1, 0, 1] = 2.0, 3.0, 5.0, -1.0
    sc = Ox.block_scores(qm, km, 0.5)
    exp = np.array([[[0, 0, 5.0], [0, -1.5, 0]]])
    return max(worst, float(np.max(np.abs(sc - exp))))


def pin_wire_layout(Ox):
    """Hand-checked element of the destination-major packing, and the head
    merge inverts it per tensor."""
    rows, H, D = 2, 4, 3
    idx = lambda t: np.arange(rows * H * D, dtype=np.float64).reshape(rows, H, D) + 100 * t
    q, k, v = idx(0), idx(1), idx(2)
    p = Ox.pack_qkv(q, k, v, 2)                  # [2 dest, 2 rows, 2 heads, 3, D]
    worst = 0.0 if (p.shape == (2, 2, 2, 3, 3) and p[1, 0, 1, 2, 1] == v[0, 3, 1]
                    and p[0, 1, 0, 1, 2] == k[1, 0, 2]) else 1.0
    for t_, x in enumerate((q, k, v)):
        worst += float(np.max(np.abs(Ox.merge_heads(p[:, :, :, t_, :]) - x)))
    return worst


def pin_ue5m3_int8(Ox):
    """UE5M3 values by hand; the scale code is the smallest with 127 * s >=
    amax; int8 group quantisation errs by at most s/2 and a group's largest
    element lands on |q| >= 112 (consecutive codes differ by <= 1.125x)."""
    vals = Ox.ue5m3_value(np.array([0, 0x78, 0x79, 0x7F, 0x80, 0xFF]))
    exp = np.array([2.0 ** -15, 1.0, 1.125, 1.875, 2.0, 2.0 ** 16 * 1.875])
    worst = float(np.max(np.abs(vals - exp)))
    amax = np.exp(np.random.default_rng(13).uniform(-9, 14, 2000))
    c = Ox.ue5m3_scale_code(amax)
    ok = (127 * Ox.ue5m3_value(c) >= amax) & ((c == 0) | (127 * Ox.ue5m3_value(np.maximum(c - 1, 0)) < amax))
    worst += 0.0 if ok.all() else 1.0
    x = np.random.default_rng(14).standard_normal((50, 128)) * 3
    x[0, :32] = 0.0
    q, codes = Ox.int8_group32(x)
    dec = Ox.int8_group32_decode(q, codes)
    s = np.repeat(Ox.ue5m3_value(codes), 32, axis=-1)
    worst += float(np.max(np.maximum(np.abs(dec - x) - s / 2, 0)))
    big = np.abs(q.astype(np.int64)).reshape(50, 4, 32).max(-1)
    worst += 0.0 if (big[1:] >= 112).all() and (dec[0, :32] == 0).all() else 1.0
    return worst


def pin_e4m3(Ox):
    """E4M3 by hand (subnormal 2^-9, the 240/248/256 tie, saturation at 448)
    and against torch's float8_e4m3fn conversion inside its finite range."""
    x = np.array([2.0 ** -9, 2.0 ** -10, 240.0, 248.0, 464.0, 500.0, -1e6, 1.0])
    exp = np.array([2.0 ** -9, 0.0, 240.0, 256.0, 448.0, 448.0, -448.0, 1.0])
    worst = float(np.max(np.abs(Ox.e4m3_round(x) - exp)))
    bits = Ox.e4m3_bits(Ox.e4m3_round(np.array([2.0 ** -9, 240.0, 256.0, 448.0, -1.0])))
    worst += 0.0 if list(bits) == [0x01, 0x77, 0x78, 0x7E, 0xB8] else 1.0
    y = np.random.default_rng(15).standard_normal(20000) * np.exp(np.random.default_rng(16).uniform(-9, 5, 20000))
    y = torch.from_numpy(y).to(torch.bfloat16).double().numpy()
    y = y[np.abs(y) <= 464.0]  # torch's cast is finite (saturating) only up to 464
    ref = torch.from_numpy(y).float().to(torch.float8_e4m3fn)
    worst += float(np.max(np.abs(Ox.e4m3_round(y) - ref.double().numpy())))
    worst += 0.0 if np.array_equal(Ox.e4m3_bits(Ox.e4m3_round(y)), ref.view(torch.uint8).numpy()) else 1.0
    return worst


def pin_wire_records(Ox):
    """Record layouts: value bytes, scale codes and zero padding in place."""
    rng = np.random.default_rng(17)
    q, k, v = (rng.standard_normal((3, 2, 128)) for _ in range(3))
    r = Ox.qkv_int8_records(q, k, v)
    vals, codes = Ox.int8_group32(k)
    worst = 0.0 if (r.shape == (3, 2, 400) and (r[..., 396:] == 0).all() and
                    np.array_equal(r[..., 128:256], vals.view(np.uint8)) and
                    np.array_equal(r[..., 388:392], codes)) else 1.0
    o = Ox.out_int8_records(q)
    worst += 0.0 if o.shape == (3, 2, 144) and (o[..., 132:] == 0).all() else 1.0
    f = Ox.out_fp8_records(q)
    worst += 0.0 if f.shape == (3, 2, 128) and f.dtype == np.uint8 else 1.0
    return worst


def pin_int8_ties_and_clamp(Ox):
    """Block-INT8 quantiser by hand (Sol-H3 section 3.2 "Quantized
    communication"; the tie and clamp rules are the reading taken there).

    A group whose largest magnitude is 126.5 * 1.125 takes code 0x79
    (127 * 1.0 < 142.3125 <= 127 * 1.125), so every value below is an exact
    multiple of s = 1.125; exact half-integer quotients round to the even
    integer: +-0.5 -> 0, +-1.5 -> +-2, +-2.5 -> +-2, +-3.5 -> +-4,
    +-126.5 -> +-126.  A second group at code 0x80 (s = 2) repeats a tie at a
    different scale.  A group past the largest code (255, value 122880) is
    clamped to the symmetric range: +-127, never -128."""
    s = 1.125
    quot = [0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 3.5, -3.5, 126.5, -126.5, 0.25, 100.75, -7.0]
    want = [0, 0, 2, -2, 2, -2, 4, -4, 126, -126, 0, 101, -7]
    x = np.zeros((1, 128))
    x[0, :len(quot)] = np.array(quot) * s
    # group 1: s = 2 (amax 125.5 * 2 = 251 lies in (127 * 1.875, 127 * 2])
    x[0, 32:36] = np.array([125.5, 0.5, -4.5, 9.0]) * 2.0
    want1 = [126, 0, -4, 9]
    # group 2: code 255, value 2^16 * 1.875 = 122880; 127 * value = 15,605,760
    x[0, 64:70] = [2.0e7, -2.0e7, -1.6e7, 15605760.0, -15605760.0, 122880.0 * 126.5]
    want2 = [127, -127, -127, 127, -127, 126]
    vals, codes = Ox.int8_group32(x)
    v = vals.astype(np.int64)[0]
    ok = (list(codes[0]) == [0x79, 0x80, 0xFF, 0x00] and list(v[:len(want)]) == want and
          list(v[32:36]) == want1 and list(v[64:70]) == want2 and
          not v[len(want):32].any() and not v[96:].any())
    return 0.0 if ok else 1.0


def _record_vector():
    """One 128-channel vector with a known INT8 encoding, group by group:
    group 0 at s = 1 (code 0x78), group 1 at s = 2 (0x80), group 2 at
    s = 1.125 (0x79), group 3 at s = 0.5 (0x70); each group's largest
    magnitude is exactly 127 * s, so its code is the one named."""
    x = np.zeros(128)
    x[0:4] = [127.0, -127.0, 3.0, -5.0]                 # -> 7F 81 03 FB
    x[32:36] = [254.0, 14.0, -1.0, 3.0]                 # -> 7F 07 00 02 (-0.5, 1.5 are ties)
    x[64:66] = [-127 * 1.125, 11.25]                    # -> 81 0A
    x[96], x[127] = 63.5, -0.75                         # -> 7F FE
    vbytes = np.zeros(128, dtype=np.uint8)
    vbytes[0:4] = [0x7F, 0x81, 0x03, 0xFB]
    vbytes[32:36] = [0x7F, 0x07, 0x00, 0x02]
    vbytes[64:66] = [0x81, 0x0A]
    vbytes[96], vbytes[127] = 0x7F, 0xFE
    return x, vbytes, [0x78, 0x80, 0x79, 0x70]


def pin_int8_record_bytes(Ox):
    """Output and QKV INT8 records byte by byte, expected bytes written out
    by hand (Sol-H3 section 3.2 "Quantized communication"; record layout as
    read there): output record = 128 value bytes, the 4 group codes in
    channel order at bytes 128-131, 12 zero bytes; QKV record = q, k, v value
    bytes, then q's 4 codes, k's 4 codes, v's 4 codes (bytes 384-395), then
    4 zero bytes.  k = 2x and v = x/2 keep every quotient (so the value
    bytes) and move each code by one exponent step (+-8)."""
    x, vbytes, codes = _record_vector()
    o = Ox.out_int8_records(x[None, None, :])[0, 0]
    want = np.zeros(144, dtype=np.uint8)
    want[:128] = vbytes
    want[128:132] = codes
    worst = 0.0 if (o.shape == (144,) and np.array_equal(o, want)) else 1.0
    r = Ox.qkv_int8_records(x[None, None, :], 2.0 * x[None, None, :], 0.5 * x[None, None, :])[0, 0]
    want = np.zeros(400, dtype=np.uint8)
    want[0:128] = want[128:256] = want[256:384] = vbytes
    want[384:388] = codes
    want[388:392] = [c + 8 for c in codes]
    want[392:396] = [c - 8 for c in codes]
    worst += 0.0 if (r.shape == (400,) and np.array_equal(r, want)) else 1.0
    return worst


def pin_block_sparse_empty_list(Ox):
    """Sol-H3 section 3.4, "Safety rails and the exact prefix KV sink": with
    no prefix a query block's list may be empty (a constant score row keeps
    nothing above its mean); its rows then output exactly 0 (the reading
    taken for a query with no key), while the other blocks attend normally."""
    rng = np.random.default_rng(18)
    B, n, H = 8, 30, 2
    q, k, v = (rng.standard_normal((32, H, 128)) for _ in range(3))
    nb = 4
    keep = np.ones((H, nb, nb), bool)
    keep[0, 1] = False                          # head 0, query block 1 (rows 8..15)
    keep[1, 3] = False                          # head 1, the partial last block (rows 24..29)
    got = Ox.block_sparse_attention(q, k, v, n, keep, B, 0.1)
    dense = Ox.attention(q, k, v, [0, 32], [0, 32], [n], 0.1)
    worst = 0.0 if (np.all(got[8:16, 0] == 0.0) and np.all(got[24:30, 1] == 0.0)) else 1.0
    mask = np.ones((32, H), bool)
    mask[8:16, 0] = mask[24:30, 1] = False
    mask[n:] = False
    worst += float(np.max(np.abs(got - dense)[mask]))
    return worst


def pin_softmax_rows(Ox):
    rng = np.random.default_rng(7)
    s = rng.standard_normal((9, 300)) * 40.0
    p = Ox.softmax_rows(s)
    # rows sum to 1; ratios follow exp of score differences
    worst = float(np.max(np.abs(p.sum(-1) - 1.0)))
    ratio = np.log(p[:, 1] / p[:, 0]) - (s[:, 1] - s[:, 0])
    return max(worst, float(np.max(np.abs(ratio))))


def pin_round_bf16(Ox):
    """bf16 rounding: hand-derived ties and overflow, fp32-exact values
    against torch's own fp32 -> bf16 conversion."""
    cases = {1.0 + 2.0 ** -8: 1.0, 1.0 + 3 * 2.0 ** -8: 1.0 + 2.0 ** -6,
             1.0 + 2.0 ** -8 + 2.0 ** -30: 1.0 + 2.0 ** -7, -(1.0 + 2.0 ** -8): -1.0,
             3.0e38: 2.0 ** 127 * (226 / 128), 3.4e38: math.inf, 0.0: 0.0,
             2.0 ** -140: 2.0 ** -140 if 2.0 ** -140 >= 2.0 ** -133 else 0.0}
    worst = 0.0
    for x, want in cases.items():
        got = float(Ox.round_bf16(np.array([x]))[0])
        worst = max(worst, 0.0 if got == want else 1.0)
    x = np.random.default_rng(8).standard_normal(20000).astype(np.float32).astype(np.float64) * 37.0
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    worst = max(worst, float(np.max(np.abs(Ox.round_bf16(x) - ref))))
    return worst


def pin_lora_prologue(Ox):
    """delta = 0 reduces to the plain prologue; otherwise the fused result is
    the prologue of the bf16-rounded sum, checked against the brute force."""
    inp, f = _tiny_inputs()
    pos = inp["pos_thw"].numpy()
    z = Ox.qk_norm_rope_lora(f["q"], np.zeros_like(f["q"]), f["wq"], pos, SECTIONS, THETA, EPS)
    worst = float(np.max(np.abs(z - Ox.qk_norm_rope(f["q"], f["wq"], pos, SECTIONS, THETA, EPS))))
    delta = np.random.default_rng(9).standard_normal(f["q"].shape) * 0.05
    got = Ox.qk_norm_rope_lora(f["q"], delta, f["wq"], pos, SECTIONS, THETA, EPS)
    for r in (0, 100, 200, 249):
        for h in range(2):
            exp = brute.norm_rope_lora_row(list(f["q"][r, h]), list(delta[r, h]), list(f["wq"][h]),
                                           tuple(int(v) for v in pos[r]), SECTIONS, THETA, EPS)
            worst = max(worst, float(np.max(np.abs(got[r, h] - np.array(exp)))))
    return worst


PINS = [
    (pin_norm_closed_form, 1e-12),
    (pin_norm_scale_invariance, 1e-12),
    (pin_rope_closed_forms, 1e-12),
    (pin_rope_invariants, 1e-10),
    (pin_prologue_brute, 1e-12),
    (pin_attention_brute, 1e-12),
    (pin_attention_closed_forms, 1e-12),
    (pin_attention_sdpa, 1e-12),
    (pin_attention_grouped_sdpa, 1e-12),
    (pin_attention_invariants, 1e-12),
    (pin_softmax_rows, 1e-9),
    (pin_round_bf16, 0.0),
    (pin_attention_groups, 1e-12),
    (pin_block_means, 0.0),
    (pin_block_selection, 0.0),
    (pin_block_sparse_attention, 1e-12),
    (pin_wire_layout, 0.0),
    (pin_ue5m3_int8, 1e-12),
    (pin_e4m3, 0.0),
    (pin_wire_records, 0.0),
    (pin_int8_ties_and_clamp, 0.0),
    (pin_int8_record_bytes, 0.0),
    (pin_block_sparse_empty_list, 1e-12),
    (pin_lora_prologue, 1e-12),
]


@pytest.mark.parametrize("pin,bound", PINS, ids=[p.__name__ for p, _ in PINS])
def test_pin(pin, bound):
    assert pin(O) <= bound


# ---------------------------------------------------- planted mistakes
def _mutant(**overrides):
    ns = types.SimpleNamespace(**{n: getattr(O, n) for n in dir(O) if not n.startswith("__")})
    for name, fn in overrides.items():
        setattr(ns, name, fn)
    # re-bind composite functions so they call the mutated parts
    def qk_norm_rope(x, w, pos, sections=SECTIONS, theta=THETA, eps=EPS):
        return ns.rope_axial(ns.rms_norm(x, w[None], eps), pos, sections, theta)

    def attention(q, k, v, cu_q, cu_kv, vl, scale, rows=None, block=256):
        if "attention" in overrides:
            return overrides["attention"](q, k, v, cu_q, cu_kv, vl, scale, rows)
        saved = O.softmax_rows
        try:
            O.softmax_rows = ns.softmax_rows
            return O.attention(q, k, v, cu_q, cu_kv, vl, scale, rows, block)
        finally:
            O.softmax_rows = saved
    if "qk_norm_rope" not in overrides:
        ns.qk_norm_rope = qk_norm_rope

    def qk_norm_rope_lora(base, delta, w, pos, sections=SECTIONS, theta=THETA, eps=EPS):
        return ns.qk_norm_rope(ns.round_bf16(base + delta), w, pos, sections, theta, eps)
    if "qk_norm_rope_lora" not in overrides:
        ns.qk_norm_rope_lora = qk_norm_rope_lora

    def int8_group32(x):
        g = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
        codes = ns.ue5m3_scale_code(np.abs(g).max(axis=-1))
        s = ns.ue5m3_value(codes)[..., None]
        vals = np.clip(np.rint(g / s), -127, 127).astype(np.int8)
        return vals.reshape(x.shape), codes.astype(np.uint8)
    if "int8_group32" not in overrides:
        ns.int8_group32 = int8_group32
    ns.attention = attention
    return ns


def _rope_sign_flip(y, pos, sections=SECTIONS, theta=THETA):
    return O.rope_axial(y, -np.asarray(pos), sections, theta)


def _rope_rotate_half(y, pos, sections=SECTIONS, theta=THETA):
    out = y.copy(); off = 0
    for a, d in enumerate(sections):
        inv = O.rope_inverse_frequencies(d, theta)
        phi = pos[:, a][:, None] * inv[None]
        c, s = np.cos(phi)[:, None], np.sin(phi)[:, None]
        y0, y1 = y[..., off:off + d // 2], y[..., off + d // 2:off + d]
        out[..., off:off + d // 2] = y0 * c - y1 * s
        out[..., off + d // 2:off + d] = y0 * s + y1 * c
        off += d
    return out


def _rope_shared_base(y, pos, sections=SECTIONS, theta=THETA):
    # frequencies from the full head width instead of each axis' own width
    out = y.copy(); off = 0
    for a, d in enumerate(sections):
        j = np.arange(d // 2)
        phi = pos[:, a][:, None] * (theta ** (-2.0 * j / 128.0))[None]
        c, s = np.cos(phi)[:, None], np.sin(phi)[:, None]
        y0, y1 = y[..., off:off + d:2], y[..., off + 1:off + d:2]
        out[..., off:off + d:2] = y0 * c - y1 * s
        out[..., off + 1:off + d:2] = y0 * s + y1 * c
        off += d
    return out


def _rope_axis_swap(y, pos, sections=SECTIONS, theta=THETA):
    return O.rope_axial(y, np.asarray(pos)[:, [1, 0, 2]], sections, theta)


def _norm_eps_outside(x, w, eps):
    return x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps) * w


def _norm_no_weight(x, w, eps):
    return O.rms_norm(x, np.ones_like(w), eps)


def _norm_sum_not_mean(x, w, eps):
    return x / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps) * w


def _softmax_no_norm(s):
    return np.exp(s - np.max(s, -1, keepdims=True))


def _attn_transposed(q, k, v, cu_q, cu_kv, vl, scale, rows=None):
    # uses V^T-like mixing: weights over queries instead of keys
    return O.attention(k, q, v, cu_kv, cu_q, vl, scale, rows)


def _attn_no_scale(q, k, v, cu_q, cu_kv, vl, scale, rows=None):
    return O.attention(q, k, v, cu_q, cu_kv, vl, 1.0, rows)


def _attn_pad_keys(q, k, v, cu_q, cu_kv, vl, scale, rows=None):
    # attends over the whole buffer, padded keys included
    return O.attention(q, np.nan_to_num(k), np.nan_to_num(v), cu_q, cu_kv, None, scale, rows)


def _round_trunc(x):
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    q = np.ldexp(1.0, e - 8)
    return np.trunc(x / q) * q


def _round_half_up(x):
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    q = np.ldexp(1.0, e - 8)
    return np.floor(x / q + 0.5) * q


def _groups_ignore_cache(q, k, v, kc, vc, groups, scale, rows=None):
    return O.attention_groups(q, k, v, kc, vc, [g[:4] + (0, 0) for g in groups], scale, rows)


def _select_sample_std(scores, tau, n_prefix):
    mu = scores.mean(-1, keepdims=True)
    sd = scores.std(-1, ddof=1, keepdims=True)
    keep = scores > mu + tau * sd
    keep[:, :, :n_prefix] = True
    keep[:, :n_prefix, :] = True
    return keep


def _select_ge(scores, tau, n_prefix):
    keep = scores >= scores.mean(-1, keepdims=True) + tau * scores.std(-1, keepdims=True)
    keep[:, :, :n_prefix] = True
    keep[:, :n_prefix, :] = True
    return keep


def _select_no_sink(scores, tau, n_prefix):
    keep = scores > scores.mean(-1, keepdims=True) + tau * scores.std(-1, keepdims=True)
    keep[:, :n_prefix, :] = True
    return keep


def _block_sums(x, n_rows, block):
    return O.block_means(x, n_rows, block) * block


def _scale_code_down(amax):
    c = O.ue5m3_scale_code(amax)
    return np.maximum(c - 1, 0)


def _e4m3_no_saturation(x):
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    q = np.ldexp(1.0, np.maximum(e, -5) - 4)
    return np.rint(x / q) * q


def _pack_tensor_major(q, k, v, n_dest):
    rows, H, D = q.shape
    x = np.stack([q, k, v], axis=0).reshape(3, rows, n_dest, H // n_dest, D)
    return x.transpose(2, 1, 3, 0, 4).reshape(n_dest, rows, 3, H // n_dest, D).transpose(0, 1, 3, 2, 4)


def _lora_no_round(base, delta, w, pos, sections=SECTIONS, theta=THETA, eps=EPS):
    return O.qk_norm_rope(base + delta, w, pos, sections, theta, eps)


def _int8_half_up(x):
    g = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
    codes = O.ue5m3_scale_code(np.abs(g).max(axis=-1))
    s = O.ue5m3_value(codes)[..., None]
    vals = np.clip(np.floor(g / s + 0.5), -127, 127).astype(np.int8)
    return vals.reshape(x.shape), codes.astype(np.uint8)


def _int8_clip_asymmetric(x):
    g = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
    codes = O.ue5m3_scale_code(np.abs(g).max(axis=-1))
    s = O.ue5m3_value(codes)[..., None]
    vals = np.clip(np.rint(g / s), -128, 127).astype(np.int8)
    return vals.reshape(x.shape), codes.astype(np.uint8)


def _out_codes_reversed(o):
    rec = O.out_int8_records(o)
    rec[..., 128:132] = rec[..., 128:132][..., ::-1].copy()
    return rec


def _sparse_empty_attends_all(q, k, v, n_rows, keep, block, scale, rows=None):
    keep = keep.copy()
    empty = ~keep.any(-1)
    keep[empty] = True
    return O.block_sparse_attention(q, k, v, n_rows, keep, block, scale, rows)


MUTANTS = {
    "rope_sign_flip": dict(rope_axial=_rope_sign_flip),
    "rope_rotate_half": dict(rope_axial=_rope_rotate_half),
    "rope_shared_base": dict(rope_axial=_rope_shared_base),
    "rope_axis_swap": dict(rope_axial=_rope_axis_swap),
    "norm_eps_outside": dict(rms_norm=_norm_eps_outside),
    "norm_no_weight": dict(rms_norm=_norm_no_weight),
    "norm_sum_not_mean": dict(rms_norm=_norm_sum_not_mean),
    "softmax_no_norm": dict(softmax_rows=_softmax_no_norm),
    "attn_transposed": dict(attention=_attn_transposed),
    "attn_no_scale": dict(attention=_attn_no_scale),
    "attn_pad_keys": dict(attention=_attn_pad_keys),
    "round_truncates": dict(round_bf16=_round_trunc),
    "round_half_up": dict(round_bf16=_round_half_up),
    "lora_skips_rounding": dict(qk_norm_rope_lora=_lora_no_round),
    "groups_ignore_cache": dict(attention_groups=_groups_ignore_cache),
    "select_sample_std": dict(select_blocks=_select_sample_std),
    "select_ge": dict(select_blocks=_select_ge),
    "select_no_sink": dict(select_blocks=_select_no_sink),
    "block_sums": dict(block_means=_block_sums),
    "scale_code_rounds_down": dict(ue5m3_scale_code=_scale_code_down),
    "e4m3_no_saturation": dict(e4m3_round=_e4m3_no_saturation),
    "pack_tensor_major": dict(pack_qkv=_pack_tensor_major),
    "int8_rounds_half_up": dict(int8_group32=_int8_half_up),
    "int8_clips_to_minus_128": dict(int8_group32=_int8_clip_asymmetric),
    "out_record_codes_reversed": dict(out_int8_records=_out_codes_reversed),
    "sparse_empty_list_attends_all": dict(block_sparse_attention=_sparse_empty_attends_all),
}


def _pins_pass(Ox):
    for pin, bound in PINS:
        try:
            val = pin(Ox)
        except Exception:
            return False
        if not (val <= bound):
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    assert _pins_pass(_mutant()), "unmutated copy must pass"
    assert not _pins_pass(_mutant(**MUTANTS[name])), f"mutant {name} slipped through"


# ------------------------------------------------------ pages' own numbers
def test_workload_shapes_match_pages():
    g = json.load(open(os.path.join(HERE, "golden", "workload_shapes.json")))
    full = W.workload("full")
    assert full.segments[0].valid == g["packed_sequence"]["valid_tokens"]
    assert full.segments[0].q_rows == g["packed_sequence"]["buffer_tokens"]
    assert full.n_heads * full.head_dim == g["hidden_width"]["value"]
    assert full.head_dim == g["projection_channels"]["value"]


def test_workload_flops_and_bytes():
    # 4 * H * D * L^2 over valid tokens
    assert W.workload("full").attention_flops() == 4 * 42 * 128 * 58758 ** 2
    assert abs(W.workload("grouped_chunk").attention_flops() - 7.255e12) / 7.255e12 < 1e-3
    assert abs(W.workload("full").prologue_bytes() - 2.527e9) / 2.527e9 < 1e-3


def test_positions_layout():
    pos = W.positions(W.workload("tiny")).numpy()
    # video grid (2, 8, 8) t-major, then audio (i,0,0), then text (i,0,0), pad 0
    assert tuple(pos[0]) == (0, 0, 0) and tuple(pos[9]) == (0, 1, 1)
    assert tuple(pos[127]) == (1, 7, 7)
    assert tuple(pos[128]) == (0, 0, 0) and tuple(pos[191]) == (63, 0, 0)
    assert tuple(pos[192]) == (0, 0, 0) and tuple(pos[249]) == (57, 0, 0)
    assert (pos[250:] == 0).all()


def test_inputs_deterministic_and_padded():
    a = W.make_inputs("tiny")
    b = W.make_inputs("tiny")
    assert torch.equal(a["q"].view(torch.int16), b["q"].view(torch.int16))
    c = W.make_inputs("tiny", fill="B")
    assert torch.isnan(c["k"][250:].float()).any() and torch.isinf(c["v"][250:].float()).any()
    assert torch.equal(a["q"][:250].view(torch.int16), c["q"][:250].view(torch.int16))
    assert torch.isnan(a["out"].float()).all()


def test_attention_medium_against_sdpa():
    """Library cross-check at the multi-tile size: the 4,000-valid-row,
    42-head packed sequence (32 key tiles of 128 rows, a ragged last one),
    prologue included, against torch SDPA in float64 on the CPU, head by
    head over every valid row (the packed sequence and valid length of the
    vLLM-Omni blog section 3.1)."""
    inp = W.make_inputs("medium")
    n = inp["valid_len"][0]
    pos = inp["pos_thw"].numpy()[:n]
    q = O.qk_norm_rope(O.widen(inp["q"][:n]), O.widen(inp["wq"]), pos, SECTIONS, THETA, EPS)
    k = O.qk_norm_rope(O.widen(inp["k"][:n]), O.widen(inp["wk"]), pos, SECTIONS, THETA, EPS)
    v = O.widen(inp["v"][:n])
    pad = np.full((inp["q"].shape[0] - n,) + q.shape[1:], np.nan)
    got = O.attention(np.concatenate([q, pad]), np.concatenate([k, pad]),
                      np.concatenate([v, pad]), inp["cu_seqlens_q"], inp["cu_seqlens_kv"],
                      inp["valid_len"], SCALE)
    assert np.all(got[n:] == 0.0)
    worst = 0.0
    for h in range(q.shape[1]):
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a[:, h]))[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=SCALE)
        worst = max(worst, float(np.max(np.abs(got[:n, h] - ref[0, 0].numpy()))))
    assert worst <= 1e-12, worst
