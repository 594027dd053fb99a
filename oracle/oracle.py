"""fp64 CPU oracle for packed-sequence attention and its fused Q/K prologue.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import or run this module.
The CUDA product path never calls it and shares no code with it.

What is computed, with the passage each step follows:

* ``qk_norm_rope`` -- "QK normalization with partial RoPE", operator group 2
  of Sol-H3 (arXiv 2609.35110) section 3.5 "Kernel Fusion", and the fused
  Q/K RMSNorm + RoPE of the vLLM-Omni blog ("MiniMax H3 on vLLM-Omni"),
  section 3.2 "fused DiT operators".  Per (row, head): RMSNorm over the
  head's 128 channels with a per-head weight, eps inside the square root,
  then an axial 3-D rotary embedding with sections (t, h, w) of widths
  (32, 48, 48); channels past the rotary sections pass through.
* ``attention`` -- exact softmax(Q K^T * scale) V per packed sequence or
  query group and per head: the packed joint sequence and valid length of
  the vLLM-Omni blog section 3.1 (the backend receives the valid length, the
  suffix padding is removed), the flat (total, heads, head_dim) layout of
  Sol-H3 section 3.2 "Optimized attention collectives", and the grouped
  condition / audio / video query ranges of the SolarWM-H3 Realtime blog,
  stage 2 "Attention Backend".
* ``attention_groups`` -- query groups over KV views into the current K/V
  and a cached K/V range (Sol-H3 reference KV caching, Fig. 4; SolarWM
  history K/V reuse).
* ``qk_norm_rope_lora`` / ``round_bf16`` -- the LoRA consumer fusion of
  Sol-H3 section 3.5 (base + delta rounded to bf16 before the prologue).
* block-sparse attention (``block_means`` ... ``block_sparse_attention``) --
  Sol-Attn with the exact prefix KV sink, Sol-H3 section 3.4.
* wire formats (``pack_qkv``, ``merge_heads``, the INT8 / FP8 records) --
  Sol-H3 section 3.2, optimized and quantized attention collectives.

Readings taken where the pages are silent (each listed in the design notes):
RMSNorm per head (128 channels) with weight [H, 128]; eps inside the root;
norm before rotation; rotary pairs are adjacent channels (2j, 2j+1) inside
each section; pair j of a section of width d turns by pos * theta^(-2j/d);
padded query rows and query rows with no valid key produce zeros.

All arithmetic is float64 on exactly widened bf16 inputs; there is no
intermediate rounding.  Matrix products and exp use NumPy as library
primitives, with no blocking beyond splitting query rows into independent
blocks (each output row depends on its own query row only).
"""
from __future__ import annotations

import numpy as np

DEFAULT_SECTIONS = (32, 48, 48)
DEFAULT_THETA = 10000.0
DEFAULT_EPS = 1e-6


def widen(t) -> np.ndarray:
    """bf16 / fp32 tensor or array -> float64 ndarray (exact for bf16)."""
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    # torch tensor (any device); bf16 -> fp32 -> fp64 is exact.
    return t.detach().to("cpu").float().numpy().astype(np.float64)


# ---------------------------------------------------------------- prologue
def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """y_c = x_c / sqrt(mean_c(x_c^2) + eps) * w_c over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_inverse_frequencies(width: int, theta: float) -> np.ndarray:
    """theta^(-2j/width) for the width/2 pairs of one axis section."""
    j = np.arange(width // 2, dtype=np.float64)
    return theta ** (-2.0 * j / width)


def rope_axial(y: np.ndarray, pos: np.ndarray,
               sections=DEFAULT_SECTIONS, theta=DEFAULT_THETA) -> np.ndarray:
    """Rotate adjacent channel pairs of y [n, H, D] by per-axis angles.

    Section a (t, h or w) covers channels [off_a, off_a + d_a); its pair j is
    (off_a + 2j, off_a + 2j + 1) and turns by phi = pos[:, a] *
    theta^(-2j/d_a):  (y0, y1) -> (y0 cos phi - y1 sin phi,
    y0 sin phi + y1 cos phi).
    """
    out = y.copy()
    off = 0
    for a, d in enumerate(sections):
        if d == 0:
            continue
        inv = rope_inverse_frequencies(d, theta)                # [d/2]
        phi = pos[:, a].astype(np.float64)[:, None] * inv[None, :]
        c = np.cos(phi)[:, None, :]                              # [n,1,d/2]
        s = np.sin(phi)[:, None, :]
        y0 = y[..., off:off + d:2]
        y1 = y[..., off + 1:off + d:2]
        out[..., off:off + d:2] = y0 * c - y1 * s
        out[..., off + 1:off + d:2] = y0 * s + y1 * c
        off += d
    return out


def qk_norm_rope(x: np.ndarray, w: np.ndarray, pos: np.ndarray,
                 sections=DEFAULT_SECTIONS, theta=DEFAULT_THETA,
                 eps=DEFAULT_EPS) -> np.ndarray:
    """x [n, H, D] float64, w [H, D] float64, pos [n, 3] int -> [n, H, D]."""
    assert sum(sections) <= x.shape[-1]
    y = rms_norm(x, w[None, :, :], eps)
    return rope_axial(y, pos, sections, theta)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significant bits,
    8-bit exponent), ties to even, as float64.  Values beyond the largest
    finite bf16 become +-inf; the subnormal range keeps a fixed quantum of
    2^-133."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0)
    m, e = np.frexp(x[finite])                 # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                    # below 2^-126 the quantum stays 2^-133
    q = np.ldexp(1.0, e - 8)                   # value of one unit in the last place
    r = np.rint(x[finite] / q) * q             # rint rounds half to even
    big = np.abs(r) >= np.ldexp(1.0, 128)      # past the largest finite bf16
    r[big] = np.copysign(np.inf, r[big])
    out[finite] = r
    return out


def qk_norm_rope_lora(base: np.ndarray, delta: np.ndarray, w: np.ndarray, pos: np.ndarray,
                      sections=DEFAULT_SECTIONS, theta=DEFAULT_THETA,
                      eps=DEFAULT_EPS) -> np.ndarray:
    """LoRA consumer fusion (Sol-H3 section 3.5 "Precision-preserving LoRA
    fusion"): the consumer rounds base + delta to bf16 before the Q/K
    normalisation and RoPE, exactly where the separate branches would store
    the sum; the rest is ``qk_norm_rope`` on that rounded sum."""
    return qk_norm_rope(round_bf16(base + delta), w, pos, sections, theta, eps)


# --------------------------------------------------------------- attention
def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row-wise softmax of a float64 score block (max-subtracted)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
              cu_seqlens_q, cu_seqlens_kv, valid_len, scale: float,
              rows=None, block: int = 256) -> np.ndarray:
    """Non-causal attention per segment and head.

    q [Rq, H, D], k / v [Rkv, H, D] float64.  Segment b owns query rows
    [cu_q[b], cu_q[b+1]) and key rows [cu_kv[b], cu_kv[b+1]).  With
    ``valid_len`` given, only the first valid_len[b] rows of each range are
    valid (queries and keys alike); otherwise all rows are.  Output rows that
    are padded, or whose segment has no valid key, are 0.

    ``rows`` selects global query-row indices to compute (default: all);
    the result has one output row per selected row, in that order.
    """
    Rq, H, D = q.shape
    if rows is None:
        rows = np.arange(Rq)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, H, D), dtype=np.float64)
    n_seg = len(cu_seqlens_q) - 1
    for b in range(n_seg):
        q0, q1 = cu_seqlens_q[b], cu_seqlens_q[b + 1]
        k0, k1 = cu_seqlens_kv[b], cu_seqlens_kv[b + 1]
        nq, nkv = q1 - q0, k1 - k0
        if valid_len is not None:
            nq = nkv = valid_len[b]
        sel = np.nonzero((rows >= q0) & (rows < q0 + nq))[0]
        if sel.size == 0 or nkv == 0:
            continue
        for h in range(H):
            kb = k[k0:k0 + nkv, h, :]
            vb = v[k0:k0 + nkv, h, :]
            for i in range(0, sel.size, block):
                idx = sel[i:i + block]
                s = scale * (q[rows[idx], h, :] @ kb.T)
                out[idx, h, :] = softmax_rows(s) @ vb
    return out


def attention_groups(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     k_cache: np.ndarray, v_cache: np.ndarray, groups, scale: float,
                     rows=None, block: int = 256) -> np.ndarray:
    """Query groups over KV views, with a cached KV range (Sol-H3 section 5,
    reference KV caching, Fig. 4: after the first step the reference query
    rows are skipped and the remaining queries attend to the cached
    reference K/V and to the current tokens' K/V; SolarWM-H3 Realtime blog,
    stage 3: pre-concatenated history K/V reused across denoising forwards).

    ``groups`` is a sequence of (q_start, q_len, kv_start, kv_len,
    cache_start, cache_len): query rows [q_start, q_start + q_len) attend to
    k/v rows [kv_start, kv_start + kv_len) together with k_cache/v_cache rows
    [cache_start, cache_start + cache_len).  Views may overlap between
    groups.  Returns (rows, out_rows): the query rows that belong to some
    group (all of them, or those listed in ``rows``) and their outputs; a
    group with no key at all outputs zeros.
    """
    H, D = q.shape[1], q.shape[2]
    sel_rows, outs = [], []
    for (q0, nq, k0, nk, c0, nc) in groups:
        grp_rows = np.arange(q0, q0 + nq)
        if rows is not None:
            grp_rows = grp_rows[np.isin(grp_rows, rows)]
        if grp_rows.size == 0:
            continue
        o = np.zeros((grp_rows.size, H, D))
        if nk + nc > 0:
            kk = np.concatenate([k[k0:k0 + nk], k_cache[c0:c0 + nc]], axis=0)
            vv = np.concatenate([v[k0:k0 + nk], v_cache[c0:c0 + nc]], axis=0)
            for h in range(H):
                for i in range(0, grp_rows.size, block):
                    r = grp_rows[i:i + block]
                    s = scale * (q[r, h, :] @ kk[:, h, :].T)
                    o[i:i + block, h, :] = softmax_rows(s) @ vv[:, h, :]
        sel_rows.append(grp_rows)
        outs.append(o)
    if not outs:
        return np.zeros(0, dtype=np.int64), np.zeros((0, H, D))
    return np.concatenate(sel_rows), np.concatenate(outs, axis=0)


# ------------------------------------------------- block-sparse attention
# Sol-Attn as Sol-H3 (arXiv 2609.35110) section 3.4 describes it: for each
# query block the threshold is mu + tau * sigma over that block's block-level
# scores against all KV blocks; KV blocks scoring above it are attended.
# "Safety rails and the exact prefix KV sink": queries of the prefix
# [text | conditioning video | audio] attend densely; the prefix KV blocks
# are always attended by the remaining (target-video) queries.
# Readings (the page leaves them open): the block-level score of query block
# a and KV block b is scale * <mean of the block's queries, mean of the
# block's keys>; sigma is the population standard deviation; "exceed" is a
# strict >; a block that contains any prefix row counts as a prefix block.

def block_means(x: np.ndarray, n_rows: int, block: int) -> np.ndarray:
    """x [rows, H, D] -> [ceil(n_rows / block), H, D]: mean over each block's
    rows among the first n_rows (the last block may be partial)."""
    nb = -(-n_rows // block)
    out = np.zeros((nb, x.shape[1], x.shape[2]))
    for b in range(nb):
        out[b] = x[b * block:min(n_rows, (b + 1) * block)].mean(axis=0)
    return out


def block_scores(q_means: np.ndarray, k_means: np.ndarray, scale: float) -> np.ndarray:
    """[nQB, H, D] x [nKB, H, D] -> [H, nQB, nKB] = scale * q_mean . k_mean."""
    return scale * np.einsum("ahd,bhd->hab", q_means, k_means)


def select_blocks(scores: np.ndarray, tau: float, n_prefix_blocks: int) -> np.ndarray:
    """bool [H, nQB, nKB]: the KV blocks each query block attends.

    Query blocks a < n_prefix_blocks attend to every KV block; otherwise KV
    block b is kept when b < n_prefix_blocks (sink) or its score exceeds
    mean + tau * std of the row (population std over all KV blocks)."""
    mu = scores.mean(axis=-1, keepdims=True)
    sd = scores.std(axis=-1, keepdims=True)
    keep = scores > mu + tau * sd
    keep[:, :, :n_prefix_blocks] = True
    keep[:, :n_prefix_blocks, :] = True
    return keep


def block_sparse_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_rows: int,
                           keep: np.ndarray, block: int, scale: float, rows=None) -> np.ndarray:
    """Exact softmax attention of each query row over the keys of the KV
    blocks its query block keeps (rows past n_rows are padding, and rows of a
    query block that keeps nothing, output 0)."""
    H, D = q.shape[1], q.shape[2]
    if rows is None:
        rows = np.arange(q.shape[0])
    rows = np.asarray(rows)
    out = np.zeros((rows.size, H, D))
    for i, r in enumerate(rows):
        if r >= n_rows:
            continue
        a = r // block
        for h in range(H):
            kb = np.nonzero(keep[h, a])[0]
            if kb.size == 0:
                continue  # a query block that keeps no KV block outputs 0
            cols = np.concatenate([np.arange(b * block, min(n_rows, (b + 1) * block)) for b in kb])
            s = scale * (k[cols, h] @ q[r, h])
            out[i, h] = softmax_rows(s[None])[0] @ v[cols, h]
    return out


# ------------------------------------------------------------ wire formats
# Sol-H3 section 3.2, "Optimized attention collectives" and "Quantized
# communication": packed QKV goes out destination-major in one pass, the
# attention output comes back through the inverse head merge, and both may
# travel in approximate record formats.  Readings (the page fixes the sizes,
# not every bit): a QKV record is one (token, head) with q, k, v back to
# back; UE5M3 is unsigned, 5 exponent bits (bias 15) and 3 mantissa bits, all
# 256 codes finite and positive (value 2^(e-15) * (1 + m/8)); a group of 32
# values takes the smallest code c with 127 * value(c) >= max |x| and stores
# rint(x / value(c)) as int8; E4M3 is the OCP FP8 E4M3 format with
# round-to-nearest-even saturating at +-448.

def pack_qkv(q, k, v, n_dest: int) -> np.ndarray:
    """[rows, H, D] x3 -> [n_dest, rows, H/n_dest, 3, D]: destination-major,
    q/k/v of one head back to back."""
    rows, H, D = q.shape
    x = np.stack([q, k, v], axis=2)                        # [rows, H, 3, D]
    return x.reshape(rows, n_dest, H // n_dest, 3, D).transpose(1, 0, 2, 3, 4)


def merge_heads(parts: np.ndarray) -> np.ndarray:
    """[n_src, rows, H/n_src, D] -> [rows, H, D] (source s owns heads
    s*H/n_src ...)."""
    n_src, rows, hl, D = parts.shape
    return parts.transpose(1, 0, 2, 3).reshape(rows, n_src * hl, D)


def ue5m3_value(code) -> np.ndarray:
    code = np.asarray(code, dtype=np.int64)
    return np.ldexp(1.0 + (code & 7) / 8.0, (code >> 3) - 15)


def ue5m3_scale_code(amax) -> np.ndarray:
    """Smallest code c with 127 * value(c) >= amax (code 255 if none)."""
    amax = np.asarray(amax, dtype=np.float64)
    table = 127.0 * ue5m3_value(np.arange(256))
    return np.minimum(np.searchsorted(table, amax, side="left"), 255)


def int8_group32(x: np.ndarray):
    """x [..., D] -> (int8 values [..., D], uint8 scale codes [..., D/32])."""
    g = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
    codes = ue5m3_scale_code(np.abs(g).max(axis=-1))
    s = ue5m3_value(codes)[..., None]
    vals = np.clip(np.rint(g / s), -127, 127).astype(np.int8)
    return vals.reshape(x.shape), codes.astype(np.uint8)


def int8_group32_decode(vals: np.ndarray, codes: np.ndarray) -> np.ndarray:
    g = vals.astype(np.float64).reshape(vals.shape[:-1] + (vals.shape[-1] // 32, 32))
    return (g * ue5m3_value(codes)[..., None]).reshape(vals.shape)


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value (3 mantissa bits, min normal 2^-6, subnormal
    quantum 2^-9), ties to even, saturated to +-448."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    q = np.ldexp(1.0, np.maximum(e, -5) - 4)   # one unit in the last place
    r = np.rint(x / q) * q
    return np.clip(r, -448.0, 448.0)


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """uint8 E4M3 encoding of values already on the E4M3 grid."""
    x = np.asarray(x, dtype=np.float64)
    sign = (np.signbit(x)).astype(np.int64) << 7
    a = np.abs(x)
    m, e = np.frexp(a)                        # a = m * 2^e, m in [0.5, 1)
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e - 1 + 7, 0)
    frac = np.where(normal, np.rint((a / np.ldexp(1.0, e - 1) - 1.0) * 8), np.rint(a / 2.0 ** -9))
    frac = np.where(a == 0, 0, frac)
    return (sign | (exp_field << 3) | frac.astype(np.int64)).astype(np.uint8)


def qkv_int8_records(q, k, v) -> np.ndarray:
    """[rows, H, D] x3 -> uint8 [rows, H, 400]: 3 x 128 int8 values, 12 scale
    codes (q groups 0-3, k groups, v groups), 4 zero bytes."""
    rows, H, D = q.shape
    rec = np.zeros((rows, H, 400), dtype=np.uint8)
    for t, x in enumerate((q, k, v)):
        vals, codes = int8_group32(x)
        rec[..., t * 128:(t + 1) * 128] = vals.view(np.uint8)
        rec[..., 384 + 4 * t:388 + 4 * t] = codes
    return rec


def out_int8_records(o) -> np.ndarray:
    """[rows, H, D] -> uint8 [rows, H, 144]: 128 int8 values, 4 scale codes,
    12 zero bytes (a 16-byte aligned record)."""
    rows, H, D = o.shape
    rec = np.zeros((rows, H, 144), dtype=np.uint8)
    vals, codes = int8_group32(o)
    rec[..., :128] = vals.view(np.uint8)
    rec[..., 128:132] = codes
    return rec


def out_fp8_records(o) -> np.ndarray:
    """[rows, H, D] -> uint8 [rows, H, 128] raw E4M3 bytes, no scale."""
    return e4m3_bits(e4m3_round(o))

