"""Pure-Python brute force for tiny cases: an independent second oracle.

TEST INFRASTRUCTURE.  Only the test suite may run this.  It shares nothing
with ``oracle.oracle`` (no NumPy, no shared helpers): plain loops over
Python floats with ``math.fsum`` sums, so that it can pin the NumPy oracle.
It follows the same passages (Sol-H3 section 3.5 operator group 2 for the
Q/K norm + RoPE; exact softmax attention over the valid rows of each
packed sequence, vLLM-Omni blog section 3.1).
"""
from __future__ import annotations

import math


def norm_rope_row(x, w, pos, sections, theta, eps):
    """One (row, head): x and w are lists of D floats, pos = (t, h, w)."""
    d_total = len(x)
    ms = math.fsum(xi * xi for xi in x) / d_total
    r = 1.0 / math.sqrt(ms + eps)
    y = [x[c] * r * w[c] for c in range(d_total)]
    out = list(y)
    off = 0
    for axis in range(3):
        width = sections[axis]
        for j in range(width // 2):
            angle = pos[axis] * theta ** (-(2.0 * j) / width)
            c0 = off + 2 * j
            a, b = y[c0], y[c0 + 1]
            out[c0] = a * math.cos(angle) - b * math.sin(angle)
            out[c0 + 1] = a * math.sin(angle) + b * math.cos(angle)
        off += width
    return out


def attention_row(qrow, keys, values, scale):
    """softmax over keys of scale * <q, k_j>, then the weighted sum of v_j."""
    if not keys:
        return [0.0] * len(qrow)
    scores = [scale * math.fsum(a * b for a, b in zip(qrow, kj)) for kj in keys]
    m = max(scores)
    e = [math.exp(s - m) for s in scores]
    z = math.fsum(e)
    d = len(values[0])
    return [math.fsum(e[j] * values[j][c] for j in range(len(values))) / z
            for c in range(d)]


def round_bf16(x):
    """Nearest bfloat16 to a Python float (8 significant bits), ties to even."""
    if x == 0.0 or math.isinf(x) or math.isnan(x):
        return x
    m, e = math.frexp(x)
    e = max(e, -125)
    q = math.ldexp(1.0, e - 8)
    return round(x / q) * q  # Python's round() is round-half-to-even


def norm_rope_lora_row(base, delta, w, pos, sections, theta, eps):
    """One (row, head) of the LoRA-fused prologue: round base + delta to bf16
    first, then the RMSNorm + axial RoPE of ``norm_rope_row``."""
    x = [round_bf16(b + d) for b, d in zip(base, delta)]
    return norm_rope_row(x, w, pos, sections, theta, eps)
