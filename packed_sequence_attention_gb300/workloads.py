"""Seeded synthetic workloads for packed-sequence attention.

This module holds only shapes, seeds and random draws.  It computes nothing
of the method itself (no normalisation, rotation or attention), so both the
CUDA path and the CPU oracle may take their inputs from here.

Workload shapes follow the pages:

* packed joint sequence of text, audio and video tokens, e.g. 58,758 valid
  tokens in a 58,816-token aligned buffer ("MiniMax H3 on vLLM-Omni",
  section 3.1 "long-sequence attention and communication");
* hidden width 5,376 in 128-channel heads, hence 42 heads (Sol-H3,
  arXiv 2609.35110, section 3.5 "Kernel Fusion"; vLLM-Omni blog section 3.1);
* grouped condition / audio / video query ranges reading different KV
  extents from a pre-concatenated history cache ("SolarWM-H3 Realtime",
  stage 2 "Attention Backend" and stage 3 "reuse of concatenated history K/V").

Token order inside one sequence is video, audio, text, then padding.  Video
rows carry their (t, h, w) latent-grid indices; audio and text rows carry
(i, 0, 0) with i counting from 0 inside each modality; padded rows carry
(0, 0, 0).  Positions restart in every sequence.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

HEAD_DIM = 128
BASE_SEED = 20260903


@dataclass(frozen=True)
class Segment:
    """One packed sequence (self-attention) or one query group (grouped)."""

    q_rows: int                     # rows the segment occupies in Q / out
    kv_rows: int                    # rows the segment occupies in K / V
    valid: Optional[int] = None     # valid rows (Q and KV alike); None = all
    video: Optional[tuple] = None   # (t, h, w) latent grid
    audio: int = 0
    text: int = 0

    def n_valid_q(self) -> int:
        return self.q_rows if self.valid is None else self.valid

    def n_valid_kv(self) -> int:
        return self.kv_rows if self.valid is None else self.valid


@dataclass(frozen=True)
class Workload:
    name: str
    n_heads: int
    segments: tuple
    self_attention: bool = True     # Q/K/V share one row layout; prologue runs
    description: str = ""
    head_dim: int = HEAD_DIM

    # ---- derived sizes -------------------------------------------------
    @property
    def q_rows(self) -> int:
        return sum(s.q_rows for s in self.segments)

    @property
    def kv_rows(self) -> int:
        return sum(s.kv_rows for s in self.segments)

    def cu_seqlens_q(self) -> list:
        out = [0]
        for s in self.segments:
            out.append(out[-1] + s.q_rows)
        return out

    def cu_seqlens_kv(self) -> list:
        out = [0]
        for s in self.segments:
            out.append(out[-1] + s.kv_rows)
        return out

    def valid_len(self) -> Optional[list]:
        if all(s.valid is None for s in self.segments):
            return None
        return [s.n_valid_q() for s in self.segments]

    def attention_flops(self) -> float:
        """4 * H * D * sum(Lq * Lkv) over valid rows only."""
        return float(4 * self.n_heads * self.head_dim *
                     sum(s.n_valid_q() * s.n_valid_kv() for s in self.segments))

    def prologue_bytes(self) -> float:
        """Bytes the fused Q/K norm + RoPE step must move over valid rows:
        read + write of Q and K (2 B each way per element), plus the per-row
        int32 positions and the two bf16 weight tables."""
        if not self.self_attention:
            return 0.0
        rows = sum(s.n_valid_q() for s in self.segments)
        per_row = 2 * 2 * 2 * self.n_heads * self.head_dim + 3 * 4
        return float(rows * per_row + 2 * 2 * self.n_heads * self.head_dim)


def _seq(buffer_rows: int, video: tuple, audio: int, text: int) -> Segment:
    t, h, w = video
    valid = t * h * w + audio + text
    assert valid <= buffer_rows
    return Segment(buffer_rows, buffer_rows, valid, video, audio, text)


WORKLOADS = {
    "tiny": Workload(
        "tiny", 2, (_seq(256, (2, 8, 8), 64, 58),),
        description="1 sequence, 250 valid of 256 rows, 2 heads"),
    "medium": Workload(
        "medium", 42, (_seq(4096, (5, 24, 28), 400, 240),),
        description="1 sequence, 4,000 valid of 4,096 rows, 42 heads"),
    "full": Workload(
        "full", 42, (_seq(58816, (21, 48, 56), 1800, 510),),
        description="1 sequence, 58,758 valid of 58,816 rows, 42 heads"),
    "stage1_batch2": Workload(
        "stage1_batch2", 42,
        (_seq(16448, (21, 24, 28), 1800, 510),) * 2,
        description="2 sequences, 16,422 valid of 16,448 rows each, 42 heads"),
    "grouped_chunk": Workload(
        "grouped_chunk", 42,
        (Segment(512, 512), Segment(1024, 4096), Segment(8160, 40800)),
        self_attention=False,
        description="3 query groups (512/512, 1,024/4,096, 8,160/40,800), "
                    "42 heads, attention only"),
}
# Index order of the five synthetic shapes.
CONFIG_ORDER = ["tiny", "medium", "full", "stage1_batch2", "grouped_chunk"]


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[CONFIG_ORDER[name_or_index]]
    return WORKLOADS[name_or_index]


def default_seed(w: Workload) -> int:
    if w.name in CONFIG_ORDER:
        return BASE_SEED + CONFIG_ORDER.index(w.name)
    return BASE_SEED + 100 + sum(ord(c) for c in w.name)


def positions(w: Workload) -> torch.Tensor:
    """int32 [q_rows, 3] (t, h, w) indices per row; see module docstring."""
    rows = []
    for s in w.segments:
        seg = torch.zeros(s.q_rows, 3, dtype=torch.int32)
        r = 0
        if s.video is not None:
            t, h, ww = s.video
            n = t * h * ww
            idx = torch.arange(n, dtype=torch.int64)
            seg[:n, 0] = (idx // (h * ww)).to(torch.int32)
            seg[:n, 1] = ((idx // ww) % h).to(torch.int32)
            seg[:n, 2] = (idx % ww).to(torch.int32)
            r = n
        for count in (s.audio, s.text):
            seg[r:r + count, 0] = torch.arange(count, dtype=torch.int32)
            r += count
        rows.append(seg)
    return torch.cat(rows, 0)


def padded_row_mask(w: Workload, kv: bool = False) -> torch.Tensor:
    """bool [rows]: True for rows past a segment's valid length."""
    parts = []
    for s in w.segments:
        n = s.kv_rows if kv else s.q_rows
        valid = s.n_valid_kv() if kv else s.n_valid_q()
        m = torch.zeros(n, dtype=torch.bool)
        m[valid:] = True
        parts.append(m)
    return torch.cat(parts, 0)


def _garbage(shape, fill: str, gen: torch.Generator, device) -> torch.Tensor:
    g = (torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
         * 2.0 - 1.0) * 1.0e4
    if fill == "B":
        flat = g.view(-1)
        flat[0::3] = float("nan")
        flat[1::5] = float("inf")
        flat[2::7] = float("-inf")
    return g


def make_inputs(w, seed: Optional[int] = None, fill: str = "A",
                device="cpu", packed_qkv: bool = False,
                row_pad: int = 0) -> dict:
    """Draw one seeded input set for workload ``w``.

    Q, K, V ~ N(0, 1) drawn in fp32 and rounded to bf16; per-head norm weights
    ~ N(1, 0.1) rounded to bf16.  Padded rows hold garbage: uniform in
    [-1e4, 1e4] (fill "A") or the same with NaN / +Inf / -Inf mixed in
    (fill "B").  The output buffer is pre-filled with NaN.

    ``packed_qkv`` places Q, K and V as views into one [rows, 3, H, D] buffer
    (row stride 3*H*D); ``row_pad`` adds that many unused elements at the end
    of every row of each separate tensor (row stride H*D + row_pad).
    The draw order is fixed: q, k, v, wq, wk, then the garbage of q, k, v.
    """
    if not isinstance(w, Workload):
        w = workload(w)
    if seed is None:
        seed = default_seed(w)
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed)
    H, D = w.n_heads, w.head_dim
    Rq, Rkv = w.q_rows, w.kv_rows
    bf = torch.bfloat16

    def normal(rows):
        return torch.randn((rows, H, D), generator=gen, device=dev,
                           dtype=torch.float32).to(bf)

    if packed_qkv:
        assert w.self_attention and Rq == Rkv and row_pad == 0
        buf = torch.empty((Rq, 3, H, D), dtype=bf, device=dev)
        q, k, v = buf[:, 0], buf[:, 1], buf[:, 2]
        q.copy_(normal(Rq)); k.copy_(normal(Rkv)); v.copy_(normal(Rkv))
    elif row_pad:
        def strided(rows):
            base = torch.full((rows, H * D + row_pad), float("nan"),
                              dtype=bf, device=dev)
            return base[:, :H * D].view(rows, H, D)
        q, k, v = strided(Rq), strided(Rkv), strided(Rkv)
        q.copy_(normal(Rq)); k.copy_(normal(Rkv)); v.copy_(normal(Rkv))
    else:
        q, k, v = normal(Rq), normal(Rkv), normal(Rkv)

    wq = (1.0 + 0.1 * torch.randn((H, D), generator=gen, device=dev)).to(bf)
    wk = (1.0 + 0.1 * torch.randn((H, D), generator=gen, device=dev)).to(bf)

    pad_q = padded_row_mask(w).to(dev)
    pad_kv = padded_row_mask(w, kv=True).to(dev)
    for t, m in ((q, pad_q), (k, pad_kv), (v, pad_kv)):
        n = int(m.sum())
        if n:
            t[m] = _garbage((n, H, D), fill, gen, dev).to(bf)

    out = torch.full((Rq, H, D), float("nan"), dtype=bf, device=dev)
    res = dict(workload=w, seed=seed, q=q, k=k, v=v, out=out,
               wq=wq, wk=wk,
               cu_seqlens_q=w.cu_seqlens_q(), cu_seqlens_kv=w.cu_seqlens_kv(),
               valid_len=w.valid_len(), pad_q=pad_q, pad_kv=pad_kv)
    if w.self_attention:
        res["pos_thw"] = positions(w).to(dev)
    return res


def ref_cached_inputs(n_refs: int = 3, seed: int = BASE_SEED + 50, device="cpu") -> dict:
    """Reference-to-video step after the first (Sol-H3 reference KV caching,
    Fig. 4): the current sequence holds video 21x24x28 (14,112), audio 1,800
    and text 510 tokens (16,422 valid of 16,448 rows); the cache holds the
    K/V of n_refs reference videos of the same latent grid (14,112 rows each)
    computed in the first step.  Reference query rows are skipped: the
    16,422 current queries attend to the cache and to the current K/V."""
    H, D = 42, HEAD_DIM
    cur_valid, cur_rows, ref_rows = 16422, 16448, 14112 * n_refs
    gen = torch.Generator(device=torch.device(device)).manual_seed(seed)

    def normal(rows):
        return torch.randn((rows, H, D), generator=gen, device=device,
                           dtype=torch.float32).to(torch.bfloat16)
    q, k, v = normal(cur_rows), normal(cur_rows), normal(cur_rows)
    kc, vc = normal(ref_rows), normal(ref_rows)
    for t in (q, k, v):
        t[cur_valid:] = float("nan")
    out = torch.full((cur_rows, H, D), float("nan"), dtype=torch.bfloat16, device=device)
    groups = [(0, cur_valid, 0, cur_valid, 0, ref_rows)]
    return dict(q=q, k=k, v=v, k_cache=kc, v_cache=vc, out=out, groups=groups, n_heads=H,
                flops=4.0 * H * D * cur_valid * (cur_valid + ref_rows))


def custom(name: str, n_heads: int, segments: Sequence[Segment],
           self_attention: bool = True) -> Workload:
    """A workload for tests: arbitrary heads and segments."""
    return Workload(name, n_heads, tuple(segments), self_attention)
