"""Packed-sequence attention for the MiniMax-H3 DiT block on GB300 (sm_103a).

Two operations, both hand-written CUDA behind the C ABI of libh3kern.so
(include/h3kern.h); this module only marshals torch tensors into pointers,
strides and the current stream:

* ``qk_norm_rope`` -- fused Q/K RMSNorm + axial 3-D RoPE, in place
  (Sol-H3, arXiv 2609.35110, section 3.5 "Kernel Fusion", operator group 2);
  ``qk_norm_rope_varlen`` does the valid rows of several packed sequences in
  one launch.
* ``qk_norm_rope_lora`` -- the same as a LoRA consumer: base + delta is
  rounded to bf16 first (Sol-H3 section 3.5, precision-preserving LoRA fusion).
* ``attention`` -- softmax(Q K^T * scale) V over packed sequences with a
  valid length, or over grouped query ranges with their own KV extents
  (vLLM-Omni blog section 3.1; SolarWM-H3 Realtime blog stage 2).
* ``attention_groups`` -- query groups over KV views into the current K/V
  plus a cached K/V range (Sol-H3 reference KV caching, Fig. 4; SolarWM
  history K/V reuse).
* ``block_means`` (``block_means_qk``) / ``block_select`` / ``sparse_attention`` (and
  ``sol_attention`` chaining them) -- Sol-Attn block-sparse attention with
  the exact prefix KV sink (Sol-H3 section 3.4).
* ``pack_qkv`` / ``unpack_qkv`` / ``pack_out`` / ``merge_heads`` -- the
  attention-boundary wire formats: destination-major packed QKV, the inverse
  head merge, and block-INT8 / FP8 records (Sol-H3 section 3.2).

There is no CPU or library fallback: without the built library, or off an
sm_103 device, every call raises ``H3Error``.
"""
from __future__ import annotations

import ctypes
import math
from typing import List, Optional, Sequence, Tuple

import torch

from . import _binding

__all__ = ["H3Error", "qk_norm_rope", "qk_norm_rope_varlen", "qk_norm_rope_lora", "attention",
           "attention_groups", "block_means", "block_means_qk", "block_select", "sparse_attention",
           "sol_attention", "WIRE_BF16", "WIRE_INT8", "WIRE_FP8", "wire_record_bytes", "pack_qkv",
           "unpack_qkv", "pack_out", "merge_heads", "status_word", "lib", "HEAD_DIM",
           "MAX_SEGMENTS", "attention_block", "copy_2d", "head_groups", "HostPipeline"]

HEAD_DIM = 128
MAX_SEGMENTS = 16


class H3Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_binding.STATUS.get(status, status)}: {message}")
        self.status = status


def lib():
    return _binding.load()


def _check(status: int):
    if status != 0:
        raise H3Error(status, lib().h3_last_error().decode())


def _on_device(t: torch.Tensor, name: str) -> torch.Tensor:
    """Every pointer the kernels read or write must be memory of the current
    CUDA device: a host tensor, or one on another GPU, would have its
    address encoded into a tensor map or dereferenced in a kernel."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got device {t.device})")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    return t


def _heads(t: torch.Tensor, name: str, n_heads: int) -> None:
    if t.dim() < 2 or t.shape[1] != n_heads:
        raise ValueError(f"{name} must have {n_heads} heads, got shape {tuple(t.shape)}")


def _row_stride(t: torch.Tensor, name: str) -> int:
    _on_device(t, name)
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 3 or t.shape[-1] != HEAD_DIM:
        raise ValueError(f"{name} must be [rows, heads, {HEAD_DIM}], got {tuple(t.shape)}")
    if t.stride(-1) != 1 or (t.shape[1] > 1 and t.stride(1) != HEAD_DIM):
        raise ValueError(f"{name}: channels must be contiguous and heads {HEAD_DIM} apart")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1] * HEAD_DIM


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def qk_norm_rope(q: torch.Tensor, k: torch.Tensor, wq: torch.Tensor, wk: torch.Tensor,
                 pos_thw: torch.Tensor, n_rows: Optional[int] = None,
                 rot=(32, 48, 48), theta: float = 10000.0, eps: float = 1e-6,
                 stream=None) -> None:
    """In place: q, k <- RoPE(RMSNorm(x) * w) for rows [0, n_rows)."""
    qs, ks = _row_stride(q, "q"), _row_stride(k, "k")
    H = q.shape[1]
    _heads(k, "k", H)
    if n_rows is None:
        n_rows = q.shape[0]
    if not (0 <= n_rows <= min(q.shape[0], k.shape[0], pos_thw.shape[0])):
        raise ValueError("n_rows exceeds the tensors")
    _prologue_small_inputs(wq, wk, pos_thw, H)
    _check(lib().h3_qk_norm_rope(q.data_ptr(), qs, k.data_ptr(), ks, wq.data_ptr(),
                                 wk.data_ptr(), pos_thw.data_ptr(), int(n_rows), H, HEAD_DIM,
                                 int(rot[0]), int(rot[1]), int(rot[2]), float(theta),
                                 float(eps), _stream(stream)))


def qk_norm_rope_varlen(q: torch.Tensor, k: torch.Tensor, wq: torch.Tensor, wk: torch.Tensor,
                        pos_thw: torch.Tensor, cu_seqlens: Sequence[int],
                        valid_len: Optional[Sequence[int]] = None, rot=(32, 48, 48),
                        theta: float = 10000.0, eps: float = 1e-6, stream=None) -> None:
    """In place, in one launch: ``qk_norm_rope`` on the first ``valid_len[b]``
    rows of each packed sequence b = rows [cu_seqlens[b], cu_seqlens[b+1]).

    ``cu_seqlens`` and ``valid_len`` are host sequences of ints; ``pos_thw``
    is indexed by buffer row.  Other rows are not touched."""
    qs, ks = _row_stride(q, "q"), _row_stride(k, "k")
    H = q.shape[1]
    _heads(k, "k", H)
    n_seq = len(cu_seqlens) - 1
    if valid_len is not None and len(valid_len) != n_seq:
        raise ValueError("cu_seqlens and valid_len disagree on n_seq")
    if n_seq >= 1 and cu_seqlens[-1] > min(q.shape[0], k.shape[0], pos_thw.shape[0]):
        raise ValueError("cu_seqlens exceed the tensors")
    _prologue_small_inputs(wq, wk, pos_thw, H)
    cu = _i32_array(cu_seqlens)
    vl = _i32_array(valid_len) if valid_len is not None else None
    _check(lib().h3_qk_norm_rope_varlen(q.data_ptr(), qs, k.data_ptr(), ks, wq.data_ptr(),
                                        wk.data_ptr(), pos_thw.data_ptr(),
                                        ctypes.cast(cu, _binding.c_i32p),
                                        ctypes.cast(vl, _binding.c_i32p) if vl is not None
                                        else None, n_seq, H, HEAD_DIM, int(rot[0]), int(rot[1]),
                                        int(rot[2]), float(theta), float(eps), _stream(stream)))


def qk_norm_rope_lora(q: torch.Tensor, q_delta: torch.Tensor, k: torch.Tensor,
                      k_delta: torch.Tensor, wq: torch.Tensor, wk: torch.Tensor,
                      pos_thw: torch.Tensor, n_rows: Optional[int] = None,
                      rot=(32, 48, 48), theta: float = 10000.0, eps: float = 1e-6,
                      stream=None) -> None:
    """In place on the base branches q, k: x = bf16(base + delta), then
    RoPE(RMSNorm(x) * w), for rows [0, n_rows)."""
    qs, ks = _row_stride(q, "q"), _row_stride(k, "k")
    dqs, dks = _row_stride(q_delta, "q_delta"), _row_stride(k_delta, "k_delta")
    H = q.shape[1]
    for t, name in ((k, "k"), (q_delta, "q_delta"), (k_delta, "k_delta")):
        _heads(t, name, H)
    if n_rows is None:
        n_rows = q.shape[0]
    if not (0 <= n_rows <= min(q.shape[0], k.shape[0], q_delta.shape[0], k_delta.shape[0],
                               pos_thw.shape[0])):
        raise ValueError("n_rows exceeds the tensors")
    _prologue_small_inputs(wq, wk, pos_thw, H)
    _check(lib().h3_qk_norm_rope_lora(q.data_ptr(), qs, q_delta.data_ptr(), dqs, k.data_ptr(), ks,
                                      k_delta.data_ptr(), dks, wq.data_ptr(), wk.data_ptr(),
                                      pos_thw.data_ptr(), int(n_rows), H, HEAD_DIM, int(rot[0]),
                                      int(rot[1]), int(rot[2]), float(theta), float(eps),
                                      _stream(stream)))


def _prologue_small_inputs(wq, wk, pos_thw, H):
    _on_device(pos_thw, "pos_thw")
    if pos_thw.dtype != torch.int32 or not pos_thw.is_contiguous() or pos_thw.shape[-1] != 3:
        raise ValueError("pos_thw must be contiguous int32 [rows, 3]")
    for w, name in ((wq, "wq"), (wk, "wk")):
        _on_device(w, name)
        if w.dtype != torch.bfloat16 or not w.is_contiguous() or tuple(w.shape) != (H, HEAD_DIM):
            raise ValueError(f"{name} must be contiguous bf16 [{H}, {HEAD_DIM}]")


def _i32_array(values: Sequence[int]):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
              cu_seqlens_q: Sequence[int], cu_seqlens_kv: Sequence[int],
              valid_len: Optional[Sequence[int]] = None, scale: Optional[float] = None,
              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[i, h] = softmax_j(scale <q_i, k_j>) v_j per segment; see h3kern.h.

    ``cu_seqlens_*`` and ``valid_len`` are host sequences of ints."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, HEAD_DIM), dtype=torch.bfloat16, device=q.device)
    strides = [_row_stride(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"))]
    for t, name in ((k, "k"), (v, "v"), (out, "out")):
        _heads(t, name, H)
    n_seq = len(cu_seqlens_q) - 1
    if len(cu_seqlens_kv) != n_seq + 1 or (valid_len is not None and len(valid_len) != n_seq):
        raise ValueError("cu_seqlens_q, cu_seqlens_kv and valid_len disagree on n_seq")
    if cu_seqlens_q[-1] > q.shape[0] or cu_seqlens_q[-1] > out.shape[0] or \
            cu_seqlens_kv[-1] > k.shape[0] or cu_seqlens_kv[-1] > v.shape[0]:
        raise ValueError("cu_seqlens exceed the tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(HEAD_DIM)
    cq, ckv = _i32_array(cu_seqlens_q), _i32_array(cu_seqlens_kv)
    vl = _i32_array(valid_len) if valid_len is not None else None
    _check(lib().h3_attention(q.data_ptr(), strides[0], k.data_ptr(), strides[1],
                              v.data_ptr(), strides[2], out.data_ptr(), strides[3],
                              ctypes.cast(cq, _binding.c_i32p), ctypes.cast(ckv, _binding.c_i32p),
                              ctypes.cast(vl, _binding.c_i32p) if vl is not None else None,
                              n_seq, H, HEAD_DIM, float(scale), _stream(stream)))
    return out


def attention_groups(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, groups,
                     k_cache: Optional[torch.Tensor] = None,
                     v_cache: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Query groups over KV views plus an optional cached KV range.

    ``groups``: sequence of (q_start, q_len, kv_start, kv_len, cache_start,
    cache_len).  Rows of ``out`` outside every group are left untouched."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, HEAD_DIM), dtype=torch.bfloat16, device=q.device)
    tensors = [(q, "q"), (k, "k"), (v, "v"), (out, "out")]
    uses_cache = any(g[5] > 0 for g in groups)
    if uses_cache:
        if k_cache is None or v_cache is None:
            raise ValueError("a group uses the cache but k_cache / v_cache are missing")
        tensors += [(k_cache, "k_cache"), (v_cache, "v_cache")]
    strides = {n: _row_stride(t, n) for t, n in tensors}
    for t, name in tensors[1:]:
        _heads(t, name, H)
    for (q0, nq, k0, nk, c0, nc) in groups:
        if q0 + nq > min(q.shape[0], out.shape[0]) or k0 + nk > min(k.shape[0], v.shape[0]) or \
                (nc and c0 + nc > min(k_cache.shape[0], v_cache.shape[0])):
            raise ValueError("a group addresses rows past the tensors")
    arr = (_binding.AttnGroup * len(groups))(*[_binding.AttnGroup(*map(int, g)) for g in groups])
    if scale is None:
        scale = 1.0 / math.sqrt(HEAD_DIM)
    kc_ptr = k_cache.data_ptr() if uses_cache else None
    vc_ptr = v_cache.data_ptr() if uses_cache else None
    _check(lib().h3_attention_groups(
        q.data_ptr(), strides["q"], k.data_ptr(), strides["k"], v.data_ptr(), strides["v"],
        kc_ptr, strides.get("k_cache", 0), vc_ptr, strides.get("v_cache", 0),
        out.data_ptr(), strides["out"], ctypes.cast(arr, ctypes.c_void_p), len(groups), H,
        HEAD_DIM, float(scale), _stream(stream)))
    return out


BLOCK = 128  # block-sparse blocks = attention tiles


def block_means(x: torch.Tensor, n_rows: Optional[int] = None, stream=None) -> torch.Tensor:
    """fp32 [ceil(n_rows / 128), H, 128]: mean of each 128-row block."""
    xs = _row_stride(x, "x")
    n_rows = x.shape[0] if n_rows is None else n_rows
    if n_rows > x.shape[0]:
        raise ValueError("n_rows exceeds the tensor")
    H = x.shape[1]
    out = torch.empty((-(-n_rows // BLOCK), H, HEAD_DIM), dtype=torch.float32, device=x.device)
    _check(lib().h3_block_means(x.data_ptr(), xs, int(n_rows), H, HEAD_DIM, out.data_ptr(),
                                _stream(stream)))
    return out


def block_means_qk(q: torch.Tensor, k: torch.Tensor, n_rows: Optional[int] = None, stream=None):
    """(q_means, k_means), each fp32 [ceil(n_rows / 128), H, 128], in one launch."""
    qs, ks = _row_stride(q, "q"), _row_stride(k, "k")
    n_rows = q.shape[0] if n_rows is None else n_rows
    H = q.shape[1]
    _heads(k, "k", H)
    if n_rows > min(q.shape[0], k.shape[0]):
        raise ValueError("n_rows exceeds the tensors")
    qm, km = (torch.empty((-(-n_rows // BLOCK), H, HEAD_DIM), dtype=torch.float32, device=q.device)
              for _ in range(2))
    _check(lib().h3_block_means_qk(q.data_ptr(), qs, k.data_ptr(), ks, int(n_rows), H, HEAD_DIM,
                                   qm.data_ptr(), km.data_ptr(), _stream(stream)))
    return qm, km


def block_select(q_means: torch.Tensor, k_means: torch.Tensor, tau: float, n_prefix_blocks: int,
                 scale: Optional[float] = None, with_scores: bool = False, stream=None):
    """(lists int32 [H, nqb, nkb], counts int32 [H, nqb][, scores fp32])."""
    nqb, H, _ = q_means.shape
    nkb = k_means.shape[0]
    for t, name in ((q_means, "q_means"), (k_means, "k_means")):
        _on_device(t, name)
        if t.dtype != torch.float32 or not t.is_contiguous() or t.shape[1:] != (H, HEAD_DIM):
            raise ValueError("means must be contiguous fp32 [n_blocks, H, 128]")
    if scale is None:
        scale = 1.0 / math.sqrt(HEAD_DIM)
    dev = q_means.device
    lists = torch.empty((H, nqb, nkb), dtype=torch.int32, device=dev)
    counts = torch.empty((H, nqb), dtype=torch.int32, device=dev)
    scores = torch.empty((H, nqb, nkb), dtype=torch.float32, device=dev) if with_scores else None
    _check(lib().h3_block_select(q_means.data_ptr(), k_means.data_ptr(), nqb, nkb, H, float(scale),
                                 float(tau), int(n_prefix_blocks),
                                 scores.data_ptr() if with_scores else None, lists.data_ptr(),
                                 counts.data_ptr(), _stream(stream)))
    return (lists, counts, scores) if with_scores else (lists, counts)


def sparse_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, lists: torch.Tensor,
                     counts: torch.Tensor, n_rows: int, scale: Optional[float] = None,
                     out: Optional[torch.Tensor] = None, stream=None,
                     n_prefix_blocks: int = 0) -> torch.Tensor:
    """Attention of each query row over the KV blocks its block keeps.

    ``n_prefix_blocks`` (the value given to ``block_select``) only orders the
    work: the dense prefix query tiles are scheduled first."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, HEAD_DIM), dtype=torch.bfloat16, device=q.device)
    strides = [_row_stride(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"))]
    for t, name in ((k, "k"), (v, "v"), (out, "out")):
        _heads(t, name, H)
    _on_device(lists, "lists")
    _on_device(counts, "counts")
    nb = -(-n_rows // BLOCK)
    if tuple(lists.shape) != (H, nb, nb) or tuple(counts.shape) != (H, nb) or \
            lists.dtype != torch.int32 or counts.dtype != torch.int32:
        raise ValueError("lists / counts do not match the sequence")
    if not lists.is_contiguous() or not counts.is_contiguous():
        raise ValueError("lists / counts must be contiguous")
    if n_rows > min(q.shape[0], k.shape[0], v.shape[0], out.shape[0]):
        raise ValueError("n_rows exceeds the tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(HEAD_DIM)
    _check(lib().h3_sparse_attention(q.data_ptr(), strides[0], k.data_ptr(), strides[1],
                                     v.data_ptr(), strides[2], out.data_ptr(), strides[3],
                                     int(n_rows), H, HEAD_DIM, lists.data_ptr(), counts.data_ptr(),
                                     int(n_prefix_blocks), float(scale), _stream(stream)))
    return out


def sol_attention(q, k, v, n_rows: int, tau: float, n_prefix_rows: int,
                  scale: Optional[float] = None, out=None, stream=None):
    """The three block-sparse stages in a row; returns (out, lists, counts)."""
    qm, km = block_means_qk(q, k, n_rows, stream)
    n_pre = -(-n_prefix_rows // BLOCK)
    lists, counts = block_select(qm, km, tau, n_pre, scale, stream=stream)
    out = sparse_attention(q, k, v, lists, counts, n_rows, scale, out, stream, n_prefix_blocks=n_pre)
    return out, lists, counts


WIRE_BF16, WIRE_INT8, WIRE_FP8 = 0, 1, 2


def wire_record_bytes(what: str, fmt: int) -> int:
    """Bytes of one (token, head) record; what is "qkv" or "out"."""
    n = lib().h3_wire_record_bytes(0 if what == "qkv" else 1, int(fmt))
    if n < 0:
        raise ValueError(f"no {what} record in format {fmt}")
    return n


def pack_qkv(q, k, v, n_dest: int, fmt: int = WIRE_BF16, stream=None) -> torch.Tensor:
    """uint8 [n_dest, rows, H/n_dest, record]: destination-major packed QKV."""
    rows, H = q.shape[0], q.shape[1]
    rec = wire_record_bytes("qkv", fmt)
    wire = torch.empty((n_dest, rows, H // n_dest, rec), dtype=torch.uint8, device=q.device)
    s = [_row_stride(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"))]
    for t, name in ((k, "k"), (v, "v")):
        _heads(t, name, H)
        if t.shape[0] < rows:
            raise ValueError(f"{name} has fewer rows than q")
    _check(lib().h3_pack_qkv(q.data_ptr(), s[0], k.data_ptr(), s[1], v.data_ptr(), s[2], rows, H,
                             int(n_dest), int(fmt), wire.data_ptr(), _stream(stream)))
    return wire


def unpack_qkv(wire: torch.Tensor, fmt: int = WIRE_BF16, stream=None):
    """wire [rows, heads, record] -> (q, k, v) bf16 [rows, heads, 128]."""
    rows, hl = wire.shape[0], wire.shape[1]
    _on_device(wire, "wire")
    if not wire.is_contiguous() or wire.shape[2] != wire_record_bytes("qkv", fmt):
        raise ValueError("wire must be contiguous [rows, heads, record]")
    q, k, v = (torch.empty((rows, hl, HEAD_DIM), dtype=torch.bfloat16, device=wire.device)
               for _ in range(3))
    _check(lib().h3_unpack_qkv(wire.data_ptr(), rows, hl, int(fmt), q.data_ptr(), hl * HEAD_DIM,
                               k.data_ptr(), hl * HEAD_DIM, v.data_ptr(), hl * HEAD_DIM,
                               _stream(stream)))
    return q, k, v


def pack_out(out: torch.Tensor, fmt: int = WIRE_BF16, stream=None) -> torch.Tensor:
    """uint8 [rows, heads, record]: attention output records."""
    rows, hl = out.shape[0], out.shape[1]
    wire = torch.empty((rows, hl, wire_record_bytes("out", fmt)), dtype=torch.uint8,
                       device=out.device)
    _check(lib().h3_pack_out(out.data_ptr(), _row_stride(out, "out"), rows, hl, int(fmt),
                             wire.data_ptr(), _stream(stream)))
    return wire


def merge_heads(wire: torch.Tensor, fmt: int = WIRE_BF16, out=None, stream=None) -> torch.Tensor:
    """wire [n_src, rows, H/n_src, record] -> out bf16 [rows, H, 128]."""
    n_src, rows, hl = wire.shape[0], wire.shape[1], wire.shape[2]
    _on_device(wire, "wire")
    if not wire.is_contiguous() or wire.shape[3] != wire_record_bytes("out", fmt):
        raise ValueError("wire must be contiguous [n_src, rows, heads, record]")
    H = n_src * hl
    if out is None:
        out = torch.empty((rows, H, HEAD_DIM), dtype=torch.bfloat16, device=wire.device)
    _heads(out, "out", H)
    if out.shape[0] < rows:
        raise ValueError("out has fewer rows than the records")
    _check(lib().h3_merge_heads(wire.data_ptr(), rows, H, n_src, int(fmt), out.data_ptr(),
                                _row_stride(out, "out"), _stream(stream)))
    return out


def attention_block(q, k, v, wq, wk, pos_thw, cu_seqlens, valid_len,
                    rot=(32, 48, 48), theta=10000.0, eps=1e-6, scale=None, out=None,
                    stream=None) -> torch.Tensor:
    """The block's hot path: fused Q/K norm + RoPE on the valid rows of each
    packed sequence, then attention over the valid rows.  Q and K are
    modified in place."""
    _block_prologue(q, k, wq, wk, pos_thw, cu_seqlens, valid_len, rot, theta, eps, stream)
    return attention(q, k, v, cu_seqlens, cu_seqlens, valid_len, scale, out, stream)


def _block_prologue(q, k, wq, wk, pos_thw, cu_seqlens, valid_len, rot, theta, eps, stream):
    """The norm + RoPE of ``attention_block``: every packed sequence's valid
    rows, in one launch."""
    qk_norm_rope_varlen(q, k, wq, wk, pos_thw, cu_seqlens, valid_len, rot=rot, theta=theta,
                        eps=eps, stream=stream)


def copy_2d(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """Asynchronous copy between two [rows, heads, 128] views with the same
    shape (for instance one group of heads of a pinned host tensor and of a
    device tensor); each row's heads must be contiguous."""
    if dst.shape != src.shape or dst.dtype != src.dtype:
        raise ValueError(f"copy_2d: shapes/dtypes differ ({tuple(dst.shape)} vs {tuple(src.shape)})")
    es = dst.element_size()
    width = dst.shape[1] * dst.shape[2] * es
    for t, name in ((dst, "dst"), (src, "src")):
        if t.stride(2) != 1 or (t.shape[1] > 1 and t.stride(1) != t.shape[2]):
            raise ValueError(f"copy_2d: {name} must hold each row's heads contiguously")
    _check(lib().h3_copy_2d(dst.data_ptr(), dst.stride(0) * es, src.data_ptr(),
                            src.stride(0) * es, width, dst.shape[0], _stream(stream)))


def head_groups(n_heads: int, heads_per_group: int = 6,
                group_sizes: Optional[Sequence[int]] = None) -> List[Tuple[int, int]]:
    """Head ranges [h0, h1) of ``HostPipeline``'s groups.

    ``group_sizes`` gives them explicitly (positive, summing to ``n_heads``).
    Otherwise groups hold up to ``heads_per_group`` heads, except that with
    more than two groups the first and the last hold half of that (at least
    one head) and the ones between share the rest evenly.  Only the first
    group's copy in and the last group's copy out are not hidden behind
    compute, so smaller end groups shorten the step; much smaller ones make
    narrow 2-D copies, which move fewer bytes per second.
    (42 heads, 6 per group, on GB300: 49.2 ms per step with seven groups of
    6, 48.6 ms with [3, 6 x 6, 3], 48.9 ms with [2, 4, 6 x 5, 4, 2].)"""
    if group_sizes is not None:
        sizes = [int(x) for x in group_sizes]
        if not sizes or min(sizes) < 1 or sum(sizes) != n_heads:
            raise ValueError(f"group_sizes must be positive and sum to {n_heads}: {sizes}")
    else:
        g = max(1, min(int(heads_per_group), n_heads))
        head = [max(1, g // 2)]
        middle = n_heads - 2 * sum(head)
        if n_heads <= 2 * g or middle < g:
            sizes = [g] * (n_heads // g) + ([n_heads % g] if n_heads % g else [])
        else:  # the middle heads in as few groups of at most g as possible, evenly
            k = -(-middle // g)
            sizes = head + [middle // k + (1 if i < middle % k else 0) for i in range(k)] + head
    out, h = [], 0
    for n in sizes:
        out.append((h, h + n))
        h += n
    return out


class HostPipeline:
    """The block's hot path on inputs in pinned host memory, with the
    transfers hidden behind the compute.

    Heads are processed in groups (``head_groups``: smaller groups at both
    ends): the Q/K/V rows of group g + 1 are copied host -> device while
    group g is normalised and attended, and group g's output is copied back
    as soon as it is done.  Consecutive groups run on
    two compute streams so that one attention launch's last partial wave
    overlaps the next launch.  Heads are independent, so the result is
    bitwise that of ``attention_block`` on the whole tensors.

    The device buffers (Q, K, V, out, weights, positions) are allocated once
    for ``rows`` (query rows; ``kv_rows`` key rows, default the same) x
    ``n_heads``; host tensors must be pinned and shaped like them.
    ``run`` is the block step (prologue then attention, self-attention);
    ``run_attention`` is attention alone over separate query and key extents
    (grouped query ranges).
    """

    def __init__(self, rows: int, n_heads: int, heads_per_group: int = 6, device=None,
                 kv_rows: Optional[int] = None, group_sizes: Optional[Sequence[int]] = None):
        dev = torch.device(device if device is not None else "cuda")
        bf = torch.bfloat16
        kv_rows = rows if kv_rows is None else kv_rows
        self.rows, self.kv_rows, self.n_heads = rows, kv_rows, n_heads
        self.q = torch.empty((rows, n_heads, HEAD_DIM), dtype=bf, device=dev)
        self.k = torch.empty((kv_rows, n_heads, HEAD_DIM), dtype=bf, device=dev)
        self.v = torch.empty_like(self.k)
        self.out = torch.empty_like(self.q)
        self.wq = torch.empty((n_heads, HEAD_DIM), dtype=bf, device=dev)
        self.wk = torch.empty_like(self.wq)
        self.pos = torch.empty((rows, 3), dtype=torch.int32, device=dev)
        self.groups = head_groups(n_heads, heads_per_group, group_sizes)
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.s_comp = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
        # Prologues run on a stream of their own, each as soon as its group's
        # Q and K have landed, so that attention launches follow one another.
        self.s_pro = torch.cuda.Stream(device=dev, priority=-1)

    def run_attention(self, q, k, v, cu_seqlens_q, cu_seqlens_kv, valid_len, out, scale=None,
                      stream=None) -> None:
        """Attention alone from pinned host Q, K, V to the pinned host out,
        with the same head-group overlap as ``run``; the arguments are those
        of ``attention``."""
        def compute(h0, h1, sc):
            attention(self.q[:, h0:h1], self.k[:, h0:h1], self.v[:, h0:h1], cu_seqlens_q,
                      cu_seqlens_kv, valid_len, scale, self.out[:, h0:h1], sc)
        self._pipeline(q, k, v, out, compute, None, stream)

    def run(self, q, k, v, wq, wk, pos_thw, cu_seqlens, valid_len, out,
            rot=(32, 48, 48), theta=10000.0, eps=1e-6, scale=None, stream=None) -> None:
        """Queue one block step after the work already on ``stream`` (default:
        the current stream); ``stream`` waits for the whole step, so a
        synchronise on it (or an event recorded on it) sees ``out`` filled.
        Q, K, V, weights and positions are read from the host tensors; the
        device copies of Q and K are normalised in place."""
        # The prologue of a group needs only its Q and K: it runs (on its own
        # stream) while the group's V is still being copied in.
        def prologue(h0, h1, sc):
            _block_prologue(self.q[:, h0:h1], self.k[:, h0:h1], self.wq[h0:h1], self.wk[h0:h1],
                            self.pos, cu_seqlens, valid_len, rot, theta, eps, sc)

        def compute(h0, h1, sc):
            attention(self.q[:, h0:h1], self.k[:, h0:h1], self.v[:, h0:h1], cu_seqlens,
                      cu_seqlens, valid_len, scale, self.out[:, h0:h1], sc)

        def small_inputs():
            self.wq.copy_(wq, non_blocking=True)
            self.wk.copy_(wk, non_blocking=True)
            self.pos.copy_(pos_thw, non_blocking=True)
        self._pipeline(q, k, v, out, compute, small_inputs, stream, prologue)

    def _pipeline(self, q, k, v, out, compute, small_inputs, stream, prologue=None):
        cur = stream if stream is not None else torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        for s in (self.s_in, self.s_out, *self.s_comp, self.s_pro):
            s.wait_event(start)
        if small_inputs is not None:
            with torch.cuda.stream(self.s_in):
                small_inputs()
        for i, (h0, h1) in enumerate(self.groups):
            sc = self.s_comp[i % 2]
            for dev_t, host_t in ((self.q, q), (self.k, k)):
                copy_2d(dev_t[:, h0:h1], host_t[:, h0:h1], self.s_in)
            if prologue is not None:
                qk_landed = torch.cuda.Event()
                qk_landed.record(self.s_in)
                self.s_pro.wait_event(qk_landed)
                prologue(h0, h1, self.s_pro)
                normed = torch.cuda.Event()
                normed.record(self.s_pro)
                sc.wait_event(normed)
            copy_2d(self.v[:, h0:h1], v[:, h0:h1], self.s_in)
            landed = torch.cuda.Event()
            landed.record(self.s_in)
            sc.wait_event(landed)
            compute(h0, h1, sc)
            done = torch.cuda.Event()
            done.record(sc)
            self.s_out.wait_event(done)
            copy_2d(out[:, h0:h1], self.out[:, h0:h1], self.s_out)
        for s in (self.s_out, *self.s_comp, self.s_pro):
            ev = torch.cuda.Event()
            ev.record(s)
            cur.wait_event(ev)


def status_word() -> int:
    """Synchronise the device; return and clear the device status bits
    (0 = no bounded wait gave up since the last read)."""
    val = ctypes.c_uint32(0)
    st = lib().h3_status_word(ctypes.byref(val))
    if st not in (0, -6):  # H3_ERR_TIMEOUT still reports the bits
        _check(st)
    return val.value
