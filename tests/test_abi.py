"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol the public headers declare, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import glob
import os
import re

import pytest
import torch

from packed_sequence_attention_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
H3_OK, ARG, ALIGN, SHAPE, ARCH, LAUNCH, TIMEOUT, DEVICE = 0, -1, -2, -3, -4, -5, -6, -7
A = 0x10000  # a 16-byte-aligned fake device address; never dereferenced on the host


def declared_symbols():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(h3_\w+)\s*\(", text))
    return sorted(names)


def test_headers_declare_the_boundary():
    names = declared_symbols()
    assert {"h3_qk_norm_rope", "h3_attention", "h3_last_error", "h3_status_word"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _binding.SIGNATURES, f"{name} has no binding"


def test_version(lib):
    assert lib.h3_version() == 10000


def _i32(vals):
    return ctypes.cast((ctypes.c_int32 * len(vals))(*vals), _binding.c_i32p)


def norm_rope(lib, **kw):
    a = dict(q=A, qs=5376, k=A + 0x100000, ks=5376, wq=A, wk=A, pos=A, n=10, H=42, D=128,
             rt=32, rh=48, rw=48, theta=10000.0, eps=1e-6, stream=None)
    a.update(kw)
    return lib.h3_qk_norm_rope(a["q"], a["qs"], a["k"], a["ks"], a["wq"], a["wk"], a["pos"],
                               a["n"], a["H"], a["D"], a["rt"], a["rh"], a["rw"], a["theta"],
                               a["eps"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), ARG), (dict(H=0), ARG), (dict(D=64), SHAPE), (dict(rt=31), SHAPE),
    (dict(H=449, qs=449 * 128, ks=449 * 128), SHAPE),
    (dict(rt=-2), SHAPE), (dict(rt=64, rh=64, rw=2), SHAPE), (dict(theta=0.0), ARG),
    (dict(theta=float("inf")), ARG), (dict(eps=-1.0), ARG), (dict(eps=float("nan")), ARG),
    (dict(qs=5375), SHAPE), (dict(ks=100), SHAPE), (dict(q=None), ARG), (dict(pos=None), ARG),
    (dict(k=A), ARG), (dict(q=A + 8), ALIGN), (dict(wk=A + 4), ALIGN), (dict(pos=A + 2), ALIGN),
    (dict(qs=5380), ALIGN), (dict(ks=5377), ALIGN),
])
def test_norm_rope_rejects_on_host(lib, kw, code):
    assert norm_rope(lib, **kw) == code
    assert lib.h3_last_error().decode() != ""


def test_norm_rope_zero_rows_is_a_no_op(lib):
    assert norm_rope(lib, n=0, q=None, k=None) == H3_OK


def norm_rope_varlen(lib, **kw):
    a = dict(q=A, qs=5376, k=A + 0x100000, ks=5376, wq=A, wk=A, pos=A, cu=[0, 256, 512],
             valid=[250, 256], n_seq=None, H=42, D=128, rt=32, rh=48, rw=48, theta=10000.0,
             eps=1e-6, stream=None)
    a.update(kw)
    n_seq = a["n_seq"] if a["n_seq"] is not None else (len(a["cu"]) - 1 if a["cu"] else 1)
    return lib.h3_qk_norm_rope_varlen(a["q"], a["qs"], a["k"], a["ks"], a["wq"], a["wk"], a["pos"],
                                      _i32(a["cu"]) if a["cu"] is not None else None,
                                      _i32(a["valid"]) if a["valid"] is not None else None,
                                      n_seq, a["H"], a["D"], a["rt"], a["rh"], a["rw"],
                                      a["theta"], a["eps"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(n_seq=0), ARG), (dict(n_seq=17, cu=[0] * 18, valid=None), ARG), (dict(cu=None), ARG),
    (dict(cu=[1, 256, 512]), ARG), (dict(cu=[0, 256, 100]), ARG), (dict(valid=[257, 0]), ARG),
    (dict(valid=[0, -1]), ARG), (dict(H=0), ARG), (dict(D=64), SHAPE), (dict(rt=31), SHAPE),
    (dict(qs=100), SHAPE), (dict(theta=0.0), ARG), (dict(eps=-1.0), ARG), (dict(k=A), ARG),
    (dict(q=None), ARG), (dict(pos=None), ARG), (dict(q=A + 8), ALIGN), (dict(pos=A + 2), ALIGN),
    (dict(ks=5377), ALIGN), (dict(cu=[0, 1 << 30, (1 << 30) + 2], valid=None), SHAPE),
])
def test_norm_rope_varlen_rejects_on_host(lib, kw, code):
    assert norm_rope_varlen(lib, **kw) == code
    assert lib.h3_last_error().decode() != ""


def test_norm_rope_varlen_no_valid_row_is_a_no_op(lib):
    assert norm_rope_varlen(lib, valid=[0, 0], q=None, k=None, pos=None) == H3_OK
    assert norm_rope_varlen(lib, cu=[0, 0, 0], valid=None, q=None, k=None) == H3_OK


def norm_rope_lora(lib, **kw):
    a = dict(q=A, qs=5376, dq=A + 0x200000, dqs=5376, k=A + 0x100000, ks=5376, dk=A + 0x300000,
             dks=5376, wq=A, wk=A, pos=A, n=10, H=42, D=128, rt=32, rh=48, rw=48, theta=10000.0,
             eps=1e-6, stream=None)
    a.update(kw)
    return lib.h3_qk_norm_rope_lora(a["q"], a["qs"], a["dq"], a["dqs"], a["k"], a["ks"], a["dk"],
                                    a["dks"], a["wq"], a["wk"], a["pos"], a["n"], a["H"], a["D"],
                                    a["rt"], a["rh"], a["rw"], a["theta"], a["eps"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dq=None), ARG), (dict(dk=None), ARG), (dict(dq=A + 8), ALIGN), (dict(dks=5380), ALIGN),
    (dict(dqs=100), SHAPE), (dict(H=221, qs=221 * 128, ks=221 * 128, dqs=221 * 128,
                                  dks=221 * 128), SHAPE),
    (dict(n=-1), ARG), (dict(D=64), SHAPE), (dict(k=A), ARG), (dict(rw=50), SHAPE),
])
def test_norm_rope_lora_rejects_on_host(lib, kw, code):
    assert norm_rope_lora(lib, **kw) == code


def test_norm_rope_lora_zero_rows_is_a_no_op(lib):
    assert norm_rope_lora(lib, n=0, q=None, k=None, dq=None, dk=None) == H3_OK


def attn(lib, **kw):
    a = dict(q=A, qs=5376, k=A, ks=5376, v=A, vs=5376, o=A + 0x100000, os=5376,
             cq=[0, 256], ckv=[0, 256], valid=[250], n_seq=None, H=42, D=128, scale=0.08838,
             stream=None)
    a.update(kw)
    n_seq = a["n_seq"] if a["n_seq"] is not None else (len(a["cq"]) - 1 if a["cq"] else 1)
    return lib.h3_attention(a["q"], a["qs"], a["k"], a["ks"], a["v"], a["vs"], a["o"], a["os"],
                            _i32(a["cq"]) if a["cq"] is not None else None,
                            _i32(a["ckv"]) if a["ckv"] is not None else None,
                            _i32(a["valid"]) if a["valid"] is not None else None,
                            n_seq, a["H"], a["D"], a["scale"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(n_seq=0), ARG), (dict(n_seq=17, cq=[0] * 18, ckv=[0] * 18, valid=None), ARG),
    (dict(H=0), ARG), (dict(D=256), SHAPE), (dict(scale=0.0), ARG), (dict(scale=-1.0), ARG),
    (dict(scale=float("nan")), ARG), (dict(cq=None), ARG), (dict(cq=[1, 256]), ARG),
    (dict(ckv=[0, 256, 100], cq=[0, 10, 20], valid=None), ARG),
    (dict(valid=[257]), ARG), (dict(valid=[-1]), ARG),
    (dict(cq=[0, 100], ckv=[0, 256], valid=[101]), ARG),
    (dict(qs=100), SHAPE), (dict(os=5000), SHAPE), (dict(v=None), ARG), (dict(o=None), ARG),
    (dict(q=A + 2), ALIGN), (dict(o=A + 8), ALIGN), (dict(ks=5377), ALIGN), (dict(os=5380), ALIGN),
])
def test_attention_rejects_on_host(lib, kw, code):
    assert attn(lib, **kw) == code
    assert lib.h3_last_error().decode() != ""


def groups_call(lib, groups, **kw):
    a = dict(q=A, qs=5376, k=A, ks=5376, v=A, vs=5376, kc=A + 0x400000, kcs=5376,
             vc=A + 0x500000, vcs=5376, o=A + 0x100000, os=5376, n=None, H=42, D=128,
             scale=0.08838, stream=None)
    a.update(kw)
    arr = (_binding.AttnGroup * max(len(groups), 1))(*[_binding.AttnGroup(*g) for g in groups])
    n = a["n"] if a["n"] is not None else len(groups)
    return lib.h3_attention_groups(a["q"], a["qs"], a["k"], a["ks"], a["v"], a["vs"], a["kc"],
                                   a["kcs"], a["vc"], a["vcs"], a["o"], a["os"],
                                   ctypes.cast(arr, ctypes.c_void_p), n, a["H"], a["D"],
                                   a["scale"], a["stream"])


G_OK = [(0, 100, 0, 100, 0, 50)]


@pytest.mark.parametrize("groups,kw,code", [
    (G_OK, dict(n=0), ARG), (G_OK, dict(n=17), ARG), ([(0, -1, 0, 1, 0, 0)], {}, ARG),
    ([(0, 10, -5, 1, 0, 0)], {}, ARG), ([(2 ** 31 - 5, 10, 0, 1, 0, 0)], {}, ARG),
    ([(0, 10, 0, 5, 0, 0), (5, 10, 0, 5, 0, 0)], {}, ARG),          # overlapping query ranges
    (G_OK, dict(kc=None), ARG), (G_OK, dict(vc=A + 8), ALIGN), (G_OK, dict(kcs=100), SHAPE),
    (G_OK, dict(D=64), SHAPE), (G_OK, dict(scale=0.0), ARG), (G_OK, dict(os=5380), ALIGN),
])
def test_attention_groups_rejects_on_host(lib, groups, kw, code):
    assert groups_call(lib, groups, **kw) == code


@pytest.mark.parametrize("args,code", [
    (dict(n=0), ARG), (dict(n=2048 * 128 + 1), ARG), (dict(D=64), SHAPE), (dict(x=None), ARG),
    (dict(x=A + 8), ALIGN), (dict(m=A + 2), ALIGN), (dict(s=100), SHAPE),
])
def test_block_means_rejects_on_host(lib, args, code):
    a = dict(x=A, s=5376, n=1000, H=42, D=128, m=A)
    a.update(args)
    assert lib.h3_block_means(a["x"], a["s"], a["n"], a["H"], a["D"], a["m"], None) == code


@pytest.mark.parametrize("args,code", [
    (dict(n=0), ARG), (dict(n=2048 * 128 + 1), ARG), (dict(D=64), SHAPE), (dict(k=None), ARG),
    (dict(km=None), ARG), (dict(k=A + 8), ALIGN), (dict(km=A + 2), ALIGN), (dict(ks=100), SHAPE),
    (dict(qs=5380), ALIGN), (dict(km=A), ARG), (dict(H=0), ARG),
])
def test_block_means_qk_rejects_on_host(lib, args, code):
    a = dict(q=A, qs=5376, k=A + 0x100000, ks=5376, n=1000, H=42, D=128, qm=A, km=A + 0x200000)
    a.update(args)
    assert lib.h3_block_means_qk(a["q"], a["qs"], a["k"], a["ks"], a["n"], a["H"], a["D"],
                                 a["qm"], a["km"], None) == code


@pytest.mark.parametrize("args,code", [
    (dict(nkb=2049), ARG), (dict(nqb=0), ARG), (dict(tau=float("inf")), ARG),
    (dict(npre=9), ARG), (dict(npre=-1), ARG), (dict(lists=None), ARG), (dict(qm=A + 4), ALIGN),
    (dict(counts=A + 2), ALIGN),
])
def test_block_select_rejects_on_host(lib, args, code):
    a = dict(qm=A, km=A, nqb=8, nkb=8, H=2, scale=0.1, tau=1.0, npre=1, sc=None, lists=A, counts=A)
    a.update(args)
    assert lib.h3_block_select(a["qm"], a["km"], a["nqb"], a["nkb"], a["H"], a["scale"], a["tau"],
                               a["npre"], a["sc"], a["lists"], a["counts"], None) == code


@pytest.mark.parametrize("args,code", [
    (dict(n=0), ARG), (dict(D=256), SHAPE), (dict(lists=None), ARG), (dict(q=A + 2), ALIGN),
    (dict(os_=100), SHAPE), (dict(scale=-1.0), ARG), (dict(counts=A + 1), ALIGN),
    (dict(npre=-1), ARG), (dict(npre=9), ARG),             # 1,000 rows: 8 blocks
])
def test_sparse_attention_rejects_on_host(lib, args, code):
    a = dict(q=A, k=A, v=A, o=A, os_=5376, n=1000, H=42, D=128, lists=A, counts=A, npre=0,
             scale=0.1)
    a.update(args)
    assert lib.h3_sparse_attention(a["q"], 5376, a["k"], 5376, a["v"], 5376, a["o"], a["os_"],
                                   a["n"], a["H"], a["D"], a["lists"], a["counts"], a["npre"],
                                   a["scale"], None) == code


def test_wire_record_sizes_on_host(lib):
    assert [lib.h3_wire_record_bytes(0, f) for f in (0, 1, 2)] == [768, 400, -1]
    assert [lib.h3_wire_record_bytes(1, f) for f in (0, 1, 2)] == [256, 144, 128]
    assert lib.h3_wire_record_bytes(2, 0) == -1


@pytest.mark.parametrize("args,code", [
    (dict(nd=4), ARG), (dict(nd=0), ARG), (dict(fmt=2), ARG), (dict(q=None), ARG),
    (dict(q=A + 4), ALIGN), (dict(ks=5375), SHAPE), (dict(wire=A + 8), ALIGN), (dict(H=0), ARG),
    (dict(n=2 ** 33), ARG), (dict(n=-1), ARG),
    (dict(v=A + 8), ALIGN), (dict(qs=5376 + 4), ALIGN),          # INT8: 16-byte vectors
])
def test_pack_qkv_rejects_on_host(lib, args, code):
    a = dict(q=A, qs=5376, k=A, ks=5376, v=A, vs=5376, n=10, H=42, nd=2, fmt=1, wire=A)
    a.update(args)
    assert lib.h3_pack_qkv(a["q"], a["qs"], a["k"], a["ks"], a["v"], a["vs"], a["n"], a["H"],
                           a["nd"], a["fmt"], a["wire"], None) == code


def test_pack_qkv_bf16_allows_8_byte_alignment(lib):
    """BF16 records move 8-byte vectors: an 8-byte aligned view passes the host
    checks (and, without a GPU, stops at the device check)."""
    st = lib.h3_pack_qkv(A + 8, 5376 + 4, A, 5376, A, 5376, 10, 42, 2, 0, A, None)
    assert st in (DEVICE, ARCH) or (torch.cuda.is_available() and st == ARG)


def unpack_qkv(lib, **kw):
    a = dict(wire=A, n=10, hl=21, fmt=1, q=A, qs=2688, k=A + 0x100000, ks=2688, v=A + 0x200000,
             vs=2688)
    a.update(kw)
    return lib.h3_unpack_qkv(a["wire"], a["n"], a["hl"], a["fmt"], a["q"], a["qs"], a["k"], a["ks"],
                             a["v"], a["vs"], None)


@pytest.mark.parametrize("args,code", [
    (dict(fmt=2), ARG), (dict(wire=None), ARG), (dict(wire=A + 8), ALIGN), (dict(qs=100), SHAPE),
    (dict(q=A + 8), ALIGN), (dict(ks=2688 + 4), ALIGN), (dict(v=A + 4), ALIGN),
])
def test_unpack_qkv_int8_rejects_on_host(lib, args, code):
    assert unpack_qkv(lib, **args) == code


def test_unpack_qkv_bf16_allows_8_byte_alignment(lib):
    """BF16 records move 8-byte vectors: 8-byte aligned outputs pass the host
    checks (and, without a GPU, stop at the device check); INT8 writes 16-byte
    vectors and needs 16-byte alignment."""
    st = unpack_qkv(lib, fmt=0, q=A + 8, qs=2688 + 4)
    assert st in (DEVICE, ARCH) or (torch.cuda.is_available() and st == ARG)
    assert unpack_qkv(lib, fmt=1, q=A + 8, qs=2688 + 4) == ALIGN


@pytest.mark.parametrize("args,code", [
    (dict(ns=5), ARG), (dict(fmt=3), ARG), (dict(o=None), ARG), (dict(os_=100), SHAPE),
    (dict(wire=None), ARG), (dict(wire=A + 4), ALIGN), (dict(n=2 ** 33), ARG),
])
def test_merge_heads_rejects_on_host(lib, args, code):
    a = dict(wire=A, n=10, H=42, ns=2, fmt=2, o=A, os_=5376)
    a.update(args)
    assert lib.h3_merge_heads(a["wire"], a["n"], a["H"], a["ns"], a["fmt"], a["o"], a["os_"],
                              None) == code


@pytest.mark.parametrize("args,code", [
    (dict(dst=None), ARG), (dict(src=None), ARG), (dict(h=-1), ARG), (dict(w=-4), ARG),
    (dict(dp=100), SHAPE), (dict(sp=100), SHAPE),
])
def test_copy_2d_rejects_on_host(lib, args, code):
    a = dict(dst=A, dp=10752, src=A, sp=10752, w=1536, h=10)
    a.update(args)
    assert lib.h3_copy_2d(a["dst"], a["dp"], a["src"], a["sp"], a["w"], a["h"], None) == code


def test_copy_2d_empty_is_a_no_op(lib):
    assert lib.h3_copy_2d(None, 0, None, 0, 1536, 0, None) == 0
    assert lib.h3_copy_2d(None, 0, None, 0, 0, 10, None) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_device_error(lib):
    assert attn(lib) == DEVICE
    assert norm_rope(lib) == DEVICE
    assert norm_rope_lora(lib) == DEVICE
    assert groups_call(lib, [(0, 10, 0, 10, 0, 0)], kc=None, vc=None) == DEVICE
    v = ctypes.c_uint32(0)
    assert lib.h3_status_word(ctypes.byref(v)) == DEVICE


def test_status_word_null(lib):
    assert lib.h3_status_word(None) == ARG


def test_fault_hook_validates(lib):
    assert lib.h3_debug_fault_next_attention(7) == ARG
    assert lib.h3_debug_fault_next_attention(0) == H3_OK


def test_python_api_fails_loudly_without_library(monkeypatch, tmp_path):
    import packed_sequence_attention_gb300 as h3
    monkeypatch.setattr(_binding, "_LIB", None)
    monkeypatch.setattr(_binding, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        h3.lib()
