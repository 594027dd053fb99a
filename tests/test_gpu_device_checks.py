"""Pointers that are not memory of the current device are rejected on the
host, before any launch: by the Python wrappers (CPU tensors, wrong head
counts) and by the C ABI itself (pinned host memory).

The C-level case passes pinned host memory, which this GPU can address
through unified virtual addressing, to a kernel that uses plain loads and
stores (the output-record pack), so the call is harmless even if the check
let it through; the test only asserts that it did not."""
import ctypes

import pytest
import torch

import packed_sequence_attention_gb300 as h3
from packed_sequence_attention_gb300 import _binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    h3.lib()
    yield
    assert h3.status_word() == 0


def _bf16(rows, H, device="cuda"):
    return torch.zeros((rows, H, 128), dtype=torch.bfloat16, device=device)


def test_wrappers_reject_host_tensors():
    q, k, v = _bf16(256, 2), _bf16(256, 2), _bf16(256, 2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        h3.attention(q.cpu(), k, v, [0, 256], [0, 256])
    with pytest.raises(ValueError, match="CUDA tensor"):
        h3.attention(q, k, v, [0, 256], [0, 256], out=_bf16(256, 2, "cpu"))
    w = torch.ones((2, 128), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros((256, 3), dtype=torch.int32)
    with pytest.raises(ValueError, match="pos_thw must be a CUDA tensor"):
        h3.qk_norm_rope(q, k, w, w, pos)
    with pytest.raises(ValueError, match="wk must be a CUDA tensor"):
        h3.qk_norm_rope(q, k, w, w.cpu(), pos.cuda())
    lists = torch.zeros((2, 2, 2), dtype=torch.int32)
    counts = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError, match="lists must be a CUDA tensor"):
        h3.sparse_attention(q, k, v, lists, counts, 256)
    with pytest.raises(ValueError, match="CUDA tensor"):
        h3.block_means(q.cpu(), 256)
    with pytest.raises(ValueError, match="CUDA tensor"):
        h3.pack_out(q.cpu(), h3.WIRE_FP8)
    torch.cuda.synchronize()


def test_wrappers_reject_head_count_mismatch():
    q, v = _bf16(256, 4), _bf16(256, 4)
    k_narrow = _bf16(256, 4)[:, :2]        # 2 heads, row stride of 4: passes the stride checks
    with pytest.raises(ValueError, match="must have 4 heads"):
        h3.attention(q, k_narrow, v, [0, 256], [0, 256])
    with pytest.raises(ValueError, match="must have 4 heads"):
        h3.attention(q, _bf16(256, 4), v, [0, 256], [0, 256], out=_bf16(256, 4)[:, :3])
    with pytest.raises(ValueError, match="must have 4 heads"):
        h3.attention_groups(q, _bf16(256, 4), v, [(0, 10, 0, 10, 0, 5)],
                            k_cache=_bf16(64, 4)[:, :1], v_cache=_bf16(64, 4))
    w = torch.ones((4, 128), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros((256, 3), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError, match="must have 4 heads"):
        h3.qk_norm_rope(q, k_narrow, w, w, pos)
    torch.cuda.synchronize()


def test_c_abi_rejects_pinned_host_memory():
    lib = h3.lib()
    host = torch.zeros((64, 2, 128), dtype=torch.bfloat16).pin_memory()
    wire = torch.empty((64, 2, 128), dtype=torch.uint8, device="cuda")
    st = lib.h3_pack_out(host.data_ptr(), 256, 64, 2, h3.WIRE_FP8, wire.data_ptr(), None)
    assert st == -1, st
    assert "host memory" in lib.h3_last_error().decode()
    dev = _bf16(64, 2)
    st = lib.h3_pack_out(dev.data_ptr(), 256, 64, 2, h3.WIRE_FP8, ctypes.c_void_p(host.data_ptr()),
                         None)
    assert st == -1 and "wire is host memory" in lib.h3_last_error().decode()
    # the same call on device memory goes through
    st = lib.h3_pack_out(dev.data_ptr(), 256, 64, 2, h3.WIRE_FP8, wire.data_ptr(), None)
    assert st == 0, lib.h3_last_error().decode()
    torch.cuda.synchronize()
    assert (wire == 0).all()
