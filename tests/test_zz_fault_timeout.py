"""Failure path of the attention kernel, exercised without faulting a GPU.

The test hook makes the TMA producer of every CTA skip K/V tile 1, so the
MMA issuer waits for data that never comes.  Its bounded wait (about 2 s of
wall clock) must give up, set a timeout bit in the status word, drain the
copies and MMAs already in flight, free TMEM and return; the CUDA context
must stay usable, which a normal launch right after checks.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import packed_sequence_attention_gb300 as h3
from oracle import oracle as O

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128.0)
TIMEOUT_BITS = 0x1 | 0x2 | 0x4


def test_bounded_wait_gives_up_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib = h3.lib()
    gen = torch.Generator().manual_seed(7)
    q, k, v = (torch.randn((300, 2, 128), generator=gen).to(torch.bfloat16).cuda() for _ in range(3))
    assert h3.status_word() == 0
    assert lib.h3_debug_fault_next_attention(1) == 0
    h3.attention(q, k, v, [0, 300], [0, 300], None, SCALE)
    val = ctypes.c_uint32(0)
    assert lib.h3_status_word(ctypes.byref(val)) == -6  # H3_ERR_TIMEOUT
    assert val.value & TIMEOUT_BITS, f"status {val.value:#x}"
    # the hook is one-shot and the context still works
    out = h3.attention(q, k, v, [0, 300], [0, 300], None, SCALE)
    torch.cuda.synchronize()
    assert h3.status_word() == 0
    ref = O.attention(O.widen(q), O.widen(k), O.widen(v), [0, 300], [0, 300], None, SCALE)
    got = O.widen(out)
    assert np.abs(got - ref).max() <= 2e-2
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3
