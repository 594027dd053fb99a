"""Host logic of bench.py that needs no GPU: the kernel-source digest that keys
the committed DRAM traffic (comments do not count), and the config object both
arms report."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from packed_sequence_attention_gb300 import workloads as W  # noqa: E402


def test_digest_ignores_comments_but_not_code():
    src = b"""// a file comment
__global__ void k(int* p) {  // trailing comment
  /* a block
     comment */
  p[0] = 1;

}
"""
    recommented = b"""// another comment
__global__ void k(int* p) {
  p[0] = 1;  /* moved */
}
"""
    changed = src.replace(b"p[0] = 1;", b"p[0] = 2;")
    assert bench._code_only(src) == bench._code_only(recommented)
    assert bench._code_only(src) != bench._code_only(changed)


def test_both_arms_report_the_same_config():
    for name in ("full", "stage1_batch2", "grouped_chunk"):
        w = W.workload(name)
        cfg = bench.workload_config(w, 1)
        assert cfg["workload"] == name
        assert cfg["attention_flop_per_step"] == w.attention_flops()
        assert cfg["parallelism"] == "single GPU"
        assert bench.workload_config(w, 4)["parallelism"] == "replicas x4"


def _oracle_step(w, inp):
    """The whole step by the oracle, rounded to bf16 like a kernel output."""
    import numpy as np
    import torch
    from oracle import oracle as O
    out = torch.zeros_like(inp["out"])
    for b, s in enumerate(w.segments):
        q0, kv0 = inp["cu_seqlens_q"][b], inp["cu_seqlens_kv"][b]
        nq, nkv = s.n_valid_q(), s.n_valid_kv()
        q = O.widen(inp["q"][q0:q0 + nq])
        k = O.widen(inp["k"][kv0:kv0 + nkv])
        if w.self_attention:
            pos = inp["pos_thw"].numpy()
            q = O.qk_norm_rope(q, O.widen(inp["wq"]), pos[q0:q0 + nq])
            k = O.qk_norm_rope(k, O.widen(inp["wk"]), pos[kv0:kv0 + nkv])
        o = O.attention(q, k, O.widen(inp["v"][kv0:kv0 + nkv]), [0, nq], [0, nkv], None,
                        bench.SCALE)
        out[q0:q0 + nq] = torch.from_numpy(np.ascontiguousarray(o)).to(torch.bfloat16)
    return out


def test_config_gate_accepts_the_oracle_and_rejects_mistakes():
    """The per-config parity gate of the bench passes a correct step output
    and fails one with a wrong row, a nonzero padded row or a NaN."""
    from oracle import oracle as O
    w = W.custom("gate_case", 2, [W._seq(256, (2, 8, 8), 64, 58), W._seq(192, (1, 8, 8), 60, 6)])
    inp = W.make_inputs(w, seed=5, fill="B")
    fresh = dict(inp)
    good = _oracle_step(w, inp)
    g = dict(inp, out=good.clone())
    ok, info = bench.config_gate(O, w, fresh, g)
    assert ok and info["rows_checked"] == 48 and info["padded_rows_zero"], info
    bad = good.clone()
    bad[256 + 129] *= 1.5                  # the last valid row of the second sequence
    ok, info = bench.config_gate(O, w, fresh, dict(inp, out=bad))
    assert not ok
    bad = good.clone()
    bad[252, 1, 7] = 1.0                   # a padded output row
    ok, info = bench.config_gate(O, w, fresh, dict(inp, out=bad))
    assert not ok and not info["padded_rows_zero"]
    bad = good.clone()
    bad[0, 0, 0] = float("nan")
    ok, _ = bench.config_gate(O, w, fresh, dict(inp, out=bad))
    assert not ok
