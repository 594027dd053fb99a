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
