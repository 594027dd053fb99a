"""GPU: launches from several host threads at once (each on its own stream,
with its own inputs) give bitwise the single-threaded results: the library's
per-device caches and the thread-local error message are safe to share."""
import threading

import pytest
import torch

import packed_sequence_attention_gb300 as h3
from packed_sequence_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu
SCALE = 128 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    h3.lib()
    yield
    assert h3.status_word() == 0


def _step(g, q, k, out, stream):
    h3.attention_block(q, k, g["v"], g["wq"], g["wk"], g["pos_thw"], g["cu_seqlens_q"],
                       g["valid_len"], scale=SCALE, out=out, stream=stream)


def test_concurrent_threads_match_single_threaded():
    n_threads, reps = 4, 3
    ws = [W.custom(f"t{i}", 6, [W.Segment(700 + 64 * i, 700 + 64 * i, 650 + 60 * i,
                                          (2, 10, 15 + i), 250, 100 + 40 * i)])
          for i in range(n_threads)]
    gs = [W.make_inputs(w, device="cuda", seed=1000 + i) for i, w in enumerate(ws)]
    refs = []
    for g in gs:
        out = torch.empty_like(g["out"])
        _step(g, g["q"].clone(), g["k"].clone(), out, torch.cuda.current_stream())
        refs.append(out)
    torch.cuda.synchronize()
    results, errors = [None] * n_threads, []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            g = gs[i]
            outs = []
            for _ in range(reps):
                out = torch.full_like(g["out"], float("nan"))
                _step(g, g["q"].clone(), g["k"].clone(), out, s)
                outs.append(out)
            s.synchronize()
            results[i] = outs
        except Exception as e:  # surfaced below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(n_threads):
        for out in results[i]:
            assert torch.equal(out.view(torch.int16), refs[i].view(torch.int16)), f"thread {i}"


def test_error_message_is_per_thread():
    lib = h3.lib()
    msgs = {}

    def bad(i):
        # each thread provokes its own argument error and reads its own message
        st = lib.h3_attention(None, 0, None, 0, None, 0, None, 0, None, None, None, i + 1, 1, 128,
                              0.1, None)
        msgs[i] = (st, lib.h3_last_error().decode())

    threads = [threading.Thread(target=bad, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert all(st < 0 and m for st, m in msgs.values())
