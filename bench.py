"""Benchmark of the packed-sequence attention hot path on GB300.

One step = the whole hot path over one packed-sequence block: the fused
Q/K RMSNorm + axial RoPE on the valid rows of every sequence, then attention
over the valid rows.  The default workload is the 58,816-row buffer holding
58,758 valid tokens, 42 heads x 128 channels (bf16).

Printed (rank 0, one JSON line): attention TFLOP/s over valid tokens for the
whole job (value), the same through the public API from pinned host buffers
(e2e), the roofline of the attention kernel, the prologue's GB/s, sampled
SM clocks, and the fp64 CPU oracle timed on a bounded sample (cpu_baseline).

``--impl reference`` times the CPU oracle instead (rank 0 only).
Multi-GPU runs are independent replicas (the method has no exchange step on
one GPU); value then sums the units of all ranks over the slowest rank.
"""
import os

os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

import argparse  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s (valid tokens) at 58,816-tok packed seq; % bf16 peak; prologue GB/s"
ROT = (32, 48, 48)
SCALE = 1.0 / math.sqrt(128.0)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"],
                    bf16_sustained=p["bf16_tflops_sustained"], source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "clocks.mem")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, mem, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
            try:
                mem.append(float(f[9]))
            except (IndexError, ValueError):
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "mem_mhz": float(np.median(mem)) if mem else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def mufu_bound(w, attn_ms, clocks, sms=152, ex2_per_clk_per_sm=32):
    """Secondary bound of the attention kernel: one ex2 per (valid query,
    valid key, head) on the MUFU, against 32 lanes per clock per SM (the rate
    the XU counters imply on this part) at the sampled median SM clock."""
    ex2 = float(w.n_heads * sum(s.n_valid_q() * s.n_valid_kv() for s in w.segments))
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz")
    if not mhz or attn_ms <= 0:
        return {"bound": "mufu_ex2", "ex2_per_launch": ex2, "frac": None}
    peak = sms * ex2_per_clk_per_sm * mhz * 1e6
    achieved = ex2 / (attn_ms * 1e-3)
    return {"bound": "mufu_ex2", "ex2_per_launch": ex2, "achieved_per_s": round(achieved, 0),
            "peak_per_s": round(peak, 0), "frac": round(achieved / peak, 4)}


# ------------------------------------------------------- replicas (N > 1)
def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings over all ranks: the slowest
    rank decides.  ``dist`` is torch.distributed (any backend) or None."""
    if dist is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_value(units_per_rank, ms_per_step, world):
    """Whole-job throughput in units/s x 1e-12 (TFLOP/s for FLOP): the units
    every rank processed in one step over the slowest rank's step time.
    Ranks are independent replicas with the same per-rank work (weak
    scaling)."""
    return units_per_rank * world / (ms_per_step * 1e-3) / 1e12


# -------------------------------------------------------------- the GPU arm
def prologue_launches(w):
    """One launch covers every sequence's valid rows (none when no row is valid)."""
    return int(w.self_attention and any(s.n_valid_q() for s in w.segments))


def launches_per_step(w):
    return prologue_launches(w) + 1


def run_prologue(h3, g, w):
    """The prologue on every sequence's valid rows, in one launch."""
    if prologue_launches(w):
        h3.qk_norm_rope_varlen(g["q"], g["k"], g["wq"], g["wk"], g["pos_thw"], g["cu_seqlens_q"],
                               g["valid_len"], rot=ROT)


def run_step(h3, g, w, ev=None):
    """Prologue on each sequence's valid rows, then attention.  With ``ev``
    (four events), records prologue and attention boundaries."""
    if ev is not None:
        ev[0].record()
    run_prologue(h3, g, w)
    if ev is not None:
        ev[1].record()
    h3.attention(g["q"], g["k"], g["v"], g["cu_seqlens_q"], g["cu_seqlens_kv"], g["valid_len"],
                 SCALE, out=g["out"])
    if ev is not None:
        ev[2].record()


def parity_gate(h3, W, O, w):
    """Fail-closed check on the same build before any number is reported:
    the tiny packed sequence against the fp64 oracle."""
    inp = W.make_inputs("tiny", fill="B")
    g = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    run_step(h3, g, W.workload("tiny"))
    torch.cuda.synchronize()
    n = inp["valid_len"][0]
    pos = inp["pos_thw"].numpy()[:n]
    q = O.qk_norm_rope(O.widen(inp["q"][:n]), O.widen(inp["wq"]), pos)
    k = O.qk_norm_rope(O.widen(inp["k"][:n]), O.widen(inp["wk"]), pos)
    ref = O.attention(q, k, O.widen(inp["v"][:n]), [0, n], [0, n], None, SCALE)
    got = O.widen(g["out"])
    err = float(np.abs(got[:n] - ref).max())
    rel = float(np.linalg.norm(got[:n] - ref) / np.linalg.norm(ref))
    ok = err <= 2e-2 and rel <= 5e-3 and bool((got[n:] == 0).all()) and h3.status_word() == 0
    return ok, {"max_abs": err, "rel_l2": rel}


def cpu_baseline(O, inp_cpu, w, n_heads_sample, n_rows_sample):
    """The fp64 oracle as it stands, on a bounded sample: n_rows_sample
    query rows of the first sequence x n_heads_sample heads, each against all
    valid keys of its sequence (prologue of those keys included)."""
    s = w.segments[0]
    q0, kv0 = inp_cpu["cu_seqlens_q"][0], inp_cpu["cu_seqlens_kv"][0]
    nq, nkv = s.n_valid_q(), s.n_valid_kv()
    rows = np.linspace(0, nq - 1, n_rows_sample).astype(np.int64) + q0
    rows_t = torch.as_tensor(rows)
    t0 = time.perf_counter()
    for h in range(n_heads_sample):
        qs = O.widen(inp_cpu["q"][rows_t, h:h + 1])
        kh = O.widen(inp_cpu["k"][kv0:kv0 + nkv, h:h + 1])
        vh = O.widen(inp_cpu["v"][kv0:kv0 + nkv, h:h + 1])
        if w.self_attention:
            pos = inp_cpu["pos_thw"].numpy()
            qs = O.qk_norm_rope(qs, O.widen(inp_cpu["wq"][h:h + 1]), pos[rows])
            kh = O.qk_norm_rope(kh, O.widen(inp_cpu["wk"][h:h + 1]), pos[kv0:kv0 + nkv])
        O.attention(qs, kh, vh, [0, len(rows)], [0, nkv], None, SCALE)
    dt = time.perf_counter() - t0
    flops = 4.0 * 128 * nkv * len(rows) * n_heads_sample
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "ms_per_query_row_head": round(dt / (len(rows) * n_heads_sample) * 1e3, 3),
            # the whole workload at the sample's rate (not run)
            "extrapolated_full_s": round(w.attention_flops() / (flops / dt), 1),
            "sample": f"{len(rows)} query rows x {n_heads_sample} heads of '{w.name}' against "
                      f"all {nkv} valid keys (fp64 NumPy oracle incl. the K prologue), "
                      f"{dt:.1f} s wall"}


def bench_gpu(args):
    import packed_sequence_attention_gb300 as h3
    from packed_sequence_attention_gb300 import workloads as W
    from oracle import oracle as O

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    h3.lib()
    pk = peaks()
    w = W.workload(args.config)

    ok, parity = parity_gate(h3, W, O, w)
    if not ok:
        raise SystemExit(f"parity gate failed: {parity}; no number reported")

    # ---- device-resident inputs (seeded, generated on the GPU)
    g = W.make_inputs(w, device=f"cuda:{local}", seed=W.default_seed(w) + rank)
    stream = torch.cuda.current_stream()
    if args.wire_only or args.next_only:
        if not w.self_attention:
            raise SystemExit("--wire-only / --next-only need a self-attention workload")
        if args.wire_only:
            res = {"wire_formats": wire_timing(h3, g, w, stream, pk)}
        else:
            res = {"lora_prologue": lora_prologue_timing(h3, g, w, stream, pk),
                   "sol_block_sparse": sol_attention_timing(h3, g, w, stream, pk)}
        if h3.status_word():
            raise SystemExit("device status word is nonzero after the timed calls")
        if rank == 0:
            print(json.dumps({"workload": w.name, "rows": w.segments[0].n_valid_q(), **res}))
        if dist is not None:
            dist.destroy_process_group()
        return
    for _ in range(args.warmup):
        run_step(h3, g, w)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            run_step(h3, g, w, evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    clk_summary = clk.summary()
    attn_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    step_each = [e[0].elapsed_time(e[2]) for e in evs]  # prologue start -> attention end
    # The prologue alone (in the step it follows the previous attention,
    # whose last output lines are still being written back from L2).
    pro_alone_ms = None
    if w.self_attention:
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(10):
            run_prologue(h3, g, w)
        a1.record(stream)
        torch.cuda.synchronize()
        pro_alone_ms = a0.elapsed_time(a1) / 10
    pro_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs])) if w.self_attention else 0.0
    ceiling = rmw_ceiling(g, w, stream) if w.self_attention else None
    lora = lora_prologue_timing(h3, g, w, stream, pk) if w.self_attention else None
    ref_cached = ref_cached_timing(h3, W, stream, pk) if w.name == "full" else None
    sol = sol_attention_timing(h3, g, w, stream, pk) if w.name == "full" else None
    wire = wire_timing(h3, g, w, stream, pk) if w.name == "full" else None
    if sol is not None:
        for r in [sol] + sol["tau_sweep"]:
            r["speedup_vs_dense_attention"] = round(attn_ms / r["total_ms"], 3)
    status = h3.status_word()
    if status:
        raise SystemExit(f"device status word {status:#x} after the timed region")
    ms_total = max_over_ranks([ms_total], dist, "cuda")[0]
    ms_step = ms_total / args.steps
    flops = w.attention_flops()
    value = whole_job_value(flops, ms_step, world)
    attn_tflops = flops / (attn_ms * 1e-3) / 1e12
    pro_gbs = w.prologue_bytes() / (pro_ms * 1e-3) / 1e9 if pro_ms > 0 else None

    if args.kernels_only:
        if rank == 0:
            print(json.dumps({"workload": w.name, "attention_ms": attn_ms, "prologue_ms": pro_ms,
                              "ms_per_step": ms_step, "attention_tflops": attn_tflops,
                              "prologue_gbs": pro_gbs, "clocks": clk.summary()}))
        if dist is not None:
            dist.destroy_process_group()
        return

    # ---- end to end through the public API, pinned host buffers
    host = {k: (v.cpu().pin_memory() if torch.is_tensor(v) else v) for k, v in
            W.make_inputs(w, device=f"cuda:{local}", seed=W.default_seed(w) + rank).items()}
    out_host = torch.empty_like(host["out"]).pin_memory()
    names = ["q", "k", "v"] + (["wq", "wk", "pos_thw"] if w.self_attention else [])
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = out_host.numel() * out_host.element_size()

    pipe = h3.HostPipeline(w.q_rows, w.n_heads, kv_rows=w.kv_rows)

    def e2e_step():
        # head groups copied in, computed and copied out on overlapping streams
        if w.self_attention:
            pipe.run(host["q"], host["k"], host["v"], host["wq"], host["wk"], host["pos_thw"],
                     host["cu_seqlens_q"], host["valid_len"], out_host, rot=ROT, scale=SCALE,
                     stream=stream)
        else:
            pipe.run_attention(host["q"], host["k"], host["v"], host["cu_seqlens_q"],
                               host["cu_seqlens_kv"], host["valid_len"], out_host, scale=SCALE,
                               stream=stream)

    for _ in range(min(args.warmup, 2)):
        e2e_step()
    torch.cuda.synchronize()
    # Each step is timed on its own (a step waits for the previous one to
    # finish, so steps do not overlap).  Host <-> device copies occasionally
    # stall for tens of milliseconds independently of this program; the
    # median step is the value, the mean and the slowest step are reported
    # beside it.
    e_steps = max(5, min(args.steps, 10))
    e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps + 1)]
    if dist is not None:
        dist.barrier()
    e_ev[0].record(stream)
    for i in range(e_steps):
        e2e_step()
        e_ev[i + 1].record(stream)
    torch.cuda.synchronize()
    e_each = [e_ev[i].elapsed_time(e_ev[i + 1]) for i in range(e_steps)]
    e_ms = float(np.median(e_each))
    e_mean = float(np.mean(e_each))
    e_ms, e_mean = max_over_ranks([e_ms, e_mean], dist, "cuda")
    e2e_value = whole_job_value(flops, e_ms, world)

    if rank != 0:
        dist.barrier()
        dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        fresh = W.make_inputs(w, device=f"cuda:{local}")  # unmodified inputs
        inp_cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in fresh.items()}
        del fresh
        cpu = cpu_baseline(O, inp_cpu, w, args.cpu_heads, args.cpu_rows)
    configs = None
    if not args.no_configs and w.name == "full":
        configs = config_sweep(h3, W, O, pk, [n for n in W.CONFIG_ORDER if n != w.name])
    traffic = committed_traffic(w)
    peak = pk["bf16_sustained"]
    mhz, max_mhz = clk_summary.get("sm_mhz"), clk_summary.get("sm_max_mhz")
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, N(1,0.1) norm weights, garbage pads)",
        "config": workload_config(w, world),
        "roofline": {"bound": "tensor", "achieved": round(attn_tflops, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(attn_tflops / peak, 4),
                     "frac_of_burst": round(attn_tflops / pk["bf16"], 4),
                     "peak_source": f"{pk['source']} bf16 (sustained; burst {pk['bf16']})",
                     "kernel": "attn_fwd_kernel", "traffic": traffic,
                     "secondary": mufu_bound(w, attn_ms, clk_summary)},
        "step_ms_percentiles": {q: round(float(np.percentile(step_each, int(q[1:]))), 4)
                                for q in ("p10", "p50", "p90")},
        "attention_ms": round(attn_ms, 4),
        "attention_tflops": round(attn_tflops, 2),
        "prologue_us": round(pro_ms * 1e3, 2) if pro_ms else None,
        "prologue_gbs": round(pro_gbs, 1) if pro_gbs else None,
        "prologue_frac_hbm_measured": round(pro_gbs / pk["hbm"], 4) if pro_gbs else None,
        "prologue_frac_8tbs": round(pro_gbs / 8000.0, 4) if pro_gbs else None,
        "prologue_alone_us": round(pro_alone_ms * 1e3, 2) if pro_alone_ms else None,
        "prologue_alone_gbs": round(w.prologue_bytes() / (pro_alone_ms * 1e-3) / 1e9, 1)
        if pro_alone_ms else None,
        "prologue_ceiling": ceiling,
        "prologue_ceiling_gbs": ceiling["gbs"] if ceiling else None,
        "prologue_frac_of_ceiling": round(pro_gbs / ceiling["gbs"], 4) if ceiling and pro_gbs
        else None,
        # The prologue's time follows the SM clock (its data path is the SM's
        # load/store pipe): the same time scaled to the part's maximum clock.
        "prologue_us_at_max_sm_clock": round(pro_ms * 1e3 * mhz / max_mhz, 2)
        if pro_ms and mhz and max_mhz else None,
        "prologue_sm_cycles": round(pro_ms * 1e-3 * mhz * 1e6) if pro_ms and mhz else None,
        "configs": configs,
        "next_rows": {"lora_prologue": lora, "ref_cached_attention": ref_cached,
                      "sol_block_sparse": sol, "wire_formats": wire},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 3),
                "statistic": f"median of {len(e_each)} individually timed steps",
                "mean_ms_per_step": round(e_mean, 3), "max_ms_per_step": round(max(e_each), 3),
                "value_at_mean": round(whole_job_value(flops, e_mean, world), 3),
                "path": f"HostPipeline: {len(pipe.groups)} head groups, copies overlapped with compute"},
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": clk_summary,
        "parity": dict(parity, passed=True),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def rmw_ceiling(g, w, stream, iters=10):
    """torch's own in-place read-modify-write (x *= 1, which changes no bit)
    over the valid Q and K rows the prologue reads and writes: the rate a
    plain streaming kernel reaches on this GPU, in this run."""
    views = []
    for b, s in enumerate(w.segments):
        if s.n_valid_q():
            r0 = g["cu_seqlens_q"][b]
            views += [g["q"][r0:r0 + s.n_valid_q()], g["k"][r0:r0 + s.n_valid_q()]]
    nbytes = sum(2 * t.numel() * t.element_size() for t in views)

    def fn():
        for t in views:
            t.mul_(1.0)
    fn()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(iters):
        fn()
    a1.record(stream)
    torch.cuda.synchronize()
    us = a0.elapsed_time(a1) / iters * 1e3
    return {"us": round(us, 2), "gbs": round(nbytes / us / 1e3, 1), "bytes": nbytes,
            "what": "torch in-place x.mul_(1.0) over the valid rows of Q and K"}


def flush_l2(buf):
    """Overwrite a buffer larger than L2 so that the next kernel reads from HBM."""
    buf.zero_()


def config_gate(O, w, fresh, g, n_sample=24):
    """Fail-closed parity of one step on sampled rows: for each segment, up
    to ``n_sample`` valid query rows (first, last and evenly spaced) over all
    heads against the fp64 oracle (prologue of those rows and of all the
    segment's valid keys, then attention), and every padded output row must
    be exactly 0."""
    errs, refs, diffs, rows_checked = [], [], [], 0
    for b, s in enumerate(w.segments):
        q0, kv0 = g["cu_seqlens_q"][b], g["cu_seqlens_kv"][b]
        nq, nkv = s.n_valid_q(), s.n_valid_kv()
        if nq == 0:
            continue
        rows = np.unique(np.linspace(0, nq - 1, min(n_sample, nq)).astype(np.int64)) + q0
        got = O.widen(g["out"][torch.as_tensor(rows, device=g["out"].device)])
        qh = O.widen(fresh["q"][torch.as_tensor(rows)])
        kh = O.widen(fresh["k"][kv0:kv0 + nkv])
        vh = O.widen(fresh["v"][kv0:kv0 + nkv])
        if w.self_attention:
            pos = fresh["pos_thw"].numpy()
            qh = O.qk_norm_rope(qh, O.widen(fresh["wq"]), pos[rows])
            kh = O.qk_norm_rope(kh, O.widen(fresh["wk"]), pos[kv0:kv0 + nkv])
        ref = O.attention(qh, kh, vh, [0, len(rows)], [0, nkv], None, SCALE)
        errs.append(float(np.abs(got - ref).max()) if np.isfinite(got).all() else float("inf"))
        diffs.append(float(np.sum((got - ref) ** 2)))
        refs.append(float(np.sum(ref ** 2)))
        rows_checked += len(rows)
    pad_ok = True
    for b, s in enumerate(w.segments):
        q0 = g["cu_seqlens_q"][b]
        if s.n_valid_q() < s.q_rows:
            pad = g["out"][q0 + s.n_valid_q():q0 + s.q_rows]
            pad_ok = pad_ok and bool((pad.float() == 0).all())
    err = max(errs)
    rel = math.sqrt(sum(diffs) / max(sum(refs), 1e-300))
    ok = err <= 2e-2 and rel <= 5e-3 and pad_ok
    return ok, {"max_abs": err, "rel_l2": rel, "rows_checked": rows_checked,
                "heads": w.n_heads, "padded_rows_zero": pad_ok, "passed": ok}


def config_sweep(h3, W, O, pk, names, min_timed_s=0.3):
    """Every shape besides the headline one, at one GPU: a fail-closed parity
    gate on the first step's output (fresh inputs), then per-kernel CUDA-event
    times of the prologue and attention with L2 flushed before every step,
    and the SM clocks sampled while they run."""
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")  # 2x L2
    res = {}
    for name in names:
        w = W.workload(name)
        g = W.make_inputs(w, device="cuda", fill="B")
        fresh = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in g.items()}
        run_step(h3, g, w)
        torch.cuda.synchronize()
        ok, gate = config_gate(O, w, fresh, g)
        del fresh
        ok = ok and h3.status_word() == 0
        if not ok:
            raise SystemExit(f"parity gate failed on {name}: {gate}; no number reported")
        for _ in range(3):
            flush_l2(flush)
            run_step(h3, g, w)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        flush_l2(flush)
        run_step(h3, g, w)
        torch.cuda.synchronize()
        steps = int(min(2000, max(10, min_timed_s / max(time.perf_counter() - t0, 1e-6))))
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        with ClockSampler(torch.cuda.current_device()) as clk:
            for i in range(steps):
                flush_l2(flush)
                run_step(h3, g, w, evs[i])
            torch.cuda.synchronize()
        if h3.status_word():
            raise SystemExit(f"device status word nonzero after timing {name}")
        attn_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
        pro_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs])) if w.self_attention else 0.0
        tf = w.attention_flops() / (attn_ms * 1e-3) / 1e12
        entry = {"description": w.description, "steps": steps,
                 "attention_ms": round(attn_ms, 4), "attention_tflops": round(tf, 2),
                 "attention_frac_of_burst": round(tf / pk["bf16"], 4),
                 "attention_frac_of_sustained": round(tf / pk["bf16_sustained"], 4),
                 "attention_flop": w.attention_flops(), "parity": gate,
                 "clocks": clk.summary(), "l2": "flushed (256 MB written) before every step"}
        if w.self_attention:
            gbs = w.prologue_bytes() / (pro_ms * 1e-3) / 1e9
            entry.update({"prologue_us": round(pro_ms * 1e3, 2), "prologue_gbs": round(gbs, 1),
                          "prologue_frac_hbm_measured": round(gbs / pk["hbm"], 4),
                          "prologue_frac_8tbs": round(gbs / 8000.0, 4),
                          "prologue_launches": prologue_launches(w),
                          "prologue_bytes": w.prologue_bytes()})
        res[name] = entry
        del g, evs
        torch.cuda.empty_cache()
    del flush
    return res


def lora_prologue_timing(h3, g, w, stream, pk, iters=10):
    """The LoRA-consumer prologue (base + delta rounded to bf16, then the
    norm + RoPE) against the separate branches it replaces (a bf16 add kernel
    writing the sum, then the plain prologue).  Bytes: base and delta read,
    result written."""
    gen = torch.Generator(device=g["q"].device).manual_seed(77)
    dq = (0.05 * torch.randn(g["q"].shape, generator=gen, device=g["q"].device)).to(torch.bfloat16)
    dk = (0.05 * torch.randn(g["k"].shape, generator=gen, device=g["k"].device)).to(torch.bfloat16)

    def fused():
        for b, s in enumerate(w.segments):
            if s.n_valid_q():
                r0, n = g["cu_seqlens_q"][b], s.n_valid_q()
                h3.qk_norm_rope_lora(g["q"][r0:], dq[r0:], g["k"][r0:], dk[r0:], g["wq"], g["wk"],
                                     g["pos_thw"][r0:], n_rows=n, rot=ROT)

    def separate():
        for b, s in enumerate(w.segments):
            if s.n_valid_q():
                r0, n = g["cu_seqlens_q"][b], s.n_valid_q()
                g["q"][r0:r0 + n].add_(dq[r0:r0 + n])
                g["k"][r0:r0 + n].add_(dk[r0:r0 + n])
                h3.qk_norm_rope(g["q"][r0:], g["k"][r0:], g["wq"], g["wk"], g["pos_thw"][r0:],
                                n_rows=n, rot=ROT)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(iters):
            fn()
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / iters * 1e3

    us = timed(fused)
    sep = timed(separate)
    nbytes = 1.5 * (w.prologue_bytes() - 2 * 2 * w.n_heads * 128) + 2 * 2 * w.n_heads * 128
    del dq, dk
    return {"us": round(us, 2), "gbs": round(nbytes / us / 1e3, 1),
            "frac_hbm_measured": round(nbytes / us / 1e3 / pk["hbm"], 4),
            "bytes": nbytes, "separate_branches_us": round(sep, 2),
            "speedup_vs_separate": round(sep / us, 3)}


def ref_cached_timing(h3, W, stream, pk, iters=5):
    """Attention of a reference-to-video step after the first: 16,422 current
    queries over the cached K/V of 3 reference videos (42,336 rows) plus the
    current K/V (16,422 rows), through h3_attention_groups."""
    inp = W.ref_cached_inputs(device=f"cuda:{torch.cuda.current_device()}")

    def run():
        h3.attention_groups(inp["q"], inp["k"], inp["v"], inp["groups"], inp["k_cache"],
                            inp["v_cache"], SCALE, out=inp["out"])
    run()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(iters):
        run()
    a1.record(stream)
    torch.cuda.synchronize()
    ms = a0.elapsed_time(a1) / iters
    tf = inp["flops"] / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 3), "tflops": round(tf, 1), "frac_of_burst": round(tf / pk["bf16"], 4),
            "queries": 16422, "keys": 16422 + 42336, "flop": inp["flops"]}


def sol_attention_timing(h3, g, w, stream, pk, taus=(1.0, 1.25, 1.5), iters=5):
    """Sol-Attn at each tau of the page's per-step schedule; the first tau's
    figures are the top-level keys, every tau is in ``tau_sweep``."""
    runs = [sol_attention_one(h3, g, w, stream, pk, tau, iters) for tau in taus]
    res = dict(runs[0])
    res["tau_sweep"] = runs
    return res


def sol_attention_one(h3, g, w, stream, pk, tau=1.0, iters=5):
    """Sol-Attn on the 58,758-token sequence read as [text | audio | video]
    (prefix 2,310 rows = 19 sink blocks): block means of Q and K (one
    launch), selection at tau, then sparse attention.  Reports the kept
    fraction of (query block, KV block) pairs, stage times, and TFLOP/s over
    the kept pairs."""
    s = w.segments[0]
    n = s.n_valid_q()
    q, k, v = g["q"], g["k"], g["v"]

    def run(ev=None):
        if ev is not None:
            ev[0].record(stream)
        qm, km = h3.block_means_qk(q, k, n)
        if ev is not None:
            ev[1].record(stream)
        lists, counts = h3.block_select(qm, km, tau, -(-2310 // 128), SCALE)
        if ev is not None:
            ev[2].record(stream)
        h3.sparse_attention(q, k, v, lists, counts, n, SCALE, out=g["out"],
                            n_prefix_blocks=-(-2310 // 128))
        if ev is not None:
            ev[3].record(stream)
        return counts

    counts = run()
    torch.cuda.synchronize()
    # Iterations are queued back to back, so that the host's launch work for
    # one stage overlaps the GPU's previous work; the first iteration (queued
    # on an idle stream, its start event firing before its first launch) is
    # not counted.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(iters + 1)]
    for ev in evs:
        run(ev)
    torch.cuda.synchronize()
    t = np.mean([[ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]), ev[2].elapsed_time(ev[3])]
                 for ev in evs[1:]], axis=0)
    nb = -(-n // 128)
    kept = float(counts.double().sum().item()) / (w.n_heads * nb * nb)
    flops_kept = kept * 4.0 * w.n_heads * 128 * n * n  # the first sequence only
    total_ms = float(t.sum())
    tf = flops_kept / (t[2] * 1e-3) / 1e12
    means_bytes = 2.0 * n * w.n_heads * 128 * 2  # Q and K valid rows read once
    return {"tau": tau, "kept_fraction": round(kept, 4), "means_ms": round(t[0], 4),
            "means_gbs": round(means_bytes / (t[0] * 1e-3) / 1e9, 1),
            "means_frac_hbm_measured": round(means_bytes / (t[0] * 1e-3) / 1e9 / pk["hbm"], 4),
            "select_ms": round(t[1], 4), "attention_ms": round(t[2], 3),
            "total_ms": round(total_ms, 3),
            "tflops_over_kept": round(tf, 1), "frac_of_burst": round(tf / pk["bf16"], 4),
            "speedup_vs_dense_attention": None}


def wire_timing(h3, g, w, stream, pk, iters=5):
    """Bandwidth of the attention-boundary wire kernels on the valid rows:
    packing Q/K/V for 2 destinations (bf16 and block-INT8 records), unpacking
    one destination's share, and packing the output as FP8 records."""
    n = w.segments[0].n_valid_q()
    q, k, v = g["q"][:n], g["k"][:n], g["v"][:n]
    res = {}
    elem = n * w.n_heads * 128

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(iters):
            fn()
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / iters * 1e3

    for name, fmt, rec in (("bf16", h3.WIRE_BF16, 768), ("int8", h3.WIRE_INT8, 400)):
        us = timed(lambda: h3.pack_qkv(q, k, v, 2, fmt))
        nbytes = 3 * elem * 2 + n * w.n_heads * rec
        res[f"pack_qkv_{name}"] = {"us": round(us, 1), "gbs": round(nbytes / us / 1e3, 1),
                                   "frac_hbm_measured": round(nbytes / us / 1e3 / pk["hbm"], 4)}
    wire8 = h3.pack_qkv(q, k, v, 2, h3.WIRE_INT8)
    us = timed(lambda: h3.unpack_qkv(wire8[0], h3.WIRE_INT8))
    nbytes = n * (w.n_heads // 2) * (400 + 3 * 256)
    res["unpack_qkv_int8"] = {"us": round(us, 1), "gbs": round(nbytes / us / 1e3, 1)}
    us = timed(lambda: h3.pack_out(g["out"][:n], h3.WIRE_FP8))
    nbytes = elem * 2 + elem
    res["pack_out_fp8"] = {"us": round(us, 1), "gbs": round(nbytes / us / 1e3, 1)}
    del wire8
    return res


def _code_only(text):
    """Source text without comments, trailing spaces or blank lines, so that a
    comment edit does not count as a kernel change."""
    import re
    text = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    text = re.sub(rb"//[^\n]*", b"", text)
    return b"\n".join(l.rstrip() for l in text.split(b"\n") if l.strip())


def kernel_source_digest():
    """First 16 hex digits of sha256 over the attention kernel's device code,
    comments left out: attention.cu up to its host-side section, then ptx.cuh."""
    import hashlib
    csrc = os.path.join(ROOT, "packed_sequence_attention_gb300", "csrc")
    text = open(os.path.join(csrc, "attention.cu"), "rb").read()
    cut = text.find(b"// ------------------------------------------------------------------ host side")
    device = text if cut < 0 else text[:cut]
    ptx = open(os.path.join(csrc, "ptx.cuh"), "rb").read()
    return hashlib.sha256(_code_only(device) + b"\n" + _code_only(ptx)).hexdigest()[:16]


def committed_traffic(w):
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on this workload and on the current kernel device code."""
    path = os.path.join(ROOT, "profiles", "attention_traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            a, b = line.split(":", 1)
            kv[a.strip()] = b.strip()
    if kv.get("kernel_source_sha256_16") != kernel_source_digest() or kv.get("workload") != w.name:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# -------------------------------------------------------- the reference arm
def workload_config(w, world):
    """The `config` object of the JSON line; both arms report the same one."""
    return {"workload": w.name, "description": w.description,
            "valid_tokens": [s.n_valid_q() for s in w.segments],
            "buffer_rows": [s.q_rows for s in w.segments],
            "heads": w.n_heads, "head_dim": 128,
            "attention_flop_per_step": w.attention_flops(),
            "prologue_bytes_per_step": w.prologue_bytes(),
            "l2": "inputs larger than L2 (Q,K,V 632 MB each); no flush"
            if w.name == "full" else "no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def bench_reference(args):
    """The CPU oracle timed as the reference arm: each step is a bounded
    sample (args.ref_rows query rows x args.ref_heads heads) of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from packed_sequence_attention_gb300 import workloads as W
    from oracle import oracle as O
    w = W.workload(args.config)
    inp = W.make_inputs(w, device="cuda" if torch.cuda.is_available() else "cpu")
    inp = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    for _ in range(args.warmup):
        cpu_baseline(O, inp, w, args.ref_heads, args.ref_rows)
    vals, t0 = [], time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(O, inp, w, args.ref_heads, args.ref_rows))
    dt = time.perf_counter() - t0
    value = float(np.mean([v["value"] for v in vals]))
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": vals[-1]["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="h3", choices=["h3", "reference"])
    ap.add_argument("--config", default="full")
    ap.add_argument("--cpu-heads", type=int, default=42)
    ap.add_argument("--cpu-rows", type=int, default=192)
    ap.add_argument("--ref-heads", type=int, default=2)
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other four shapes (measured by default with the full one)")
    ap.add_argument("--kernels-only", action="store_true",
                    help="profiling mode: warm-up and timed steps only (no e2e, no CPU baseline)")
    ap.add_argument("--wire-only", action="store_true",
                    help="profiling mode: the wire-format kernels on the first sequence only")
    ap.add_argument("--next-only", action="store_true",
                    help="profiling mode: the LoRA-fused prologue and the Sol-Attn stages only")
    args = ap.parse_args()
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
