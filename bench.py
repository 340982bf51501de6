"""Benchmark of the sink-attention hot path on GB300.

Headline (one JSON line on rank 0): the gpt-oss-120b-shaped split-KV decode
(64 sequences, 64 query / 8 KV heads, d 64, q_len 1, kv_len ~ U[1024, 8192])
as KV-read HBM GB/s: algorithmic bytes (Q + visible K + visible V + O + LSE +
sinks + kv_indptr) per step divided by the device time of one step (split
kernel + merge kernel). The same line carries the prefill workloads'
TFLOP/s (algorithmic flops 4 * d * Hq * visible pairs) under "also", the
roofline of the dominant kernel, the float64 oracle timed on the host's cores
("cpu_baseline"), an end-to-end number through the C ABI with host buffers
("e2e"), and the SM clocks sampled during the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Multi-GPU runs go through torchrun; every rank runs its own replica of the
workload (the path needs no exchange), rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

HEADLINE = "gptoss_decode"
ALSO = ["qwen_mtp_decode", "gptoss_prefill", "gptoss_prefill_w128", "qwen_prefill",
        "gptoss_mtp2_decode", "gptoss_mtp4_decode", "qwen_mtp2_decode", "qwen_mtp4_decode",
        "qwen_mtp16_decode", "gptoss_decode_paged", "qwen_mtp_decode_paged", "gptoss_decode_fp8",
        "qwen_mtp_decode_fp8"]
# secondary workloads that get the oracle timed beside them (the other named
# configurations; the headline has its own cpu_baseline)
CPU_ALSO = ("qwen_mtp_decode", "gptoss_prefill", "gptoss_prefill_w128", "qwen_prefill")
ALSO_FIELDS = "value, unit, frac of measured peak, ms/step, oracle on host cores (same unit)"
METRIC = "decode KV-read HBM GB/s and prefill TFLOP/s, each as % of GB300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2**20


# ----------------------------------------------------------------------------
# algorithmic work
# ----------------------------------------------------------------------------
def visible_pairs(q_lens, kv_lens, causal, window):
    """Visible (query, key) pairs per head, in closed form per query row."""
    total = 0
    for lq, lk in zip(q_lens, kv_lens):
        if lq == 0:
            continue
        p = np.arange(lk - lq, lk, dtype=np.int64)          # query positions
        hi = np.minimum(p, lk - 1) if causal else np.full_like(p, lk - 1)
        lo = np.maximum(0, p - window + 1) if window > 0 else np.zeros_like(p)
        total += int(np.maximum(0, hi - lo + 1).sum())
    return total


def work(w, inp):
    """(algorithmic bytes, algorithmic flops) of one pass, and the split kernel's
    input bytes (Q + visible K + V)."""
    Hq, Hkv, d = w.num_qo_heads, w.num_kv_heads, w.head_dim
    pairs = visible_pairs(inp["q_lens"], inp["kv_lens"], w.causal, w.window)
    flops = 4.0 * d * Hq * pairs
    tq = inp["total_q"]
    q_bytes = tq * Hq * d * 2
    if w.window > 0:
        # keys any query of the sequence can see
        kv_tok = sum(min(lk, lq + w.window - 1) for lq, lk in zip(inp["q_lens"], inp["kv_lens"]))
    else:
        kv_tok = sum(inp["kv_lens"])
    kv_bytes = 2 * Hkv * kv_tok * d * (1 if w.kv_fp8 else 2)
    small = Hq * 4 + (inp["batch"] + 1) * 4 * (1 if w.kind == "decode" else 2)
    if w.kv_fp8:          # per-KV-head key and value scales
        small += 2 * Hkv * 4
    if w.page_size > 0:   # page lists
        small += 4 * (inp["batch"] + 1 + sum(-(-lk // w.page_size) for lk in inp["kv_lens"]))
    total = q_bytes + kv_bytes + q_bytes + tq * Hq * 4 + small
    return float(total), float(flops), float(q_bytes + kv_bytes)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"]))}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text):
    """C++/CUDA source without comments or blank lines: a comment edit does
    not change the kernel the counters were taken on."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gqa_attention_softmax_gb300", "csrc", n)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(key, sources):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources are unchanged since the capture; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(key)
    if not e or e.get("source_sha") != kernel_source_sha(sources):
        return None
    return float(e["dram_bytes_per_launch"])


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        loaded = [s for s, r in zip(sm, rows) if r[3].strip() and float(r[3] or 0) > 0]
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------
def time_workload(name, steps, warmup, dist_ctx=None, want_kernel_split=False, batch=None):
    """Device time of `steps` passes (events on the launching stream) after
    `warmup` untimed passes. Returns (ms_per_step, split_ms_per_launch or None,
    inputs, runner). `batch` overrides a decode workload's batch (profiling)."""
    from gqa_attention_softmax_gb300 import runner, workloads, _binding as B
    w = workloads.WORKLOADS[name]
    rank = int(os.environ.get("RANK", "0"))
    inp = workloads.make_inputs(w, device="cuda", seed=runner.rank_seed(w.seed, rank), batch=batch)
    run = runner.Runner(w, inp)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        run()
    split_ms = None
    # the step: `steps` calls back to back (for decode the merge is launched
    # as a programmatic dependent of the partial kernel, so nothing may sit
    # between them on the stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _sync(dist_ctx)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    _sync(dist_ctx)
    ms = e0.elapsed_time(e1) / steps
    if w.kind == "decode" and want_kernel_split and not run.fused and not single_pass_decode(w):
        # the dominant kernel's own time: the same partial launches back to
        # back, bracketed by events on the launching stream
        n_acc = inp["total_q"] * w.num_qo_heads * run.num_splits * w.head_dim * 4
        off = (n_acc + 255) // 256 * 256
        acc = run.workspace[:n_acc].view(torch.float32).view(inp["total_q"], w.num_qo_heads,
                                                            run.num_splits, w.head_dim)
        md = run.workspace[off: off + inp["total_q"] * w.num_qo_heads * run.num_splits * 8].view(
            torch.float32).view(inp["total_q"], w.num_qo_heads, run.num_splits, 2)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _sync(dist_ctx)
        s0.record(stream)
        for _ in range(steps):
            if w.kv_fp8:
                B.sinkattn_decode_split_fp8(inp["q"], inp["k_fp8"], inp["v_fp8"], inp["k_scale"],
                                            inp["v_scale"], inp["cu_k"], w.q_len, inp["max_k"],
                                            run.num_splits, w.scale, w.causal, w.window,
                                            part_acc=acc, part_md=md)
            elif w.page_size > 0:
                B.sinkattn_decode_split_paged(inp["q"], inp["k_pages"], inp["v_pages"], inp["cu_k"],
                                              inp["page_indptr"], inp["page_indices"], w.q_len,
                                              inp["max_k"], run.num_splits, w.scale, w.causal,
                                              w.window, part_acc=acc, part_md=md)
            else:
                B.sinkattn_decode_split(inp["q"], inp["k"], inp["v"], inp["cu_k"], w.q_len,
                                        inp["max_k"], w.num_kv_heads, run.num_splits, w.scale,
                                        w.causal, w.window, part_acc=acc, part_md=md)
        s1.record(stream)
        _sync(dist_ctx)
        split_ms = s0.elapsed_time(s1) / steps
    elif w.kind == "decode":
        split_ms = ms   # one launch (cluster-fused, or single pass) is the whole step
    ms = _max_over_ranks(ms, dist_ctx)
    if split_ms is not None:
        split_ms = _max_over_ranks(split_ms, dist_ctx)
    return ms, split_ms, w, inp, run


def time_flushed(run, steps, dist_ctx=None, flush_bytes=256 * 2**20):
    """Device time of one pass with L2 flushed before it: a `flush_bytes`
    write between passes, outside the events. Returns ms per pass (median)."""
    stream = torch.cuda.current_stream()
    buf = torch.empty(flush_bytes, dtype=torch.uint8, device="cuda")
    times = []
    _sync(dist_ctx)
    for _ in range(steps):
        buf.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    _sync(dist_ctx)
    del buf
    return _max_over_ranks(statistics.median(times), dist_ctx)


def _sync(ctx):
    torch.cuda.synchronize()
    if ctx is not None:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


def _max_over_ranks(x, ctx):
    from gqa_attention_softmax_gb300 import runner
    return runner.max_over_ranks(x)


def runner_call(run, inp):
    """One pass of the runner's workload on the given (device) inputs."""
    saved = run.inp
    run.inp = inp
    try:
        return run()
    finally:
        run.inp = saved


def e2e_decode(w, inp, run, steps):
    """Same metric through the C ABI with host buffers: H2D of the step's
    inputs from pinned memory, the decode, D2H of out + lse, all timed."""
    from gqa_attention_softmax_gb300 import _binding as B
    host = {k: inp[k].cpu().pin_memory() for k in ("q", "k", "v", "cu_k", "sinks")}
    dev = {k: torch.empty_like(inp[k]) for k in host}
    out_h = torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory()
    lse_h = torch.empty(run.lse.shape, dtype=run.lse.dtype).pin_memory()
    stream = torch.cuda.current_stream()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

    run_dev = dict(inp)
    run_dev.update(dev)

    def step():
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        runner_call(run, run_dev)
        out_h.copy_(run.out, non_blocking=True)
        lse_h.copy_(run.lse, non_blocking=True)

    step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


# ----------------------------------------------------------------------------
# the float64 oracle on the host (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------
def oracle_sample(w, inp, target_s):
    """Time the oracle on a bounded sample of the workload: whole sequences
    (decode) or random query rows of every sequence (prefill), grown until the
    work takes about `target_s`. Returns (GB/s or GFLOP/s, unit, cores, sample text)."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    Hq, Hkv, d = w.num_qo_heads, w.num_kv_heads, w.head_dim
    cu_q = inp["cu_q"].cpu().tolist()
    cu_k = inp["cu_k"].cpu().tolist()
    B = len(cu_q) - 1
    rng = np.random.default_rng(0)
    if w.kind == "decode":
        # whole sequences, all heads and rows; grow the sample, then repeat
        # passes over it until about target_s seconds of work
        n = 1
        while True:
            seqs = list(range(min(n, B)))
            sub = _sub(inp, Hkv, seqs, cu_q, cu_k)
            t0 = time.perf_counter()
            oracle.attend(sub["q"], sub["k"], sub["v"], sub["sinks"], sub["cu_q"], sub["cu_k"], Hq,
                          Hkv, d, w.scale, w.causal, w.window)
            dt = time.perf_counter() - t0
            if dt >= target_s or n >= B:
                break
            n = min(B, max(n + 1, int(n * min(8.0, 1.5 * target_s / max(dt, 1e-3)))))
        passes, total = 1, dt
        while total < target_s and passes < 1000:
            t0 = time.perf_counter()
            oracle.attend(sub["q"], sub["k"], sub["v"], sub["sinks"], sub["cu_q"], sub["cu_k"], Hq,
                          Hkv, d, w.scale, w.causal, w.window)
            total += time.perf_counter() - t0
            passes += 1
        wl = {"q_lens": [cu_q[b + 1] - cu_q[b] for b in seqs], "kv_lens": [cu_k[b + 1] - cu_k[b] for b in seqs],
              "total_q": sum(cu_q[b + 1] - cu_q[b] for b in seqs), "batch": len(seqs)}
        nbytes, _, _ = work(w, wl)
        return (passes * nbytes / total / 1e9, "GB/s", oracle.num_threads(),
                "%d passes over %d of %d seqs, all rows, %.1f s" % (passes, len(seqs), B, total))
    # prefill: random rows, flops counted per row
    n = 64
    while True:
        toks = rng.integers(0, cu_q[-1], size=n)
        heads = rng.integers(0, Hq, size=n)
        rows = toks * Hq + heads
        t0 = time.perf_counter()
        oracle.attend(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["cu_q"], inp["cu_k"], Hq, Hkv,
                      d, w.scale, w.causal, w.window, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= 1 << 20:
            break
        n = int(n * min(8.0, 1.5 * target_s / max(dt, 1e-3)))
    pairs = 0
    for t in toks:
        b = int(np.searchsorted(cu_q, t, side="right") - 1)
        lq, lk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        p = lk - lq + (t - cu_q[b])
        hi = p if w.causal else lk - 1
        lo = max(0, p - w.window + 1) if w.window > 0 else 0
        pairs += max(0, hi - lo + 1)
    return 4.0 * d * pairs / dt / 1e12, "TFLOP/s", oracle.num_threads(), "%d random rows, %.1f s" % (n, dt)


def _sub(inp, Hkv, seqs, cu_q, cu_k):
    qs, ks, vs = [], [], []
    ncq, nck = [0], [0]
    for b in seqs:
        qs.append(inp["q"][cu_q[b]:cu_q[b + 1]].cpu())
        ks.append(inp["k"][Hkv * cu_k[b]:Hkv * cu_k[b + 1]].cpu())
        vs.append(inp["v"][Hkv * cu_k[b]:Hkv * cu_k[b + 1]].cpu())
        ncq.append(ncq[-1] + cu_q[b + 1] - cu_q[b])
        nck.append(nck[-1] + cu_k[b + 1] - cu_k[b])
    return dict(q=torch.cat(qs), k=torch.cat(ks), v=torch.cat(vs), sinks=inp["sinks"].cpu(),
                cu_q=torch.tensor(ncq, dtype=torch.int32), cu_k=torch.tensor(nck, dtype=torch.int32))


def reference_arm(args, rank, world):
    """The oracle, as it stands, on the host's cores: each step is a bounded
    sample of the headline workload (whole sequences, all heads)."""
    from gqa_attention_softmax_gb300 import workloads
    if rank != 0:
        return
    w = workloads.WORKLOADS[HEADLINE]
    inp = workloads.make_inputs(w, device="cpu")
    import oracle
    oracle.build()
    cu_q = inp["cu_q"].tolist()
    cu_k = inp["cu_k"].tolist()
    # one sequence per step: bounded, ~tens of ms each
    seq_times, nbytes_all = [], 0.0
    total_steps = args.warmup + args.steps
    budget = 150.0
    t_start = time.perf_counter()
    done = 0
    for i in range(total_steps):
        b = i % inp["batch"]
        sub = _sub(inp, w.num_kv_heads, [b], cu_q, cu_k)
        t0 = time.perf_counter()
        oracle.attend(sub["q"], sub["k"], sub["v"], sub["sinks"], sub["cu_q"], sub["cu_k"],
                      w.num_qo_heads, w.num_kv_heads, w.head_dim, w.scale, w.causal, w.window)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            wl = {"q_lens": [1], "kv_lens": [cu_k[b + 1] - cu_k[b]], "total_q": 1, "batch": 1}
            nbytes_all += work(w, wl)[0]
            seq_times.append(dt)
            done += 1
        if time.perf_counter() - t_start > budget and done >= 1:
            break
    tsum = sum(seq_times)
    value = nbytes_all / tsum / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": done, "warmup": args.warmup, "ms_per_step": 1e3 * tsum / max(done, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": _workload_desc(w), "sample_per_step": "one whole sequence (all 64 heads)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": "%d steps of one sequence each (cycling through the batch)" % done},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def single_pass_decode(w):
    """True when the library's default runs this decode as one single-pass
    launch: more query rows per KV head (G x q_len) than one 128-row tile."""
    return not w.kv_fp8 and (w.num_qo_heads // w.num_kv_heads) * w.q_len > 128


def decode_kernel_name(w):
    """The kernel the library's default selection runs for this shape."""
    if single_pass_decode(w):
        return "prefill_tc_kernel (tcgen05, single pass: the drafts are its queries)"
    if w.kv_fp8:
        g = w.num_qo_heads // w.num_kv_heads
        if w.head_dim == 128 and g <= 64:
            return "decode_tc_kernel (tcgen05 f16, e4m3 codes widened in shared memory)"
        return "attn_mma_kernel (mma.sync f16, e4m3 codes widened in shared memory)"
    return "decode_tc_kernel (tcgen05)" if w.head_dim == 128 else "attn_mma_kernel (mma.sync)"


def decode_traffic(w):
    """ncu DRAM bytes per launch of the split kernel for this decode workload,
    from the committed summaries (None if absent or the sources changed)."""
    if single_pass_decode(w):
        return ncu_traffic("prefill_tc_kernel/" + w.name, ["prefill_tc.cu", "common.cuh", "tc.cuh"])
    if "decode_tc" in decode_kernel_name(w):
        return ncu_traffic("decode_tc_kernel/" + w.name, ["decode_tc.cu", "common.cuh", "tc.cuh"])
    return ncu_traffic("attn_mma_kernel/" + w.name, ["attn_mma.cu", "common.cuh"])


def _workload_desc(w):
    if w.kind == "decode":
        layout = ("paged HND bf16, %d-key pages in random order" % w.page_size if w.page_size > 0
                  else "HND FP8 e4m3 with per-KV-head scales" if w.kv_fp8 else "HND bf16")
        return ("%s: batch %d, %d query / %d KV heads, head_dim %d, q_len %d, kv_len ~ U[%d, %d], "
                "%s, fp32 sinks" % (w.name, w.batch, w.num_qo_heads, w.num_kv_heads,
                                    w.head_dim, w.q_len, w.kv_range[0], w.kv_range[1], layout))
    return ("%s: seqlens %s, %d query / %d KV heads, head_dim %d, causal, window %d, bf16" % (
        w.name, list(w.kv_lens), w.num_qo_heads, w.num_kv_heads, w.head_dim, w.window))


# ----------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-also", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--profile", metavar="WORKLOAD", default=None,
                    help="profiling mode: time only this workload (no extras), for ncu")
    ap.add_argument("--batch", type=int, default=None, help="decode batch override (profiling)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist_ctx = None
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
        dist_ctx = True
    else:
        torch.cuda.set_device(0)
    args.warmup = max(3, args.warmup)

    import __graft_entry__
    __graft_entry__.build()
    from gqa_attention_softmax_gb300 import workloads
    peaks, peak_src = load_peaks()

    if args.profile:
        ms, split_ms, w, inp, run = time_workload(args.profile, args.steps, args.warmup, dist_ctx,
                                                  want_kernel_split=True, batch=args.batch)
        nb, fl, sb = work(w, inp)
        if rank == 0:
            print(json.dumps({"profile": args.profile, "batch": inp["batch"], "ms_per_step": ms,
                              "split_ms": split_ms, "bytes": nb, "flops": fl,
                              "GB/s": nb / (ms * 1e-3) / 1e9, "TFLOP/s": fl / (ms * 1e-3) / 1e12}),
                  flush=True)
        return

    sampler = ClockSampler(local_rank)
    with sampler:
        ms, split_ms, w, inp, run = time_workload(HEADLINE, args.steps, args.warmup, dist_ctx,
                                                  want_kernel_split=True)
    clocks = sampler.summary()
    nbytes, flops, split_bytes = work(w, inp)
    value = world * nbytes / (ms * 1e-3) / 1e9
    if run.fused:
        # one launch does split and merge: its algorithmic bytes are the step's
        split_bytes = nbytes
        kernel_name = "attn_mma_kernel, cluster-fused split-KV decode (%d chunks per cluster)" % run.num_splits
    else:
        kernel_name = decode_kernel_name(w).split(" ")[0]
    split_gbs = split_bytes / (split_ms * 1e-3) / 1e9
    traffic = ncu_traffic(("attn_mma_kernel_fused/" if run.fused else "attn_mma_kernel/") + HEADLINE,
                          ["attn_mma.cu", "common.cuh"])

    flushed_ms = time_flushed(run, max(3, min(args.steps, 50)), dist_ctx)

    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_decode(w, inp, run, steps=min(args.steps, 20))
        e2e = {"value": _r(world * nbytes / (e2e_ms * 1e-3) / 1e9), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    also, detail = {}, {}
    if not args.no_also:
        for name in ALSO:
            wa = workloads.WORKLOADS[name]
            steps = max(3, min(args.steps, 200))
            ms_a, split_a, wa, inp_a, _ = time_workload(name, steps, args.warmup, dist_ctx,
                                                        want_kernel_split=(wa.kind == "decode"))
            nb, fl, sb = work(wa, inp_a)
            cpu_a = None
            if rank == 0 and not args.no_cpu and name in CPU_ALSO:
                inp_c = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp_a.items()}
                cpu_a = oracle_sample(wa, inp_c, target_s=4.0)[0]
                del inp_c
            gbs = nb / (ms_a * 1e-3) / 1e9
            if wa.kind == "decode":
                also[name] = [_r(gbs), "GB/s", _r(gbs / peaks["hbm_gbs"], 3), _r(ms_a, 3), _r(cpu_a, 3)]
                detail[name] = {"workload": _workload_desc(wa), "num_splits": splits_of(wa, inp_a),
                                "kernel": decode_kernel_name(wa) + (
                                    "" if single_pass_decode(wa) else " + merge_kernel"),
                                "split_kernel_ms": _r(split_a),
                                "traffic": decode_traffic(wa), "tflops": _r(fl / (ms_a * 1e-3) / 1e12)}
            else:
                tf = fl / (ms_a * 1e-3) / 1e12
                also[name] = [_r(tf), "TFLOP/s", _r(tf / peaks["bf16_tflops"], 3), _r(ms_a, 3),
                              _r(cpu_a, 3)]
                if wa.window > 0:   # the HBM roofline binds (arithmetic intensity below the ridge)
                    also[name + "_hbm"] = [_r(gbs), "GB/s", _r(gbs / peaks["hbm_gbs"], 3),
                                           _r(ms_a, 3), None]
                detail[name] = {"workload": _workload_desc(wa),
                                "kernel": "prefill_tc_kernel or prefill_tc_persistent_kernel "
                                          "(tcgen05; the library's launch choice)",
                                "traffic": ncu_traffic("prefill_tc_kernel/" + name,
                                                       ["prefill_tc.cu", "common.cuh", "tc.cuh"])}
            del inp_a
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu:
        inp_cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
        v_cpu, unit, cores, sample = oracle_sample(w, inp_cpu, target_s=10.0)
        cpu = {"value": _r(v_cpu), "unit": unit, "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        if detail:
            # kernel names, splits and ncu traffic of the secondary workloads
            # (stderr: stdout carries the one JSON result line)
            print(json.dumps({"detail": detail}), file=sys.stderr, flush=True)
        line = {
            "metric": METRIC, "value": _r(value), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": _r(ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": _workload_desc(w), "num_splits": run.num_splits,
                       "l2": "inputs > L2 (%.0f MB K/V per step); l2_flushed: 256 MB written "
                             "before each pass" % (split_bytes / 1e6),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": kernel_name,
                         "achieved": _r(split_gbs), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": _r(split_gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                         "bytes_per_launch": split_bytes, "peak_source": peak_src},
            "l2_flushed": {"value": _r(world * nbytes / (flushed_ms * 1e-3) / 1e9),
                           "ms_per_step": _r(flushed_ms)},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": run.launches_per_call * args.steps,
            "clocks": clocks,
            "also_fields": ALSO_FIELDS,
            "also": also,
        }
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if dist_ctx is not None:
        import torch.distributed as dist
        dist.destroy_process_group()


def _r(x, digits=4):
    """x to `digits` significant digits (None stays None): keeps the JSON line short."""
    if x is None:
        return None
    return float("%.*g" % (digits, x))


def splits_of(w, inp):
    from gqa_attention_softmax_gb300 import runner
    return runner.splits_for(w, inp)


if __name__ == "__main__":
    main()
