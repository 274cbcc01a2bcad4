#!/usr/bin/env python
"""Benchmark of layer-major batched int8 prefill on GB300.

One step = one prefill of the whole prompt through every layer (all kernels
of the path) with weights resident in HBM, last-position logits produced.
Default workload: Llama-3-8B-shaped int8 decoder, 4096-token prompt, chunks
of 512 (synthetic, seeded weights and tokens). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 8b|...]

Multi-GPU (torchrun, N > 1): independent replicas, one prompt per rank, no
collective on the data path ("scaling": "weak").
`--impl reference` times the CPU oracle (test infrastructure, plain C) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill tok/s (int8 8B-shape, 4096-tok prompt); % of int8-TC/HBM roofline"
NORTH_HBM_GBS = 8000.0  # the 8 TB/s of the roofline definition
FP32_LANES = 128  # FP32 FMA lanes per SM


def sm_count() -> int:
    """SMs of the current CUDA device (152 on a GB300)."""
    import torch

    return int(torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count)

# DRAM bytes (read + write) per launch of a kernel class at the 8B / chunk 512
# workload, from one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum),
# valid only while the kernel's source file hashes to the value recorded with
# it. profiles/ holds the capture summaries and commands.
KERNEL_TRAFFIC = {
    # k_attention, mean over the 8 launches of one layer (chunk starts 0, 512, ..., 3584); the range merge
    # kernel's own bytes are listed in its profile summary
    "attention": {"bytes_per_launch": 33144704.0, "source": "prompt_prefill_gb300/csrc/k_attention.cu",
                  "sha256": "3126986e9cac0e39cadbd1c23e1552acda354fd2ad8b3df0a9b5b4c944e9d375"},
}


def kernel_traffic(kernel: str, workload: str):
    """Captured DRAM bytes per launch, or None when none was captured for this
    kernel and workload or its source has changed since."""
    import hashlib

    t = KERNEL_TRAFFIC.get(kernel)
    if t is None or workload != "8b":
        return None
    with open(os.path.join(ROOT, t["source"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != t["sha256"]:
            return None
    return t["bytes_per_launch"]


# ----------------------------------------------------------------------------- accounting
def layer_weight_bytes(c) -> int:
    """int8 weights + f32 row scales of one layer (what its GEMMs read)."""
    return c.layer_bytes() + 4 * (c.qkv_rows + c.dim + 2 * c.ffn + c.dim)


def weight_bytes_read(c, prompt: int, chunk: int) -> int:
    """Layer weights once per chunk plus the output projection once per call
    ("Batched Prefill", "The arithmetic": the per-token path reads the model
    once per token; chunking reads it once per chunk)."""
    n_chunks = -(-prompt // chunk)
    return layer_weight_bytes(c) * c.n_layers * n_chunks + c.vocab * c.dim + 4 * c.vocab


def macs_per_weight_byte(prompt: int, chunk: int) -> float:
    """Work per weight byte fetched ("Batched Prefill", "The Solution" table): 1 for GEMV, chunk for GEMM."""
    return prompt / -(-prompt // chunk)


def tok_per_s(prompt: int, seconds: float) -> float:
    return prompt / seconds


def algorithmic_work(c, prompt: int, chunk: int) -> dict:
    """Algorithmic work of one step, per kernel class (flops or bytes)."""
    D, H, Hkv, hd, F, V, L = c.dim, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn, c.vocab, c.n_layers
    QD, QKV = H * hd, (H + 2 * Hkv) * hd
    gemm_flops = 2 * prompt * c.layer_bytes() * L
    pairs = prompt * (prompt + 1) // 2  # causal (query, key) pairs at start_pos 0
    attn_flops = 4 * hd * H * pairs * L  # q.k and p.v, 2 flops per multiply-add each
    # HBM bytes each row kernel must move per token and layer (f32 in, int8 out, plus the row scale)
    nq_bytes = L * prompt * ((4 + 1) * (2 * D + QD + F) + 4 * 4) + (4 + 1) * D
    rope_bytes = L * prompt * (4 * QKV + 4 * QD + 4 * 2 * Hkv * hd)
    lm_head_bytes = V * D + 4 * V + 4 * V
    embed_bytes = 2 * 4 * prompt * D
    # attention must read each K/V row of its head group once per chunk and write o
    n_chunks = -(-prompt // chunk)
    kv_reads = sum(min(prompt, (i + 1) * chunk) for i in range(n_chunks))
    attn_bytes = L * (kv_reads * 2 * Hkv * hd * 4 + prompt * 2 * QD * 4)
    return {
        "gemm": {"bound": "tensor", "work": gemm_flops, "unit": "TFLOP/s"},
        "attention": {"bound": "alu", "work": attn_flops, "unit": "TFLOP/s", "bytes": attn_bytes},
        "norm_quant": {"bound": "hbm", "work": nq_bytes, "unit": "GB/s"},
        "rope_kv": {"bound": "hbm", "work": rope_bytes, "unit": "GB/s"},
        "lm_head": {"bound": "hbm", "work": lm_head_bytes, "unit": "GB/s"},
        "embed": {"bound": "hbm", "work": embed_bytes, "unit": "GB/s"},
    }


def step_bytes(c, prompt: int, chunk: int) -> int:
    """HBM bytes of one step for the prefill roofline: weights once per chunk,
    the K/V cache written once and read once per chunk, embeddings, activations."""
    w = algorithmic_work(c, prompt, chunk)
    return weight_bytes_read(c, prompt, chunk) + w["attention"]["bytes"] + w["norm_quant"]["work"] + \
        w["rope_kv"]["work"] + w["embed"]["work"]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


def peak_for(bound: str, peaks: dict, sms: int | None = None) -> tuple[float, str]:
    if bound == "tensor":
        # the exact-integer GEMMs run at f16 operand rate; bf16 and f16 dense rates are equal
        return float(peaks["bf16_tflops_sustained"]), f"bf16/f16 dense sustained ({peaks['source']})"
    if bound == "alu":
        clk = float(peaks.get("sm_max_mhz", 2070.0))
        sms = sms or sm_count()
        return sms * FP32_LANES * 2 * clk * 1e6 / 1e12, f"FP32 FMA: {sms} SMs x {FP32_LANES} lanes x 2 x {clk:.0f} MHz"
    return float(peaks["hbm_gbs"]), f"HBM copy ({peaks['source']})"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.device)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float) -> float:
    if pg is None:
        return value
    import torch

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def replica_tok_per_s(world: int, tokens_per_rank: int, steps: int, seconds_max: float) -> float:
    """Whole-job throughput of N replicas: every rank prefills its own
    `tokens_per_rank`-token prompt `steps` times; the job takes as long as the
    slowest rank (`seconds_max`, the max over ranks)."""
    return world * tokens_per_rank * steps / seconds_max


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(model, cfg, sample_tokens: int, toks) -> tuple[float, int, float]:
    """Time the oracle (as it stands) prefilling the first `sample_tokens`
    tokens of the prompt in one chunk, one thread per host core."""
    import oracle

    cores = os.cpu_count() or 1
    om = oracle.OracleModel(model, max_seq=sample_tokens, n_threads=cores)
    t0 = time.perf_counter()
    om.prefill(toks[:sample_tokens], 0, sample_tokens)
    dt = time.perf_counter() - t0
    om.close()
    return sample_tokens / dt, cores, dt


def run_reference(args, cfg, world, rank, pg):
    """--impl reference: the oracle on the host cores, bounded sample per step."""
    if rank != 0:
        return 0
    import synth

    model = synth.make_model(cfg)
    toks = synth.prompt(cfg, cfg.prompt_len)
    sample = args.ref_sample_tokens
    for _ in range(args.warmup):
        oracle_sample(model, cfg, sample, toks)
    times = []
    cores = os.cpu_count() or 1
    for _ in range(args.steps):
        _, cores, dt = oracle_sample(model, cfg, sample, toks)
        times.append(dt)
    total = sum(times)
    value = sample * args.steps / total
    desc = (f"oracle prefill of the first {sample} tokens of the {cfg.prompt_len}-token prompt, one chunk, "
            f"{cores} threads, per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic", "config": workload_config(cfg, args),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg, args) -> dict:
    names = {"8b": "Llama-3-8B-shaped int8 decoder, weights resident in HBM",
             "350m": "350M-class int8 decoder", "1b": "1B-class int8 decoder", "tiny": "tiny int8 decoder"}
    return {"workload": f"{names.get(cfg.name, cfg.name)}: {cfg.prompt_len}-token prompt, chunk {args.chunk}, "
                        f"start_pos 0, last-position logits",
            "dim": cfg.dim, "layers": cfg.n_layers, "heads": cfg.n_heads, "kv_heads": cfg.n_kv_heads,
            "head_dim": cfg.head_dim, "ffn": cfg.ffn, "vocab": cfg.vocab, "prompt_tokens": cfg.prompt_len,
            "chunk": args.chunk, "weights": "resident",
            "l2": "inputs larger than L2 (every step reads all layer weights, %.2f GB int8)" % (
                cfg.layer_bytes() * cfg.n_layers / 1e9),
            "parallelism": "replicas" if int(os.environ.get("WORLD_SIZE", "1")) > 1 else "single GPU"}


# ----------------------------------------------------------------------------- our arm
def time_calls(stream, fn, steps: int, warmup: int) -> float:
    """Milliseconds per call of fn() (enqueued on `stream`), CUDA events on that stream."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_calls_each(stream, fn, calls: int) -> list:
    """Milliseconds of each of `calls` calls of fn() (CUDA events around every call on `stream`)."""
    import torch

    out = []
    for _ in range(calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def profile_classes(g, step, steps_dominant: int = 1):
    """Per kernel class: summed launch time of one step with every launch of the class bracketed by CUDA
    events on its stream (chunks in serial order, so no other kernel runs inside a bracket). The
    dominant class is then profiled over `steps_dominant` further steps. Returns ({class: ms per step},
    {class: launches per step}, dominant)."""
    import prompt_prefill_gb300 as pp

    class_ms, class_launches = {}, {}
    for cls, name in pp.KERNEL_NAMES.items():
        g.set_profile_kernel(cls)
        g.reset_stats()
        step()
        s = g.stats()
        class_ms[name] = s["prof_ms"]
        class_launches[name] = s["prof_launches"]
    dominant = max(class_ms, key=class_ms.get)
    if steps_dominant > 1:
        g.set_profile_kernel({v: k for k, v in pp.KERNEL_NAMES.items()}[dominant])
        g.reset_stats()
        for _ in range(steps_dominant):
            step()
        s = g.stats()
        class_ms[dominant] = s["prof_ms"] / steps_dominant
        class_launches[dominant] = s["prof_launches"] // steps_dominant
    g.set_profile_kernel(pp.PP_KERNEL_NONE)
    g.reset_stats()
    return class_ms, class_launches, dominant


def prefill_roofline_ms(cfg, P, chunk, peaks, start_pos: int = 0) -> dict:
    """max(int8 GEMM ops / tensor peak, bytes / 8 TB/s) for one call of P tokens."""
    gemm_ops = 2 * P * cfg.layer_bytes() * cfg.n_layers
    n_chunks = -(-P // chunk)
    kv_row = 2 * cfg.n_kv_heads * cfg.head_dim * 4
    kv_reads = sum(start_pos + min(P, (i + 1) * chunk) for i in range(n_chunks))
    bytes_ = weight_bytes_read(cfg, P, chunk) + cfg.n_layers * kv_reads * kv_row
    t_tc = gemm_ops / (peak_for("tensor", peaks)[0] * 1e12)
    t_hbm = bytes_ / (NORTH_HBM_GBS * 1e9)
    return {"t_roof_ms": 1000 * max(t_tc, t_hbm), "bound": "tensor" if t_tc >= t_hbm else "hbm",
            "gemm_tops": gemm_ops / 1e12, "bytes_gb": bytes_ / 1e9}


def run_small_configs(args, peaks) -> dict:
    """The 350M-class (747 tokens, chunk 32) and 1B-class (2048 tokens, chunks 32..2048, then a call at
    start_pos 2048 continuing the K/V cache) workloads: tok/s, prefill roofline fraction, and for
    350M how much of a call the host spends enqueueing launches against the kernels' summed time."""
    import time as _time

    import torch

    import prompt_prefill_gb300 as pp
    import synth

    stream = torch.cuda.current_stream()
    steps, warm = max(3, min(args.steps, 10)), 3
    out = {}
    # ---- 350M: 747 tokens in chunks of 32
    cfg = synth.CONFIGS["350m"]
    model = synth.make_model(cfg)
    P, chunk = cfg.prompt_len, cfg.chunk
    g = pp.PrefillModel(cfg, model, max_seq=cfg.max_seq, max_chunk=chunk, gemm_engine=args.engine)
    d_tok = torch.from_numpy(synth.prompt(cfg)).cuda()
    d_logits = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
    step = lambda: g.prefill_device(d_tok, P, 0, chunk, d_logits, stream)  # noqa: E731
    res = {}
    for graphs in (0, 1):
        g.set_graphs(bool(graphs))
        for overlap in (0, 1):
            g.set_chunk_overlap(bool(overlap))
            ms = time_calls(stream, step, steps, warm)
            res[("overlap" if overlap else "serial") + ("_graph" if graphs else "")] = {
                "ms": ms, "tok_per_s": P / (ms / 1000)}
    g.set_graphs(False)
    g.set_chunk_overlap(False)
    # host enqueue time of one call (the library's launches, no device wait) against the GPU time
    torch.cuda.synchronize()
    t0 = _time.perf_counter()
    step()
    host_ms = 1000 * (_time.perf_counter() - t0)
    torch.cuda.synchronize()
    g.reset_stats()
    step()
    launches = g.stats()["kernel_launches"]
    class_ms, _, _ = profile_classes(g, step)
    kernel_ms = sum(class_ms.values())
    roof = prefill_roofline_ms(cfg, P, chunk, peaks)
    best = min(v["ms"] for v in res.values())
    out["350m"] = {
        "workload": f"350M-class int8 decoder (D{cfg.dim}, L{cfg.n_layers}, {cfg.n_heads}/{cfg.n_kv_heads} heads, "
                    f"F{cfg.ffn}, V{cfg.vocab}): {P}-token prompt, chunk {chunk}",
        "calls": res, "roofline": roof, "frac_of_roofline": roof["t_roof_ms"] / best,
        "launches_per_call": launches, "host_enqueue_ms_per_call": host_ms,
        "kernel_ms_per_call_serial_profiled": kernel_ms, "kernel_ms_by_class": class_ms,
        # launch by launch vs the same call replayed from a CUDA graph: the host's share of a call
        "graph_speedup_serial": res["serial"]["ms"] / res["serial_graph"]["ms"],
        "graph_speedup_overlap": res["overlap"]["ms"] / res["overlap_graph"]["ms"]}
    g.close()
    del model
    # ---- 1B: chunk sweep, then a continuation call at start_pos 2048
    cfg = synth.CONFIGS["1b"]
    model = synth.make_model(cfg)
    P = cfg.prompt_len
    toks = synth.prompt(cfg, 2 * P)
    g = pp.PrefillModel(cfg, model, max_seq=2 * P, max_chunk=2048, gemm_engine=args.engine)
    g.set_chunk_overlap(True)
    g.set_graphs(bool(args.graphs))
    d_tok = torch.from_numpy(toks).cuda()
    d_logits = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
    sweep = {}
    for chunk in cfg.extra["chunks"]:
        ms = time_calls(stream, lambda: g.prefill_device(d_tok, P, 0, chunk, d_logits, stream), steps, warm)
        roof = prefill_roofline_ms(cfg, P, chunk, peaks)
        sweep[str(chunk)] = {"ms": ms, "tok_per_s": P / (ms / 1000), "frac_of_roofline": roof["t_roof_ms"] / ms,
                             "roofline": roof, "weight_bytes_read": weight_bytes_read(cfg, P, chunk)}
    # continuation: positions 2048..4095 after the first call wrote 0..2047
    chunk = 512
    g.prefill_device(d_tok, P, 0, chunk, d_logits, stream)
    ms = time_calls(stream, lambda: g.prefill_device(d_tok[P:], P, P, chunk, d_logits, stream), steps, warm)
    roof = prefill_roofline_ms(cfg, P, chunk, peaks, start_pos=P)
    g.close()
    out["1b"] = {"workload": f"1B-class int8 decoder (D{cfg.dim}, L{cfg.n_layers}, {cfg.n_heads}/{cfg.n_kv_heads} "
                             f"heads, F{cfg.ffn}, V{cfg.vocab}): {P}-token prompt, chunk sweep, chunk overlap on",
                 "chunk_sweep": sweep,
                 "continuation_start_pos_2048_chunk_512": {"ms": ms, "tok_per_s": P / (ms / 1000),
                                                           "frac_of_roofline": roof["t_roof_ms"] / ms,
                                                           "roofline": roof}}
    return out


def run_streamed_config(args, model, cfg8) -> dict:
    """Weights in pinned host memory streamed into a 2-slot device ring ("Predictive prefetch"), prompts
    122 / 512 / 2048 at chunk 512, chunk-outer and layer-outer: tok/s against the host-link bound,
    host-to-device bytes against the per-token naive bytes, prefetch hits and misses."""
    import torch

    import prompt_prefill_gb300 as pp
    import synth

    stream = torch.cuda.current_stream()
    cfg = synth.CONFIGS["8b-streamed"]
    chunk = 512
    bw = h2d_bandwidth_gbs()
    # the host link is shared with the machine's other work: every call is timed on its own and the median of
    # five reported (with the fastest and slowest), so one disturbed copy does not move the figure
    steps, warm = 5, 3
    out = {"h2d_gbs_measured": bw, "ring_slots": 2, "chunk": chunk,
           "weights": "the resident workload's 8B-shaped weights, held in pinned host memory by the library"}
    for order, tag in ((pp.PP_LOOP_CHUNK_OUTER, "chunk_outer"), (pp.PP_LOOP_LAYER_OUTER, "layer_outer")):
        g = pp.PrefillModel(cfg8, model, max_seq=max(cfg.extra["prompt_lens"]), max_chunk=chunk,
                            mode=pp.PP_MODE_STREAMED, ring_slots=2, gemm_engine=args.engine, loop_order=order)
        if order == pp.PP_LOOP_LAYER_OUTER:
            g.set_chunk_overlap(True)  # chunk-outer streaming is bound by the host link and stays serial
        res = {}
        for P in cfg.extra["prompt_lens"]:
            d_tok = torch.from_numpy(synth.prompt(cfg, P)).cuda()
            d_logits = torch.empty(cfg8.vocab, dtype=torch.float32, device="cuda")
            for _ in range(warm):
                g.prefill_device(d_tok, P, 0, chunk, d_logits, stream)
            torch.cuda.synchronize()
            g.reset_stats()
            each = sorted(time_calls_each(stream, lambda: g.prefill_device(d_tok, P, 0, chunk, d_logits, stream), steps))
            ms = each[len(each) // 2]
            st = g.stats()
            h2d = st["h2d_bytes"] / steps
            visits = (1 if order == pp.PP_LOOP_LAYER_OUTER else -(-P // chunk)) * cfg8.n_layers
            layer_block = h2d / visits  # device-resident ids: the layer copies are the only host-to-device bytes
            res[str(P)] = {"tok_per_s": P / (ms / 1000), "ms": ms, "ms_min_max": [each[0], each[-1]],
                           "h2d_bytes_per_prompt": h2d,
                           "h2d_bytes_naive_per_prompt": layer_block * cfg8.n_layers * P,
                           "prefetch_hits": st["prefetch_hits"] // steps, "prefetch_misses": st["prefetch_misses"] // steps,
                           "h2d_bound_tok_per_s": P / (h2d / (bw * 1e9)), "frac_of_h2d_bound": (h2d / (bw * 1e9)) / (ms / 1000)}
        out[tag] = res
        g.close()
    return out


def run_ours(args, cfg, world, rank, local, pg):
    import torch

    import prompt_prefill_gb300 as pp
    import synth

    torch.cuda.set_device(local)
    peaks = load_peaks()
    sms = sm_count()
    P, chunk = cfg.prompt_len, args.chunk
    model = synth.make_model(cfg)
    toks = synth.prompt(cfg, P, seed=cfg.seed + rank)
    g = pp.PrefillModel(cfg, model, max_seq=max(cfg.max_seq, P), max_chunk=chunk, gemm_engine=args.engine)
    stream = torch.cuda.current_stream()
    d_tok = torch.from_numpy(toks).cuda()
    d_logits = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")

    def step():
        g.prefill_device(d_tok, P, 0, chunk, d_logits, stream)

    # Warm-up, then profiled steps with the chunks in serial order: every launch of one kernel class
    # bracketed by CUDA events on its stream, so each bracket holds that kernel alone (with chunk overlap a
    # bracket would also hold the other streams' kernels). They give the per-class breakdown and the
    # dominant kernel's own duration for `roofline`. Profiling is off again before the timed region.
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert g.device_status() == pp.PP_OK
    class_ms, class_launches, dominant = profile_classes(g, step, steps_dominant=max(1, min(args.steps, 5)))
    if args.overlap:
        g.set_chunk_overlap(True)
    g.set_graphs(bool(args.graphs))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    g.reset_stats()

    # timed region: K steps, device-resident inputs, nothing but the prefill calls on the streams
    clocks = ClockSampler(local).start()
    barrier(pg)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(pg, ms)
    stats = g.stats()
    launches = stats["kernel_launches"]
    logits = d_logits.cpu().numpy()
    assert np.all(np.isfinite(logits)), "non-finite logits"
    assert g.device_status() == pp.PP_OK

    # e2e: the host C-ABI call (token ids host->device, logits device->host inside), from and into pinned
    # host buffers; warmed up like the device path (its first call captures its own graph)
    h_tok = torch.from_numpy(toks).pin_memory().numpy()
    h_logits = torch.empty(cfg.vocab, dtype=torch.float32).pin_memory().numpy()
    for _ in range(args.warmup):
        g.prefill(h_tok, 0, chunk, out=h_logits)
    barrier(pg)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        g.prefill(h_tok, 0, chunk, out=h_logits)
    t_e2e = time.perf_counter() - t0
    host_logits = h_logits.copy()
    t_e2e = max_over_ranks(pg, t_e2e)
    assert np.array_equal(host_logits.view(np.uint32), logits.view(np.uint32)), "host and device paths differ"
    if args.profile_step:
        # one more step, after everything timed, between cudaProfilerStart and cudaProfilerStop: the launch
        # list of exactly one step under `ncu --profile-from-start off`
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()

    value = replica_tok_per_s(world, P, args.steps, ms_max / 1000.0)
    e2e_value = replica_tok_per_s(world, P, args.steps, t_e2e)
    awork = algorithmic_work(cfg, P, chunk)
    work = awork[dominant]
    scale = 1e12 if work["unit"] == "TFLOP/s" else 1e9
    peak, peak_src = peak_for(work["bound"], peaks, sms)
    # the dominant kernel's average launch duration in the profiled serial steps
    per_launch_work = work["work"] / max(1, class_launches[dominant])
    launch_ms = class_ms[dominant] / max(1, class_launches[dominant])
    achieved = per_launch_work / (launch_ms / 1000.0) / scale

    # prefill roofline of the metric: max(GEMM ops / tensor peak, bytes / 8 TB/s)
    gemm_ops = awork["gemm"]["work"]
    bytes_step = step_bytes(cfg, P, chunk)
    t_tc = gemm_ops / (peak_for("tensor", peaks)[0] * 1e12)
    t_roof = max(t_tc, bytes_step / (NORTH_HBM_GBS * 1e9))
    t_roof_meas = max(t_tc, bytes_step / (float(peaks["hbm_gbs"]) * 1e9))
    step_s = ms_max / 1000.0 / args.steps
    tensor_peak = peak_for("tensor", peaks)[0]

    default_workload = (args.workload, P, chunk) == ("8b", 4096, 512)
    metric = METRIC if default_workload else f"prefill tok/s ({cfg.name}-class int8 decoder, {P}-tok prompt, chunk {chunk})"
    line = {
        "metric": metric, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic (seeded N(0,0.02) int8 per-row weights, uniform ids)",
        "config": workload_config(cfg, args),
        "gemm_engine": {pp.PP_GEMM_MMA: "mma.sync s8", pp.PP_GEMM_TC: "tcgen05 exact-integer f16"}.get(g.gemm_engine),
        "chunk_overlap": bool(args.overlap), "cuda_graphs": bool(args.graphs),
        "prefill_roofline": {"t_roof_ms": 1000 * t_roof, "frac": t_roof / step_s, "tensor_peak_tflops": tensor_peak,
                             "hbm_gbs": NORTH_HBM_GBS, "frac_vs_measured_hbm": t_roof_meas / step_s,
                             "gemm_tops": gemm_ops / 1e12, "bytes_gb": bytes_step / 1e9},
        "roofline": {"kernel": dominant, "bound": work["bound"], "achieved": achieved, "peak": peak,
                     "unit": work["unit"], "frac": achieved / peak,
                     "traffic": kernel_traffic(dominant, "8b" if (args.workload, args.prompt, args.chunk) == ("8b", None, 512) else ""),
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu)", "peak_source": peak_src,
                     "launch_ms": launch_ms, "launches_per_step": class_launches[dominant],
                     "measured_in": "profiled steps with the chunks in serial order: CUDA events on the launching "
                                    "stream around each launch of the kernel, averaged over its launches"},
        # the projection GEMMs as one class: the step's int8 GEMM work over their summed launch times (each
        # launch bracketed by CUDA events in a profiled serial step), against the measured dense f16/bf16 rate
        # (the tensor path they run on; sm_103a has no integer MMA kind)
        "gemm_roofline": {"bound": "tensor", "achieved": gemm_ops / (class_ms["gemm"] / 1000.0) / 1e12,
                          "peak": tensor_peak, "unit": "TFLOP/s",
                          "frac": gemm_ops / (class_ms["gemm"] / 1000.0) / 1e12 / tensor_peak},
        "kernel_ms_per_step": {k: v for k, v in class_ms.items()},  # serial profiled steps
        "weight_bytes_read_per_step": weight_bytes_read(cfg, P, chunk),
        "weight_bytes_naive_per_step": layer_weight_bytes(cfg) * cfg.n_layers * P + cfg.vocab * cfg.dim + 4 * cfg.vocab,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
        "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": 4 * P, "d2h_bytes_per_step": 4 * cfg.vocab},
        "gpu_launches": launches,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, dt = oracle_sample(model, cfg, args.cpu_sample_tokens, toks)
        line["cpu_baseline"] = {"value": v, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                "sample": f"oracle prefill of the first {args.cpu_sample_tokens} tokens of the prompt "
                                          f"in one chunk ({dt:.1f} s)"}
    g.close()
    if rank == 0 and world == 1 and args.workload == "8b" and not args.no_configs:
        # the other measured configurations, each on its own (not part of `value`)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["configs"] = run_small_configs(args, peaks)
        line["streamed"] = run_streamed_config(args, model, cfg)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- streamed weights
def h2d_bandwidth_gbs(nbytes: int = 1 << 30) -> float:
    """Pinned host -> device copy bandwidth (best of 5, CUDA events)."""
    import torch

    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1000) / 1e9)
    return best


def run_streamed(args, cfg, world, rank, local, pg):
    """Weights in pinned host memory, streamed into a device ring ("Predictive
    prefetch"): tok/s per prompt length for the 2-slot ring and the 1-slot
    synchronous loader (chunk-outer: each layer copied once per chunk), and for
    the layer-outer loop (each layer copied once per call), host-to-device
    bytes, prefetch hits and misses."""
    import torch

    import prompt_prefill_gb300 as pp
    import synth

    torch.cuda.set_device(local)
    chunk = args.chunk
    lens = tuple(cfg.extra.get("prompt_lens", (cfg.prompt_len,)))
    model = synth.make_model(cfg)
    bw = h2d_bandwidth_gbs()
    layer_block = None
    results = {}
    layer_profiles = {}
    for slots, order in ((2, pp.PP_LOOP_CHUNK_OUTER), (1, pp.PP_LOOP_CHUNK_OUTER), (2, pp.PP_LOOP_LAYER_OUTER)):
        g = pp.PrefillModel(cfg, model, max_seq=max(lens), max_chunk=chunk, mode=pp.PP_MODE_STREAMED,
                            ring_slots=slots, gemm_engine=args.engine, loop_order=order)
        tag = "" if order == pp.PP_LOOP_CHUNK_OUTER else "_layer_outer"
        overlap = bool(args.overlap) and order == pp.PP_LOOP_LAYER_OUTER  # chunk-outer streaming is H2D-bound
        if overlap:
            g.set_chunk_overlap(True)
        stream = torch.cuda.current_stream()
        for P in lens:
            toks = synth.prompt(cfg, P)
            d_tok = torch.from_numpy(toks).cuda()
            d_logits = torch.empty(cfg.vocab, dtype=torch.float32, device="cuda")
            for _ in range(args.warmup):
                g.prefill_device(d_tok, P, 0, chunk, d_logits, stream)
            torch.cuda.synchronize()
            g.reset_stats()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                g.prefill_device(d_tok, P, 0, chunk, d_logits, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            st = g.stats()
            h2d = st["h2d_bytes"] / args.steps
            n_chunks = -(-P // chunk)
            layer_block = h2d / ((1 if order == pp.PP_LOOP_LAYER_OUTER else n_chunks) * cfg.n_layers)
            results[f"{P}_slots{slots}{tag}"] = {
                "prompt": P, "ring_slots": slots, "loop": "layer-outer" if tag else "chunk-outer",
                "chunk_overlap": overlap,
                "tok_per_s": P / (ms / 1000), "ms": ms,
                "h2d_bytes_per_prompt": h2d, "h2d_bytes_naive_per_prompt": layer_block * cfg.n_layers * P,
                "prefetch_hits": st["prefetch_hits"] // args.steps, "prefetch_misses": st["prefetch_misses"] // args.steps,
                "h2d_bound_tok_per_s": P / (h2d / (bw * 1e9)), "frac_of_h2d_bound": (h2d / (bw * 1e9)) / (ms / 1000)}
        # per-layer profile (an extra, untimed call with the profiler on): sync vs async loader per layer
        P = lens[-1]
        toks = synth.prompt(cfg, P)
        d_tok = torch.from_numpy(toks).cuda()
        g.set_layer_profile(True)
        g.reset_stats()
        g.prefill_device(d_tok, P, 0, chunk, d_logits, stream)
        prof = g.layer_profile()
        g.set_layer_profile(False)
        v = sum(p["visits"] for p in prof)
        layer_profiles[f"{P}_slots{slots}{tag}"] = {
            "per_visit_ms": {k: sum(p[k] for p in prof) / v for k in ("compute_ms", "io_ms", "wait_ms")},
            "visits": v, "wait_ms_by_layer": [round(p["wait_ms"], 3) for p in prof]}
        g.close()
    main = results[f"{lens[-1]}_slots2"]
    line = {"metric": "prefill tok/s, 8B-shaped int8 decoder, weights streamed from pinned host memory",
            "value": main["tok_per_s"], "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": main["ms"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic", "config": {"workload": f"8B-shaped int8 decoder, weights streamed (2-slot ring), "
                                                    f"prompts {lens}, chunk {chunk}"},
            "h2d_gbs_measured": bw, "per_prompt": results, "layer_profile": layer_profiles}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- one kernel
def graph_ms_per_launch(launch, n: int, reps: int = 5) -> float:
    """Replay `n` launches captured in one CUDA graph and return the best average device time per launch
    (CUDA events on the replay stream): the host's launch path is out of the figure, the gap between two
    kernels is in it, as in a model step."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        launch(0)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(n):
            launch(i)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1) / n)
    del graph
    return best


def run_row_op(args, peaks):
    """The per-token quantiser (--op quant) or RMSNorm + quantiser (--op norm_quant) over --m rows of --k,
    int8 and fp16 codes and the row scale written. Timed as graph replays of max(--steps, 96) launches:
    with the inputs rotating through more than twice the L2 (every launch reads its rows from HBM; the
    reported figure) and with one input that stays in L2 (the model's case: the previous kernel has just
    written the rows). A torch f32 -> fp16 copy of the same rows is timed the same way for context."""
    import torch

    import prompt_prefill_gb300 as pp

    m, k = args.m, args.k
    n = max(args.steps, 96)
    nbuf = max(2, -(-(2 * 129 * 2**20) // (4 * m * k)))
    gen = torch.Generator(device="cuda").manual_seed(7)
    xs = [torch.randn((m, k), device="cuda", generator=gen) for _ in range(nbuf)]
    g = 1.0 + 0.02 * torch.randn((k,), device="cuda", generator=gen)
    q8 = torch.empty((m, k), dtype=torch.int8, device="cuda")
    q16 = torch.empty((m, k), dtype=torch.float16, device="cuda")
    asc = torch.empty((m,), device="cuda")
    if args.op == "norm_quant":
        def op(x):
            pp.pp_op_rmsnorm_quantize(x, g, m, k, 1e-5, None, q8, q16, asc)
    else:
        def op(x):
            pp.pp_op_quantize(x, m, k, q8, q16, asc)
    ms_hbm = graph_ms_per_launch(lambda i: op(xs[i % nbuf]), n)
    ms_l2 = graph_ms_per_launch(lambda i: op(xs[0]), n)
    ms_copy = graph_ms_per_launch(lambda i: q16.copy_(xs[i % nbuf]), n)
    # bytes the kernel must move: f32 rows in, int8 + fp16 codes and the row scale out (+ the gains)
    work = m * (4 * k + k + 2 * k + 4) + (4 * k if args.op == "norm_quant" else 0)
    achieved = work / (ms_hbm / 1000) / 1e9
    peak, src = peak_for("hbm", peaks)
    print(json.dumps({"op": args.op, "m": m, "k": k, "launches_per_graph": n, "input_buffers": nbuf,
                      "ms": ms_hbm, "achieved": achieved, "unit": "GB/s", "peak": peak, "frac": achieved / peak,
                      "peak_source": src, "bytes_per_launch": work, "ms_l2_resident": ms_l2,
                      "achieved_l2_resident": work / (ms_l2 / 1000) / 1e9,
                      "ms_torch_f32_to_f16_copy": ms_copy}), flush=True)
    return 0


def run_op(args):
    """Time one kernel alone at a given shape (for ncu captures and per-kernel
    rooflines): --op gemm --engine 1|2 --m --n --k, --op attention --m
    (query rows) --start (start position) on the 8B head layout, or
    --op quant | norm_quant --m (rows) --k (row length)."""
    import torch

    import prompt_prefill_gb300 as pp
    import synth

    peaks = load_peaks()
    torch.cuda.set_device(0)
    m, n, k = args.m, args.n, args.k
    if args.op == "gemm":
        a = torch.from_numpy(synth.uniform_i8(1, 1, (m, k))).cuda()
        a16 = a.to(torch.float16)
        w = torch.from_numpy(synth.uniform_i8(1, 2, (n, k))).cuda()
        ws = torch.full((n,), 1e-3, device="cuda")
        as_ = torch.full((m,), 1e-2, device="cuda")
        out = torch.empty((m, n), device="cuda")
        engine = args.engine or pp.PP_GEMM_TC

        def once():
            pp.pp_op_gemm(engine, pp.PP_EPI_STORE, a, a16, w, ws, as_, m, n, k, out, n)
        work, unit, bound = 2.0 * m * n * k, "TFLOP/s", "tensor"
    elif args.op == "attention":
        H, Hkv, hd = args.heads, args.kv_heads, args.hd
        start = args.start
        q = torch.randn((m, H, hd), device="cuda")
        kc = torch.randn((start + m, Hkv, hd), device="cuda")
        vc = torch.randn((start + m, Hkv, hd), device="cuda")
        o = torch.empty_like(q)

        def once():
            pp.pp_op_attention(q, kc, vc, m, start, H, Hkv, hd, o)
        pairs = sum(start + i + 1 for i in range(m))
        work, unit, bound = 4.0 * hd * H * pairs, "TFLOP/s", "alu"
    elif args.op in ("quant", "norm_quant"):
        return run_row_op(args, peaks)
    else:
        raise SystemExit(f"unknown --op {args.op}")
    for _ in range(args.warmup):
        once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        once()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    achieved = work / (ms / 1000) / (1e9 if unit == "GB/s" else 1e12)
    peak, src = peak_for(bound, peaks)
    print(json.dumps({"op": args.op, "m": m, "n": n, "k": k, "start": args.start, "engine": args.engine,
                      "ms": ms, "achieved": achieved, "unit": unit, "peak": peak, "frac": achieved / peak,
                      "peak_source": src}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="8b")
    ap.add_argument("--chunk", type=int, default=None)
    ap.add_argument("--prompt", type=int, default=None)
    ap.add_argument("--engine", type=int, default=0, help="0 auto, 1 mma.sync, 2 tcgen05")
    ap.add_argument("--cpu-sample-tokens", type=int, default=16)
    ap.add_argument("--ref-sample-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the 350M, 1B and streamed measurements that follow the 8B line")
    ap.add_argument("--overlap", type=int, default=1,
                    help="1 (default): consecutive chunks on their own streams, up to 32 (pp_set_chunk_overlap); 0: serial")
    ap.add_argument("--graphs", type=int, default=1,
                    help="1 (default): each prefill call replayed from a CUDA graph after its first (pp_set_graphs)")
    ap.add_argument("--profile-step", action="store_true",
                    help="after the timed steps, run one more step between cudaProfilerStart and cudaProfilerStop "
                         "(for ncu --profile-from-start off)")
    ap.add_argument("--op", default=None, help="time one kernel alone: gemm | attention | quant | norm_quant")
    ap.add_argument("--heads", type=int, default=32, help="--op attention: query heads")
    ap.add_argument("--kv-heads", type=int, default=8, help="--op attention: KV heads")
    ap.add_argument("--hd", type=int, default=128, help="--op attention: head dim (64 or 128)")
    ap.add_argument("--m", type=int, default=512)
    ap.add_argument("--n", type=int, default=28672)
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--start", type=int, default=3584)
    args = ap.parse_args(argv)
    if args.op:
        return run_op(args)
    if args.warmup < 3:
        args.warmup = 3  # timing rule: at least 3 warm-up steps
    import synth

    cfg = synth.CONFIGS[args.workload]
    if args.prompt:
        cfg.prompt_len = args.prompt
    args.chunk = args.chunk or cfg.chunk
    world, rank, local, pg = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, cfg, world, rank, pg)
        if args.workload == "8b-streamed":
            return run_streamed(args, cfg, world, rank, local, pg)
        return run_ours(args, cfg, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
