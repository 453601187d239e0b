"""Benchmark of the GPT-2 forward pass on GB300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gpt2-124m-b16] [--precision fp16] [--gemm-diag]

A step is one gpt2_forward over a batch of B sequences of T tokens of
seeded synthetic input (random-init GPT-2 weights, uniform token ids), with
the logits and the softmax probabilities written.  `value` is tokens/s of
the whole job (all ranks), timed with CUDA events around exactly K steps
bracketed by a barrier and a device synchronisation, max over ranks.  The
working set (logits plus probabilities alone are 6.6 GB at B=16) is far
larger than the 129 MB L2, so no L2 flush runs between steps.

Several GPUs run independent replicas (the forward pass of one batch needs
no exchange between GPUs): each rank processes its own batch, no collective
touches the data path, and scaling is weak.

--impl reference times the CPU oracle (the plain double-precision C
implementation) on the host cores, on a bounded sample of the same workload
per step; rank 0 alone runs it.

--workload gpt2-124m-decode measures KV-cached decoding instead: per run a
prefill of 32 prompts of 512 tokens (reported apart), then 128 greedy steps
(argmax + gpt2_decode_step), K runs timed; value = decoded tokens/s.
--gemm-diag adds each GEMM site's time beside cuBLAS at the same shape.
--attention-forward / --attention-backward time one layer's attention
forward (16-bit operands) / backward (fp32) instead.
--train times whole training steps (forward, softmax cross-entropy,
backward, AdamW; tf32 GEMMs, or fp32 with --precision fp32) instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gpt_transformer_forward_gb300 import inputs  # noqa: E402

METRIC = "GPT-2 124M forward tokens/s (B=16,T=1024) on 1 GB300; % of roofline"


def metric_name(w, probs="fp32"):
    """The metric string of a forward workload: the headline string for the
    124M B=16 T=1024 pass with fp32 probabilities, the same wording with its
    own model, shape and probabilities type for every other one."""
    if w.name == "gpt2-124m-b16" and probs == "fp32":
        return METRIC
    model = {12: "124M", 24: "medium"}.get(w.cfg.num_layers, f"L{w.cfg.num_layers}")
    extra = "" if probs == "fp32" else f", {probs} probabilities"
    return f"GPT-2 {model} forward tokens/s (B={w.B},T={w.T}{extra}) on 1 GB300; % of roofline"

UNIT = "tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------- algorithmic cost
def stage_costs(cfg, B, T, act_bytes=2, probs_bytes=4):
    """Algorithmic FLOPs and bytes of each stage of one forward pass (every
    layer summed): bytes count each input read once and each output written
    once, with operand buffers of act_bytes (2 for bf16/fp16), the residual
    stream and logits fp32, probabilities of probs_bytes, weights 16-bit, and the causal
    attention FLOPs only (j <= t).  With 16-bit operands the two projections
    write their output y in 16 bits and the residual add x += y runs in the
    LayerNorm that follows (layer 0's first LayerNorm has no y to add; the
    final one does not write x back)."""
    C, L, NH, Vp = cfg.channels, cfg.num_layers, cfg.num_heads, cfg.padded_vocab_size
    hs = C // NH
    N = B * T
    a, w = act_bytes, 2
    fused = act_bytes == 2
    ln_bytes = N * C * 4 + N * C * a + 2 * C * 4
    fused_ln = ln_bytes + N * C * a + N * C * 4   # + read y, + write x
    proj_out = N * C * a if fused else 2 * N * C * 4
    pairs = T * (T + 1) // 2
    return {
        "encoder": (0, 4 * N + N * C * 4 + T * C * 4 + N * C * 4),
        "ln1": (0, ln_bytes + (L - 1) * (fused_ln if fused else ln_bytes)),
        "qkv": (L * 2 * N * C * 3 * C, L * (N * C * a + 3 * C * C * w + 3 * C * 4 + N * 3 * C * a)),
        "attention": (L * B * NH * 4 * hs * pairs, L * (N * 3 * C * a + N * C * a)),
        "attproj": (L * 2 * N * C * C, L * (N * C * a + C * C * w + C * 4 + proj_out)),
        "ln2": (0, L * (fused_ln if fused else ln_bytes)),
        "fc": (L * 2 * N * C * 4 * C, L * (N * C * a + 4 * C * C * w + 4 * C * 4 + N * 4 * C * a)),
        "fcproj": (L * 2 * N * 4 * C * C, L * (N * 4 * C * a + 4 * C * C * w + C * 4 + proj_out)),
        "lnf": (0, ln_bytes + (N * C * a if fused else 0)),
        "lm_head": (2 * N * C * Vp, N * C * a + Vp * C * w + N * Vp * 4),
        "softmax": (0, N * Vp * (4 + probs_bytes)),
    }


def decode_step_bytes(cfg, B, pos, act_bytes=2):
    """Algorithmic HBM bytes of one KV-cached decode step at position pos:
    the weights of the blocks and of the tied LM head (16-bit, or fp32 when
    act_bytes is 4), the fp32 biases and LayerNorm parameters, the cache
    read of positions 0..pos-1 and the append at pos (keys and values,
    act_bytes each), the token ids, embedding rows, and the B rows of
    logits (written, then read by the softmax) and probabilities, as the
    forward pass's stage sum counts them.  The activations passed between
    kernels (a few B x C rows, under 0.1 % here) are left out."""
    C, L, Vp = cfg.channels, cfg.num_layers, cfg.padded_vocab_size
    weights = (L * 12 * C * C + Vp * C) * act_bytes
    small = (L * 13 * C + 2 * C) * 4  # per layer 9C of biases and 4C of LayerNorm; LN_f
    kv = 2 * L * B * C * act_bytes * (pos + 1)  # pos rows read, one row written
    rows = B * 4 + (B + 1) * C * 4 + 3 * B * Vp * 4
    return weights + small + kv + rows


def measured_traffic(stage):
    """DRAM bytes per launch of a stage's kernel from the committed ncu
    record, or None when absent or taken on a different kernel source."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[stage]
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        return rec["bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# -------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle
def oracle_sample_run(w, params, tok, T_s):
    """One oracle forward pass over sequence 0's first T_s tokens (logits and
    probabilities, every column); returns seconds."""
    import oracle
    t0 = time.perf_counter()
    oracle.forward(w.cfg, params, tok[:1, :T_s])
    return time.perf_counter() - t0


def oracle_threads():
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def cpu_baseline(w, params, tok, target_s=15.0):
    """The oracle timed on a bounded sample (about target_s seconds)."""
    t8 = oracle_sample_run(w, params, tok, 8)
    T_s = int(max(8, min(w.T, 8 * target_s / max(t8, 1e-3))))
    dt = oracle_sample_run(w, params, tok, T_s)
    return {"value": T_s / dt, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"1 sequence x {T_s} tokens of {w.name} (double precision, logits and probs), {dt:.1f} s"}


# ------------------------------------------------------------------- arms
def dist_setup(n_gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist
    return rank, world, local, pg


def gemm_vs_library(cfg, N, stage_ms):
    """Diagnostic (--gemm-diag): per GEMM site, this library's time per launch
    (its stage time from gpt2_forward_profile, epilogue included) beside the
    vendor library's plain fp16 matrix product of the same shape
    (torch.matmul: cuBLAS; fp16 out, fp32 out for the LM head)."""
    import torch
    C, L, Vp = cfg.channels, cfg.num_layers, cfg.padded_vocab_size
    sites = {"qkv": (C, 3 * C, L), "attproj": (C, C, L), "fc": (C, 4 * C, L), "fcproj": (4 * C, C, L),
             "lm_head": (C, Vp, 1)}
    out = {}
    for name, (K, OC, launches) in sites.items():
        a = torch.randn(N, K, device="cuda", dtype=torch.float16)
        wt = torch.randn(OC, K, device="cuda", dtype=torch.float16)
        f32 = name == "lm_head"
        f = (lambda: torch.mm(a, wt.t(), out_dtype=torch.float32)) if f32 else (lambda: a @ wt.t())
        try:
            f()
        except (TypeError, RuntimeError):  # no fp32-output matmul in this torch: fp16 out
            f32 = False
            f = lambda: a @ wt.t()
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            f()
        e1.record()
        torch.cuda.synchronize()
        lib_us = e0.elapsed_time(e1) / 10 * 1e3
        ours_us = stage_ms[name] / launches * 1e3
        out[name] = {"shape_mnk": [N, OC, K], "ours_us": round(ours_us, 1), "cublas_us": round(lib_us, 1),
                     "cublas_out": "fp32" if f32 else "fp16"}
        del a, wt
    return out


def rank_tokens(w, tok, rank):
    """The token batch of replica `rank`: the workload's own on rank 0, a
    differently seeded batch of the same shape on every other rank."""
    if rank == 0:
        return tok
    return inputs.make_tokens(w.token_seed + 7919 * rank, w.B, w.T, w.cfg.vocab_size)


def max_over_ranks(value, pg, device):
    """The largest of every rank's `value` (a float), on every rank; `device`
    holds the reduction tensor ("cuda" with NCCL, "cpu" with gloo)."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, ms_per_step):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def run_reference(args):
    rank, world, _, pg = dist_setup(args.gpus)
    if rank != 0:
        if pg is not None:
            pg.barrier()
        return
    w = inputs.WORKLOADS[args.workload]
    params, tok = inputs.workload_inputs(w)
    # size one step's sample so that warm-up plus timed steps take ~2 minutes
    t8 = oracle_sample_run(w, params, tok, 8)
    per_step = 120.0 / (args.steps + args.warmup)
    T_s = int(max(1, min(w.T, 8 * per_step / max(t8, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample_run(w, params, tok, T_s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_run(w, params, tok, T_s)
    dt = time.perf_counter() - t0
    value = args.steps * T_s / dt
    sample = f"per step: 1 sequence x {T_s} tokens of {w.name} (double precision, logits and probs)"
    line = {"impl": "reference", "metric": metric_name(w, args.probs), "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": w.B, "T": w.T},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()


DECODE_METRIC = "GPT-2 124M KV-cached decode tokens/s (B=32, prompt 512, 128 greedy steps) on 1 GB300"


def run_decode(args, w, precision):
    """The KV-cached decode workload: per run, a prefill of the B prompts of T
    tokens (gpt2_forward filling the cache; timed and reported apart), then
    w.decode_steps steps of greedy argmax + gpt2_decode_step (timed).  K runs
    after W warm-up runs; tokens/s = B x steps x K / decode time."""
    import torch
    from gpt_transformer_forward_gb300 import binding as ab
    from gpt_transformer_forward_gb300.runner import GPT2Model

    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    params, tok = inputs.workload_inputs(w)
    tok = rank_tokens(w, tok, rank)
    cfg, B, T, n = w.cfg, w.B, w.T, w.decode_steps
    model = GPT2Model(cfg, params, B, T, precision)
    cache = model.new_kvcache(B)
    tok_d = torch.from_numpy(tok).cuda()
    prefill_logits, _ = model.new_outputs(B, T, probs=False)
    last = torch.empty((B, cfg.padded_vocab_size), dtype=torch.float32, device="cuda")
    logits, probs = model.new_outputs(B, None)
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    prefill_ms = decode_ms = 0.0
    for run in range(args.warmup + args.steps):
        cache.zero_()
        p0.record(stream)
        model.forward(tok_d, prefill_logits, None, cache)
        p1.record(stream)
        last.copy_(prefill_logits[:, T - 1])
        e0.record(stream)
        src = last
        for i in range(n):
            ab.gpt2_argmax(nxt, src, B, cfg.vocab_size, cfg.padded_vocab_size)
            model.decode_step(cache, nxt, T + i, logits, probs)
            src = logits
        e1.record(stream)
        torch.cuda.synchronize()
        if run >= args.warmup:
            prefill_ms += p0.elapsed_time(p1)
            decode_ms += e0.elapsed_time(e1)
    err = ab.gpt2_get_error()
    decode_ms = max_over_ranks(decode_ms, pg, "cuda")
    tokens = B * n * args.steps
    # HBM floor of the timed steps (positions T .. T + n - 1) at the measured
    # copy bandwidth
    peaks, peak_src = load_peaks()
    act = 2 if precision in (ab.GPT2_BF16, ab.GPT2_FP16) else 4
    step_bytes = sum(decode_step_bytes(cfg, B, T + i, act) for i in range(n)) / n
    ms_step = decode_ms / (args.steps * n)
    floor_ms = step_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    line = {
        "metric": DECODE_METRIC, "value": job_tokens_per_s(world, tokens, decode_ms), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.precision,
        "data": "synthetic",
        "config": {"workload": w.name, "B": B, "prompt": T, "decode_steps": n, "layers": cfg.num_layers,
                   "outputs": "logits+probs per step, greedy argmax", "parallelism": f"replicas{world}"},
        "prefill_ms": prefill_ms / args.steps,
        "step_roofline": {"bound": "hbm", "bytes_per_step": step_bytes, "floor_ms": floor_ms, "measured_ms": ms_step,
                          "frac": floor_ms / ms_step, "peak_gbs": peaks["hbm_gbs"], "peak_source": peak_src},
        # per step: argmax, encoder, 7 per layer (LN, QKV, attention with the
        # cache append, projection, LN, FC, FC-proj), LN_f, LM head, softmax
        "gpu_launches": (7 * cfg.num_layers + 5) * n * args.steps,
        "device_error_word": err,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


ATTN_BWD_METRIC = "GPT-2 124M causal attention backward, one layer (B=16,T=1024,12 heads of 64), {}, ms"


def attention_backward_flops(B, T, C, NH):
    """Algorithmic FLOPs of one attention backward: the four gradient
    products dV = P^T dO, dP = dO V^T, dQ = dS K, dK = dS^T Q over the causal
    (t, j) pairs, 2 hs FLOPs each (the recomputation of S is not counted)."""
    hs = C // NH
    return B * NH * (T * (T + 1) // 2) * 4 * 2 * hs


ATTN_FWD_METRIC = "GPT-2 124M causal attention forward, one layer (B=16,T=1024,12 heads of 64), ms"


def run_attention_forward(args, w):
    """One layer's attention forward at the workload's shape through
    attention_forward (16-bit operands per --precision; the call converts
    the fp32 qkv to the operand type, then runs the attention kernel):
    K timed calls after W warm-up calls; the attention kernel alone is
    timed by the forward pass's stage profile."""
    import torch
    from gpt_transformer_forward_gb300 import binding as ab

    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    precision = ab.PRECISIONS[args.precision]
    cfg, B, T = w.cfg, w.B, w.T
    C, NH = cfg.channels, cfg.num_heads
    qkv = torch.from_numpy(inputs.make_normal(803 + rank, (B, T, 3 * C), 0.55).astype("float32")).cuda()
    out = torch.empty((B, T, C), dtype=torch.float32, device="cuda")
    wsz = ab.attention_workspace_size(B, T, C, precision)
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        ab.attention_forward(out, qkv, B, T, C, NH, precision, ws, wsz)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        ab.attention_forward(out, qkv, B, T, C, NH, precision, ws, wsz)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, "cuda")
    line = {"metric": ATTN_FWD_METRIC, "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": args.precision, "data": "synthetic",
            "config": {"workload": w.name + "-attention-forward", "B": B, "T": T, "C": C, "heads": NH,
                       "includes": "fp32 -> 16-bit conversion of qkv"},
            "gpu_launches": 2 * args.steps, "device_error_word": ab.gpt2_get_error()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_attention_backward(args, w):
    """One layer's attention backward at the workload's shape through
    attention_backward: fp32 CUDA cores with --precision fp32, else the bf16
    tensor-core path (the call converts qkv and dout to bf16, reruns the
    forward for the row statistic, then runs the two backward kernels).  K
    timed calls after W warm-up calls, CUDA events on the stream."""
    import torch
    from gpt_transformer_forward_gb300 import binding as ab

    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    precision = ab.GPT2_FP32 if args.precision == "fp32" else ab.GPT2_BF16
    cfg, B, T = w.cfg, w.B, w.T
    C, NH = cfg.channels, cfg.num_heads
    qkv = torch.from_numpy(inputs.make_normal(801 + rank, (B, T, 3 * C), 0.55).astype("float32")).cuda()
    dout = torch.from_numpy(inputs.make_normal(802 + rank, (B, T, C), 1.0).astype("float32")).cuda()
    out = torch.empty((B, T, C), dtype=torch.float32, device="cuda")
    ab.attention_forward(out, qkv, B, T, C, NH, ab.GPT2_FP32, None, 0)
    dqkv = torch.empty((B, T, 3 * C), dtype=torch.float32, device="cuda")
    wsz = ab.attention_backward_workspace_size(B, T, C, NH, precision)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        ab.attention_backward(dqkv, dout, qkv, out, B, T, C, NH, precision, ws, wsz)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        ab.attention_backward(dqkv, dout, qkv, out, B, T, C, NH, precision, ws, wsz)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, "cuda")
    flops = attention_backward_flops(B, T, C, NH)
    f32 = precision == ab.GPT2_FP32
    line = {"metric": ATTN_BWD_METRIC.format("fp32" if f32 else "bf16 tensor cores"), "value": ms, "unit": "ms",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32" if f32 else "bf16",
            "data": "synthetic",
            "config": {"workload": w.name + "-attention-backward", "B": B, "T": T, "C": C, "heads": NH,
                       "includes": "the fp32 kernels" if f32 else
                       "qkv and dout to bf16, the forward rerun for the row statistic, dO prep, dK/dV and dQ"},
            "tflops": flops / (ms * 1e-3) / 1e12, "algorithmic_flops": flops,
            "gpu_launches": (3 if f32 else 5) * args.steps, "device_error_word": ab.gpt2_get_error()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


TRAIN_METRIC = "GPT-2 training step tokens/s (forward, softmax cross-entropy, backward, AdamW) on 1 GB300"


def run_train(args, w):
    """Training steps at the workload's shape: gpt2_forward_backward then
    gpt2_adamw, K timed steps after W warm-up steps (fp32 activations; tf32
    tensor-core operands unless --precision fp32)."""
    import torch
    from gpt_transformer_forward_gb300 import binding as ab

    precision = ab.GPT2_FP32 if args.precision == "fp32" else ab.GPT2_TF32
    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    params, tok = inputs.workload_inputs(w)
    tok = rank_tokens(w, tok, rank)
    cfg, B, T = w.cfg, w.B, w.T
    tgt = np.roll(tok, -1, axis=1)  # next-token targets (the last wraps to the first)
    P = torch.from_numpy(params).cuda()
    G, M, V = torch.empty_like(P), torch.zeros_like(P), torch.zeros_like(P)
    tk, tg = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    wsz = ab.gpt2_train_workspace_size(cfg, B, T, precision)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")

    def step(t):
        ab.gpt2_forward_backward(cfg, P, G, tk, tg, B, T, loss, ws, wsz, precision)
        ab.gpt2_adamw(P, G, M, V, P.numel(), 3e-4, 0.9, 0.95, 1e-8, 0.0, t)

    for t in range(1, args.warmup + 1):
        step(t)
    torch.cuda.synchronize()
    first = float(loss.item())
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for t in range(args.warmup + 1, args.warmup + args.steps + 1):
        step(t)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, "cuda")
    line = {"metric": TRAIN_METRIC, "value": job_tokens_per_s(world, B * T, ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32" if precision == ab.GPT2_FP32 else "f32 (tf32 GEMMs)",
            "data": "synthetic", "config": {"workload": w.name + "-train", "B": B, "T": T, "layers": cfg.num_layers},
            "loss_after_warmup": first, "loss_last": float(loss.item()),
            "workspace_gb": wsz / 1e9, "device_error_word": ab.gpt2_get_error()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_ours(args):
    import torch
    from gpt_transformer_forward_gb300 import binding as ab
    from gpt_transformer_forward_gb300.runner import GPT2Model

    w = inputs.WORKLOADS[args.workload]
    precision = ab.PRECISIONS[args.precision]
    if args.attention_backward:
        return run_attention_backward(args, w)
    if args.attention_forward:
        return run_attention_forward(args, w)
    if args.train:
        return run_train(args, w)
    if w.decode_steps:
        return run_decode(args, w, precision)
    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev_index = torch.cuda.current_device()
    params, tok = inputs.workload_inputs(w)
    tok = rank_tokens(w, tok, rank)  # replicas: each rank its own batch of token ids
    model = GPT2Model(w.cfg, params, w.B, w.T, precision)
    probs_dtype = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}[args.probs]
    logits, probs = model.new_outputs(w.B, w.T, probs_dtype=probs_dtype)
    tok_d = torch.from_numpy(tok).cuda()
    stream = torch.cuda.current_stream()

    def barrier():
        if pg is not None:
            pg.barrier()

    for _ in range(args.warmup):
        model.forward(tok_d, logits, probs)
    torch.cuda.synchronize()
    assert ab.gpt2_get_error() == 0

    # ---- device-resident timed region
    clocks = ClockSampler(dev_index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        model.forward(tok_d, logits, probs)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, "cuda")
    err = ab.gpt2_get_error()

    # ---- end to end: pinned host tokens in, logits and probabilities out.
    # A serving loop: two sets of device outputs, and the device-to-host
    # copy of step i (6.6 GB at B=16, bound by the host link) runs on a copy
    # stream while step i + 1 computes; every step's copies are inside the
    # timed region, the last one included.
    tok_h = torch.from_numpy(tok).pin_memory()
    logits_h = torch.empty(logits.shape, dtype=torch.float32, pin_memory=True)
    probs_h = torch.empty(probs.shape, dtype=probs_dtype, pin_memory=True)
    bufs = [(logits, probs), model.new_outputs(w.B, w.T, probs_dtype=probs_dtype)]
    copy_stream = torch.cuda.Stream()
    copied = [None, None]  # event: the copy out of buffer set b is done
    e2e_steps = max(3, min(args.steps, 20))
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(e2e_steps):
        lg, pr = bufs[i & 1]
        if copied[i & 1] is not None:
            stream.wait_event(copied[i & 1])
        tok_d.copy_(tok_h, non_blocking=True)
        model.forward(tok_d, lg, pr)
        computed = torch.cuda.Event()
        computed.record(stream)
        copy_stream.wait_event(computed)
        with torch.cuda.stream(copy_stream):
            logits_h.copy_(lg, non_blocking=True)
            probs_h.copy_(pr, non_blocking=True)
        copied[i & 1] = torch.cuda.Event()
        copied[i & 1].record(copy_stream)
    stream.wait_stream(copy_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    del bufs
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, pg, "cuda")

    # ---- per-stage times (CUDA events between stages) and the roofline
    prof_runs = 5
    stage_ms = {k: 0.0 for k in ab.STAGES}
    for _ in range(prof_runs):
        for k, v in model.forward_profile(tok_d, logits, probs).items():
            stage_ms[k] += v / prof_runs
    peaks, peak_src = load_peaks()
    costs = stage_costs(w.cfg, w.B, w.T, act_bytes=2 if precision in (ab.GPT2_BF16, ab.GPT2_FP16) else 4,
                        probs_bytes=probs.element_size())
    hbm = peaks["hbm_gbs"] * 1e9
    tensor = peaks["bf16_tflops_sustained"] * 1e12
    stages, roof_ms = {}, 0.0
    for k, (flops, nbytes) in costs.items():
        t_roof = max(flops / tensor, nbytes / hbm) * 1e3
        roof_ms += t_roof
        stages[k] = {"ms": round(stage_ms[k], 4), "roofline_ms": round(t_roof, 4),
                     "bound": "tensor" if flops / tensor > nbytes / hbm else "hbm"}
    dom = max(stage_ms, key=stage_ms.get)
    flops, nbytes = costs[dom]
    launches = w.cfg.num_layers if dom not in ("encoder", "lnf", "lm_head", "softmax") else 1
    per_launch_ms = stage_ms[dom] / launches
    if flops / tensor > nbytes / hbm:
        achieved = flops / launches / (per_launch_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s"}
    else:
        achieved = nbytes / launches / (per_launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    # the committed DRAM records are of the headline pass (fp32 probabilities)
    roof["traffic"] = measured_traffic(dom) if args.workload == "gpt2-124m-b16" and args.probs == "fp32" else None
    roof["algorithmic_per_launch"] = flops / launches if roof["bound"] == "tensor" else nbytes / launches
    roof["kernel"] = dom
    roof["peak_source"] = peak_src

    tokens = w.B * w.T
    value = job_tokens_per_s(world, tokens, ms)
    launches_per_step = 1 + 7 * w.cfg.num_layers + 3
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, params, tok)
    line = {
        "metric": metric_name(w, args.probs), "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.precision, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "layers": w.cfg.num_layers,
                   "channels": w.cfg.channels, "heads": w.cfg.num_heads, "vocab": w.cfg.vocab_size,
                   "padded_vocab": w.cfg.padded_vocab_size,
                   "outputs": "logits+probs" if args.probs == "fp32" else f"logits (fp32) + probs ({args.probs})",
                   "l2": "no flush: working set > 7 GB, L2 129 MB", "parallelism": f"replicas{world}"},
        "e2e": {"value": job_tokens_per_s(world, tokens, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": int(tok.nbytes),
                "d2h_bytes_per_step": int(logits.numel() * 4 + probs.numel() * probs.element_size())},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roof,
        "pass_roofline": {"roofline_ms": roof_ms, "measured_ms": ms, "frac": roof_ms / ms,
                          "peaks": "hbm_gbs, bf16_tflops_sustained of " + peak_src},
        "stages": stages,
        "clocks": clk,
        "device_error_word": err,
        "cpu_baseline": cpu,
    }
    if args.gemm_diag and rank == 0:
        line["gemm_vs_cublas"] = gemm_vs_library(w.cfg, w.B * w.T, stage_ms)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gpt2-124m-b16", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--precision", default="fp16", choices=["fp16", "bf16", "tf32", "fp32"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--probs", default="fp32", choices=["fp32", "fp16", "bf16"],
                    help="element type of the forward pass's probabilities output (fp32: the headline)")
    ap.add_argument("--train", action="store_true",
                    help="time training steps (forward, loss, backward, AdamW) at the workload's shape instead")
    ap.add_argument("--attention-forward", action="store_true",
                    help="time one layer's attention_forward at the workload's shape instead")
    ap.add_argument("--attention-backward", action="store_true",
                    help="time one layer's attention backward at the workload's shape instead (fp32 with --precision fp32, "
                         "else bf16 tensor cores)")
    ap.add_argument("--gemm-diag", action="store_true",
                    help="add each GEMM site's time beside cuBLAS at the same shape (diagnostic)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
