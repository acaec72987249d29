"""Benchmark of the TSP-folded block on GB300: tokens/s and TFLOP/s at 1 GPU.

Workload (default): 7B-shaped TSP block forward, S=16384 tokens, D=8 virtual
ranks under zigzag causal partitioning, d_model=4096, 32 heads x 128, SwiGLU
inter=11008, bf16 storage with fp32 accumulation; synthetic Gaussian inputs
(x ~ N(0,1), weights ~ N(0,0.02), gains 1).

One step = the whole hot path on one batch resident in HBM: zigzag-permute x,
RMSNorm, shard-streamed Q|K|V GEMM, zigzag causal flash attention, W_O split-K
GEMM + residual, RMSNorm, W_1|W_3 SwiGLU GEMM, W_2 ring-order split-K GEMM +
residual, un-permute y.  The step's working set (x 128 MiB, weights 405 MiB,
activations > 1 GiB) is larger than L2, so no explicit flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload fwd16k|fwd128k|fwdbwd32k|fwdbwd8k|mlp16k|
                                fwd512k|fwd1m|fwdbwd512k|stack32_16k|stack32train_16k]

With N > 1 (torchrun, one rank per GPU) every rank runs its own replica
("replicas only": the block has no data-path exchange on one node's GPUs in
this form); value = all ranks' tokens / max-over-ranks time.
The reference arm is the CPU float64 oracle, timed on this host's cores, one
bounded sample of the same workload per step (cpu_sample: for the forward
workloads a virtual rank's step of the TSP schedule on mirrored row pairs,
which carry exactly the block's average work per token).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: (S, D, d, H, inter, kind)
    "fwd16k": (16384, 8, 4096, 32, 11008, "fwd"),
    "fwd128k": (131072, 8, 4096, 32, 11008, "fwd"),
    "fwdbwd32k": (32768, 8, 4096, 32, 11008, "fwdbwd"),
    "fwdbwd8k": (8192, 8, 4096, 32, 11008, "fwdbwd"),   # small case for profiler captures
    # long context on one GPU without sequence tiling: the forward fits up to
    # ~1M tokens (92 GB of workspace), the training step up to 512K (179 GB)
    "fwd512k": (524288, 8, 4096, 32, 11008, "fwd"),
    "fwd1m": (1048576, 8, 4096, 32, 11008, "fwd"),
    "fwdbwd512k": (524288, 8, 4096, 32, 11008, "fwdbwd"),
    # beyond the untiled limit: the MLP in sequence tiles of 16384 rows, its
    # G and pre-activations recomputed in the backward instead of kept
    "fwdbwd768k_tiled": (786432, 8, 4096, 32, 11008, "fwdbwd"),
    "mlp16k": (16384, 4, 4096, 32, 11008, "mlp"),
    # 32-layer stacks of the 7B-shaped block (each layer its own weights)
    "stack32_16k": (16384, 8, 4096, 32, 11008, "fwd"),
    "stack32train_16k": (16384, 8, 4096, 32, 11008, "fwdbwd"),
    # the 7B-shaped block with grouped-query attention (8 K/V heads, four
    # query heads per group) and rotary embedding
    "fwd16k_gqa8": (16384, 8, 4096, 32, 11008, "fwd"),
    # the same forward computed rank by rank by the TSP schedule: every virtual
    # rank's per-rank calls in turn (tsp_rank_*), the shard broadcast, K/V
    # all-gather and MLP ring as device copies on a copy stream
    "fwd16k_by_rank": (16384, 8, 4096, 32, 11008, "fwd"),
    # ... and the training step that way (the backward schedule's exchanges
    # as device copies and sums; each shard's gradient left at its owner)
    "fwdbwd16k_by_rank": (16384, 8, 4096, 32, 11008, "fwdbwd"),
    "fwdbwd8k_gqa8": (8192, 8, 4096, 32, 11008, "fwdbwd"),
    # inference: one new token per step after a 16384-token prompt held in the
    # zigzag KV cache (the prefill runs once, untimed)
    "decode16k": (16384, 8, 4096, 32, 11008, "decode"),
    "decode16k_gqa8": (16384, 8, 4096, 32, 11008, "decode"),
}
DECODE_T = 1        # new tokens per decode call
DECODE_GEN = 256    # decode calls per step: a step generates 256 tokens after the prompt
LAYERS = {"stack32_16k": 32, "stack32train_16k": 32}   # other workloads: one block
# block variants of a workload (default: multi-head attention, no positional encoding)
VARIANTS = {"fwd16k_gqa8": {"Hkv": 8, "rope_base": 500000.0},
            "fwdbwd8k_gqa8": {"Hkv": 8, "rope_base": 500000.0},
            "decode16k_gqa8": {"Hkv": 8, "rope_base": 500000.0},
            "fwdbwd768k_tiled": {"mlp_tile": 16384},
            "fwd16k_by_rank": {"by_rank": True},
            "fwdbwd16k_by_rank": {"by_rank": True}}


def decode_bytes(name, d, inter, dkv, n_rows, T=DECODE_T):
    """Algorithmic HBM bytes of one decode-step kernel: every bf16 weight
    once, the fp16 K/V of every cached row once (the activations of T tokens
    are negligible and left out)."""
    table = {
        "gemv_qkv": 2.0 * d * (d + 2 * dkv),
        "gemv_oproj": 2.0 * d * d,
        "gemv_w13_swiglu": 4.0 * d * inter,
        "gemv_w2": 2.0 * d * inter,
        "decode_attn": 2.0 * 2 * dkv * n_rows,
    }
    return table.get(name)

DEFAULT_WORKLOAD = "fwd16k"
NOMINAL_BF16_TFLOPS = 2250.0   # GB300 rated dense bf16 (context; the measured peaks are the denominators)


def block_flops(S, d, inter, kind, dkv=None):
    """Algorithmic flops: 8Sd^2 (Q,K,V,O) + 6SdI (SwiGLU) + 2S(S+1)d (causal pairs);
    with K/V of width dkv < d the projections take 4Sd^2 + 4Sd*dkv."""
    if kind == "mlp":
        return 6.0 * S * d * inter
    dkv = d if dkv is None else dkv
    f = 4.0 * S * d * d + 4.0 * S * d * dkv + 6.0 * S * d * inter + 2.0 * S * (S + 1) * d
    return 3.0 * f if kind == "fwdbwd" else f


def gemm_flops(name, S, d, inter, dkv=None):
    dkv = d if dkv is None else dkv
    table = {
        "gemm_qkv": 2.0 * S * d * (d + 2 * dkv),
        # grouped K/V heads: Q and K|V are separate GEMMs
        "gemm_q": 2.0 * S * d * d,
        "gemm_kv": 4.0 * S * d * dkv,
        "gemm_wgrad_q": 2.0 * S * d * d,
        "gemm_wgrad_kv": 4.0 * S * d * dkv,
        "gemm_oproj": 2.0 * S * d * d,
        "gemm_w13_swiglu": 4.0 * S * d * inter,
        "gemm_w2": 2.0 * S * d * inter,
        # the per-rank calls of the schedule: every rank's launches of a step
        # together do the block's work
        "rank_gemm_qkv": 2.0 * S * d * (d + 2 * dkv),
        "rank_gemm_q": 2.0 * S * d * d,
        "rank_gemm_kv": 4.0 * S * d * dkv,
        "rank_gemm_oproj": 2.0 * S * d * d,
        "rank_gemm_w13_swiglu": 4.0 * S * d * inter,
        "rank_gemm_w2": 2.0 * S * d * inter,
        "rank_gemm_w13_recompute": 4.0 * S * d * inter,   # the backward's ring recomputes G, A|B
        "rank_gemm_dgrad_w2_swiglu": 2.0 * S * d * inter,
        "rank_gemm_dgrad_w13": 4.0 * S * d * inter,
        "rank_gemm_wgrad_w13": 4.0 * S * d * inter,
        "rank_gemm_wgrad_w2": 2.0 * S * d * inter,
        "rank_gemm_dgrad_wo": 2.0 * S * d * d,
        "rank_gemm_wgrad_wo": 2.0 * S * d * d,
        "rank_gemm_wgrad_q": 2.0 * S * d * d,
        "rank_gemm_wgrad_kv": 4.0 * S * d * dkv,
        "rank_gemm_dgrad_qkv": 2.0 * S * d * (d + 2 * dkv),
        "rank_attn_bwd": 5.0 * S * (S + 1) * d,
        "attn_fwd": 2.0 * S * (S + 1) * d,
        # backward: dgrad and wgrad of every projection, and the attention
        # backward's five causal products (S recomputed, dP, dV, dK, dQ)
        "gemm_dgrad_w2_swiglu": 2.0 * S * d * inter,
        "gemm_wgrad_w2": 2.0 * S * d * inter,
        "gemm_wgrad_w13": 4.0 * S * d * inter,
        # MLP tiling: the backward recomputes G and A|B (work beyond the model's flops)
        "gemm_w13_recompute": 4.0 * S * d * inter,
        "gemm_dgrad_w13": 4.0 * S * d * inter,
        "gemm_wgrad_wo": 2.0 * S * d * d,
        "gemm_dgrad_wo": 2.0 * S * d * d,
        "gemm_wgrad_qkv": 2.0 * S * d * (d + 2 * dkv),
        "gemm_dgrad_qkv": 2.0 * S * d * (d + 2 * dkv),
        "attn_bwd": 5.0 * S * (S + 1) * d,
    }
    return table.get(name)


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant kernel, from one ncu capture of `bench.py --workload <w>`; each entry
# holds the SHA-256 of the kernel's source file at capture time, and the figure
# is reported only while that source is unchanged (otherwise traffic is null).
MEASURED_TRAFFIC = {
    # (kernel, workload): (bytes per launch, source file, sha256 of the source);
    # first (cold) launch of the process, from the captures summarised under profiles/
    ("gemm_w13_swiglu", "fwd16k"): (
        944034816 + 348202240, "folded_tensor_sequence_zigzag_gb300/csrc/gemm_tc.cu",
        "e83ee7a870f45b96341ece6c71e6c262d62c017a8ea9d8649962054a2391ec7b"),
    ("attn_fwd", "fwd16k"): (
        422576384 + 114971648, "folded_tensor_sequence_zigzag_gb300/csrc/attn_fwd.cu",
        "e15ab810a491d18f59761817c11bd61ea0997429e80e87acca851d2c5e0afd5a"),
    ("attn_bwd", "fwdbwd8k"): (
        407518976 + 227177216, "folded_tensor_sequence_zigzag_gb300/csrc/attn_bwd.cu",
        "6153d18e49ffa1c13d3bd1855a0b850efe2e96017d7d90ce197a4972184c4fc6"),
    ("decode_attn", "decode16k"): (
        268713728 + 2905600, "folded_tensor_sequence_zigzag_gb300/csrc/decode.cu",
        "f18fb1543642fef5e3c46c60d884bcc4fec2def3a9b08aa0a04305815fe27910"),
    ("decode_attn", "decode16k_gqa8"): (
        67188224 + 7424, "folded_tensor_sequence_zigzag_gb300/csrc/decode.cu",
        "f18fb1543642fef5e3c46c60d884bcc4fec2def3a9b08aa0a04305815fe27910"),
}


def measured_traffic(kernel, workload):
    import hashlib
    ent = MEASURED_TRAFFIC.get((kernel, workload))
    if ent is None:
        return None
    nbytes, src, sha = ent
    try:
        with open(os.path.join(ROOT, src), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha:
                return None
    except OSError:
        return None
    return nbytes


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.idx = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
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
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle legs

_SAMPLE_CACHE = {}

# rows (mirrored pairs per sample: 2 * CPU_PAIRS tokens) of one oracle sample
# of a forward workload, shared by the GPU arm's cpu_baseline and every step
# of the reference arm so that the two legs time the same thing
CPU_PAIRS = 512
# causal prefix of a training-step sample (the oracle's backward is unsharded)
CPU_PREFIX_BWD = 512
# rows of an MLP-only sample (the MLP is row-local: every row costs the same)
CPU_ROWS_MLP = 2048


def _oracle_inputs(S, d, H, inter, kind, variant):
    import torch
    from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs
    variant = variant or {}
    key = (S, d, H, inter, kind, tuple(sorted(variant.items())))
    if key not in _SAMPLE_CACHE:
        _SAMPLE_CACHE.clear()
        shape = BlockShape(S=S, d=d, H=H, inter=inter, D=1, Hkv=variant.get("Hkv", 0))
        inp = make_block_inputs(shape, torch.bfloat16, seed=0, with_dy=(kind == "fwdbwd"),
                                mlp_only=(kind == "mlp"))
        if variant.get("rope_base"):
            inp["rope_base"] = variant["rope_base"]
        _SAMPLE_CACHE[key] = {"inp": inp}
    return _SAMPLE_CACHE[key]


def cpu_sample(S, D, d, H, inter, kind, variant, r=0):
    """Time the float64 oracle on one bounded sample of the workload.

    Returns (tokens, seconds, equiv_seconds, exact, description): the sample
    took `seconds`; `equiv_seconds` is the time `tokens` of the workload's
    tokens take at that rate, so tokens / equiv_seconds is the oracle's
    throughput on the workload.  `exact`: the sampled tokens carry exactly the
    workload's average work per token (equiv_seconds == seconds); otherwise
    equiv_seconds is an estimate scaled by the algorithmic flop ratio.

    Forward: virtual rank r's step of the TSP schedule on CPU_PAIRS mirrored
    row pairs of its zigzag rows -- its own Q/K/V projection shard by shard,
    causal attention against the gathered K/V of the whole sequence, the W_O
    shard loop and the MLP ring.  Every mirrored pair attends S + 1 keys, so
    the sample's work per token is the block's average exactly.  The gathered
    K/V (what the other ranks' projections and the all-gather deliver) is
    prepared once, untimed.
    MLP only: the oracle's MLP on the first CPU_ROWS_MLP rows (row-local).
    Forward + backward: the oracle's (unsharded) backward on a causal prefix
    of CPU_PREFIX_BWD tokens, scaled by the algorithmic flop ratio (an
    estimate, labelled as such).
    """
    import numpy as np
    import oracle.tsp_oracle as O
    variant = variant or {}
    H_kv = variant.get("Hkv", H)
    dkv = H_kv * (d // H)
    c = S // (2 * D)
    if kind == "mlp":
        ent = _oracle_inputs(CPU_ROWS_MLP, d, H, inter, kind, variant)
        inp = ent["inp"]
        t0 = time.perf_counter()
        O.mlp_fwd(inp["x"], inp, 1e-6, norm=False, residual=False)
        dt = time.perf_counter() - t0
        return CPU_ROWS_MLP, dt, dt, True, (f"oracle (numpy float64) MLP on {CPU_ROWS_MLP} rows "
                                        f"(row-local: every row carries the same work)")
    if kind == "fwdbwd":
        rows = CPU_PREFIX_BWD
        inp = _oracle_inputs(rows, d, H, inter, kind, variant)["inp"]
        t0 = time.perf_counter()
        O.block_bwd(inp["x"], inp, inp["dy"], H, 1e-6)
        dt = time.perf_counter() - t0
        scale = block_flops(S, d, inter, kind, dkv) / block_flops(rows, d, inter, kind, dkv)
        return rows, dt, dt * rows * scale / S, False, (
            f"oracle (numpy float64) training step on the first {rows} tokens, time scaled to "
            f"the workload by algorithmic flops x{scale:.1f} (an estimate)")
    ent = _oracle_inputs(S, d, H, inter, kind, variant)
    inp = ent["inp"]
    if "x64" not in ent:
        ent["x64"] = O.f64(inp["x"])
        ent["kv"] = O.gather_kv(inp["x"], inp, H, D, 1e-6)
    x64 = ent["x64"]
    K_all, V_all = ent["kv"]
    n = min(c, CPU_PAIRS)
    p = O.mirrored_rows(S, D, r, n)
    t0 = time.perf_counter()
    Q_r, _, _ = O.rank_project(x64[p], p, inp, H, D, 1e-6)
    O.rank_fwd(r, x64[p], p, Q_r, K_all, V_all, inp, H, D, 1e-6, c)
    dt = time.perf_counter() - t0
    return 2 * n, dt, dt, True, (
        f"oracle (numpy float64), virtual rank {r}'s step of the TSP schedule on {n} mirrored "
        f"row pairs of its zigzag rows ({2 * n} tokens: own Q/K/V projection by shards, causal "
        f"attention against the gathered K/V of all {S} tokens, W_O shard loop, MLP ring); each "
        f"pair attends S+1 keys, so the sample carries the block's average work per token; "
        f"gathered K/V prepared untimed")


def cpu_cores():
    return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.barrier()
            dist.destroy_process_group()
            return
    S, D, d, H, inter, kind = WORKLOADS[args.workload]
    L = LAYERS.get(args.workload, 1)
    if kind == "decode":
        return run_reference_decode(args, rank, world)
    var = VARIANTS.get(args.workload)
    # each step is one bounded sample (virtual rank = step mod D for the
    # forward workloads); ms_per_step is the sample's own time
    for i in range(args.warmup):
        cpu_sample(S, D, d, H, inter, kind, var, r=i % D)
    times, equiv, toks = [], [], 0
    desc, exact = "", True
    for i in range(args.steps):
        n_tok, dt, dt_eq, exact, desc = cpu_sample(S, D, d, H, inter, kind, var, r=i % D)
        times.append(dt)
        equiv.append(dt_eq * L)
        toks += n_tok
    if L > 1:
        desc += f"; x{L} layers (each layer its own weights, same work)"
    value = toks / sum(equiv)
    line = {
        "impl": "reference", "metric": "TSP-block tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(times) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload),
        "step": f"one bounded sample of the workload: {desc}",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc, "exact_work_per_token": exact},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def oracle_decode_sample(S_full, d, H, inter, variant, prompt_rows):
    """Time the oracle's decode of one token after a `prompt_rows` prompt.
    The oracle keeps no cache (it recomputes the prefix's K/V), so its cost
    grows with the prompt; the time is scaled to the workload's prompt by
    the row ratio.  Returns (seconds estimate, seconds measured, description)."""
    import torch
    import oracle.tsp_oracle as O
    from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs
    variant = variant or {}
    key = ("decode", prompt_rows, d, H, inter, tuple(sorted(variant.items())))
    if key not in _SAMPLE_CACHE:
        shape = BlockShape(S=prompt_rows + 1, d=d, H=H, inter=inter, D=1, Hkv=variant.get("Hkv", 0))
        _SAMPLE_CACHE.clear()
        _SAMPLE_CACHE[key] = make_block_inputs(shape, torch.bfloat16, seed=0)
        if variant.get("rope_base"):
            _SAMPLE_CACHE[key]["rope_base"] = variant["rope_base"]
    inp = _SAMPLE_CACHE[key]
    x = inp["x"]
    t0 = time.perf_counter()
    O.block_decode(x[:prompt_rows], [x[prompt_rows:prompt_rows + 1]], inp, H, 1e-6)
    dt = time.perf_counter() - t0
    scale = (S_full + 1) / (prompt_rows + 1)
    desc = (f"oracle (numpy float64) decoding one token after a {prompt_rows}-token prompt "
            f"(it recomputes the prefix K/V), scaled to the {S_full}-token prompt by x{scale:.1f}")
    return dt * scale, dt, desc


def run_reference_decode(args, rank, world):
    S, D, d, H, inter, kind = WORKLOADS[args.workload]
    rows = args.ref_rows or 1024
    var = VARIANTS.get(args.workload)
    for _ in range(args.warmup):
        oracle_decode_sample(S, d, H, inter, var, rows)
    times, desc = [], ""
    for _ in range(args.steps):
        est, _, desc = oracle_decode_sample(S, d, H, inter, var, rows)
        times.append(est)
    t = statistics.median(times) * DECODE_GEN / DECODE_T     # one step: DECODE_GEN tokens
    value = DECODE_GEN / t
    line = {
        "impl": "reference", "metric": "decode tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def workload_config(name):
    S, D, d, H, inter, kind = WORKLOADS[name]
    desc = {"fwd": "7B-shaped TSP block forward", "fwdbwd": "7B-shaped TSP block forward+backward",
            "mlp": "sharded SwiGLU MLP only (no norm, no residual)",
            "decode": f"7B-shaped TSP block decode, {DECODE_GEN} tokens generated one at a time "
                      f"after the prompt, against its zigzag KV cache"}[kind]
    L = LAYERS.get(name, 1)
    if L > 1:
        desc = f"{L}-layer stack of the {desc}"
    var = VARIANTS.get(name, {})
    extra = ""
    if "Hkv" in var:
        extra += f", grouped-query attention with {var['Hkv']} K/V heads"
    if var.get("rope_base"):
        extra += f", rotary embedding base {var['rope_base']:g}"
    if var.get("mlp_tile"):
        extra += f", MLP in sequence tiles of {var['mlp_tile']} rows (recomputed in the backward)"
    if var.get("by_rank"):
        extra += (", computed rank by rank by the TSP schedule (each virtual rank's per-rank "
                  "calls in turn; shard broadcast, K/V all-gather and MLP ring as device copies "
                  "on a copy stream)")
    return {"workload": f"{desc}, S={S}, D={D} zigzag virtual ranks, d_model={d}, "
                        f"{H} heads x {d // H}, SwiGLU inter={inter}, causal{extra}",
            "S": S, "D": D, "d_model": d, "heads": H, "kv_heads": var.get("Hkv", H),
            "rope_base": var.get("rope_base", 0.0), "inter": inter, "global_batch": 1,
            "seq_len": S, "parallelism": "replicas (one TSP-emulated block per GPU)",
            "l2": "working set larger than L2 (no flush needed)"}


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch
    import torch.distributed as dist
    from folded_tensor_sequence_zigzag_gb300 import build, tsp
    from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    tsp.load()

    S, D, d, H, inter, kind = WORKLOADS[args.workload]
    if kind == "decode":
        return run_gpu_decode(args, rank, world, local, dev)
    var = VARIANTS.get(args.workload, {})
    shape = BlockShape(S=S, d=d, H=H, inter=inter, D=D, Hkv=var.get("Hkv", 0))
    inp = make_block_inputs(shape, torch.bfloat16, seed=rank, with_dy=(kind == "fwdbwd"),
                            mlp_only=(kind == "mlp"))
    cfg = tsp.make_cfg(S, d, H, inter, D, torch.bfloat16, rope_base=var.get("rope_base", 0.0),
                       Hkv=var.get("Hkv", 0), mlp_tile=var.get("mlp_tile", 0))
    dkv = shape.dkv
    if kind == "mlp":
        inp.update({k: torch.zeros(1, dtype=torch.bfloat16) for k in ("wq", "wk", "wv", "wo")})
    W = tsp.BlockWeights.from_dict(inp, dev)
    L = LAYERS.get(args.workload, 1)
    Ws = [W]
    gen = torch.Generator(device=dev).manual_seed(1000 + rank)
    for _ in range(1, L):   # further layers drawn on the device, same distributions
        def rnd(*shp):
            return (torch.randn(*shp, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        Ws.append(tsp.BlockWeights(rnd(d, d), rnd(dkv, d), rnd(dkv, d), rnd(d, d), rnd(inter, d),
                                   rnd(inter, d), rnd(d, inter),
                                   torch.ones(d, dtype=torch.bfloat16, device=dev),
                                   torch.ones(d, dtype=torch.bfloat16, device=dev)))
    x = inp["x"].to(dev)
    xz = torch.empty_like(x)
    yz = torch.empty_like(x)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    saved = ws = wsb = dy = dyz = None
    if L > 1:
        if kind == "fwd":
            ws = torch.empty(tsp.stack_workspace_bytes(cfg, L, tsp.TSP_OP_BLOCK_FWD),
                             dtype=torch.uint8, device=dev)
        else:
            saved = torch.empty(tsp.stack_saved_bytes(cfg, L), dtype=torch.uint8, device=dev)
            ws = torch.empty(tsp.stack_workspace_bytes(cfg, L, tsp.TSP_OP_BLOCK_FWD),
                             dtype=torch.uint8, device=dev)
            wsb = torch.empty(tsp.stack_workspace_bytes(cfg, L, tsp.TSP_OP_BLOCK_BWD),
                              dtype=torch.uint8, device=dev)
            dy = inp["dy"].to(dev)
            dyz = torch.empty_like(dy)
            y = torch.empty(x.shape, dtype=torch.float32, device=dev)
    elif kind == "fwd":
        ws = torch.empty(tsp.workspace_bytes(cfg, tsp.TSP_OP_BLOCK_FWD), dtype=torch.uint8, device=dev)
    elif kind == "mlp":
        ws = torch.empty(tsp.workspace_bytes(cfg, tsp.TSP_OP_MLP_FWD), dtype=torch.uint8, device=dev)
    else:
        saved = torch.empty(tsp.saved_bytes(cfg), dtype=torch.uint8, device=dev)
        wsb = torch.empty(tsp.workspace_bytes(cfg, tsp.TSP_OP_BLOCK_BWD), dtype=torch.uint8, device=dev)
        dy = inp["dy"].to(dev)
        dyz = torch.empty_like(dy)
        y = torch.empty(x.shape, dtype=torch.float32, device=dev)  # dx (fp32) in global order

    # The block's weights in the fp16 operand type, converted once per weight
    # update (tsp_block_weights_prepare): for a forward (inference) workload
    # once before timing, as a deployment holds them; for a training step once
    # per step, inside it, shared by the forward and the backward.  The
    # workspaces above are sized for the calls that convert their own weights,
    # which is more than the prepared calls need, so they serve both.
    prep_mode = "per-step" if kind == "fwdbwd" else ("once" if kind == "fwd" else "none")
    sched = None
    if var.get("by_rank"):
        # packed shards once before timing (what the broadcast and the ring
        # carry); each rank's calls convert the shard they hold as it arrives
        from folded_tensor_sequence_zigzag_gb300 import schedule
        prep_mode = "shards"
        rows = S // D
        sched = (schedule.LocalComm(cfg, W, overlap=True),
                 schedule.GpuRankOps(cfg, W, {r: xz[r * rows:(r + 1) * rows] for r in range(D)}))
        if kind == "fwdbwd":
            for r in range(D):   # each rank's dy rows: views of the step's permuted dy
                sched[1].set_dy(r, dyz[r * rows:(r + 1) * rows])
            dxz = torch.empty(x.shape, dtype=torch.float32, device=dev)
    preps = None
    if prep_mode != "none":
        preps = [tsp.prepare_weights(cfg, Wl) for Wl in Ws]
    if prep_mode == "per-step" and L == 1:
        ws = torch.empty(tsp.workspace_bytes(cfg, tsp.TSP_OP_BLOCK_FWD_TRAIN | tsp.TSP_OP_PREPARED),
                         dtype=torch.uint8, device=dev)

    def step(xin, yout=None, convert_per_call=False):
        yout = y if yout is None else yout
        tsp.zigzag_permute(xin, D, out=xz)
        pp = None if convert_per_call else preps
        if sched is not None:
            comm, ops = sched
            schedule.forward(comm, ops, D)
            if kind == "fwdbwd":
                tsp.zigzag_permute(dy, D, out=dyz)
                dx = schedule.backward(comm, ops, D)
                for r in range(D):
                    dxz[r * rows:(r + 1) * rows].copy_(dx[r])
                tsp.zigzag_permute(dxz, D, inverse=True, out=yout)
                return yout
            for r in range(D):
                yz[r * rows:(r + 1) * rows].copy_(ops.output(r))
            tsp.zigzag_permute(yz, D, inverse=True, out=yout)
            return yout
        if prep_mode == "per-step":
            for Wl, p in zip(Ws, preps):
                tsp.prepare_weights(cfg, Wl, out=p)
        if L > 1 and kind == "fwd":
            tsp.stack_fwd(cfg, xz, Ws, out=yz, ws=ws, preps=pp)
            tsp.zigzag_permute(yz, D, inverse=True, out=yout)
            return yout
        if L > 1:
            tsp.stack_fwd(cfg, xz, Ws, saved=saved, out=yz, ws=ws, preps=preps)
            tsp.zigzag_permute(dy, D, out=dyz)
            dx, _ = tsp.stack_bwd(cfg, dyz, saved, Ws, ws=wsb, preps=preps)
            tsp.zigzag_permute(dx, D, inverse=True, out=yout)
            return yout
        if kind == "fwd":
            tsp.block_fwd(cfg, xz, W, out=yz, ws=ws, prep=pp[0] if pp else None)
            tsp.zigzag_permute(yz, D, inverse=True, out=yout)
            return yout
        if kind == "mlp":
            tsp.gated_mlp_fwd(cfg, xz, W, norm=False, residual=False, out=yz, ws=ws)
            tsp.zigzag_permute(yz, D, inverse=True, out=yout)
            return yout
        tsp.block_fwd(cfg, xz, W, saved=saved, out=yz, ws=ws, prep=preps[0])
        tsp.zigzag_permute(dy, D, out=dyz)
        g = tsp.block_bwd(cfg, xz, dyz, saved, W, ws=wsb, prep=preps[0])
        tsp.zigzag_permute(g["dx"], D, inverse=True, out=yout)
        return yout

    # ---- warm-up
    for _ in range(max(args.warmup, 0)):
        step(x)
    torch.cuda.synchronize(dev)
    if tsp.device_status() != tsp.TSP_OK:
        raise RuntimeError("device status not OK after warm-up")

    # The rank-by-rank step is ~500 small launches: it is captured once as a
    # CUDA graph and replayed, so the timed region carries no host launch
    # overhead, and the per-kernel times come from an eager pass of the same
    # steps right after it (events cannot sit inside a replayed graph).
    graph = None
    if sched is not None:
        graph = torch.cuda.CUDAGraph()
        n_cap = tsp.launch_count()
        with torch.cuda.graph(graph):
            step(x)
        graph_kernels = tsp.launch_count() - n_cap
        torch.cuda.synchronize(dev)

    # ---- device-timed region: inputs resident in HBM; per-kernel CUDA events
    # are recorded on the launch stream inside the same region (eager steps)
    n0 = tsp.launch_count()
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    clocks.start()
    tsp.profile_enable(graph is None)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(x)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    launches = graph_kernels * args.steps if graph is not None else tsp.launch_count() - n0
    t_eager = None
    if graph is not None:
        tsp.profile_enable(True)
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        for _ in range(args.steps):
            step(x)
        q1.record(stream)
        torch.cuda.synchronize(dev)
        t_eager = q0.elapsed_time(q1) / 1e3 / args.steps
    prof = tsp.profile_report()
    tsp.profile_enable(False)
    t_dev = ev0.elapsed_time(ev1) / 1e3 / args.steps
    t_dev = reduce_max(t_dev, world, dev if world > 1 else None)

    # ---- the same step with the weights converted inside every call (the
    # calls without prepared copies), for comparison
    conv = None
    if prep_mode == "once":
        for _ in range(2):
            step(x, convert_per_call=True)
        torch.cuda.synchronize(dev)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(args.steps):
            step(x, convert_per_call=True)
        c1.record(stream)
        torch.cuda.synchronize(dev)
        t_conv = reduce_max(c0.elapsed_time(c1) / 1e3 / args.steps, world, dev if world > 1 else None)
        conv = {"value": world * S / t_conv, "unit": "tokens/s", "ms_per_step": t_conv * 1e3}

    # ---- end to end through the public API with host buffers: every step
    # uploads its input from pinned host memory and reads its result back.
    # Uploads and read-backs run on streams of their own with double-buffered
    # device copies, so step i+1's upload and step i-1's read-back overlap step
    # i's compute; the timed region runs from the first upload to the last
    # read-back.
    x_host = inp["x"].pin_memory()
    y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    y_dev = [torch.empty_like(y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(s_in)
    # the captured step reads x and writes y: every step uploads into x, replays
    # the graph and reads y back, in order on the launch stream
    for i in range(args.steps if graph is not None else 0):
        with torch.cuda.stream(stream):
            if i == 0:
                stream.wait_stream(s_in)
            x.copy_(x_host, non_blocking=True)
            graph.replay()
            y_host[0].copy_(y, non_blocking=True)
        if i == args.steps - 1:
            s_out.wait_stream(stream)
    for i in range(args.steps if graph is None else 0):
        p = i & 1
        if i >= 2:
            s_in.wait_event(comp_done[p])      # x_dev[p] no longer read
        with torch.cuda.stream(s_in):
            x_dev[p].copy_(x_host, non_blocking=True)
        h2d_done[p].record(s_in)
        stream.wait_event(h2d_done[p])
        if i >= 2:
            stream.wait_event(d2h_done[p])     # y_dev[p] read back
        with torch.cuda.stream(stream):
            step(x_dev[p], y_dev[p])
        comp_done[p].record(stream)
        s_out.wait_event(comp_done[p])
        with torch.cuda.stream(s_out):
            y_host[p].copy_(y_dev[p], non_blocking=True)
        d2h_done[p].record(s_out)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    t_e2e = e0.elapsed_time(e1) / 1e3 / args.steps
    t_e2e = reduce_max(t_e2e, world, dev if world > 1 else None)
    if tsp.device_status() != tsp.TSP_OK:
        raise RuntimeError("device status not OK after the timed region")

    # ---- roofline of the dominant kernel
    peaks, peak_src = measured_peaks()
    kernel_rows = []
    for name, (k, ms) in prof.items():
        kernel_rows.append((ms, name, k))
    kernel_rows.sort(reverse=True)
    top_name = kernel_rows[0][1] if kernel_rows else None
    roof = None
    per_kernel = {}
    for ms, name, k in kernel_rows:
        per_launch_ms = ms / max(k, 1)
        f = gemm_flops(name, S, d, inter, dkv)   # one layer-step's flops over all its launches
        if (f is not None and sched is not None and kind == "fwdbwd" and
                name in ("attn_fwd", "rank_gemm_qkv", "rank_gemm_q", "rank_gemm_kv")):
            f *= 2   # rank by rank the backward recomputes each rank's Q, K|V, O and LSE
        entry = {"launches": k, "ms_per_launch": per_launch_ms}
        if f is not None and kind != "mlp":
            entry["tflops"] = f * L * args.steps / (ms / 1e3) / 1e12
        elif name.startswith("gemm_w13") and kind == "mlp":
            entry["tflops"] = 4.0 * S * d * inter / (per_launch_ms / 1e3) / 1e12
        elif name.startswith("gemm_w2") and kind == "mlp":
            entry["tflops"] = 2.0 * S * d * inter / (per_launch_ms / 1e3) / 1e12
        per_kernel[name] = entry
    # the dominant tensor-core kernel of the step
    dom = None
    for ms, name, k in kernel_rows:
        if "tflops" in per_kernel[name]:
            dom = name
            break
    # the burst peak (cuBLAS timed alone) for a timed region shorter than a
    # second, the sustained one (seconds-long loop under the power cap) beyond
    timed_s = t_dev * args.steps
    sustained = timed_s >= 1.0
    peak = peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops", peaks.get("bf16_tflops"))
    peak_label = (f"{peak_src} bf16 {'sustained' if sustained else 'burst'} (MEASURED_PEAKS.json; "
                  f"timed region {timed_s:.2f} s {'>=' if sustained else '<'} 1 s)")
    # the tensor core's own rate at the clock the run saw: 8192 dense fp16/bf16
    # flop per clock per SM (M=128, N=128, K=16 in 64 cycles) x SMs x the
    # median sampled SM clock
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    clock_peak = (n_sm * 8192.0 * clk["sm_mhz"] * 1e6 / 1e12) if clk.get("sm_mhz") else None
    if dom is not None:
        ach = per_kernel[dom]["tflops"]
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "peak_source": peak_label,
                "traffic": measured_traffic(dom, args.workload),
                "clock_peak": clock_peak,
                "frac_of_clock_peak": ach / clock_peak if clock_peak else None,
                "clock_peak_source": f"{n_sm} SMs x 8192 flop/clk x median sampled SM clock",
                "frac_of_nominal": ach / NOMINAL_BF16_TFLOPS,
                "nominal_source": "GB300 rated dense bf16, 2.25 PFLOP/s"}
    flops = block_flops(S, d, inter, kind, dkv) * L
    value = world * S / t_dev
    tflops = world * flops / t_dev / 1e12
    line = {
        "metric": "TSP-block tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_dev * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (x~N(0,1), weights~N(0,0.02), gains 1)",
        "config": workload_config(args.workload),
        "tflops": tflops, "tflops_per_gpu": tflops / world,
        "frac_of_peak": (tflops / world) / peak,
        "peak_tflops": peak, "peak_source": peak_label,
        "frac_of_nominal": (tflops / world) / NOMINAL_BF16_TFLOPS,
        "timed_region_s": timed_s,
        "e2e": {"value": world * S / t_e2e, "unit": "tokens/s",
                "h2d_bytes_per_step": int(x.numel() * x.element_size()),
                "d2h_bytes_per_step": int(y.numel() * y.element_size())},
        "gpu_launches": int(launches),
        "launches_per_step": launches / args.steps,
        "weights": {"once": "bf16 weights converted to the fp16 tensor-core operand copies once, "
                            "before the timed region (tsp_block_weights_prepare), as a deployment "
                            "holds them",
                    "per-step": "bf16 weights converted to the fp16 operand copies once per step, "
                                "inside the timed region, shared by the forward and the backward",
                    "none": "the MLP call converts its weights inside every call",
                    "shards": "bf16 weights packed into the schedule's shards once, before the "
                              "timed region (tsp_pack_attn_shards, tsp_pack_mlp_shards); each "
                              "rank's calls convert the shard they hold to fp16 as it "
                              "arrives"}[prep_mode],
        "with_weight_conversion_per_call": conv,
        "timed_as": ("CUDA graph of one step, replayed; kernels and eager_ms_per_step from an "
                     "eager pass of the same steps with per-kernel CUDA events"
                     if graph is not None else
                     "eager steps with per-kernel CUDA events on the launch stream"),
        "eager_ms_per_step": t_eager * 1e3 if t_eager is not None else None,
        "kernels": per_kernel,
        "roofline": roof,
        "clocks": clk,
        "memory": {
            "layers": L, "device_peak_gb": torch.cuda.max_memory_allocated(dev) / 1e9,
            # bytes one rank would hold for this many layers (the fold against the
            # layouts the pages compare), from the kernels' own buffer plan
            "per_rank_gb": {nm: tsp.rank_memory(cfg, L, kind == "fwdbwd", sch)["total"] / 1e9
                            for nm, sch in (("tsp", tsp.TSP_MEM_TSP), ("dp", tsp.TSP_MEM_DP),
                                            ("tp", tsp.TSP_MEM_TP), ("sp", tsp.TSP_MEM_SP),
                                            ("tp_sp_on_D2_devices", tsp.TSP_MEM_TP_SP))}},
    }
    if rank == 0 and not args.no_cpu_baseline:
        n_tok, dt, dt_eq, exact, desc = cpu_sample(S, D, d, H, inter, kind, var, r=0)
        if L > 1:
            desc += f"; x{L} layers (each layer its own weights, same work)"
        line["cpu_baseline"] = {"value": n_tok / (dt_eq * L), "unit": "tokens/s", "cores": cpu_cores(),
                                "kind": "oracle", "sample": desc, "sample_seconds": dt,
                                "exact_work_per_token": exact}
    if rank == 0 and args.cpu_full:
        # the oracle's unsharded block forward over the whole workload, once
        # (minutes of CPU time: a check of the bounded sample above, not part
        # of the default run)
        import oracle.tsp_oracle as O
        ent = _oracle_inputs(S, d, H, inter, kind, var)
        t0 = time.perf_counter()
        if kind == "fwd":
            O.block_fwd(ent["inp"]["x"], ent["inp"], H, 1e-6)
        elif kind == "mlp":
            O.mlp_fwd(ent["inp"]["x"], ent["inp"], 1e-6, norm=False, residual=False)
        else:
            O.block_bwd(ent["inp"]["x"], ent["inp"], ent["inp"]["dy"], H, 1e-6)
        dt = time.perf_counter() - t0
        line["cpu_full"] = {"value": S / dt, "unit": "tokens/s", "seconds": dt,
                            "cores": cpu_cores(), "kind": "oracle",
                            "what": f"oracle (numpy float64), whole workload ({kind}), one layer"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_gpu_decode(args, rank, world, local, dev):
    """A step generates DECODE_GEN tokens after a prefilled prompt, one
    tsp_block_decode call of DECODE_T tokens at a time (positions S, S+1, ...).
    The prompt runs once through tsp_block_prefill, untimed; every step starts
    again from the prompt (the cache's decoded rows are overwritten), so all
    steps do the same work."""
    import torch
    import torch.distributed as dist
    from folded_tensor_sequence_zigzag_gb300 import tsp
    from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs

    S, D, d, H, inter, kind = WORKLOADS[args.workload]
    var = VARIANTS.get(args.workload, {})
    T, n_gen = DECODE_T, DECODE_GEN
    calls = n_gen // T
    shape = BlockShape(S=S + n_gen, d=d, H=H, inter=inter, D=D, Hkv=var.get("Hkv", 0))
    inp = make_block_inputs(shape, torch.bfloat16, seed=rank)
    cfg = tsp.make_cfg(S, d, H, inter, D, torch.bfloat16, rope_base=var.get("rope_base", 0.0),
                       Hkv=var.get("Hkv", 0))
    dkv = shape.dkv
    W = tsp.BlockWeights.from_dict(inp, dev)
    cache = tsp.KVCache(cfg, S + n_gen, dev)
    stream = torch.cuda.current_stream(dev)
    xs_host = inp["x"][S:].contiguous()          # the generated tokens' inputs, position order
    xs = xs_host.to(dev)
    ys = torch.empty_like(xs)
    ws = torch.empty(tsp.decode_workspace_bytes(cfg, T, cache.rows_cap), dtype=torch.uint8,
                     device=dev)
    ws_pre = torch.empty(tsp.workspace_bytes(cfg, tsp.TSP_OP_BLOCK_FWD), dtype=torch.uint8,
                         device=dev)
    xz = tsp.zigzag_permute(inp["x"][:S].to(dev), D)
    tsp.block_prefill(cfg, xz, W, cache, ws=ws_pre)
    del ws_pre, xz
    xv = [xs[i * T:(i + 1) * T] for i in range(calls)]
    yv = [ys[i * T:(i + 1) * T] for i in range(calls)]

    def step(x_in=None, y_out=None):
        xin = xv if x_in is None else [x_in[i * T:(i + 1) * T] for i in range(calls)]
        yout = yv if y_out is None else [y_out[i * T:(i + 1) * T] for i in range(calls)]
        cache.n = S
        for i in range(calls):
            tsp.block_decode(cfg, xin[i], W, cache, out=yout[i], ws=ws)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    if tsp.device_status() != tsp.TSP_OK:
        raise RuntimeError("device status not OK after warm-up")

    # A step's DECODE_GEN calls always run at the same positions, so the step
    # is captured once as a CUDA graph and replayed: the timed region has no
    # host launch overhead between the ~2000 small kernels of a step.
    graph = torch.cuda.CUDAGraph()
    n_cap = tsp.launch_count()
    with torch.cuda.graph(graph):
        step()
    graph_kernels = tsp.launch_count() - n_cap
    torch.cuda.synchronize(dev)
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    launches = graph_kernels * args.steps
    t_dev = reduce_max(ev0.elapsed_time(ev1) / 1e3 / args.steps, world, dev if world > 1 else None)
    n_rows_mid = S + (n_gen + 1) / 2           # cached rows an attention call reads, on average

    # per-kernel durations: the same steps once more, eagerly, with CUDA events
    # around every kernel on the launch stream (events cannot sit inside the
    # replayed graph), and the eager step time beside them
    tsp.profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    prof = tsp.profile_report()
    tsp.profile_enable(False)
    t_eager = e0.elapsed_time(e1) / 1e3 / args.steps

    # end to end through the public API: every step uploads its tokens' inputs
    # from pinned host memory into the buffer the graph reads, replays the
    # step, and reads the outputs back
    x_host = xs_host.pin_memory()
    y_host = torch.empty(ys.shape, dtype=ys.dtype).pin_memory()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        xs.copy_(x_host, non_blocking=True)
        graph.replay()
        y_host.copy_(ys, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_e2e = reduce_max(e0.elapsed_time(e1) / 1e3 / args.steps, world, dev if world > 1 else None)
    if tsp.device_status() != tsp.TSP_OK:
        raise RuntimeError("device status not OK after the timed region")

    peaks, peak_src = measured_peaks()
    hbm = peaks.get("hbm_gbs")
    per_kernel = {}
    for name, (k, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
        per_launch_ms = ms / max(k, 1)
        entry = {"launches": k, "ms_per_launch": per_launch_ms}
        b = decode_bytes(name, d, inter, dkv, n_rows_mid)
        if b is not None:
            entry["gbs"] = b / (per_launch_ms / 1e3) / 1e9
        per_kernel[name] = entry
    dom = next((n for n in per_kernel if "gbs" in per_kernel[n]), None)
    roof = None
    if dom is not None:
        ach = per_kernel[dom]["gbs"]
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "peak_source": f"{peak_src} HBM copy bandwidth (MEASURED_PEAKS.json)",
                "traffic": measured_traffic(dom, args.workload)}
    call_bytes = sum(decode_bytes(n, d, inter, dkv, n_rows_mid) for n in
                     ("gemv_qkv", "gemv_oproj", "gemv_w13_swiglu", "gemv_w2", "decode_attn"))
    line = {
        "metric": "decode tokens/s", "value": world * n_gen / t_dev, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_dev * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (x~N(0,1), weights~N(0,0.02), gains 1)",
        "config": dict(workload_config(args.workload), tokens_per_call=T, tokens_per_step=n_gen,
                       l2="working set (weights + KV cache) larger than L2 (no flush needed)"),
        "hbm_bytes_per_token": call_bytes / T,
        "hbm_gbs_per_step": call_bytes * calls / t_dev / 1e9,
        "frac_of_hbm_peak": call_bytes * calls / t_dev / 1e9 / hbm,
        "e2e": {"value": world * n_gen / t_e2e, "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_host.numel() * 2),
                "d2h_bytes_per_step": int(y_host.numel() * 2)},
        "gpu_launches": int(launches),
        "launches_per_step": launches / args.steps,
        "timed_as": "CUDA graph of one step, replayed; kernels and eager_ms_per_step from an "
                    "eager pass of the same steps with per-kernel CUDA events",
        "eager_ms_per_step": t_eager * 1e3,
        "kernels": per_kernel,
        "roofline": roof,
        "clocks": clk,
        "memory": {"device_peak_gb": torch.cuda.max_memory_allocated(dev) / 1e9,
                   "kv_cache_gb": tsp.kv_cache_bytes(cfg, cache.rows_cap) / 1e9},
    }
    if rank == 0 and not args.no_cpu_baseline:
        rows = args.ref_rows or 1024
        est, dt, desc = oracle_decode_sample(S, d, H, inter, var, rows)
        line["cpu_baseline"] = {"value": T / est, "unit": "tokens/s", "cores": cpu_cores(),
                                "kind": "oracle", "sample": desc, "sample_seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--ref-rows", type=int, default=0, help="prompt rows of the decode sample")
    ap.add_argument("--cpu-full", action="store_true",
                    help="also time the oracle once on the whole workload (minutes)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
