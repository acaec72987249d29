"""Host-side logic of bench.py: flop counts, max-over-ranks reduction across
two gloo ranks, and the CPU reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_flop_counts():
    S, d, I = 16384, 4096, 11008
    assert bench.block_flops(S, d, I, "fwd") == 8 * S * d * d + 6 * S * d * I + 2 * S * (S + 1) * d
    assert abs(bench.block_flops(S, d, I, "fwd") - 8.83e12) / 8.83e12 < 1e-2
    assert bench.block_flops(S, d, I, "fwdbwd") == 3 * bench.block_flops(S, d, I, "fwd")
    assert bench.block_flops(S, d, I, "mlp") == 6 * S * d * I


def test_kernel_flop_table_adds_up():
    """The per-kernel table covers the step: forward kernels sum to the block's
    forward flops, backward GEMMs to twice the forward projections."""
    S, d, I = 8192, 4096, 11008
    fwd = ["gemm_qkv", "gemm_oproj", "gemm_w13_swiglu", "gemm_w2", "attn_fwd"]
    assert sum(bench.gemm_flops(k, S, d, I) for k in fwd) == bench.block_flops(S, d, I, "fwd")
    bwd_gemms = ["gemm_dgrad_w2_swiglu", "gemm_wgrad_w2", "gemm_wgrad_w13", "gemm_dgrad_w13",
                 "gemm_wgrad_wo", "gemm_dgrad_wo", "gemm_wgrad_qkv", "gemm_dgrad_qkv"]
    proj = sum(bench.gemm_flops(k, S, d, I) for k in fwd[:4])
    assert sum(bench.gemm_flops(k, S, d, I) for k in bwd_gemms) == 2 * proj
    assert bench.gemm_flops("attn_bwd", S, d, I) == 2.5 * bench.gemm_flops("attn_fwd", S, d, I)


def test_grouped_kv_flops():
    """8 K/V heads of 128 (dkv = 1024): the K and V projections shrink by
    d/dkv, attention does not; the kernel table still adds up."""
    S, d, I, dkv = 8192, 4096, 11008, 1024
    full = bench.block_flops(S, d, I, "fwd")
    assert bench.block_flops(S, d, I, "fwd", dkv) == full - 4 * S * d * (d - dkv)
    fwd = ["gemm_q", "gemm_kv", "gemm_oproj", "gemm_w13_swiglu", "gemm_w2", "attn_fwd"]
    assert sum(bench.gemm_flops(k, S, d, I, dkv) for k in fwd) == bench.block_flops(S, d, I, "fwd", dkv)
    assert bench.gemm_flops("gemm_q", S, d, I, dkv) + bench.gemm_flops("gemm_kv", S, d, I, dkv) == \
        bench.gemm_flops("gemm_qkv", S, d, I, dkv)
    bwd_gemms = ["gemm_dgrad_w2_swiglu", "gemm_wgrad_w2", "gemm_wgrad_w13", "gemm_dgrad_w13",
                 "gemm_wgrad_wo", "gemm_dgrad_wo", "gemm_wgrad_q", "gemm_wgrad_kv", "gemm_dgrad_qkv"]
    proj = sum(bench.gemm_flops(k, S, d, I, dkv) for k in fwd[:5])
    assert sum(bench.gemm_flops(k, S, d, I, dkv) for k in bwd_gemms) == 2 * proj
    cfg = bench.workload_config("fwd16k_gqa8")
    assert cfg["kv_heads"] == 8 and cfg["rope_base"] > 0


def test_rank_schedule_flops_cover_its_launches():
    """The rank-by-rank workload: every per-rank GEMM launch name the library
    labels has a flop count, and the forward ones (one Q|K|V GEMM, or Q and
    K|V apart) add up, with the attention, to the block's forward flops."""
    import re
    src = open(os.path.join(ROOT, "folded_tensor_sequence_zigzag_gb300", "csrc", "rank.cu")).read()
    names = set(re.findall(r'name = "(rank_gemm_\w+)"', src))
    assert names, "no rank GEMM labels found"
    S, d, I = 16384, 4096, 11008
    for n in names:
        assert bench.gemm_flops(n, S, d, I) is not None, n
    fused = ["rank_gemm_qkv", "rank_gemm_oproj", "rank_gemm_w13_swiglu", "rank_gemm_w2", "attn_fwd"]
    apart = ["rank_gemm_q", "rank_gemm_kv"] + fused[1:]
    for ks in (fused, apart):
        assert sum(bench.gemm_flops(k, S, d, I) for k in ks) == bench.block_flops(S, d, I, "fwd")
    bwd = ["rank_gemm_dgrad_w2_swiglu", "rank_gemm_wgrad_w2", "rank_gemm_dgrad_w13",
           "rank_gemm_wgrad_w13", "rank_gemm_dgrad_wo", "rank_gemm_wgrad_wo", "rank_gemm_wgrad_q",
           "rank_gemm_wgrad_kv", "rank_gemm_dgrad_qkv"]
    proj = sum(bench.gemm_flops(k, S, d, I) for k in fused[:4])
    assert sum(bench.gemm_flops(k, S, d, I) for k in bwd) == 2 * proj
    S_, D, d_, H, I_, kind = bench.WORKLOADS["fwd16k_by_rank"]
    assert kind == "fwd" and bench.VARIANTS["fwd16k_by_rank"].get("by_rank")
    assert "rank by rank" in bench.workload_config("fwd16k_by_rank")["workload"]


def test_traffic_figure_tracks_its_source(tmp_path, monkeypatch):
    """A stored ncu traffic figure is reported only while the kernel source
    it was taken on is unchanged."""
    import hashlib
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    sha = hashlib.sha256(b"kernel v1").hexdigest()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "MEASURED_TRAFFIC", {("k", "w"): (1234, "k.cu", sha)})
    assert bench.measured_traffic("k", "w") == 1234
    assert bench.measured_traffic("k", "other") is None
    src.write_text("kernel v2")
    assert bench.measured_traffic("k", "w") is None


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q.put((rank, bench.reduce_max(1.0 + rank * 2.5, world)))
    dist.destroy_process_group()


def test_reduce_max_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 1000
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get() for _ in range(2))
    assert got == {0: 3.5, 1: 3.5}


@pytest.mark.slow
def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "mlp16k", "--ref-rows", "32", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["unit"] == "tokens/s" and j["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["e2e"]["h2d_bytes_per_step"] == 0
