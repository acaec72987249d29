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
