"""The checked build on the GPU: the same calls through libtsp_check.so (every
computed global index -- zigzag rows, shard and segment indices, tile rows,
cache rows, partial slots -- tested before its access, a failure recorded as
TSP_ERR_BOUNDS) run clean and give bit-identical outputs to the normal build,
whose arithmetic they share.  Each library runs in its own process (a process
holds one copy of the library); the outputs meet here."""
import os
import subprocess
import sys

import pytest
import torch

from folded_tensor_sequence_zigzag_gb300 import tsp

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, torch
sys.path.insert(0, sys.argv[3])
from folded_tensor_sequence_zigzag_gb300 import tsp, schedule
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs
tsp.load(sys.argv[1])
out = {}

def check(what):
    torch.cuda.synchronize()
    st = tsp.device_status()
    if st != tsp.TSP_OK:
        raise SystemExit(f"{what}: status {st} ({tsp.strerror(st)})")

def train(tag, shape, **kw):
    inp = make_block_inputs(shape, torch.bfloat16, seed=7, with_dy=True)
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, torch.bfloat16, shape.eps,
                       kw.get("rope", 0.0), shape.Hkv)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    xz = tsp.zigzag_permute(inp["x"].cuda(), shape.D)
    dyz = tsp.zigzag_permute(inp["dy"].cuda(), shape.D)
    saved = tsp.empty(tsp.saved_bytes(cfg), torch.uint8, "cuda")
    out[tag + "/y"] = tsp.block_fwd(cfg, xz, W, saved=saved).cpu()
    for k, v in tsp.block_bwd(cfg, xz, dyz, saved, W).items():
        out[tag + "/" + k] = v.cpu()
    check(tag)

# multi-head, ragged MLP shards (inter / D = 853.3), D = 3
train("mha", BlockShape(S=4608, d=1024, H=8, inter=2560, D=3))
# grouped K/V heads with rotary embedding
train("gqa", BlockShape(S=4096, d=1024, H=8, inter=2048, D=4, Hkv=2), rope=10000.0)

# prefill into the zigzag cache, then decode three tokens
shape = BlockShape(S=4096 + 3, d=1024, H=8, inter=2048, D=4, Hkv=2)
inp = make_block_inputs(shape, torch.bfloat16, seed=8)
S = 4096
cfg = tsp.make_cfg(S, 1024, 8, 2048, 4, torch.bfloat16, shape.eps, 10000.0, 2)
W = tsp.BlockWeights.from_dict(inp, "cuda")
cache = tsp.KVCache(cfg, S + 3, "cuda")
out["pre/y"] = tsp.block_prefill(cfg, tsp.zigzag_permute(inp["x"][:S].cuda(), 4), W, cache).cpu()
for t in range(3):
    out[f"dec/{t}"] = tsp.block_decode(cfg, inp["x"][S + t:S + t + 1].cuda(), W, cache).cpu()
check("decode")

# the forward schedule rank by rank (per-rank calls, packed shards)
shape = BlockShape(S=4096, d=1024, H=8, inter=2048, D=4)
inp = make_block_inputs(shape, torch.bfloat16, seed=9)
cfg = tsp.make_cfg(4096, 1024, 8, 2048, 4, torch.bfloat16, shape.eps)
W = tsp.BlockWeights.from_dict(inp, "cuda")
out["sched/y"] = schedule.block_fwd_by_schedule(cfg, tsp.zigzag_permute(inp["x"].cuda(), 4), W).cpu()
check("schedule")
# and its training step rank by rank (the one-rank attention backward among them)
inp = make_block_inputs(shape, torch.bfloat16, seed=10, with_dy=True)
W = tsp.BlockWeights.from_dict(inp, "cuda")
g = schedule.block_bwd_by_schedule(cfg, tsp.zigzag_permute(inp["x"].cuda(), 4),
                                   tsp.zigzag_permute(inp["dy"].cuda(), 4), W)
for k, v in g.items():
    out["sched_bwd/" + k] = v.cpu()
check("schedule backward")
torch.save(out, sys.argv[2])
"""


def _run(lib_path, out_path):
    r = subprocess.run([sys.executable, "-c", SCRIPT, lib_path, out_path, ROOT],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return torch.load(out_path)


def test_checked_build_runs_clean_and_matches(tmp_path):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    plain = _run(build.build(), str(tmp_path / "plain.pt"))
    checked = _run(build.build(check=True), str(tmp_path / "checked.pt"))
    assert plain.keys() == checked.keys()
    # the backward's dQ and the gain gradients sum with atomics in whatever
    # order the run takes, so those few are compared to 1e-4 of their scale
    atomic = ("/dx", "/dwq", "/dg_attn", "/dg_mlp")
    for k in plain:
        a, b = plain[k].float(), checked[k].float()
        if k.endswith(atomic):
            scale = float(a.abs().max()) or 1.0
            assert float((a - b).abs().max()) <= 1e-4 * scale, k
        else:
            assert torch.equal(plain[k], checked[k]), k
