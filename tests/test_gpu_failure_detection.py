"""Failure detection on the GPU without a fault: a pipeline wait that can never
be satisfied (one stage of one CTA is deliberately left unfilled, through the
tsp_debug_skip_stage knob) must run out after TSP_WAIT_LIMIT_MS, be reported as
TSP_ERR_TIMEOUT by tsp_device_status, and leave the context usable: after the
status is cleared the same call gives the correct result again.  Runs in a
child process so the short wait limit applies to nothing else."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys, time
sys.path.insert(0, os.environ["TSP_ROOT"])
import torch
from folded_tensor_sequence_zigzag_gb300 import build, tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs
build.build()
shape = BlockShape(S=512, d=256, H=2, inter=384, D=4)
inp = make_block_inputs(shape, torch.bfloat16, seed=3, mlp_only=True)
inp.update({k: torch.zeros(1, dtype=torch.bfloat16) for k in ("wq", "wk", "wv", "wo")})
W = tsp.BlockWeights.from_dict(inp, "cuda")
cfg = tsp.make_cfg(512, 256, 2, 384, 4, torch.bfloat16)
h = tsp.zigzag_permute(inp["x"].cuda(), 4)
good = tsp.gated_mlp_fwd(cfg, h, W, norm=False, residual=False)
assert tsp.device_status(reset=True) == tsp.TSP_OK
tsp.debug_skip_stage(1)
t0 = time.time()
tsp.gated_mlp_fwd(cfg, h, W, norm=False, residual=False)
st = tsp.device_status(reset=True)
dt = time.time() - t0
assert st == tsp.TSP_ERR_TIMEOUT, st
assert dt < 30, dt
again = tsp.gated_mlp_fwd(cfg, h, W, norm=False, residual=False)
assert tsp.device_status(reset=True) == tsp.TSP_OK
assert torch.equal(again, good)
print("timeout detected in %.2f s; context usable" % dt)
"""


def test_bounded_wait_reports_timeout_and_context_survives():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    env = dict(os.environ, TSP_WAIT_LIMIT_MS="300", TSP_ROOT=ROOT)
    out = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True,
                         timeout=300, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "context usable" in out.stdout
