"""GPU tests of the fp16 range check of the bf16 path.

The bf16 configuration holds its tensor-core operands in fp16 (weights,
normalised activations, Q/K/V, G, the upstream gradient ...).  A value fp16
cannot hold (|v| >= 65520, or not finite) must be reported as TSP_ERR_RANGE
through the device status word instead of silently becoming inf; values that
only the fp32 residual stream or the bf16 output carry must not be reported.
All inputs are made on the host; nothing here faults the GPU.
"""
import pytest
import torch

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs
from tests.helpers import assert_bf16_close

pytestmark = pytest.mark.gpu

SHAPE = BlockShape(S=1024, d=256, H=2, inter=512, D=2)


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    lib = tsp.load()
    tsp.device_status(reset=True)
    return lib


def _inputs(seed=3):
    return make_block_inputs(SHAPE, torch.bfloat16, seed=seed, with_dy=True)


def _cfg():
    return tsp.make_cfg(SHAPE.S, SHAPE.d, SHAPE.H, SHAPE.inter, SHAPE.D, torch.bfloat16)


def _forward(inp):
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    xz = tsp.zigzag_permute(inp["x"].cuda(), SHAPE.D)
    yz = tsp.block_fwd(_cfg(), xz, W)
    return tsp.zigzag_permute(yz, SHAPE.D, inverse=True), tsp.device_status(reset=True)


@pytest.mark.parametrize("what", ["w1", "wq", "w2", "g_attn"])
def test_out_of_fp16_range_operand_is_reported(what):
    inp = _inputs()
    if what == "g_attn":
        # the normalised activations are about x * g: a gain of 1e5 takes every
        # |x| > 0.66 beyond fp16 range (while the gain itself is a fine bf16)
        inp["g_attn"] = torch.full_like(inp["g_attn"], 1.0e5)
    else:
        inp[what] = inp[what].clone()
        inp[what][5, 7] = 1.0e5          # a bf16 weight fp16 cannot hold
    _, st = _forward(inp)
    assert st == tsp.TSP_ERR_RANGE, tsp.strerror(st)
    # the status was cleared and the context still works
    y, st = _forward(_inputs())
    assert st == tsp.TSP_OK
    assert torch.isfinite(y).all()


def test_large_residual_values_are_not_a_range_error():
    """x carries values far beyond fp16 range; only the fp32 residual stream
    and the bf16 output hold them (the normalised a stays near sqrt(d)), so
    nothing is reported and y still matches the oracle."""
    inp = _inputs(seed=4)
    x = inp["x"].float()
    x[::97, ::13] *= 3.0e5
    inp["x"] = x.to(torch.bfloat16)
    y, st = _forward(inp)
    assert st == tsp.TSP_OK, tsp.strerror(st)
    ref, _ = O.block_fwd(inp["x"], inp, SHAPE.H, SHAPE.eps)
    assert_bf16_close(y.cpu(), ref, "y with large residual values")


def test_out_of_range_upstream_gradient_is_reported():
    inp = _inputs(seed=5)
    cfg = _cfg()
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    xz = tsp.zigzag_permute(inp["x"].cuda(), SHAPE.D)
    saved = tsp.empty(tsp.saved_bytes(cfg), torch.uint8, "cuda")
    tsp.block_fwd(cfg, xz, W, saved=saved)
    assert tsp.device_status(reset=True) == tsp.TSP_OK
    dy = inp["dy"].clone()
    dy[3, 3] = 2.0e5
    dyz = tsp.zigzag_permute(dy.cuda(), SHAPE.D)
    tsp.block_bwd(cfg, xz, dyz, saved, W)
    assert tsp.device_status(reset=True) == tsp.TSP_ERR_RANGE


def test_decode_reports_out_of_range_projection():
    """The decode path streams the bf16 weights directly; a projection that
    overflows fp16 in its fp16 output is reported too."""
    inp = _inputs(seed=6)
    cfg = _cfg()
    W_ok = tsp.BlockWeights.from_dict(inp, "cuda")
    xz = tsp.zigzag_permute(inp["x"].cuda(), SHAPE.D)
    cache = tsp.KVCache(cfg, SHAPE.S + 1, "cuda")
    tsp.block_prefill(cfg, xz, W_ok, cache)
    assert tsp.device_status(reset=True) == tsp.TSP_OK
    bad = dict(inp)
    bad["wq"] = inp["wq"].float()
    bad["wq"][:, :] *= 1.0e7               # |q| far beyond fp16
    bad["wq"] = bad["wq"].to(torch.bfloat16)
    W_bad = tsp.BlockWeights.from_dict(bad, "cuda")
    x_new = torch.randn(1, SHAPE.d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    tsp.block_decode(cfg, x_new.cuda(), W_bad, cache)
    assert tsp.device_status(reset=True) == tsp.TSP_ERR_RANGE
