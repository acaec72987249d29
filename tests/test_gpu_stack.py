"""GPU parity of the L-block stack (forward, inference and training, and
backward) through the C ABI against the float64 oracle's composition."""
import numpy as np
import pytest
import torch

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, TINY_FP32, make_block_inputs
from tests.helpers import assert_bf16_close, assert_f32_close


pytestmark = pytest.mark.gpu

WEIGHTS = ("wq", "wk", "wv", "wo", "w1", "w3", "w2", "g_attn", "g_mlp")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    return tsp.load()


def _stack_inputs(shape, dtype, L, seed):
    inp = make_block_inputs(shape, dtype, seed=seed, with_dy=True)
    layers = []
    for l in range(L):
        w = make_block_inputs(shape, dtype, seed=seed + 100 + l)
        layers.append({k: w[k] for k in WEIGHTS})
    return inp["x"], inp["dy"], layers


def _run_stack(shape, dtype, x, dy, layers, training, rope_base=0.0, mlp_tile=0):
    dev = "cuda"
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, dtype, shape.eps,
                       rope_base, shape.Hkv, mlp_tile)
    Ws = [tsp.BlockWeights.from_dict(w, dev) for w in layers]
    xz = tsp.zigzag_permute(x.to(dev), shape.D)
    L = len(layers)
    saved = None
    if training:
        saved = tsp.empty(tsp.stack_saved_bytes(cfg, L), torch.uint8, dev)
    yz = tsp.stack_fwd(cfg, xz, Ws, saved=saved)
    y = tsp.zigzag_permute(yz, shape.D, inverse=True)
    out = {"y": y}
    if training:
        dyz = tsp.zigzag_permute(dy.to(dev), shape.D)
        dx, grads = tsp.stack_bwd(cfg, dyz, saved, Ws)
        out["dx"] = tsp.zigzag_permute(dx, shape.D, inverse=True)
        out["grads"] = grads
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    return out


@pytest.mark.parametrize("training", [False, True])
def test_tiny_fp32_stack_matches_oracle(training):
    L = 3
    x, dy, layers = _stack_inputs(TINY_FP32, torch.float32, L, seed=3)
    got = _run_stack(TINY_FP32, torch.float32, x, dy, layers, training)
    yref = O.stack_fwd(x, layers, TINY_FP32.H, TINY_FP32.eps)
    assert_f32_close(got["y"].cpu(), yref, "stack y")
    if training:
        dx_ref, g_ref = O.stack_bwd(x, layers, dy, TINY_FP32.H, TINY_FP32.eps)
        assert_f32_close(got["dx"].cpu(), dx_ref, "stack dx",
                         tol=1e-4 * max(1.0, float(np.max(np.abs(dx_ref)))))
        for l in range(L):
            for k, v in g_ref[l].items():
                scale = max(1.0, float(np.max(np.abs(v))))
                assert_f32_close(got["grads"][l][k].cpu(), v, f"layer {l} {k}", tol=1e-4 * scale)


@pytest.mark.parametrize("training", [False, True])
def test_bf16_stack_matches_oracle(training):
    L = 3
    shape = BlockShape(S=2048, d=256, H=2, inter=512, D=4)
    x, dy, layers = _stack_inputs(shape, torch.bfloat16, L, seed=9)
    got = _run_stack(shape, torch.bfloat16, x, dy, layers, training)
    # the residual stream between layers stays fp32, so the stack is held to
    # the block's own bf16 bounds (2e-2 * RMS max, 5e-3 mean relative)
    yref = O.stack_fwd(x, layers, shape.H, shape.eps)
    report = [("y",) + assert_bf16_close(got["y"].float().cpu(), yref, "bf16 stack y")]
    if training:
        dx_ref, g_ref = O.stack_bwd(x, layers, dy, shape.H, shape.eps)
        report.append(("dx",) + assert_bf16_close(got["dx"].cpu(), dx_ref, "bf16 stack dx"))
        for l in range(L):
            for k, v in g_ref[l].items():
                report.append((f"{l}.{k}",) + assert_bf16_close(got["grads"][l][k].cpu(), v,
                                                                 f"bf16 stack layer {l} {k}"))
    for name, mx, mean in report:
        print(f"bf16 stack {name}: max|err|/RMS {mx:.3e}  mean rel {mean:.3e}")


def test_bf16_stack_with_every_variant_matches_oracle():
    """Two layers with grouped K/V heads, rotary embedding and the MLP in
    sequence tiles together: forward and every gradient."""
    L, base = 2, 10000.0
    shape = BlockShape(S=2048, d=512, H=4, inter=512, D=4, Hkv=2)
    x, dy, layers = _stack_inputs(shape, torch.bfloat16, L, seed=21)
    got = _run_stack(shape, torch.bfloat16, x, dy, layers, True, rope_base=base, mlp_tile=256)
    ref_layers = [dict(w, rope_base=base) for w in layers]
    yref = O.stack_fwd(x, ref_layers, shape.H, shape.eps)
    assert_bf16_close(got["y"].float().cpu(), yref, "variant stack y")
    dx_ref, g_ref = O.stack_bwd(x, ref_layers, dy, shape.H, shape.eps)
    assert_bf16_close(got["dx"].cpu(), dx_ref, "variant stack dx")
    for l in range(L):
        for k, v in g_ref[l].items():
            assert got["grads"][l][k].shape == v.shape, (l, k)
            assert_bf16_close(got["grads"][l][k].cpu(), v, f"variant stack layer {l} {k}")


def test_stack_rejects_bad_arguments():
    shape = TINY_FP32
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, torch.float32, shape.eps)
    assert tsp.load().tsp_stack_fwd(cfg, 0, None, None, None, None, None, None, 0, None) == \
        tsp.TSP_ERR_INVALID_ARG
    assert tsp.stack_workspace_bytes(cfg, 0, tsp.TSP_OP_BLOCK_FWD) == 0
    assert tsp.stack_saved_bytes(cfg, 0) == 0
