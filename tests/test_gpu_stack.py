"""GPU parity of the L-block stack (forward, inference and training, and
backward) through the C ABI against the float64 oracle's composition."""
import numpy as np
import pytest
import torch

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, TINY_FP32, make_block_inputs
from tests.helpers import BF16_MAX_REL_RMS, BF16_MEAN_REL, assert_f32_close, bf16_metrics, to64


def assert_stack_bf16_close(got, ref, boundaries, what=""):
    """The block's bf16 bounds, with the max-error bound widened by one bf16
    ulp of the largest reference value per stored layer boundary: a value
    within rounding distance of a bf16 tie can round to different neighbours
    on the GPU (fp32 before rounding) and in the oracle (fp64), and the
    residual path carries that one-ulp step to the output.  The mean relative
    bound is unchanged."""
    ref64 = to64(ref)
    rms = float(np.sqrt(np.mean(ref64 ** 2)))
    top = float(np.max(np.abs(ref64)))
    ulp = 2.0 ** (np.floor(np.log2(top)) - 7) if top > 0 else 0.0
    mx, mean = bf16_metrics(got, ref)
    bound = BF16_MAX_REL_RMS + boundaries * ulp / rms
    assert np.all(np.isfinite(to64(got))), f"{what}: non-finite output"
    assert mx <= bound and mean <= BF16_MEAN_REL, \
        f"{what}: max|err|/RMS={mx:.3e} (<= {bound:.3e}), mean rel={mean:.3e} (<= {BF16_MEAN_REL})"

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
        saved = torch.empty(tsp.stack_saved_bytes(cfg, L), dtype=torch.uint8, device=dev)
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
    # the stack stores activations (and the gradient between layers) in bf16
    yref = O.stack_fwd(x, layers, shape.H, shape.eps, store="bf16")
    assert_stack_bf16_close(got["y"].float().cpu(), yref, L - 1, "bf16 stack y")
    if training:
        dx_ref, g_ref = O.stack_bwd(x, layers, dy, shape.H, shape.eps, store="bf16")
        # dx crosses the L-1 forward boundaries and the L-1 gradient boundaries
        assert_stack_bf16_close(got["dx"].cpu(), dx_ref, 2 * (L - 1), "bf16 stack dx")
        for l in range(L):
            for k, v in g_ref[l].items():
                assert_stack_bf16_close(got["grads"][l][k].cpu(), v, 2 * (L - 1),
                                        f"bf16 stack layer {l} {k}")


def test_bf16_stack_with_every_variant_matches_oracle():
    """Two layers with grouped K/V heads, rotary embedding and the MLP in
    sequence tiles together: forward and every gradient."""
    L, base = 2, 10000.0
    shape = BlockShape(S=2048, d=512, H=4, inter=512, D=4, Hkv=2)
    x, dy, layers = _stack_inputs(shape, torch.bfloat16, L, seed=21)
    got = _run_stack(shape, torch.bfloat16, x, dy, layers, True, rope_base=base, mlp_tile=256)
    ref_layers = [dict(w, rope_base=base) for w in layers]
    yref = O.stack_fwd(x, ref_layers, shape.H, shape.eps, store="bf16")
    assert_stack_bf16_close(got["y"].float().cpu(), yref, L - 1, "variant stack y")
    dx_ref, g_ref = O.stack_bwd(x, ref_layers, dy, shape.H, shape.eps, store="bf16")
    assert_stack_bf16_close(got["dx"].cpu(), dx_ref, 2 * (L - 1), "variant stack dx")
    for l in range(L):
        for k, v in g_ref[l].items():
            assert got["grads"][l][k].shape == v.shape, (l, k)
            assert_stack_bf16_close(got["grads"][l][k].cpu(), v, 2 * (L - 1),
                                    f"variant stack layer {l} {k}")


def test_stack_rejects_bad_arguments():
    shape = TINY_FP32
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, torch.float32, shape.eps)
    assert tsp.load().tsp_stack_fwd(cfg, 0, None, None, None, None, None, None, 0, None) == \
        tsp.TSP_ERR_INVALID_ARG
    assert tsp.stack_workspace_bytes(cfg, 0, tsp.TSP_OP_BLOCK_FWD) == 0
    assert tsp.stack_saved_bytes(cfg, 0) == 0
