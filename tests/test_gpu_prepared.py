"""GPU tests of the weights-converted-once entry points: the block and the
stack with fp16 weight copies made by tsp_block_weights_prepare give what the
calls that convert the weights themselves give -- bit for bit wherever the
kernels are deterministic (the same kernels read the same fp16 copies).  Two
sums are order-dependent from run to run: the attention backward adds dQ over
key tiles with fp32 atomic reductions (so dQ and what is computed from it --
dW_Q, the attention input gradient, dx, dg_attn -- vary), and the RMSNorm
backward of widths that are not a multiple of 1024 adds the gain gradients in
shared memory with atomics (dg_mlp, dg_attn).  Those agree to fp32
reassociation instead."""
import ctypes

import pytest
import torch

from folded_tensor_sequence_zigzag_gb300 import tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs

pytestmark = pytest.mark.gpu

# outputs that go through an order-dependent fp32 sum (see above)
ATOMIC = ("dwq", "dx", "dg_attn", "dg_mlp")


def _same(a, b, k):
    if k in ATOMIC:
        err = float((a - b).abs().max())
        assert err <= 1e-4 * float(a.abs().max()), (k, err)
    else:
        assert torch.equal(a, b), k


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    return tsp.load()


@pytest.mark.parametrize("shape,tile,base", [
    (BlockShape(S=2048, d=256, H=2, inter=512, D=4), 0, 0.0),
    (BlockShape(S=4096, d=512, H=4, inter=768, D=8, Hkv=2), 256, 10000.0),
])
def test_block_prepared_equals_per_call_conversion(shape, tile, base):
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, torch.bfloat16, shape.eps,
                       base, shape.Hkv, tile)
    inp = make_block_inputs(shape, torch.bfloat16, seed=17, with_dy=True)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    prep = tsp.prepare_weights(cfg, W)
    assert prep.numel() >= tsp.block_weights_bytes(cfg) > 0
    xz = tsp.zigzag_permute(inp["x"].cuda(), shape.D)
    dyz = tsp.zigzag_permute(inp["dy"].cuda(), shape.D)
    # inference forward
    y0 = tsp.block_fwd(cfg, xz, W)
    y1 = tsp.block_fwd(cfg, xz, W, prep=prep)
    # training forward + backward
    s0 = tsp.empty(tsp.saved_bytes(cfg), torch.uint8, "cuda")
    s1 = tsp.empty(tsp.saved_bytes(cfg), torch.uint8, "cuda")
    t0 = tsp.block_fwd(cfg, xz, W, saved=s0)
    t1 = tsp.block_fwd(cfg, xz, W, saved=s1, prep=prep)
    g0 = tsp.block_bwd(cfg, xz, dyz, s0, W)
    g1 = tsp.block_bwd(cfg, xz, dyz, s1, W, prep=prep)
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    assert torch.equal(y0, y1) and torch.equal(t0, t1) and torch.equal(y0, t0)
    for k in g0:
        _same(g0[k], g1[k], k)


def test_stack_prepared_equals_per_call_conversion():
    shape = BlockShape(S=2048, d=256, H=2, inter=512, D=4)
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, torch.bfloat16)
    L = 3
    Ws = [tsp.BlockWeights.from_dict(make_block_inputs(shape, torch.bfloat16, seed=30 + l), "cuda")
          for l in range(L)]
    preps = [tsp.prepare_weights(cfg, W) for W in Ws]
    inp = make_block_inputs(shape, torch.bfloat16, seed=29, with_dy=True)
    xz = tsp.zigzag_permute(inp["x"].cuda(), shape.D)
    dyz = tsp.zigzag_permute(inp["dy"].cuda(), shape.D)
    y0 = tsp.stack_fwd(cfg, xz, Ws)
    y1 = tsp.stack_fwd(cfg, xz, Ws, preps=preps)
    s0 = tsp.empty(tsp.stack_saved_bytes(cfg, L), torch.uint8, "cuda")
    s1 = tsp.empty(tsp.stack_saved_bytes(cfg, L), torch.uint8, "cuda")
    tsp.stack_fwd(cfg, xz, Ws, saved=s0)
    tsp.stack_fwd(cfg, xz, Ws, saved=s1, preps=preps)
    dx0, g0 = tsp.stack_bwd(cfg, dyz, s0, Ws)
    dx1, g1 = tsp.stack_bwd(cfg, dyz, s1, Ws, preps=preps)
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    assert torch.equal(y0, y1)
    _same(dx0, dx1, "dx")
    for l in range(L):
        for k in g0[l]:
            # below the top layer every gradient depends on dQ of the layers above
            _same(g0[l][k], g1[l][k], k if l == L - 1 else "dx")


def test_prepared_block_reads_no_weight_matrix():
    """With prepared copies the matrix pointers may be NULL: only the gains
    and the fp16 copies are read."""
    shape = BlockShape(S=1024, d=256, H=2, inter=512, D=2)
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, torch.bfloat16)
    inp = make_block_inputs(shape, torch.bfloat16, seed=8)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    prep = tsp.prepare_weights(cfg, W)
    xz = tsp.zigzag_permute(inp["x"].cuda(), shape.D)
    want = tsp.block_fwd(cfg, xz, W)
    aw = tsp.AttnW(None, None, None, None, tsp._ptr(W.g_attn))
    mw = tsp.MlpW(None, None, None, tsp._ptr(W.g_mlp), 1)
    ws = tsp.empty(tsp.workspace_bytes(cfg, tsp.TSP_OP_BLOCK_FWD | tsp.TSP_OP_PREPARED),
                   torch.uint8, "cuda")
    out = torch.empty_like(xz)
    st = tsp.load().tsp_block_fwd_prepared(ctypes.byref(cfg), tsp._ptr(xz), tsp._ptr(prep),
                                           ctypes.byref(aw), ctypes.byref(mw), tsp._ptr(out), None,
                                           tsp._ptr(ws), ws.numel(), tsp._stream())
    assert st == tsp.TSP_OK
    torch.cuda.synchronize()
    assert torch.equal(out, want)
