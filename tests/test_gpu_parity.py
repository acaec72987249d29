"""GPU parity: the CUDA path (through the C ABI) against the CPU float64 oracle.

Every input is drawn by folded_tensor_sequence_zigzag_gb300.inputs; the GPU
permutes it into zigzag order with its own kernel and the result is permuted
back with its own kernel before the comparison.  The oracle never sees a GPU
value as input.
"""
import numpy as np
import pytest
import torch

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import tsp
from folded_tensor_sequence_zigzag_gb300.inputs import (BlockShape, TINY_FP32, make_block_inputs,
                                                         sample_rows)
from tests.helpers import assert_bf16_close, assert_f32_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    return tsp.load()


def _run_block(shape: BlockShape, inp: dict, dtype, mode="block", norm=True, residual=True,
               rope_base=0.0):
    dev = "cuda"
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, dtype, shape.eps, rope_base,
                       shape.Hkv)
    W = tsp.BlockWeights.from_dict(inp, dev)
    x = inp["x"].to(dev)
    xz = tsp.zigzag_permute(x, shape.D)
    if mode == "block":
        yz = tsp.block_fwd(cfg, xz, W)
    elif mode == "attn":
        yz = tsp.attn_block_fwd(cfg, xz, W)
    else:
        yz = tsp.gated_mlp_fwd(cfg, xz, W, norm=norm, residual=residual)
    y = tsp.zigzag_permute(yz, shape.D, inverse=True)
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    return y.cpu()


# ------------------------------------------------------------------ K1 permute

@pytest.mark.parametrize("S,D,cols,dtype", [(256, 4, 64, torch.float32), (2048, 8, 512, torch.bfloat16),
                                            (48, 3, 5, torch.float32), (16, 1, 7, torch.bfloat16),
                                            (64, 2, 3, torch.uint8), (131072, 8, 4096, torch.bfloat16)])
def test_zigzag_permute_bit_exact(S, D, cols, dtype):
    g = torch.Generator().manual_seed(S + D)
    if dtype == torch.uint8:
        x = torch.randint(0, 256, (S, cols), generator=g, dtype=torch.uint8)
    else:
        x = torch.randn(S, cols, generator=g).to(dtype)
    xd = x.cuda()
    z = tsp.zigzag_permute(xd, D).cpu()
    pos = torch.from_numpy(O.zigzag_positions(S, D))
    assert torch.equal(z, x[pos])
    back = tsp.zigzag_permute(z.cuda(), D, inverse=True).cpu()
    assert torch.equal(back, x)


# ------------------------------------------------------------------ K2 RMSNorm

@pytest.mark.parametrize("rows,n,dtype", [(300, 64, torch.float32), (1000, 4096, torch.bfloat16),
                                          (37, 200, torch.float32), (257, 11008, torch.bfloat16),
                                          (5, 12, torch.bfloat16)])
def test_rmsnorm_fwd(rows, n, dtype):
    g0 = torch.Generator().manual_seed(rows)
    u = (torch.randn(rows, n, generator=g0) * 3).to(dtype)
    gain = (1 + 0.5 * torch.randn(n, generator=g0)).to(dtype)
    out, rstd = tsp.rmsnorm_fwd(u.cuda(), gain.cuda(), 1e-6, with_rstd=True)
    ref, rref = O.rmsnorm(to64(u), to64(gain), 1e-6)
    if dtype == torch.float32:
        assert_f32_close(out.cpu(), ref, "rmsnorm", tol=1e-5)
    else:
        # one bf16 rounding of an fp32 value: |err| <= 2^-9 |ref| (+ fp32 noise), checked with 2x margin
        err = np.abs(to64(out.cpu()) - ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-6), float((err / (np.abs(ref) + 1e-6)).max())
    assert np.max(np.abs(to64(rstd.cpu()) - rref) / rref) < 1e-5


# ------------------------------------------------------------------ fp32 tiny block (exact path)

def test_tiny_fp32_block_matches_oracle():
    inp = make_block_inputs(TINY_FP32, torch.float32, seed=0)
    y = _run_block(TINY_FP32, inp, torch.float32)
    ref, _ = O.block_fwd(inp["x"], inp, TINY_FP32.H, TINY_FP32.eps)
    assert_f32_close(y, ref, "tiny fp32 block")


@pytest.mark.parametrize("D", [1, 2, 3, 4, 5, 6, 7, 8])
def test_fp32_block_virtual_rank_sweep(D):
    shape = BlockShape(S=2 * D * 16, d=64, H=4, inter=128, D=D)
    inp = make_block_inputs(shape, torch.float32, seed=D)
    y = _run_block(shape, inp, torch.float32)
    ref = O.block_fwd_sharded(inp["x"], inp, shape.H, D, shape.eps)
    assert_f32_close(y, ref, f"fp32 block D={D}")


@pytest.mark.parametrize("D", [1, 2, 4, 8])
def test_fp32_block_S256_rank_sweep(D):
    shape = BlockShape(S=256, d=64, H=4, inter=128, D=D)
    inp = make_block_inputs(shape, torch.float32, seed=0)
    y = _run_block(shape, inp, torch.float32)
    ref, _ = O.block_fwd(inp["x"], inp, 4, shape.eps)
    assert_f32_close(y, ref, f"fp32 S=256 D={D}")


def test_fp32_halves_match_oracle():
    shape = BlockShape(S=96, d=48, H=3, inter=80, D=3)
    inp = make_block_inputs(shape, torch.float32, seed=3)
    h = _run_block(shape, inp, torch.float32, mode="attn")
    href, _ = O.attn_block_fwd(inp["x"], inp, shape.H, shape.eps)
    assert_f32_close(h, href, "fp32 attention half")
    y = _run_block(shape, inp, torch.float32, mode="mlp", norm=False, residual=False)
    yref = O.mlp_fwd_sharded(inp["x"], inp, shape.D, shape.eps, norm=False, residual=False)
    assert_f32_close(y, yref, "fp32 mlp half (no norm, no residual)")


# ------------------------------------------------------------------ bf16 tensor-core path

@pytest.mark.parametrize("S,d,I,D,norm,res", [
    (512, 256, 384, 4, False, False),     # several N and M tiles, I/D = 96 (not a 64 multiple)
    (660, 512, 640, 3, True, True),       # ragged last M tile (660 = 5 x 128 + 20), shards 213/214
    (384, 512, 512, 1, True, False),
    (1000 * 2, 256, 512, 8, False, True),  # S not a multiple of 128 -> ragged M
])
def test_bf16_mlp_half(S, d, I, D, norm, res):
    shape = BlockShape(S=S, d=d, H=2, inter=I, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=S + D)
    y = _run_block(shape, inp, torch.bfloat16, mode="mlp", norm=norm, residual=res)
    ref, _ = O.mlp_fwd(inp["x"], inp, shape.eps, norm=norm, residual=res)
    assert_bf16_close(y, ref, f"bf16 mlp S={S} D={D}")


@pytest.mark.parametrize("S,H,D", [(2048, 2, 4), (512, 2, 1), (4096, 4, 8), (1536, 2, 3)])
def test_bf16_attention_half(S, H, D):
    shape = BlockShape(S=S, d=128 * H, H=H, inter=256, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=S + H)
    h = _run_block(shape, inp, torch.bfloat16, mode="attn")
    ref, _ = O.attn_block_fwd(inp["x"], inp, shape.H, shape.eps)
    assert_bf16_close(h, ref, f"bf16 attention S={S} D={D}")


@pytest.mark.parametrize("S,H,D", [(2048, 2, 4), (4096, 2, 8), (1536, 2, 3)])
def test_bf16_attention_dominated(S, H, D):
    """Sharper softmax (W_Q, W_K x8) and a large W_O (x60) so that the attention
    term, not the residual x, dominates h: checks the attention kernel itself."""
    shape = BlockShape(S=S, d=128 * H, H=H, inter=256, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=S + 11)
    for k, f in (("wq", 8.0), ("wk", 8.0), ("wo", 60.0)):
        inp[k] = (inp[k].float() * f).to(torch.bfloat16)
    h = _run_block(shape, inp, torch.bfloat16, mode="attn")
    ref, _ = O.attn_block_fwd(inp["x"], inp, shape.H, shape.eps)
    x = to64(inp["x"])
    assert np.sqrt(np.mean((ref - x) ** 2)) > 2 * np.sqrt(np.mean(x ** 2))
    assert_bf16_close(h, ref, f"attention-dominated S={S} D={D}")


@pytest.mark.parametrize("S,d,H,I,D", [(2048, 512, 4, 1024, 4), (4096, 256, 2, 512, 8),
                                       (1024, 256, 2, 768, 2)])
def test_bf16_block_small(S, d, H, I, D):
    shape = BlockShape(S=S, d=d, H=H, inter=I, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=7)
    y = _run_block(shape, inp, torch.bfloat16)
    ref, _ = O.block_fwd(inp["x"], inp, H, shape.eps)
    assert_bf16_close(y, ref, f"bf16 block S={S} D={D}")


# ------------------------------------------------------------------ the 7B-shaped workloads

@pytest.mark.parametrize("S", [1024, 2048, 4096, 8192, 16384])
def test_mlp_only_4096_11008_D4(S):
    """SwiGLU MLP alone, d=4096, inter=11008, D=4; no norm, no residual (y = G W_2^T)."""
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=4)
    inp = make_block_inputs(shape, torch.bfloat16, seed=0, mlp_only=True)
    dev = "cuda"
    cfg = tsp.make_cfg(S, 4096, 32, 11008, 4, torch.bfloat16)
    W = tsp.BlockWeights(*(inp[k].to(dev) if k in inp else torch.zeros(1, device=dev)
                           for k in ("wq", "wk", "wv", "wo", "w1", "w3", "w2", "g_attn", "g_mlp")))
    xz = tsp.zigzag_permute(inp["x"].to(dev), 4)
    yz = tsp.gated_mlp_fwd(cfg, xz, W, norm=False, residual=False)
    y = tsp.zigzag_permute(yz, 4, inverse=True).cpu()
    assert tsp.device_status() == tsp.TSP_OK
    rows = sample_rows(S, 4).numpy() if S > 1024 else np.arange(S)
    ref, _ = O.mlp_fwd(inp["x"][rows], inp, shape.eps, norm=False, residual=False)
    assert_bf16_close(y[rows], ref, f"MLP-only S={S}")


@pytest.mark.parametrize("S", [16384, 131072, 262144])
def test_7b_block_fwd_sampled_rows(S):
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=8)
    inp = make_block_inputs(shape, torch.bfloat16, seed=0)
    y = _run_block(shape, inp, torch.bfloat16)
    rows = sample_rows(S, 8).numpy()
    assert len(rows) == 256
    ref = O.block_fwd_rows(inp["x"], inp, shape.H, shape.eps, rows)
    assert_bf16_close(y[rows], ref, f"7B block S={S}")


# ------------------------------------------------------------------ backward

def _run_bwd(shape, inp, dtype, rope_base=0.0, mlp_tile=0):
    dev = "cuda"
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, dtype, shape.eps, rope_base,
                       shape.Hkv, mlp_tile)
    W = tsp.BlockWeights.from_dict(inp, dev)
    xz = tsp.zigzag_permute(inp["x"].to(dev), shape.D)
    dyz = tsp.zigzag_permute(inp["dy"].to(dev), shape.D)
    saved = tsp.empty(tsp.saved_bytes(cfg), torch.uint8, dev)
    yz = tsp.block_fwd(cfg, xz, W, saved=saved)
    g = tsp.block_bwd(cfg, xz, dyz, saved, W)
    g["dx"] = tsp.zigzag_permute(g["dx"], shape.D, inverse=True)
    y = tsp.zigzag_permute(yz, shape.D, inverse=True)
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    return y.cpu(), {k: v.cpu() for k, v in g.items()}


def test_tiny_fp32_backward_matches_oracle():
    inp = make_block_inputs(TINY_FP32, torch.float32, seed=0, with_dy=True)
    y, g = _run_bwd(TINY_FP32, inp, torch.float32)
    ref = O.block_bwd(inp["x"], inp, inp["dy"], TINY_FP32.H, TINY_FP32.eps)
    yref, _ = O.block_fwd(inp["x"], inp, TINY_FP32.H, TINY_FP32.eps)
    assert_f32_close(y, yref, "fwd (training)")
    for k, v in ref.items():
        scale = max(1.0, float(np.max(np.abs(v))))
        assert_f32_close(g[k], v, k, tol=1e-4 * scale)


@pytest.mark.parametrize("D", [1, 3, 8])
def test_fp32_backward_rank_sweep(D):
    shape = BlockShape(S=2 * D * 16, d=32, H=2, inter=48, D=D)
    inp = make_block_inputs(shape, torch.float32, seed=10 + D, with_dy=True)
    _, g = _run_bwd(shape, inp, torch.float32)
    ref = O.block_bwd_sharded(inp["x"], inp, inp["dy"], shape.H, D, shape.eps)
    for k, v in ref.items():
        scale = max(1.0, float(np.max(np.abs(v))))
        assert_f32_close(g[k], v, f"{k} D={D}", tol=1e-4 * scale)


@pytest.mark.parametrize("S,d,H,I,D", [(2048, 256, 2, 512, 4), (4096, 512, 4, 768, 8),
                                       # d = 1024 and 2048: the vectorised RMSNorm backward
                                       (2048, 1024, 8, 1024, 4), (1024, 2048, 16, 512, 2)])
def test_bf16_backward_small(S, d, H, I, D):
    shape = BlockShape(S=S, d=d, H=H, inter=I, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=5, with_dy=True)
    _, g = _run_bwd(shape, inp, torch.bfloat16)
    ref = O.block_bwd(inp["x"], inp, inp["dy"], H, shape.eps)
    for k, v in ref.items():
        assert_bf16_close(g[k], v, f"bf16 {k}")


# ------------------------------------------------------------------ training step at 7B shapes

def test_7b_fwd_bwd_S8192_all_outputs():
    """Config-5 shapes (d=4096, 32x128 heads, inter=11008, D=8) at S=8192:
    every output of the training step against the dense float64 backward,
    once as is and once with the MLP in sequence tiles of 512 rows
    (recomputed in the backward, weight gradients summed over 16 tiles)."""
    shape = BlockShape(S=8192, d=4096, H=32, inter=11008, D=8)
    inp = make_block_inputs(shape, torch.bfloat16, seed=0, with_dy=True)
    yref, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    ref = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)
    for tile in (0, 512):
        y, g = _run_bwd(shape, inp, torch.bfloat16, mlp_tile=tile)
        assert_bf16_close(y, yref, f"y (S=8192, mlp_tile={tile})")
        for k, v in ref.items():
            assert_bf16_close(g[k], v, f"{k} (S=8192, mlp_tile={tile})")


def test_long_context_training_step_S262144_tail():
    """Beyond 131K tokens on one GPU with no sequence tiling: the training step
    at S=262144 (D=8, 7B shapes); dx at the last 256 positions is exact in the
    oracle, every gradient finite."""
    S, D = 262144, 8
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=1, with_dy=True)
    _, g = _run_bwd(shape, inp, torch.bfloat16)
    n_tail = 256
    dx_ref = O.block_bwd_tail(inp["x"], inp, inp["dy"], shape.H, shape.eps, n_tail)
    assert_bf16_close(g["dx"][S - n_tail:], dx_ref, "dx (S=262144, last 256 positions)")
    for k in ("dwq", "dwk", "dwv", "dwo", "dw1", "dw3", "dw2", "dg_attn", "dg_mlp"):
        assert torch.isfinite(g[k]).all(), k


def test_7b_fwd_bwd_S32768_sampled():
    """Config 5 at full size (S=32768, D=8): y on 256 seeded rows and dx on the
    last 256 positions (both exact in the oracle), every gradient finite."""
    S, D = 32768, 8
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=0, with_dy=True)
    y, g = _run_bwd(shape, inp, torch.bfloat16)
    rows = sample_rows(S, D).numpy()
    assert_bf16_close(y[rows], O.block_fwd_rows(inp["x"], inp, shape.H, shape.eps, rows),
                      "y (S=32768, sampled rows)")
    n_tail = 256
    dx_ref = O.block_bwd_tail(inp["x"], inp, inp["dy"], shape.H, shape.eps, n_tail)
    assert_bf16_close(g["dx"][S - n_tail:], dx_ref, "dx (S=32768, last 256 positions)")
    for k in ("dwq", "dwk", "dwv", "dwo", "dw1", "dw3", "dw2", "dg_attn", "dg_mlp"):
        assert torch.isfinite(g[k]).all(), k


def test_7b_fwd_bwd_S32768_sparse_dy_every_gradient():
    """Config 5 at full size (S=32768, D=8) with dy non-zero on 256 seeded rows
    only: every output of the backward (dx at all positions, all weight and
    gain gradients) against the float64 oracle, which needs the forward only
    at those rows (block_bwd_rows).  The kernels run at the full size: every
    key tile, every query tile, the whole dQ reduction stream."""
    S, D = 32768, 8
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=3, with_dy=True)
    rows = np.sort(sample_rows(S, D).numpy())
    dy = inp["dy"].clone()
    keep = torch.zeros(S, dtype=torch.bool)
    keep[torch.from_numpy(rows)] = True
    dy[~keep] = 0
    inp_s = dict(inp)
    inp_s["dy"] = dy
    _, g = _run_bwd(shape, inp_s, torch.bfloat16)
    ref = O.block_bwd_rows(inp["x"], inp, O.f64(dy)[rows], rows, shape.H, shape.eps)
    # dx is dy-sized on the 256 rows and only the attention's share elsewhere,
    # and that share falls off along the sequence (the first keys are seen by
    # every sampled query): the rows of dy against their own RMS, every other
    # row (one position's gradient) against its own RMS at the same 2e-2 bound
    dx, dx_ref = g.pop("dx"), ref.pop("dx")
    assert_bf16_close(dx[rows], dx_ref[rows], "dx at the dy rows (S=32768)")
    other = np.setdiff1d(np.arange(S), rows)
    a, b = O.f64(dx)[other], dx_ref[other]
    row_rms = np.sqrt(np.mean(b * b, axis=1))
    floor = 1e-6 * float(np.sqrt(np.mean(b * b)))   # rows past the last dy row are zero
    worst = float(np.max(np.abs(a - b).max(axis=1) / (row_rms + floor)))
    assert worst <= 2e-2, ("dx elsewhere: max over rows of max|err|/row RMS", worst)
    assert float(np.abs(a - b).sum() / np.abs(b).sum()) <= 5e-3, "dx elsewhere: mean rel"
    for k, v in ref.items():
        assert_bf16_close(g[k], v, f"{k} (S=32768, dy on 256 rows)")


# ------------------------------------------------------------------ rotary embedding (variant)

def _with_rope(inp, base):
    out = dict(inp)
    out["rope_base"] = base
    return out


def test_tiny_fp32_rope_forward_backward():
    base = 10000.0
    inp = make_block_inputs(TINY_FP32, torch.float32, seed=4, with_dy=True)
    y, g = _run_bwd(TINY_FP32, inp, torch.float32, rope_base=base)
    ref_in = _with_rope(inp, base)
    yref, _ = O.block_fwd(inp["x"], ref_in, TINY_FP32.H, TINY_FP32.eps)
    assert_f32_close(y, yref, "rope fwd")
    ref = O.block_bwd(inp["x"], ref_in, inp["dy"], TINY_FP32.H, TINY_FP32.eps)
    for k, v in ref.items():
        scale = max(1.0, float(np.max(np.abs(v))))
        assert_f32_close(g[k], v, f"rope {k}", tol=1e-4 * scale)


def test_bf16_rope_forward_backward_small():
    base = 10000.0
    shape = BlockShape(S=2048, d=256, H=2, inter=512, D=4)
    inp = make_block_inputs(shape, torch.bfloat16, seed=6, with_dy=True)
    y, g = _run_bwd(shape, inp, torch.bfloat16, rope_base=base)
    ref_in = _with_rope(inp, base)
    yref, _ = O.block_fwd(inp["x"], ref_in, shape.H, shape.eps)
    assert_bf16_close(y, yref, "bf16 rope y")
    ref = O.block_bwd(inp["x"], ref_in, inp["dy"], shape.H, shape.eps)
    for k, v in ref.items():
        assert_bf16_close(g[k], v, f"bf16 rope {k}")


def test_7b_rope_block_fwd_sampled_rows():
    base, S = 500000.0, 16384
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=8)
    inp = make_block_inputs(shape, torch.bfloat16, seed=2)
    y = _run_block(shape, inp, torch.bfloat16, rope_base=base)
    rows = sample_rows(S, 8).numpy()
    ref = O.block_fwd_rows(inp["x"], _with_rope(inp, base), shape.H, shape.eps, rows)
    assert_bf16_close(y[rows], ref, "7B rope block S=16384")


# ------------------------------------------------------------------ grouped-query attention (variant)

@pytest.mark.parametrize("Hkv,base", [(2, 0.0), (1, 10000.0)])
def test_tiny_fp32_gqa_forward_backward(Hkv, base):
    shape = BlockShape(S=256, d=64, H=4, inter=128, D=4, Hkv=Hkv)
    inp = make_block_inputs(shape, torch.float32, seed=20 + Hkv, with_dy=True)
    y, g = _run_bwd(shape, inp, torch.float32, rope_base=base)
    ref_in = _with_rope(inp, base)
    yref, _ = O.block_fwd(inp["x"], ref_in, shape.H, shape.eps)
    assert_f32_close(y, yref, f"gqa Hkv={Hkv} fwd")
    ref = O.block_bwd(inp["x"], ref_in, inp["dy"], shape.H, shape.eps)
    for k, v in ref.items():
        assert g[k].shape == v.shape, k
        scale = max(1.0, float(np.max(np.abs(v))))
        assert_f32_close(g[k], v, f"gqa Hkv={Hkv} {k}", tol=1e-4 * scale)


def test_fp32_gqa_backward_three_ranks_matches_sharded_oracle():
    shape = BlockShape(S=2 * 3 * 16, d=64, H=4, inter=48, D=3, Hkv=2)
    inp = make_block_inputs(shape, torch.float32, seed=33, with_dy=True)
    _, g = _run_bwd(shape, inp, torch.float32)
    ref = O.block_bwd_sharded(inp["x"], inp, inp["dy"], shape.H, shape.D, shape.eps)
    for k, v in ref.items():
        scale = max(1.0, float(np.max(np.abs(v))))
        assert_f32_close(g[k], v, f"gqa D=3 {k}", tol=1e-4 * scale)


@pytest.mark.parametrize("S,d,H,Hkv,D,base", [(2048, 512, 4, 2, 4, 0.0), (4096, 1024, 8, 2, 8, 10000.0),
                                               (2048, 1024, 8, 8, 2, 0.0)])
def test_bf16_gqa_forward_backward_small(S, d, H, Hkv, D, base):
    shape = BlockShape(S=S, d=d, H=H, inter=512, D=D, Hkv=Hkv)
    inp = make_block_inputs(shape, torch.bfloat16, seed=7, with_dy=True)
    y, g = _run_bwd(shape, inp, torch.bfloat16, rope_base=base)
    ref_in = _with_rope(inp, base)
    yref, _ = O.block_fwd(inp["x"], ref_in, H, shape.eps)
    assert_bf16_close(y, yref, f"bf16 gqa y (H={H}, Hkv={Hkv})")
    ref = O.block_bwd(inp["x"], ref_in, inp["dy"], H, shape.eps)
    for k, v in ref.items():
        assert g[k].shape == v.shape, k
        assert_bf16_close(g[k], v, f"bf16 gqa {k} (H={H}, Hkv={Hkv})")


def test_7b_gqa8_training_step_S8192_sampled():
    """7B shapes with 8 K/V heads (four query heads per group), RoPE on:
    y on 256 seeded rows and dx on the last 256 positions, both exact in the
    oracle; every gradient finite and of the grouped shapes."""
    S, D, base = 8192, 8, 500000.0
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=D, Hkv=8)
    inp = make_block_inputs(shape, torch.bfloat16, seed=3, with_dy=True)
    y, g = _run_bwd(shape, inp, torch.bfloat16, rope_base=base)
    ref_in = _with_rope(inp, base)
    rows = sample_rows(S, D).numpy()
    assert_bf16_close(y[rows], O.block_fwd_rows(inp["x"], ref_in, shape.H, shape.eps, rows),
                      "gqa8 y (S=8192, sampled rows)")
    n_tail = 256
    dx_ref = O.block_bwd_tail(inp["x"], ref_in, inp["dy"], shape.H, shape.eps, n_tail)
    assert_bf16_close(g["dx"][S - n_tail:], dx_ref, "gqa8 dx (S=8192, last 256 positions)")
    assert g["dwk"].shape == (1024, 4096) and g["dwv"].shape == (1024, 4096)
    for k in ("dwq", "dwk", "dwv", "dwo", "dw1", "dw3", "dw2", "dg_attn", "dg_mlp"):
        assert torch.isfinite(g[k]).all(), k


# ------------------------------------------------------------------ MLP sequence tiling (variant)

@pytest.mark.parametrize("tile,base,Hkv", [(128, 0.0, 0), (256, 10000.0, 2)])
def test_bf16_mlp_tiling_forward_backward(tile, base, Hkv):
    """The training step with the MLP run in sequence tiles (recomputed in the
    backward) against the oracle: every output."""
    shape = BlockShape(S=4096, d=512, H=4, inter=768, D=8, Hkv=Hkv)
    inp = make_block_inputs(shape, torch.bfloat16, seed=12, with_dy=True)
    y, g = _run_bwd(shape, inp, torch.bfloat16, rope_base=base, mlp_tile=tile)
    ref_in = _with_rope(inp, base)
    yref, _ = O.block_fwd(inp["x"], ref_in, shape.H, shape.eps)
    assert_bf16_close(y, yref, f"tiled y (tile={tile})")
    ref = O.block_bwd(inp["x"], ref_in, inp["dy"], shape.H, shape.eps)
    for k, v in ref.items():
        assert_bf16_close(g[k], v, f"tiled {k} (tile={tile})")
