"""GPU parity of the per-rank calls (tsp_rank_attn_project / tsp_rank_attn_heads
/ tsp_rank_mlp_step): the block computed rank by rank by the TSP forward
schedule, with explicit broadcast, all-gather and ring exchanges between the
virtual ranks' buffers on one GPU, against the float64 oracle and against
the one-pass tsp_block_fwd."""
import numpy as np
import pytest
import torch

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import schedule, tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs, sample_rows
from tests.helpers import assert_bf16_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    return tsp.load()


def _assert_same_up_to_bf16_rounding(y, y_other, what):
    """Two bf16 outputs of the same block computed with the work cut
    differently.  Their fp32 values before the final rounding differ by the
    summation order and by the internal fp16 roundings -- the attention's P
    among them, which a rank whose key range is split into chunks (a short
    sequence: too few 256-row blocks to fill the GPU) forms against each
    chunk's own running maximum and merges by log-sum-exp -- so every element
    is within two bf16 spacings (2^-6 of its magnitude) of the other, up to a
    small absolute term for elements near zero, and on average far closer."""
    a, b = O.f64(y), O.f64(y_other)
    rms = float(np.sqrt(np.mean(b * b)))
    diff = np.abs(a - b)
    bound = 2.0 ** -6 * np.maximum(np.abs(a), np.abs(b)) + 2e-3 * rms
    mean_rel = float(diff.sum() / np.abs(b).sum())
    assert np.all(diff <= bound), (what, float((diff / bound).max()), mean_rel)
    assert mean_rel <= 1e-3, (what, mean_rel)


def _run(shape, seed):
    inp = make_block_inputs(shape, torch.bfloat16, seed=seed)
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, torch.bfloat16, shape.eps)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    xz = tsp.zigzag_permute(inp["x"].cuda(), shape.D)
    yz = schedule.block_fwd_by_schedule(cfg, xz, W)
    # the weight transfers on a copy stream, overlapped with the compute: the
    # same kernels on the same data, so the same bits
    yz_ov = schedule.block_fwd_by_schedule(cfg, xz, W, overlap=True)
    y = tsp.zigzag_permute(yz, shape.D, inverse=True)
    y_batched = tsp.zigzag_permute(tsp.block_fwd(cfg, xz, W), shape.D, inverse=True)
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    assert torch.equal(yz, yz_ov)
    return inp, y.cpu(), y_batched.cpu()


@pytest.mark.parametrize("S,d,H,I,D", [(4096, 1024, 8, 2048, 4), (2048, 512, 4, 1024, 2),
                                       (4096, 1024, 8, 2048, 1),
                                       # three heads a shard (384 columns): Q and K|V
                                       # projected by two GEMMs instead of one
                                       (2048, 1536, 12, 1024, 4)])
def test_schedule_by_rank_matches_oracle(S, d, H, I, D):
    shape = BlockShape(S=S, d=d, H=H, inter=I, D=D)
    inp, y, y_batched = _run(shape, seed=S + D)
    ref, _ = O.block_fwd(inp["x"], inp, H, shape.eps)
    assert_bf16_close(y, ref, f"schedule by rank S={S} D={D}")
    _assert_same_up_to_bf16_rounding(y, y_batched, "schedule vs one-pass block")


def test_schedule_by_rank_7b_shapes_S16384():
    """d=4096, 32 heads x 128, inter=11008, D=8 (4 heads, 1376 MLP rows a
    shard): 256 sampled rows against the oracle."""
    S, D = 16384, 8
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=D)
    inp, y, y_batched = _run(shape, seed=0)
    rows = sample_rows(S, D).numpy()
    ref = O.block_fwd_rows(inp["x"], inp, shape.H, shape.eps, rows)
    assert_bf16_close(y[rows], ref, "schedule by rank, 7B shapes")
    _assert_same_up_to_bf16_rounding(y, y_batched, "schedule vs one-pass block, 7B shapes")
    # the rank path (its attention split into chunks here) is as close to the
    # oracle as the one-pass block on the sampled rows
    err = lambda v: float(np.abs(O.f64(v[rows]) - ref).max())
    assert err(y) <= 1.25 * err(y_batched), (err(y), err(y_batched))


def test_rank_calls_reject_what_they_do_not_take():
    S, d, H, I, D = 4096, 1024, 8, 2048, 4
    bf = tsp.make_cfg(S, d, H, I, D, torch.bfloat16)
    assert tsp.rank_workspace_bytes(bf) > 0
    for cfg in (tsp.make_cfg(S, d, H, I, D, torch.float32),          # fp32 path
                tsp.make_cfg(S, d, H, I, D, torch.bfloat16, Hkv=2),  # grouped K/V heads
                tsp.make_cfg(S, d, H, I, D, torch.bfloat16, rope_base=1e4),
                tsp.make_cfg(S, d, H, I, 8, torch.bfloat16),         # one head a shard
                tsp.make_cfg(S, d, H, 2040, D, torch.bfloat16)):     # MLP shard not 32-wide
        assert tsp.rank_workspace_bytes(cfg) == 0
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(tsp.TspError) as e:
        tsp.rank_attn_project(bf, D, 0, x, x, x, x, ws)                # rank out of range
    assert e.value.code == tsp.TSP_ERR_INVALID_ARG
    with pytest.raises(tsp.TspError) as e:
        tsp.rank_attn_project(bf, 0, 0, x, x, x, x, ws)                # workspace too small
    assert e.value.code == tsp.TSP_ERR_INVALID_ARG
    assert np.isfinite(tsp.rank_workspace_bytes(bf))


@pytest.mark.parametrize("S,d,H,I,D", [(4096, 1024, 8, 2048, 4), (2048, 512, 4, 1024, 2),
                                       (4096, 1024, 8, 2048, 1)])
def test_backward_schedule_by_rank_matches_oracle(S, d, H, I, D):
    """The training step rank by rank: the forward schedule, then its reverse
    (schedule.backward: the MLP ring carrying each shard's gradient home, the
    attention shards re-broadcast, the K|V re-gathered, the dK|dV
    reduce-scatter, each shard's gradient summed at its owner, the gains
    all-reduced), every rank's steps in the tsp_rank_* kernels including the
    one-rank attention backward.  Every gradient against the dense float64
    backward."""
    shape = BlockShape(S=S, d=d, H=H, inter=I, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=S + D + 1, with_dy=True)
    cfg = tsp.make_cfg(S, d, H, I, D, torch.bfloat16, shape.eps)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    xz = tsp.zigzag_permute(inp["x"].cuda(), D)
    dyz = tsp.zigzag_permute(inp["dy"].cuda(), D)
    g = schedule.block_bwd_by_schedule(cfg, xz, dyz, W)
    g["dx"] = tsp.zigzag_permute(g["dx"], D, inverse=True)
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    ref = O.block_bwd(inp["x"], inp, inp["dy"], H, shape.eps)
    for k, v in ref.items():
        assert_bf16_close(g[k].cpu(), v, f"{k} by rank (S={S}, D={D})")


def test_backward_schedule_by_rank_7b_shapes_S8192_sparse_dy():
    """d=4096, 32 heads x 128, inter=11008, D=8 (4 heads and 1376 MLP rows a
    shard) at S=8192, with dy on 256 seeded rows: every gradient of the
    rank-by-rank training step against the oracle's exact backward for such a
    dy (block_bwd_rows); dx row by row off the dy rows, as in the batched
    full-size test."""
    S, D = 8192, 8
    shape = BlockShape(S=S, d=4096, H=32, inter=11008, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=11, with_dy=True)
    rows = np.sort(sample_rows(S, D).numpy())
    dy = torch.zeros_like(inp["dy"])
    dy[torch.from_numpy(rows)] = inp["dy"][torch.from_numpy(rows)]
    cfg = tsp.make_cfg(S, shape.d, shape.H, shape.inter, D, torch.bfloat16, shape.eps)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    g = schedule.block_bwd_by_schedule(cfg, tsp.zigzag_permute(inp["x"].cuda(), D),
                                       tsp.zigzag_permute(dy.cuda(), D), W)
    g["dx"] = tsp.zigzag_permute(g["dx"], D, inverse=True)
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    ref = O.block_bwd_rows(inp["x"], inp, O.f64(dy)[rows], rows, shape.H, shape.eps)
    dx, dx_ref = O.f64(g.pop("dx").cpu()), ref.pop("dx")
    assert_bf16_close(torch.from_numpy(dx[rows]), dx_ref[rows], "dx at the dy rows, by rank")
    other = np.setdiff1d(np.arange(S), rows)
    a, b = dx[other], dx_ref[other]
    row_rms = np.sqrt(np.mean(b * b, axis=1))
    floor = 1e-6 * float(np.sqrt(np.mean(b * b)))
    assert float(np.max(np.abs(a - b).max(axis=1) / (row_rms + floor))) <= 2e-2
    for k, v in ref.items():
        assert_bf16_close(g[k].cpu(), v, f"{k} by rank, 7B shapes, dy on 256 rows")
