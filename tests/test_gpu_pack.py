"""GPU test of tsp_pack_attn_shards, the packed attention shard that one step
of the broadcast schedule carries ("Folding Tensor and Sequence Parallelism
for Memory-Efficient Transformer Training & Inference", section 2, "Runtime
schedules", attention bullet: each rank's packed W_Q, W_K, W_V, W_O shard).

The packed layout is a pure copy, so it must match, bit for bit, slicing the
weights at the oracle's shard boundaries: shard k (columns C_k) is
[W_Q[C_k,:]; W_K[C_k,:]; W_V[C_k,:]; W_O[:,C_k]^T], shards one after another.
"""
import numpy as np
import pytest
import torch

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    return tsp.load()


def _packed_by_slicing(inp, d, D):
    b = O.shard_bounds(d, D)
    parts = []
    for k in range(D):
        lo, hi = b[k], b[k + 1]
        parts += [inp["wq"][lo:hi], inp["wk"][lo:hi], inp["wv"][lo:hi], inp["wo"][:, lo:hi].T]
    return torch.cat(parts, 0)


@pytest.mark.parametrize("d,H,D,dtype", [(64, 4, 3, torch.float32), (48, 3, 5, torch.float32),
                                         (256, 2, 8, torch.bfloat16), (512, 4, 3, torch.bfloat16),
                                         (4096, 32, 8, torch.bfloat16), (96, 2, 1, torch.bfloat16)])
def test_pack_attn_shards_bit_exact(d, H, D, dtype):
    shape = BlockShape(S=2 * D, d=d, H=H, inter=2 * D, D=D)
    inp = make_block_inputs(shape, dtype, seed=d + D)
    cfg = tsp.make_cfg(shape.S, d, H, shape.inter, D, dtype)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    got = tsp.pack_attn_shards(cfg, W)
    torch.cuda.synchronize()
    want = _packed_by_slicing(inp, d, D)
    assert got.shape == want.shape == (4 * d, d)
    assert torch.equal(got.cpu(), want)
    # every shard's rows start where the previous shard's end
    sizes = np.diff(O.shard_bounds(d, D))
    assert int(4 * sizes.sum()) == 4 * d


def test_pack_attn_shards_rejects_grouped_kv():
    shape = BlockShape(S=8, d=256, H=2, inter=8, D=4, Hkv=1)
    inp = make_block_inputs(shape, torch.bfloat16, seed=1)
    cfg = tsp.make_cfg(8, 256, 2, 8, 4, torch.bfloat16, Hkv=1)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    with pytest.raises(tsp.TspError) as e:
        tsp.pack_attn_shards(cfg, W)
    assert e.value.code == tsp.TSP_ERR_UNSUPPORTED
