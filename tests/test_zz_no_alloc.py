"""GPU test of tsp_gated_mlp_fwd_noalloc, the gated-MLP forward for callers
that cannot allocate device memory during the call (for instance a plugin
running inside an engine that has planned all device memory up front, or a
latency-critical loop that must not pay for a cudaMalloc).

It must give what tsp_gated_mlp_fwd gives, on two calls in a row with
different inputs (the shared scratch keeps the previous call's contents, which
must not leak into the next result), and refuse a problem whose scratch does
not fit in its fixed 32 MiB array.  This file is collected last on purpose.
"""
import pytest
import torch

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


@pytest.mark.parametrize("S,d,I,D,dtype,norm,res", [
    (512, 256, 384, 4, torch.bfloat16, False, False),
    (660, 512, 640, 3, torch.bfloat16, True, True),
    (96, 48, 80, 3, torch.float32, True, True),
])
def test_noalloc_matches_workspace_entry_point_twice(S, d, I, D, dtype, norm, res):
    """Two calls in a row with different inputs give exactly (bit for bit: the
    same kernels on the same grid) what the workspace entry point gives, and
    device memory stays as it was across them: the calls allocate nothing."""
    shape = BlockShape(S=S, d=d, H=2, inter=I, D=D)
    cfg = tsp.make_cfg(S, d, 2, I, D, dtype)
    assert tsp.workspace_bytes(cfg, tsp.TSP_OP_MLP_FWD) <= tsp.NOALLOC_SCRATCH_BYTES
    calls = []
    for seed in (S, S + 1):
        inp = make_block_inputs(shape, dtype, seed=seed, mlp_only=True)
        inp.update({k: torch.zeros(1, dtype=dtype) for k in ("wq", "wk", "wv", "wo")})
        W = tsp.BlockWeights.from_dict(inp, "cuda")
        hz = tsp.zigzag_permute(inp["x"].cuda(), D)
        ref = tsp.gated_mlp_fwd(cfg, hz, W, norm=norm, residual=res)
        out = torch.full_like(hz, float("nan"))
        calls.append((W, hz, ref, out))
    # a first call looks the scratch array up (and may load the module)
    warm = torch.empty_like(calls[0][1])
    tsp.gated_mlp_fwd_noalloc(cfg, calls[0][1], calls[0][0], warm, norm=norm, residual=res)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    held0 = torch.cuda.memory_allocated()
    for W, hz, _, out in calls:
        tsp.gated_mlp_fwd_noalloc(cfg, hz, W, out, norm=norm, residual=res)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == held0
    assert tsp.device_status() == tsp.TSP_OK
    for call, (_, _, ref, out) in enumerate(calls):
        assert torch.equal(out, ref), f"no-alloc MLP call {call} differs from the workspace path"


def test_noalloc_rejects_a_problem_larger_than_its_scratch():
    cfg = tsp.make_cfg(16384, 4096, 32, 11008, 4, torch.bfloat16)
    assert tsp.workspace_bytes(cfg, tsp.TSP_OP_MLP_FWD) > tsp.NOALLOC_SCRATCH_BYTES
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    W = tsp.BlockWeights(*([x] * 9))
    with pytest.raises(tsp.TspError) as e:
        tsp.gated_mlp_fwd_noalloc(cfg, x, W, torch.empty_like(x))
    assert e.value.code == tsp.TSP_ERR_INVALID_ARG
