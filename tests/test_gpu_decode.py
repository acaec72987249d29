"""GPU parity of the inference path: prefill into the zigzag KV cache, then
decode steps of T new tokens, against the CPU float64 oracle.

The oracle's decode output is the causal block forward over the whole
sequence at the new positions; its cache is the prompt's K/V in zigzag row
order.  Every input comes from the seeded generators; the oracle never sees a
GPU value.
"""
import numpy as np
import pytest
import torch

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs
from tests.helpers import assert_bf16_close, assert_f32_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    return tsp.load()


def _run(S, shape_kw, dtype, steps, rope_base=0.0, seed=0, spare=5):
    """Prefill S prompt tokens, then decode `steps` tokens at a time.
    Returns (inputs, y of the prompt (global order), [y of each step], cache)."""
    n_new = sum(steps)
    shape = BlockShape(S=S + n_new, **shape_kw)
    inp = make_block_inputs(shape, dtype, seed=seed)
    cfg = tsp.make_cfg(S, shape.d, shape.H, shape.inter, shape.D, dtype, shape.eps, rope_base,
                       shape.Hkv)
    dev = "cuda"
    W = tsp.BlockWeights.from_dict(inp, dev)
    x = inp["x"].to(dev)
    cache = tsp.KVCache(cfg, S + n_new + spare, dev)
    yz = tsp.block_prefill(cfg, tsp.zigzag_permute(x[:S].contiguous(), shape.D), W, cache)
    y_prompt = tsp.zigzag_permute(yz, shape.D, inverse=True)
    outs = []
    n = S
    for T in steps:
        outs.append(tsp.block_decode(cfg, x[n:n + T].contiguous(), W, cache))
        n += T
    torch.cuda.synchronize()
    assert tsp.device_status() == tsp.TSP_OK
    assert cache.n == S + n_new
    ref_in = dict(inp)
    if rope_base:
        ref_in["rope_base"] = rope_base
    return shape, ref_in, y_prompt.cpu(), [o.cpu() for o in outs], cache, cfg


def _oracle_steps(ref_in, S, steps, H, eps):
    x = ref_in["x"]
    chunks, n = [], S
    for T in steps:
        chunks.append(x[n:n + T])
        n += T
    return O.block_decode(x[:S], chunks, ref_in, H, eps)


@pytest.mark.parametrize("Hkv,base,steps", [(0, 0.0, [1, 3, 8, 2]), (2, 10000.0, [2, 5]),
                                            (1, 0.0, [8])])
def test_fp32_prefill_and_decode(Hkv, base, steps):
    S = 256
    shape, ref_in, y_prompt, outs, cache, cfg = _run(
        S, dict(d=64, H=4, inter=128, D=4, Hkv=Hkv), torch.float32, steps, base, seed=40 + Hkv)
    yref, _ = O.block_fwd(ref_in["x"][:S], ref_in, shape.H, shape.eps)
    assert_f32_close(y_prompt, yref, "prefill y")
    kv_ref = O.kv_cache_zigzag(ref_in["x"][:S], ref_in, shape.H, shape.eps, shape.D)
    assert_f32_close(cache.view(cfg)[:S].cpu(), kv_ref, "cache rows (zigzag order)")
    for k, (got, want) in enumerate(zip(outs, _oracle_steps(ref_in, S, steps, shape.H, shape.eps))):
        assert got.shape == want.shape
        assert_f32_close(got, want, f"decode step {k} (T={steps[k]})")


@pytest.mark.parametrize("S,kw,base,steps", [
    (2048, dict(d=512, H=4, inter=512, D=4), 0.0, [1, 4, 8]),
    (4096, dict(d=1024, H=8, inter=512, D=8, Hkv=2), 10000.0, [1, 8, 3]),
])
def test_bf16_prefill_and_decode(S, kw, base, steps):
    shape, ref_in, y_prompt, outs, cache, cfg = _run(S, kw, torch.bfloat16, steps, base, seed=3)
    kv_ref = O.kv_cache_zigzag(ref_in["x"][:S], ref_in, shape.H, shape.eps, shape.D)
    got_kv = cache.view(cfg)[:S].cpu()
    dkv = kv_ref.shape[1] // 2
    assert_bf16_close(got_kv[:, :dkv], kv_ref[:, :dkv], "cache K (zigzag order)")
    assert_bf16_close(got_kv[:, dkv:], kv_ref[:, dkv:], "cache V (zigzag order)")
    for k, (got, want) in enumerate(zip(outs, _oracle_steps(ref_in, S, steps, shape.H, shape.eps))):
        assert_bf16_close(got, want, f"bf16 decode step {k} (T={steps[k]})")


@pytest.mark.parametrize("Hkv,base,steps", [(0, 0.0, [1, 4]), (8, 500000.0, [1])])
def test_7b_decode_after_16k_prompt(Hkv, base, steps):
    """7B shapes, a 16384-token prompt over D=8 virtual ranks, then decode."""
    S = 16384
    shape, ref_in, _, outs, _, _ = _run(
        S, dict(d=4096, H=32, inter=11008, D=8, Hkv=Hkv), torch.bfloat16, steps, base, seed=11)
    for k, (got, want) in enumerate(zip(outs, _oracle_steps(ref_in, S, steps, shape.H, shape.eps))):
        assert_bf16_close(got, want, f"7B decode step {k} (T={steps[k]}, Hkv={Hkv or 32})")


def test_fp32_decode_crosses_split_boundaries():
    """130 tokens decoded 8 at a time (the last call 2) after a prompt whose
    ranks own 64 rows each (D=8): the decoded rows cross the 128-row split
    boundary of the appended region, with grouped K/V heads and RoPE on."""
    S, steps = 512, [8] * 16 + [2]
    shape, ref_in, _, outs, cache, cfg = _run(
        S, dict(d=64, H=4, inter=128, D=8, Hkv=2), torch.float32, steps, 500.0, seed=77, spare=0)
    assert cache.n == cache.rows_cap
    want = _oracle_steps(ref_in, S, steps, shape.H, shape.eps)
    for k, (got, w) in enumerate(zip(outs, want)):
        assert_f32_close(got, w, f"decode step {k} (T={steps[k]})")


def test_bf16_decode_streaming_across_split_boundaries():
    """Calls of 4 tokens (then 3) with one query head per K/V head: at most
    four query rows per K/V head, the streaming kernel's case, for 131 tokens
    after a 1024-token prompt over D=2 ranks; the appended rows cross the
    128-row split boundary, with RoPE on.  (The 16K-prompt 7B cases above
    give that kernel slices of many splits each.)"""
    S, steps = 1024, [4] * 32 + [3]
    shape, ref_in, _, outs, cache, cfg = _run(
        S, dict(d=256, H=2, inter=512, D=2), torch.bfloat16, steps, 10000.0, seed=21, spare=0)
    assert cache.n == cache.rows_cap
    want = _oracle_steps(ref_in, S, steps, shape.H, shape.eps)
    for k, (got, w) in enumerate(zip(outs, want)):
        assert_bf16_close(got, w, f"bf16 decode step {k} (T={steps[k]})")
