"""Seeded synthetic inputs for the TSP-folded block.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests.  It holds no arithmetic of the method itself: it only draws Gaussian
tensors in a fixed order and rounds them to the storage dtype.

Workload recipe (the pages print no dataset; every input is synthetic):
  * activations x  ~ N(0, 1), shape [S, d], in global token order;
  * weight matrices ~ N(0, 0.02), nn.Linear convention [out, in]:
      W_Q, W_O : [d, d];  W_K, W_V : [Hkv*dh, d] ([d, d] unless the shape
      sets Hkv, grouped-query attention);  W_1, W_3 : [inter, d];
      W_2 : [d, inter];
  * RMSNorm gains g_attn, g_mlp = 1 (learnable; not drawn);
  * upstream gradient dy ~ N(0, 1), shape [S, d] (training step only).
Draw order on one ``torch.Generator('cpu')``: x, W_Q, W_K, W_V, W_O, W_1,
W_3, W_2, dy; each ``normal_`` in fp32, then round-to-nearest-even to bf16
when the config is bf16.  The exact same bytes are handed to the GPU path and
to the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class BlockShape:
    S: int          # tokens
    d: int          # d_model
    H: int          # heads
    inter: int      # SwiGLU intermediate size
    D: int          # virtual ranks
    eps: float = 1e-6
    Hkv: int = 0    # K/V heads (0: as many as query heads)

    @property
    def dh(self) -> int:
        return self.d // self.H

    @property
    def dkv(self) -> int:
        return (self.Hkv or self.H) * self.dh


# The five workloads the method is exercised on (7B-shaped unless noted).
TINY_FP32 = BlockShape(S=256, d=64, H=4, inter=128, D=4)
MLP_4096 = lambda S: BlockShape(S=S, d=4096, H=32, inter=11008, D=4)  # noqa: E731
BLOCK_7B_16K = BlockShape(S=16384, d=4096, H=32, inter=11008, D=8)
BLOCK_7B_128K = BlockShape(S=131072, d=4096, H=32, inter=11008, D=8)
BLOCK_7B_32K_TRAIN = BlockShape(S=32768, d=4096, H=32, inter=11008, D=8)


def _normal(gen: torch.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float32)
    t.normal_(0.0, std, generator=gen)
    return t.to(dtype) if dtype != torch.float32 else t


def make_block_inputs(shape: BlockShape, dtype: torch.dtype, seed: int = 0,
                      with_dy: bool = False, mlp_only: bool = False) -> dict:
    """Draw the block's inputs on the CPU.

    Returns a dict of CPU tensors: x, wq, wk, wv, wo, w1, w3, w2, g_attn,
    g_mlp and (if ``with_dy``) dy.  With ``mlp_only`` the attention weights
    are skipped (draw order of the rest is unchanged: x, W_1, W_3, W_2).
    """
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    S, d, inter = shape.S, shape.d, shape.inter
    out = {"x": _normal(gen, (S, d), 1.0, dtype)}
    if not mlp_only:
        for name in ("wq", "wk", "wv", "wo"):
            rows = shape.dkv if name in ("wk", "wv") else d
            out[name] = _normal(gen, (rows, d), 0.02, dtype)
    out["w1"] = _normal(gen, (inter, d), 0.02, dtype)
    out["w3"] = _normal(gen, (inter, d), 0.02, dtype)
    out["w2"] = _normal(gen, (d, inter), 0.02, dtype)
    out["g_attn"] = torch.ones(d, dtype=dtype)
    out["g_mlp"] = torch.ones(d, dtype=dtype)
    if with_dy:
        out["dy"] = _normal(gen, (S, d), 1.0, dtype)
    return out


def sample_rows(S: int, D: int, n: int = 256, seed: int = 1234) -> torch.Tensor:
    """Seeded sample of global token positions used to check large workloads.

    Always contains 0, S-1 and the first and last position of every one of
    the 2D zigzag chunks (these count toward the ``n`` rows); the rest are
    drawn without replacement.  Returned sorted, int64.
    """
    c = S // (2 * D)
    must = {0, S - 1}
    for j in range(2 * D):
        must.add(j * c)
        must.add(j * c + c - 1)
    must = sorted(must)
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    perm = torch.randperm(S, generator=gen).tolist()
    rest = []
    chosen = set(must)
    for p in perm:
        if len(must) + len(rest) >= min(n, S):
            break
        if p not in chosen:
            rest.append(p)
            chosen.add(p)
    return torch.tensor(sorted(must + rest), dtype=torch.int64)
