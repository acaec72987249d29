"""The TSP forward schedule, rank by rank.

Source: "Folding Tensor and Sequence Parallelism for Memory-Efficient
Transformer Training & Inference" (gist.science summary), section 2.  Every
rank owns 1/D of the weights (attention shard r, MLP shard r: "unified
sharding") and its 2c zigzag token rows.  Attention layers: the owners of
the packed W_Q/W_K/W_V/W_O shards broadcast them one after another; every
rank projects its own rows with the shard it has just received, the K/V of
the sequence is all-gathered, and every rank attends with its zigzag rows.
Gated-MLP layers: the W_1/W_2/W_3 shards travel around a ring -- at step t
rank r holds shard (r - t) mod D, received from rank r - 1 -- and every rank
accumulates its partial outputs locally, with no all-reduce.

`forward` runs those steps in that order for the ranks this process holds,
with the data movement behind a `comm` object and one rank's computation
behind an `ops` object.  `LocalComm` holds all D virtual ranks in one
process on one GPU (an exchange is a device copy into the receiving rank's
buffer); `GpuRankOps` is one rank's computation in the library's kernels
(the tsp_rank_* calls).  Nothing here computes any of the block's
arithmetic.
"""
from __future__ import annotations

import torch

from . import tsp


def shard_bounds(n: int, D: int) -> list[int]:
    """Shard boundaries floor(k n / D), k = 0..D (the library's split)."""
    return [(k * n) // D for k in range(D + 1)]


def ring_shard(r: int, t: int, D: int) -> int:
    """The MLP shard rank r holds at ring step t."""
    return (r - t) % D


def forward(comm, ops, D: int):
    """One block forward by the schedule; returns {rank: output rows} for the
    ranks `comm` holds."""
    local = comm.local_ranks()
    for k in range(D):
        shard = comm.broadcast_attn_shard(k)          # from its owner, rank k
        parts = {r: ops.attn_project(r, k, shard) for r in local}
        kv_all = comm.all_gather_kv(k, parts)         # every rank's K|V, rank order
        for r in local:
            ops.attn_heads(r, k, kv_all)
    held = {r: comm.own_mlp_shard(r) for r in local}  # step 0: each rank its own shard
    for t in range(D):
        for r in local:
            ops.mlp_step(r, t, held[r])
        if t + 1 < D:
            held = comm.ring_pass(t, held)            # rank r receives from rank r - 1
    return {r: ops.output(r) for r in local}


class LocalComm:
    """All D virtual ranks in this process, on one GPU.  The broadcast shard is
    copied into one receive buffer that every local rank reads; the all-gather
    copies each rank's K|V rows into one gathered buffer (rank q's rows at
    q * 2c, the zigzag row order); the ring copies each held MLP shard into the
    next rank's receive buffer (two buffers a rank, alternating)."""

    def __init__(self, cfg, W: tsp.BlockWeights, stream=None):
        self.cfg, self.D = cfg, cfg.D
        self.attn_packed = tsp.pack_attn_shards(cfg, W, stream=stream)   # [4d, d]
        self.mlp_packed = tsp.pack_mlp_shards(cfg, W, stream=stream)     # [3I, d]
        self.Cb = shard_bounds(cfg.d, cfg.D)
        self.Ib = shard_bounds(cfg.inter, cfg.D)
        dev, dt = W.wq.device, W.wq.dtype
        wC = max(self.Cb[k + 1] - self.Cb[k] for k in range(self.D))
        wI = max(self.Ib[k + 1] - self.Ib[k] for k in range(self.D))
        self.attn_rx = tsp.empty((4 * wC, cfg.d), dt, dev)
        self.kv_all = tsp.empty((cfg.S, 2 * wC), torch.float16, dev)
        self.mlp_rx = [[tsp.empty((3 * wI, cfg.d), dt, dev) for _ in range(2)] for _ in range(self.D)]

    def local_ranks(self):
        return list(range(self.D))

    def attn_shard(self, k):
        return self.attn_packed[4 * self.Cb[k]:4 * self.Cb[k + 1]]

    def broadcast_attn_shard(self, k):
        src = self.attn_shard(k)
        dst = self.attn_rx[:src.shape[0]]
        dst.copy_(src)
        return dst

    def all_gather_kv(self, k, parts):
        rows = self.cfg.S // self.D
        w = 2 * (self.Cb[k + 1] - self.Cb[k])
        out = self.kv_all[:, :w] if w == self.kv_all.shape[1] else \
            self.kv_all.view(-1)[:self.cfg.S * w].view(self.cfg.S, w)
        for r, p in parts.items():
            out[r * rows:(r + 1) * rows].copy_(p)
        return out

    def own_mlp_shard(self, r):
        return self.mlp_packed[3 * self.Ib[r]:3 * self.Ib[r + 1]]

    def ring_pass(self, t, held):
        out = {}
        for r in range(self.D):
            src = held[(r - 1) % self.D]
            dst = self.mlp_rx[r][t & 1][:src.shape[0]]
            dst.copy_(src)
            out[r] = dst
        return out


class GpuRankOps:
    """One rank's computation in the library's kernels, for the ranks in
    `x_rows` ({rank: that rank's 2c zigzag rows of x}); each rank keeps its own
    workspace, K|V part, fp32 residual and MLP accumulator."""

    def __init__(self, cfg, W: tsp.BlockWeights, x_rows: dict, stream=None):
        self.cfg, self.W, self.stream = cfg, W, stream
        self.rows = cfg.S // cfg.D
        self.x = dict(x_rows)
        dev = next(iter(self.x.values())).device
        nb = tsp.rank_workspace_bytes(cfg)
        if nb == 0:
            raise tsp.TspError(tsp.TSP_ERR_UNSUPPORTED, "tsp_rank_workspace_bytes")
        b = shard_bounds(cfg.d, cfg.D)
        wC = max(hi - lo for lo, hi in zip(b[:-1], b[1:]))
        dt = next(iter(self.x.values())).dtype
        self.ws = {r: tsp.empty(nb, torch.uint8, dev) for r in self.x}
        self.kv = {r: tsp.empty((self.rows, 2 * wC), torch.float16, dev) for r in self.x}
        self.h = {r: tsp.empty((self.rows, cfg.d), torch.float32, dev) for r in self.x}
        self.y = {r: tsp.empty((self.rows, cfg.d), torch.float32, dev) for r in self.x}
        self.out = {r: tsp.empty((self.rows, cfg.d), dt, dev) for r in self.x}

    def attn_project(self, r, k, shard):
        Ck = shard.shape[0] // 4
        kv = self.kv[r].view(-1)[:self.rows * 2 * Ck].view(self.rows, 2 * Ck)
        tsp.rank_attn_project(self.cfg, r, k, self.x[r], self.W.g_attn, shard, kv, self.ws[r],
                              self.stream)
        return kv

    def attn_heads(self, r, k, kv_all):
        tsp.rank_attn_heads(self.cfg, r, k, self.x[r], kv_all, self.h[r], self.ws[r], self.stream)

    def mlp_step(self, r, t, shard):
        last = t == self.cfg.D - 1
        tsp.rank_mlp_step(self.cfg, r, t, self.h[r], self.W.g_mlp, shard, self.y[r],
                          self.out[r] if last else None, self.ws[r], self.stream)

    def output(self, r):
        return self.out[r]


def block_fwd_by_schedule(cfg, x_z, W: tsp.BlockWeights, stream=None):
    """y_z of the block computed rank by rank by the schedule, all D virtual
    ranks on this GPU (the same value tsp_block_fwd computes in one pass)."""
    rows = cfg.S // cfg.D
    comm = LocalComm(cfg, W, stream)
    ops = GpuRankOps(cfg, W, {r: x_z[r * rows:(r + 1) * rows] for r in range(cfg.D)}, stream)
    y = forward(comm, ops, cfg.D)
    return torch.cat([y[r] for r in range(cfg.D)], 0)
