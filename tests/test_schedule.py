"""The TSP forward schedule with real exchanges between processes, on CPU.

`schedule.forward` runs the pages' schedule ("Folding Tensor and Sequence
Parallelism for Memory-Efficient Transformer Training & Inference", section
2, "Runtime schedules") over the ranks a process holds.  Here every rank is
its own process (torch.distributed, gloo, world sizes 2 and 3) holding only
its own attention and MLP shards and its own zigzag rows; the exchanges are
real collectives (broadcast of the attention shard by its owner, K/V
all-gather, ring send/receive of the MLP shards).  One rank's steps are
computed in float64 from the oracle's primitives, so the test checks the
schedule's bookkeeping -- which shard is used when, the all-gather order,
the ring direction, where the residual enters -- against the unsharded block
to 1e-12.  (The GPU runs of the same runner are in test_gpu_schedule.py.)
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import schedule
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs


def _shape(D):
    H, dh = 2 * D, 4
    return BlockShape(S=2 * D * 8, d=H * dh, H=H, inter=12 * D, D=D)


def _weights(D):
    shape = _shape(D)
    inp = make_block_inputs(shape, torch.float32, seed=70 + D)
    gen = torch.Generator().manual_seed(171 + D)
    inp["g_attn"] = 1 + 0.5 * torch.randn(shape.d, generator=gen)
    inp["g_mlp"] = 1 + 0.5 * torch.randn(shape.d, generator=gen)
    for k in ("wq", "wk", "wv", "wo", "w1", "w3", "w2"):
        inp[k] = inp[k] * 10           # far from uniform attention, non-linear MLP
    return shape, {k: O.f64(v) for k, v in inp.items()}


def _attn_shard(W, k, D):
    b = O.shard_bounds(W["wq"].shape[0], D)
    lo, hi = b[k], b[k + 1]
    return np.concatenate([W["wq"][lo:hi], W["wk"][lo:hi], W["wv"][lo:hi], W["wo"][:, lo:hi].T], 0)


def _mlp_shard(W, s, D):
    b = O.shard_bounds(W["w1"].shape[0], D)
    lo, hi = b[s], b[s + 1]
    return np.concatenate([W["w1"][lo:hi], W["w3"][lo:hi], W["w2"][:, lo:hi].T], 0)


class OracleRankOps:
    """One rank's steps in float64, from the packed shards it receives."""

    def __init__(self, shape, W, x):
        self.shape, self.W, self.D = shape, W, shape.D
        self.c = shape.S // (2 * shape.D)
        self.pos = O.zigzag_positions(shape.S, shape.D)
        self.x = x
        self.a, self.q, self.shard, self.h, self.b, self.y = {}, {}, {}, {}, {}, {}

    def _rows(self, r):
        return self.pos[r * 2 * self.c:(r + 1) * 2 * self.c]

    def attn_project(self, r, k, shard):
        if k == 0:
            self.a[r] = O.rmsnorm(self.x[self._rows(r)], self.W["g_attn"], self.shape.eps)[0]
        Ck = shard.shape[0] // 4
        a = self.a[r]
        self.q[r] = a @ shard[:Ck].T
        self.shard[r] = shard
        return np.concatenate([a @ shard[Ck:2 * Ck].T, a @ shard[2 * Ck:3 * Ck].T], 1)

    def attn_heads(self, r, k, kv_all):
        Ck = kv_all.shape[1] // 2
        Ok, _ = O.causal_attention(self.q[r], kv_all[:, :Ck], kv_all[:, Ck:], Ck // self.shape.dh,
                                   q_pos=self._rows(r), k_pos=self.pos)
        base = self.x[self._rows(r)] if k == 0 else self.h[r]
        self.h[r] = base + Ok @ self.shard[r][3 * Ck:]

    def mlp_step(self, r, t, shard):
        if t == 0:
            self.b[r] = O.rmsnorm(self.h[r], self.W["g_mlp"], self.shape.eps)[0]
            self.y[r] = self.h[r].copy()
        Is = shard.shape[0] // 3
        b = self.b[r]
        G = O.silu(b @ shard[:Is].T) * (b @ shard[Is:2 * Is].T)
        self.y[r] = self.y[r] + G @ shard[2 * Is:]

    def output(self, r):
        return self.y[r]


class DistComm:
    """This process is rank `rank` of D and holds its own shards only."""

    def __init__(self, rank, D, W):
        self.rank, self.D, self.W = rank, D, W
        self.own_attn = torch.from_numpy(_attn_shard(W, rank, D))
        self.own_mlp = torch.from_numpy(_mlp_shard(W, rank, D))
        self.Cb = O.shard_bounds(W["wq"].shape[0], D)
        self.Ib = O.shard_bounds(W["w1"].shape[0], D)
        self.log = []

    def local_ranks(self):
        return [self.rank]

    def broadcast_attn_shard(self, k):
        rows = 4 * (self.Cb[k + 1] - self.Cb[k])
        buf = self.own_attn.clone() if self.rank == k else torch.empty(rows, self.own_attn.shape[1],
                                                                       dtype=torch.float64)
        dist.broadcast(buf, src=k)
        self.log.append(("bcast", k))
        return buf.numpy()

    def all_gather_kv(self, k, parts):
        mine = torch.from_numpy(np.ascontiguousarray(parts[self.rank]))
        lst = [torch.empty_like(mine) for _ in range(self.D)]
        dist.all_gather(lst, mine)
        return torch.cat(lst, 0).numpy()       # rank q's rows at q * 2c: the zigzag row order

    def own_mlp_shard(self, r):
        return self.own_mlp.numpy()

    def ring_pass(self, t, held):
        src = torch.from_numpy(np.ascontiguousarray(held[self.rank]))
        prev = (self.rank - 1) % self.D
        s_in = schedule.ring_shard(self.rank, t + 1, self.D)     # what arrives from rank r - 1
        rows = 3 * (self.Ib[s_in + 1] - self.Ib[s_in])
        rx = torch.empty(rows, src.shape[1], dtype=torch.float64)
        ops = [dist.P2POp(dist.isend, src, (self.rank + 1) % self.D),
               dist.P2POp(dist.irecv, rx, prev)]
        for req in dist.batch_isend_irecv(ops):
            req.wait()
        self.log.append(("ring", t, s_in))
        return {self.rank: rx.numpy()}


def _worker(rank, D, port, q):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=D)
        shape, W = _weights(D)
        x = O.f64(make_block_inputs(shape, torch.float32, seed=90 + D)["x"])
        comm = DistComm(rank, D, W)
        ops = OracleRankOps(shape, W, x)
        y_r = schedule.forward(comm, ops, D)[rank]
        ref, _ = O.block_fwd(x, W, shape.H, shape.eps)
        rows = O.zigzag_positions(shape.S, D)[rank * shape.S // D:(rank + 1) * shape.S // D]
        err = float(np.max(np.abs(y_r - ref[rows])) / np.max(np.abs(ref)))
        # the ring hands rank r shard (r - t) mod D at step t, from rank r - 1
        ring = [e for e in comm.log if e[0] == "ring"]
        ok_ring = [s for (_, _, s) in ring] == [(rank - t) % D for t in range(1, D)]
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, err, ok_ring, None))
    except Exception as e:  # noqa: BLE001
        q.put((rank, None, False, repr(e)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("D", [2, 3])
def test_schedule_over_gloo_ranks_equals_unsharded_block(D):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, D, port, q)) for r in range(D)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(D)]
    for p in procs:
        p.join(timeout=60)
    for rank, err, ok_ring, exc in sorted(res, key=lambda t: t[0]):
        assert exc is None, f"rank {rank}: {exc}"
        assert err <= 1e-12, (rank, err)
        assert ok_ring, rank


def test_ring_hands_every_shard_to_every_rank_once():
    for D in range(1, 9):
        for r in range(D):
            seen = [schedule.ring_shard(r, t, D) for t in range(D)]
            assert sorted(seen) == list(range(D))
            # the shard rank r holds at step t + 1 is the one rank r - 1 held at step t
            for t in range(D - 1):
                assert schedule.ring_shard(r, t + 1, D) == schedule.ring_shard((r - 1) % D, t, D)
        assert schedule.shard_bounds(10, D) == O.shard_bounds(10, D)
