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

    # --- backward (schedule.backward), after the forward ran on this object
    def set_dy(self, r, dy_r):
        self.dy = getattr(self, "dy", {})
        self.dy[r] = dy_r

    def mlp_bwd_step(self, r, t, shard, g):
        if t == 0:
            self.db = getattr(self, "db", {})
            self.db[r] = np.zeros_like(self.h[r])
        Is = shard.shape[0] // 3
        w1s, w3s, w2t = shard[:Is], shard[Is:2 * Is], shard[2 * Is:]   # w2t = W_2[:, I_s]^T
        b = self.b[r]
        A, B = b @ w1s.T, b @ w3s.T
        sA = O.sigmoid(A)
        G = A * sA * B
        dG = self.dy[r] @ w2t.T
        dA = dG * B * sA * (1.0 + A * (1.0 - sA))
        dB = dG * A * sA
        self.db[r] += dA @ w1s + dB @ w3s
        part = np.concatenate([dA.T @ b, dB.T @ b, G.T @ self.dy[r]], 0)
        return part if g is None else g + part

    def mlp_bwd_finish(self, r):
        self.dh, self.da, self.dg = (getattr(self, n, {}) for n in ("dh", "da", "dg"))
        _, rstd2 = O.rmsnorm(self.h[r], self.W["g_mlp"], self.shape.eps)
        du2, dg2 = O.rmsnorm_bwd(self.db[r], self.h[r], self.W["g_mlp"], rstd2)
        self.dh[r] = self.dy[r] + du2
        self.da[r] = np.zeros_like(self.h[r])
        self.dg[r] = [None, dg2]

    def attn_bwd_heads(self, r, k, kv_all):
        Ck = kv_all.shape[1] // 2
        K, V = kv_all[:, :Ck], kv_all[:, Ck:]
        nh = Ck // self.shape.dh
        Ok, _ = O.causal_attention(self.q[r], K, V, nh, q_pos=self._rows(r), k_pos=self.pos)
        dO = self.dh[r] @ self.shard[r][3 * Ck:].T          # dh W_O[:, C_k]
        dq, dk, dv = O.causal_attention_bwd(self.q[r], K, V, Ok, dO, nh, q_pos=self._rows(r),
                                            k_pos=self.pos)
        self.ok, self.dq = getattr(self, "ok", {}), getattr(self, "dq", {})
        self.ok[r], self.dq[r] = Ok, dq
        return np.concatenate([dk, dv], 1)

    def attn_bwd_weights(self, r, k, dkv_r):
        Ck = dkv_r.shape[1] // 2
        dk, dv = dkv_r[:, :Ck], dkv_r[:, Ck:]
        sh, a = self.shard[r], self.a[r]
        self.da[r] += self.dq[r] @ sh[:Ck] + dk @ sh[Ck:2 * Ck] + dv @ sh[2 * Ck:3 * Ck]
        return np.concatenate([self.dq[r].T @ a, dk.T @ a, dv.T @ a, self.ok[r].T @ self.dh[r]], 0)

    def attn_bwd_finish(self, r):
        x_r = self.x[self._rows(r)]
        _, rstd1 = O.rmsnorm(x_r, self.W["g_attn"], self.shape.eps)
        du1, dg1 = O.rmsnorm_bwd(self.da[r], x_r, self.W["g_attn"], rstd1)
        self.dxr = getattr(self, "dxr", {})
        self.dxr[r] = self.dh[r] + du1
        self.dg[r][0] = dg1

    def gain_grads(self, r):
        return np.concatenate(self.dg[r])

    def dx(self, r):
        return self.dxr[r]


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

    # --- backward exchanges
    def ring_pass_with_grad(self, t, held, grad):
        src, gsrc = (torch.from_numpy(np.ascontiguousarray(v[self.rank])) for v in (held, grad))
        prev, nxt = (self.rank - 1) % self.D, (self.rank + 1) % self.D
        s_in = schedule.ring_shard(self.rank, t + 1, self.D)
        rows = 3 * (self.Ib[s_in + 1] - self.Ib[s_in])
        rx = torch.empty(rows, src.shape[1], dtype=torch.float64)
        grx = torch.empty_like(rx)
        ops = [dist.P2POp(dist.isend, src, nxt), dist.P2POp(dist.irecv, rx, prev),
               dist.P2POp(dist.isend, gsrc, nxt), dist.P2POp(dist.irecv, grx, prev)]
        for req in dist.batch_isend_irecv(ops):
            req.wait()
        self.log.append(("bring", t, s_in))
        return {self.rank: rx.numpy()}, {self.rank: grx.numpy()}

    def keep_mlp_grads(self, grad):
        self.mlp_grad = grad[self.rank]        # the gradient of this rank's own shard

    def reduce_scatter_kv(self, k, dkv):
        full = torch.from_numpy(np.ascontiguousarray(dkv[self.rank]))
        dist.all_reduce(full)
        rows = full.shape[0] // self.D
        return {self.rank: full[self.rank * rows:(self.rank + 1) * rows].numpy()}

    def reduce_attn_grad(self, k, gparts):
        t = torch.from_numpy(np.ascontiguousarray(gparts[self.rank]))
        dist.reduce(t, dst=k)
        if self.rank == k:
            self.attn_grad = t.numpy().copy()

    def all_reduce_gains(self, g):
        t = torch.from_numpy(np.ascontiguousarray(g[self.rank]))
        dist.all_reduce(t)
        self.gains = t.numpy().copy()


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


def _bwd_worker(rank, D, port, q):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=D)
        shape, W = _weights(D)
        inp = make_block_inputs(shape, torch.float32, seed=90 + D, with_dy=True)
        x, dy = O.f64(inp["x"]), O.f64(inp["dy"])
        comm = DistComm(rank, D, W)
        ops = OracleRankOps(shape, W, x)
        schedule.forward(comm, ops, D)
        ops.set_dy(rank, dy[ops._rows(rank)])
        dx_r = schedule.backward(comm, ops, D)[rank]
        bring = [e for e in comm.log if e[0] == "bring"]
        ok_ring = [s for (_, _, s) in bring] == [(rank - t) % D for t in range(1, D + 1)]
        q.put((rank, dx_r, comm.attn_grad, comm.mlp_grad, comm.gains, ok_ring, None))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # noqa: BLE001
        q.put((rank, None, None, None, None, False, repr(e)))


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


@pytest.mark.parametrize("D", [2, 3])
def test_backward_schedule_over_gloo_ranks_equals_dense_backward(D):
    """schedule.backward with every rank its own process: the MLP ring with
    each shard's gradient riding along (D hops, the last one home), the
    re-broadcast attention shards, the K|V all-gather, the reduce-scatter of
    dK|dV to the key owners, the reduction of each shard's weight gradient to
    its owner and the all-reduced gains.  dx (from each rank's rows) and every
    weight and gain gradient (from the owners' shards) against the dense
    float64 backward to 1e-12."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bwd_worker, args=(r, D, port, q)) for r in range(D)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(D)]
    for p in procs:
        p.join(timeout=60)
    res.sort(key=lambda t: t[0])
    for rank, *_, ok_ring, exc in res:
        assert exc is None, f"rank {rank}: {exc}"
        assert ok_ring, rank
    shape, W = _weights(D)
    inp = make_block_inputs(shape, torch.float32, seed=90 + D, with_dy=True)
    ref = O.block_bwd(inp["x"], W, inp["dy"], shape.H, shape.eps)
    S, d, c = shape.S, shape.d, shape.S // (2 * D)
    pos = O.zigzag_positions(S, D)
    Cb, Ib = O.shard_bounds(d, D), O.shard_bounds(shape.inter, D)
    got = {k: np.zeros_like(v) for k, v in ref.items()}
    for rank, dx_r, ag, mg, gains, _, _ in res:
        got["dx"][pos[rank * 2 * c:(rank + 1) * 2 * c]] = dx_r
        C, n = slice(Cb[rank], Cb[rank + 1]), Cb[rank + 1] - Cb[rank]
        got["dwq"][C], got["dwk"][C], got["dwv"][C] = ag[:n], ag[n:2 * n], ag[2 * n:3 * n]
        got["dwo"][:, C] = ag[3 * n:].T
        I, m = slice(Ib[rank], Ib[rank + 1]), Ib[rank + 1] - Ib[rank]
        got["dw1"][I], got["dw3"][I] = mg[:m], mg[m:2 * m]
        got["dw2"][:, I] = mg[2 * m:].T
        got["dg_attn"], got["dg_mlp"] = gains[:d], gains[d:]
    for k, v in ref.items():
        assert np.max(np.abs(got[k] - v)) <= 1e-12 * np.max(np.abs(v)), k
