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


def backward(comm, ops, D: int):
    """One block backward by the schedule, after `forward` ran with the same
    `ops` (which keeps what each rank's forward left).  Returns {rank: dx
    rows} for the ranks `comm` holds; each shard's weight gradient ends at its
    owner (comm keeps it) and the gain gradients are all-reduced.

    The pages describe the forward only; this is its reverse, moving the same
    shards (reading R17):
      * MLP: the ring again, rank r holding shard (r - t) mod D at step t; the
        shard's weight gradient travels with it, each rank adding its rows'
        part, and one more hop after the last step brings it to its owner;
      * attention: the owners broadcast their packed shards again; every rank
        recomputes its K|V of the shard and the K|V is all-gathered; each rank
        back-propagates its own query rows through the shard's heads, which
        gives dK|dV for every key, and a reduce-scatter returns to each rank
        the sum over all query ranks for its own rows; the shard's weight
        gradient (summed over ranks) goes to its owner;
      * the RMSNorm gains are replicated, so their gradients are all-reduced.
    """
    local = comm.local_ranks()
    held = {r: comm.own_mlp_shard(r) for r in local}
    grad = {r: None for r in local}                 # running gradient of the held shard
    for t in range(D):
        for r in local:
            grad[r] = ops.mlp_bwd_step(r, t, held[r], grad[r])
        held, grad = comm.ring_pass_with_grad(t, held, grad)
    comm.keep_mlp_grads(grad)                       # rank r: the gradient of its own shard
    for r in local:
        ops.mlp_bwd_finish(r)
    for k in range(D):
        shard = comm.broadcast_attn_shard(k)
        parts = {r: ops.attn_project(r, k, shard) for r in local}
        kv_all = comm.all_gather_kv(k, parts)
        dkv = {r: ops.attn_bwd_heads(r, k, kv_all) for r in local}   # every key's dK|dV
        dkv_own = comm.reduce_scatter_kv(k, dkv)                      # own rows, all query ranks
        comm.reduce_attn_grad(k, {r: ops.attn_bwd_weights(r, k, dkv_own[r]) for r in local})
    for r in local:
        ops.attn_bwd_finish(r)
    comm.all_reduce_gains({r: ops.gain_grads(r) for r in local})
    return {r: ops.dx(r) for r in local}


class LocalComm:
    """All D virtual ranks in this process, on one GPU.  The broadcast copies
    the owner's packed shard into a receive buffer that every local rank
    reads; the all-gather copies each rank's K|V rows into one gathered buffer
    (rank q's rows at q * 2c, the zigzag row order); the ring copies each held
    MLP shard into the next rank's receive buffer.  Receive buffers come in
    pairs, alternating by step.

    overlap=True moves the weight transfers (broadcast and ring) to a copy
    stream, the single-GPU picture of the pages' transfer hidden behind the
    shard GEMMs: shard k + 1 is copied while step k computes, and the compute
    stream waits for a copy only where it reads the buffer.  The K|V
    all-gather stays on the compute stream (its data is made by the same
    step)."""

    def __init__(self, cfg, W: tsp.BlockWeights, stream=None, overlap=False):
        self.cfg, self.D = cfg, cfg.D
        dev = W.wq.device
        self.dev, self._stream = dev, stream
        self.attn_packed = tsp.pack_attn_shards(cfg, W, stream=self.stream)   # [4d, d]
        self.mlp_packed = tsp.pack_mlp_shards(cfg, W, stream=self.stream)     # [3I, d]
        self.Cb = shard_bounds(cfg.d, cfg.D)
        self.Ib = shard_bounds(cfg.inter, cfg.D)
        dt = W.wq.dtype
        wC = max(self.Cb[k + 1] - self.Cb[k] for k in range(self.D))
        wI = max(self.Ib[k + 1] - self.Ib[k] for k in range(self.D))
        self.attn_rx = [tsp.empty((4 * wC, cfg.d), dt, dev) for _ in range(2)]
        self.kv_all = tsp.empty((cfg.S, 2 * wC), torch.float16, dev)
        self.mlp_rx = [[tsp.empty((3 * wI, cfg.d), dt, dev) for _ in range(2)] for _ in range(self.D)]
        self.overlap = overlap
        self._copy = torch.cuda.Stream(dev) if overlap else None
        if overlap:
            self._copy.wait_stream(self.stream)   # the packed shards are written
        # per receive slot: the copy into it is done / the compute reading it is done
        self.a_copied = [torch.cuda.Event() for _ in range(2)]
        self.a_used = [torch.cuda.Event() for _ in range(2)]
        self.m_copied = [torch.cuda.Event() for _ in range(2)]
        self.m_used = [torch.cuda.Event() for _ in range(2)]

    @property
    def stream(self):
        """The compute stream: the one given, else the current one at each call
        (so a CUDA-graph capture records the exchanges too)."""
        return self._stream if self._stream is not None else torch.cuda.current_stream(self.dev)

    @property
    def copy(self):
        return self._copy if self.overlap else self.stream

    def local_ranks(self):
        return list(range(self.D))

    def attn_shard(self, k):
        return self.attn_packed[4 * self.Cb[k]:4 * self.Cb[k + 1]]

    def _copy_attn(self, k):
        b = k & 1
        src = self.attn_shard(k)
        dst = self.attn_rx[b][:src.shape[0]]
        with torch.cuda.stream(self.copy):
            if self.overlap and k >= 2:
                self.copy.wait_event(self.a_used[b])   # step k - 2 has read the slot
            dst.copy_(src)
            self.a_copied[b].record(self.copy)
        return dst

    def broadcast_attn_shard(self, k):
        b = k & 1
        if k >= 1:
            self.a_used[(k - 1) & 1].record(self.stream)   # step k - 1 is fully issued
        elif self.overlap:
            self.copy.wait_stream(self.stream)   # fork the copy stream from this point
        if not self.overlap or k == 0:
            dst = self._copy_attn(k)
        else:
            dst = self.attn_rx[b][:self.attn_shard(k).shape[0]]
        if self.overlap:
            self.stream.wait_event(self.a_copied[b])
            if k + 1 < self.D:
                self._copy_attn(k + 1)   # runs while step k computes
        return dst

    def all_gather_kv(self, k, parts):
        rows = self.cfg.S // self.D
        w = 2 * (self.Cb[k + 1] - self.Cb[k])
        out = self.kv_all[:, :w] if w == self.kv_all.shape[1] else \
            self.kv_all.view(-1)[:self.cfg.S * w].view(self.cfg.S, w)
        with torch.cuda.stream(self.stream):
            for r, p in parts.items():
                out[r * rows:(r + 1) * rows].copy_(p)
        return out

    def own_mlp_shard(self, r):
        return self.mlp_packed[3 * self.Ib[r]:3 * self.Ib[r + 1]]

    def ring_pass(self, t, held):
        b = (t + 1) & 1
        self.m_used[t & 1].record(self.stream)   # step t is fully issued
        out = {}
        with torch.cuda.stream(self.copy):
            # the held shards are the packed ones (t = 0) or this stream's own
            # earlier copies, so only the slots being overwritten need a wait
            if self.overlap and t >= 1:
                self.copy.wait_event(self.m_used[b])   # step t - 1 has read the slots
            for r in self.local_ranks():
                src = held[(r - 1) % self.D]
                dst = self.mlp_rx[r][b][:src.shape[0]]
                dst.copy_(src)
                out[r] = dst
            self.m_copied[b].record(self.copy)
        if self.overlap:
            # the copy runs beside step t's kernels, queued before this wait
            self.stream.wait_event(self.m_copied[b])
        return out

    # --- backward exchanges (on this GPU: copies, and the sums the collectives form)
    def ring_pass_with_grad(self, t, held, grad):
        if not hasattr(self, "grad_rx"):
            wI = max(self.Ib[s + 1] - self.Ib[s] for s in range(self.D))
            dev = self.attn_packed.device
            self.grad_rx = [[tsp.empty((3 * wI, self.cfg.d), torch.float32, dev) for _ in range(2)]
                            for _ in range(self.D)]
        b = (t + 1) & 1
        out_s, out_g = {}, {}
        with torch.cuda.stream(self.stream):
            for r in self.local_ranks():
                src, gsrc = held[(r - 1) % self.D], grad[(r - 1) % self.D]
                dst = self.mlp_rx[r][b][:src.shape[0]]
                gdst = self.grad_rx[r][b][:gsrc.shape[0]]
                dst.copy_(src)
                gdst.copy_(gsrc)
                out_s[r], out_g[r] = dst, gdst
        return out_s, out_g

    def keep_mlp_grads(self, grad):
        self.mlp_grads = {r: g.clone() for r, g in grad.items()}   # rank r: its own shard's gradient

    def reduce_scatter_kv(self, k, dkv):
        rows = self.cfg.S // self.D
        with torch.cuda.stream(self.stream):
            total = None
            for p in dkv.values():
                total = p.float() if total is None else total + p.float()
            return {r: total[r * rows:(r + 1) * rows].to(torch.float16).contiguous()
                    for r in self.local_ranks()}

    def reduce_attn_grad(self, k, gparts):
        if not hasattr(self, "attn_grads"):
            self.attn_grads = {}
        with torch.cuda.stream(self.stream):
            acc = None
            for g in gparts.values():
                acc = g.clone() if acc is None else acc + g
            self.attn_grads[k] = acc        # summed at the owner, rank k

    def all_reduce_gains(self, g):
        with torch.cuda.stream(self.stream):
            self.gains = sum(v for v in g.values())


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

    # --- backward (schedule.backward), after the forward ran on this object
    def set_dy(self, r, dy_r):
        if not hasattr(self, "dy"):
            dev, cfg = self.x[r].device, self.cfg
            b = shard_bounds(cfg.d, cfg.D)
            wC = max(hi - lo for lo, hi in zip(b[:-1], b[1:]))
            bi = shard_bounds(cfg.inter, cfg.D)
            wI = max(hi - lo for lo, hi in zip(bi[:-1], bi[1:]))
            f32 = torch.float32
            mk = lambda shape, dt=f32: {q: tsp.empty(shape, dt, dev) for q in self.x}
            self.dy = {}
            self.db, self.dh, self.da, self.dxr = (mk((self.rows, cfg.d)) for _ in range(4))
            self.dgm, self.dga = mk((cfg.d,)), mk((cfg.d,))
            self.dkv = mk((cfg.S, 2 * wC), torch.float16)
            self.gk = mk((4 * wC, cfg.d))
            self.g0 = mk((3 * wI, cfg.d))
        self.dy[r] = dy_r

    def mlp_bwd_step(self, r, t, shard, g):
        if g is None:                        # the first holder starts the shard's gradient
            g = self.g0[r][:shard.shape[0]]
            g.zero_()
        tsp.rank_mlp_bwd_step(self.cfg, r, t, self.h[r], self.W.g_mlp, shard, self.dy[r], g,
                              self.db[r], self.ws[r], self.stream)
        return g

    def mlp_bwd_finish(self, r):
        tsp.rank_mlp_bwd_finish(self.cfg, r, self.h[r], self.W.g_mlp, self.db[r], self.dy[r],
                                self.dh[r], self.dgm[r], self.ws[r], self.stream)

    def attn_bwd_heads(self, r, k, kv_all):
        Ck = kv_all.shape[1] // 2
        dkv = self.dkv[r].view(-1)[:self.cfg.S * 2 * Ck].view(self.cfg.S, 2 * Ck)
        gk = self.gk[r].view(-1)[:4 * Ck * self.cfg.d].view(4 * Ck, self.cfg.d)
        tsp.rank_attn_bwd_heads(self.cfg, r, k, kv_all, gk, dkv, self.ws[r], self.stream)
        return dkv

    def attn_bwd_weights(self, r, k, dkv_own):
        Ck = dkv_own.shape[1] // 2
        gk = self.gk[r].view(-1)[:4 * Ck * self.cfg.d].view(4 * Ck, self.cfg.d)
        tsp.rank_attn_bwd_weights(self.cfg, r, k, dkv_own, gk, self.da[r], self.ws[r], self.stream)
        return gk

    def attn_bwd_finish(self, r):
        tsp.rank_attn_bwd_finish(self.cfg, r, self.x[r], self.W.g_attn, self.da[r], self.dh[r],
                                 self.dxr[r], self.dga[r], self.ws[r], self.stream)

    def gain_grads(self, r):
        return torch.cat([self.dga[r], self.dgm[r]])

    def dx(self, r):
        return self.dxr[r]


def block_fwd_by_schedule(cfg, x_z, W: tsp.BlockWeights, stream=None, overlap=False):
    """y_z of the block computed rank by rank by the schedule, all D virtual
    ranks on this GPU (the same value tsp_block_fwd computes in one pass)."""
    rows = cfg.S // cfg.D
    comm = LocalComm(cfg, W, stream, overlap=overlap)
    ops = GpuRankOps(cfg, W, {r: x_z[r * rows:(r + 1) * rows] for r in range(cfg.D)}, stream)
    y = forward(comm, ops, cfg.D)
    return torch.cat([y[r] for r in range(cfg.D)], 0)


class OneRankComm(LocalComm):
    """Rank r0 alone, as one GPU of a D-GPU deployment sees the schedule: the
    broadcast shard and the ring shard arrive by copies into its receive
    buffers, and the all-gather copies every rank's K|V of the shard into the
    gathered buffer -- the other ranks' parts taken from `kv_shards` (each
    shard's K|V of all S rows, computed beforehand)."""

    def __init__(self, cfg, W, r0, kv_shards, overlap=False):
        super().__init__(cfg, W, overlap=overlap)
        self.r0, self.kv_shards = r0, kv_shards

    def local_ranks(self):
        return [self.r0]

    def all_gather_kv(self, k, parts):
        rows = self.cfg.S // self.D
        out = super().all_gather_kv(k, {})
        with torch.cuda.stream(self.stream):
            out.copy_(self.kv_shards[k])
            out[self.r0 * rows:(self.r0 + 1) * rows].copy_(parts[self.r0])
        return out

    def ring_pass(self, t, held):
        full = {r: self.own_mlp_shard(ring_shard(r, t, self.D)) for r in range(self.D)}
        full[self.r0] = held[self.r0]
        out = super().ring_pass(t, full)
        return {self.r0: out[self.r0]}


def block_bwd_by_schedule(cfg, x_z, dy_z, W: tsp.BlockWeights, stream=None):
    """The block's gradients computed rank by rank by the forward and backward
    schedule, all D virtual ranks on this GPU: the same dict as tsp.block_bwd
    (dx_z fp32 in the zigzag layout, weight and gain gradients fp32), each
    shard's weight gradient taken from its owner."""
    D, d, rows = cfg.D, cfg.d, cfg.S // cfg.D
    comm = LocalComm(cfg, W, stream)
    ops = GpuRankOps(cfg, W, {r: x_z[r * rows:(r + 1) * rows] for r in range(D)}, stream)
    forward(comm, ops, D)
    for r in range(D):
        ops.set_dy(r, dy_z[r * rows:(r + 1) * rows])
    dx = backward(comm, ops, D)
    dev = x_z.device
    g = {n: torch.zeros(shape, dtype=torch.float32, device=dev) for n, shape in
         (("dwq", (d, d)), ("dwk", (d, d)), ("dwv", (d, d)), ("dwo", (d, d)),
          ("dw1", (cfg.inter, d)), ("dw3", (cfg.inter, d)), ("dw2", (d, cfg.inter)))}
    Cb, Ib = shard_bounds(d, D), shard_bounds(cfg.inter, D)
    for k in range(D):
        n, C, a = Cb[k + 1] - Cb[k], slice(Cb[k], Cb[k + 1]), comm.attn_grads[k]
        g["dwq"][C], g["dwk"][C], g["dwv"][C] = a[:n], a[n:2 * n], a[2 * n:3 * n]
        g["dwo"][:, C] = a[3 * n:4 * n].T
        m, I, b = Ib[k + 1] - Ib[k], slice(Ib[k], Ib[k + 1]), comm.mlp_grads[k]
        g["dw1"][I], g["dw3"][I] = b[:m], b[m:2 * m]
        g["dw2"][:, I] = b[2 * m:3 * m].T
    g["dg_attn"], g["dg_mlp"] = comm.gains[:d].clone(), comm.gains[d:].clone()
    g["dx"] = torch.cat([dx[r] for r in range(D)], 0)
    return g


def _time_main():
    """Times the 7B-shaped block forward on this GPU and prints one JSON line:
    the one-pass tsp_block_fwd (all D ranks' work), and one rank's schedule
    (what one GPU of a D-GPU deployment computes: 1/D of the work) replayed
    from a CUDA graph, with its weight transfers on the compute stream and on
    a copy stream.  python -m folded_tensor_sequence_zigzag_gb300.schedule"""
    import argparse
    import json

    from .inputs import BlockShape, make_block_inputs

    ap = argparse.ArgumentParser()
    ap.add_argument("--S", type=int, default=16384)
    ap.add_argument("--D", type=int, default=8)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    a = ap.parse_args()
    shape = BlockShape(S=a.S, d=4096, H=32, inter=11008, D=a.D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=0)
    cfg = tsp.make_cfg(shape.S, shape.d, shape.H, shape.inter, shape.D, torch.bfloat16, shape.eps)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    xz = tsp.zigzag_permute(inp["x"].cuda(), a.D)
    rows = a.S // a.D

    def timed(fn, graph):
        for _ in range(a.warmup):
            fn()
        torch.cuda.synchronize()
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            fn = g.replay
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(a.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / a.steps

    # every shard's K|V of all rows, from one full run of the schedule
    class Keep(LocalComm):
        kept = []

        def all_gather_kv(self, k, parts):
            out = super().all_gather_kv(k, parts)
            self.kept.append(out.clone())
            return out

    all_ops = GpuRankOps(cfg, W, {r: xz[r * rows:(r + 1) * rows] for r in range(a.D)})
    forward(Keep(cfg, W), all_ops, a.D)
    kv_shards = Keep.kept

    res = {"workload": f"7B-shaped block forward, S={a.S}, D={a.D}",
           "one_pass_ms": timed(lambda: tsp.block_fwd(cfg, xz, W), False)}
    res["one_pass_per_rank_ms"] = res["one_pass_ms"] / a.D
    y_ref = all_ops.output(0).clone()
    for overlap in (False, True):
        comm = OneRankComm(cfg, W, 0, kv_shards, overlap=overlap)
        ops = GpuRankOps(cfg, W, {0: xz[:rows]})
        key = "one_rank_overlap_ms" if overlap else "one_rank_serial_ms"
        res[key] = timed(lambda: forward(comm, ops, a.D), True)
        if not torch.equal(ops.output(0), y_ref):
            raise RuntimeError("one rank's schedule differs from the full run")
    # the training step: one pass (tsp_block_fwd + tsp_block_bwd) against all D
    # ranks' schedule steps run one after another on this GPU (so 1/D of it is
    # one rank's work), both replayed from CUDA graphs
    dyz = tsp.zigzag_permute(make_block_inputs(shape, torch.bfloat16, seed=1, with_dy=True)["dy"]
                             .cuda(), a.D)
    saved = tsp.empty(tsp.saved_bytes(cfg), torch.uint8, "cuda")

    def one_pass_train():
        tsp.block_fwd(cfg, xz, W, saved=saved)
        tsp.block_bwd(cfg, xz, dyz, saved, W)

    res["train_one_pass_per_rank_ms"] = timed(one_pass_train, True) / a.D
    res["train_by_rank_per_rank_ms"] = timed(
        lambda: block_bwd_by_schedule(cfg, xz, dyz, W), True) / a.D
    if tsp.device_status() != tsp.TSP_OK:
        raise RuntimeError("device status not OK")
    print(json.dumps(res))


if __name__ == "__main__":
    _time_main()
