"""The TSP forward schedule with every virtual rank in its own process.

"Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer
Training & Inference" (gist.science summary), section 2, "Runtime schedules":
the owner of each packed W_Q/W_K/W_V/W_O shard broadcasts it, the ranks
all-gather the K/V of their zigzag rows, and the W_1/W_3/W_2 shards travel
around a ring.  Here D processes share one GPU; each holds only its own
attention and MLP shards and its own 2c zigzag rows, runs its steps through
the per-rank calls (tsp_rank_attn_project / tsp_rank_attn_heads /
tsp_rank_mlp_step), and exchanges shards and K|V through host memory over
gloo between its kernel launches (no kernel waits on another process).  The
gathered output is compared with the float64 oracle and with the one-process
tsp_block_fwd.
"""
import os
import socket
import types

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300 import tsp
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, make_block_inputs
from tests.helpers import assert_bf16_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    return tsp.load()


def _bytes(t):
    """A tensor's bytes as a flat uint8 CPU tensor (what gloo carries)."""
    return t.contiguous().view(torch.uint8).reshape(-1).cpu()


class HostStagedComm:
    """Rank `rank` of D in its own process: each exchange copies the device
    data to host memory, runs the gloo collective, and copies the result back
    to the device."""

    def __init__(self, rank, D, own_attn, own_mlp, Cb, Ib, d, dev):
        self.rank, self.D, self.d, self.dev = rank, D, d, dev
        self.own_attn, self.own_mlp = own_attn, own_mlp
        self.Cb, self.Ib = Cb, Ib
        self.ring_log = []
        self.bring_log = []

    def local_ranks(self):
        return [self.rank]

    def broadcast_attn_shard(self, k):
        rows = 4 * (self.Cb[k + 1] - self.Cb[k])
        if self.rank == k:
            buf = _bytes(self.own_attn)
        else:
            buf = torch.empty(rows * self.d * 2, dtype=torch.uint8)
        dist.broadcast(buf, src=k)
        return buf.view(torch.bfloat16).view(rows, self.d).to(self.dev)

    def all_gather_kv(self, k, parts):
        mine = parts[self.rank]
        w = mine.shape[1]
        flat = _bytes(mine)
        lst = [torch.empty_like(flat) for _ in range(self.D)]
        dist.all_gather(lst, flat)
        # rank q's rows land at q * 2c: the zigzag row order
        return torch.cat(lst, 0).view(torch.float16).view(-1, w).to(self.dev)

    def own_mlp_shard(self, r):
        return self.own_mlp

    def ring_pass(self, t, held):
        from folded_tensor_sequence_zigzag_gb300 import schedule
        src = _bytes(held[self.rank])
        s_in = schedule.ring_shard(self.rank, t + 1, self.D)   # what arrives from rank r - 1
        rows = 3 * (self.Ib[s_in + 1] - self.Ib[s_in])
        rx = torch.empty(rows * self.d * 2, dtype=torch.uint8)
        ops = [dist.P2POp(dist.isend, src, (self.rank + 1) % self.D),
               dist.P2POp(dist.irecv, rx, (self.rank - 1) % self.D)]
        for req in dist.batch_isend_irecv(ops):
            req.wait()
        self.ring_log.append(s_in)
        return {self.rank: rx.view(torch.bfloat16).view(rows, self.d).to(self.dev)}

    # --- backward exchanges
    def ring_pass_with_grad(self, t, held, grad):
        from folded_tensor_sequence_zigzag_gb300 import schedule
        src, gsrc = _bytes(held[self.rank]), grad[self.rank].float().cpu().contiguous()
        s_in = schedule.ring_shard(self.rank, t + 1, self.D)
        rows = 3 * (self.Ib[s_in + 1] - self.Ib[s_in])
        rx = torch.empty(rows * self.d * 2, dtype=torch.uint8)
        grx = torch.empty(rows, self.d, dtype=torch.float32)
        nxt, prev = (self.rank + 1) % self.D, (self.rank - 1) % self.D
        ops = [dist.P2POp(dist.isend, src, nxt), dist.P2POp(dist.irecv, rx, prev),
               dist.P2POp(dist.isend, gsrc, nxt), dist.P2POp(dist.irecv, grx, prev)]
        for req in dist.batch_isend_irecv(ops):
            req.wait()
        self.bring_log.append(s_in)
        return ({self.rank: rx.view(torch.bfloat16).view(rows, self.d).to(self.dev)},
                {self.rank: grx.to(self.dev)})

    def keep_mlp_grads(self, grad):
        self.mlp_grad = grad[self.rank].cpu()

    def reduce_scatter_kv(self, k, dkv):
        full = dkv[self.rank].float().cpu().contiguous()
        dist.all_reduce(full)                       # the sum over the query ranks
        rows = full.shape[0] // self.D
        own = full[self.rank * rows:(self.rank + 1) * rows].to(torch.float16).contiguous()
        return {self.rank: own.to(self.dev)}

    def reduce_attn_grad(self, k, gparts):
        t = gparts[self.rank].cpu().contiguous()
        dist.reduce(t, dst=k)
        if self.rank == k:
            self.attn_grad = t

    def all_reduce_gains(self, g):
        t = g[self.rank].cpu().contiguous()
        dist.all_reduce(t)
        self.gains = t


def _worker(rank, D, port, q, dims, seed):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=D)
        from folded_tensor_sequence_zigzag_gb300 import schedule
        S, d, H, I = dims
        dev = torch.device("cuda", 0)
        shape = BlockShape(S=S, d=d, H=H, inter=I, D=D)
        inp = make_block_inputs(shape, torch.bfloat16, seed=seed)
        cfg = tsp.make_cfg(S, d, H, I, D, torch.bfloat16, shape.eps)
        W = tsp.BlockWeights.from_dict(inp, dev)
        Cb, Ib = schedule.shard_bounds(d, D), schedule.shard_bounds(I, D)
        # the owner's packing step; afterwards this process keeps only its own shards
        own_attn = tsp.pack_attn_shards(cfg, W)[4 * Cb[rank]:4 * Cb[rank + 1]].clone()
        own_mlp = tsp.pack_mlp_shards(cfg, W)[3 * Ib[rank]:3 * Ib[rank + 1]].clone()
        # the norm gains are replicated on every rank
        gains = types.SimpleNamespace(g_attn=W.g_attn, g_mlp=W.g_mlp)
        del W
        rows = S // D
        x_r = tsp.zigzag_permute(inp["x"].to(dev), D)[rank * rows:(rank + 1) * rows].clone()
        comm = HostStagedComm(rank, D, own_attn, own_mlp, Cb, Ib, d, dev)
        ops = schedule.GpuRankOps(cfg, gains, {rank: x_r})
        y = schedule.forward(comm, ops, D)[rank]
        torch.cuda.synchronize(dev)
        status = tsp.device_status()
        q.put((rank, y.cpu(), status, comm.ring_log, None))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # noqa: BLE001
        q.put((rank, None, None, None, repr(e)))


def _bwd_worker(rank, D, port, q, dims, seed):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=D)
        from folded_tensor_sequence_zigzag_gb300 import schedule
        S, d, H, I = dims
        dev = torch.device("cuda", 0)
        shape = BlockShape(S=S, d=d, H=H, inter=I, D=D)
        inp = make_block_inputs(shape, torch.bfloat16, seed=seed, with_dy=True)
        cfg = tsp.make_cfg(S, d, H, I, D, torch.bfloat16, shape.eps)
        W = tsp.BlockWeights.from_dict(inp, dev)
        Cb, Ib = schedule.shard_bounds(d, D), schedule.shard_bounds(I, D)
        own_attn = tsp.pack_attn_shards(cfg, W)[4 * Cb[rank]:4 * Cb[rank + 1]].clone()
        own_mlp = tsp.pack_mlp_shards(cfg, W)[3 * Ib[rank]:3 * Ib[rank + 1]].clone()
        gains = types.SimpleNamespace(g_attn=W.g_attn, g_mlp=W.g_mlp)
        del W
        rows = S // D
        x_r = tsp.zigzag_permute(inp["x"].to(dev), D)[rank * rows:(rank + 1) * rows].clone()
        dy_r = tsp.zigzag_permute(inp["dy"].to(dev), D)[rank * rows:(rank + 1) * rows].clone()
        comm = HostStagedComm(rank, D, own_attn, own_mlp, Cb, Ib, d, dev)
        ops = schedule.GpuRankOps(cfg, gains, {rank: x_r})
        schedule.forward(comm, ops, D)
        ops.set_dy(rank, dy_r)
        dx_r = schedule.backward(comm, ops, D)[rank]
        torch.cuda.synchronize(dev)
        status = tsp.device_status()
        q.put((rank, dx_r.cpu(), comm.attn_grad, comm.mlp_grad, comm.gains, status,
               comm.bring_log, None))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # noqa: BLE001
        q.put((rank, None, None, None, None, None, None, repr(e)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("S,d,H,I,D", [(4096, 1024, 8, 2048, 2), (3072, 768, 6, 1536, 3)])
def test_schedule_one_process_per_rank(S, d, H, I, D):
    seed = 40 + D
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, D, port, q, (S, d, H, I), seed)) for r in range(D)]
    for p in procs:
        p.start()
    res = [q.get(timeout=900) for _ in range(D)]
    for p in procs:
        p.join(timeout=120)
    res.sort(key=lambda t: t[0])
    for rank, _, status, ring, exc in res:
        assert exc is None, f"rank {rank}: {exc}"
        assert status == tsp.TSP_OK, (rank, status)
        # rank r receives shard (r - t) mod D from rank r - 1 at ring step t
        assert ring == [(rank - t) % D for t in range(1, D)], (rank, ring)
    yz = torch.cat([y for _, y, _, _, _ in res], 0)
    y = tsp.zigzag_permute(yz.cuda(), D, inverse=True).cpu()

    shape = BlockShape(S=S, d=d, H=H, inter=I, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=seed)
    ref, _ = O.block_fwd(inp["x"], inp, H, shape.eps)
    assert_bf16_close(y, ref, f"schedule over {D} processes")

    # the same block in one pass on this GPU: equal up to the final bf16 rounding
    cfg = tsp.make_cfg(S, d, H, I, D, torch.bfloat16, shape.eps)
    W = tsp.BlockWeights.from_dict(inp, "cuda")
    y1 = tsp.zigzag_permute(tsp.block_fwd(cfg, tsp.zigzag_permute(inp["x"].cuda(), D), W), D,
                            inverse=True).cpu()
    a, b = O.f64(y), O.f64(y1)
    rms = float(np.sqrt(np.mean(b * b)))
    diff = np.abs(a - b)
    assert np.all(diff <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-3 * rms)
    assert float(diff.sum() / np.abs(b).sum()) <= 1e-3


@pytest.mark.parametrize("S,d,H,I,D", [(4096, 1024, 8, 2048, 2), (3072, 768, 6, 1536, 3)])
def test_backward_schedule_one_process_per_rank(S, d, H, I, D):
    """The training step with every rank its own process on the one GPU: the
    forward schedule, then its reverse with host-staged gloo exchanges (the
    gradient-carrying ring, the dK|dV reduce-scatter, each shard's gradient
    reduced to its owner, the gains all-reduced).  dx from every rank's rows
    and every weight and gain gradient from the owners against the dense
    float64 backward."""
    seed = 50 + D
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bwd_worker, args=(r, D, port, q, (S, d, H, I), seed))
             for r in range(D)]
    for p in procs:
        p.start()
    res = [q.get(timeout=900) for _ in range(D)]
    for p in procs:
        p.join(timeout=120)
    res.sort(key=lambda t: t[0])
    for rank, *_, status, bring, exc in res:
        assert exc is None, f"rank {rank}: {exc}"
        assert status == tsp.TSP_OK, (rank, status)
        assert bring == [(rank - t) % D for t in range(1, D + 1)], (rank, bring)
    shape = BlockShape(S=S, d=d, H=H, inter=I, D=D)
    inp = make_block_inputs(shape, torch.bfloat16, seed=seed, with_dy=True)
    ref = O.block_bwd(inp["x"], inp, inp["dy"], H, shape.eps)
    c = S // (2 * D)
    pos = O.zigzag_positions(S, D)
    Cb, Ib = O.shard_bounds(d, D), O.shard_bounds(I, D)
    got = {k: np.zeros_like(v) for k, v in ref.items()}
    for rank, dx_r, ag, mg, gains, *_ in res:
        got["dx"][pos[rank * 2 * c:(rank + 1) * 2 * c]] = O.f64(dx_r)
        ag, mg = O.f64(ag), O.f64(mg)
        C, n = slice(Cb[rank], Cb[rank + 1]), Cb[rank + 1] - Cb[rank]
        got["dwq"][C], got["dwk"][C], got["dwv"][C] = ag[:n], ag[n:2 * n], ag[2 * n:3 * n]
        got["dwo"][:, C] = ag[3 * n:].T
        Ik, m = slice(Ib[rank], Ib[rank + 1]), Ib[rank + 1] - Ib[rank]
        got["dw1"][Ik], got["dw3"][Ik] = mg[:m], mg[m:2 * m]
        got["dw2"][:, Ik] = mg[2 * m:].T
        got["dg_attn"], got["dg_mlp"] = O.f64(gains)[:d], O.f64(gains)[d:]
    for k, v in ref.items():
        assert_bf16_close(torch.from_numpy(got[k]), v, f"{k} over {D} processes")
