"""Thin ctypes binding of libtsp.so (include/tsp.h).

Argument marshalling only: torch tensors give device pointers and the current
stream; every step of the block runs in the library's CUDA kernels.  There is
no fallback: if the library is missing or no GPU is present the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtsp.so")
# the checked build (build.build(check=True)): the same library with every
# computed global index tested before its access (TSP_ERR_BOUNDS)
CHECK_LIB_PATH = os.path.join(_PKG, "libtsp_check.so")

(TSP_OK, TSP_ERR_INVALID_ARG, TSP_ERR_UNSUPPORTED, TSP_ERR_CUDA, TSP_ERR_TIMEOUT, TSP_ERR_RANGE,
 TSP_ERR_BOUNDS) = range(7)
TSP_F32, TSP_BF16 = 0, 1
TSP_OP_ATTN_FWD, TSP_OP_MLP_FWD, TSP_OP_BLOCK_FWD, TSP_OP_BLOCK_BWD, TSP_OP_BLOCK_FWD_TRAIN = range(5)
TSP_OP_PREPARED = 16

EXPORTED = ("tsp_zigzag_permute", "tsp_rmsnorm_fwd", "tsp_workspace_bytes", "tsp_saved_bytes",
            "tsp_attn_block_fwd", "tsp_gated_mlp_fwd", "tsp_block_fwd", "tsp_block_bwd",
            "tsp_pack_attn_shards", "tsp_device_status", "tsp_strerror", "tsp_num_sms",
            "tsp_profile_enable", "tsp_profile_report", "tsp_launch_count",
            "tsp_gated_mlp_fwd_noalloc", "tsp_stack_saved_bytes", "tsp_stack_workspace_bytes",
            "tsp_stack_fwd", "tsp_stack_bwd", "tsp_rank_memory", "tsp_kv_cache_bytes",
            "tsp_decode_workspace_bytes", "tsp_block_prefill", "tsp_block_decode",
            "tsp_debug_skip_stage", "tsp_block_weights_bytes", "tsp_block_weights_prepare",
            "tsp_block_fwd_prepared", "tsp_block_bwd_prepared", "tsp_stack_fwd_prepared",
            "tsp_stack_bwd_prepared", "tsp_pack_mlp_shards", "tsp_rank_workspace_bytes",
            "tsp_rank_attn_project", "tsp_rank_attn_heads", "tsp_rank_mlp_step",
            "tsp_rank_mlp_bwd_step", "tsp_rank_mlp_bwd_finish", "tsp_rank_attn_bwd_heads",
            "tsp_rank_attn_bwd_weights", "tsp_rank_attn_bwd_finish")
DECODE_MAX_T = 8   # TSP_DECODE_MAX_T


class TspError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (status {code})")


class Cfg(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int64), ("d", ctypes.c_int32), ("H", ctypes.c_int32),
                ("dh", ctypes.c_int32), ("inter", ctypes.c_int32), ("D", ctypes.c_int32),
                ("eps", ctypes.c_float), ("dtype", ctypes.c_int32), ("rope_base", ctypes.c_float),
                ("Hkv", ctypes.c_int32), ("mlp_tile", ctypes.c_int32)]


class AttnW(ctypes.Structure):
    _fields_ = [("wq", ctypes.c_void_p), ("wk", ctypes.c_void_p), ("wv", ctypes.c_void_p),
                ("wo", ctypes.c_void_p), ("g_attn", ctypes.c_void_p)]


class MlpW(ctypes.Structure):
    _fields_ = [("w1", ctypes.c_void_p), ("w3", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("g_mlp", ctypes.c_void_p), ("add_residual", ctypes.c_int32)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtsp.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run folded_tensor_sequence_zigzag_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "tsp_zigzag_permute": (i32, [vp, vp, i64, i32, i64, i32, vp]),
        "tsp_rmsnorm_fwd": (i32, [vp, vp, vp, vp, i64, i32, f32, i32, vp]),
        "tsp_workspace_bytes": (sz, [P(Cfg), i32]),
        "tsp_saved_bytes": (sz, [P(Cfg)]),
        "tsp_attn_block_fwd": (i32, [P(Cfg), vp, P(AttnW), vp, vp, sz, vp]),
        "tsp_gated_mlp_fwd": (i32, [P(Cfg), vp, P(MlpW), vp, vp, sz, vp]),
        "tsp_block_fwd": (i32, [P(Cfg), vp, P(AttnW), P(MlpW), vp, vp, vp, sz, vp]),
        "tsp_block_bwd": (i32, [P(Cfg), vp, vp, vp, P(AttnW), P(MlpW), vp] + [vp] * 9 + [vp, sz, vp]),
        "tsp_pack_attn_shards": (i32, [P(Cfg), P(AttnW), vp, vp]),
        "tsp_device_status": (i32, [vp, i32]),
        "tsp_strerror": (ctypes.c_char_p, [i32]),
        "tsp_num_sms": (i32, []),
        "tsp_profile_enable": (None, [i32]),
        "tsp_profile_report": (i32, [ctypes.c_char_p, i64]),
        "tsp_launch_count": (i64, []),
        "tsp_debug_skip_stage": (None, [i32]),
        "tsp_block_weights_bytes": (sz, [P(Cfg)]),
        "tsp_block_weights_prepare": (i32, [P(Cfg), P(AttnW), P(MlpW), vp, vp]),
        "tsp_block_fwd_prepared": (i32, [P(Cfg), vp, vp, P(AttnW), P(MlpW), vp, vp, vp, sz, vp]),
        "tsp_block_bwd_prepared": (i32, [P(Cfg), vp, vp, vp, vp, P(AttnW), P(MlpW), vp] + [vp] * 9
                                   + [vp, sz, vp]),
        "tsp_stack_fwd_prepared": (i32, [P(Cfg), i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_stack_bwd_prepared": (i32, [P(Cfg), i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_pack_mlp_shards": (i32, [P(Cfg), P(MlpW), vp, vp]),
        "tsp_rank_workspace_bytes": (sz, [P(Cfg)]),
        "tsp_rank_attn_project": (i32, [P(Cfg), i32, i32, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_rank_attn_heads": (i32, [P(Cfg), i32, i32, vp, vp, vp, vp, sz, vp]),
        "tsp_rank_mlp_step": (i32, [P(Cfg), i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_rank_mlp_bwd_step": (i32, [P(Cfg), i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_rank_mlp_bwd_finish": (i32, [P(Cfg), i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_rank_attn_bwd_heads": (i32, [P(Cfg), i32, i32, vp, vp, vp, vp, sz, vp]),
        "tsp_rank_attn_bwd_weights": (i32, [P(Cfg), i32, i32, vp, vp, vp, vp, sz, vp]),
        "tsp_rank_attn_bwd_finish": (i32, [P(Cfg), i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_gated_mlp_fwd_noalloc": (i32, [P(Cfg), vp, P(MlpW), vp, vp]),
        "tsp_stack_saved_bytes": (sz, [P(Cfg), i32]),
        "tsp_stack_workspace_bytes": (sz, [P(Cfg), i32, i32]),
        "tsp_stack_fwd": (i32, [P(Cfg), i32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_stack_bwd": (i32, [P(Cfg), i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "tsp_rank_memory": (i32, [P(Cfg), i32, i32, i32, P(RankMem)]),
        "tsp_kv_cache_bytes": (sz, [P(Cfg), i64]),
        "tsp_decode_workspace_bytes": (sz, [P(Cfg), i32, i64]),
        "tsp_block_prefill": (i32, [P(Cfg), vp, P(AttnW), P(MlpW), vp, vp, i64, vp, sz, vp]),
        "tsp_block_decode": (i32, [P(Cfg), vp, i32, i64, P(AttnW), P(MlpW), vp, vp, i64, vp, sz,
                                   vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().tsp_strerror(code).decode()
    except Exception:  # noqa: BLE001
        return f"status {code}"


def _check(code: int, where: str):
    if code != TSP_OK:
        raise TspError(code, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must live on the GPU")


class RankMem(ctypes.Structure):
    _fields_ = [("weights", ctypes.c_double), ("activations", ctypes.c_double),
                ("transient", ctypes.c_double), ("total", ctypes.c_double),
                ("devices", ctypes.c_double)]


TSP_MEM_TSP, TSP_MEM_DP, TSP_MEM_TP, TSP_MEM_SP, TSP_MEM_TP_SP = range(5)


@dataclass
class BlockWeights:
    """Device tensors of one block (nn.Linear layout [out, in])."""
    wq: torch.Tensor
    wk: torch.Tensor
    wv: torch.Tensor
    wo: torch.Tensor
    w1: torch.Tensor
    w3: torch.Tensor
    w2: torch.Tensor
    g_attn: torch.Tensor
    g_mlp: torch.Tensor

    @classmethod
    def from_dict(cls, d: dict, device="cuda"):
        return cls(**{k: d[k].to(device).contiguous() for k in
                      ("wq", "wk", "wv", "wo", "w1", "w3", "w2", "g_attn", "g_mlp")})

    def attn(self) -> AttnW:
        return AttnW(_ptr(self.wq), _ptr(self.wk), _ptr(self.wv), _ptr(self.wo), _ptr(self.g_attn))

    def mlp(self, norm=True, residual=True) -> MlpW:
        return MlpW(_ptr(self.w1), _ptr(self.w3), _ptr(self.w2), _ptr(self.g_mlp) if norm else None,
                    1 if residual else 0)


def make_cfg(S, d, H, inter, D, dtype: torch.dtype, eps=1e-6, rope_base=0.0, Hkv=0,
             mlp_tile=0) -> Cfg:
    return Cfg(int(S), int(d), int(H), int(d // H), int(inter), int(D), float(eps),
               TSP_BF16 if dtype == torch.bfloat16 else TSP_F32, float(rope_base), int(Hkv),
               int(mlp_tile))


def _grad_shapes(cfg: Cfg) -> dict:
    d, I = cfg.d, cfg.inter
    dkv = (cfg.Hkv if cfg.Hkv > 0 else cfg.H) * cfg.dh
    return {"dwq": (d, d), "dwk": (dkv, d), "dwv": (dkv, d), "dwo": (d, d), "dw1": (I, d),
            "dw3": (I, d), "dw2": (d, I), "dg_attn": (d,), "dg_mlp": (d,)}


def workspace_bytes(cfg: Cfg, op: int) -> int:
    return int(load().tsp_workspace_bytes(ctypes.byref(cfg), op))


def saved_bytes(cfg: Cfg) -> int:
    return int(load().tsp_saved_bytes(ctypes.byref(cfg)))


# Poison mode (for tests): every buffer the binding allocates -- outputs,
# gradients, workspaces, caches -- starts as all-ones bytes (NaN in fp32,
# bf16 and fp16) instead of whatever the caching allocator hands back, so an
# element the library fails to write cannot pass as a previous call's value.
POISON = False


def empty(shape, dtype, device) -> torch.Tensor:
    """An uninitialised buffer, or a poisoned one while POISON is set."""
    t = torch.empty(shape, dtype=dtype, device=device)
    if POISON:
        t.view(torch.uint8).fill_(0xFF)
    return t


def empty_like(t: torch.Tensor) -> torch.Tensor:
    return empty(t.shape, t.dtype, t.device)


def _ws(nbytes: int, device) -> torch.Tensor:
    return empty(max(nbytes, 256), torch.uint8, device)


def zigzag_permute(src: torch.Tensor, D: int, inverse: bool = False, out=None, stream=None):
    """Rows of src (global order) -> zigzag rank-major order (or back)."""
    _require_cuda(src)
    src = src.contiguous()
    out = empty_like(src) if out is None else out
    S = src.shape[0]
    row_bytes = src.numel() // max(S, 1) * src.element_size()
    _check(load().tsp_zigzag_permute(_ptr(src), _ptr(out), S, D, row_bytes, 1 if inverse else 0,
                                     _stream(stream)), "tsp_zigzag_permute")
    return out


def rmsnorm_fwd(u: torch.Tensor, g: torch.Tensor, eps: float = 1e-6, with_rstd=False, stream=None):
    _require_cuda(u, g)
    out = empty_like(u)
    rstd = empty(u.shape[0], torch.float32, u.device) if with_rstd else None
    dt = TSP_BF16 if u.dtype == torch.bfloat16 else TSP_F32
    _check(load().tsp_rmsnorm_fwd(_ptr(u), _ptr(g), _ptr(out), _ptr(rstd), u.shape[0], u.shape[1],
                                  eps, dt, _stream(stream)), "tsp_rmsnorm_fwd")
    return (out, rstd) if with_rstd else out


def attn_block_fwd(cfg: Cfg, x_z, W: BlockWeights, out=None, ws=None, stream=None):
    _require_cuda(x_z)
    out = empty_like(x_z) if out is None else out
    nb = workspace_bytes(cfg, TSP_OP_ATTN_FWD)
    ws = _ws(nb, x_z.device) if ws is None else ws
    aw = W.attn()
    _check(load().tsp_attn_block_fwd(ctypes.byref(cfg), _ptr(x_z), ctypes.byref(aw), _ptr(out),
                                     _ptr(ws), ws.numel(), _stream(stream)), "tsp_attn_block_fwd")
    return out


def gated_mlp_fwd(cfg: Cfg, h_z, W: BlockWeights, norm=True, residual=True, out=None, ws=None,
                  stream=None):
    _require_cuda(h_z)
    out = empty_like(h_z) if out is None else out
    nb = workspace_bytes(cfg, TSP_OP_MLP_FWD)
    ws = _ws(nb, h_z.device) if ws is None else ws
    mw = W.mlp(norm, residual)
    _check(load().tsp_gated_mlp_fwd(ctypes.byref(cfg), _ptr(h_z), ctypes.byref(mw), _ptr(out),
                                    _ptr(ws), ws.numel(), _stream(stream)), "tsp_gated_mlp_fwd")
    return out


def block_weights_bytes(cfg: Cfg) -> int:
    return int(load().tsp_block_weights_bytes(ctypes.byref(cfg)))


def prepare_weights(cfg: Cfg, W: BlockWeights, out=None, stream=None):
    """The block's fp16 operand copies, converted once (bf16 configurations;
    None for fp32, which reads the weights as they are).  ``out``: a buffer of
    block_weights_bytes(cfg) bytes to refill instead of a new one."""
    nb = block_weights_bytes(cfg)
    if nb == 0:
        return None
    prep = _ws(nb, W.wq.device) if out is None else out
    aw, mw = W.attn(), W.mlp()
    _check(load().tsp_block_weights_prepare(ctypes.byref(cfg), ctypes.byref(aw), ctypes.byref(mw),
                                            _ptr(prep), _stream(stream)), "tsp_block_weights_prepare")
    return prep


def block_fwd(cfg: Cfg, x_z, W: BlockWeights, saved=None, out=None, ws=None, stream=None,
              prep=None):
    """y_z = block(x_z).  Pass ``saved`` (uint8, saved_bytes(cfg)) to keep activations for bwd,
    ``prep`` (prepare_weights) to use weights converted once.

    Without ``prep`` the workspace holds the fp16 operand copies of the weights;
    without ``saved`` it also holds the activations."""
    _require_cuda(x_z)
    out = empty_like(x_z) if out is None else out
    pf = TSP_OP_PREPARED if prep is not None else 0
    if ws is None:
        op = TSP_OP_BLOCK_FWD if saved is None else TSP_OP_BLOCK_FWD_TRAIN
        ws = _ws(workspace_bytes(cfg, op | pf), x_z.device)
    aw, mw = W.attn(), W.mlp()
    if prep is not None:
        _check(load().tsp_block_fwd_prepared(ctypes.byref(cfg), _ptr(x_z), _ptr(prep),
                                             ctypes.byref(aw), ctypes.byref(mw), _ptr(out),
                                             _ptr(saved), _ptr(ws), ws.numel(), _stream(stream)),
               "tsp_block_fwd_prepared")
        return out
    _check(load().tsp_block_fwd(ctypes.byref(cfg), _ptr(x_z), ctypes.byref(aw), ctypes.byref(mw),
                                _ptr(out), _ptr(saved), _ptr(ws), 0 if ws is None else ws.numel(),
                                _stream(stream)), "tsp_block_fwd")
    return out


def kv_cache_bytes(cfg: Cfg, rows_cap: int) -> int:
    return int(load().tsp_kv_cache_bytes(ctypes.byref(cfg), int(rows_cap)))


def decode_workspace_bytes(cfg: Cfg, T: int, rows_cap: int) -> int:
    return int(load().tsp_decode_workspace_bytes(ctypes.byref(cfg), int(T), int(rows_cap)))


class KVCache:
    """Device KV cache of ``rows_cap`` rows for one block (layout in tsp.h):
    the prompt's rows in zigzag order, then the decoded tokens'."""

    def __init__(self, cfg: Cfg, rows_cap: int, device="cuda"):
        nb = kv_cache_bytes(cfg, rows_cap)
        if nb == 0:
            raise ValueError("invalid configuration or capacity for a KV cache")
        self.buf = empty(nb, torch.uint8, device)
        self.rows_cap = int(rows_cap)
        self.n = 0          # rows filled

    def view(self, cfg: Cfg) -> torch.Tensor:
        """[rows_cap, 2*Hkv*dh] view in the internal element type (K | V)."""
        dt = torch.float16 if cfg.dtype == TSP_BF16 else torch.float32
        return self.buf.view(dt).view(self.rows_cap, -1)


def block_prefill(cfg: Cfg, x_z, W: BlockWeights, cache: KVCache, out=None, ws=None, stream=None):
    """Inference forward over the S prompt tokens (zigzag order) that also
    fills cache rows [0, S) with their K and V."""
    _require_cuda(x_z)
    out = empty_like(x_z) if out is None else out
    if ws is None:
        ws = _ws(workspace_bytes(cfg, TSP_OP_BLOCK_FWD), x_z.device)
    aw, mw = W.attn(), W.mlp()
    _check(load().tsp_block_prefill(ctypes.byref(cfg), _ptr(x_z), ctypes.byref(aw), ctypes.byref(mw),
                                    _ptr(out), _ptr(cache.buf), cache.rows_cap, _ptr(ws), ws.numel(),
                                    _stream(stream)), "tsp_block_prefill")
    cache.n = cfg.S
    return out


def block_decode(cfg: Cfg, x, W: BlockWeights, cache: KVCache, out=None, ws=None, stream=None):
    """y [T, d] of T new tokens (position order) at positions cache.n ..;
    appends their K/V to the cache."""
    _require_cuda(x)
    T = x.shape[0]
    out = empty_like(x) if out is None else out
    if ws is None:
        ws = _ws(decode_workspace_bytes(cfg, T, cache.rows_cap), x.device)
    aw, mw = W.attn(), W.mlp()
    _check(load().tsp_block_decode(ctypes.byref(cfg), _ptr(x), T, cache.n, ctypes.byref(aw),
                                   ctypes.byref(mw), _ptr(out), _ptr(cache.buf), cache.rows_cap,
                                   _ptr(ws), ws.numel(), _stream(stream)), "tsp_block_decode")
    cache.n += T
    return out


GRAD_NAMES = ("dwq", "dwk", "dwv", "dwo", "dw1", "dw3", "dw2", "dg_attn", "dg_mlp")


def block_bwd(cfg: Cfg, x_z, dy_z, saved, W: BlockWeights, ws=None, stream=None,
              prep=None) -> dict:
    """Gradients of sum(dy * y), all fp32: dx_z (zigzag order) and the weight/gain grads."""
    _require_cuda(x_z, dy_z, saved)
    dev = x_z.device
    shapes = _grad_shapes(cfg)
    g = {k: empty(shapes[k], torch.float32, dev) for k in GRAD_NAMES}
    g["dx"] = empty(x_z.shape, torch.float32, dev)
    pf = TSP_OP_PREPARED if prep is not None else 0
    ws = _ws(workspace_bytes(cfg, TSP_OP_BLOCK_BWD | pf), dev) if ws is None else ws
    aw, mw = W.attn(), W.mlp()
    if prep is not None:
        _check(load().tsp_block_bwd_prepared(ctypes.byref(cfg), _ptr(x_z), _ptr(dy_z), _ptr(saved),
                                             _ptr(prep), ctypes.byref(aw), ctypes.byref(mw),
                                             _ptr(g["dx"]), *[_ptr(g[k]) for k in GRAD_NAMES],
                                             _ptr(ws), ws.numel(), _stream(stream)),
               "tsp_block_bwd_prepared")
        return g
    _check(load().tsp_block_bwd(ctypes.byref(cfg), _ptr(x_z), _ptr(dy_z), _ptr(saved),
                                ctypes.byref(aw), ctypes.byref(mw), _ptr(g["dx"]),
                                *[_ptr(g[k]) for k in GRAD_NAMES], _ptr(ws), ws.numel(),
                                _stream(stream)), "tsp_block_bwd")
    return g


def stack_saved_bytes(cfg: Cfg, L: int) -> int:
    return int(load().tsp_stack_saved_bytes(ctypes.byref(cfg), int(L)))


def stack_workspace_bytes(cfg: Cfg, L: int, op: int) -> int:
    return int(load().tsp_stack_workspace_bytes(ctypes.byref(cfg), int(L), op))


def _weight_arrays(Ws):
    L = len(Ws)
    aws = (AttnW * L)(*[W.attn() for W in Ws])
    mws = (MlpW * L)(*[W.mlp() for W in Ws])
    return aws, mws


def _prep_array(preps):
    return (ctypes.c_void_p * len(preps))(*[p.data_ptr() for p in preps])


def stack_fwd(cfg: Cfg, x_z, Ws, saved=None, out=None, ws=None, stream=None, preps=None):
    """y_z of the L-block stack with weights Ws[0..L-1].  ``saved`` (uint8,
    stack_saved_bytes(cfg, L)) keeps every layer's input and activations;
    ``preps``: every layer's prepare_weights buffer (weights converted once)."""
    _require_cuda(x_z)
    L = len(Ws)
    out = empty_like(x_z) if out is None else out
    pf = TSP_OP_PREPARED if preps is not None else 0
    if ws is None:
        ws = _ws(stack_workspace_bytes(cfg, L, TSP_OP_BLOCK_FWD | pf), x_z.device)
    aws, mws = _weight_arrays(Ws)
    if preps is not None:
        _check(load().tsp_stack_fwd_prepared(ctypes.byref(cfg), L, _ptr(x_z), _prep_array(preps), aws,
                                             mws, _ptr(out), _ptr(saved), _ptr(ws), ws.numel(),
                                             _stream(stream)), "tsp_stack_fwd_prepared")
        return out
    _check(load().tsp_stack_fwd(ctypes.byref(cfg), L, _ptr(x_z), aws, mws, _ptr(out), _ptr(saved),
                                _ptr(ws), ws.numel(), _stream(stream)), "tsp_stack_fwd")
    return out


def stack_bwd(cfg: Cfg, dy_z, saved, Ws, ws=None, stream=None, preps=None):
    """Gradients of sum(dy * y) through the stack: (dx_z fp32, [grads of layer l])."""
    _require_cuda(dy_z, saved)
    dev = dy_z.device
    L = len(Ws)
    shapes = _grad_shapes(cfg)
    grads = [{k: empty(shapes[k], torch.float32, dev) for k in GRAD_NAMES}
             for _ in range(L)]
    ptrs = (ctypes.c_void_p * (9 * L))(*[g[k].data_ptr() for g in grads for k in GRAD_NAMES])
    dx = empty(dy_z.shape, torch.float32, dev)
    pf = TSP_OP_PREPARED if preps is not None else 0
    if ws is None:
        ws = _ws(stack_workspace_bytes(cfg, L, TSP_OP_BLOCK_BWD | pf), dev)
    aws, mws = _weight_arrays(Ws)
    if preps is not None:
        _check(load().tsp_stack_bwd_prepared(ctypes.byref(cfg), L, _ptr(dy_z), _ptr(saved),
                                             _prep_array(preps), aws, mws, _ptr(dx), ptrs, _ptr(ws),
                                             ws.numel(), _stream(stream)), "tsp_stack_bwd_prepared")
        return dx, grads
    _check(load().tsp_stack_bwd(ctypes.byref(cfg), L, _ptr(dy_z), _ptr(saved), aws, mws, _ptr(dx),
                                ptrs, _ptr(ws), ws.numel(), _stream(stream)), "tsp_stack_bwd")
    return dx, grads


def rank_memory(cfg: Cfg, L: int, training: bool, scheme: int) -> dict:
    """Bytes one rank holds for an L-layer stack under a parallel scheme (host only)."""
    m = RankMem()
    _check(load().tsp_rank_memory(ctypes.byref(cfg), int(L), 1 if training else 0, int(scheme),
                                  ctypes.byref(m)), "tsp_rank_memory")
    return {k: getattr(m, k) for k, _ in RankMem._fields_}


def pack_attn_shards(cfg: Cfg, W: BlockWeights, stream=None):
    out = empty((4 * cfg.d, cfg.d), W.wq.dtype, W.wq.device)
    aw = W.attn()
    _check(load().tsp_pack_attn_shards(ctypes.byref(cfg), ctypes.byref(aw), _ptr(out),
                                       _stream(stream)), "tsp_pack_attn_shards")
    return out


def pack_mlp_shards(cfg: Cfg, W: BlockWeights, stream=None):
    """[3*inter, d]: shard k = [W_1[I_k]; W_3[I_k]; W_2[:, I_k]^T], shards in order."""
    out = empty((3 * cfg.inter, cfg.d), W.w1.dtype, W.w1.device)
    mw = W.mlp()
    _check(load().tsp_pack_mlp_shards(ctypes.byref(cfg), ctypes.byref(mw), _ptr(out),
                                      _stream(stream)), "tsp_pack_mlp_shards")
    return out


def rank_workspace_bytes(cfg: Cfg) -> int:
    return int(load().tsp_rank_workspace_bytes(ctypes.byref(cfg)))


def rank_attn_project(cfg: Cfg, r: int, k: int, x_r, g_attn, shard_k, kv_k, ws, stream=None):
    _check(load().tsp_rank_attn_project(ctypes.byref(cfg), r, k, _ptr(x_r), _ptr(g_attn),
                                        _ptr(shard_k), _ptr(kv_k), _ptr(ws), ws.numel(),
                                        _stream(stream)), "tsp_rank_attn_project")


def rank_attn_heads(cfg: Cfg, r: int, k: int, x_r, kv_all_k, h_r, ws, stream=None):
    _check(load().tsp_rank_attn_heads(ctypes.byref(cfg), r, k, _ptr(x_r), _ptr(kv_all_k),
                                      _ptr(h_r), _ptr(ws), ws.numel(), _stream(stream)),
           "tsp_rank_attn_heads")


def rank_mlp_step(cfg: Cfg, r: int, t: int, h_r, g_mlp, shard, y_r, y_out, ws, stream=None):
    _check(load().tsp_rank_mlp_step(ctypes.byref(cfg), r, t, _ptr(h_r), _ptr(g_mlp), _ptr(shard),
                                    _ptr(y_r), _ptr(y_out), _ptr(ws), ws.numel(), _stream(stream)),
           "tsp_rank_mlp_step")


def rank_mlp_bwd_step(cfg: Cfg, r: int, t: int, h_r, g_mlp, shard, dy_r, grad, db_r, ws,
                      stream=None):
    _check(load().tsp_rank_mlp_bwd_step(ctypes.byref(cfg), r, t, _ptr(h_r), _ptr(g_mlp),
                                        _ptr(shard), _ptr(dy_r), _ptr(grad), _ptr(db_r), _ptr(ws),
                                        ws.numel(), _stream(stream)), "tsp_rank_mlp_bwd_step")


def rank_mlp_bwd_finish(cfg: Cfg, r: int, h_r, g_mlp, db_r, dy_r, dh_r, dg_mlp, ws, stream=None):
    _check(load().tsp_rank_mlp_bwd_finish(ctypes.byref(cfg), r, _ptr(h_r), _ptr(g_mlp), _ptr(db_r),
                                          _ptr(dy_r), _ptr(dh_r), _ptr(dg_mlp), _ptr(ws),
                                          ws.numel(), _stream(stream)), "tsp_rank_mlp_bwd_finish")


def rank_attn_bwd_heads(cfg: Cfg, r: int, k: int, kv_all_k, grad_k, dkv_k, ws, stream=None):
    _check(load().tsp_rank_attn_bwd_heads(ctypes.byref(cfg), r, k, _ptr(kv_all_k), _ptr(grad_k),
                                          _ptr(dkv_k), _ptr(ws), ws.numel(), _stream(stream)),
           "tsp_rank_attn_bwd_heads")


def rank_attn_bwd_weights(cfg: Cfg, r: int, k: int, dkv_own, grad_k, da_r, ws, stream=None):
    _check(load().tsp_rank_attn_bwd_weights(ctypes.byref(cfg), r, k, _ptr(dkv_own), _ptr(grad_k),
                                            _ptr(da_r), _ptr(ws), ws.numel(), _stream(stream)),
           "tsp_rank_attn_bwd_weights")


def rank_attn_bwd_finish(cfg: Cfg, r: int, x_r, g_attn, da_r, dh_r, dx_r, dg_attn, ws,
                         stream=None):
    _check(load().tsp_rank_attn_bwd_finish(ctypes.byref(cfg), r, _ptr(x_r), _ptr(g_attn),
                                           _ptr(da_r), _ptr(dh_r), _ptr(dx_r), _ptr(dg_attn),
                                           _ptr(ws), ws.numel(), _stream(stream)),
           "tsp_rank_attn_bwd_finish")


def device_status(reset: bool = True, stream=None) -> int:
    return int(load().tsp_device_status(_stream(stream), 1 if reset else 0))


def profile_enable(on: bool = True):
    load().tsp_profile_enable(1 if on else 0)


def profile_report() -> dict:
    """{label: (kernels, total_ms)} of the launches recorded since profile_enable(True)."""
    buf = ctypes.create_string_buffer(1 << 16)
    n = load().tsp_profile_report(buf, len(buf))
    if n < 0:
        raise RuntimeError("tsp_profile_report failed")
    out = {}
    for line in buf.value.decode().splitlines():
        name, k, ms = line.split("\t")
        out[name] = (int(k), float(ms))
    return out


def launch_count() -> int:
    return int(load().tsp_launch_count())


def debug_skip_stage(n: int):
    """Failure-detection knob: the next n GEMM launches each leave one pipeline
    stage unfilled so a bounded wait runs out (TSP_ERR_TIMEOUT, no fault)."""
    load().tsp_debug_skip_stage(int(n))


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def gated_mlp_fwd_noalloc(cfg: Cfg, h_z, W: BlockWeights, out, norm=True, residual=True,
                          stream=None):
    """tsp_gated_mlp_fwd without a workspace: for callers that must not allocate
    device memory during the call.  ``out`` must be preallocated by the caller;
    the library works in its fixed 32 MiB device scratch and allocates nothing.
    Calls that overlap on the GPU share that scratch and race."""
    _require_cuda(h_z, out)
    mw = W.mlp(norm, residual)
    _check(load().tsp_gated_mlp_fwd_noalloc(ctypes.byref(cfg), _ptr(h_z), ctypes.byref(mw),
                                            _ptr(out), _stream(stream)),
           "tsp_gated_mlp_fwd_noalloc")
    return out
