"""The C ABI library loads, exports every declared entry point, and rejects
bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from folded_tensor_sequence_zigzag_gb300 import tsp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(tsp_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    from folded_tensor_sequence_zigzag_gb300 import build
    build.build()
    return tsp.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"tsp_zigzag_permute", "tsp_attn_block_fwd", "tsp_gated_mlp_fwd", "tsp_block_fwd",
            "tsp_block_bwd"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(tsp.EXPORTED) == names


def test_strerror(lib):
    for code in range(7):
        assert lib.tsp_strerror(code) and lib.tsp_strerror(code) != b"unknown status"
    assert b"invalid" in lib.tsp_strerror(tsp.TSP_ERR_INVALID_ARG)
    assert b"fp16" in lib.tsp_strerror(tsp.TSP_ERR_RANGE)
    assert b"bounds" in lib.tsp_strerror(tsp.TSP_ERR_BOUNDS)


def test_checked_build_exports_the_same_entry_points():
    """The checked build (TSP_CHECK: every computed global index tested
    before its access) is the same library otherwise: it builds from the same
    sources and exports every declared entry point."""
    from folded_tensor_sequence_zigzag_gb300 import build
    path = build.build(check=True)
    chk = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(chk, n), n


def _cfg(**kw):
    base = dict(S=256, d=64, H=4, inter=128, D=4, dtype=tsp.TSP_F32, rope_base=0.0, Hkv=0,
                mlp_tile=0)
    base.update(kw)
    return tsp.Cfg(base["S"], base["d"], base["H"], base.get("dh", base["d"] // base["H"]),
                   base["inter"], base["D"], 1e-6, base["dtype"], base["rope_base"], base["Hkv"],
                   base["mlp_tile"])


@pytest.mark.parametrize("bad", [dict(S=250), dict(D=0), dict(D=65), dict(d=66), dict(dh=8),
                                 dict(inter=0), dict(dtype=7), dict(S=0), dict(d=2, H=1, D=4),
                                 dict(rope_base=-1.0), dict(d=60, H=4, rope_base=10000.0),
                                 dict(Hkv=3), dict(Hkv=-1), dict(Hkv=8), dict(H=8, Hkv=1, D=16),
                                 dict(mlp_tile=-128), dict(mlp_tile=64, S=512, D=2),
                                 dict(mlp_tile=384, S=2048, D=4, dtype=tsp.TSP_BF16)])
def test_invalid_cfg_rejected_without_launch(lib, bad):
    cfg = _cfg(**bad)
    assert lib.tsp_workspace_bytes(ctypes.byref(cfg), tsp.TSP_OP_BLOCK_FWD) == 0
    assert lib.tsp_saved_bytes(ctypes.byref(cfg)) == 0
    fake = ctypes.c_void_p(0x10000)
    aw = tsp.AttnW(fake, fake, fake, fake, fake)
    mw = tsp.MlpW(fake, fake, fake, fake, 1)
    r = lib.tsp_block_fwd(ctypes.byref(cfg), fake, ctypes.byref(aw), ctypes.byref(mw), fake, None,
                          fake, 1 << 40, None)
    assert r == tsp.TSP_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_rejected(lib):
    cfg = _cfg()
    ok = ctypes.c_void_p(0x10000)
    mis = ctypes.c_void_p(0x10008)
    aw = tsp.AttnW(ok, ok, ok, ok, ok)
    mw = tsp.MlpW(ok, ok, ok, ok, 1)
    big = 1 << 40
    assert lib.tsp_block_fwd(ctypes.byref(cfg), None, ctypes.byref(aw), ctypes.byref(mw), ok,
                             None, ok, big, None) == tsp.TSP_ERR_INVALID_ARG
    assert lib.tsp_block_fwd(ctypes.byref(cfg), mis, ctypes.byref(aw), ctypes.byref(mw), ok,
                             None, ok, big, None) == tsp.TSP_ERR_INVALID_ARG
    bad_aw = tsp.AttnW(ok, mis, ok, ok, ok)
    assert lib.tsp_block_fwd(ctypes.byref(cfg), ok, ctypes.byref(bad_aw), ctypes.byref(mw), ok,
                             None, ok, big, None) == tsp.TSP_ERR_INVALID_ARG
    # block forward needs the MLP norm and residual
    no_norm = tsp.MlpW(ok, ok, ok, None, 1)
    assert lib.tsp_block_fwd(ctypes.byref(cfg), ok, ctypes.byref(aw), ctypes.byref(no_norm), ok,
                             None, ok, big, None) == tsp.TSP_ERR_INVALID_ARG
    # short workspace
    assert lib.tsp_block_fwd(ctypes.byref(cfg), ok, ctypes.byref(aw), ctypes.byref(mw), ok,
                             None, ok, 16, None) == tsp.TSP_ERR_INVALID_ARG
    assert lib.tsp_zigzag_permute(None, ok, 16, 2, 16, 0, None) == tsp.TSP_ERR_INVALID_ARG
    assert lib.tsp_zigzag_permute(ok, ok, 18, 2, 16, 0, None) == tsp.TSP_ERR_INVALID_ARG
    assert lib.tsp_zigzag_permute(ok, ok, 16, 2, 0, 0, None) == tsp.TSP_ERR_INVALID_ARG
    assert lib.tsp_rmsnorm_fwd(ok, None, ok, None, 4, 8, 1e-6, 1, None) == tsp.TSP_ERR_INVALID_ARG


def test_bf16_shapes_the_kernels_do_not_take_are_unsupported(lib):
    ok = ctypes.c_void_p(0x10000)
    aw = tsp.AttnW(ok, ok, ok, ok, ok)
    mw = tsp.MlpW(ok, ok, ok, ok, 1)
    # dh = 64 (tensor-core attention takes dh = 128 only)
    cfg = _cfg(S=2048, d=256, H=4, inter=512, D=4, dtype=tsp.TSP_BF16)
    assert lib.tsp_block_fwd(ctypes.byref(cfg), ok, ctypes.byref(aw), ctypes.byref(mw), ok,
                             None, ok, 1 << 40, None) == tsp.TSP_ERR_UNSUPPORTED
    # chunk of 64 rows (not a multiple of the 256-row attention block)
    cfg = _cfg(S=512, d=256, H=2, inter=512, D=4, dtype=tsp.TSP_BF16)
    assert lib.tsp_attn_block_fwd(ctypes.byref(cfg), ok, ctypes.byref(aw), ok, ok, 1 << 40,
                                  None) == tsp.TSP_ERR_UNSUPPORTED
    # grouped K/V of width 128 (the K|V GEMM's N tiles are 256 columns wide)
    cfg = _cfg(S=2048, d=512, H=4, inter=512, D=4, dtype=tsp.TSP_BF16, Hkv=1)
    assert lib.tsp_block_fwd(ctypes.byref(cfg), ok, ctypes.byref(aw), ctypes.byref(mw), ok,
                             None, ok, 1 << 40, None) == tsp.TSP_ERR_UNSUPPORTED
    # the MLP alone takes it
    cfg = _cfg(S=500 * 8, d=256, H=2, inter=384, D=4, dtype=tsp.TSP_BF16)
    assert lib.tsp_workspace_bytes(ctypes.byref(cfg), tsp.TSP_OP_MLP_FWD) > 0


def test_workspace_sizes_are_consistent(lib):
    cfg = _cfg(S=16384, d=4096, H=32, inter=11008, D=8, dtype=tsp.TSP_BF16)
    S, d, I, H = 16384, 4096, 11008, 32
    fwd = lib.tsp_workspace_bytes(ctypes.byref(cfg), tsp.TSP_OP_BLOCK_FWD)
    saved = lib.tsp_saved_bytes(ctypes.byref(cfg))
    acts = S * (d * 2 * (1 + 3 + 1 + 1) + d * 4 + I * 2 + 4 * (2 + H))  # a,QKV,O,b,G fp16; h fp32
    wcopy = 2 * (4 * d * d + 3 * d * I)                                    # fp16 weight copies
    # inference keeps the activations and the fp16 weight copies in the workspace
    assert fwd >= acts + wcopy
    # training keeps the activations plus the SwiGLU pre-activations A|B in `saved`
    assert saved >= acts + S * 2 * I * 2
    assert saved < acts + S * 2 * I * 2 + 64 * 256
    assert lib.tsp_workspace_bytes(ctypes.byref(cfg), tsp.TSP_OP_BLOCK_BWD) > 0


def test_decode_arguments_checked_without_launch(lib):
    cfg = _cfg()            # S=256, d=64, H=4, fp32
    ok = ctypes.c_void_p(0x10000)
    aw = tsp.AttnW(ok, ok, ok, ok, ok)
    mw = tsp.MlpW(ok, ok, ok, ok, 1)
    cap = 300
    assert lib.tsp_kv_cache_bytes(ctypes.byref(cfg), cap) == cap * 2 * 64 * 4
    assert lib.tsp_kv_cache_bytes(ctypes.byref(cfg), 255) == 0          # below the prompt
    assert lib.tsp_decode_workspace_bytes(ctypes.byref(cfg), 0, cap) == 0
    assert lib.tsp_decode_workspace_bytes(ctypes.byref(cfg), tsp.DECODE_MAX_T + 1, cap) == 0
    ws = lib.tsp_decode_workspace_bytes(ctypes.byref(cfg), 4, cap)
    assert ws > 0
    # grouped K/V: a narrower cache
    g = _cfg(Hkv=2)
    assert lib.tsp_kv_cache_bytes(ctypes.byref(g), cap) == cap * 2 * 32 * 4
    big = 1 << 40

    def dec(T, n_cached, cap_=cap, x=ok, wsb=big):
        return lib.tsp_block_decode(ctypes.byref(cfg), x, T, n_cached, ctypes.byref(aw),
                                    ctypes.byref(mw), ok, ok, cap_, ok, wsb, None)
    assert dec(0, 256) == tsp.TSP_ERR_INVALID_ARG
    assert dec(tsp.DECODE_MAX_T + 1, 256) == tsp.TSP_ERR_INVALID_ARG
    assert dec(1, 255) == tsp.TSP_ERR_INVALID_ARG              # inside the prompt
    assert dec(4, 297) == tsp.TSP_ERR_INVALID_ARG              # past the cache
    assert dec(1, 256, x=ctypes.c_void_p(0x10004)) == tsp.TSP_ERR_INVALID_ARG
    assert dec(1, 256, wsb=16) == tsp.TSP_ERR_INVALID_ARG      # short workspace
    # prefill: the cache must hold the prompt
    assert lib.tsp_block_prefill(ctypes.byref(cfg), ok, ctypes.byref(aw), ctypes.byref(mw), ok, ok,
                                 255, ok, big, None) == tsp.TSP_ERR_INVALID_ARG


def test_mlp_tiling_configuration(lib):
    """Tiles of 128-multiples that divide a virtual rank's rows; bf16 only;
    the training record loses G and A|B, the backward workspace shrinks."""
    big = dict(S=16384, d=4096, H=32, inter=11008, D=8, dtype=tsp.TSP_BF16)
    plain, tiled = _cfg(**big), _cfg(mlp_tile=1024, **big)
    S, I = 16384, 11008
    saved_gap = lib.tsp_saved_bytes(ctypes.byref(plain)) - lib.tsp_saved_bytes(ctypes.byref(tiled))
    assert saved_gap == S * I * 2 + S * 2 * I * 2            # G and A|B, fp16
    bwd_plain = lib.tsp_workspace_bytes(ctypes.byref(plain), tsp.TSP_OP_BLOCK_BWD)
    bwd_tiled = lib.tsp_workspace_bytes(ctypes.byref(tiled), tsp.TSP_OP_BLOCK_BWD)
    assert bwd_plain - bwd_tiled == (S - 1024) * 2 * I * 2 - 1024 * 3 * I * 2
    train = lib.tsp_workspace_bytes(ctypes.byref(tiled), tsp.TSP_OP_BLOCK_FWD_TRAIN)
    assert train - lib.tsp_workspace_bytes(ctypes.byref(plain), tsp.TSP_OP_BLOCK_FWD_TRAIN) == 1024 * I * 2
    # fp32: valid shape, not taken by the tiled path
    f32 = _cfg(mlp_tile=128, S=1024, d=64, H=4, inter=128, D=4)
    assert lib.tsp_saved_bytes(ctypes.byref(f32)) == 0
    ok = ctypes.c_void_p(0x10000)
    aw = tsp.AttnW(ok, ok, ok, ok, ok)
    mw = tsp.MlpW(ok, ok, ok, ok, 1)
    assert lib.tsp_block_fwd(ctypes.byref(f32), ok, ctypes.byref(aw), ctypes.byref(mw), ok, ok, ok,
                             1 << 40, None) == tsp.TSP_ERR_UNSUPPORTED


def test_prepared_weights_sizes(lib):
    """Prepared fp16 copies: one block's seven matrices in fp16; the whole-block
    workspaces shrink by exactly that; fp32 has nothing to prepare; the
    prepared calls reject a missing buffer on the host."""
    d, I = 4096, 11008
    cfg = _cfg(S=16384, d=d, H=32, inter=I, D=8, dtype=tsp.TSP_BF16)
    nb = lib.tsp_block_weights_bytes(ctypes.byref(cfg))
    assert 2 * (4 * d * d + 3 * d * I) <= nb < 2 * (4 * d * d + 3 * d * I) + 7 * 256
    for op in (tsp.TSP_OP_BLOCK_FWD, tsp.TSP_OP_BLOCK_BWD):
        full = lib.tsp_workspace_bytes(ctypes.byref(cfg), op)
        assert lib.tsp_workspace_bytes(ctypes.byref(cfg), op | tsp.TSP_OP_PREPARED) == full - nb
    assert lib.tsp_workspace_bytes(ctypes.byref(cfg), tsp.TSP_OP_MLP_FWD | tsp.TSP_OP_PREPARED) == 0
    L = 4
    assert (lib.tsp_stack_workspace_bytes(ctypes.byref(cfg), L, tsp.TSP_OP_BLOCK_FWD)
            - lib.tsp_stack_workspace_bytes(ctypes.byref(cfg), L,
                                             tsp.TSP_OP_BLOCK_FWD | tsp.TSP_OP_PREPARED)) == nb
    assert lib.tsp_block_weights_bytes(ctypes.byref(_cfg())) == 0      # fp32
    assert lib.tsp_block_fwd_prepared(ctypes.byref(cfg), None, None, None, None, None, None, None,
                                      0, None) == tsp.TSP_ERR_INVALID_ARG
    assert lib.tsp_stack_fwd_prepared(ctypes.byref(cfg), 2, None, None, None, None, None, None,
                                      None, 0, None) == tsp.TSP_ERR_INVALID_ARG
