"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong chunk order) fails at
least one of them:
  * hand-worked fixtures under tests/golden/ (zigzag map, pair counts);
  * closed forms (constant-row RMSNorm, S=1 attention, K = 0 attention,
    zero W_O / W_2, the c*(S+1) pair count);
  * invariants (bijection, softmax rows sum to 1, causality, sharded ==
    unsharded for D = 1..8);
  * an independent library evaluation in torch CPU float64 (F.rms_norm,
    scaled_dot_product_attention, F.silu, autograd);
  * central finite differences for the backward.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.tsp_oracle as O
from folded_tensor_sequence_zigzag_gb300.inputs import BlockShape, TINY_FP32, make_block_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return np.array(rows, dtype=np.int64)


# --------------------------------------------------------------- zigzag map

def test_zigzag_golden_S12_D3():
    g = _load("zigzag_S12_D3.txt")
    pos = O.zigzag_positions(12, 3)
    assert np.array_equal(pos, g[:, 1])
    assert np.array_equal(O.zigzag_owner(12, 3)[pos], g[:, 2])


@pytest.mark.parametrize("S,D", [(2, 1), (16, 1), (16, 2), (48, 3), (256, 4), (320, 5), (96, 6), (112, 7), (256, 8), (4096, 8)])
def test_zigzag_is_bijection_and_owner_consistent(S, D):
    pos = O.zigzag_positions(S, D)
    assert np.array_equal(np.sort(pos), np.arange(S))
    c = S // (2 * D)
    owner = O.zigzag_owner(S, D)
    for r in range(D):
        rows = pos[r * 2 * c:(r + 1) * 2 * c]
        assert np.all(owner[rows] == r)
        assert np.all(np.diff(rows[:c]) == 1) and np.all(np.diff(rows[c:]) == 1)
    x = np.random.default_rng(0).standard_normal((S, 3))
    assert np.array_equal(O.zigzag_permute(O.zigzag_permute(x, D), D, inverse=True), x)


def test_causal_pairs_closed_form_golden():
    for S, D, per_rank, total in _load("causal_pairs.txt"):
        pairs = O.causal_pairs_per_rank(int(S), int(D))
        assert np.all(pairs == per_rank), (S, D, pairs)
        assert pairs.sum() == total == S * (S + 1) // 2


def test_zigzag_rejects_bad_sizes():
    with pytest.raises(ValueError):
        O.zigzag_positions(10, 3)


def test_shard_bounds_cover_once():
    for n in (64, 128, 4096, 11008):
        for D in range(1, 9):
            b = O.shard_bounds(n, D)
            assert b[0] == 0 and b[-1] == n and all(b[k] <= b[k + 1] for k in range(D))
    assert O.shard_bounds(11008, 8)[1] == 1376 and O.shard_bounds(11008, 4)[1] == 2752


# --------------------------------------------------------------- elementary layers

def test_rmsnorm_closed_form_constant_rows():
    vals = np.array([0.5, -3.0, 7.25])
    u = np.repeat(vals[:, None], 8, axis=1)
    g = np.linspace(0.5, 2.0, 8)
    eps = 1e-6
    out, rstd = O.rmsnorm(u, g, eps)
    expect = vals[:, None] / np.sqrt(vals[:, None] ** 2 + eps) * g[None, :]
    assert np.allclose(out, expect, rtol=0, atol=1e-15)
    assert np.allclose(rstd, 1 / np.sqrt(vals ** 2 + eps))


def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(1)
    u = rng.standard_normal((17, 33)) * 3
    g = rng.standard_normal(33)
    out, _ = O.rmsnorm(u, g, 1e-6)
    ref = F.rms_norm(torch.from_numpy(u), (33,), torch.from_numpy(g), eps=1e-6).numpy()
    assert np.max(np.abs(out - ref)) < 1e-13


def test_silu_matches_torch_and_is_stable():
    z = np.linspace(-800, 800, 2001)
    ref = F.silu(torch.from_numpy(z)).numpy()
    assert np.allclose(O.silu(z), ref, rtol=1e-14, atol=1e-300)
    assert np.all(np.isfinite(O.silu(z)))


def _rand_qkv(S, H, dh, seed=0):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((S, H * dh)) for _ in range(3)]


def test_attention_single_token_returns_v():
    Q, K, V = _rand_qkv(1, 2, 4)
    out, lse = O.causal_attention(Q, K, V, 2)
    assert np.array_equal(out, V)
    for h in range(2):
        s = Q[0, h * 4:(h + 1) * 4] @ K[0, h * 4:(h + 1) * 4] / 2.0
        assert abs(lse[h, 0] - s) < 1e-14


def test_attention_zero_keys_is_prefix_mean():
    Q, K, V = _rand_qkv(37, 3, 8, seed=2)
    out, lse = O.causal_attention(Q, np.zeros_like(K), V, 3, row_block=8)
    prefix = np.cumsum(V, axis=0) / np.arange(1, 38)[:, None]
    assert np.max(np.abs(out - prefix)) < 1e-13
    assert np.allclose(lse, np.log(np.arange(1, 38))[None, :].repeat(3, 0))


def test_attention_rows_sum_to_one_and_mask():
    Q, K, V = _rand_qkv(29, 2, 8, seed=3)
    P = O.attention_probs(Q * 4, K * 4, 2)
    assert np.max(np.abs(P.sum(axis=2) - 1)) <= 1e-12
    assert np.all(np.triu(P[0], 1) == 0) and np.all(np.triu(P[1], 1) == 0)
    assert np.all(np.diagonal(P, axis1=1, axis2=2) > 0)


def test_attention_matches_torch_sdpa():
    H, dh, S = 4, 16, 70
    Q, K, V = _rand_qkv(S, H, dh, seed=4)
    out, lse = O.causal_attention(Q, K, V, H, row_block=16)
    t = lambda a: torch.from_numpy(a).view(S, H, dh).transpose(0, 1)  # noqa: E731
    ref = F.scaled_dot_product_attention(t(Q), t(K), t(V), is_causal=True)
    ref = ref.transpose(0, 1).reshape(S, H * dh).numpy()
    assert np.max(np.abs(out - ref)) < 1e-13
    sc = torch.einsum("hid,hjd->hij", t(Q), t(K)) / math.sqrt(dh)
    sc = sc.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    assert np.max(np.abs(lse - torch.logsumexp(sc, dim=2).numpy())) < 1e-12


def test_attention_with_positions_equals_permuted_attention():
    # zigzag-ordered queries/keys with their global positions give the same
    # rows as the global-order computation, permuted
    S, D, H, dh = 48, 3, 2, 8
    Q, K, V = _rand_qkv(S, H, dh, seed=5)
    pos = O.zigzag_positions(S, D)
    ref, lref = O.causal_attention(Q, K, V, H)
    out, lout = O.causal_attention(Q[pos], K[pos], V[pos], H, q_pos=pos, k_pos=pos, row_block=7)
    assert np.max(np.abs(out - ref[pos])) < 1e-13
    assert np.max(np.abs(lout - lref[:, pos])) < 1e-12


# --------------------------------------------------------------- whole block

def _torch_block(inp, H, eps, requires_grad=False):
    """Independent float64 evaluation with torch library routines."""
    T = {k: v.to(torch.float64).clone().requires_grad_(requires_grad) for k, v in inp.items()}
    x = T["x"]
    S, d = x.shape
    dh = d // H
    Hk = T["wk"].shape[0] // dh          # K/V heads (grouped-query attention if < H)
    a = F.rms_norm(x, (d,), T["g_attn"], eps=eps)
    heads = lambda m, n: m.view(S, n, dh).transpose(0, 1)  # noqa: E731
    o = F.scaled_dot_product_attention(heads(F.linear(a, T["wq"]), H),
                                       heads(F.linear(a, T["wk"]), Hk),
                                       heads(F.linear(a, T["wv"]), Hk), is_causal=True,
                                       enable_gqa=Hk != H)
    h = x + F.linear(o.transpose(0, 1).reshape(S, d), T["wo"])
    b = F.rms_norm(h, (d,), T["g_mlp"], eps=eps)
    y = h + F.linear(F.silu(F.linear(b, T["w1"])) * F.linear(b, T["w3"]), T["w2"])
    return y, h, T


def _small(S=64, d=32, H=4, inter=48, D=4, seed=0, dtype=torch.float32, Hkv=0):
    shape = BlockShape(S=S, d=d, H=H, inter=inter, D=D, Hkv=Hkv)
    inp = make_block_inputs(shape, dtype, seed=seed, with_dy=True)
    # non-trivial gains so a dropped gain shows up
    gen = torch.Generator().manual_seed(seed + 100)
    inp["g_attn"] = (1 + 0.5 * torch.randn(d, generator=gen)).to(dtype)
    inp["g_mlp"] = (1 + 0.5 * torch.randn(d, generator=gen)).to(dtype)
    # larger weights so attention is far from uniform and the MLP is non-linear
    for k in ("wq", "wk", "wv", "wo", "w1", "w3", "w2"):
        inp[k] = (inp[k] * 10).to(dtype)
    return shape, inp


def test_block_fwd_matches_torch_fp64():
    shape, inp = _small()
    y, s = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    yt, ht, _ = _torch_block(inp, shape.H, shape.eps)
    assert np.max(np.abs(y - yt.detach().numpy())) < 1e-11
    assert np.max(np.abs(s["h"] - ht.detach().numpy())) < 1e-11


def test_block_fwd_tiny_config_matches_torch_fp64():
    inp = make_block_inputs(TINY_FP32, torch.float32, seed=0)
    y, _ = O.block_fwd(inp["x"], inp, TINY_FP32.H, TINY_FP32.eps)
    yt, _, _ = _torch_block(inp, TINY_FP32.H, TINY_FP32.eps)
    assert np.max(np.abs(y - yt.detach().numpy())) < 1e-12


@pytest.mark.parametrize("D", [1, 2, 3, 4, 5, 6, 7, 8])
def test_sharded_equals_unsharded(D):
    shape, inp = _small(S=2 * D * 16, D=D, seed=D)
    y, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    ys = O.block_fwd_sharded(inp["x"], inp, shape.H, D, shape.eps)
    rel = np.max(np.abs(ys - y)) / np.max(np.abs(y))
    assert rel <= 1e-12
    if D == 1:
        assert np.max(np.abs(ys - y)) <= 1e-12 * np.max(np.abs(y))


@pytest.mark.parametrize("D", [1, 2, 4, 8])
def test_sharded_equals_unsharded_tiny_S256(D):
    inp = make_block_inputs(TINY_FP32, torch.float32, seed=0)
    y, _ = O.block_fwd(inp["x"], inp, 4, 1e-6)
    ys = O.block_fwd_sharded(inp["x"], inp, 4, D, 1e-6)
    assert np.max(np.abs(ys - y)) <= 1e-12 * np.max(np.abs(y))


def test_mlp_sharded_equals_unsharded_no_norm_no_residual():
    shape, inp = _small(S=64, D=4)
    ref, _ = O.mlp_fwd(inp["x"], inp, shape.eps, norm=False, residual=False)
    got = O.mlp_fwd_sharded(inp["x"], inp, 4, shape.eps, norm=False, residual=False)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
    t = {k: v.to(torch.float64) for k, v in inp.items()}
    tref = F.linear(F.silu(F.linear(t["x"], t["w1"])) * F.linear(t["x"], t["w3"]), t["w2"]).numpy()
    assert np.max(np.abs(ref - tref)) < 1e-11


def test_causality_perturbing_future_rows():
    shape, inp = _small(S=48, D=3)
    y0, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    for i in (0, 17, 30, 46):
        pert = dict(inp)
        x = inp["x"].clone()
        x[i + 1:] += torch.randn(x[i + 1:].shape, generator=torch.Generator().manual_seed(i)) * 5
        pert["x"] = x
        y1, _ = O.block_fwd(x, pert, shape.H, shape.eps)
        assert np.array_equal(y0[: i + 1], y1[: i + 1])
        if i + 1 < 48:
            assert not np.array_equal(y0[i + 1:], y1[i + 1:])


def test_zero_w2_gives_h_and_zero_wo_gives_x():
    shape, inp = _small(S=32, D=2)
    z = dict(inp)
    z["w2"] = torch.zeros_like(inp["w2"])
    y, s = O.block_fwd(inp["x"], z, shape.H, shape.eps)
    assert np.array_equal(y, s["h"])
    z = dict(inp)
    z["wo"] = torch.zeros_like(inp["wo"])
    h, _ = O.attn_block_fwd(inp["x"], z, shape.H, shape.eps)
    assert np.array_equal(h, O.f64(inp["x"]))


def test_block_fwd_rows_matches_full():
    shape, inp = _small(S=96, D=3)
    y, s = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    rows = np.array([0, 5, 15, 16, 40, 95])
    assert np.max(np.abs(O.block_fwd_rows(inp["x"], inp, shape.H, shape.eps, rows) - y[rows])) < 1e-12
    h = O.block_fwd_rows(inp["x"], inp, shape.H, shape.eps, rows, attn_only=True)
    assert np.max(np.abs(h - s["h"][rows])) < 1e-12


# --------------------------------------------------------------- backward

def _loss(inp, H, eps):
    y, _ = O.block_fwd(inp["x"], inp, H, eps)
    return float(np.sum(O.f64(inp["dy"]) * y))


GRAD_OF = {"dx": "x", "dwq": "wq", "dwk": "wk", "dwv": "wv", "dwo": "wo", "dw1": "w1",
           "dw3": "w3", "dw2": "w2", "dg_attn": "g_attn", "dg_mlp": "g_mlp"}


def test_backward_matches_torch_autograd():
    shape, inp = _small(S=40, d=16, H=2, inter=24, D=2)
    g = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)
    y, _, T = _torch_block(inp, shape.H, shape.eps, requires_grad=True)
    (y * T["dy"].detach()).sum().backward()
    for gname, pname in GRAD_OF.items():
        ref = T[pname].grad.numpy()
        err = np.max(np.abs(g[gname] - ref)) / max(np.max(np.abs(ref)), 1e-30)
        assert err < 1e-11, (gname, err)


def test_backward_central_finite_differences():
    shape, inp = _small(S=32, d=16, H=2, inter=24, D=2, seed=7)
    inp = {k: v.to(torch.float64) for k, v in inp.items()}
    g = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)
    rng = np.random.default_rng(11)
    step = 1e-6
    for gname, pname in GRAD_OF.items():
        base = inp[pname]
        scale = np.sqrt(np.mean(g[gname] ** 2))
        flat = base.reshape(-1)
        idx = rng.choice(flat.numel(), size=min(16, flat.numel()), replace=False)
        for i in idx:
            plus, minus = dict(inp), dict(inp)
            p = base.clone(); p.view(-1)[i] += step; plus[pname] = p
            m = base.clone(); m.view(-1)[i] -= step; minus[pname] = m
            fd = (_loss(plus, shape.H, shape.eps) - _loss(minus, shape.H, shape.eps)) / (2 * step)
            an = g[gname].reshape(-1)[i]
            assert abs(fd - an) <= 1e-6 * max(abs(an), scale), (gname, i, fd, an)
        # a random direction
        v = torch.from_numpy(rng.standard_normal(tuple(base.shape)))
        plus, minus = dict(inp), dict(inp)
        plus[pname] = base + step * v
        minus[pname] = base - step * v
        fd = (_loss(plus, shape.H, shape.eps) - _loss(minus, shape.H, shape.eps)) / (2 * step)
        an = float(np.sum(g[gname] * v.numpy()))
        assert abs(fd - an) <= 1e-6 * max(abs(an), scale * math.sqrt(v.numel())), (gname, fd, an)


@pytest.mark.parametrize("D", [1, 2, 3, 4])
def test_backward_sharded_equals_unsharded(D):
    shape, inp = _small(S=2 * D * 8, d=16, H=2, inter=24, D=D, seed=20 + D)
    g = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)
    gs = O.block_bwd_sharded(inp["x"], inp, inp["dy"], shape.H, D, shape.eps)
    for k in GRAD_OF:
        ref = g[k]
        assert np.max(np.abs(gs[k] - ref)) <= 1e-12 * np.max(np.abs(ref)), k


@pytest.mark.parametrize("n_tail", [1, 7, 24])
def test_backward_tail_rows_equal_full_backward(n_tail):
    shape, inp = _small(S=48, d=16, H=2, inter=24, D=3, seed=31)
    full = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)["dx"]
    tail = O.block_bwd_tail(inp["x"], inp, inp["dy"], shape.H, shape.eps, n_tail)
    assert np.max(np.abs(tail - full[48 - n_tail:])) <= 1e-12 * np.max(np.abs(full))


# --------------------------------------------------------------- planted mistakes

def test_planted_mistakes_are_caught(monkeypatch):
    """Plant typical slips in the oracle (CPU only) and check a pin fails."""
    shape, inp = _small(S=48, D=3)
    yt, _, _ = _torch_block(inp, shape.H, shape.eps)
    yt = yt.detach().numpy()

    def off():
        y, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
        return np.max(np.abs(y - yt))

    assert off() < 1e-11
    # (1) SiLU on the wrong branch / wrong sign in the sigmoid
    with monkeypatch.context() as m:
        m.setattr(O, "sigmoid", lambda z: 1 / (1 + np.exp(z)))
        assert off() > 1e-3
    # (2) RMSNorm without eps inside the root -> the constant-row closed form
    with monkeypatch.context() as m:
        m.setattr(O, "rmsnorm", lambda u, g, eps: (u / np.sqrt(np.mean(u * u, 1))[:, None] * g,
                                                   1 / np.sqrt(np.mean(u * u, 1))))
        out, _ = O.rmsnorm(np.full((1, 4), 1e-4), np.ones(4), 1e-6)
        assert abs(out[0, 0] - 1e-4 / math.sqrt(1e-8 + 1e-6)) > 1e-3
    # (3) zigzag with the two chunks of a rank swapped -> golden fixture
    with monkeypatch.context() as m:
        def swapped(S, D):
            c = S // (2 * D)
            return np.concatenate([np.r_[(2 * D - 1 - r) * c:(2 * D - r) * c, r * c:(r + 1) * c]
                                   for r in range(D)])
        m.setattr(O, "zigzag_positions", swapped)
        assert not np.array_equal(O.zigzag_positions(12, 3), _load("zigzag_S12_D3.txt")[:, 1])
    # (4) attention mask without the diagonal -> S=1 closed form breaks
    Q, K, V = _rand_qkv(5, 1, 4)
    P = O.attention_probs(Q, K, 1)
    strict = np.tril(P[0], -1)
    assert not np.allclose(strict.sum(axis=1), 1)


# ------------------------------------------------------------------ stack of blocks

def _layers(shape, seeds):
    """Weight sets of the _small kind (non-trivial gains, larger weights)."""
    ws = []
    for sd in seeds:
        _, inp = _small(S=shape.S, d=shape.d, H=shape.H, inter=shape.inter, D=shape.D, seed=sd)
        ws.append({k: inp[k].to(torch.float64) for k in GRAD_OF.values() if k != "x"})
    return ws


def test_stack_of_one_is_the_block():
    shape, inp = _small(S=24, d=16, H=2, inter=24, D=3, seed=41)
    y1 = O.stack_fwd(inp["x"], [inp], shape.H, shape.eps)
    yb, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    assert np.array_equal(y1, yb)


def test_stack_identity_layer_is_transparent():
    """A layer with W_O = 0 and W_2 = 0 adds nothing to either residual, so it
    passes its input through unchanged wherever it sits in the stack."""
    shape, inp = _small(S=24, d=16, H=2, inter=24, D=3, seed=42)
    ident = dict(inp)
    ident["wo"] = torch.zeros_like(inp["wo"])
    ident["w2"] = torch.zeros_like(inp["w2"])
    yb, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    for Ws in ([inp, ident], [ident, inp], [ident, inp, ident]):
        y = O.stack_fwd(inp["x"], Ws, shape.H, shape.eps)
        assert np.max(np.abs(y - yb)) <= 1e-13 * np.max(np.abs(yb))


def test_stack_backward_central_finite_differences():
    """dx and one weight of every layer of a 3-layer stack against central
    differences of sum(dy * y): a dropped or misplaced link of the chain rule
    between layers fails."""
    shape, inp = _small(S=16, d=8, H=2, inter=12, D=2, seed=43)
    inp = {k: v.to(torch.float64) for k, v in inp.items()}
    Ws = _layers(shape, [43, 44, 45])
    x, dy = inp["x"], inp["dy"]
    dx, grads = O.stack_bwd(x, Ws, dy, shape.H, shape.eps)

    def loss(xx, WW):
        return float(np.sum(O.f64(dy) * O.stack_fwd(xx, WW, shape.H, shape.eps)))

    rng = np.random.default_rng(5)
    step = 1e-6
    v = torch.from_numpy(rng.standard_normal(tuple(x.shape)))
    fd = (loss(x + step * v, Ws) - loss(x - step * v, Ws)) / (2 * step)
    an = float(np.sum(dx * v.numpy()))
    assert abs(fd - an) <= 1e-6 * abs(an), ("dx", fd, an)
    for l in range(3):
        for gname, pname in (("dwq", "wq"), ("dw2", "w2"), ("dg_mlp", "g_mlp")):
            base = Ws[l][pname]
            u = torch.from_numpy(rng.standard_normal(tuple(base.shape)))
            plus = [dict(W) for W in Ws]
            minus = [dict(W) for W in Ws]
            plus[l][pname] = base + step * u
            minus[l][pname] = base - step * u
            fd = (loss(x, plus) - loss(x, minus)) / (2 * step)
            an = float(np.sum(grads[l][gname] * u.numpy()))
            assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-8), (l, gname, fd, an)


def test_two_layer_stack_backward_is_the_composition_of_block_backwards():
    """The gradient handed from layer 1 to layer 0 is layer 1's dx, unrounded:
    a two-layer stack's dx and every gradient equal two block backwards
    chained by hand, and layer 1 sees layer 0's exact output as its input."""
    shape, inp = _small(S=24, d=16, H=2, inter=24, D=3, seed=46)
    W0 = inp
    W1 = _layers(shape, [47])[0]
    x, dy = inp["x"], inp["dy"]
    dx, grads = O.stack_bwd(x, [W0, W1], dy, shape.H, shape.eps)
    y0, _ = O.block_fwd(x, W0, shape.H, shape.eps)
    g1 = O.block_bwd(y0, W1, dy, shape.H, shape.eps)
    g0 = O.block_bwd(x, W0, g1["dx"], shape.H, shape.eps)
    assert np.array_equal(dx, g0["dx"])
    for k in grads[0]:
        assert np.array_equal(grads[0][k], g0[k]), k
        assert np.array_equal(grads[1][k], g1[k]), k
    # and the forward: layer 1 reads layer 0's output as it is
    y = O.stack_fwd(x, [W0, W1], shape.H, shape.eps)
    assert np.array_equal(y, O.block_fwd(y0, W1, shape.H, shape.eps)[0])


# ------------------------------------------------------------------ rotary embedding (variant)

def _rope_rand(n=12, H=2, dh=8, seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, H * dh)), rng.integers(0, 5000, size=n)


def test_rope_closed_form_on_unit_vectors():
    """Element j of a head alone turns into (cos, sin) of pos * base^(-2j/dh)
    at positions j and j + dh/2: pins the frequency formula and the pairing."""
    H, dh, base = 2, 8, 10000.0
    half = dh // 2
    pos = np.array([0, 1, 7, 4095])
    for h in range(H):
        for j in range(half):
            X = np.zeros((len(pos), H * dh))
            X[:, h * dh + j] = 1.0
            Y = O.rope(X, pos, H, base)
            ang = pos * base ** (-2.0 * j / dh)
            assert np.allclose(Y[:, h * dh + j], np.cos(ang), atol=1e-15)
            assert np.allclose(Y[:, h * dh + j + half], np.sin(ang), atol=1e-15)
            others = np.delete(Y, [h * dh + j, h * dh + j + half], axis=1)
            assert np.all(others == 0)


def test_rope_norms_roundtrip_and_identity():
    X, pos = _rope_rand()
    Y = O.rope(X, pos, 2, 10000.0)
    assert np.allclose(np.linalg.norm(Y, axis=1), np.linalg.norm(X, axis=1), rtol=1e-14)
    assert np.allclose(O.rope(Y, pos, 2, 10000.0, inverse=True), X, atol=1e-13)
    assert np.array_equal(O.rope(X, np.zeros_like(pos), 2, 10000.0), X)
    assert O.rope(X, pos, 2, 0.0) is X


def test_rope_scores_depend_on_relative_position_only():
    q, _ = _rope_rand(n=1, seed=1)
    k, _ = _rope_rand(n=1, seed=2)
    H, dh = 2, 8
    for m, n in ((5, 3), (100, 100), (17, 2000)):
        for t in (0, 1, 999):
            a = O.rope(q, [m + t], H, 500.0)
            b = O.rope(k, [n + t], H, 500.0)
            ref = O.rope(q, [m], H, 500.0), O.rope(k, [n], H, 500.0)
            for h in range(H):
                sl = slice(h * dh, (h + 1) * dh)
                assert np.isclose(a[0, sl] @ b[0, sl], ref[0][0, sl] @ ref[1][0, sl], rtol=1e-12)


def _rope_small(seed, D=2, S=32):
    shape, inp = _small(S=S, d=16, H=2, inter=24, D=D, seed=seed)
    inp = {k: v.to(torch.float64) for k, v in inp.items()}
    inp["rope_base"] = 1000.0
    return shape, inp


def test_rope_block_backward_central_finite_differences():
    shape, inp = _rope_small(51)
    g = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)
    rng = np.random.default_rng(3)
    step = 1e-6
    for gname, pname in (("dx", "x"), ("dwq", "wq"), ("dwk", "wk"), ("dwv", "wv")):
        base = inp[pname]
        v = torch.from_numpy(rng.standard_normal(tuple(base.shape)))
        plus, minus = dict(inp), dict(inp)
        plus[pname] = base + step * v
        minus[pname] = base - step * v
        fd = (_loss(plus, shape.H, shape.eps) - _loss(minus, shape.H, shape.eps)) / (2 * step)
        an = float(np.sum(g[gname] * v.numpy()))
        assert abs(fd - an) <= 1e-6 * abs(an), (gname, fd, an)


@pytest.mark.parametrize("D", [1, 2, 4])
def test_rope_sharded_and_tail_equal_unsharded(D):
    shape, inp = _rope_small(60 + D, D=D, S=2 * D * 8)
    y, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    ys = O.block_fwd_sharded(inp["x"], inp, shape.H, D, shape.eps)
    assert np.max(np.abs(ys - y)) <= 1e-12 * np.max(np.abs(y))
    rows = np.array([0, 3, shape.S - 1])
    yr = O.block_fwd_rows(inp["x"], inp, shape.H, shape.eps, rows)
    assert np.max(np.abs(yr - y[rows])) <= 1e-12 * np.max(np.abs(y))
    g = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)
    gs = O.block_bwd_sharded(inp["x"], inp, inp["dy"], shape.H, D, shape.eps)
    for k in GRAD_OF:
        assert np.max(np.abs(gs[k] - g[k])) <= 1e-12 * np.max(np.abs(g[k])), k
    tail = O.block_bwd_tail(inp["x"], inp, inp["dy"], shape.H, shape.eps, 5)
    assert np.max(np.abs(tail - g["dx"][-5:])) <= 1e-12 * np.max(np.abs(g["dx"]))


# ------------------------------------------------------------------ grouped-query attention (variant)

@pytest.mark.parametrize("Hkv", [1, 2])
def test_gqa_block_matches_torch_fp64_forward_and_autograd(Hkv):
    """torch's own grouped-query attention (query head h on K/V head
    h // (H / Hkv)) pins the head mapping, the forward and every gradient,
    including dW_K / dW_V, which sum over a group's query heads."""
    shape, inp = _small(S=40, d=32, H=4, inter=24, D=2, seed=70 + Hkv, Hkv=Hkv)
    assert inp["wk"].shape == (Hkv * 8, 32)
    y, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    yt, _, T = _torch_block(inp, shape.H, shape.eps, requires_grad=True)
    assert np.max(np.abs(y - yt.detach().numpy())) < 1e-11
    g = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)
    (yt * T["dy"].detach()).sum().backward()
    for gname, pname in GRAD_OF.items():
        ref = T[pname].grad.numpy()
        assert g[gname].shape == ref.shape, gname
        err = np.max(np.abs(g[gname] - ref)) / max(np.max(np.abs(ref)), 1e-30)
        assert err < 1e-11, (gname, err)


def test_gqa_equals_mha_with_each_kv_head_repeated_over_its_group():
    rng = np.random.default_rng(5)
    S, H, Hkv, dh = 24, 6, 2, 8
    Q = rng.standard_normal((S, H * dh))
    K = rng.standard_normal((S, Hkv * dh))
    V = rng.standard_normal((S, Hkv * dh))
    grp = H // Hkv
    rep = lambda M: np.concatenate(  # noqa: E731
        [M[:, (h // grp) * dh:(h // grp + 1) * dh] for h in range(H)], axis=1)
    O1, L1 = O.causal_attention(Q, K, V, H)
    O2, L2 = O.causal_attention(Q, rep(K), rep(V), H)
    assert np.allclose(O1, O2, atol=1e-14) and np.allclose(L1, L2, atol=1e-14)
    dO = rng.standard_normal(O1.shape)
    dq1, dk1, dv1 = O.causal_attention_bwd(Q, K, V, O1, dO, H)
    dq2, dk2, dv2 = O.causal_attention_bwd(Q, rep(K), rep(V), O2, dO, H)
    assert np.allclose(dq1, dq2, atol=1e-13)
    for g in range(Hkv):      # a K/V head's gradient = the sum over its group
        sl = slice(g * dh, (g + 1) * dh)
        want_k = sum(dk2[:, h * dh:(h + 1) * dh] for h in range(g * grp, (g + 1) * grp))
        want_v = sum(dv2[:, h * dh:(h + 1) * dh] for h in range(g * grp, (g + 1) * grp))
        assert np.allclose(dk1[:, sl], want_k, atol=1e-13)
        assert np.allclose(dv1[:, sl], want_v, atol=1e-13)


@pytest.mark.parametrize("D", [1, 2, 4])
def test_gqa_with_rope_sharded_rows_and_tail_equal_unsharded(D):
    shape, inp = _small(S=2 * D * 8, d=32, H=4, inter=24, D=D, seed=80 + D, Hkv=2)
    inp = {k: v.to(torch.float64) for k, v in inp.items()}
    inp["rope_base"] = 1000.0
    y, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    ys = O.block_fwd_sharded(inp["x"], inp, shape.H, D, shape.eps)
    assert np.max(np.abs(ys - y)) <= 1e-12 * np.max(np.abs(y))
    rows = np.array([0, 3, shape.S - 1])
    yr = O.block_fwd_rows(inp["x"], inp, shape.H, shape.eps, rows)
    assert np.max(np.abs(yr - y[rows])) <= 1e-12 * np.max(np.abs(y))
    g = O.block_bwd(inp["x"], inp, inp["dy"], shape.H, shape.eps)
    gs = O.block_bwd_sharded(inp["x"], inp, inp["dy"], shape.H, D, shape.eps)
    for k in GRAD_OF:
        assert np.max(np.abs(gs[k] - g[k])) <= 1e-12 * np.max(np.abs(g[k])), k
    tail = O.block_bwd_tail(inp["x"], inp, inp["dy"], shape.H, shape.eps, 5)
    assert np.max(np.abs(tail - g["dx"][-5:])) <= 1e-12 * np.max(np.abs(g["dx"]))
    # finite differences through RoPE on grouped K heads
    rng = np.random.default_rng(9)
    step = 1e-6
    for gname, pname in (("dwk", "wk"), ("dwv", "wv")):
        base = inp[pname]
        v = torch.from_numpy(rng.standard_normal(tuple(base.shape)))
        plus, minus = dict(inp), dict(inp)
        plus[pname] = base + step * v
        minus[pname] = base - step * v
        fd = (_loss(plus, shape.H, shape.eps) - _loss(minus, shape.H, shape.eps)) / (2 * step)
        an = float(np.sum(g[gname] * v.numpy()))
        assert abs(fd - an) <= 1e-6 * abs(an), (gname, fd, an)


# ------------------------------------------------------------------ inference: KV cache, decode (variant)

@pytest.mark.parametrize("Hkv,base", [(0, 0.0), (2, 500.0)])
def test_kv_cache_rows_follow_the_zigzag_layout(Hkv, base):
    """Cache row i holds K/V of the token the hand-worked zigzag map puts at
    buffer row i; K and V are torch's own projections (rotated by the closed
    form for RoPE)."""
    shape, inp = _small(S=12, d=16, H=4, inter=24, D=3, seed=90, Hkv=Hkv)
    inp = {k: v.to(torch.float64) for k, v in inp.items()}
    if base:
        inp["rope_base"] = base
    cache = O.kv_cache_zigzag(inp["x"], inp, shape.H, shape.eps, 3)
    a = F.rms_norm(inp["x"], (16,), inp["g_attn"], eps=shape.eps)
    K = F.linear(a, inp["wk"]).numpy()
    V = F.linear(a, inp["wv"]).numpy()
    if base:
        dh, half = 4, 2
        for p in range(12):
            for h in range(K.shape[1] // dh):
                for j in range(half):
                    ang = p * base ** (-2.0 * j / dh)
                    x1, x2 = K[p, h * dh + j], K[p, h * dh + j + half]
                    K[p, h * dh + j] = x1 * math.cos(ang) - x2 * math.sin(ang)
                    K[p, h * dh + j + half] = x1 * math.sin(ang) + x2 * math.cos(ang)
    # buffer row -> global position, from the hand-worked S=12, D=3 fixture
    pos_of_row = {int(r[0]): int(r[1]) for r in _load("zigzag_S12_D3.txt")}
    want = np.concatenate([K, V], axis=1)
    for row in range(12):
        assert np.allclose(cache[row], want[pos_of_row[row]], atol=1e-13), row


@pytest.mark.parametrize("Hkv,base", [(0, 0.0), (2, 1000.0)])
def test_decode_steps_match_torch_full_forward(Hkv, base):
    """Decoding 1, 3 and 2 tokens after a prompt gives the rows of torch's
    causal block forward over the whole sequence."""
    S = 16
    shape, inp = _small(S=S + 6, d=32, H=4, inter=24, D=2, seed=95, Hkv=Hkv)
    inp = {k: v.to(torch.float64) for k, v in inp.items()}
    if base:
        inp["rope_base"] = base
    x = inp["x"].numpy()
    outs = O.block_decode(x[:S], [x[S:S + 1], x[S + 1:S + 4], x[S + 4:S + 6]], inp, shape.H,
                          shape.eps)
    if base:   # torch has no rotary block here: compare with the oracle's own full forward,
        # itself pinned against torch with RoPE off and by the RoPE pins above
        y, _ = O.block_fwd(x, inp, shape.H, shape.eps)
    else:
        y = _torch_block({k: v for k, v in inp.items() if k != "rope_base"}, shape.H,
                         shape.eps)[0].detach().numpy()
    got = np.concatenate(outs, axis=0)
    assert got.shape == (6, 32)
    assert np.max(np.abs(got - y[S:])) < 1e-11


# ------------------------------------------------------------------ per-rank steps of the schedule

def test_mirrored_row_pairs_each_attend_S_plus_1_keys():
    """Closed form: position p attends p + 1 keys; a mirrored pair of virtual
    rank r attends S + 1 keys in all, and n = c pairs are exactly rank r's
    zigzag rows."""
    for S, D in ((48, 3), (256, 4), (16384, 8)):
        c = S // (2 * D)
        for r in range(D):
            n = min(c, 5)
            p = O.mirrored_rows(S, D, r, n)
            keys = p + 1
            assert np.all(keys[:n] + keys[n:][::-1] == S + 1)
            full = O.mirrored_rows(S, D, r, c)
            zz = O.zigzag_positions(S, D)[r * 2 * c:(r + 1) * 2 * c]
            assert np.array_equal(np.sort(full), np.sort(zz))


def test_gather_kv_is_the_unsharded_projection():
    shape, inp = _small(S=48, d=24, H=3, inter=40, D=3, seed=61)
    K_all, V_all = O.gather_kv(inp["x"], inp, shape.H, shape.D, shape.eps)
    _, s = O.attn_block_fwd(inp["x"], inp, shape.H, shape.eps)
    assert np.max(np.abs(K_all - s["K"])) <= 1e-12 * np.max(np.abs(s["K"]))
    assert np.max(np.abs(V_all - s["V"])) <= 1e-12 * np.max(np.abs(s["V"]))


@pytest.mark.parametrize("D,n", [(3, 2), (4, 8), (2, 1)])
def test_rank_step_on_mirrored_rows_is_the_block_at_those_rows(D, n):
    """One virtual rank's step on a subset of its rows (its own Q/K/V
    projection, attention against the gathered K/V, the W_O loop and the MLP
    ring) gives the unsharded block's output at exactly those positions."""
    shape, inp = _small(S=2 * D * 8, d=16, H=2, inter=24, D=D, seed=62 + D)
    S, c = shape.S, shape.S // (2 * D)
    yb, _ = O.block_fwd(inp["x"], inp, shape.H, shape.eps)
    K_all, V_all = O.gather_kv(inp["x"], inp, shape.H, D, shape.eps)
    x = O.f64(inp["x"])
    for r in range(D):
        p = O.mirrored_rows(S, D, r, n)
        Q_r, _, _ = O.rank_project(x[p], p, inp, shape.H, D, shape.eps)
        y_r = O.rank_fwd(r, x[p], p, Q_r, K_all, V_all, inp, shape.H, D, shape.eps, c)
        assert np.max(np.abs(y_r - yb[p])) <= 1e-12 * np.max(np.abs(yb)), r


@pytest.mark.parametrize("Hkv,base", [(0, 0.0), (2, 10000.0)])
def test_backward_of_sparse_dy_is_the_dense_backward(Hkv, base):
    """block_bwd_rows (the gradients when dy is non-zero on a few rows only,
    computed without the other rows' forward) against the dense block_bwd
    with the same dy, including grouped K/V heads and the rotary embedding;
    a key reached only by later rows, and the last position, are among the
    cases."""
    shape = BlockShape(S=64, d=32, H=4, inter=48, D=2, Hkv=Hkv)
    inp = make_block_inputs(shape, torch.float32, seed=5 + Hkv, with_dy=True)
    if base:
        inp["rope_base"] = base
    for rows in (np.array([3, 17, 40, 63]), np.array([0, 31, 32, 50])):
        dy = O.f64(inp["dy"])
        dys = np.zeros_like(dy)
        dys[rows] = dy[rows]
        ref = O.block_bwd(inp["x"], inp, dys, shape.H, shape.eps)
        got = O.block_bwd_rows(inp["x"], inp, dy[rows], rows, shape.H, shape.eps)
        for k, v in ref.items():
            assert np.max(np.abs(got[k] - v)) <= 1e-12 * max(1e-30, np.max(np.abs(v))), (k, rows)
