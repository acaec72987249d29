"""CPU float64 oracle for the TSP-folded transformer block.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package's smoke check and
the benchmark's CPU-baseline leg may import this module; the library never
does, and it shares no code with the CUDA path.

Source pages (cited below by short tag):
  [TSP]  "Folding Tensor and Sequence Parallelism for Memory-Efficient
         Transformer Training & Inference" (gist.science summaries, Arabic and
         Japanese editions).  Section 2 ("Methodology: TSP") defines the fold:
         every rank holds 1/D of the parameters and 1/D of the tokens
         (2, "Unified sharding"); attention layers walk the packed
         W_Q/W_K/W_V/W_O shards, project locally, all-gather K/V and run
         FlashAttention over zigzag-partitioned causal rows (2, "Runtime
         schedules", attention bullet); gated-MLP layers rotate W_1/W_2/W_3
         shards around a ring and accumulate partial outputs locally with no
         all-reduce (2, "Runtime schedules", gated-MLP bullet).
The pages give no formula for any step.  Where they are silent this module
takes the plain readings listed below; each one is also listed in the
design notes of the repository.

  R1  RMSNorm: rms(u) = u / sqrt(mean(u^2) + eps) * g, eps = 1e-6, learnable
      gain g, no bias (pre-norm block).
  R2  No biases anywhere; no positional encoding (NoPE) unless R12 is selected.
  R3  Attention: multi-head, scale 1/sqrt(dh), causal with the diagonal
      included (no row is ever fully masked).
  R4  Gated MLP: G = silu(b W_1^T) * (b W_3^T), y = h + G W_2^T
      (SiLU on the W_1 branch), silu(z) = z * sigmoid(z).
  R5  Zigzag: the S tokens are cut into 2D equal chunks of c = S/(2D); rank r
      owns chunks r and 2D-1-r, stored rank-major, chunk r first, ascending
      position inside each chunk.
  R6  Shards: contiguous column ranges with boundaries floor(k*n/D).
  R7  Shard arrival order: attention broadcasts shard k = 0..D-1 in turn;
      the MLP ring hands rank r shard (r - t) mod D at step t.
  R8  Backward: the exact gradient of the forward above; weight gradients of
      the virtual ranks are summed (what TSP's reduction to shard owners
      delivers).
  R12 Rotary position embedding (a variant, off by default): rotate-half
      form, pair (j, j + dh/2) of every head turned by pos * base^(-2j/dh)
      at the token's global position; Q and K only.  Selected by a
      "rope_base" entry next to the weights (0 or absent: none).
  R13 Grouped-query attention (a variant, off by default): H query heads
      share Hkv K/V heads, Hkv dividing H; query head h reads K/V head
      floor(h / (H / Hkv)), so consecutive query heads form a group.  The K/V
      head count follows from the shapes (W_K, W_V have Hkv*dh rows); Hkv = H
      is plain multi-head attention.
  R14 Inference (a variant the pages name in their title but do not
      detail): the prefill is the block forward over the prompt; the KV
      cache keeps the prompt's K (after R12's rotation, if selected) and V
      rows in zigzag row order, each virtual rank's 2c rows contiguous;
      decoded tokens are appended after the prompt in position order (they
      are not re-zigzagged).  A decode step's output is what the causal
      block forward over the whole sequence gives at the new positions.
  R11 Stack of L layers: plain composition, each layer its own weights.  The
      residual stream between layers is not rounded to the storage dtype (it
      stays fp32 on the GPU, as inside one block), so in this float64 oracle
      the stack is the exact composition of the blocks.

Every floating-point step runs in numpy float64; inputs are converted
exactly from their bf16/fp32 storage.  No step here rounds to bf16.

Parity pins: every function below is pinned by tests under tests/ against
closed forms, invariants, brute force and an independent library
evaluation (torch CPU float64); none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np
import torch

# ----------------------------------------------------------------------------
# Zigzag causal partitioning  [TSP 2, attention bullet: zigzag partitioning]
# ----------------------------------------------------------------------------


def zigzag_positions(S: int, D: int) -> np.ndarray:
    """Global token position held at every row of the rank-major zigzag buffer.

    Buffer row r*2c + slot*c + t holds chunk (r if slot == 0 else 2D-1-r),
    offset t, i.e. global position chunk*c + t (reading R5).
    """
    if D < 1 or S % (2 * D) != 0:
        raise ValueError("S must be a positive multiple of 2D")
    c = S // (2 * D)
    pos = np.empty(S, dtype=np.int64)
    row = 0
    for r in range(D):
        for chunk in (r, 2 * D - 1 - r):
            for t in range(c):
                pos[row] = chunk * c + t
                row += 1
    return pos


def zigzag_owner(S: int, D: int) -> np.ndarray:
    """Virtual rank that owns each global position (reading R5)."""
    c = S // (2 * D)
    chunk = np.arange(S) // c
    return np.where(chunk < D, chunk, 2 * D - 1 - chunk)


def zigzag_permute(x: np.ndarray, D: int, inverse: bool = False) -> np.ndarray:
    """Global order -> rank-major zigzag order (or back with ``inverse``)."""
    pos = zigzag_positions(x.shape[0], D)
    out = np.empty_like(x)
    if inverse:
        out[pos] = x
    else:
        out[:] = x[pos]
    return out


def causal_pairs_per_rank(S: int, D: int) -> np.ndarray:
    """Number of causal (query, key) pairs j <= i whose query rank r owns.

    Counted by brute force over the owner map; the closed form c*(S+1) for
    every rank is what zigzag balancing promises.
    """
    owner = zigzag_owner(S, D)
    pairs = np.zeros(D, dtype=np.int64)
    for i in range(S):
        pairs[owner[i]] += i + 1  # keys 0..i
    return pairs


def shard_bounds(n: int, D: int) -> list[int]:
    """Contiguous shard boundaries floor(k*n/D), k = 0..D (reading R6)."""
    return [(k * n) // D for k in range(D + 1)]


# ----------------------------------------------------------------------------
# Elementary layers
# ----------------------------------------------------------------------------


def f64(t) -> np.ndarray:
    """Exact conversion of a CPU torch tensor (bf16/fp32/fp64) or array to float64."""
    if hasattr(t, "detach"):
        import torch
        return t.detach().to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def rmsnorm(u: np.ndarray, g: np.ndarray, eps: float):
    """Reading R1.  Returns (u * rstd * g, rstd) with rstd = 1/sqrt(mean(u^2)+eps)."""
    rstd = 1.0 / np.sqrt(np.mean(u * u, axis=1) + eps)
    return u * rstd[:, None] * g[None, :], rstd


def sigmoid(z: np.ndarray) -> np.ndarray:
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def silu(z: np.ndarray) -> np.ndarray:
    return z * sigmoid(z)


def causal_attention(Q, K, V, H, q_pos=None, k_pos=None, row_block=512):
    """Softmax attention of every query row over the keys at positions <= its own.

    [TSP 2, attention bullet] runs FlashAttention over the gathered K/V; the
    value it computes is exact softmax attention (readings R3).  For query i
    and head h:  s_ij = q_i . k_j / sqrt(dh) for pos(j) <= pos(i),
    p_ij = exp(s_ij - m_i) / sum_j exp(s_ij - m_i),  o_i = sum_j p_ij v_j.
    Rows are evaluated a group at a time only to bound memory.

    With fewer K/V heads than query heads (reading R13) query head h reads
    K/V head h // (H / Hkv), Hkv = K.shape[1] / dh.

    Returns (O [nq, H*dh], LSE [H, nq]) with LSE_i = log sum_j exp(s_ij).
    """
    nq = Q.shape[0]
    nk = K.shape[0]
    dh = Q.shape[1] // H
    grp = H // (K.shape[1] // dh)
    if q_pos is None:
        q_pos = np.arange(nq)
    if k_pos is None:
        k_pos = np.arange(nk)
    scale = 1.0 / math.sqrt(dh)
    O = np.zeros((nq, H * dh))
    LSE = np.zeros((H, nq))
    for r0 in range(0, nq, row_block):
        r1 = min(nq, r0 + row_block)
        allowed = k_pos[None, :] <= q_pos[r0:r1, None]
        kmax = int(np.nonzero(allowed.any(axis=0))[0].max()) + 1 if allowed.any() else 0
        allowed = allowed[:, :kmax]
        for h in range(H):
            cols = slice(h * dh, (h + 1) * dh)
            kc = slice((h // grp) * dh, (h // grp + 1) * dh)
            s = (Q[r0:r1, cols] @ K[:kmax, kc].T) * scale
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            z = e.sum(axis=1, keepdims=True)
            O[r0:r1, cols] = (e / z) @ V[:kmax, kc]
            LSE[h, r0:r1] = (m + np.log(z))[:, 0]
    return O, LSE


def attention_probs(Q, K, H, q_pos=None, k_pos=None):
    """Full probability matrices P[h, i, j] (small inputs only; used by pins)."""
    nq, nk = Q.shape[0], K.shape[0]
    dh = Q.shape[1] // H
    grp = H // (K.shape[1] // dh)
    q_pos = np.arange(nq) if q_pos is None else q_pos
    k_pos = np.arange(nk) if k_pos is None else k_pos
    allowed = k_pos[None, :] <= q_pos[:, None]
    P = np.zeros((H, nq, nk))
    for h in range(H):
        cols = slice(h * dh, (h + 1) * dh)
        kc = slice((h // grp) * dh, (h // grp + 1) * dh)
        s = (Q[:, cols] @ K[:, kc].T) / math.sqrt(dh)
        s = np.where(allowed, s, -np.inf)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        P[h] = e / e.sum(axis=1, keepdims=True)
    return P


# ----------------------------------------------------------------------------
# Unsharded block (the value TSP must reproduce)
# ----------------------------------------------------------------------------


def _w(W, name):
    return f64(W[name])


def _rope_base(W):
    return float(W.get("rope_base", 0.0)) if hasattr(W, "get") else 0.0


def _kv_heads(W, H):
    """K/V head count of the weights: W_K rows / dh (reading R13)."""
    return W["wk"].shape[0] // (W["wq"].shape[0] // H)


def rope(X, pos, H, base, inverse=False):
    """Rotary position embedding (a variant; the pages' block has none,
    reading R12): within each head of width dh, element j < dh/2 pairs with
    element j + dh/2 and the pair turns by the angle pos * base^(-2j/dh);
    ``inverse`` applies the transposed rotation (the map of gradients).
    base = 0 leaves X as it is."""
    if not base:
        return X
    X = np.asarray(X, dtype=np.float64)
    d = X.shape[1]
    dh = d // H
    half = dh // 2
    f = float(base) ** (-2.0 * np.arange(half) / dh)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * f[None, :]
    cs, sn = np.cos(ang), np.sin(ang)
    if inverse:
        sn = -sn
    Y = X.copy()
    for h in range(H):
        a = X[:, h * dh:h * dh + half]
        b = X[:, h * dh + half:(h + 1) * dh]
        Y[:, h * dh:h * dh + half] = a * cs - b * sn
        Y[:, h * dh + half:(h + 1) * dh] = a * sn + b * cs
    return Y


def attn_block_fwd(x, W, H, eps):
    """h = x + Attn(rms(x; g_attn)) W_O^T.  Returns (h, saved dict)."""
    x = f64(x)
    a, rstd1 = rmsnorm(x, _w(W, "g_attn"), eps)
    p = np.arange(x.shape[0])
    Q = rope(a @ _w(W, "wq").T, p, H, _rope_base(W))
    K = rope(a @ _w(W, "wk").T, p, _kv_heads(W, H), _rope_base(W))
    V = a @ _w(W, "wv").T
    O, LSE = causal_attention(Q, K, V, H)
    h = x + O @ _w(W, "wo").T
    return h, dict(x=x, a=a, rstd1=rstd1, Q=Q, K=K, V=V, O=O, LSE=LSE)


def mlp_fwd(h, W, eps, norm=True, residual=True):
    """y = [h +] silu(b W_1^T) * (b W_3^T) W_2^T with b = rms(h; g_mlp) or b = h."""
    h = f64(h)
    if norm:
        b, rstd2 = rmsnorm(h, _w(W, "g_mlp"), eps)
    else:
        b, rstd2 = h, None
    A = b @ _w(W, "w1").T
    B = b @ _w(W, "w3").T
    G = silu(A) * B
    y = G @ _w(W, "w2").T
    if residual:
        y = h + y
    return y, dict(h=h, b=b, rstd2=rstd2, A=A, B=B, G=G)


def block_fwd(x, W, H, eps):
    """Pre-norm block: h = x + Attn(rms(x)), y = h + MLP(rms(h))."""
    h, s1 = attn_block_fwd(x, W, H, eps)
    y, s2 = mlp_fwd(h, W, eps)
    s1.update(s2)
    return y, s1


# ----------------------------------------------------------------------------
# Sharded emulation: D virtual ranks following the TSP schedules
# ----------------------------------------------------------------------------


def rank_project(x_r, pos_r, W, H, D, eps):
    """Step 2 of the attention schedule for one rank's rows x_r (global
    positions pos_r): a_r = rms(x_r; g_attn), then shard k = 0..D-1 of the
    packed W_Q/W_K/W_V columns arrives and the rank projects its own rows
    with it (K/V columns cut the same way over their own width, which is d
    unless reading R13 applies); Q and K are rotated at the rows' global
    positions when reading R12 applies.  Returns (Q_r, K_r, V_r)."""
    x_r = f64(x_r)
    wq, wk, wv = (_w(W, n) for n in ("wq", "wk", "wv"))
    d, dkv = wq.shape[0], wk.shape[0]
    Cb, Kb = shard_bounds(d, D), shard_bounds(dkv, D)
    a_r = rmsnorm(x_r, _w(W, "g_attn"), eps)[0]
    Q = np.zeros((x_r.shape[0], d)); K = np.zeros((x_r.shape[0], dkv)); V = np.zeros_like(K)
    for k in range(D):
        C, Ck = slice(Cb[k], Cb[k + 1]), slice(Kb[k], Kb[k + 1])
        Q[:, C] = a_r @ wq[C].T
        K[:, Ck] = a_r @ wk[Ck].T
        V[:, Ck] = a_r @ wv[Ck].T
    Q = rope(Q, pos_r, H, _rope_base(W))
    K = rope(K, pos_r, _kv_heads(W, H), _rope_base(W))
    return Q, K, V


def rank_fwd(r, x_r, pos_r, Q_r, K_all, V_all, W, H, D, eps, c, parts=("attn", "mlp")):
    """Steps 4-6 of the schedule for virtual rank r, given the gathered K/V.

    x_r, pos_r: the rank's rows and their global positions; Q_r from
    rank_project; K_all, V_all: the all-gathered keys and values of the whole
    sequence, row p holding position p.  Attention of the rank's rows runs
    chunk by chunk (chunk length c) against the keys at positions <= each
    query's own; the rank accumulates O[:, C_k] W_O[:, C_k]^T shard by shard
    onto its residual rows; then the MLP ring hands it shard (r - t) mod D of
    W_1/W_3 (rows) and W_2 (columns) at step t and it accumulates
    G[:, I_k] W_2[:, I_k]^T onto its rows.  ``parts`` selects the halves.
    Returns y_r (h_r if only the attention half runs)."""
    x_r = f64(x_r)
    pos_r = np.asarray(pos_r)
    h_r = x_r.copy()
    if "attn" in parts:
        wo = _w(W, "wo")
        Cb = shard_bounds(wo.shape[0], D)
        O_r = np.zeros_like(Q_r)
        kpos = np.arange(K_all.shape[0])
        for ch in np.unique(pos_r // c):        # each chunk's rows have ascending positions
            sel = np.nonzero(pos_r // c == ch)[0]
            O_r[sel], _ = causal_attention(Q_r[sel], K_all, V_all, H, q_pos=pos_r[sel], k_pos=kpos)
        for k in range(D):
            C = slice(Cb[k], Cb[k + 1])
            h_r += O_r[:, C] @ wo[:, C].T
    y_r = h_r.copy()
    if "mlp" in parts:
        w1, w3, w2 = (_w(W, n) for n in ("w1", "w3", "w2"))
        Ib = shard_bounds(w1.shape[0], D)
        b_r = rmsnorm(h_r, _w(W, "g_mlp"), eps)[0]
        for t in range(D):
            k = (r - t) % D
            I = slice(Ib[k], Ib[k + 1])
            G = silu(b_r @ w1[I].T) * (b_r @ w3[I].T)
            y_r += G @ w2[:, I].T
    return y_r


def gather_kv(x, W, H, D, eps):
    """The K/V all-gather: every rank projects its own zigzag rows
    (rank_project) and the rows are placed at their global positions.
    Returns (K_all, V_all) in position order."""
    x = f64(x)
    S = x.shape[0]
    c = S // (2 * D)
    pos = zigzag_positions(S, D)
    dkv = W["wk"].shape[0]
    K_all = np.zeros((S, dkv)); V_all = np.zeros((S, dkv))
    for r in range(D):
        R = pos[r * 2 * c:(r + 1) * 2 * c]
        _, K_all[R], V_all[R] = rank_project(x[R], R, W, H, D, eps)
    return K_all, V_all


def block_fwd_sharded(x, W, H, D, eps, parts=("attn", "mlp")):
    """The TSP schedule, one virtual rank at a time, in float64.

    1. zigzag-partition the tokens (reading R5): rank r holds chunks r and
       2D-1-r;
    2. attention broadcast loop: every rank projects its own rows with each
       arriving shard (rank_project);
    3. "all-gather" of K/V: every rank's K/V rows placed at their global
       positions (gather_kv);
    4.-6. per rank: causal attention of its rows against the gathered K/V,
       the W_O shard loop onto its residual rows, the MLP ring (rank_fwd);
    7. un-permute.
    ``parts`` selects which half runs (both by default); the MLP half keeps
    its norm and residual.
    """
    x = f64(x)
    S = x.shape[0]
    c = S // (2 * D)
    pos = zigzag_positions(S, D)
    K_all = V_all = None
    if "attn" in parts:
        K_all, V_all = gather_kv(x, W, H, D, eps)
    out = np.empty_like(x)
    for r in range(D):
        R = pos[r * 2 * c:(r + 1) * 2 * c]
        Q_r = rank_project(x[R], R, W, H, D, eps)[0] if "attn" in parts else None
        out[R] = rank_fwd(r, x[R], R, Q_r, K_all, V_all, W, H, D, eps, c, parts)
    return out


def mirrored_rows(S, D, r, n):
    """n mirrored row pairs of virtual rank r, as global positions: the first
    n rows of chunk r and the last n rows of chunk 2D-1-r.  Row i of chunk r
    (position r*c + i) attends r*c + i + 1 keys and its mirror (position
    (2D-r)*c - 1 - i) attends (2D-r)*c - i, so every pair attends S + 1 keys:
    a set of mirrored pairs carries exactly the block's average work per
    token (the balance the zigzag layout is built for)."""
    c = S // (2 * D)
    lo = r * c + np.arange(n)
    hi = (2 * D - 1 - r) * c + c - n + np.arange(n)
    return np.concatenate([lo, hi])


def mlp_fwd_sharded(h, W, D, eps, norm=True, residual=True):
    """The gated-MLP ring on its own: rank r accumulates shards (r - t) mod D."""
    h = f64(h)
    S = h.shape[0]
    c = S // (2 * D)
    pos = zigzag_positions(S, D)
    hz = h[pos]
    w1, w3, w2 = (_w(W, n) for n in ("w1", "w3", "w2"))
    Ib = shard_bounds(w1.shape[0], D)
    yz = hz.copy() if residual else np.zeros_like(hz)
    for r in range(D):
        R = slice(r * 2 * c, (r + 1) * 2 * c)
        b_r = rmsnorm(hz[R], _w(W, "g_mlp"), eps)[0] if norm else hz[R]
        for t in range(D):
            k = (r - t) % D
            I = slice(Ib[k], Ib[k + 1])
            yz[R] += (silu(b_r @ w1[I].T) * (b_r @ w3[I].T)) @ w2[:, I].T
    out = np.empty_like(yz)
    out[pos] = yz
    return out


# ----------------------------------------------------------------------------
# Sampled rows of a large forward (exact on the rows it returns)
# ----------------------------------------------------------------------------


def block_fwd_rows(x, W, H, eps, rows, attn_only=False):
    """y (or h with ``attn_only``) at the given global positions only.

    Keys and values are needed at every position <= max(rows); queries,
    attention, W_O and the MLP only at the requested rows (every step after
    K/V is row-local).
    """
    x = f64(x)
    rows = np.asarray(rows, dtype=np.int64)
    kmax = int(rows.max()) + 1
    g1 = _w(W, "g_attn")
    a_all = rmsnorm(x[:kmax], g1, eps)[0]
    K = rope(a_all @ _w(W, "wk").T, np.arange(kmax), _kv_heads(W, H), _rope_base(W))
    V = a_all @ _w(W, "wv").T
    Q = rope(a_all[rows] @ _w(W, "wq").T, rows, H, _rope_base(W))
    O, _ = causal_attention(Q, K, V, H, q_pos=rows, k_pos=np.arange(kmax))
    h = x[rows] + O @ _w(W, "wo").T
    if attn_only:
        return h
    return mlp_fwd(h, W, eps)[0]


# ----------------------------------------------------------------------------
# Inference: KV cache and decode (reading R14)
# ----------------------------------------------------------------------------


def kv_cache_zigzag(x, W, H, eps, D):
    """Cache rows of a prompt x [S, d]: row i = [K | V] of the token at
    position zigzag_positions(S, D)[i] ([TSP 2, attention bullet]: every rank
    keeps the K/V of its own zigzag rows).  Returns [S, 2 * K-width]."""
    x = f64(x)
    S = x.shape[0]
    a, _ = rmsnorm(x, _w(W, "g_attn"), eps)
    K = rope(a @ _w(W, "wk").T, np.arange(S), _kv_heads(W, H), _rope_base(W))
    V = a @ _w(W, "wv").T
    pos = zigzag_positions(S, D)
    return np.concatenate([K[pos], V[pos]], axis=1)


def block_decode(x_prompt, steps, W, H, eps):
    """Outputs of consecutive decode steps after a prompt.

    ``steps`` is a list of [T_k, d] arrays: step k's tokens follow the prompt
    and every earlier step's tokens.  Each step's output is the causal block
    forward over the whole sequence so far, at the step's positions (reading
    R14), evaluated row-wise with block_fwd_rows.  Returns a list of [T_k, d].
    """
    seq = [f64(x_prompt)]
    n = seq[0].shape[0]
    outs = []
    for xs in steps:
        xs = f64(xs)
        seq.append(xs)
        rows = np.arange(n, n + xs.shape[0])
        outs.append(block_fwd_rows(np.concatenate(seq, axis=0), W, H, eps, rows))
        n += xs.shape[0]
    return outs


# ----------------------------------------------------------------------------
# Backward: exact gradient of block_fwd (reading R8)
# ----------------------------------------------------------------------------


def rmsnorm_bwd(dout, u, g, rstd):
    """Gradient of n*g, n = u*rstd, rstd = (mean(u^2)+eps)^-1/2.

    dg = sum_rows dout*n;  du = rstd * (dout*g - n * mean_cols(dout*g*n)).
    """
    n = u * rstd[:, None]
    dg = (dout * n).sum(axis=0)
    gd = dout * g[None, :]
    du = rstd[:, None] * (gd - n * np.mean(gd * n, axis=1, keepdims=True))
    return du, dg


def causal_attention_bwd(Q, K, V, O, dO, H, q_pos=None, k_pos=None, row_block=512):
    """dQ, dK, dV of causal_attention.

    With P the probabilities:  dV = P^T dO,  dP = dO V^T,
    Delta_i = sum_c dO_ic O_ic,  dS = P * (dP - Delta),
    dQ = dS K / sqrt(dh),  dK = dS^T Q / sqrt(dh).  The sums over query
    rows are taken a row group at a time only to bound memory; with grouped
    K/V heads (reading R13) a K/V head's dK and dV sum over its group's query
    heads.
    """
    nq, nk = Q.shape[0], K.shape[0]
    dh = Q.shape[1] // H
    grp = H // (K.shape[1] // dh)
    q_pos = np.arange(nq) if q_pos is None else q_pos
    k_pos = np.arange(nk) if k_pos is None else k_pos
    scale = 1.0 / math.sqrt(dh)
    dQ = np.zeros_like(Q); dK = np.zeros_like(K); dV = np.zeros_like(V)
    for r0 in range(0, nq, row_block):
        r1 = min(nq, r0 + row_block)
        allowed = k_pos[None, :] <= q_pos[r0:r1, None]
        kmax = int(np.nonzero(allowed.any(axis=0))[0].max()) + 1
        allowed = allowed[:, :kmax]
        for h in range(H):
            cols = slice(h * dh, (h + 1) * dh)
            kc = slice((h // grp) * dh, (h // grp + 1) * dh)
            s = (Q[r0:r1, cols] @ K[:kmax, kc].T) * scale
            s = np.where(allowed, s, -np.inf)
            e = np.exp(s - s.max(axis=1, keepdims=True))
            P = e / e.sum(axis=1, keepdims=True)
            do = dO[r0:r1, cols]
            dV[:kmax, kc] += P.T @ do
            dP = do @ V[:kmax, kc].T
            delta = (do * O[r0:r1, cols]).sum(axis=1, keepdims=True)
            dS = P * (dP - delta)
            dQ[r0:r1, cols] = (dS @ K[:kmax, kc]) * scale
            dK[:kmax, kc] += (dS.T @ Q[r0:r1, cols]) * scale
    return dQ, dK, dV


def stack_fwd(x, Ws, H, eps):
    """y of an L-layer stack: the blocks applied in order, each with its own
    weights Ws[l] ([TSP] sections 1-3: the fold is applied to every layer of
    the model; the stack is plain composition, reading R11)."""
    y = f64(x)
    for W in Ws:
        y, _ = block_fwd(y, W, H, eps)
    return y


def stack_bwd(x, Ws, dy, H, eps):
    """dx and per-layer gradients of L = sum(dy * y), y = stack_fwd(x): the
    chain rule through the layers, the dx of layer l being the dy of layer
    l - 1.  Returns (dx, [dict of layer l's weight and gain gradients])."""
    xs = [f64(x)]
    for W in Ws[:-1]:
        xs.append(block_fwd(xs[-1], W, H, eps)[0])
    g = f64(dy)
    grads = [None] * len(Ws)
    for l in range(len(Ws) - 1, -1, -1):
        gl = block_bwd(xs[l], Ws[l], g, H, eps)
        g = gl.pop("dx")
        grads[l] = gl
    return g, grads


def block_bwd(x, W, dy, H, eps):
    """All gradients of L = sum(dy * y) for y = block_fwd(x).

    Returns dict: dx, dwq, dwk, dwv, dwo, dw1, dw3, dw2, dg_attn, dg_mlp.
    """
    y, s = block_fwd(x, W, H, eps)
    dy = f64(dy)
    w1, w3, w2 = _w(W, "w1"), _w(W, "w3"), _w(W, "w2")
    # MLP
    dw2 = dy.T @ s["G"]
    dG = dy @ w2
    sA = sigmoid(s["A"])
    silu_A = s["A"] * sA
    dA = dG * s["B"] * sA * (1.0 + s["A"] * (1.0 - sA))
    dB = dG * silu_A
    dw1 = dA.T @ s["b"]
    dw3 = dB.T @ s["b"]
    db = dA @ w1 + dB @ w3
    du2, dg_mlp = rmsnorm_bwd(db, s["h"], _w(W, "g_mlp"), s["rstd2"])
    dh = dy + du2
    # attention
    wq, wk, wv, wo = (_w(W, n) for n in ("wq", "wk", "wv", "wo"))
    dwo = dh.T @ s["O"]
    dO = dh @ wo
    dQ, dK, dV = causal_attention_bwd(s["Q"], s["K"], s["V"], s["O"], dO, H)
    p = np.arange(s["x"].shape[0])
    dQ = rope(dQ, p, H, _rope_base(W), inverse=True)   # back through the rotation
    dK = rope(dK, p, _kv_heads(W, H), _rope_base(W), inverse=True)
    dwq = dQ.T @ s["a"]
    dwk = dK.T @ s["a"]
    dwv = dV.T @ s["a"]
    da = dQ @ wq + dK @ wk + dV @ wv
    du1, dg_attn = rmsnorm_bwd(da, s["x"], _w(W, "g_attn"), s["rstd1"])
    dx = dh + du1
    return dict(dx=dx, dwq=dwq, dwk=dwk, dwv=dwv, dwo=dwo, dw1=dw1, dw3=dw3,
                dw2=dw2, dg_attn=dg_attn, dg_mlp=dg_mlp)


def block_bwd_rows(x, W, dy_rows, rows, H, eps):
    """All gradients of L = sum over the given positions of dy_rows * y, that
    is block_bwd with dy zero at every other position, computed exactly
    without the forward of the other rows.

    The MLP, W_O and the query side of attention are row-local, so they run on
    the given rows only; the keys and values at positions <= max(rows) are
    projected for all of those positions, and the attention backward of the
    given query rows reaches every one of them (dK, dV), so the K/V weight
    gradients, the first RMSNorm's backward and dx cover positions
    0 .. max(rows).  Returns the dict of block_bwd (dx over all S positions).
    """
    x = f64(x)
    dy_r = f64(dy_rows)
    rows = np.asarray(rows, dtype=np.int64)
    S = x.shape[0]
    kmax = int(rows.max()) + 1
    keys = np.arange(kmax)
    g1, g2 = _w(W, "g_attn"), _w(W, "g_mlp")
    wq, wk, wv, wo = (_w(W, n) for n in ("wq", "wk", "wv", "wo"))
    w1, w3, w2 = _w(W, "w1"), _w(W, "w3"), _w(W, "w2")
    Hk = _kv_heads(W, H)
    # forward: keys and values of positions < kmax, the rest at the rows
    a_all, rstd1 = rmsnorm(x[:kmax], g1, eps)
    K = rope(a_all @ wk.T, keys, Hk, _rope_base(W))
    V = a_all @ wv.T
    a_r = a_all[rows]
    Q_r = rope(a_r @ wq.T, rows, H, _rope_base(W))
    O_r, _ = causal_attention(Q_r, K, V, H, q_pos=rows, k_pos=keys)
    h_r = x[rows] + O_r @ wo.T
    b_r, rstd2 = rmsnorm(h_r, g2, eps)
    A = b_r @ w1.T
    B = b_r @ w3.T
    sA = sigmoid(A)
    G = A * sA * B
    # MLP backward at the rows
    dw2 = dy_r.T @ G
    dG = dy_r @ w2
    dA = dG * B * sA * (1.0 + A * (1.0 - sA))
    dB = dG * A * sA
    dw1 = dA.T @ b_r
    dw3 = dB.T @ b_r
    du2, dg_mlp = rmsnorm_bwd(dA @ w1 + dB @ w3, h_r, g2, rstd2)
    dh_r = dy_r + du2
    # attention backward: the rows' queries against every key they see
    dwo = dh_r.T @ O_r
    dO_r = dh_r @ wo
    dQ_r, dK, dV = causal_attention_bwd(Q_r, K, V, O_r, dO_r, H, q_pos=rows, k_pos=keys)
    dQ_r = rope(dQ_r, rows, H, _rope_base(W), inverse=True)
    dK = rope(dK, keys, Hk, _rope_base(W), inverse=True)
    dwq = dQ_r.T @ a_r
    dwk = dK.T @ a_all
    dwv = dV.T @ a_all
    da = dK @ wk + dV @ wv
    da[rows] += dQ_r @ wq
    du1, dg_attn = rmsnorm_bwd(da, x[:kmax], g1, rstd1)
    dx = np.zeros_like(x)
    dx[:kmax] = du1
    dx[rows] += dh_r
    return dict(dx=dx, dwq=dwq, dwk=dwk, dwv=dwv, dwo=dwo, dw1=dw1, dw3=dw3,
                dw2=dw2, dg_attn=dg_attn, dg_mlp=dg_mlp)


def block_bwd_sharded(x, W, dy, H, D, eps):
    """Backward in the D-virtual-rank layout.

    Activations stay on their zigzag rows; every rank contributes the weight
    and gain gradients of its own 2c rows and they are summed over ranks
    (reading R8).  dK/dV reach a key's owner from every rank whose queries
    attend to it (summed over the query ranks).  dx is returned in global
    order.
    """
    x = f64(x)
    dy = f64(dy)
    S, d = x.shape
    c = S // (2 * D)
    pos = zigzag_positions(S, D)
    R = [slice(r * 2 * c, (r + 1) * 2 * c) for r in range(D)]
    xz, dyz = x[pos], dy[pos]
    g1, g2 = _w(W, "g_attn"), _w(W, "g_mlp")
    wq, wk, wv, wo = (_w(W, n) for n in ("wq", "wk", "wv", "wo"))
    w1, w3, w2 = _w(W, "w1"), _w(W, "w3"), _w(W, "w2")
    # forward, per rank (row-local steps) + gathered K/V
    az = np.zeros_like(xz); rstd1 = np.zeros(S)
    for r in range(D):
        az[R[r]], rstd1[R[r]] = rmsnorm(xz[R[r]], g1, eps)
    Qz, Kz, Vz = az @ wq.T, az @ wk.T, az @ wv.T
    Qz = rope(Qz, pos, H, _rope_base(W))
    Kz = rope(Kz, pos, _kv_heads(W, H), _rope_base(W))
    Oz = np.zeros_like(xz)
    for r in range(D):
        Oz[R[r]] = causal_attention(Qz[R[r]], Kz, Vz, H, q_pos=pos[R[r]], k_pos=pos)[0]
    hz = xz + Oz @ wo.T
    grads = {k: 0.0 for k in ("dwq", "dwk", "dwv", "dwo", "dw1", "dw3", "dw2", "dg_attn", "dg_mlp")}
    dOz = np.zeros_like(xz); dhz = np.zeros_like(xz)
    for r in range(D):
        h_r = hz[R[r]]
        b_r, rstd2 = rmsnorm(h_r, g2, eps)
        A = b_r @ w1.T; B = b_r @ w3.T
        sA = sigmoid(A)
        G = A * sA * B
        dy_r = dyz[R[r]]
        grads["dw2"] = grads["dw2"] + dy_r.T @ G
        dG = dy_r @ w2
        dA = dG * B * sA * (1.0 + A * (1.0 - sA))
        dB = dG * A * sA
        grads["dw1"] = grads["dw1"] + dA.T @ b_r
        grads["dw3"] = grads["dw3"] + dB.T @ b_r
        du2, dg2 = rmsnorm_bwd(dA @ w1 + dB @ w3, h_r, g2, rstd2)
        grads["dg_mlp"] = grads["dg_mlp"] + dg2
        dhz[R[r]] = dy_r + du2
        grads["dwo"] = grads["dwo"] + dhz[R[r]].T @ Oz[R[r]]
        dOz[R[r]] = dhz[R[r]] @ wo
    dQz = np.zeros_like(xz); dKz = np.zeros_like(Kz); dVz = np.zeros_like(Vz)
    for r in range(D):
        dq, dk, dv = causal_attention_bwd(Qz[R[r]], Kz, Vz, Oz[R[r]], dOz[R[r]], H,
                                          q_pos=pos[R[r]], k_pos=pos)
        dQz[R[r]] = dq
        dKz += dk            # returned to the key owners
        dVz += dv
    dQz = rope(dQz, pos, H, _rope_base(W), inverse=True)
    dKz = rope(dKz, pos, _kv_heads(W, H), _rope_base(W), inverse=True)
    dxz = np.zeros_like(xz)
    for r in range(D):
        a_r = az[R[r]]
        grads["dwq"] = grads["dwq"] + dQz[R[r]].T @ a_r
        grads["dwk"] = grads["dwk"] + dKz[R[r]].T @ a_r
        grads["dwv"] = grads["dwv"] + dVz[R[r]].T @ a_r
        da = dQz[R[r]] @ wq + dKz[R[r]] @ wk + dVz[R[r]] @ wv
        du1, dg1 = rmsnorm_bwd(da, xz[R[r]], g1, rstd1[R[r]])
        grads["dg_attn"] = grads["dg_attn"] + dg1
        dxz[R[r]] = dhz[R[r]] + du1
    dx = np.empty_like(dxz)
    dx[pos] = dxz
    grads["dx"] = dx
    return grads


def block_bwd_tail(x, W, dy, H, eps, n_tail):
    """dx of L = sum(dy * y) at the last n_tail positions, exactly.

    A key at position >= S - n_tail is attended only by queries at positions
    >= its own, all inside the tail, so its dK and dV are complete once the
    tail queries are back-propagated; dQ of a tail query needs every key, which
    only takes the K/V projections of all rows.  Everything else is row-local.
    Returns dx[S - n_tail:] (global order).
    """
    x = f64(x)
    dy = f64(dy)
    S = x.shape[0]
    t0 = S - n_tail
    g1, g2 = _w(W, "g_attn"), _w(W, "g_mlp")
    wq, wk, wv, wo = (_w(W, n) for n in ("wq", "wk", "wv", "wo"))
    w1, w3, w2 = _w(W, "w1"), _w(W, "w3"), _w(W, "w2")
    a_all, rstd1 = rmsnorm(x, g1, eps)
    tail = np.arange(t0, S)
    keys = np.arange(S)
    K = rope(a_all @ wk.T, keys, _kv_heads(W, H), _rope_base(W))
    V = a_all @ wv.T
    Q_t = rope(a_all[t0:] @ wq.T, tail, H, _rope_base(W))
    O_t, _ = causal_attention(Q_t, K, V, H, q_pos=tail, k_pos=keys)
    h_t = x[t0:] + O_t @ wo.T
    b_t, rstd2 = rmsnorm(h_t, g2, eps)
    A = b_t @ w1.T
    B = b_t @ w3.T
    sA = sigmoid(A)
    dG = dy[t0:] @ w2
    dA = dG * B * sA * (1.0 + A * (1.0 - sA))
    dB = dG * A * sA
    du2, _ = rmsnorm_bwd(dA @ w1 + dB @ w3, h_t, g2, rstd2)
    dh_t = dy[t0:] + du2
    dO_t = dh_t @ wo
    dQ_t, dK, dV = causal_attention_bwd(Q_t, K, V, O_t, dO_t, H, q_pos=tail, k_pos=keys)
    dQ_t = rope(dQ_t, tail, H, _rope_base(W), inverse=True)
    dK_t = rope(dK[t0:], tail, _kv_heads(W, H), _rope_base(W), inverse=True)
    da = dQ_t @ wq + dK_t @ wk + dV[t0:] @ wv
    du1, _ = rmsnorm_bwd(da, x[t0:], g1, rstd1[t0:])
    return dh_t + du1

