"""Per-rank memory account of the fold against the other layouts the pages
compare (host only, no GPU).  The pages state the claim in words: the fold is
the only layout that cuts both weight and activation memory per rank by the
degree D without D^2 devices; these checks pin the account to that claim, to
closed forms of the parameter count, and to the buffers the kernels use."""
import pytest
import torch

from folded_tensor_sequence_zigzag_gb300 import build, tsp

M = (tsp.TSP_MEM_TSP, tsp.TSP_MEM_DP, tsp.TSP_MEM_TP, tsp.TSP_MEM_SP, tsp.TSP_MEM_TP_SP)


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return tsp.load()


def _cfg(S=16384, d=4096, H=32, I=11008, D=8, dtype=torch.bfloat16):
    return tsp.make_cfg(S, d, H, I, D, dtype)


def _all(cfg, L, training):
    return {m: tsp.rank_memory(cfg, L, training, m) for m in M}


@pytest.mark.parametrize("training", [True, False])
@pytest.mark.parametrize("D", [1, 2, 8])
def test_shares_follow_the_layouts(training, D):
    cfg = _cfg(D=D)
    r = _all(cfg, 4, training)
    tsp_, dp, tp, sp, tpsp = (r[m] for m in M)
    assert tsp_["weights"] * D == pytest.approx(dp["weights"])
    assert tsp_["activations"] * D == pytest.approx(dp["activations"])
    assert tp["weights"] == pytest.approx(tsp_["weights"]) and tp["activations"] == dp["activations"]
    assert sp["weights"] == dp["weights"] and sp["activations"] == pytest.approx(tsp_["activations"])
    assert tpsp["devices"] == D * D and tsp_["devices"] == D
    for m in M:
        v = r[m]
        assert v["total"] == pytest.approx(v["weights"] + v["activations"] + v["transient"])


def test_weights_closed_form():
    d, I, L = 4096, 11008, 32
    r = tsp.rank_memory(_cfg(d=d, I=I), L, True, tsp.TSP_MEM_DP)
    assert r["weights"] == L * (4 * d * d + 3 * d * I + 2 * d) * 2        # bf16
    r32 = tsp.rank_memory(_cfg(S=256, d=64, H=4, I=128, D=4, dtype=torch.float32), 3, True,
                          tsp.TSP_MEM_DP)
    assert r32["weights"] == 3 * (4 * 64 * 64 + 3 * 64 * 128 + 2 * 64) * 4   # fp32
    # grouped-query attention: W_K, W_V have Hkv*dh = 1024 rows
    g = tsp.rank_memory(tsp.make_cfg(16384, d, 32, I, 8, torch.bfloat16, Hkv=8), L, True,
                        tsp.TSP_MEM_DP)
    assert g["weights"] == L * (2 * d * d + 2 * 1024 * d + 3 * d * I + 2 * d) * 2
    # ... and its saved activations hold the narrower K|V columns
    full = tsp.stack_saved_bytes(_cfg(), L)
    assert tsp.stack_saved_bytes(tsp.make_cfg(16384, d, 32, I, 8, torch.bfloat16, Hkv=8), L) < full


def test_training_activations_are_the_stack_record():
    """The whole-sequence activation term is exactly the buffer tsp_stack_fwd
    fills for the backward (every layer's input plus its saved activations)."""
    cfg, L = _cfg(), 32
    dp = tsp.rank_memory(cfg, L, True, tsp.TSP_MEM_DP)
    assert dp["activations"] == tsp.stack_saved_bytes(cfg, L)


def test_only_the_fold_cuts_both_without_d_squared_devices():
    r = _all(_cfg(D=8), 32, True)
    on_d = [m for m in M if r[m]["devices"] == 8]
    best = min(on_d, key=lambda m: r[m]["total"])
    assert best == tsp.TSP_MEM_TSP
    assert r[tsp.TSP_MEM_TSP]["total"] < r[tsp.TSP_MEM_SP]["total"] < r[tsp.TSP_MEM_TP]["total"]


def test_gathered_kv_transient_does_not_shrink_with_d():
    """The one term the fold does not divide: every rank holds the gathered K
    and V of all S tokens while it runs attention."""
    t2 = tsp.rank_memory(_cfg(D=2), 1, True, tsp.TSP_MEM_TSP)["transient"]
    t8 = tsp.rank_memory(_cfg(D=8), 1, True, tsp.TSP_MEM_TSP)["transient"]
    kv = 2 * 16384 * 4096 * 2
    assert kv < t8 < t2 <= kv + 4 * 4096 * 4096 * 2 / 2
