"""Shared test utilities: tolerance checks and CPU<->GPU plumbing.

Tolerances (from the block's stated accuracy targets):
  * permutation / indexing: bit-exact;
  * bf16 path: max|err| <= 2e-2 * RMS(ref) and sum|err| / sum|ref| <= 5e-3,
    per output tensor, RMS(ref) = sqrt(mean(ref^2)) over the checked elements;
  * exact-fp32 path: max|err| <= 1e-4.
"""
import numpy as np
import torch

BF16_MAX_REL_RMS = 2e-2
BF16_MEAN_REL = 5e-3
F32_MAX_ABS = 1e-4


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def bf16_metrics(got, ref):
    got, ref = to64(got), to64(ref)
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(err.max()) / rms, float(err.sum() / np.abs(ref).sum())


def assert_bf16_close(got, ref, what=""):
    mx, mean = bf16_metrics(got, ref)
    assert np.all(np.isfinite(to64(got))), f"{what}: non-finite output"
    assert mx <= BF16_MAX_REL_RMS and mean <= BF16_MEAN_REL, \
        f"{what}: max|err|/RMS={mx:.3e} (<= {BF16_MAX_REL_RMS}), mean rel={mean:.3e} (<= {BF16_MEAN_REL})"
    return mx, mean


def assert_f32_close(got, ref, what="", tol=F32_MAX_ABS):
    err = float(np.max(np.abs(to64(got) - to64(ref))))
    assert err <= tol, f"{what}: max|err|={err:.3e} > {tol}"
    return err
