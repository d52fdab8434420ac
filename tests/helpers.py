"""Shared test helpers: tolerances, comparisons and GPU availability."""
import numpy as np
import torch

# Output tolerances for bf16-input / fp32-accumulate attention (stated targets).
MAX_ABS = 2e-2
MIN_COS = 0.9999
MAX_REL_L2 = 2e-3
# lse: fp32 accumulation of exact bf16 products plus exp2 approximation and log;
# the error budget is a few ulp of |lse| ~ 10, far below this bound.
LSE_ABS = 1e-3


def have_gpu() -> bool:
    return torch.cuda.is_available()


def compare(got, ref):
    """max-abs, cosine and relative L2 of got (any float) against ref (float64)."""
    g = np.asarray(got, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    diff = g - r
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    nr = float(np.linalg.norm(r))
    ng = float(np.linalg.norm(g))
    cos = float(np.dot(g, r) / (ng * nr)) if ng > 0 and nr > 0 else (1.0 if ng == nr else 0.0)
    rel = float(np.linalg.norm(diff) / nr) if nr > 0 else float(np.linalg.norm(diff))
    return max_abs, cos, rel


def assert_close_attn(got, ref, what=""):
    max_abs, cos, rel = compare(got, ref)
    assert max_abs <= MAX_ABS and cos >= MIN_COS and rel <= MAX_REL_L2, (
        f"{what}: max_abs={max_abs:.3e} cos={cos:.7f} rel_l2={rel:.3e}")
    return max_abs, cos, rel


def assert_lse_close(got, ref, what=""):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(g) & np.isneginf(r)
    assert np.array_equal(np.isneginf(g), np.isneginf(r)), f"{what}: -inf pattern differs"
    with np.errstate(invalid="ignore"):
        d = np.abs(np.where(both_inf, 0.0, g - r))
    assert np.all(np.isfinite(d)) and d.max(initial=0.0) <= LSE_ABS, f"{what}: lse err {d.max()}"
