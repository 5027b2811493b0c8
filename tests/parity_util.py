"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances: o (and merged o) max-abs <= 2e-2; lse |d| <= 1e-3 * max(1, |lse|)
(-inf must match -inf exactly); dq, dk, dv relative Frobenius error <= 1e-2.
"""
import numpy as np
import torch

O_ATOL = 2e-2
LSE_RTOL = 1e-3
GRAD_RTOL = 1e-2


def host(t: torch.Tensor, dtype=np.float64) -> np.ndarray:
    return t.detach().to(torch.float32).cpu().numpy().astype(dtype, copy=False)


def check_o(got, ref, what="o"):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= O_ATOL, f"{what}: max abs err {err:.3e} > {O_ATOL}"
    return err


def check_lse(got, ref, what="lse"):
    got = np.asarray(got, dtype=np.float64)
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), f"{what}: -inf pattern differs ({ninf_g.sum()} vs {ninf_r.sum()})"
    fin = ~ninf_r
    if not fin.any():
        return 0.0
    err = np.abs(got[fin] - ref[fin]) / np.maximum(1.0, np.abs(ref[fin]))
    assert np.isfinite(got[fin]).all(), f"{what}: non-finite values"
    assert err.max() <= LSE_RTOL, f"{what}: max rel err {err.max():.3e} > {LSE_RTOL}"
    return float(err.max())


def check_grad(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / (den if den > 0 else 1.0)
    assert rel <= GRAD_RTOL, f"{what}: rel Frobenius err {rel:.3e} > {GRAD_RTOL}"
    return float(rel)
