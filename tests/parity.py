"""Tolerances and comparison helpers for the CUDA-vs-oracle parity tests.

Tolerances (floating point; the integer accounting is compared bit-exactly):
  O    : max |O - O_ref| <= 1e-2 on float32-output O, and bf16 O must equal
         round-to-nearest-even(float32 O) bit for bit;
  LSE  : |LSE - LSE_ref| <= 1e-3 * max(1, |LSE_ref|); rows with an empty
         visible set must give exactly -inf (and O = 0);
  dQ/dK/dV : ||X - X_ref||_F / ||X_ref||_F <= 2e-2 over the checked rows.
"""
import os

import numpy as np
import torch

O_ATOL = 1e-2
LSE_RTOL = 1e-3
GRAD_RFRO = 2e-2

# Largest error seen per test and quantity (O, LSE, dQ, dK, dV), written to
# the file named by CA_PARITY_REPORT at the end of the session (conftest.py).
REPORT = {}


def _record(what: str, err: float):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    kind = what.split(":")[-1].strip().split(" ")[0]
    d = REPORT.setdefault(test, {})
    d[kind] = max(d.get(kind, 0.0), float(err))


def to64(x: torch.Tensor) -> np.ndarray:
    return x.detach().to(torch.float64).cpu().numpy()


def check_o(o_gpu: np.ndarray, o_ref: np.ndarray, what="O"):
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite values"
    err = np.abs(o_gpu - o_ref).max() if o_ref.size else 0.0
    _record(what, err)
    assert err <= O_ATOL, f"{what}: max abs error {err:.3e} > {O_ATOL}"
    return float(err)


def check_lse(lse_gpu: np.ndarray, lse_ref: np.ndarray, what="LSE"):
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), f"{what}: -inf pattern differs"
    assert np.all(lse_gpu[~fin] == -np.inf), f"{what}: empty rows must be -inf"
    if not fin.any():
        return 0.0
    rel = np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
    err = float(rel.max())
    _record(what, err)
    assert err <= LSE_RTOL, f"{what}: relative error {err:.3e} > {LSE_RTOL}"
    return err


def rel_fro(x: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


def check_grad(x: np.ndarray, ref: np.ndarray, what: str):
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    err = rel_fro(x, ref)
    _record(what, err)
    assert err <= GRAD_RFRO, f"{what}: relative Frobenius error {err:.3e} > {GRAD_RFRO}"
    return err


def bf16_rne(x: torch.Tensor) -> torch.Tensor:
    """float32 -> bf16 with round-to-nearest-even (torch's conversion)."""
    return x.to(torch.bfloat16)
