"""Comparison rules between the CUDA library and the fp64 oracle.

The tolerances are the ones the method's specification fixes:
  * group scales within 1e-5 relative;
  * integer codes bit-exact, except codes whose oracle pre-round value lies
    within 1e-4 of a rounding boundary (k + 1/2), which may differ by one;
  * dequantised vectors within one quantisation step of the oracle's
    dequantised vectors (per vector, the largest scale_{g(i)} / lambda_i),
    plus half an fp16 ulp of the output;
  * attention outputs within 2e-3 max-abs of the oracle run on the same
    quantised cache.
"""

from __future__ import annotations

import numpy as np

from oracle import srft_oracle as O

SCALE_RTOL = 1e-5
BOUNDARY_BAND = 1e-4
ATTN_ATOL = 2e-3


def compare_codes(gpu_codes: np.ndarray, r: np.ndarray, bits: int) -> dict:
    """Codes from the GPU against the oracle's pre-round values r (same shape as the codes' coordinates)."""
    q_gpu = O.unpack_codes(gpu_codes, bits)
    Q = O.qmax(bits)
    q_ref = np.clip(np.rint(r), -Q, Q).astype(np.int64)
    diff = q_gpu - q_ref
    near = np.abs(np.abs(r - np.floor(r)) - 0.5) < BOUNDARY_BAND
    bad = (diff != 0) & ~(near & (np.abs(diff) == 1))
    return {"n": int(q_ref.size), "mismatch": int((diff != 0).sum()), "bad": int(bad.sum()),
            "near_boundary": int(near.sum()), "first_bad": None if not bad.any() else tuple(np.argwhere(bad)[0])}


def assert_codes(gpu_codes, r, bits):
    st = compare_codes(gpu_codes, r, bits)
    assert st["bad"] == 0, f"code mismatches outside the rounding-boundary band: {st}"
    return st


def assert_scales(gpu_scales: np.ndarray, ref_scales: np.ndarray):
    g = np.asarray(gpu_scales, dtype=np.float64)
    err = np.abs(g - ref_scales)
    tol = SCALE_RTOL * np.abs(ref_scales) + 1e-30
    worst = float((err / tol).max()) if err.size else 0.0
    assert np.all(err <= tol), f"scale relative error above 1e-5 (worst err/tol = {worst:.3g})"


def quant_step(scales: np.ndarray, lam, group: int) -> np.ndarray:
    """Per-vector bound: max_i scale_{g(i)} / lambda_i."""
    step = np.repeat(np.asarray(scales, dtype=np.float64), group, axis=-1)
    if lam is not None:
        step = step / np.asarray(lam, dtype=np.float64)
    return step.max(axis=-1)


def assert_dequant_within_step(x_gpu: np.ndarray, x_oracle_hat: np.ndarray, scales: np.ndarray, lam, group: int):
    """GPU-dequantised vectors against the oracle's dequantisation of its own codes: max-abs difference per
    vector within one quantisation step (a code that differs by one moves x_hat by scale * R^T e_i, whose
    entries are at most scale * sqrt(2/d)), plus half an fp16 ulp of the GPU output."""
    x_gpu = np.asarray(x_gpu, dtype=np.float64)
    x_ref = np.asarray(x_oracle_hat, dtype=np.float64)
    half_ulp = np.abs(x_gpu) * 2.0**-11 + 2.0**-25
    err = (np.abs(x_gpu - x_ref) - half_ulp).max(axis=-1)
    bound = quant_step(scales, lam, group)
    assert np.all(err <= bound), f"dequantised error above one quantisation step: worst {float((err - bound).max()):.3g}"


def assert_reconstruction_bound(x_gpu: np.ndarray, x: np.ndarray, scales: np.ndarray, lam, group: int):
    """||x_hat - x||_2 <= ||(scale_{g(i)} / (2 lambda_i))_i||_2 (the rotation is orthogonal), plus fp16 rounding."""
    x_gpu = np.asarray(x_gpu, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    step = np.repeat(np.asarray(scales, dtype=np.float64), group, axis=-1) / 2
    if lam is not None:
        step = step / np.asarray(lam, dtype=np.float64)
    bound = np.linalg.norm(step, axis=-1) + np.linalg.norm(x_gpu, axis=-1) * 2.0**-11 + 1e-6
    err = np.linalg.norm(x_gpu - x, axis=-1)
    assert np.all(err <= bound), f"reconstruction error above the orthogonality bound: worst {float((err - bound).max()):.3g}"
