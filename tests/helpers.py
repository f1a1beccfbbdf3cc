"""Shared helpers for the GPU parity tests (comparison rules and tolerances).

Tolerances: fp32 storage -> max-abs error <= 1e-5; bf16 / fp16 / FP8 storage
-> max-abs error <= 2e-2 * max|y_oracle|.  Index status and present K/V are
compared bit for bit.
"""
import numpy as np
import torch

TOL_F32 = 1e-5
TOL_REL_LOW = 2e-2


def tol_for(dtype, ref):
    if dtype == torch.float32:
        return TOL_F32
    return TOL_REL_LOW * float(np.abs(ref).max())


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    tol = tol_for(dtype, ref)
    assert err <= tol, f"{what}: max|got - oracle| = {err:.3e} > tol {tol:.3e}"
    return err


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()
