"""Helpers shared by the GPU parity tests (tolerances and transfers)."""
import numpy as np

import oracle


def dev_tensor(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def gemv_tol(fmt, W, r0, r1, in_dim, x):
    """Per-row bound max|y_gpu - y_ref| <= 1e-3 * ||W_r||_2 * ||x||_2."""
    return 1e-3 * oracle.row_norms(fmt, W, r0, r1, in_dim) * float(
        np.linalg.norm(np.asarray(x, dtype=np.float64)))


def assert_gemv_close(y_gpu, y_ref, tol, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, (f"{what}: {bad.size} rows out of tolerance, first row {bad[0]}: "
                           f"gpu {y_gpu[bad[0]]} ref {y_ref[bad[0]]} tol {tol[bad[0]]}")
    return float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0


def swiglu_h_tol(g_ref, u_ref, tg, tu):
    """Bound on |h_gpu - h_ref| for h = silu(g)*u given |dg| <= tg, |du| <= tu:
    |silu'| <= 1.1, plus fp32 rounding of the epilogue."""
    silu = g_ref / (1.0 + np.exp(-g_ref))
    return 1.1 * tg * (np.abs(u_ref) + tu) + np.abs(silu) * tu + 1e-6 * np.abs(silu * u_ref)
