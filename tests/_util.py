"""Shared helpers of the parity tests (comparison and tolerances only)."""
import numpy as np
import torch

# bf16: max|err| <= 1e-2 * max|ref| + 1e-3 per tensor; fp32: <= 1e-5.
BF16_REL, BF16_ABS = 1e-2, 1e-3
F32_ABS = 1e-5


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def bound(ref, dtype):
    ref = np.asarray(ref)
    if dtype == torch.float32:
        return F32_ABS
    mx = float(np.max(np.abs(ref))) if ref.size else 0.0
    return BF16_REL * mx + BF16_ABS


def assert_close(name, got, ref, dtype, mask=None):
    got = to_np(got)
    ref = np.asarray(ref, dtype=np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = float(np.max(np.abs(got - ref)))
    tol = bound(ref, dtype)
    assert err <= tol, f"{name}: max|err| {err:.3e} > tol {tol:.3e} (max|ref| {np.max(np.abs(ref)):.3e})"
    return err


def valid_rows(seg, B, H, S):
    """bool [B,H,S] of non-padding query rows."""
    if seg is None:
        return np.ones((B, H, S), dtype=bool)
    v = to_np(seg) >= 0
    return np.broadcast_to(v[:, None, :], (B, H, S))
