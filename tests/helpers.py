"""Shared helpers for the GPU parity tests.

Tolerances (bf16 inputs and outputs, fp32 accumulation, against the fp64 oracle):
  out, dq, dk, dv: max-abs <= 2e-2 and relative L2 <= 5e-3
  lse:             max-abs <= 1e-3
  permutations:    bit-exact
"""
import numpy as np
import torch

TOL_MAX_ABS = 2e-2
TOL_REL_L2 = 5e-3
TOL_LSE = 1e-3


def f64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def assert_close(name, got, ref, max_abs=TOL_MAX_ABS, rel_l2=TOL_REL_L2):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = np.abs(got - ref)
    mx = float(err.max()) if err.size else 0.0
    assert mx <= max_abs, f"{name}: max-abs {mx:.3e} > {max_abs} at {np.unravel_index(err.argmax(), err.shape)}"
    if rel_l2 is not None and err.size:
        rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
        assert rel <= rel_l2, f"{name}: rel-L2 {rel:.3e} > {rel_l2}"


def assert_lse_close(name, got, ref, tol=TOL_LSE):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape
    both_inf = np.isneginf(got) & np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{name}: -inf pattern differs"
    err = np.zeros_like(got)
    err[~both_inf] = np.abs(got[~both_inf] - ref[~both_inf])
    mx = float(err.max()) if err.size else 0.0
    assert mx <= tol, f"{name}: max-abs {mx:.3e} > {tol}"


def to_layout(ra, x, layout, n):
    """Original order -> layout order through the library's own permute kernel."""
    return ra.ring_attn_permute(x, layout, n, seq_dim=2)


def to_original(ra, y, layout, n):
    return ra.ring_attn_unpermute(y, layout, n, seq_dim=2)


def lse_to_original(ra, lse, layout, n):
    return ra.ring_attn_unpermute(lse.contiguous(), layout, n, seq_dim=2)


def check_no_device_error(ra):
    st, info = ra.ring_attn_check_device_error()
    assert st == 0, f"device-side error status {st} info {info:#x}"
