"""Comparison rules of the parity tests (CUDA library vs CPU oracle).

* Indexing is bit-exact: a canary NaN pattern fills every output buffer on
  both sides first, and the set of elements each side overwrote must match.
* bf16 outputs: |gpu - ref| <= 2e-3 * max|ref| per tensor, where ref is the
  oracle's bf16 rounding of its exact value.  The one exception is a rounding
  tie the fp32 arithmetic cannot decide: when the exact value lies within
  2e-5 * max|ref| of a bf16 rounding boundary, either neighbour of the exact
  value is accepted (a one-ulp difference).
* fp32 corrections and committed states: |gpu - exact| <= 1e-4 * max|exact|
  per tensor (exact = the oracle's double value).
* Conv outputs (the key half of the key/gate records), the raw-gate half and
  the rolled conv state are compared bit for bit.
"""
from __future__ import annotations

import numpy as np

BF16_CANARY = 0x7FA5
F32_CANARY = 0x7FC0DEAD


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_order(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns as integers in numeric order (adjacent values differ by 1)."""
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def assert_bf16_outputs(gpu_bits, ref_bits, ref_exact, mask, tol=2e-3, tie=2e-5, what="out"):
    """gpu_bits / ref_bits: uint16 arrays; ref_exact: double; mask: elements written."""
    g = bf16_to_f64(gpu_bits[mask])
    r = bf16_to_f64(ref_bits[mask])
    e = ref_exact[mask]
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    scale = np.abs(e).max() if e.size else 0.0
    err = np.abs(g - r)
    bad = err > tol * scale
    n_ties = 0
    if bad.any():
        gb, rb = gpu_bits[mask][bad], ref_bits[mask][bad]
        one_ulp = np.abs(_bf16_order(gb) - _bf16_order(rb)) == 1
        near_tie = np.abs(e[bad] - (g[bad] + r[bad]) / 2) <= tie * scale
        ok = near_tie & one_ulp
        n_ties = int(ok.sum())
        if not ok.all():
            i = np.flatnonzero(bad)[~ok][:5]
            raise AssertionError(
                f"{what}: {int((~ok).sum())} elements exceed {tol}*max|ref| = {tol * scale:.3g}; "
                f"gpu {g[i]}, ref {r[i]}, exact {e[i]}")
    return dict(max_err=float(err.max()) if err.size else 0.0, scale=float(scale), tie_flips=n_ties)


def assert_f32_close(gpu, exact, mask, tol=1e-4, what="corr"):
    g = gpu[mask].astype(np.float64)
    e = exact[mask]
    assert np.isfinite(g).all(), f"{what}: non-finite GPU values"
    scale = np.abs(e).max() if e.size else 0.0
    err = np.abs(g - e).max() if e.size else 0.0
    assert err <= tol * scale, f"{what}: max|err| {err:.3g} > {tol}*max|ref| {tol * scale:.3g}"
    return dict(max_err=float(err), scale=float(scale), rel=float(err / scale) if scale else 0.0)


def written_bf16(bits):
    return bits != BF16_CANARY


def written_f32(arr):
    return arr.view(np.uint32) != F32_CANARY


def assert_same_written(gpu_written, ref_written, what):
    if not np.array_equal(gpu_written, ref_written):
        extra = np.argwhere(gpu_written & ~ref_written)[:5]
        missing = np.argwhere(~gpu_written & ref_written)[:5]
        raise AssertionError(f"{what}: written sets differ; GPU-only {extra.tolist()}, "
                             f"oracle-only {missing.tolist()}")


def conv_adversarial_rows():
    """The rows of tests/golden/conv_adversarial.txt: (kinds [n], fp32 conv
    weights [n, 4] as doubles), for a conv fed with inputs of 1.0."""
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "conv_adversarial.txt")
    kinds, rows = [], []
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            kinds.append(parts[0])
            rows.append([float.fromhex(v) for v in parts[1:5]])
    return np.array(kinds), np.array(rows, np.float64)
