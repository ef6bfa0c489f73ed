"""Shared helpers of the parity tests: the tolerance, device upload, sampling."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Per-element bound: |C_gpu - C_ref| <= RTOL * |C_ref| + ATOL_RMS * rms(C_ref).
# The kernels accumulate each 128-wide group exactly in fp32 as far as the
# products allow and promote with one fp32 FMA per group; the output cast adds
# at most half an ulp of the output type (2^-9 relative for bf16).  1e-2 of the
# element plus 1e-2 of the matrix rms covers both with a wide margin while
# still catching a wrong scale, a dropped group or a swapped index.
RTOL = 1e-2
ATOL_RMS = 1e-2

OUT_TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def to_device(x, device="cuda"):
    """Upload synth inputs: returns (A, a_s, B, b_s) CUDA tensors."""
    return (x.A.to(device), x.a_s.to(device), x.B.to(device), x.b_s.to(device))


def assert_close(got, ref, rows=None, cols=None, rms=None, what=""):
    """got: torch tensor (any float dtype, any device) of the GPU result;
    ref: float64 numpy array of the oracle result at the same positions."""
    g = got.detach().to("cpu", torch.float64).numpy()
    if rows is not None:
        g = g[rows, cols]
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    if rms is None:
        rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    assert not np.isnan(g[~np.isnan(ref)]).any(), f"{what}: NaN in the GPU result"
    err = np.abs(g - ref)
    bound = RTOL * np.abs(ref) + ATOL_RMS * rms
    bad = err > bound
    if bad.any():
        i = np.argmax(err - bound)
        idx = np.unravel_index(i, err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements outside the bound; "
                             f"worst at {idx}: got {g[idx]!r} want {ref[idx]!r} "
                             f"(bound {bound[idx]:.3g}, rms {rms:.3g})")


def sample_rows(M: int, count: int = 192) -> np.ndarray:
    """Rows spread over every 128-row tile plus the ragged tail, at most ~count."""
    if M <= count:
        return np.arange(M)
    step = max(1, M // count)
    rows = set(range(0, M, step))
    rows.update(range(max(0, M - 8), M))
    rows.update(t * 128 + 127 for t in range(M // 128) if t * 128 + 127 < M)
    return np.array(sorted(rows))


def reference_rows(x, rows):
    """Oracle result of the given rows of A against all of B (float64)."""
    return oracle.reference_c(x.A[rows], x.a_s[rows], x.B, x.b_s)


def rms_estimate(ref_rows: np.ndarray) -> float:
    return float(np.sqrt(np.mean(ref_rows ** 2)))
