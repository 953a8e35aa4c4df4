"""Shared helpers for the GPU parity tests: tolerances and device plumbing.

Tolerances (written out here, derived in the design notes):
  fp32 workloads: |gpu - ref| <= 1e-4 + 1e-4 * |ref| per element.
  bf16 workloads: the relative bound applies to each output row (the last
                  axis: one head's d-vector, or one latent / k / v row):
                  |gpu - ref| <= 2e-2 * |ref| + 2e-2 * rms(ref row) per element,
                  ||gpu - ref row||_2 <= 2e-2 * ||ref row||_2 per row, and
                  ||gpu - ref||_2 <= 2e-2 * ||ref||_2 over the compared set.
                  (Rows at small t average few values and are several times
                  larger than the global rms, so the scale is the row's own.)
"""
import numpy as np
import torch


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def assert_f32_close(gpu, ref, what=""):
    g, r = to_np(gpu), to_np(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bound = 1e-4 + 1e-4 * np.abs(r)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements off; "
                           f"max abs err {err.max():.3e}")


def bf16_errors(gpu, ref):
    g, r = to_np(gpu), to_np(ref)
    err = np.abs(g - r)
    row_rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    row_norm = np.linalg.norm(r, axis=-1)
    row_err = np.linalg.norm(g - r, axis=-1)
    return dict(max_abs=float(err.max()),
                normwise=float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)),
                worst_row=float((row_err / np.maximum(row_norm, 1e-300)).max()),
                worst_ratio=float((err / (2e-2 * np.abs(r) + 2e-2 * row_rms + 1e-30)).max()))


def assert_bf16_close(gpu, ref, what=""):
    g, r = to_np(gpu), to_np(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    e = bf16_errors(g, r)
    assert e["worst_ratio"] <= 1.0, f"{what}: elementwise bound exceeded {e}"
    assert e["worst_row"] <= 2e-2, f"{what}: row-relative error {e}"
    assert e["normwise"] <= 2e-2, f"{what}: normwise error {e}"
    return e


def cuda(t):
    return t.to("cuda").contiguous()


def sample_rows(B, Tq, n, seed=0, must=((0, 0),)):
    """(b, i) pairs: the given ones, the last row of each end batch, then random."""
    rng = np.random.default_rng(seed)
    rows = list(must) + [(B - 1, Tq - 1)]
    while len(rows) < n:
        rows.append((int(rng.integers(B)), int(rng.integers(Tq))))
    out, seen = [], set()
    for r in rows:
        if r not in seen:
            seen.add(r)
            out.append(r)
    return out
