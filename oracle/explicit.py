"""Brute-force float64 cross-check of latent causal attention (numpy, no torch).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Same definition as the C oracle, reached a different way: K and V are
materialised once for every position and head (K[b,s,h,:] =
kv_latent[b,s] @ w_up_k[:,h], likewise V), then each head runs ordinary
causal softmax attention with a hand-written, max-subtracted softmax.
Page "FW-GLM-5-1 l2_p31" (fused MLA-style attention from compressed KV
latents), "The algorithm" passage; the inclusive mask s <= t is the page's;
queries are the last Tq positions when Tq < Tkv.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def materialise_kv(kv_latent, w_up_k, w_up_v):
    """K, V of shape (B, Tkv, H, d): every position's latent times each head's weights."""
    lat, wk, wv = _f64(kv_latent), _f64(w_up_k), _f64(w_up_v)
    R, H, d = wk.shape
    K = (lat.reshape(-1, R) @ wk.reshape(R, H * d)).reshape(lat.shape[0], lat.shape[1], H, d)
    V = (lat.reshape(-1, R) @ wv.reshape(R, H * d)).reshape(lat.shape[0], lat.shape[1], H, d)
    return K, V


def softmax_rows(x: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax along the last axis; -inf entries get weight 0."""
    m = x.max(axis=-1, keepdims=True)
    w = np.exp(x - m)
    return w / w.sum(axis=-1, keepdims=True)


def attention_kv(q, k, v, scale: float, causal: bool = True, query_rows=None) -> np.ndarray:
    """Ordinary softmax attention over given keys and values: q (B,Tq,H,d),
    k, v (B,Tkv,H,d) -> out (B,Tq,H,d) float64 (or (B,len(query_rows),H,d)).
    The same definition with k_s and v_s supplied instead of rebuilt from the
    latent; queries are the last Tq positions, mask s <= t when causal."""
    qf, K, V = _f64(q), _f64(k), _f64(v)
    B, Tq, H, d = qf.shape
    Tkv = K.shape[1]
    idx = np.arange(Tq) if query_rows is None else np.asarray(query_rows)
    t = (Tkv - Tq) + idx
    out = np.empty((B, len(idx), H, d))
    s = np.arange(Tkv)
    for b in range(B):
        for h in range(H):
            x = (qf[b, idx, h, :] @ K[b, :, h, :].T) * scale
            if causal:
                x = np.where(s[None, :] <= t[:, None], x, -np.inf)
            out[b, :, h, :] = softmax_rows(x) @ V[b, :, h, :]
    return out


def attention(q, kv_latent, w_up_k, w_up_v, scale: float, causal: bool = True,
              query_rows=None) -> np.ndarray:
    """out (B, Tq, H, d) float64; ``query_rows`` restricts to a subset of i
    (then out has shape (B, len(query_rows), H, d))."""
    qf = _f64(q)
    B, Tq, H, d = qf.shape
    K, V = materialise_kv(kv_latent, w_up_k, w_up_v)
    Tkv = K.shape[1]
    idx = np.arange(Tq) if query_rows is None else np.asarray(query_rows)
    t = (Tkv - Tq) + idx                                   # absolute query positions
    out = np.empty((B, len(idx), H, d))
    s = np.arange(Tkv)
    for b in range(B):
        for h in range(H):
            x = (qf[b, idx, h, :] @ K[b, :, h, :].T) * scale  # (n, Tkv)
            if causal:
                x = np.where(s[None, :] <= t[:, None], x, -np.inf)
            out[b, :, h, :] = softmax_rows(x) @ V[b, :, h, :]
    return out
