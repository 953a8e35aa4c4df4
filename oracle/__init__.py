"""Float64 CPU oracle for latent causal attention and the latent projection.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package's smoke check
and by the benchmark's CPU-baseline leg, never by the library's product path.
It shares no code with the CUDA path; both sides only share the seeded input
generator, which holds none of the method's arithmetic.

Two independent forms of the same definition:

* ``attention`` / ``attention_rows`` / ``project`` etc. call the plain C loops
  in ``mla_oracle.c`` (literal form: k and v rebuilt from the latent for every
  (b, h, t, s), float64, max-subtracted softmax).
* ``explicit.py`` materialises K and V once with numpy float64 and applies a
  hand-written causal softmax (no torch); it is the brute-force cross-check.

Sources: page "FW-GLM-5-1 l2_p31" (fused MLA-style attention from compressed
KV latents), "The algorithm" passage; page "FW-GLM-5-1 l2_p1" (fused latent
projection), problem statement; page "Kimi-K2.6 l2_p29" (MSA gated
attention), online-softmax derivation and its -inf worked example.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_CACHE = {}

_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)


def build(mutant: int = 0, out_dir: Optional[str] = None) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP) and return the library path.

    ``mutant`` > 0 compiles a copy with one planted mistake (see the
    ORACLE_MUTANT list in the C source) for the tests that check the pins.
    """
    if mutant:
        out_dir = out_dir or os.path.join(_HERE, "_mutants")
        os.makedirs(out_dir, exist_ok=True)
        path = os.path.join(out_dir, f"libmla_oracle_m{mutant}.so")
    else:
        path = os.path.join(out_dir or _HERE, "libmla_oracle.so")
    if (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", f"-DORACLE_MUTANT={mutant}",
               _SRC, "-o", path + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(path + ".tmp", path)
    return path


class Oracle:
    """ctypes view of one compiled oracle library (the real one or a mutant)."""

    def __init__(self, mutant: int = 0, path: Optional[str] = None):
        self.lib = ctypes.CDLL(path or build(mutant))
        L = self.lib
        L.mla_oracle_project.argtypes = [_D, _D, _D, _D, _D, _D, _D, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.mla_oracle_attention.argtypes = [_D, _D, _D, _D, _D] + [ctypes.c_int] * 6 + [
            ctypes.c_double, ctypes.c_int]
        L.mla_oracle_attention_absorbed.argtypes = L.mla_oracle_attention.argtypes
        L.mla_oracle_attention_rows.argtypes = [_D, _D, _D, _D, _I32, ctypes.c_int, _D] + [
            ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_int]
        L.mla_oracle_attention_absorbed_rows.argtypes = L.mla_oracle_attention_rows.argtypes
        L.mla_oracle_attention_weights.argtypes = [_D, _D, _D] + [ctypes.c_int] * 9 + [
            ctypes.c_double, ctypes.c_int, _D]
        L.mla_oracle_attention_weights.restype = ctypes.c_int
        L.mla_oracle_online_softmax.argtypes = [_D, _D, ctypes.c_int, ctypes.c_int, _D]
        L.mla_oracle_merge_partials.argtypes = [_D, _D, _D, ctypes.c_int, ctypes.c_int, _D]

    # -- helpers ----------------------------------------------------------
    @staticmethod
    def _f64(a) -> np.ndarray:
        if hasattr(a, "detach"):              # torch tensor (bf16 -> f64 is exact)
            import torch
            a = a.detach().to("cpu", torch.float64).numpy()
        return np.ascontiguousarray(a, dtype=np.float64)

    @staticmethod
    def _p(a: Optional[np.ndarray]):
        return None if a is None else a.ctypes.data_as(_D)

    # -- projection -------------------------------------------------------
    def project(self, hidden, w_down, w_up_k=None, w_up_v=None):
        """latent = hidden @ w_down (and k, v = latent @ w_up_k / w_up_v).

        hidden (..., Dm) is flattened to (M, Dm); w_up_* are (R, C) or (R, H, d).
        Returns (latent, k, v) as float64 arrays of shape (M, R), (M, C), (M, C).
        """
        h = self._f64(hidden)
        wd = self._f64(w_down)
        Dm, R = wd.shape
        h = h.reshape(-1, Dm)
        M = h.shape[0]
        wk = None if w_up_k is None else self._f64(w_up_k).reshape(R, -1)
        wv = None if w_up_v is None else self._f64(w_up_v).reshape(R, -1)
        C = (wk if wk is not None else wv).shape[1] if (wk is not None or wv is not None) else 0
        lat = np.empty((M, R))
        k = np.empty((M, C)) if wk is not None else None
        v = np.empty((M, C)) if wv is not None else None
        self.lib.mla_oracle_project(self._p(h), self._p(wd), self._p(wk), self._p(wv),
                                    self._p(lat), self._p(k), self._p(v), M, Dm, R, C)
        return lat, k, v

    # -- attention --------------------------------------------------------
    def _attn_args(self, q, lat, wk, wv):
        q, lat, wk, wv = (self._f64(x) for x in (q, lat, wk, wv))
        B, Tq, H, d = q.shape
        Tkv, R = lat.shape[1], lat.shape[2]
        assert lat.shape[0] == B and wk.shape == (R, H, d) and wv.shape == (R, H, d)
        return q, lat, wk, wv, (B, Tq, Tkv, H, d, R)

    def attention(self, q, kv_latent, w_up_k, w_up_v, scale: float, causal: bool = True):
        """Literal form over every row: out (B, Tq, H, d) float64."""
        q, lat, wk, wv, (B, Tq, Tkv, H, d, R) = self._attn_args(q, kv_latent, w_up_k, w_up_v)
        out = np.empty((B, Tq, H, d))
        self.lib.mla_oracle_attention(self._p(q), self._p(lat), self._p(wk), self._p(wv),
                                      self._p(out), B, Tq, Tkv, H, d, R, float(scale),
                                      int(causal))
        return out

    def attention_absorbed(self, q, kv_latent, w_up_k, w_up_v, scale: float,
                           causal: bool = True):
        """Absorbed form (q' = w_up_k q, softmax over q'.latent, then w_up_v)."""
        q, lat, wk, wv, (B, Tq, Tkv, H, d, R) = self._attn_args(q, kv_latent, w_up_k, w_up_v)
        out = np.empty((B, Tq, H, d))
        self.lib.mla_oracle_attention_absorbed(self._p(q), self._p(lat), self._p(wk),
                                               self._p(wv), self._p(out), B, Tq, Tkv, H, d,
                                               R, float(scale), int(causal))
        return out

    def attention_rows(self, q, kv_latent, w_up_k, w_up_v, scale: float,
                       rows: Sequence[Sequence[int]], causal: bool = True,
                       prepared=None, form: str = "literal"):
        """Selected (b, i) rows only, all heads: returns (n, H, d).

        ``form="literal"`` rebuilds k, v per key (the definition as written);
        ``form="absorbed"`` uses the pinned absorbed identity, far cheaper at
        rank >> head_dim, for sampled checks of large workloads."""
        if prepared is None:
            prepared = self._attn_args(q, kv_latent, w_up_k, w_up_v)
        q, lat, wk, wv, (B, Tq, Tkv, H, d, R) = prepared
        bi = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        assert (bi[:, 0] >= 0).all() and (bi[:, 0] < B).all()
        assert (bi[:, 1] >= 0).all() and (bi[:, 1] < Tq).all()
        n = bi.shape[0]
        out = np.empty((n, H, d))
        fn = {"literal": self.lib.mla_oracle_attention_rows,
              "absorbed": self.lib.mla_oracle_attention_absorbed_rows}[form]
        fn(self._p(q), self._p(lat), self._p(wk), self._p(wv), bi.ctypes.data_as(_I32), n,
           self._p(out), B, Tq, Tkv, H, d, R, float(scale), int(causal))
        return out

    def prepare(self, q, kv_latent, w_up_k, w_up_v):
        """Convert once to float64 for repeated ``attention_rows`` calls."""
        return self._attn_args(q, kv_latent, w_up_k, w_up_v)

    def attention_weights(self, q, kv_latent, w_up_k, scale: float, b: int, h: int, i: int,
                          causal: bool = True):
        """Normalised softmax weights of row (b, h, i) over its keys."""
        q, lat, wk = (self._f64(x) for x in (q, kv_latent, w_up_k))
        B, Tq, H, d = q.shape
        Tkv, R = lat.shape[1], lat.shape[2]
        w = np.empty(Tkv)
        n = self.lib.mla_oracle_attention_weights(self._p(q), self._p(lat), self._p(wk), b, h, i,
                                                  B, Tq, Tkv, H, d, R, float(scale),
                                                  int(causal), self._p(w))
        return w[:n].copy()

    # -- online softmax and the partial merge -------------------------------
    def online_softmax(self, x, v):
        x = self._f64(x)
        v = self._f64(v).reshape(x.shape[0], -1)
        out = np.empty(v.shape[1])
        self.lib.mla_oracle_online_softmax(self._p(x), self._p(v), x.shape[0], v.shape[1],
                                           self._p(out))
        return out

    def merge_partials(self, m_i, l_i, o_i):
        m_i, l_i = self._f64(m_i), self._f64(l_i)
        o_i = self._f64(o_i).reshape(m_i.shape[0], -1)
        out = np.empty(o_i.shape[1])
        self.lib.mla_oracle_merge_partials(self._p(m_i), self._p(l_i), self._p(o_i),
                                           m_i.shape[0], o_i.shape[1], self._p(out))
        return out


def get(mutant: int = 0) -> Oracle:
    """The (cached) oracle; ``mutant`` > 0 only for the pin tests."""
    if mutant not in _LIB_CACHE:
        _LIB_CACHE[mutant] = Oracle(mutant)
    return _LIB_CACHE[mutant]
