"""Seeded synthetic inputs for latent causal attention and the latent projection.

This module is shared by the CUDA path's tests, the benchmark and the float64
oracle's tests.  It holds no arithmetic of the method: it only names the five
workloads (shapes, standard deviations, softmax scale, dtype) and draws their
tensors from a seeded CPU generator.

Workloads (the shapes are the ones the attention and projection pages work
with, scaled up to prefill and decode sizes):

  tiny_f32      fp32 causal attention, q (2,32,4,16), latent (2,32,24)
  proj_f32      fp32 projection (4,96,256)->rank 48->k,v (4,96,128), then
                attention with q (4,96,4,32)
  mid_bf16      bf16 causal attention B4 T1024 H16 d64 rank 256
  prefill_bf16  bf16 projection (2,4096,4096)@(4096,512), then causal attention
                B2 T4096 H32 d128 rank 512
  decode_bf16   bf16 attention of one query at t=4095 over 4096 latent rows,
                B64 H128 d128 rank 512

Recipe: generator = torch.Generator('cpu').manual_seed(1234 + index); tensors
are drawn in the order hidden, w_down, w_up_k, w_up_v, q, kv_latent (absent
ones skipped) as ``randn(shape, float32) * std``.  ``N(0, x)`` in a workload's
description is read as standard deviation x.  bf16 workloads round each tensor
to bf16 with round-to-nearest-even (torch's cast).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dtype: str                      # "f32" or "bf16": the dtype of every input
    B: int
    Tq: int
    Tkv: int
    H: int
    d: int
    rank: int
    scale: float
    causal: bool = True
    model_dim: Optional[int] = None  # set when the workload starts with the projection
    std_q: float = 1.0
    std_latent: float = 1.0
    std_w_up: float = 1.0
    std_hidden: float = 1.0
    std_w_down: float = 1.0

    @property
    def kv_dim(self) -> int:
        return self.H * self.d

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def pairs(self) -> int:
        """Number of (query, key) pairs per head summed over the batch."""
        if self.causal and self.Tq == self.Tkv:
            return self.B * self.Tq * (self.Tq + 1) // 2
        if self.causal:
            off = self.Tkv - self.Tq
            return self.B * sum(off + i + 1 for i in range(self.Tq))
        return self.B * self.Tq * self.Tkv

    def attention_flops(self) -> int:
        """Algorithmic FLOPs of the absorbed attention: q.latent and p.latent
        over rank for every causal pair and head, plus the query absorption
        and the value up-projection once per output row."""
        H, R, d = self.H, self.rank, self.d
        return 4 * R * self.pairs() * H + 4 * self.B * self.Tq * H * R * d

    def projection_flops(self, with_kv: bool = False) -> int:
        if self.model_dim is None:
            return 0
        M = self.B * self.Tkv
        f = 2 * M * self.model_dim * self.rank
        if with_kv:
            f += 2 * 2 * M * self.rank * self.kv_dim
        return f

    def attention_bytes(self, out_bytes: int = 4) -> int:
        """Each attention input read once plus the output written once."""
        es = 4 if self.dtype == "f32" else 2
        n_in = (self.B * self.Tq * self.H * self.d + self.B * self.Tkv * self.rank
                + 2 * self.rank * self.H * self.d)
        return n_in * es + self.B * self.Tq * self.H * self.d * out_bytes


WORKLOADS: Dict[str, Workload] = {
    "tiny_f32": Workload("tiny_f32", 0, "f32", B=2, Tq=32, Tkv=32, H=4, d=16, rank=24,
                         scale=1.0 / math.sqrt(16), std_w_up=1.0 / math.sqrt(24)),
    "proj_f32": Workload("proj_f32", 1, "f32", B=4, Tq=96, Tkv=96, H=4, d=32, rank=48,
                         scale=1.0 / math.sqrt(32), model_dim=256,
                         std_w_up=1.0 / math.sqrt(48), std_w_down=1.0 / 16),
    "mid_bf16": Workload("mid_bf16", 2, "bf16", B=4, Tq=1024, Tkv=1024, H=16, d=64, rank=256,
                         scale=1.0 / 8, std_w_up=1.0 / math.sqrt(256)),
    "prefill_bf16": Workload("prefill_bf16", 3, "bf16", B=2, Tq=4096, Tkv=4096, H=32, d=128,
                             rank=512, scale=1.0 / math.sqrt(128), model_dim=4096,
                             std_w_up=1.0 / math.sqrt(512), std_w_down=1.0 / 64),
    "decode_bf16": Workload("decode_bf16", 4, "bf16", B=64, Tq=1, Tkv=4096, H=128, d=128,
                            rank=512, scale=1.0 / math.sqrt(128),
                            std_w_up=1.0 / math.sqrt(512)),
}


def custom_workload(name: str, *, dtype: str, B: int, Tq: int, Tkv: int, H: int, d: int,
                    rank: int, scale: Optional[float] = None, causal: bool = True,
                    model_dim: Optional[int] = None, index: int = 100) -> Workload:
    """A workload of arbitrary shape with the standard deviations of the
    named ones (weights 1/sqrt(fan_in), activations 1)."""
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return Workload(name, index, dtype, B=B, Tq=Tq, Tkv=Tkv, H=H, d=d, rank=rank, scale=scale,
                    causal=causal, model_dim=model_dim, std_w_up=1.0 / math.sqrt(rank),
                    std_w_down=(1.0 / math.sqrt(model_dim)) if model_dim else 1.0)


def make_inputs(w: Workload, seed: Optional[int] = None, *, with_latent: bool = True,
                with_projection: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Draw the workload's tensors on the CPU (contiguous, in the workload's dtype).

    Keys: hidden (B,Tkv,model_dim), w_down (model_dim,rank) when the workload
    has a projection; w_up_k, w_up_v (rank,H,d); q (B,Tq,H,d);
    kv_latent (B,Tkv,rank).
    """
    g = torch.Generator("cpu").manual_seed(1234 + w.index if seed is None else seed)
    dt = w.torch_dtype
    out: Dict[str, torch.Tensor] = {}
    if with_projection is None:
        with_projection = w.model_dim is not None

    def draw(shape, std):
        t = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(dt).contiguous()

    if with_projection and w.model_dim is not None:
        out["hidden"] = draw((w.B, w.Tkv, w.model_dim), w.std_hidden)
        out["w_down"] = draw((w.model_dim, w.rank), w.std_w_down)
    out["w_up_k"] = draw((w.rank, w.H, w.d), w.std_w_up)
    out["w_up_v"] = draw((w.rank, w.H, w.d), w.std_w_up)
    out["q"] = draw((w.B, w.Tq, w.H, w.d), w.std_q)
    if with_latent:
        out["kv_latent"] = draw((w.B, w.Tkv, w.rank), w.std_latent)
    return out


def make_kv_inputs(w: Workload, seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Queries, keys and values drawn directly (for attention over given k, v):
    q (B,Tq,H,d), k and v (B,Tkv,H,d), N(0, 1) each (the spread of latent @
    w_up with the workloads' weight scaling), in the workload's dtype.  Same
    generator recipe as make_inputs; drawn in the order q, k, v."""
    g = torch.Generator("cpu").manual_seed(4321 + w.index if seed is None else seed)
    dt = w.torch_dtype

    def draw(shape):
        return torch.randn(shape, generator=g, dtype=torch.float32).to(dt).contiguous()

    return {"q": draw((w.B, w.Tq, w.H, w.d)), "k": draw((w.B, w.Tkv, w.H, w.d)),
            "v": draw((w.B, w.Tkv, w.H, w.d))}
