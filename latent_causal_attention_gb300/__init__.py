"""Latent causal attention for GB300 (sm_103a): Python binding of the C ABI.

Every call below only marshals torch tensors (device memory, the current CUDA
stream) into the C functions declared in include/mla.h; all arithmetic runs
in the library's CUDA kernels.  There is no CPU fallback: without the built
library or without a GPU the calls raise.

    project(hidden, w_down, w_up_k=None, w_up_v=None)  -> latent, k, v
    attention(q, kv_latent, w_up_k, w_up_v, scale, causal=True) -> out
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import MLAError, MLA_BF16, MLA_F32

__all__ = ["project", "attention", "attention_varlen", "explicit_attention", "attention_from_host",
           "workspace_size", "kv_splits",
           "merge_partials",
           "set_option", "device_error", "launch_count", "StageEvents", "MLAError",
           "dtype_code"]


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return MLA_F32
    if dt == torch.bfloat16:
        return MLA_BF16
    raise TypeError(f"unsupported dtype {dt}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _require(name: str, t: Optional[torch.Tensor], shape=None, numel=None, dtype=None,
             device=None) -> None:
    """Shape, element count, dtype and device of one argument, checked before
    any pointer crosses the C ABI (the library trusts the sizes it is given)."""
    if t is None:
        return
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def project(hidden: torch.Tensor, w_down: torch.Tensor, w_up_k: Optional[torch.Tensor] = None,
            w_up_v: Optional[torch.Tensor] = None, *, out_dtype: Optional[torch.dtype] = None,
            latent: Optional[torch.Tensor] = None
            ) -> Tuple[torch.Tensor, Optional[torch.Tensor], Optional[torch.Tensor]]:
    """latent = hidden @ w_down; k = latent @ w_up_k; v = latent @ w_up_v.

    hidden (..., model_dim); w_down (model_dim, rank); w_up_k / w_up_v
    (rank, kv_dim) or (rank, H, d).  Returns latent (..., rank) and k, v
    (..., kv_dim) (None where the weight is None)."""
    lib = _lib.load()
    out_dtype = out_dtype or hidden.dtype
    Dm, R = w_down.shape
    lead = hidden.shape[:-1]
    if hidden.shape[-1] != Dm:
        raise ValueError(f"hidden: last dimension {hidden.shape[-1]}, w_down has {Dm} rows")
    M = hidden.numel() // Dm
    kvd = 0
    for w in (w_up_k, w_up_v):
        if w is not None:
            kvd = w.numel() // R
    dev = hidden.device
    _require("w_down", w_down, dtype=hidden.dtype, device=dev)
    for name, w in (("w_up_k", w_up_k), ("w_up_v", w_up_v)):
        _require(name, w, numel=R * kvd, dtype=hidden.dtype, device=dev)
        if w is not None and (w.shape[0] != R or w.numel() % R != 0):
            raise ValueError(f"{name}: leading dimension {w.shape[0]}, expected rank {R}")
    _require("latent", latent, numel=M * R, dtype=out_dtype, device=dev)
    if latent is None:
        latent = torch.empty(*lead, R, device=dev, dtype=out_dtype)
    k = torch.empty(*lead, kvd, device=dev, dtype=out_dtype) if w_up_k is not None else None
    v = torch.empty(*lead, kvd, device=dev, dtype=out_dtype) if w_up_v is not None else None
    st = lib.mla_kv_latent_project(_ptr(hidden), _ptr(w_down), _ptr(w_up_k), _ptr(w_up_v),
                                   _ptr(latent), _ptr(k), _ptr(v), M, Dm, R, kvd,
                                   dtype_code(hidden.dtype), dtype_code(out_dtype), _stream(dev))
    _lib.check("mla_kv_latent_project", st)
    return latent, k, v


def workspace_size(B: int, Tq: int, Tkv: int, H: int, d: int, rank: int,
                   dtype: torch.dtype, causal: bool = True) -> int:
    lib = _lib.load()
    return int(lib.mla_latent_attention_workspace_size(B, Tq, Tkv, H, d, rank, dtype_code(dtype),
                                                       int(causal)))


def kv_splits(B: int, Tq: int, Tkv: int, H: int, d: int, rank: int,
              dtype: torch.dtype, causal: bool = True) -> int:
    """Key-range partitions the attention call plans for these sizes (0: the
    warp-per-query path)."""
    lib = _lib.load()
    return int(lib.mla_latent_attention_kv_splits(B, Tq, Tkv, H, d, rank, dtype_code(dtype),
                                                  int(causal)))


def attention(q: torch.Tensor, kv_latent: torch.Tensor, w_up_k: torch.Tensor,
              w_up_v: torch.Tensor, scale: float, causal: bool = True, *,
              out_dtype: torch.dtype = torch.float32, out: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Causal latent attention.  q (B,Tq,H,d), kv_latent (B,Tkv,rank),
    w_up_k / w_up_v (rank,H,d); returns out (B,Tq,H,d) in ``out_dtype``.
    ``workspace`` (uint8, at least workspace_size(...) bytes) is allocated
    here when not given."""
    lib = _lib.load()
    B, Tq, H, d = q.shape
    Tkv, R = kv_latent.shape[1], kv_latent.shape[2]
    dev = q.device
    _require("kv_latent", kv_latent, shape=(B, Tkv, R), dtype=q.dtype, device=dev)
    _require("w_up_k", w_up_k, numel=R * H * d, dtype=q.dtype, device=dev)
    _require("w_up_v", w_up_v, numel=R * H * d, dtype=q.dtype, device=dev)
    _require("out", out, shape=(B, Tq, H, d), device=dev)
    _require("workspace", workspace, dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(B, Tq, H, d, device=dev, dtype=out_dtype)
    ws_bytes = workspace_size(B, Tq, Tkv, H, d, R, q.dtype, causal)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    st = lib.mla_latent_attention(_ptr(q), _ptr(kv_latent), _ptr(w_up_k), _ptr(w_up_v), _ptr(out),
                                  B, Tq, Tkv, H, d, R, float(scale), int(causal),
                                  dtype_code(q.dtype), dtype_code(out.dtype), _ptr(workspace),
                                  0 if workspace is None else workspace.numel(), _stream(dev))
    _lib.check("mla_latent_attention", st)
    return out


def attention_varlen(q: torch.Tensor, kv_latent: torch.Tensor, w_up_k: torch.Tensor,
                     w_up_v: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_kv: torch.Tensor,
                     max_seqlen_q: int, scale: float, causal: bool = True, *,
                     out_dtype: torch.dtype = torch.float32,
                     out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Variable-length batch: q (total_q,H,d), kv_latent (total_kv,rank) packed
    back to back, cu_seqlens_q / cu_seqlens_kv (B+1,) int32 on the device;
    returns out (total_q,H,d)."""
    lib = _lib.load()
    total_q, H, d = q.shape
    total_kv, R = kv_latent.shape
    B = cu_seqlens_q.numel() - 1
    dev = q.device
    _require("kv_latent", kv_latent, dtype=q.dtype, device=dev)
    _require("w_up_k", w_up_k, numel=R * H * d, dtype=q.dtype, device=dev)
    _require("w_up_v", w_up_v, numel=R * H * d, dtype=q.dtype, device=dev)
    _require("cu_seqlens_q", cu_seqlens_q, shape=(B + 1,), dtype=torch.int32, device=dev)
    _require("cu_seqlens_kv", cu_seqlens_kv, shape=(B + 1,), dtype=torch.int32, device=dev)
    _require("out", out, shape=(total_q, H, d), device=dev)
    if out is None:
        out = torch.empty(total_q, H, d, device=q.device, dtype=out_dtype)
    st = lib.mla_latent_attention_varlen(_ptr(q), _ptr(kv_latent), _ptr(w_up_k), _ptr(w_up_v),
                                         _ptr(out), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B,
                                         int(max_seqlen_q), total_q, total_kv, H, d, R,
                                         float(scale), int(causal), dtype_code(q.dtype),
                                         dtype_code(out.dtype), _stream(q.device))
    _lib.check("mla_latent_attention_varlen", st)
    return out


def explicit_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                       causal: bool = True, *, out_dtype: torch.dtype = torch.float32,
                       out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Attention over materialised keys and values (the comparator of the
    absorbed path): q (B,Tq,H,d), k / v (B,Tkv,H,d), all bf16, d 64 or 128;
    returns out (B,Tq,H,d) in ``out_dtype``.  k and v come from ``project``
    with w_up_k / w_up_v."""
    lib = _lib.load()
    B, Tq, H, d = q.shape
    Tkv = k.shape[1]
    _require("k", k, shape=(B, Tkv, H, d), dtype=q.dtype, device=q.device)
    _require("v", v, shape=(B, Tkv, H, d), dtype=q.dtype, device=q.device)
    _require("out", out, shape=(B, Tq, H, d), device=q.device)
    if out is None:
        out = torch.empty(B, Tq, H, d, device=q.device, dtype=out_dtype)
    st = lib.mla_explicit_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Tq, Tkv, H, d,
                                    float(scale), int(causal), dtype_code(q.dtype),
                                    dtype_code(out.dtype), _stream(q.device))
    _lib.check("mla_explicit_attention", st)
    return out


def attention_from_host(q: torch.Tensor, kv_latent: torch.Tensor, w_up_k: torch.Tensor,
                        w_up_v: torch.Tensor, scale: float, causal: bool = True, *,
                        device: torch.device, out_dtype: torch.dtype = torch.float32,
                        dev_buffers: Optional[dict] = None) -> torch.Tensor:
    """The same call for inputs in (pinned) host memory: copies the inputs to
    the device, runs the attention and copies the result back; returns a host
    tensor.  ``dev_buffers`` may hold preallocated device tensors keyed by
    name to avoid allocation per call."""
    bufs = dev_buffers if dev_buffers is not None else {}
    dq = bufs.get("q") if "q" in bufs else torch.empty_like(q, device=device)
    dl = bufs.get("kv_latent") if "kv_latent" in bufs else torch.empty_like(kv_latent, device=device)
    dk = bufs.get("w_up_k") if "w_up_k" in bufs else torch.empty_like(w_up_k, device=device)
    dv = bufs.get("w_up_v") if "w_up_v" in bufs else torch.empty_like(w_up_v, device=device)
    dq.copy_(q, non_blocking=True)
    dl.copy_(kv_latent, non_blocking=True)
    dk.copy_(w_up_k, non_blocking=True)
    dv.copy_(w_up_v, non_blocking=True)
    out = attention(dq, dl, dk, dv, scale, causal, out_dtype=out_dtype, out=bufs.get("out"),
                    workspace=bufs.get("workspace"))
    host = bufs.get("host_out")
    if host is None:
        host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    host.copy_(out, non_blocking=True)
    return host


def merge_partials(m: torch.Tensor, l: torch.Tensor, o: torch.Tensor,
                   out_dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """Split-KV merge of partial softmax states: m, l (parts, rows) fp32 in log2
    units, o (parts, rows, width) fp32 -> (rows, width)."""
    lib = _lib.load()
    parts, rows, width = o.shape
    _require("m", m, shape=(parts, rows), dtype=torch.float32, device=o.device)
    _require("l", l, shape=(parts, rows), dtype=torch.float32, device=o.device)
    _require("o", o, dtype=torch.float32)
    out = torch.empty(rows, width, device=o.device, dtype=out_dtype)
    st = lib.mla_merge_partials(_ptr(m), _ptr(l), _ptr(o), _ptr(out), parts, rows, width,
                                dtype_code(out_dtype), _stream(o.device))
    _lib.check("mla_merge_partials", st)
    return out


def set_option(option: int, value: int) -> None:
    _lib.check("mla_set_option", _lib.load().mla_set_option(option, value))


class StageEvents:
    """Per-stage CUDA events recorded by the library around its kernels (see
    mla_set_stage_events).  Stages: 0 absorb, 1 flash, 2 merge, 3 value
    up-projection, 4 projection, 5 projection k/v."""

    NSTAGE = 6

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * self.NSTAGE)]
        for e in self.events:          # create the underlying cudaEvent_t now
            e.record()
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self.used = set()

    def install(self) -> None:
        _lib.check("mla_set_stage_events",
                   _lib.load().mla_set_stage_events(self._arr, len(self.events)))

    @staticmethod
    def uninstall() -> None:
        _lib.load().mla_set_stage_events(None, 0)

    def elapsed_ms(self, stage: int) -> float:
        return self.events[2 * stage].elapsed_time(self.events[2 * stage + 1])


def launch_count() -> int:
    return int(_lib.load().mla_launch_count())


def device_error(clear: bool = False) -> int:
    code = ctypes.c_uint(0)
    _lib.check("mla_get_device_error", _lib.load().mla_get_device_error(ctypes.byref(code),
                                                                        int(clear)))
    return code.value
