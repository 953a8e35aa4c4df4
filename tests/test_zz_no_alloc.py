"""The allocation-free attention entry point (mla_latent_attention_noalloc).

It is meant for callers that cannot allocate device memory where they run
attention: code that must not call cudaMalloc / cudaFree on its hot path,
plugins inside a framework that owns all GPU memory, runtimes with a fixed
memory budget.  Such a caller passes inputs and output only; the scratch is
the library's own fixed device array.

These tests call it through the C ABI, twice in a row per case (the second
call reuses scratch that still holds the first call's data), and compare both
results with the regular entry point, which gets a caller-provided workspace,
using the same tolerances as the other parity tests.  The file is named so
that pytest collects it last.
"""
import ctypes

import pytest
import torch

import latent_causal_attention_gb300 as mla
from latent_causal_attention_gb300 import _lib
from latent_causal_attention_gb300.inputs import WORKLOADS, custom_workload, make_inputs

from _util import assert_bf16_close, assert_f32_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from latent_causal_attention_gb300.build import build
    build()
    lib = _lib.load()
    mla.set_option(_lib.OPT_ATTN_PATH, 0)
    mla.set_option(_lib.OPT_KV_SPLITS, 0)
    mla.set_option(_lib.OPT_PREFILL_FUSED, 1)
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def call_noalloc(lib, x, w, out):
    st = lib.mla_latent_attention_noalloc(
        _p(x["q"]), _p(x["kv_latent"]), _p(x["w_up_k"]), _p(x["w_up_v"]), _p(out),
        w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, float(w.scale), int(w.causal),
        mla.dtype_code(x["q"].dtype), mla.dtype_code(out.dtype),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


CASES = [
    custom_workload("decode_pair", dtype="bf16", B=4, Tq=1, Tkv=777, H=16, d=64, rank=512),
    custom_workload("prefill_single", dtype="bf16", B=2, Tq=300, Tkv=300, H=4, d=64, rank=256),
    custom_workload("chunk_pair", dtype="bf16", B=1, Tq=40, Tkv=200, H=8, d=128, rank=384),
    WORKLOADS["tiny_f32"],
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_regular_entry_point(lib, w):
    need = mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, w.torch_dtype, w.causal)
    assert need <= 32 * 1024 * 1024
    x = {k: v.cuda() for k, v in make_inputs(w, seed=21).items()}
    ref = mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, w.causal)
    torch.cuda.synchronize()
    check = assert_f32_close if w.dtype == "f32" else assert_bf16_close
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert call_noalloc(lib, x, w, out) == 0
        torch.cuda.synchronize()
        check(out, ref, f"{w.name} call {call}")
    assert mla.device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    """A decode batch with 32 queries per sequence over 4096 positions, 128
    heads, rank 512 needs ~67 MB of scratch: refused, nothing launched."""
    w = custom_workload("big", dtype="bf16", B=8, Tq=32, Tkv=4096, H=128, d=128, rank=512)
    need = mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, torch.bfloat16)
    assert need > 32 * 1024 * 1024
    dummy = ctypes.c_void_p(256)            # never dereferenced: the size check comes first
    before = mla.launch_count()
    st = lib.mla_latent_attention_noalloc(dummy, dummy, dummy, dummy, dummy, w.B, w.Tq, w.Tkv,
                                          w.H, w.d, w.rank, float(w.scale), 1, 1, 0, None)
    assert st == 5                           # MLA_ERR_WORKSPACE
    assert mla.launch_count() == before
