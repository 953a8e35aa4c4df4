"""The allocation-free attention entry point (mla_latent_attention_noalloc).

It is meant for callers that cannot allocate device memory where they run
attention: code that must not call cudaMalloc / cudaFree on its hot path
(both synchronise the device), plugins inside a framework that owns all GPU
memory, runtimes with a fixed memory budget.  Such a caller passes inputs and
output only; the scratch is the library's own fixed device array, shared by
every call on the device.

Each case calls the entry point through the C ABI, twice in a row.  Before
each checked call, a call with other inputs, another shape and much larger
values goes through the same entry point, so the shared array holds
different data wherever the checked call might read it.  A checked result
must equal, bit for bit, the result of the regular entry point with a
caller-provided workspace (the same kernels run with the same plan).  The
interleaved calls are checked the same way.  Any byte that a call reads from
the array before writing it would show up as a difference.  The file is
named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import latent_causal_attention_gb300 as mla
from latent_causal_attention_gb300 import _lib
from latent_causal_attention_gb300.inputs import WORKLOADS, custom_workload, make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024


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
    return lib.mla_latent_attention_noalloc(
        _p(x["q"]), _p(x["kv_latent"]), _p(x["w_up_k"]), _p(x["w_up_v"]), _p(out),
        w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, float(w.scale), int(w.causal),
        mla.dtype_code(x["q"].dtype), mla.dtype_code(out.dtype),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def regular(x, w):
    """The regular entry point with a workspace of exactly the size it asks for."""
    ws = mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, w.torch_dtype, w.causal)
    buf = torch.empty(max(ws, 1), device="cuda", dtype=torch.uint8)
    return mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, w.causal,
                         workspace=buf)


def inputs(w, seed, gain=1.0):
    x = {k: v.cuda() for k, v in make_inputs(w, seed=seed).items()}
    if gain != 1.0:
        x["q"] = (x["q"].float() * gain).to(x["q"].dtype)
        x["kv_latent"] = (x["kv_latent"].float() * gain).to(x["kv_latent"].dtype)
    return x


CASES = [
    # head-packed kernels, CTA pair, key range split in 13 parts: q', o_lat,
    # partial O and (m, l) all live in the scratch
    custom_workload("decode_pair", dtype="bf16", B=4, Tq=1, Tkv=777, H=16, d=64, rank=512),
    # head-packed kernels with a short chunk (Tq < 64), 4 key-range parts
    custom_workload("chunk_pair", dtype="bf16", B=1, Tq=40, Tkv=200, H=8, d=128, rank=384),
    # fused prefill kernel: no scratch
    custom_workload("prefill_single", dtype="bf16", B=2, Tq=300, Tkv=300, H=4, d=64, rank=256),
    # fp32: warp-per-query path, no scratch
    WORKLOADS["tiny_f32"],
]

# Written into the shared array before each checked call: larger scratch
# regions (more rows, more key-range parts) than any case above, other
# values (another seed, inputs scaled up) so that leftovers differ.
POISON = custom_workload("poison", dtype="bf16", B=8, Tq=1, Tkv=2000, H=32, d=64, rank=512)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_regular_entry_point(lib, w):
    need = mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, w.torch_dtype, w.causal)
    poison_need = mla.workspace_size(POISON.B, POISON.Tq, POISON.Tkv, POISON.H, POISON.d,
                                     POISON.rank, torch.bfloat16)
    assert need <= SCRATCH_BYTES and need <= poison_need <= SCRATCH_BYTES
    x = inputs(w, seed=21)
    px = inputs(POISON, seed=22, gain=8.0)
    ref = regular(x, w)
    pref = regular(px, POISON)
    torch.cuda.synchronize()
    for call in range(2):
        pout = torch.full_like(pref, float("nan"))
        assert call_noalloc(lib, px, POISON, pout) == 0
        out = torch.full_like(ref, float("nan"))
        assert call_noalloc(lib, x, w, out) == 0
        torch.cuda.synchronize()
        assert torch.equal(pout, pref), f"poison call before {w.name} call {call}"
        assert torch.equal(out, ref), f"{w.name} call {call}"
    assert mla.device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    """A decode batch with 32 queries per sequence over 4096 positions, 128
    heads, rank 512 needs ~67 MB of scratch: refused, nothing launched."""
    w = custom_workload("big", dtype="bf16", B=8, Tq=32, Tkv=4096, H=128, d=128, rank=512)
    need = mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, torch.bfloat16)
    assert need > SCRATCH_BYTES
    dummy = ctypes.c_void_p(256)            # never dereferenced: the size check comes first
    before = mla.launch_count()
    st = lib.mla_latent_attention_noalloc(dummy, dummy, dummy, dummy, dummy, w.B, w.Tq, w.Tkv,
                                          w.H, w.d, w.rank, float(w.scale), 1, 1, 0, None)
    assert st == 5                           # MLA_ERR_WORKSPACE
    assert mla.launch_count() == before
