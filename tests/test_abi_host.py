"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every function include/mla.h declares, and argument validation
rejects bad calls before anything reaches the GPU."""
import ctypes
import os
import re

import pytest

from latent_causal_attention_gb300 import _lib
from latent_causal_attention_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(mla_[a-z_0-9]+)\s*\(",
                                 src, flags=re.M)))


def test_header_declares_the_two_calls():
    names = declared_functions()
    assert "mla_kv_latent_project" in names and "mla_latent_attention" in names
    assert len(names) >= 7


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    assert lib.mla_status_string(0) == b"ok"
    assert lib.mla_status_string(5).startswith(b"workspace")


P = ctypes.c_void_p(16)      # a non-null, 16-byte aligned dummy (never dereferenced)


def attn(lib, **kw):
    a = dict(q=P, lat=P, wk=P, wv=P, out=P, B=2, Tq=8, Tkv=8, H=2, d=64, R=64, scale=0.1,
             causal=1, ind=1, outd=0, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.mla_latent_attention(a["q"], a["lat"], a["wk"], a["wv"], a["out"], a["B"], a["Tq"],
                                    a["Tkv"], a["H"], a["d"], a["R"], a["scale"], a["causal"],
                                    a["ind"], a["outd"], a["ws"], a["wsb"], a["stream"])


def test_attention_validation(lib):
    assert attn(lib, q=None) == 1
    assert attn(lib, out=None) == 1
    assert attn(lib, B=0) == 2
    assert attn(lib, Tq=9, Tkv=8) == 2            # more queries than keys
    assert attn(lib, d=-1) == 2
    assert attn(lib, ind=7) == 3
    assert attn(lib, ind=0, outd=1) == 3          # fp32 in -> bf16 out is not offered
    # tensor-core path (bf16, d and rank multiples of 64) needs a workspace
    assert attn(lib, ws=None, wsb=0) == 5
    need = lib.mla_latent_attention_workspace_size(2, 8, 8, 2, 64, 64, 1, 1)
    assert need > 0
    assert attn(lib, ws=ctypes.c_void_p(256), wsb=need - 1) == 5
    assert attn(lib, ws=ctypes.c_void_p(16), wsb=need) == 4     # workspace not 256-aligned


def test_explicit_attention_validation(lib):
    """Host-side checks of mla_explicit_attention (no launch reaches a GPU)."""
    P = ctypes.c_void_p(256)

    def call(q=P, k=P, v=P, out=P, B=1, Tq=8, Tkv=8, H=2, d=64, ind=1, outd=0):
        return lib.mla_explicit_attention(q, k, v, out, B, Tq, Tkv, H, d, 0.125, 1, ind, outd,
                                          None)
    assert call(k=None) == 1
    assert call(out=None) == 1
    assert call(B=0) == 2
    assert call(Tq=9, Tkv=8) == 2
    assert call(d=96) == 2                       # d must be 64 or 128
    assert call(ind=0) == 3                      # bf16 inputs only
    assert call(outd=5) == 3
    assert call(v=ctypes.c_void_p(264)) == 4     # not 16-byte aligned


def test_varlen_validation(lib):
    """Host-side checks of mla_latent_attention_varlen (no launch reaches a GPU)."""
    P = ctypes.c_void_p(256)

    def call(q=P, cu=P, B=2, maxq=8, tq=16, tkv=16, H=2, d=64, R=128, ind=1, outd=0, cuk=P):
        return lib.mla_latent_attention_varlen(q, P, P, P, P, cu, cuk, B, maxq, tq, tkv, H, d, R,
                                               0.125, 1, ind, outd, None)
    assert call(q=None) == 1
    assert call(cu=None) == 1
    assert call(B=0) == 2
    assert call(maxq=17) == 2                    # longer than all queries together
    assert call(d=192) == 2                      # d 64 or 128
    assert call(R=96) == 2                       # rank a multiple of 64
    assert call(ind=0) == 3                      # bf16 inputs only
    assert call(cuk=ctypes.c_void_p(258)) == 4   # int32 offsets 4-byte aligned


def test_workspace_size_rules(lib):
    ws = lib.mla_latent_attention_workspace_size
    assert ws(2, 32, 32, 4, 16, 24, 0, 1) == 0                 # fp32: warp path, no workspace
    assert ws(2, 32, 32, 4, 16, 24, 1, 1) == 0                 # bf16, d=16: warp path
    assert ws(4, 1024, 1024, 16, 64, 256, 1, 1) == 0           # fused prefill kernel: none
    assert lib.mla_set_option(_lib.OPT_PREFILL_FUSED, 0) == 0
    try:                                                        # head-packed kernels
        assert ws(4, 1024, 1024, 16, 64, 256, 1, 1) >= 2 * 4 * 1024 * 16 * 256 * 2
    finally:
        lib.mla_set_option(_lib.OPT_PREFILL_FUSED, 1)
    assert ws(4, 1024, 1024, 16, 192, 256, 1, 1) > 0            # d > 128: head-packed
    assert ws(0, 1, 1, 1, 64, 64, 1, 1) == 0
    # forcing several key partitions adds the partial buffers
    base = ws(64, 1, 4096, 128, 128, 512, 1, 1)
    assert lib.mla_set_option(_lib.OPT_KV_SPLITS, 4) == 0
    try:
        assert ws(64, 1, 4096, 128, 128, 512, 1, 1) >= base + 4 * 64 * 128 * 512 * 4
    finally:
        lib.mla_set_option(_lib.OPT_KV_SPLITS, 0)


def test_project_validation(lib):
    f = lib.mla_kv_latent_project
    assert f(None, P, None, None, P, None, None, 8, 64, 64, 0, 0, 0, None) == 1
    assert f(P, P, None, None, P, P, None, 8, 64, 64, 64, 0, 0, None) == 1   # k without w_up_k
    assert f(P, P, None, None, P, None, None, 0, 64, 64, 0, 0, 0, None) == 2
    assert f(P, P, None, None, P, None, None, 8, 64, 64, 0, 0, 1, None) == 3


def test_wait_check_validation(lib):
    assert lib.mla_check_wait_timeout(0, None) == 2
    assert lib.mla_check_wait_timeout(20_000_000, None) == 2


def test_options(lib):
    assert lib.mla_set_option(0, 3) == 2
    assert lib.mla_set_option(99, 0) == 8
    assert lib.mla_set_option(0, 0) == 0
    for opt in (_lib.OPT_PREFILL_FUSED, _lib.OPT_PERSISTENT):
        assert lib.mla_set_option(opt, 2) == 2
        assert lib.mla_set_option(opt, -1) == 2
        assert lib.mla_set_option(opt, 1) == 0
    assert lib.mla_merge_partials(None, P, P, P, 1, 1, 4, 0, None) == 1
    assert lib.mla_merge_partials(P, P, P, P, 1, 1, 6, 0, None) == 2


def test_product_path_has_no_fallback():
    """Without the built library the binding raises instead of computing."""
    with pytest.raises(RuntimeError):
        _lib.load(path=os.path.join(ROOT, "does_not_exist.so"))


def test_planner_follows_the_sm_count(lib):
    """The key-range split is sized from the SM count the planner is given
    (MLA_OPT_NUM_SMS), not from a fixed figure: when the head-packed kernels
    have fewer CTAs than half the SMs, the range is split into about
    SMs / CTAs parts (capped by the number of 64-key tiles)."""
    sp = lib.mla_latent_attention_kv_splits
    # decode, 64 sequences x 128 heads, rank 512: 64 CTA pairs = 128 CTAs
    dec = (64, 1, 4096, 128, 128, 512, 1, 1)
    # four sequences: 8 CTAs
    few = (4, 1, 4096, 128, 128, 512, 1, 1)
    try:
        assert lib.mla_set_option(_lib.OPT_NUM_SMS, 152) == 0
        assert sp(*dec) == 1                       # 128 CTAs >= 76: no split
        assert sp(*few) == 19                      # ceil(152 / 8)
        assert lib.mla_set_option(_lib.OPT_NUM_SMS, 512) == 0
        assert sp(*dec) == 4                       # 128 < 256: ceil(512 / 128)
        assert sp(*few) == 64                      # ceil(512 / 8), 64 tiles of keys
        assert sp(4, 1, 1000, 128, 128, 512, 1, 1) == 16   # capped at 16 key tiles
        assert lib.mla_set_option(_lib.OPT_NUM_SMS, 16) == 0
        assert sp(*few) == 1                       # 8 CTAs >= 8
        # the workspace follows the split count (partial O and (m, l) per part)
        ws16 = lib.mla_latent_attention_workspace_size(*few)
        assert lib.mla_set_option(_lib.OPT_NUM_SMS, 152) == 0
        ws152 = lib.mla_latent_attention_workspace_size(*few)
        assert ws152 >= ws16 + 19 * 4 * 128 * 512 * 4
        # paths that never split
        assert sp(2, 4096, 4096, 32, 128, 512, 1, 1) == 1   # fused prefill kernel
        assert sp(2, 32, 32, 4, 16, 24, 0, 1) == 0          # fp32: warp path
        assert lib.mla_set_option(_lib.OPT_NUM_SMS, -1) == 2
    finally:
        lib.mla_set_option(_lib.OPT_NUM_SMS, 0)


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="host-only: without a device no kernel can start")
def test_planner_without_a_device_assumes_152_sms(lib):
    assert lib.mla_latent_attention_kv_splits(4, 1, 4096, 128, 128, 512, 1, 1) == 19


def test_row_count_limit_is_exclusive(lib):
    """B*Tq*H must stay below 2^31 (the kernels index rows with int32):
    exactly 2^31 rows is refused before anything is planned or launched."""
    assert attn(lib, B=1, Tq=1 << 30, Tkv=1 << 30, H=2) == 2
    assert attn(lib, B=2, Tq=8, Tkv=1 << 30, H=1) == 2            # B*Tkv = 2^31
    # one row fewer passes the shape checks and stops at the missing workspace
    # of the head-packed kernels (the fused kernel, which needs none, is
    # switched off so that nothing can be launched)
    assert lib.mla_set_option(_lib.OPT_PREFILL_FUSED, 0) == 0
    try:
        assert attn(lib, B=1, Tq=(1 << 31) - 1, Tkv=(1 << 31) - 1, H=1) == 5
    finally:
        lib.mla_set_option(_lib.OPT_PREFILL_FUSED, 1)
    f = lib.mla_kv_latent_project
    assert f(P, P, None, None, P, None, None, 1 << 31, 64, 64, 0, 1, 1, None) == 2


def test_noalloc_refuses_only_what_its_scratch_cannot_hold(lib):
    """The allocation-free call refuses sizes whose tensor-core scratch would
    exceed its fixed array, before launching anything; sizes that need no
    scratch (fp32, the warp path) are never refused for their size."""
    big = (8, 32, 4096, 128, 128, 512)              # ~67 MB of head-packed scratch
    assert lib.mla_latent_attention_workspace_size(*big, 1, 1) > 32 * 1024 * 1024
    before = lib.mla_launch_count()
    st = lib.mla_latent_attention_noalloc(P, P, P, P, P, *big, 0.1, 1, 1, 0, None)
    assert st == 5
    assert lib.mla_launch_count() == before
    assert lib.mla_latent_attention_noalloc(None, P, P, P, P, *big, 0.1, 1, 1, 0, None) in (1, 5)
