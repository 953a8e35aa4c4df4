"""GPU parity over the WHOLE output of the two full-size bf16 workloads.

* prefill: causal latent attention B2 T4096 H32 d128 rank 512 (the fused
  per-head kernel that the benchmark times, and the head-packed kernels);
* decode: one query at t = 4095 over 4096 latent rows, B64 H128 d128 rank 512
  (the automatic plan and a forced four-way split of the key range).

Every output element is compared with two float64 oracles that reach the
definition differently: the C oracle's absorbed form (pinned equal to the
literal form) and the numpy brute force that materialises k and v
(``oracle/explicit.py``), the latter one head (prefill) or one sequence
(decode) at a time to bound its memory.  The literal form (k and v rebuilt for
every key) is run on a sample of rows: 16 (b, i) rows of the prefill,
including i = 0, 127, 128 and 4095, and 8 whole decode sequences.
Definition: page "FW-GLM-5-1 l2_p31" (fused MLA-style attention from
compressed KV latents), "The algorithm".
"""
import numpy as np
import pytest
import torch

import latent_causal_attention_gb300 as mla
from latent_causal_attention_gb300 import _lib
from latent_causal_attention_gb300.inputs import WORKLOADS, make_inputs
from oracle import explicit

from _util import assert_bf16_close, cuda, sample_rows, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from latent_causal_attention_gb300.build import build
    build()
    mla.set_option(_lib.OPT_ATTN_PATH, 0)
    mla.set_option(_lib.OPT_KV_SPLITS, 0)
    mla.set_option(_lib.OPT_PREFILL_FUSED, 1)
    yield
    mla.set_option(_lib.OPT_KV_SPLITS, 0)
    mla.set_option(_lib.OPT_PREFILL_FUSED, 1)
    assert mla.device_error() == 0


def gpu_attention(x, w, splits=0, fused=1):
    mla.set_option(_lib.OPT_KV_SPLITS, splits)
    mla.set_option(_lib.OPT_PREFILL_FUSED, fused)
    try:
        out = mla.attention(cuda(x["q"]), cuda(x["kv_latent"]), cuda(x["w_up_k"]),
                            cuda(x["w_up_v"]), w.scale, w.causal)
        torch.cuda.synchronize()
    finally:
        mla.set_option(_lib.OPT_KV_SPLITS, 0)
        mla.set_option(_lib.OPT_PREFILL_FUSED, 1)
    assert mla.device_error() == 0
    return to_np(out)


# ------------------------------------------------------------------ prefill
@pytest.fixture(scope="module")
def prefill(oracle):
    w = WORKLOADS["prefill_bf16"]
    x = make_inputs(w, with_projection=False)
    outs = {"fused": gpu_attention(x, w), "head_packed": gpu_attention(x, w, fused=0)}
    absorbed = oracle.attention_absorbed(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"],
                                         w.scale, w.causal)
    expl = np.empty_like(absorbed)
    for h in range(w.H):
        expl[:, :, h:h + 1] = explicit.attention(
            x["q"][:, :, h:h + 1], x["kv_latent"], x["w_up_k"][:, h:h + 1],
            x["w_up_v"][:, h:h + 1], w.scale, w.causal)
    rows = sample_rows(w.B, w.Tq, 18, seed=12,
                       must=((0, 0), (1, 127), (0, 128), (1, 4095), (0, 4095), (1, 0)))
    assert len(rows) >= 16
    prep = oracle.prepare(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"])
    literal = oracle.attention_rows(None, None, None, None, w.scale, rows, prepared=prep,
                                    form="literal")
    return dict(w=w, outs=outs, absorbed=absorbed, explicit=expl, rows=rows, literal=literal)


def test_prefill_oracles_agree(prefill):
    """The two full float64 oracles and the literal rows agree with each other
    (float64 rounding only), so each is a check of the other."""
    a, e = prefill["absorbed"], prefill["explicit"]
    assert np.abs(a - e).max() <= 1e-9 * max(1.0, np.abs(a).max())
    r = prefill["rows"]
    sel = a[[b for b, _ in r], [i for _, i in r]]
    assert np.abs(sel - prefill["literal"]).max() <= 1e-9 * max(1.0, np.abs(sel).max())


@pytest.mark.parametrize("path", ["fused", "head_packed"])
def test_prefill_full_output(prefill, path):
    got = prefill["outs"][path]
    assert_bf16_close(got, prefill["absorbed"], f"prefill {path}, all outputs, absorbed oracle")
    assert_bf16_close(got, prefill["explicit"], f"prefill {path}, all outputs, explicit oracle")
    r = prefill["rows"]
    assert_bf16_close(got[[b for b, _ in r], [i for _, i in r]], prefill["literal"],
                      f"prefill {path}, literal rows")


def test_prefill_every_block_and_head_within_bound(prefill):
    """The error bound holds for every 128-row block of every head on its
    own (a fault confined to one CTA's rows or one half of a CTA pair would
    show here even where the global norm hides it)."""
    w = prefill["w"]
    got, ref = prefill["outs"]["fused"], prefill["absorbed"]
    for b in range(w.B):
        for rb in range(0, w.Tq, 128):
            for h in range(w.H):
                assert_bf16_close(got[b, rb:rb + 128, h], ref[b, rb:rb + 128, h],
                                  f"prefill b{b} rows {rb}.. head {h}")


# ------------------------------------------------------------------ decode
@pytest.fixture(scope="module")
def decode(oracle):
    w = WORKLOADS["decode_bf16"]
    x = make_inputs(w)
    outs = {"auto": gpu_attention(x, w), "split4": gpu_attention(x, w, splits=4)}
    absorbed = oracle.attention_absorbed(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"],
                                         w.scale, w.causal)
    expl = np.empty_like(absorbed)
    for b in range(w.B):
        expl[b:b + 1] = explicit.attention(x["q"][b:b + 1], x["kv_latent"][b:b + 1],
                                           x["w_up_k"], x["w_up_v"], w.scale, w.causal)
    seqs = [0, 7, 17, 29, 38, 46, 55, 63]
    prep = oracle.prepare(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"])
    literal = oracle.attention_rows(None, None, None, None, w.scale, [(b, 0) for b in seqs],
                                    prepared=prep, form="literal")
    return dict(w=w, outs=outs, absorbed=absorbed, explicit=expl, seqs=seqs, literal=literal)


def test_decode_oracles_agree(decode):
    a, e = decode["absorbed"], decode["explicit"]
    assert np.abs(a - e).max() <= 1e-9 * max(1.0, np.abs(a).max())
    sel = a[decode["seqs"], 0]
    assert np.abs(sel - decode["literal"]).max() <= 1e-9 * max(1.0, np.abs(sel).max())


@pytest.mark.parametrize("path", ["auto", "split4"])
def test_decode_full_output(decode, path):
    got = decode["outs"][path]
    assert_bf16_close(got, decode["absorbed"], f"decode {path}, all outputs, absorbed oracle")
    assert_bf16_close(got, decode["explicit"], f"decode {path}, all outputs, explicit oracle")
    assert_bf16_close(got[decode["seqs"], 0], decode["literal"],
                      f"decode {path}, literal sequences")
    for b in range(decode["w"].B):                 # every sequence on its own
        assert_bf16_close(got[b], decode["absorbed"][b], f"decode {path} sequence {b}")
