"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Small cases compare every element; the full-size workloads compare sampled
rows (every head of the chosen (b, i) rows) against the oracle's literal and
absorbed forms.  Inputs come from the shared seeded generator only.
"""
import math

import numpy as np
import pytest
import torch

import latent_causal_attention_gb300 as mla
from latent_causal_attention_gb300 import _lib
from latent_causal_attention_gb300.inputs import (WORKLOADS, custom_workload, make_inputs,
                                                   make_kv_inputs)
from oracle import explicit

from _util import assert_bf16_close, assert_f32_close, cuda, sample_rows, to_np

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
    assert mla.device_error() == 0


def run_attention(x, w, out_dtype=torch.float32, lat=None):
    return mla.attention(cuda(x["q"]), cuda(x["kv_latent"]) if lat is None else lat,
                         cuda(x["w_up_k"]), cuda(x["w_up_v"]), w.scale, w.causal,
                         out_dtype=out_dtype)


# ----------------------------------------------------------------- fp32 workloads
def test_tiny_f32_full(oracle):
    w = WORKLOADS["tiny_f32"]
    x = make_inputs(w)
    out = run_attention(x, w)
    ref = oracle.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale)
    assert_f32_close(out, ref, "tiny_f32")


def test_proj_f32_projection_then_attention(oracle):
    w = WORKLOADS["proj_f32"]
    x = make_inputs(w)
    wk2, wv2 = x["w_up_k"].reshape(w.rank, -1), x["w_up_v"].reshape(w.rank, -1)
    lat, k, v = mla.project(cuda(x["hidden"]), cuda(x["w_down"]), cuda(wk2), cuda(wv2))
    rl, rk, rv = oracle.project(x["hidden"], x["w_down"], wk2, wv2)
    assert_f32_close(lat.reshape(-1, w.rank), rl, "latent")
    assert_f32_close(k.reshape(-1, w.kv_dim), rk, "k")
    assert_f32_close(v.reshape(-1, w.kv_dim), rv, "v")
    out = run_attention(x, w, lat=lat)
    ref = oracle.attention(x["q"], rl.reshape(w.B, w.Tkv, w.rank), x["w_up_k"], x["w_up_v"],
                           w.scale)
    assert_f32_close(out, ref, "proj_f32 attention")


@pytest.mark.parametrize("shape", [
    dict(B=2, Tq=9, Tkv=13, H=3, d=5, rank=7, causal=True),
    dict(B=1, Tq=1, Tkv=1, H=1, d=1, rank=1, causal=True),
    dict(B=3, Tq=17, Tkv=17, H=2, d=40, rank=100, causal=False),
    dict(B=1, Tq=5, Tkv=70, H=4, d=33, rank=300, causal=True),
])
def test_warp_path_f32_shapes(oracle, shape):
    w = custom_workload("odd", dtype="f32", **shape)
    x = make_inputs(w, seed=7)
    out = run_attention(x, w)
    ref = oracle.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, w.causal)
    assert_f32_close(out, ref, str(shape))


def test_projection_f32_odd(oracle):
    g = torch.Generator().manual_seed(3)
    h = torch.randn(17, 30, generator=g)
    wd = torch.randn(30, 7, generator=g) / 5
    wk = torch.randn(7, 10, generator=g) / 3
    lat, k, v = mla.project(cuda(h), cuda(wd), cuda(wk), None)
    rl, rk, _ = oracle.project(h, wd, wk, None)
    assert v is None
    assert_f32_close(lat, rl, "latent")
    assert_f32_close(k, rk, "k")


# ----------------------------------------------------------------- bf16 workloads
def test_mid_bf16_full(oracle):
    w = WORKLOADS["mid_bf16"]
    x = make_inputs(w)
    out = run_attention(x, w)
    ref = explicit.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale)
    assert_bf16_close(out, ref, "mid_bf16 vs explicit oracle")
    rows = sample_rows(w.B, w.Tq, 4, seed=1)
    lit = oracle.attention_rows(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, rows)
    got = to_np(out)[[r[0] for r in rows], [r[1] for r in rows]]
    assert_bf16_close(got, lit, "mid_bf16 vs literal oracle rows")


def test_prefill_bf16_attention_sampled(oracle):
    w = WORKLOADS["prefill_bf16"]
    x = make_inputs(w, with_projection=False)
    out = run_attention(x, w)
    assert torch.isfinite(out).all()
    prep = oracle.prepare(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"])
    rows = sample_rows(w.B, w.Tq, 8, seed=2, must=((0, 0), (1, 4095), (0, 127), (1, 128)))
    ref = oracle.attention_rows(None, None, None, None, w.scale, rows, prepared=prep,
                                form="absorbed")
    got = to_np(out)[[r[0] for r in rows], [r[1] for r in rows]]
    assert_bf16_close(got, ref, "prefill_bf16 sampled rows")
    lit = oracle.attention_rows(None, None, None, None, w.scale, rows[:2], prepared=prep)
    assert_bf16_close(got[:2], lit, "prefill_bf16 literal rows")


def test_prefill_bf16_projection_chain(oracle):
    """hidden -> latent (GPU, bf16) -> attention (GPU), against the oracle's
    own float64 projection and attention of one sequence."""
    w = WORKLOADS["prefill_bf16"]
    x = make_inputs(w)
    lat, _, _ = mla.project(cuda(x["hidden"]), cuda(x["w_down"]))
    assert lat.dtype == torch.bfloat16 and lat.shape == (w.B, w.Tkv, w.rank)
    b = 1
    rl, _, _ = oracle.project(x["hidden"][b], x["w_down"])
    assert_bf16_close(lat[b].float(), rl, "latent of sequence 1")
    out = run_attention(x, w, lat=lat)
    q1 = x["q"][b:b + 1]
    rows = [(0, 0), (0, 1000), (0, 4095)]
    ref = oracle.attention_rows(q1, rl.reshape(1, w.Tkv, w.rank), x["w_up_k"], x["w_up_v"],
                                w.scale, rows, form="absorbed")
    got = to_np(out)[b, [r[1] for r in rows]]
    assert_bf16_close(got, ref, "projection -> attention chain")


@pytest.mark.parametrize("splits", [0, 4])
def test_decode_bf16_sampled(oracle, splits):
    w = WORKLOADS["decode_bf16"]
    x = make_inputs(w)
    mla.set_option(_lib.OPT_KV_SPLITS, splits)
    try:
        out = run_attention(x, w)
    finally:
        mla.set_option(_lib.OPT_KV_SPLITS, 0)
    prep = oracle.prepare(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"])
    rows = [(0, 0), (17, 0), (63, 0)]
    ref = oracle.attention_rows(None, None, None, None, w.scale, rows, prepared=prep,
                                form="absorbed")
    got = to_np(out)[[r[0] for r in rows], 0]
    assert_bf16_close(got, ref, f"decode_bf16 splits={splits}")


EDGE = [
    dict(B=1, Tq=200, Tkv=200, H=3, d=64, rank=64, causal=True),       # ragged rows, small rank
    dict(B=2, Tq=70, Tkv=300, H=5, d=128, rank=192, causal=True),      # chunked prefill
    dict(B=1, Tq=130, Tkv=130, H=2, d=64, rank=384, causal=True),      # CTA pair, RC=192
    dict(B=2, Tq=33, Tkv=100, H=4, d=64, rank=128, causal=False),      # no mask
    dict(B=3, Tq=1, Tkv=1, H=1, d=64, rank=64, causal=True),           # a single key
    dict(B=1, Tq=64, Tkv=64, H=2, d=192, rank=512, causal=True),       # pair, wide head
    dict(B=1, Tq=96, Tkv=500, H=2, d=128, rank=512, causal=True),      # pair, chunked, ragged
    dict(B=1, Tq=100, Tkv=260, H=2, d=64, rank=512, causal=False),     # pair, no mask
]


MODES = {"auto": (0, 1), "packed": (0, 0), "split3": (3, 1)}   # (kv splits, prefill fused)


@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "x".join(str(v) for v in s.values()))
@pytest.mark.parametrize("mode", list(MODES))
def test_tensor_core_path_edges(oracle, shape, mode):
    """Auto (fused per-head prefill kernel when Tq >= 64 and d <= 128, else the
    head-packed kernels), the head-packed kernels forced, and split-KV forced."""
    w = custom_workload("edge", dtype="bf16", **shape)
    x = make_inputs(w, seed=11)
    splits, fused = MODES[mode]
    mla.set_option(_lib.OPT_KV_SPLITS, splits)
    mla.set_option(_lib.OPT_PREFILL_FUSED, fused)
    try:
        out = run_attention(x, w)
        outb = run_attention(x, w, out_dtype=torch.bfloat16)
    finally:
        mla.set_option(_lib.OPT_KV_SPLITS, 0)
        mla.set_option(_lib.OPT_PREFILL_FUSED, 1)
    ref = oracle.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, w.causal)
    assert_bf16_close(out, ref, f"{shape} {mode}")
    assert_bf16_close(outb.float(), ref, f"{shape} {mode} bf16 out")


def test_bf16_small_head_takes_warp_path(oracle):
    w = custom_workload("small_bf16", dtype="bf16", B=2, Tq=40, Tkv=40, H=3, d=32, rank=48)
    assert mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, torch.bfloat16) == 0
    x = make_inputs(w, seed=5)
    out = run_attention(x, w)
    ref = oracle.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale)
    assert_bf16_close(out, ref, "bf16 warp path")


def test_projection_bf16_with_kv(oracle):
    g = torch.Generator().manual_seed(9)
    M, Dm, R, C = 200, 128, 64, 192
    h = torch.randn(M, Dm, generator=g).bfloat16()
    wd = (torch.randn(Dm, R, generator=g) / math.sqrt(Dm)).bfloat16()
    wk = (torch.randn(R, C, generator=g) / 8).bfloat16()
    wv = (torch.randn(R, C, generator=g) / 8).bfloat16()
    lat, k, v = mla.project(cuda(h), cuda(wd), cuda(wk), cuda(wv))
    rl, rk, rv = oracle.project(h, wd, wk, wv)
    assert_bf16_close(lat.float(), rl, "latent")
    assert_bf16_close(k.float(), rk, "k")
    assert_bf16_close(v.float(), rv, "v")


@pytest.mark.parametrize("R", [64, 256])
def test_projection_bf16_in_fp32_latent(oracle, R):
    """bf16 inputs, fp32 latent (tensor-core GEMM, fp32 output tiles; 200 rows:
    a full and a ragged 128-row tile): fp32 accumulation against float64."""
    g = torch.Generator().manual_seed(10 + R)
    M, Dm = 200, 256
    h = torch.randn(M, Dm, generator=g).bfloat16()
    wd = (torch.randn(Dm, R, generator=g) / math.sqrt(Dm)).bfloat16()
    lat, _, _ = mla.project(cuda(h), cuda(wd), out_dtype=torch.float32)
    rl, _, _ = oracle.project(h, wd)
    assert lat.dtype == torch.float32
    assert_f32_close(lat, rl, f"latent fp32 R{R}")


# ----------------------------------------------------------------- split-KV merge
def test_merge_worked_example(oracle):
    """Scores [-inf, 0, 0] as three one-key parts give (v1 + v2) / 2 (page
    Kimi-K2.6 l2_p29's worked example), through mla_merge_partials."""
    v = torch.tensor([[1.0, 2.0, -4.0, 9.0], [3.0, 5.0, 0.5, 1.0], [7.0, 11.0, -2.5, 3.0]])
    m = torch.tensor([[-math.inf], [0.0], [0.0]])
    l = torch.tensor([[0.0], [1.0], [1.0]])
    o = (v * l).reshape(3, 1, 4)
    out = mla.merge_partials(cuda(m), cuda(l), cuda(o))
    np.testing.assert_array_equal(to_np(out)[0], (to_np(v[1]) + to_np(v[2])) / 2)


def test_merge_random_against_oracle(oracle):
    rng = np.random.default_rng(4)
    parts, rows, width = 5, 37, 64
    m = rng.standard_normal((parts, rows)) * 4
    m[1, :5] = -np.inf                                   # empty parts
    l = np.where(np.isinf(m), 0.0, rng.uniform(0.5, 3, (parts, rows)))
    o = rng.standard_normal((parts, rows, width)) * l[..., None]
    out = mla.merge_partials(cuda(torch.tensor(m, dtype=torch.float32)),
                             cuda(torch.tensor(l, dtype=torch.float32)),
                             cuda(torch.tensor(o, dtype=torch.float32)))
    ln2 = math.log(2.0)
    m32 = torch.tensor(m, dtype=torch.float32).double().numpy()
    l32 = torch.tensor(l, dtype=torch.float32).double().numpy()
    o32 = torch.tensor(o, dtype=torch.float32).double().numpy()
    for r in range(rows):
        ref = oracle.merge_partials(m32[:, r] * ln2, l32[:, r], o32[:, r])
        assert_f32_close(to_np(out)[r], ref, f"row {r}")


# ----------------------------------------------------------------- failure detection
def test_bounded_wait_reports_timeout_and_context_survives(oracle):
    """A wait that can never complete runs out after its limit, records the
    timeout in the device error word and returns; later work still runs."""
    lib = _lib.load()
    assert mla.device_error(clear=True) == 0
    assert lib.mla_check_wait_timeout(2000, None) == 0          # 2 ms limit
    torch.cuda.synchronize()
    assert mla.device_error(clear=True) == 0x17F
    assert mla.device_error() == 0
    test_tiny_f32_full(oracle)                                  # the context is still usable


# ----------------------------------------------------- explicit K/V comparator
EXPLICIT = [
    dict(B=2, Tq=200, Tkv=200, H=3, d=128, causal=True),     # ragged row block
    dict(B=1, Tq=70, Tkv=300, H=4, d=64, causal=True),       # chunked prefill
    dict(B=2, Tq=33, Tkv=100, H=2, d=128, causal=False),     # no mask
    dict(B=3, Tq=1, Tkv=1, H=1, d=64, causal=True),          # a single key
    dict(B=2, Tq=1, Tkv=777, H=5, d=128, causal=True),       # one query over a ragged key range
]


@pytest.mark.parametrize("shape", EXPLICIT, ids=lambda s: "x".join(str(v) for v in s.values()))
def test_explicit_attention_parity(shape):
    """Attention over given k, v (the comparator kernel) against the float64
    softmax attention over the same bf16 k, v."""
    w = custom_workload("explicit", dtype="bf16", rank=64, **shape)
    x = make_kv_inputs(w, seed=31)
    q, k, v = (cuda(x[n]) for n in ("q", "k", "v"))
    out = mla.explicit_attention(q, k, v, w.scale, w.causal)
    outb = mla.explicit_attention(q, k, v, w.scale, w.causal, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ref = explicit.attention_kv(x["q"], x["k"], x["v"], w.scale, w.causal)
    assert_bf16_close(to_np(out), ref, f"explicit {shape}")
    assert_bf16_close(to_np(outb.float()), ref, f"explicit {shape} bf16 out")
    assert mla.device_error() == 0


def test_explicit_path_chain_matches_latent_oracle(oracle):
    """hidden -> latent, k, v (projection kernels, bf16) -> explicit attention,
    against the oracle's float64 projection and literal latent attention: the
    comparator computes the same attention as the absorbed path."""
    w = custom_workload("explicit_chain", dtype="bf16", B=2, Tq=160, Tkv=160, H=4, d=128,
                        rank=128, model_dim=256)
    x = make_inputs(w, seed=33, with_latent=False)
    _, k, v = mla.project(cuda(x["hidden"]), cuda(x["w_down"]), cuda(x["w_up_k"]),
                          cuda(x["w_up_v"]))
    shp = (w.B, w.Tkv, w.H, w.d)
    out = mla.explicit_attention(cuda(x["q"]), k.reshape(shp), v.reshape(shp), w.scale, True)
    rl = np.stack([oracle.project(x["hidden"][b], x["w_down"])[0] for b in range(w.B)])
    # The explicit path stores the latent, k and v as bf16 (the latent feeds the
    # up-projection in bf16): the same three roundings in the reference, then
    # the float64 attention over those k, v.  Against the unrounded literal
    # attention only the normwise error is held to the bf16 bound.
    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()
    kr, vr = explicit.materialise_kv(bf16(rl), x["w_up_k"], x["w_up_v"])
    ref = explicit.attention_kv(x["q"], bf16(kr), bf16(vr), w.scale, True)
    assert_bf16_close(to_np(out), ref, "explicit chain")
    lit = oracle.attention(x["q"], rl, x["w_up_k"], x["w_up_v"], w.scale, True)
    g = to_np(out)
    assert np.linalg.norm(g - lit) <= 2e-2 * np.linalg.norm(lit)


# ------------------------------------------------------ variable-length batch
VARLEN = [
    dict(lens=[(130, 130), (1, 50), (64, 300), (200, 257)], H=3, d=128, rank=512, causal=True),
    dict(lens=[(70, 70), (5, 9), (128, 128)], H=2, d=64, rank=256, causal=True),
    dict(lens=[(33, 100), (129, 140)], H=2, d=128, rank=512, causal=False),
]


@pytest.mark.parametrize("case", VARLEN, ids=lambda c: f"R{c['rank']}d{c['d']}n{len(c['lens'])}"
                         f"{'c' if c['causal'] else 'nc'}")
def test_varlen_batch_matches_per_sequence_oracle(oracle, case):
    """Sequences of different lengths packed back to back, one call, against
    the oracle run on each sequence alone."""
    H, d, R = case["H"], case["d"], case["rank"]
    w0 = custom_workload("varlen", dtype="bf16", B=1, Tq=1, Tkv=1, H=H, d=d, rank=R)
    wts = make_inputs(w0, seed=40)
    qs, lats = [], []
    for n, (tq, tkv) in enumerate(case["lens"]):
        ws = custom_workload("varlen", dtype="bf16", B=1, Tq=tq, Tkv=tkv, H=H, d=d, rank=R)
        x = make_inputs(ws, seed=41 + n)
        qs.append(x["q"][0]); lats.append(x["kv_latent"][0])
    cu_q = [0]; cu_kv = [0]
    for tq, tkv in case["lens"]:
        cu_q.append(cu_q[-1] + tq); cu_kv.append(cu_kv[-1] + tkv)
    q = cuda(torch.cat(qs)); lat = cuda(torch.cat(lats))
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_kv, dtype=torch.int32, device="cuda")
    maxq = max(t for t, _ in case["lens"])
    scale = w0.scale
    out = mla.attention_varlen(q, lat, cuda(wts["w_up_k"]), cuda(wts["w_up_v"]), cq, ck, maxq,
                               scale, case["causal"])
    outb = mla.attention_varlen(q, lat, cuda(wts["w_up_k"]), cuda(wts["w_up_v"]), cq, ck, maxq,
                                scale, case["causal"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert mla.device_error() == 0
    for n, (tq, tkv) in enumerate(case["lens"]):
        ref = oracle.attention(qs[n][None], lats[n][None], wts["w_up_k"], wts["w_up_v"], scale,
                               case["causal"])[0]
        got = to_np(out)[cu_q[n]:cu_q[n + 1]]
        assert_bf16_close(got, ref, f"varlen sequence {n} ({tq},{tkv})")
        assert_bf16_close(to_np(outb.float())[cu_q[n]:cu_q[n + 1]], ref, f"varlen seq {n} bf16")


def test_varlen_bad_lengths_are_reported_not_written():
    """A sequence whose key range is shorter than its query range is skipped
    (its rows stay untouched) and recorded in the device error word."""
    H, d, R = 2, 64, 128
    w0 = custom_workload("varlen", dtype="bf16", B=1, Tq=40, Tkv=40, H=H, d=d, rank=R)
    x = make_inputs(w0, seed=50)
    q = cuda(torch.cat([x["q"][0], x["q"][0]]))
    lat = cuda(x["kv_latent"][0])
    cq = torch.tensor([0, 40, 80], dtype=torch.int32, device="cuda")
    ck = torch.tensor([0, 40, 30], dtype=torch.int32, device="cuda")   # second range is negative
    out = torch.full((80, H, d), 7.0, device="cuda")
    assert mla.device_error(clear=True) == 0
    mla.attention_varlen(q, lat, cuda(x["w_up_k"]), cuda(x["w_up_v"]), cq, ck, 40, w0.scale,
                         out=out)
    torch.cuda.synchronize()
    assert mla.device_error(clear=True) == 0x201
    assert (out[40:] == 7.0).all()
    assert torch.isfinite(out[:40]).all() and not (out[:40] == 7.0).all()


def test_explicit_attention_prefill_size_sampled():
    """The comparator kernel at the prefill size (B2 T4096 H32 d128), sampled
    query rows (all heads) against the float64 attention over the same k, v."""
    w = custom_workload("explicit_prefill", dtype="bf16", B=2, Tq=4096, Tkv=4096, H=32, d=128,
                        rank=64)
    x = make_kv_inputs(w, seed=61)
    out = mla.explicit_attention(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), w.scale, True)
    torch.cuda.synchronize()
    rows = [0, 127, 128, 2049, 4095]
    ref = explicit.attention_kv(x["q"], x["k"], x["v"], w.scale, True, query_rows=rows)
    assert_bf16_close(to_np(out)[:, rows], ref, "explicit prefill sampled rows")


def test_two_streams_run_independent_calls(oracle):
    """Calls on two CUDA streams at once (each with its own workspace and
    output) give the same results as one at a time: no hidden shared state."""
    shapes = [custom_workload("s1", dtype="bf16", B=2, Tq=1, Tkv=700, H=16, d=64, rank=512),
              custom_workload("s2", dtype="bf16", B=1, Tq=256, Tkv=256, H=4, d=128, rank=512)]
    xs = [{k: cuda(v) for k, v in make_inputs(w, seed=70 + n).items()}
          for n, w in enumerate(shapes)]
    refs = [mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale)
            for x, w in zip(xs, shapes)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in shapes]
    outs = []
    for _ in range(3):
        outs = []
        for x, w, s in zip(xs, shapes, streams):
            with torch.cuda.stream(s):
                outs.append(mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"],
                                          w.scale))
        torch.cuda.synchronize()
        for o, r in zip(outs, refs):
            assert torch.equal(o, r)
    assert mla.device_error() == 0


def test_stream_order_with_neighbouring_kernels():
    """The library's kernels start their set-up while the previous kernel on the
    stream finishes (programmatic dependent launch) and touch global memory only
    after it completes.  Torch kernels rewrite the inputs in place right before
    each call and copy, then poison, the output right after it; every copy must
    equal the result of a call made in isolation, and no write may land after
    the poison."""
    shapes = [custom_workload("dec", dtype="bf16", B=2, Tq=1, Tkv=700, H=16, d=64, rank=512),
              custom_workload("pre", dtype="bf16", B=1, Tq=256, Tkv=256, H=4, d=128, rank=512),
              custom_workload("mid", dtype="bf16", B=2, Tq=192, Tkv=192, H=2, d=64, rank=256)]
    for w in shapes:
        xs = [{k: cuda(v) for k, v in make_inputs(w, seed=90 + s).items()} for s in range(2)]
        refs = []
        for x in xs:
            refs.append(mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale))
            torch.cuda.synchronize()
        q, lat = torch.empty_like(xs[0]["q"]), torch.empty_like(xs[0]["kv_latent"])
        out = torch.empty_like(refs[0])
        ws = torch.empty(max(1, mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank,
                                                   torch.bfloat16)),
                         device="cuda", dtype=torch.uint8)
        snaps = []
        for i in range(6):
            x = xs[i % 2]
            q.copy_(x["q"])
            lat.copy_(x["kv_latent"])
            mla.attention(q, lat, x["w_up_k"], x["w_up_v"], w.scale, out=out, workspace=ws)
            snaps.append(out.clone())
            out.fill_(float("nan"))
        torch.cuda.synchronize()
        for i, snap in enumerate(snaps):
            assert torch.equal(snap, refs[i % 2]), (w.name, i)
        assert torch.isnan(out).all(), w.name
    # the projection's latent consumed by the attention on the same stream
    w = custom_workload("chain", dtype="bf16", B=1, Tq=256, Tkv=256, H=4, d=64, rank=256)
    x = {k: cuda(v) for k, v in make_inputs(w, seed=95).items()}
    hidden = torch.randn(w.B, w.Tkv, 512, generator=torch.Generator().manual_seed(96)
                         ).to(torch.bfloat16).cuda()
    w_down = (torch.randn(512, w.rank, generator=torch.Generator().manual_seed(97)) / 22.6
              ).to(torch.bfloat16).cuda()
    lat_ref = mla.project(hidden, w_down)[0]
    ref = mla.attention(x["q"], lat_ref, x["w_up_k"], x["w_up_v"], w.scale)
    torch.cuda.synchronize()
    lat = torch.empty_like(lat_ref)
    for _ in range(4):
        lat.fill_(float("nan"))
        mla.project(hidden, w_down, latent=lat)
        out = mla.attention(x["q"], lat, x["w_up_k"], x["w_up_v"], w.scale)
        got = out.clone()
        lat.fill_(float("nan"))
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
    assert mla.device_error() == 0


def test_calls_capture_into_a_cuda_graph():
    """The calls make no host synchronisation or allocation of their own, so
    they can be captured into a CUDA graph (the programmatic launches become
    programmatic graph edges); replays equal eager calls bit for bit."""
    cases = [custom_workload("dec", dtype="bf16", B=4, Tq=1, Tkv=900, H=32, d=64, rank=512),
             custom_workload("pre", dtype="bf16", B=1, Tq=384, Tkv=384, H=4, d=128, rank=512)]
    for w in cases:
        x = {k: cuda(v) for k, v in make_inputs(w, seed=110).items()}
        out = torch.empty(w.B, w.Tq, w.H, w.d, device="cuda", dtype=torch.float32)
        ws = torch.empty(max(1, mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank,
                                                   torch.bfloat16)),
                         device="cuda", dtype=torch.uint8)
        eager = mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):          # warm-up on the capture stream
            mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, out=out,
                          workspace=ws)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, out=out,
                          workspace=ws)
        for _ in range(3):
            out.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, eager), w.name
    # projection + attention in one graph
    w = custom_workload("chain", dtype="bf16", B=1, Tq=256, Tkv=256, H=4, d=64, rank=256)
    x = {k: cuda(v) for k, v in make_inputs(w, seed=111).items()}
    hidden = torch.randn(w.B, w.Tkv, 512, generator=torch.Generator().manual_seed(112)
                         ).to(torch.bfloat16).cuda()
    w_down = (torch.randn(512, w.rank, generator=torch.Generator().manual_seed(113)) / 22.6
              ).to(torch.bfloat16).cuda()
    lat = torch.empty(w.B, w.Tkv, w.rank, device="cuda", dtype=torch.bfloat16)
    out = torch.empty(w.B, w.Tq, w.H, w.d, device="cuda", dtype=torch.float32)
    mla.project(hidden, w_down, latent=lat)
    eager = mla.attention(x["q"], lat, x["w_up_k"], x["w_up_v"], w.scale)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mla.project(hidden, w_down, latent=lat)
        mla.attention(x["q"], lat, x["w_up_k"], x["w_up_v"], w.scale, out=out)
    for _ in range(3):
        lat.fill_(float("nan"))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert mla.device_error() == 0


# ------------------------------------------- persistent prefill (single CTA and CTA pair)
PERSIST = [
    dict(B=2, Tq=300, Tkv=300, H=4, d=64, rank=256, causal=True),     # ragged row blocks
    dict(B=1, Tq=200, Tkv=700, H=3, d=64, rank=128, causal=True),     # chunked prefill
    dict(B=3, Tq=128, Tkv=128, H=2, d=64, rank=64, causal=False),     # no mask
    dict(B=4, Tq=256, Tkv=256, H=40, d=64, rank=192, causal=True),    # 320 items: three rounds
    # CTA pairs (rank > 256): items of one to five tiles, so that every receive
    # buffer takes q tiles and partial outputs in turn
    dict(B=2, Tq=300, Tkv=300, H=3, d=128, rank=512, causal=True),    # ragged, 2..5 tiles
    dict(B=1, Tq=200, Tkv=700, H=2, d=64, rank=384, causal=True),     # chunked, d 64, RC 192
    dict(B=3, Tq=64, Tkv=64, H=2, d=128, rank=512, causal=True),      # one-tile items
    dict(B=2, Tq=130, Tkv=130, H=2, d=128, rank=512, causal=False),   # no mask, 3-tile items
    dict(B=4, Tq=256, Tkv=256, H=40, d=128, rank=512, causal=True),   # 320 items: five rounds
    dict(B=2, Tq=320, Tkv=320, H=30, d=64, rank=384, causal=True),    # 180 items, RC 192
]


@pytest.mark.parametrize("shape", PERSIST, ids=lambda s: "x".join(str(v) for v in s.values()))
def test_persistent_prefill_matches_per_block_kernel(oracle, shape):
    """Long prefill runs resident CTAs (rank <= 256, d = 64) or resident CTA
    pairs (rank 384 / 512) over all row blocks; they do the same arithmetic as
    one CTA (pair) per row block, so the two agree bit for bit, and both match
    the oracle."""
    w = custom_workload("persist", dtype="bf16", **shape)
    x = make_inputs(w, seed=13)
    outs = {}
    for persistent in (1, 0):
        mla.set_option(_lib.OPT_PERSISTENT, persistent)
        try:
            outs[persistent] = (run_attention(x, w), run_attention(x, w, out_dtype=torch.bfloat16))
            torch.cuda.synchronize()
        finally:
            mla.set_option(_lib.OPT_PERSISTENT, 1)
    assert torch.equal(outs[1][0], outs[0][0]) and torch.equal(outs[1][1], outs[0][1])
    ref = oracle.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, w.causal)
    assert_bf16_close(outs[1][0], ref, f"persistent {shape}")
    assert_bf16_close(outs[1][1].float(), ref, f"persistent {shape} bf16 out")
    assert mla.device_error() == 0


@pytest.mark.parametrize("shape", [
    dict(B=2, Tq=300, Tkv=300, H=3, d=128, rank=512, causal=True),    # 18 items on 4 pairs
    dict(B=2, Tq=640, Tkv=640, H=4, d=64, rank=384, causal=True),     # 40 items on 4 pairs
    dict(B=3, Tq=512, Tkv=512, H=4, d=64, rank=256, causal=True),     # 48 items on 8 CTAs
], ids=lambda s: "x".join(str(v) for v in s.values()))
def test_persistent_prefill_few_workers_many_items(shape):
    """With the planner told of 8 SMs, 4 resident CTA pairs (or 8 single CTAs)
    work through every item: each crosses many item boundaries, where q tiles
    and partial outputs rotate through the receive buffers.  Bitwise equal to
    one CTA (pair) per row block."""
    w = custom_workload("persist_few", dtype="bf16", **shape)
    x = make_inputs(w, seed=17)
    outs = {}
    try:
        mla.set_option(_lib.OPT_NUM_SMS, 8)
        for persistent in (1, 0):
            mla.set_option(_lib.OPT_PERSISTENT, persistent)
            outs[persistent] = (run_attention(x, w), run_attention(x, w, out_dtype=torch.bfloat16))
            torch.cuda.synchronize()
    finally:
        mla.set_option(_lib.OPT_PERSISTENT, 1)
        mla.set_option(_lib.OPT_NUM_SMS, 0)
    assert torch.equal(outs[1][0], outs[0][0]) and torch.equal(outs[1][1], outs[0][1])
    assert mla.device_error() == 0
