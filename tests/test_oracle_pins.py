"""Pins that tie the float64 oracle to facts other than itself (CPU only).

Each pin is a function ``pin_*(o) -> None`` that raises AssertionError on
failure, so that the same set can be run against copies of the oracle with a
planted mistake (``test_every_planted_mistake_is_caught``).

What pins what:
  weights sum to one ......... softmax normalisation (page FW-GLM-5-1 l2_p31, softmax step)
  t = 0 row equals v_0 ....... inclusive causal mask and the value rebuild
  absorbed == literal ........ the identity (latent W_k) . q = latent . (W_k q)
  explicit == literal ........ brute force: K, V materialised once, numpy softmax
  q = 0 -> causal mean of v .. closed form (all logits equal)
  textbook reduction ......... H = 1, rank = d, W_k = W_v = I is plain causal
                               attention with K = V = latent (torch SDPA, float64)
  peaked logit ............... one dominant key gives that key's value
  last-Tq queries ............ decode rows equal the last rows of the full prefill
  projection ................. one-hot weights select columns; numpy matmul
  online softmax / merge ..... page Kimi-K2.6 l2_p29's worked example [-inf, 0, 0]
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as oracle_mod
from oracle import explicit

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, std=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * std


def _small(seed=0, B=2, Tq=9, Tkv=9, H=3, d=5, R=7):
    q = _rand((B, Tq, H, d), seed)
    lat = _rand((B, Tkv, R), seed + 1)
    wk = _rand((R, H, d), seed + 2, 1 / math.sqrt(R))
    wv = _rand((R, H, d), seed + 3, 1 / math.sqrt(R))
    return q, lat, wk, wv


# --------------------------------------------------------------------------- pins
def pin_weights_sum_to_one(o):
    q, lat, wk, wv = _small(1)
    for (b, h, i) in [(0, 0, 0), (1, 2, 8), (0, 1, 4)]:
        w = o.attention_weights(q, lat, wk, 0.4, b, h, i)
        assert len(w) == i + 1
        assert abs(w.sum() - 1.0) < 1e-15 * 16
        assert (w > 0).all()


def pin_first_row_is_v0(o):
    q, lat, wk, wv = _small(2)
    out = o.attention(q, lat, wk, wv, 0.7)
    R, H, d = wv.shape
    v0 = (lat[:, 0, :] @ wv.reshape(R, H * d)).reshape(lat.shape[0], H, d)
    np.testing.assert_allclose(out[:, 0], v0, rtol=0, atol=1e-13)


def pin_absorbed_equals_literal(o):
    q, lat, wk, wv = _small(3, Tq=6, Tkv=11)
    for causal in (True, False):
        a = o.attention(q, lat, wk, wv, 0.3, causal)
        b = o.attention_absorbed(q, lat, wk, wv, 0.3, causal)
        assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(a)))


def pin_explicit_equals_literal(o):
    q, lat, wk, wv = _small(4, B=2, Tq=13, Tkv=13, H=2, d=4, R=6)
    a = o.attention(q, lat, wk, wv, 0.5)
    b = explicit.attention(q, lat, wk, wv, 0.5)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    q2, lat2, wk2, wv2 = _small(5, B=1, Tq=4, Tkv=10)
    for causal in (True, False):
        a = o.attention(q2, lat2, wk2, wv2, 0.9, causal)
        b = explicit.attention(q2, lat2, wk2, wv2, 0.9, causal)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def pin_zero_query_gives_causal_mean(o):
    q, lat, wk, wv = _small(6, Tq=10, Tkv=10)
    q[:] = 0.0
    out = o.attention(q, lat, wk, wv, 1.3)
    R, H, d = wv.shape
    V = (lat.reshape(-1, R) @ wv.reshape(R, H * d)).reshape(lat.shape[0], lat.shape[1], H, d)
    mean = np.cumsum(V, axis=1) / np.arange(1, lat.shape[1] + 1)[None, :, None, None]
    np.testing.assert_allclose(out, mean, rtol=0, atol=1e-13)


def pin_textbook_reduction(o):
    # H = 1, rank = d, w_up_k = w_up_v = I: K = V = latent (scale != 1 on purpose).
    B, T, d = 2, 12, 8
    q = _rand((B, T, 1, d), 7)
    lat = _rand((B, T, d), 8)
    eye = np.eye(d).reshape(d, 1, d)
    for causal in (True, False):
        out = o.attention(q, lat, eye, eye, 0.37, causal)
        qt = torch.from_numpy(q[:, :, 0, :]).unsqueeze(1)          # (B,1,T,d)
        kt = torch.from_numpy(lat).unsqueeze(1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, kt, is_causal=causal, scale=0.37)
        np.testing.assert_allclose(out[:, :, 0, :], ref[:, 0].numpy(), rtol=1e-12, atol=1e-12)


def pin_peaked_logit(o):
    # Latent rows are orthogonal one-hots e_s; q' selects key j with a huge logit.
    T, d = 6, 6
    lat = np.eye(T).reshape(1, T, T)
    wk = np.eye(T).reshape(T, 1, d)
    wv = _rand((T, 1, d), 9)
    q = np.zeros((1, T, 1, d))
    j = 2
    q[0, T - 1, 0, j] = 60.0
    out = o.attention(q, lat, wk, wv, 1.0)
    np.testing.assert_allclose(out[0, T - 1, 0], wv[j, 0], rtol=0, atol=1e-20 + 1e-12)


def pin_last_queries(o):
    q, lat, wk, wv = _small(10, Tq=12, Tkv=12)
    full = o.attention(q, lat, wk, wv, 0.6)
    last = o.attention(q[:, -3:], lat, wk, wv, 0.6)
    np.testing.assert_allclose(last, full[:, -3:], rtol=0, atol=1e-14)
    rows = o.attention_rows(q, lat, wk, wv, 0.6, [(0, 0), (1, 11), (0, 5)])
    np.testing.assert_allclose(rows, full[[0, 1, 0], [0, 11, 5]], rtol=0, atol=0)
    rows_a = o.attention_rows(q, lat, wk, wv, 0.6, [(0, 0), (1, 11), (0, 5)], form="absorbed")
    np.testing.assert_allclose(rows_a, rows, rtol=1e-12, atol=1e-13)


def pin_projection(o):
    M, Dm, R, C = 7, 10, 4, 6
    hidden = _rand((M, Dm), 11)
    w_down = np.zeros((Dm, R))
    cols = [3, 0, 9, 5]
    for r, j in enumerate(cols):
        w_down[j, r] = 1.0
    wk = np.zeros((R, C)); wk[2, 1] = 1.0; wk[0, 4] = 1.0
    wv = np.zeros((R, C)); wv[3, 0] = 1.0
    lat, k, v = o.project(hidden, w_down, wk, wv)
    assert np.array_equal(lat, hidden[:, cols])
    assert np.array_equal(k[:, 1], hidden[:, cols[2]]) and np.array_equal(k[:, 4], hidden[:, cols[0]])
    assert np.array_equal(v[:, 0], hidden[:, cols[3]]) and not v[:, 1:].any()
    w_down = _rand((Dm, R), 12)
    wk, wv = _rand((R, C), 13), _rand((R, C), 14)
    lat, k, v = o.project(hidden, w_down, wk, wv)
    np.testing.assert_allclose(lat, hidden @ w_down, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(k, (hidden @ w_down) @ wk, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(v, (hidden @ w_down) @ wv, rtol=1e-12, atol=1e-12)
    lat2, k2, v2 = o.project(hidden, w_down)
    assert k2 is None and v2 is None and np.array_equal(lat2, lat)


def _read_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "online_softmax_neg_inf.txt")) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = np.array([float(x) for x in v.split()])
    return vals


def pin_online_softmax_worked_example(o):
    g = _read_golden()
    V = np.stack([g["v0"], g["v1"], g["v2"]])
    out = o.online_softmax(g["scores"], V)
    np.testing.assert_array_equal(out, g["expected"])
    # the same scores as three one-element partitions of the merge
    m = g["scores"]
    l = np.where(np.isinf(m), 0.0, 1.0)
    merged = o.merge_partials(m, l, V * l[:, None])
    np.testing.assert_array_equal(merged, g["expected"])


def pin_merge_matches_full_softmax(o):
    rng = np.random.default_rng(15)
    x = rng.standard_normal(37) * 3
    V = rng.standard_normal((37, 5))
    w = np.exp(x - x.max()); ref = (w / w.sum()) @ V
    np.testing.assert_allclose(o.online_softmax(x, V), ref, rtol=1e-13, atol=1e-13)
    bounds = [0, 5, 6, 20, 20, 37]                    # includes an empty part
    m_i, l_i, o_i = [], [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if a == b:
            m_i.append(-np.inf); l_i.append(0.0); o_i.append(np.zeros(5)); continue
        m = x[a:b].max(); e = np.exp(x[a:b] - m)
        m_i.append(m); l_i.append(e.sum()); o_i.append(e @ V[a:b])
    merged = o.merge_partials(np.array(m_i), np.array(l_i), np.stack(o_i))
    np.testing.assert_allclose(merged, ref, rtol=1e-13, atol=1e-13)


PINS = [pin_weights_sum_to_one, pin_first_row_is_v0, pin_absorbed_equals_literal,
        pin_explicit_equals_literal, pin_zero_query_gives_causal_mean, pin_textbook_reduction,
        pin_peaked_logit, pin_last_queries, pin_projection, pin_online_softmax_worked_example,
        pin_merge_matches_full_softmax]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle):
    pin(oracle)


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7])
def test_every_planted_mistake_is_caught(mutant, tmp_path):
    """Each oracle copy with one planted mistake fails at least one pin."""
    o = oracle_mod.Oracle(path=oracle_mod.build(mutant, out_dir=str(tmp_path)))
    failed = []
    for pin in PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"


def test_config_workloads_match_their_descriptions():
    """The five workloads' shapes, spreads and scales (host logic)."""
    from latent_causal_attention_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS["prefill_bf16"]
    assert (w.B, w.Tq, w.H, w.d, w.rank, w.model_dim) == (2, 4096, 32, 128, 512, 4096)
    assert abs(w.attention_flops() - 1.1682e12) / 1.1682e12 < 1e-3
    assert WORKLOADS["decode_bf16"].pairs() == 64 * 4096
    t = make_inputs(WORKLOADS["tiny_f32"])
    assert t["q"].shape == (2, 32, 4, 16) and t["kv_latent"].shape == (2, 32, 24)
    assert abs(t["w_up_k"].std().item() * math.sqrt(24) - 1) < 0.1
    t2 = make_inputs(WORKLOADS["tiny_f32"])
    assert torch.equal(t["q"], t2["q"])                  # seeded


# ------------------------------------------------- explicit K/V oracle (numpy)
def test_explicit_kv_oracle_matches_literal(oracle):
    """attention_kv over K, V materialised in float64 equals the C oracle's
    literal form, which rebuilds k_s and v_s for every (b, h, t, s)."""
    q, lat, wk, wv = _small(21, B=2, Tq=6, Tkv=11, H=3, d=5, R=7)
    K, V = explicit.materialise_kv(lat, wk, wv)
    for causal in (True, False):
        ref = oracle.attention(q, lat, wk, wv, 0.6, causal)
        np.testing.assert_allclose(explicit.attention_kv(q, K, V, 0.6, causal), ref,
                                   rtol=1e-12, atol=1e-12)


def test_explicit_kv_oracle_matches_sdpa():
    """attention_kv equals torch's float64 scaled-dot-product attention (a
    library routine) with the queries at the last Tq positions."""
    rng = np.random.default_rng(22)
    B, Tq, Tkv, H, d = 2, 5, 9, 2, 4
    q, k, v = (rng.standard_normal(s) for s in [(B, Tq, H, d), (B, Tkv, H, d), (B, Tkv, H, d)])
    t = (Tkv - Tq) + np.arange(Tq)
    mask = torch.from_numpy(np.arange(Tkv)[None, :] <= t[:, None])
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (q, k, v))
    for causal in (True, False):
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=mask if causal else None, scale=0.35).permute(0, 2, 1, 3)
        np.testing.assert_allclose(explicit.attention_kv(q, k, v, 0.35, causal), ref.numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_projection_flop_count_matches_the_printed_toy_figures():
    """The FLOP accounting the benchmark uses, on the toy projection workload,
    against the totals the projection page prints (rounded to 0.1 MFLOP)."""
    from latent_causal_attention_gb300.inputs import WORKLOADS
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "projection_flops.txt")
    printed = {}
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            name, val = line.split(":")
            printed[name.strip()] = float(val)
    w = WORKLOADS["proj_f32"]
    assert (w.B * w.Tkv, w.model_dim, w.rank, w.kv_dim) == (384, 256, 48, 128)
    latent = w.projection_flops(with_kv=False)
    kv = w.projection_flops(with_kv=True) - latent
    assert round(latent / 1e6, 1) == printed["latent"]
    assert round(kv / 2 / 1e6, 1) == printed["k"] == printed["v"]
