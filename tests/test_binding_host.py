"""The Python binding's argument checks (no GPU): mismatched shapes, dtypes
and devices are refused before any pointer reaches the C ABI, whose kernels
trust the sizes they are given."""
import pytest
import torch

import latent_causal_attention_gb300 as mla


def _attn_args(B=1, Tq=4, Tkv=4, H=2, d=64, R=64, dt=torch.bfloat16):
    return (torch.zeros(B, Tq, H, d, dtype=dt), torch.zeros(B, Tkv, R, dtype=dt),
            torch.zeros(R, H, d, dtype=dt), torch.zeros(R, H, d, dtype=dt))


def test_attention_refuses_mismatched_arguments():
    q, lat, wk, wv = _attn_args()
    with pytest.raises(ValueError, match="w_up_k"):
        mla.attention(q, lat, wk[:32], wv, 0.1)                  # too few rank rows
    with pytest.raises(TypeError, match="kv_latent"):
        mla.attention(q, lat.float(), wk, wv, 0.1)               # latent dtype differs from q
    with pytest.raises(ValueError, match="kv_latent"):
        mla.attention(q, torch.zeros(2, 4, 64, dtype=torch.bfloat16), wk, wv, 0.1)  # batch
    with pytest.raises(ValueError, match="out"):
        mla.attention(q, lat, wk, wv, 0.1, out=torch.zeros(1, 4, 2, 32))
    with pytest.raises(TypeError, match="workspace"):
        mla.attention(q, lat, wk, wv, 0.1, workspace=torch.zeros(16))
    with pytest.raises(ValueError, match="GPU"):             # well-formed, but on the host
        mla.attention(q, lat, wk, wv, 0.1)


def test_project_refuses_mismatched_arguments():
    h = torch.zeros(8, 128, dtype=torch.bfloat16)
    wd = torch.zeros(128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="hidden"):
        mla.project(torch.zeros(8, 96, dtype=torch.bfloat16), wd)
    with pytest.raises(TypeError, match="w_down"):
        mla.project(h, wd.float())
    with pytest.raises(ValueError, match="w_up_k"):
        mla.project(h, wd, torch.zeros(32, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="latent"):
        mla.project(h, wd, latent=torch.zeros(8, 32, dtype=torch.bfloat16))


def test_varlen_and_explicit_refuse_mismatched_arguments():
    q = torch.zeros(10, 2, 64, dtype=torch.bfloat16)
    lat = torch.zeros(12, 64, dtype=torch.bfloat16)
    w = torch.zeros(64, 2, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 10], dtype=torch.int32)
    with pytest.raises(TypeError, match="cu_seqlens_q"):
        mla.attention_varlen(q, lat, w, w, cu.long(), cu, 10, 0.1)
    with pytest.raises(ValueError, match="cu_seqlens_kv"):
        mla.attention_varlen(q, lat, w, w, cu, torch.tensor([0, 5, 12], dtype=torch.int32),
                             10, 0.1)
    qe = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="v"):
        mla.explicit_attention(qe, torch.zeros(1, 6, 2, 64, dtype=torch.bfloat16),
                               torch.zeros(1, 5, 2, 64, dtype=torch.bfloat16), 0.1)
