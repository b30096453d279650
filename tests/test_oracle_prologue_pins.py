"""Pins for the oracle's index prologue (hidden states -> index query and key
heads: linear projection, RMSNorm, RoPE on the first 64 of 128 dims; "MiniMax
Sparse Attention: let each query pick its own blocks", Figure 1, and the atlas
record's d_model 3072 / RoPE dimension 64), against facts outside the oracle:
  * torch.nn.functional.rms_norm (a library routine) on identity projections;
  * RMSNorm's scale invariance and the constant-vector case;
  * RoPE as multiplication of each pair (z_j + i z_{j+half}) by the unit complex
    number exp(i * pos * theta_j) (Python's cmath), position 0 as the identity,
    and dot products that depend only on the difference of positions.
No GPU is needed.
"""
import cmath

import numpy as np
import pytest
import torch

import oracle


def bf(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def _case(T=6, d_model=32, hkv=2, d_idx=8, seed=0, kv_extra=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d_model, generator=g).to(torch.bfloat16)
    wq = (torch.randn(hkv * d_idx, d_model, generator=g) / d_model ** 0.5).to(torch.bfloat16)
    wk = (torch.randn(d_idx, d_model, generator=g) / d_model ** 0.5).to(torch.bfloat16)
    gq = (1 + 0.1 * torch.randn(d_idx, generator=g)).to(torch.bfloat16)
    gk = (1 + 0.1 * torch.randn(d_idx, generator=g)).to(torch.bfloat16)
    cu_q = np.array([0, T], np.int32)
    cu_k = np.array([0, T + kv_extra], np.int32)
    return cu_q, cu_k, x, wq, wk, gq, gk


def test_identity_projection_matches_torch_rms_norm():
    cu_q, cu_k, x, _, _, gq, gk = _case(d_model=24, hkv=2, d_idx=8)
    eye = torch.eye(24)
    wq = eye[:16].to(torch.bfloat16)       # head h reads features 8h .. 8h + 7
    wk = eye[16:24].to(torch.bfloat16)
    q, k = oracle.index_prologue(cu_q, cu_k, x, wq, wk, gq, gk, rope_dim=0, eps=1e-6)
    xd = x.double()
    ref_q = torch.nn.functional.rms_norm(xd[:, :16].reshape(-1, 2, 8), (8,), weight=gq.double(), eps=1e-6)
    ref_k = torch.nn.functional.rms_norm(xd[:, 16:24], (8,), weight=gk.double(), eps=1e-6)
    np.testing.assert_allclose(q, ref_q.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(k, ref_k.numpy(), rtol=1e-12, atol=1e-12)


def test_rms_norm_is_scale_invariant_and_normalises_constants():
    cu_q, cu_k, x, wq, wk, gq, gk = _case(seed=1)
    a = oracle.index_prologue(cu_q, cu_k, x, wq, wk, gq, gk, rope_dim=8, eps=0.0)
    b = oracle.index_prologue(cu_q, cu_k, (x.float() * 4).to(torch.bfloat16), wq, wk, gq, gk, rope_dim=8, eps=0.0)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    # every output of a head the same projection c * sum(x): normalised to sign(c) * gamma (no RoPE, eps 0)
    d_model, d_idx = x.shape[1], 8
    w = torch.zeros(d_idx, d_model)
    w[:, :4] = 0.5
    q, k = oracle.index_prologue(cu_q, cu_k, x, w.repeat(2, 1).to(torch.bfloat16), (-w).to(torch.bfloat16),
                                 gq, gk, rope_dim=0, eps=0.0)
    s = np.sign(x[:, :4].double().sum(1).numpy())
    np.testing.assert_allclose(q, np.broadcast_to(s[:, None, None] * gq.double().numpy()[None, None, :], q.shape),
                               rtol=1e-15)
    np.testing.assert_allclose(k, -s[:, None] * gk.double().numpy()[None, :], rtol=1e-15)


@pytest.mark.parametrize("rope_dim,base", [(2, 10000.0), (4, 100.0), (8, 10000.0)])
def test_rope_is_a_complex_rotation_of_each_pair(rope_dim, base):
    cu_q, cu_k, x, wq, wk, gq, gk = _case(T=7, seed=2, kv_extra=1000)
    plain_q, plain_k = oracle.index_prologue(cu_q, cu_k, x, wq, wk, gq, gk, rope_dim=0)
    q, k = oracle.index_prologue(cu_q, cu_k, x, wq, wk, gq, gk, rope_dim=rope_dim, rope_base=base)
    half = rope_dim // 2
    pos = oracle.query_positions(cu_q, cu_k)
    for i in range(len(pos)):
        for j in range(half):
            rot = cmath.exp(1j * pos[i] * base ** (-j / half))
            for got, src in ((q[i, 0], plain_q[i, 0]), (q[i, 1], plain_q[i, 1]), (k[i], plain_k[i])):
                want = complex(src[j], src[j + half]) * rot
                assert abs(complex(got[j], got[j + half]) - want) < 1e-12
        np.testing.assert_array_equal(q[i, :, rope_dim:], plain_q[i, :, rope_dim:])   # dims past rope_dim untouched
        np.testing.assert_array_equal(k[i, rope_dim:], plain_k[i, rope_dim:])


def test_rope_position_zero_is_identity_and_dots_depend_on_offsets_only():
    cu_q, cu_k, x, wq, wk, gq, gk = _case(T=9, seed=3)
    plain_q, plain_k = oracle.index_prologue(cu_q, cu_k, x, wq, wk, gq, gk, rope_dim=0)
    q0, k0 = oracle.index_prologue(cu_q, cu_k, x, wq, wk, gq, gk, rope_dim=8)
    np.testing.assert_array_equal(q0[0], plain_q[0])   # token 0 sits at position 0
    # the same tokens 5000 positions later: query-key dot products are unchanged
    q1, k1 = oracle.index_prologue(cu_q, np.array([0, 9 + 5000], np.int32), x, wq, wk, gq, gk, rope_dim=8)
    d0 = np.einsum("ihd,jd->ihj", q0, k0)
    d1 = np.einsum("ihd,jd->ihj", q1, k1)
    np.testing.assert_allclose(d1, d0, rtol=0, atol=1e-9)
    assert np.abs(q1 - q0).max() > 1e-3                 # while the vectors themselves did rotate
