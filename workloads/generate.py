"""Seeded input recipe (topic-planted index keys and queries).

* Q, K, V: i.i.d. N(0, 1), rounded to bf16 (round-to-nearest-even).
* Topics u_1..u_n: N(0, I_{d_idx}) vectors normalised to unit length.
* Every key block of every sequence draws a topic t_b ~ U{1..n};
  K_idx[j] = N(0, I) + 3 u_{t_{block(j)}}.
* Every (query, group) draws its own topic t ~ U{1..n};
  Q_idx[i, g] = N(0, I) + 3 u_t.  (One random topic per query, drawn per group
  so that the groups select differently.)
* Decode batches: kv_len = ctx - block + U{1..block}, so the query's own block
  is partial and its position is uniform inside it.

All draws come from one ``torch.Generator`` seeded with the workload's seed, on
the device the tensors are made on; large tensors are drawn in fixed row
chunks so memory stays bounded.  Draw order is fixed by this file.
"""
from __future__ import annotations

import dataclasses
import math

import torch

from .configs import Workload

_CHUNK_ELEMS = 1 << 26  # draw at most 64M normals at a time


@dataclasses.dataclass
class Inputs:
    cfg: Workload
    q: torch.Tensor        # [T, Hq, D] bf16
    k: torch.Tensor        # [N, Hkv, D] bf16
    v: torch.Tensor        # [N, Hkv, D] bf16
    q_idx: torch.Tensor    # [T, Hkv, d_idx] bf16
    k_idx: torch.Tensor    # [N, d_idx] bf16
    cu_q: torch.Tensor     # [S+1] int32
    cu_k: torch.Tensor     # [S+1] int32
    seqs: tuple            # ((q_len, kv_len), ...)

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def total_k(self) -> int:
        return int(self.k.shape[0])

    @property
    def max_q(self) -> int:
        return max(s[0] for s in self.seqs)

    @property
    def max_k(self) -> int:
        return max(s[1] for s in self.seqs)


def _normal_bf16(shape, gen, device, extra=None):
    """N(0,1) in fp32, plus an optional fp32 offset row-block, rounded to bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rows = shape[0]
    per_row = math.prod(shape[1:]) if len(shape) > 1 else 1
    step = max(1, _CHUNK_ELEMS // max(per_row, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen, device=device,
                        dtype=torch.float32)
        if extra is not None:
            x += extra(r0, r1)
        out[r0:r1] = x.to(torch.bfloat16)
    return out


def sequence_lengths(cfg: Workload, gen, device) -> tuple:
    if cfg.seqs is not None:
        return tuple(cfg.seqs)
    assert cfg.decode_batch > 0
    jitter = torch.randint(1, cfg.block + 1, (cfg.decode_batch,), generator=gen, device=device)
    return tuple((1, cfg.decode_ctx - cfg.block + int(j)) for j in jitter.tolist())


def generate(cfg: Workload, device="cpu") -> Inputs:
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed)
    seqs = sequence_lengths(cfg, gen, device)
    for ql, kl in seqs:
        assert 0 <= ql <= kl, (ql, kl)
    cu_q = torch.tensor([0] + [sum(s[0] for s in seqs[:i + 1]) for i in range(len(seqs))],
                        dtype=torch.int32)
    cu_k = torch.tensor([0] + [sum(s[1] for s in seqs[:i + 1]) for i in range(len(seqs))],
                        dtype=torch.int32)
    T, N = int(cu_q[-1]), int(cu_k[-1])

    # topics
    u = torch.randn((cfg.n_topics, cfg.d_idx), generator=gen, device=device, dtype=torch.float32)
    u = u / u.norm(dim=1, keepdim=True)
    # per key-block topic, per sequence (blocks counted from each sequence's start)
    key_topic = torch.empty(N, dtype=torch.int64, device=device)
    for s, (ql, kl) in enumerate(seqs):
        nb = (kl + cfg.block - 1) // cfg.block
        tb = torch.randint(0, cfg.n_topics, (max(nb, 1),), generator=gen, device=device)
        j = torch.arange(kl, device=device)
        key_topic[int(cu_k[s]):int(cu_k[s]) + kl] = tb[j // cfg.block]
    q_topic = torch.randint(0, cfg.n_topics, (T, cfg.hkv), generator=gen, device=device)

    k_idx = _normal_bf16((N, cfg.d_idx), gen, device,
                         extra=lambda a, b: 3.0 * u[key_topic[a:b]])
    q_idx = _normal_bf16((T, cfg.hkv, cfg.d_idx), gen, device,
                         extra=lambda a, b: 3.0 * u[q_topic[a:b]])
    q = _normal_bf16((T, cfg.hq, cfg.head_dim), gen, device)
    k = _normal_bf16((N, cfg.hkv, cfg.head_dim), gen, device)
    v = _normal_bf16((N, cfg.hkv, cfg.head_dim), gen, device)
    return Inputs(cfg, q, k, v, q_idx, k_idx, cu_q.to(device), cu_k.to(device), seqs)


@dataclasses.dataclass
class PrologueInputs:
    x: torch.Tensor        # [T, d_model] bf16 hidden states of the new tokens
    w_q: torch.Tensor      # [hkv * d_idx, d_model] bf16
    w_k: torch.Tensor      # [d_idx, d_model] bf16
    gamma_q: torch.Tensor  # [d_idx] bf16
    gamma_k: torch.Tensor  # [d_idx] bf16


def prologue_inputs(total_q: int, hkv: int, d_idx: int = 128, d_model: int = 3072, seed: int = 2000,
                    device="cpu") -> PrologueInputs:
    """Synthetic index-projection inputs (no trained weights exist here): hidden states N(0, 1), projection
    weights N(0, 1 / d_model) so the projected heads are about N(0, 1), norm weights 1 + 0.1 N(0, 1); all
    rounded to bf16, drawn from one seeded generator in this order."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = _normal_bf16((total_q, d_model), gen, device)
    std = d_model ** -0.5
    w_q = (torch.randn((hkv * d_idx, d_model), generator=gen, device=device) * std).to(torch.bfloat16)
    w_k = (torch.randn((d_idx, d_model), generator=gen, device=device) * std).to(torch.bfloat16)
    gamma_q = (1 + 0.1 * torch.randn((d_idx,), generator=gen, device=device)).to(torch.bfloat16)
    gamma_k = (1 + 0.1 * torch.randn((d_idx,), generator=gen, device=device)).to(torch.bfloat16)
    return PrologueInputs(x, w_q, w_k, gamma_q, gamma_k)
