"""GPU parity of the index prologue (hidden states -> index query and key heads:
projection, RMSNorm, RoPE on dims 0..63; "MiniMax Sparse Attention: let each
query pick its own blocks", Figure 1; readings stated in include/msa.h) against
the oracle's unrounded values.

Tolerance: the kernel accumulates the projection in fp32 on the tensor cores
and rounds each output once to bf16, the oracle works in double, so every
output is within one bf16 unit in the last place (2^-7 relative to the power
of two below it) of the oracle's value plus the fp32 accumulation error, which
matters only for outputs near zero: about k u sum_c |x_c w_c| with u = 2^-24,
a partial-sum depth k of about 16 and sum_c |x_c w_c| of about 36 at d_model
3072 (|x| ~ 0.8, |w| ~ 0.8 / sqrt(3072)), so 5e-5 absolute is allowed on top;
at least 99 % of the outputs must equal the oracle's value rounded to bf16.
K_idx rows other than the new tokens' must be left untouched.
"""
import types

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads.configs import small

from parity import problem_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_05_gb300 as m
    torch.cuda.set_device(0)
    return m


def _bf16_ulp(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.exp2(e - 7)


def _check(got, ref, what):
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    bound = _bf16_ulp(ref) + 5e-5
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs beyond one bf16 ulp, worst {err[bad].max():.3e}"
    same = got == torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert same.mean() > 0.99, f"{what}: only {same.mean():.4f} of the outputs equal the rounded oracle value"
    return float(err.max()), float(same.mean())


def _run(msa, x, cfg, d_model, rows=None, seed=2001):
    prob = problem_for(msa, x)
    pin = workloads.prologue_inputs(x.total_q, cfg.hkv, d_model=d_model, seed=seed, device="cuda")
    k_idx = torch.full((x.total_k, 128), 7.0, dtype=torch.bfloat16, device="cuda")   # sentinel
    ws = msa.workspace(prob, msa.Op.INDEX_PROLOGUE)
    q_idx = msa.msa_index_prologue(prob, pin.x, pin.w_q, pin.w_k, pin.gamma_q, pin.gamma_k, k_idx, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    rq, rk = oracle.index_prologue(x.cu_q, x.cu_k, pin.x, pin.w_q, pin.w_k, pin.gamma_q, pin.gamma_k, rows=rows)
    pos = oracle.query_positions(x.cu_q, x.cu_k)
    cu_q, cu_k = x.cu_q.cpu().numpy(), x.cu_k.cpu().numpy()
    seq = np.searchsorted(cu_q, np.arange(x.total_q), side="right") - 1
    krow = cu_k[seq] + pos
    sel = np.arange(x.total_q) if rows is None else rows
    gq = q_idx.float().cpu().numpy()[sel]
    gk = k_idx.float().cpu().numpy()
    out = _check(gq, rq, "Q_idx") + _check(gk[krow[sel]], rk, "K_idx")
    # rows of the cache that are not new tokens keep their contents
    untouched = np.ones(x.total_k, bool)
    untouched[krow] = False
    assert np.all(gk[untouched] == 7.0)
    return out


CASES = {
    # packed varlen with chunked sequences (queries are the last q_len positions), ragged last row tile
    "varlen_d512": (dict(seqs=((300, 300), (1000, 1777), (1, 129), (129, 900), (640, 640)), hq=64, hkv=4, d_idx=128,
                         topk=16, n_topics=4), 512),
    "hkv2_d3072": (dict(seqs=((700, 2000),), hq=64, hkv=2, d_idx=128, topk=16, n_topics=4), 3072),
    "hkv1_d1024": (dict(seqs=((260, 260),), hq=16, hkv=1, d_idx=128, topk=4, n_topics=4), 1024),
    "hkv8_d256": (dict(seqs=((333, 5000),), hq=64, hkv=8, d_idx=128, topk=16, n_topics=4), 256),
    # 17 heads: eight head pairs and the lone key head per 256 rows
    "hkv16_d512": (dict(seqs=((300, 900),), hq=128, hkv=16, d_idx=128, topk=8, n_topics=4), 512),
    # a decode step: three new tokens, so the second CTA of the pair has no rows at all
    "decode_step_d1024": (dict(seqs=((1, 5000), (1, 300), (1, 77)), hq=64, hkv=4, d_idx=128, topk=16, n_topics=4),
                          1024),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_index_prologue_matches_oracle(msa, name):
    kw, d_model = CASES[name]
    kw = dict(kw)
    cfg = small(name, kw.pop("seqs"), seed=51, **kw)
    x = workloads.generate(cfg, device="cuda")
    _run(msa, x, cfg, d_model)


def test_index_prologue_at_large_positions(msa, parity_report):
    """The last 1024 tokens of a 1,048,576-token sequence and two decode tokens near 1M: the RoPE angles reach
    10^6 radians, where an fp32 product pos * theta would be off by ~0.06 rad."""
    cfg = small("far", ((1024, 1048576), (1, 1048000), (1, 999999)), hq=64, hkv=4, d_idx=128, topk=16,
                n_topics=4, seed=52)
    cu_q = torch.tensor([0, 1024, 1025, 1026], dtype=torch.int32, device="cuda")
    cu_k = torch.tensor([0, 1048576, 1048576 + 1048000, 1048576 + 1048000 + 999999], dtype=torch.int32,
                        device="cuda")
    # only the sizes and sequence layout are needed: the prologue reads hidden states, not Q/K/V
    x = types.SimpleNamespace(cfg=cfg, cu_q=cu_q, cu_k=cu_k, total_q=1026, total_k=int(cu_k[-1]), max_q=1024,
                              max_k=1048576)
    emax, same = _run(msa, x, cfg, 3072, rows=np.arange(0, 1026, 3, dtype=np.int32))[:2]
    parity_report.append(f"index prologue at positions ~1M: max |err| {emax:.3e}, {same:.4f} equal to the "
                         f"rounded oracle value")
