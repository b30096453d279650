"""Pins for the CPU oracle, against facts fixed outside the oracle itself.

Each test ties one step of the oracle to something it does not compute:
  * a hand-worked example (tests/golden/three_block_example.json);
  * a library routine on a special case (torch float64 matmul for the index
    scores, torch scaled_dot_product_attention with a mask built from the
    selection for the Main Branch, Python's sort for the ranking);
  * invariants and closed forms of the method (local block present, fixed
    token budget, q = 0 gives the mean of V and lse = ln n, constant V).
The method: "MiniMax Sparse Attention: let each query pick its own blocks",
section "The mechanism, precisely".  No GPU is needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads.configs import small

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "three_block_example.json")


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64)


# ---------------------------------------------------------------- golden example
def _golden_inputs(d):
    T = len(d["q_idx"])
    q_idx = bf16(d["q_idx"]).reshape(T, 1, 1)
    k_idx = bf16(d["k_idx"]).reshape(T, 1)
    q = bf16([d["q_main_per_head"]] * T).reshape(T, 2, 1)
    k = bf16(d["k_main_bf16"]).reshape(T, 1, 1)
    v = bf16(d["v_main"]).reshape(T, 1, 1)
    cu = np.array([0, T], np.int32)
    return cu, q, k, v, q_idx, k_idx


def test_golden_three_block_example():
    d = json.load(open(GOLDEN))
    cu, q, k, v, q_idx, k_idx = _golden_inputs(d)
    out = oracle.forward(cu, cu, q, k, v, q_idx, k_idx, block=d["block"], topk=d["topk"],
                         scale=d["scale"])
    np.testing.assert_array_equal(out["idx"][:, 0, :], np.array(d["expected_idx"], np.int32))
    pooled = oracle.pooled(cu, cu, q_idx, k_idx, block=d["block"])
    for i, row in enumerate(d["expected_pooled"]):
        np.testing.assert_array_equal(pooled[i, 0, :len(row)], np.array(row, np.float32))
        assert np.all(np.isneginf(pooled[i, 0, len(row):]))
    for i in d["expected_gap_zero_rows"]:
        assert out["gap"][i, 0] == 0.0
    for i_s, exp in d["expected_attention_bf16_inputs"].items():
        i = int(i_s)
        np.testing.assert_allclose(out["o"][i, :, 0], exp["o"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(out["lse"][i], exp["lse"], rtol=0, atol=1e-12)
    # the ideal (exact ln2 / ln3) values agree to within the bf16 rounding of the logits
    ideal = d["expected_attention"]["4"]
    np.testing.assert_allclose(out["o"][4, :, 0], [1.5, 38 / 11], atol=2e-3)
    np.testing.assert_allclose(out["lse"][4], [math.log(6), math.log(11 / 6)], atol=2e-3)
    assert ideal["o"][0] == 1.5


# ---------------------------------------------------------------- index scores
def _varlen_case(seed=0, seqs=((5, 9), (17, 17), (1, 40), (30, 70)), hq=4, hkv=2, d=8, d_idx=8,
                 block=4):
    cfg = small("case", seqs, hq=hq, hkv=hkv, head_dim=d, d_idx=d_idx, block=block, topk=3,
                n_topics=3, seed=seed)
    return cfg, workloads.generate(cfg)


def _torch_pooled(x, block):
    """Index scores with torch float64 matmul, rounded to fp32, max-pooled with torch."""
    cu_q, cu_k = x.cu_q.tolist(), x.cu_k.tolist()
    pos = oracle.query_positions(cu_q, cu_k)
    nbmax = oracle.max_blocks(np.array(cu_k), block)
    out = np.full((x.total_q, x.q_idx.shape[1], nbmax), -np.inf, np.float32)
    for s in range(len(cu_q) - 1):
        kk = f64(x.k_idx[cu_k[s]:cu_k[s + 1]])                 # [kv, d]
        qq = f64(x.q_idx[cu_q[s]:cu_q[s + 1]])                 # [ql, hkv, d]
        sc = torch.einsum("thd,jd->thj", qq, kk).to(torch.float32)
        for t in range(qq.shape[0]):
            p = int(pos[cu_q[s] + t])
            for b in range(p // block + 1):
                seg = sc[t, :, b * block:min((b + 1) * block, p + 1)]
                out[cu_q[s] + t, :, b] = seg.max(dim=1).values.numpy()
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_pooled_matches_torch_matmul(seed):
    cfg, x = _varlen_case(seed)
    got = oracle.pooled(x.cu_q, x.cu_k, x.q_idx, x.k_idx, block=cfg.block)
    ref = _torch_pooled(x, cfg.block)
    np.testing.assert_array_equal(got, ref)


def test_pooled_row_subset_matches_full():
    cfg, x = _varlen_case(3)
    full = oracle.pooled(x.cu_q, x.cu_k, x.q_idx, x.k_idx, block=cfg.block)
    rows = np.array([0, 7, 22, x.total_q - 1, 5], np.int32)
    sub = oracle.pooled(x.cu_q, x.cu_k, x.q_idx, x.k_idx, block=cfg.block, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])


# ---------------------------------------------------------------- selection
def _sorted_reference(row, nb, k):
    """Full sort of the non-local blocks by (score desc, index asc), local forced."""
    local = nb - 1
    order = sorted((b for b in range(nb) if b != local), key=lambda b: (-float(row[b]), b))
    chosen = order[:max(0, min(k - 1, nb - 1))]
    sel = sorted(chosen + ([local] if k > 0 else []))
    return sel + [-1] * (k - len(sel))


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_full_sort_with_ties(seed):
    rng = np.random.default_rng(seed)
    for _ in range(300):
        nb = int(rng.integers(1, 70))
        k = int(rng.integers(1, 20))
        # few distinct values -> many exact ties; include +0 and -0
        vals = rng.choice(np.array([-2.5, -0.0, 0.0, 1.0, 3.25, 3.25, 7.0], np.float32), size=nb)
        if rng.random() < 0.5:
            vals = rng.standard_normal(nb).astype(np.float32)
        sel, gap = oracle.select(vals, nb, k)
        assert sel.tolist() == _sorted_reference(vals, nb, k)


def test_select_dominance_property():
    """Every selected non-local block beats every unselected one under (score desc, index asc)."""
    rng = np.random.default_rng(7)
    for _ in range(500):
        nb = int(rng.integers(2, 40))
        k = int(rng.integers(2, 10))
        vals = rng.integers(-3, 4, size=nb).astype(np.float32)
        sel, _ = oracle.select(vals, nb, k)
        chosen = set(int(b) for b in sel if b >= 0) - {nb - 1}
        rest = set(range(nb - 1)) - chosen
        for a in chosen:
            for b in rest:
                assert vals[a] > vals[b] or (vals[a] == vals[b] and a < b)


def test_select_gap_definition():
    row = np.array([5.0, 4.0, 4.0 * (1 + 1e-7), 1.0, 9.0], np.float32)  # local = 4
    sel, gap = oracle.select(row, 5, 3)                                 # picks 0 and 2
    assert sel.tolist() == [0, 2, 4]
    a, c = np.float32(4.0 * (1 + 1e-7)), np.float32(4.0)
    assert gap == pytest.approx(abs(float(a) - float(c)) / float(a), rel=1e-12)
    _, gap_all = oracle.select(row, 5, 16)
    assert gap_all == math.inf
    _, gap_one = oracle.select(row, 5, 1)
    assert gap_one == math.inf


# ---------------------------------------------------------------- main branch
def _sdpa_masked(x, idx, block, scale):
    """Main Branch via torch SDPA (float64) with a boolean mask built from the selection."""
    cu_q, cu_k = x.cu_q.tolist(), x.cu_k.tolist()
    hq, hkv = x.q.shape[1], x.k.shape[1]
    G = hq // hkv
    pos = oracle.query_positions(cu_q, cu_k)
    o = np.zeros((x.total_q, hq, x.q.shape[2]))
    lse = np.zeros((x.total_q, hq))
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if q1 == q0:
            continue
        kv = k1 - k0
        for h in range(hq):
            g = h // G
            mask = torch.zeros(q1 - q0, kv, dtype=torch.bool)
            for t in range(q1 - q0):
                p = int(pos[q0 + t])
                for b in idx[q0 + t, g]:
                    if b >= 0:
                        mask[t, b * block:min((b + 1) * block, p + 1)] = True
            qh = f64(x.q[q0:q1, h])[None, None]
            kh = f64(x.k[k0:k1, g])[None, None]
            vh = f64(x.v[k0:k1, g])[None, None]
            oh = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask[None, None],
                                                                   scale=scale)
            o[q0:q1, h] = oh[0, 0].numpy()
            logits = (qh[0, 0] @ kh[0, 0].T) * scale
            lse[q0:q1, h] = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=1).numpy()
    return o, lse


def _random_selection(x, block, k, rng):
    pos = oracle.query_positions(x.cu_q, x.cu_k)
    hkv = x.k.shape[1]
    idx = np.full((x.total_q, hkv, k), -1, np.int32)
    for i in range(x.total_q):
        nb = int(pos[i]) // block + 1
        for g in range(hkv):
            others = rng.permutation(nb - 1)[:min(k - 1, nb - 1)]
            sel = sorted(list(others) + [nb - 1])
            idx[i, g, :len(sel)] = sel
    return idx


@pytest.mark.parametrize("seed", [0, 1])
def test_attention_matches_masked_sdpa(seed):
    cfg, x = _varlen_case(seed, hq=6, hkv=2, d=16)
    idx = _random_selection(x, cfg.block, 3, np.random.default_rng(seed))
    scale = 0.37
    o, lse = oracle.attention(x.cu_q, x.cu_k, x.q, x.k, x.v, idx, block=cfg.block, scale=scale)
    o_ref, lse_ref = _sdpa_masked(x, idx, cfg.block, scale)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_forward_equals_dense_causal_when_k_covers_all_blocks():
    """k >= number of causal blocks -> every block is kept -> dense causal attention."""
    cfg, x = _varlen_case(5, hq=4, hkv=2, d=16, seqs=((9, 9), (3, 21), (12, 33)))
    k = 16  # > 33/4 + 1 blocks
    out = oracle.forward(x.cu_q, x.cu_k, x.q, x.k, x.v, x.q_idx, x.k_idx, block=cfg.block, topk=k)
    cu_q, cu_k = x.cu_q.tolist(), x.cu_k.tolist()
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        ql, kl = q1 - q0, k1 - k0
        # bottom-right causal mask: query t sees keys j <= kl - ql + t
        mask = torch.ones(ql, kl, dtype=torch.bool).tril(diagonal=kl - ql)
        for h in range(4):
            g = h // 2
            ref = torch.nn.functional.scaled_dot_product_attention(
                f64(x.q[q0:q1, h])[None, None], f64(x.k[k0:k1, g])[None, None],
                f64(x.v[k0:k1, g])[None, None], attn_mask=mask[None, None])
            np.testing.assert_allclose(out["o"][q0:q1, h], ref[0, 0].numpy(), atol=1e-12, rtol=0)


# ---------------------------------------------------------------- invariants & closed forms
def test_invariants_on_tiny_workload():
    cfg = workloads.get("tiny")
    x = workloads.generate(cfg)
    rows = np.arange(0, x.total_q, 37, dtype=np.int32)
    out = oracle.forward(x.cu_q, x.cu_k, x.q, x.k, x.v, x.q_idx, x.k_idx, block=cfg.block,
                         topk=cfg.topk, rows=rows)
    pos = oracle.query_positions(x.cu_q, x.cu_k)[rows]
    for r, p in enumerate(pos):
        nb = int(p) // cfg.block + 1
        for g in range(cfg.hkv):
            sel = out["idx"][r, g]
            valid = sel[sel >= 0]
            assert (nb - 1) in valid                                  # local block kept
            assert len(valid) == min(cfg.topk, nb)                    # fixed budget
            assert np.all(np.diff(valid) > 0)                         # ascending, no repeats
            assert np.all(sel[len(valid):] == -1)                     # -1 only at the tail
            assert valid.max() <= nb - 1                              # nothing in the future


def test_token_budget_and_closed_forms():
    """q = 0 -> uniform weights -> lse = ln n_tok and o = mean of V over the kept tokens;
    with nb > k the kept token count is (k-1)*block + (pos mod block) + 1."""
    cfg, x = _varlen_case(11, seqs=((6, 40), (4, 23)), hq=4, hkv=2, d=8, block=4)
    k = 3
    x.q.zero_()
    out = oracle.forward(x.cu_q, x.cu_k, x.q, x.k, x.v, x.q_idx, x.k_idx, block=cfg.block, topk=k)
    pos = oracle.query_positions(x.cu_q, x.cu_k)
    cu_k = x.cu_k.tolist()
    cu_q = x.cu_q.tolist()
    for i in range(x.total_q):
        s = 0 if i < cu_q[1] else 1
        nb = int(pos[i]) // cfg.block + 1
        for h in range(4):
            g = h // 2
            toks = [j for b in out["idx"][i, g] if b >= 0
                    for j in range(b * cfg.block, min((b + 1) * cfg.block, int(pos[i]) + 1))]
            if nb > k:
                assert len(toks) == (k - 1) * cfg.block + int(pos[i]) % cfg.block + 1
            assert out["lse"][i, h] == pytest.approx(math.log(len(toks)), abs=1e-12)
            vmean = f64(x.v[[cu_k[s] + j for j in toks], g]).mean(0).numpy()
            np.testing.assert_allclose(out["o"][i, h], vmean, atol=1e-12)


def test_constant_values_give_constant_output():
    cfg, x = _varlen_case(12)
    x.v.fill_(1.5)
    out = oracle.forward(x.cu_q, x.cu_k, x.q, x.k, x.v, x.q_idx, x.k_idx, block=cfg.block, topk=2)
    np.testing.assert_allclose(out["o"], 1.5, atol=1e-12)


def test_rejects_bad_sequence_lengths():
    cfg, x = _varlen_case(0)
    bad_k = x.cu_k.clone()
    bad_k[1] = 2  # first sequence: 5 queries but 2 keys
    with pytest.raises(ValueError):
        oracle.pooled(x.cu_q, bad_k, x.q_idx, x.k_idx, block=cfg.block)
