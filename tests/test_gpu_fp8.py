"""GPU parity of the fp8 K/V path (E4M3 codes, one scale per key block and KV
head; the atlas record of the report: the kernels handle fp8 as well, format
read as stated in include/msa.h) against the CPU oracle:

  * quantization: codes and scales bit-exact against oracle.quantize_fp8 (an
    integer result decided by fp32 division on both sides);
  * Main Branch, prefill and decode, on the oracle's indices: O and LSE within
    the parity tolerance of oracle.attention_fp8 (the Main Branch over the
    dequantized values), every row;
  * end to end (msa_forward_fp8): indices as the bf16 path (the Index Branch is
    bf16), O and LSE against oracle.attention_fp8;
  * against the bf16 oracle the results differ by the quantization only:
    O max-abs below 0.3 and mean-abs below 1e-2, LSE max-abs below 0.15 (a row
    attending to one token returns one V row, whose elements carry up to 2^-4
    relative rounding: 0.28 for |v| = 4.5; averaging over tokens shrinks it).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads.configs import small

from parity import assert_attention_close, compare_indices, problem_for, to_np

pytestmark = pytest.mark.gpu

FP8_VS_BF16 = dict(o_max=0.3, o_mean=1e-2, lse_max=0.15)


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_05_gb300 as m
    torch.cuda.set_device(0)
    return m


def _quantized(msa, x, prob, cfg):
    k8, v8, ks, vs = msa.msa_quantize_kv_fp8(prob, x.k, x.v)
    torch.cuda.synchronize()
    nkb = oracle.key_blocks(x.cu_k, cfg.block)
    return k8, v8, ks, vs, nkb


PREFILL = {
    "varlen": dict(seqs=((300, 300), (1000, 1777), (1, 129), (129, 900), (0, 77), (640, 640)),
                   hq=64, hkv=4, d_idx=128, topk=16, n_topics=16),
    "g32_k24": dict(seqs=((600, 2600),), hq=64, hkv=2, d_idx=128, topk=24, n_topics=8),
    "g8": dict(seqs=((500, 500), (200, 1300)), hq=32, hkv=4, d_idx=64, topk=8, n_topics=8),
}


@pytest.mark.parametrize("name", sorted(PREFILL))
def test_quantize_matches_oracle(msa, name):
    kw = dict(PREFILL[name])
    cfg = small(name, kw.pop("seqs"), seed=41, **kw)
    x = workloads.generate(cfg, device="cuda")
    k = x.k.clone()
    k[:128, 0] = 0.0                     # an all-zero (block, head): scale 1, codes 0
    k[200, 1, 5] = 3.0e4                 # a large value: its block's scale follows it
    prob = problem_for(msa, x)
    k8, v8, ks, vs = msa.msa_quantize_kv_fp8(prob, k, x.v)
    torch.cuda.synchronize()
    rk8, rks = oracle.quantize_fp8(x.cu_k, k, block=cfg.block)
    rv8, rvs = oracle.quantize_fp8(x.cu_k, x.v, block=cfg.block)
    nkb = rks.shape[0]
    assert np.array_equal(k8.cpu().numpy(), rk8) and np.array_equal(v8.cpu().numpy(), rv8)
    assert np.array_equal(ks[:nkb].cpu().numpy().view(np.uint32), rks.view(np.uint32))
    assert np.array_equal(vs[:nkb].cpu().numpy().view(np.uint32), rvs.view(np.uint32))


@pytest.mark.parametrize("name", sorted(PREFILL))
def test_prefill_fp8_on_oracle_indices(msa, name):
    kw = dict(PREFILL[name])
    cfg = small(name, kw.pop("seqs"), seed=42, **kw)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    k8, v8, ks, vs, nkb = _quantized(msa, x, prob, cfg)
    ref = oracle.index(x.cu_q, x.cu_k, x.q_idx, x.k_idx, block=cfg.block, topk=cfg.topk)
    idx = torch.from_numpy(ref["idx"]).cuda()
    ws = msa.workspace(prob, msa.Op.SPARSE_ATTN_PREFILL_FP8)
    o, lse = msa.msa_sparse_attn_prefill_fp8(prob, x.q, k8, v8, ks, vs, idx, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    o8, l8 = oracle.attention_fp8(x.cu_q, x.cu_k, x.q, k8, v8, ks[:nkb], vs[:nkb], ref["idx"], block=cfg.block)
    G = cfg.hq // cfg.hkv
    assert_attention_close(to_np(o), to_np(lse), {"o": o8, "lse": l8}, G, what=f"{name} fp8")
    # the same rows against the bf16 oracle: the quantization error only
    o16, l16 = oracle.attention(x.cu_q, x.cu_k, x.q, x.k, x.v, ref["idx"], block=cfg.block)
    e = np.abs(to_np(o).astype(np.float64) - o16)
    assert e.max() < FP8_VS_BF16["o_max"] and e.mean() < FP8_VS_BF16["o_mean"], (e.max(), e.mean())
    assert np.abs(to_np(lse) - l16).max() < FP8_VS_BF16["lse_max"]


DECODE = [(8, 3000, 16, 64, 4), (16, 20000, 16, 64, 4), (5, 7000, 32, 128, 4), (6, 5000, 16, 32, 4),
          (3, 200, 16, 64, 4)]


@pytest.mark.parametrize("n,ctx,topk,hq,hkv", DECODE)
def test_decode_fp8(msa, n, ctx, topk, hq, hkv):
    cfg = workloads.configs.Workload("dec8", None, seed=n * 7 + ctx, decode_batch=n, decode_ctx=ctx, topk=topk,
                                     n_topics=16, hq=hq, hkv=hkv)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    k8, v8, ks, vs, nkb = _quantized(msa, x, prob, cfg)
    ref = oracle.index(x.cu_q, x.cu_k, x.q_idx, x.k_idx, block=cfg.block, topk=cfg.topk)
    o8, l8 = oracle.attention_fp8(x.cu_q, x.cu_k, x.q, k8, v8, ks[:nkb], vs[:nkb], ref["idx"], block=cfg.block)
    G = hq // hkv
    # the decode Main Branch on the oracle's indices
    ws = msa.workspace(prob, msa.Op.SPARSE_ATTN_DECODE_FP8)
    o, lse = msa.msa_sparse_attn_decode_fp8(prob, x.q, k8, v8, ks, vs, torch.from_numpy(ref["idx"]).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    assert_attention_close(to_np(o), to_np(lse), {"o": o8, "lse": l8}, G, what="decode fp8, oracle indices")
    # end to end: the Index Branch is the bf16 one
    ws = msa.workspace(prob, msa.Op.FORWARD_FP8)
    idx, o2, lse2 = msa.msa_forward_fp8(prob, x.q, k8, v8, ks, vs, x.q_idx, x.k_idx, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    tie, mism = compare_indices(to_np(idx), ref)
    assert mism == 0
    assert_attention_close(to_np(o2), to_np(lse2), {"o": o8, "lse": l8}, G, exempt=tie, what="decode fp8")


def test_forward_fp8_prefill_end_to_end(msa):
    kw = dict(PREFILL["varlen"])
    cfg = small("fwd8", kw.pop("seqs"), seed=43, **kw)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    k8, v8, ks, vs, nkb = _quantized(msa, x, prob, cfg)
    ws = msa.workspace(prob, msa.Op.FORWARD_FP8)
    idx, o, lse = msa.msa_forward_fp8(prob, x.q, k8, v8, ks, vs, x.q_idx, x.k_idx, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    ref = oracle.index(x.cu_q, x.cu_k, x.q_idx, x.k_idx, block=cfg.block, topk=cfg.topk)
    tie, mism = compare_indices(to_np(idx), ref)
    assert mism == 0
    o8, l8 = oracle.attention_fp8(x.cu_q, x.cu_k, x.q, k8, v8, ks[:nkb], vs[:nkb], ref["idx"], block=cfg.block)
    assert_attention_close(to_np(o), to_np(lse), {"o": o8, "lse": l8}, cfg.hq // cfg.hkv, exempt=tie,
                           what="forward fp8")


# ------------------------------------------------------------------ paged fp8 decode caches
@pytest.mark.parametrize("n,ctx,seed", [(6, 9000, 51), (3, 40000, 52), (2, 200, 53)])
def test_forward_decode_paged_fp8(msa, n, ctx, seed):
    """Paged fp8 caches (E4M3 codes in pages of 128 rows, one scale row per page) give the packed fp8 path's
    results bit for bit, and quantizing the bf16 page pool as one sequence of num_pages * 128 keys yields
    exactly those codes and per-page scales."""
    cfg = workloads.configs.Workload("dec8p", None, seed=seed, decode_batch=n, decode_ctx=ctx, topk=16,
                                     n_topics=16, hq=64, hkv=4)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    k8, v8, ks, vs, nkb = _quantized(msa, x, prob, cfg)
    cu_k = x.cu_k.cpu().numpy()
    nbs = [int(cu_k[s + 1] - cu_k[s] + 127) // 128 for s in range(n)]
    n_pages = sum(nbs) + 3
    perm = np.random.default_rng(seed).permutation(n_pages)
    bt = np.full((n, max(nbs) + 2), -7, np.int32)
    rows = (n_pages * 128,) + tuple(x.k.shape[1:])
    k8c = torch.zeros(rows, dtype=torch.uint8, device="cuda")
    v8c = torch.zeros_like(k8c)
    k_c = torch.zeros(rows, dtype=torch.bfloat16, device="cuda")
    v_c = torch.zeros_like(k_c)
    ki_c = torch.zeros((n_pages * 128,) + tuple(x.k_idx.shape[1:]), dtype=x.k_idx.dtype, device="cuda")
    ksc = torch.ones((n_pages, cfg.hkv), dtype=torch.float32, device="cuda")
    vsc = torch.ones_like(ksc)
    at = blk = 0
    used = []
    for s in range(n):
        for b in range(nbs[s]):
            pg = int(perm[at])
            at += 1
            bt[s, b] = pg
            lo, hi = int(cu_k[s]) + 128 * b, min(int(cu_k[s]) + 128 * (b + 1), int(cu_k[s + 1]))
            dst = slice(pg * 128, pg * 128 + hi - lo)
            k8c[dst], v8c[dst], k_c[dst], v_c[dst], ki_c[dst] = k8[lo:hi], v8[lo:hi], x.k[lo:hi], x.v[lo:hi], \
                x.k_idx[lo:hi]
            ksc[pg], vsc[pg] = ks[blk], vs[blk]
            used.append((pg, hi - lo))
            blk += 1
    bt = torch.from_numpy(bt).cuda()
    ws = msa.workspace(prob, msa.Op.FORWARD_FP8)
    idx, o, lse = msa.msa_forward_decode_paged_fp8(prob, x.q, k8c, v8c, ksc, vsc, x.q_idx, ki_c, bt, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    idx_r, o_r, lse_r = msa.msa_forward_fp8(prob, x.q, k8, v8, ks, vs, x.q_idx, x.k_idx)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_r) and torch.equal(o, o_r) and torch.equal(lse, lse_r)
    # the recommended quantization of a page pool: one sequence of num_pages * 128 keys, a key block per page
    pool = msa.problem_from_seqlens([1], [n_pages * 128], hq=cfg.hq, hkv=cfg.hkv, d_idx=cfg.d_idx, topk=cfg.topk)
    k8q, v8q, ksq, vsq = msa.msa_quantize_kv_fp8(pool, k_c, v_c)
    torch.cuda.synchronize()
    for pg, nrow in used:
        r = slice(pg * 128, pg * 128 + nrow)
        assert torch.equal(k8q[r], k8c[r]) and torch.equal(v8q[r], v8c[r]), pg
        assert torch.equal(ksq[pg], ksc[pg]) and torch.equal(vsq[pg], vsc[pg]), pg
