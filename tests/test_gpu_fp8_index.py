"""GPU parity of the fp8 index path (Q_idx and K_idx as E4M3 codes with one
scale per query row and group and one per key block) against the oracle's
Index Branch over the same codes.

The codes always come from the CPU (the oracle's quantizer on small cases, the
tests' torch-based quantizer, pinned to it bit for bit, at full size) and are
uploaded for the GPU, so the oracle never reads anything the CUDA path made.
The GPU quantizer is compared with the oracle's quantizer on its own.
Selections are bit-exact except near-ties (oracle gap below 1e-5 relative),
which are counted; the Main Branch over fp8 K/V is compared at the fp8
tolerances of test_gpu_fp8.

Sources: the atlas record of the report, provenance of section 4.2 (the
kernels handle fp8 as well; the format is a reading, stated in msa.h);
"MiniMax Sparse Attention: let each query pick its own blocks", section "The
mechanism, precisely".
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads.configs import small

from parity import assert_attention_close, compare_indices, problem_for, quantize_index_cpu, to_np

pytestmark = pytest.mark.gpu

PREFILL = {
    # several index tiles, ragged tails, chunked sequences, an empty one; fused top-k (k <= 16)
    "varlen_g16": dict(seqs=((300, 300), (1000, 1777), (1, 129), (129, 900), (0, 77), (640, 640)),
                       hq=64, hkv=4, topk=16, n_topics=16),
    "g32_k8": dict(seqs=((600, 600), (333, 1400)), hq=64, hkv=2, topk=8, n_topics=8),
    # k > 16: pooled scores in the workspace, then the separate top-k
    "k32": dict(seqs=((900, 2600),), hq=64, hkv=4, topk=32, n_topics=8),
    "g128_hkv1": dict(seqs=((400, 400), (130, 700)), hq=128, hkv=1, topk=4, n_topics=4),
    "k64": dict(seqs=((700, 3000), (64, 64)), hq=64, hkv=4, topk=64, n_topics=8),
    "k1": dict(seqs=((300, 1000),), hq=64, hkv=4, topk=1, n_topics=8),
}
# a decode batch whose caches hold 1, 2, 128, 129, 257 and 5,000 keys (its lengths far apart, so the scan
# keeps its few large work units instead of the small ones of the even batches below)
MIXED_DECODE = ((1, 1), (1, 2), (1, 128), (1, 129), (1, 257), (1, 5000))
# decode batches: (sequences, context, topk, hq, hkv)
DECODE = [(12, 9000, 16, 64, 4), (3, 40000, 16, 64, 8), (5, 700, 64, 64, 4), (2, 200, 16, 32, 1),
          (4, 20000, 32, 32, 4)]


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_05_gb300 as m
    torch.cuda.set_device(0)
    return m


def _prefill(name, seed=3):
    kw = dict(PREFILL[name])
    return small(name, kw.pop("seqs"), d_idx=128, seed=seed, **kw)


def _decode(n, ctx, topk, hq, hkv, seed):
    rng = np.random.default_rng(seed)
    kv = [int(v) for v in rng.integers(max(1, ctx // 2), ctx + 1, size=n)]
    return small(f"decode_{n}x{ctx}", [(1, v) for v in kv], hq=hq, hkv=hkv, d_idx=128, topk=topk,
                 n_topics=8, seed=seed)


def _oracle_codes(x, cfg):
    return oracle.quantize_index_fp8(x.cu_q, x.cu_k, x.q_idx, x.k_idx, cfg.block)


def _cuda(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


def _cases():
    return [("prefill", name) for name in sorted(PREFILL)] + [("decode", i) for i in range(len(DECODE))]


def _make(kind, key):
    if kind == "mixed":
        cfg = small("fp8_dec_mixed", MIXED_DECODE, hq=64, hkv=4, d_idx=128, topk=16, n_topics=8, seed=78)
    else:
        cfg = _prefill(key) if kind == "prefill" else _decode(*DECODE[key], seed=60 + key)
    return cfg, workloads.generate(cfg, device="cuda")


@pytest.mark.parametrize("kind,key", _cases())
def test_quantize_index_matches_oracle(msa, kind, key):
    cfg, x = _make(kind, key)
    prob = problem_for(msa, x)
    q8, qs, k8, ks = msa.msa_quantize_index_fp8(prob, x.q_idx, x.k_idx)
    torch.cuda.synchronize()
    rq8, rqs, rk8, rks = _oracle_codes(x, cfg)
    assert np.array_equal(to_np(q8), rq8) and np.array_equal(to_np(qs), rqs)
    assert np.array_equal(to_np(k8), rk8) and np.array_equal(to_np(ks)[:rks.size], rks)


def test_quantize_index_one_side_only(msa):
    cfg, x = _make("prefill", "g32_k8")
    prob = problem_for(msa, x)
    rq8, rqs, rk8, rks = _oracle_codes(x, cfg)
    q8, qs, k8, ks = msa.msa_quantize_index_fp8(prob, q_idx=x.q_idx)
    assert k8 is None and ks is None
    assert np.array_equal(to_np(q8), rq8) and np.array_equal(to_np(qs), rqs)
    k8 = torch.full(x.k_idx.shape, 0x55, dtype=torch.uint8, device="cuda")
    _, _, k8, ks = msa.msa_quantize_index_fp8(prob, k_idx=x.k_idx, k_idx8=k8)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(k8), rk8) and np.array_equal(to_np(ks)[:rks.size], rks)


@pytest.mark.parametrize("name", ["varlen_g16", "g128_hkv1"])
def test_index_pool_fp8_matches_oracle(msa, name):
    cfg, x = _make("prefill", name)
    prob = problem_for(msa, x)
    rq8, rqs, rk8, rks = _oracle_codes(x, cfg)
    pooled = msa.msa_index_pool_fp8(prob, *_cuda(rq8, rqs, rk8, rks))
    torch.cuda.synchronize()
    got = to_np(pooled).reshape(x.total_q, cfg.hkv, -1)
    ref = oracle.pooled_fp8(x.cu_q, x.cu_k, rq8, rqs, rk8, rks, cfg.block, nb_stride=got.shape[2])
    valid = np.isfinite(ref)
    assert np.all(np.isnan(got[~valid])), "entries past the causal end must be left untouched"
    # the code products are exact; the sums differ in order (fp32 on the tensor cores, double in the oracle)
    np.testing.assert_allclose(got[valid], ref[valid], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("kind,key", _cases())
def test_index_topk_fp8_matches_oracle(msa, kind, key, parity_report):
    cfg, x = _make(kind, key)
    prob = problem_for(msa, x)
    rq8, rqs, rk8, rks = _oracle_codes(x, cfg)
    ws = msa.workspace(prob, msa.Op.INDEX_TOPK)
    idx = to_np(msa.msa_index_topk_fp8(prob, *_cuda(rq8, rqs, rk8, rks), ws=ws))
    assert msa.msa_read_device_status(ws) == 0
    ref = oracle.index_fp8(x.cu_q, x.cu_k, rq8, rqs, rk8, rks, cfg.block, cfg.topk)
    tie, mism = compare_indices(idx, ref)
    excused = int(((idx != ref["idx"]).any(axis=-1) & tie).sum())
    parity_report.append(f"fp8 index {cfg.name}: {tie.size} rows x groups, {mism} mismatches, "
                         f"{int(tie.sum())} near-ties, {excused} of them selected differently")
    assert mism == 0, f"{mism} rows select differently from the oracle"
    # E4M3 codes sit on a coarse grid, so equal pooled scores are more common than with bf16 inputs; the
    # near-tie count is a property of the inputs, and the rows it excuses (selected differently) must stay
    # under 0.1 % (or be a single row of a small case)
    assert excused <= 1 or excused / tie.size < 1e-3, f"{excused} near-tie rows differ"


@pytest.mark.parametrize("kind,key", [("prefill", "varlen_g16"), ("prefill", "g32_k8"), ("decode", 0),
                                      ("decode", 1), ("mixed", 0)])
def test_forward_fp8_index_end_to_end(msa, kind, key):
    """All-fp8 forward: selection against the oracle's Index Branch over the codes, O and LSE against the
    oracle's fp8 Main Branch on the oracle's selection (near-tie rows exempt)."""
    cfg, x = _make(kind, key)
    prob = problem_for(msa, x)
    rq8, rqs, rk8, rks = _oracle_codes(x, cfg)
    k8, ksc = oracle.quantize_fp8(x.cu_k, x.k, cfg.block)
    v8, vsc = oracle.quantize_fp8(x.cu_k, x.v, cfg.block)
    ws = msa.workspace(prob, msa.Op.FORWARD_FP8)
    idx, o, lse = msa.msa_forward_fp8_index(prob, x.q, *_cuda(k8, v8, ksc, vsc, rq8, rqs, rk8, rks), ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    ref = oracle.index_fp8(x.cu_q, x.cu_k, rq8, rqs, rk8, rks, cfg.block, cfg.topk)
    tie, mism = compare_indices(to_np(idx), ref)
    assert mism == 0
    ro, rlse = oracle.attention_fp8(x.cu_q, x.cu_k, x.q, k8, v8, ksc, vsc, ref["idx"], cfg.block)
    if x.total_q:
        assert_attention_close(to_np(o), to_np(lse), {"o": ro, "lse": rlse}, cfg.hq // cfg.hkv, exempt=tie,
                               what=cfg.name)


# Full size, in the launch configuration of the benchmark's fp8 record: every row of the decode batches,
# 4096 position-stratified rows of the prefills.
FULL_ROWS = {"decode_1m": None, "decode_128k": None, "prefill_32k": 4096, "prefill_128k": 4096, "varlen": 4096,
             "chunked_1m": 4096}


@pytest.mark.parametrize("name", sorted(FULL_ROWS))
def test_full_size_fp8_index_selection(msa, name, parity_report):
    cfg = workloads.get(name)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    q8, qs, k8, ks = quantize_index_cpu(x, cfg.block)
    ws = msa.workspace(prob, msa.Op.INDEX_TOPK)
    idx = msa.msa_index_topk_fp8(prob, *_cuda(q8, qs, k8, ks), ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    n = FULL_ROWS[name]
    rows = None
    if n is not None and n < x.total_q:
        rng = np.random.default_rng(23)
        edges = np.linspace(0, x.total_q, n + 1).astype(np.int64)
        rows = np.array([rng.integers(edges[j], max(edges[j] + 1, edges[j + 1])) for j in range(n)], np.int32)
    ref = oracle.index_fp8(x.cu_q, x.cu_k, q8, qs, k8, ks, cfg.block, cfg.topk, rows=rows)
    got = to_np(idx) if rows is None else to_np(idx[torch.from_numpy(rows).long().cuda()])
    tie, mism = compare_indices(got, ref)
    excused = int(((got != ref["idx"]).any(axis=-1) & tie).sum())
    parity_report.append(f"fp8 index selection {name}: {tie.size} rows x groups checked, {mism} mismatches, "
                         f"{int(tie.sum())} near-ties, {excused} of them selected differently")
    assert mism == 0, f"{mism} rows select differently from the oracle"
    assert excused / tie.size < 1e-3


@pytest.mark.parametrize("n,ctx,seed", [(6, 9000, 71), (3, 40000, 72), (2, 200, 73)])
def test_forward_decode_paged_fp8_index(msa, n, ctx, seed):
    """Paged fp8 caches with the index keys in fp8 too (one scale per page) give the packed all-fp8 path's
    results bit for bit, and quantizing the bf16 index-key page pool as one sequence of num_pages * 128 keys
    yields exactly those codes and per-page scales."""
    cfg = workloads.configs.Workload("dec8pi", None, seed=seed, decode_batch=n, decode_ctx=ctx, topk=16,
                                     n_topics=16, hq=64, hkv=4, d_idx=128)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    k8, v8, ks, vs = msa.msa_quantize_kv_fp8(prob, x.k, x.v)
    q8, qs, ki8, kis = msa.msa_quantize_index_fp8(prob, x.q_idx, x.k_idx)
    cu_k = x.cu_k.cpu().numpy()
    nbs = [int(cu_k[s + 1] - cu_k[s] + 127) // 128 for s in range(n)]
    n_pages = sum(nbs) + 3
    perm = np.random.default_rng(seed).permutation(n_pages)
    bt = np.full((n, max(nbs) + 2), -7, np.int32)
    rows = (n_pages * 128,) + tuple(x.k.shape[1:])
    k8c = torch.zeros(rows, dtype=torch.uint8, device="cuda")
    v8c = torch.zeros_like(k8c)
    ki8c = torch.zeros((n_pages * 128, cfg.d_idx), dtype=torch.uint8, device="cuda")
    ki_c = torch.zeros((n_pages * 128, cfg.d_idx), dtype=torch.bfloat16, device="cuda")
    ksc = torch.ones((n_pages, cfg.hkv), dtype=torch.float32, device="cuda")
    vsc = torch.ones_like(ksc)
    kisc = torch.ones(n_pages, dtype=torch.float32, device="cuda")
    at = blk = 0
    used = []
    for s in range(n):
        for b in range(nbs[s]):
            pg = int(perm[at])
            at += 1
            bt[s, b] = pg
            lo, hi = int(cu_k[s]) + 128 * b, min(int(cu_k[s]) + 128 * (b + 1), int(cu_k[s + 1]))
            dst = slice(pg * 128, pg * 128 + hi - lo)
            k8c[dst], v8c[dst], ki8c[dst], ki_c[dst] = k8[lo:hi], v8[lo:hi], ki8[lo:hi], x.k_idx[lo:hi]
            ksc[pg], vsc[pg], kisc[pg] = ks[blk], vs[blk], kis[blk]
            used.append((pg, hi - lo))
            blk += 1
    bt = torch.from_numpy(bt).cuda()
    ws = msa.workspace(prob, msa.Op.FORWARD_FP8)
    idx, o, lse = msa.msa_forward_decode_paged_fp8_index(prob, x.q, k8c, v8c, ksc, vsc, q8, qs, ki8c, kisc, bt,
                                                         ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws) == 0
    idx_r, o_r, lse_r = msa.msa_forward_fp8_index(prob, x.q, k8, v8, ks, vs, q8, qs, ki8, kis)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_r) and torch.equal(o, o_r) and torch.equal(lse, lse_r)
    pool = msa.problem_from_seqlens([1], [n_pages * 128], hq=cfg.hq, hkv=cfg.hkv, d_idx=cfg.d_idx, topk=cfg.topk)
    _, _, ki8q, kisq = msa.msa_quantize_index_fp8(pool, k_idx=ki_c)
    torch.cuda.synchronize()
    for pg, nrow in used:
        r = slice(pg * 128, pg * 128 + nrow)
        assert torch.equal(ki8q[r], ki8c[r]) and torch.equal(kisq[pg], kisc[pg]), pg
