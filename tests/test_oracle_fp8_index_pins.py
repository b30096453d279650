"""Pins for the oracle's fp8 index path (Q_idx and K_idx as E4M3 codes: K_idx
with one scale per key block of a sequence, Q_idx with one per query row and
group), against facts fixed outside the oracle:
  * the bf16 Index Branch of the oracle (pinned on its own in test_oracle_pins)
    must give bit-identical pooled scores when the fp8 inputs, decoded by torch's
    float8_e4m3fn dtype and multiplied by power-of-two scales, are exact bf16
    values;
  * a brute-force numpy evaluation of the definition (float64 einsum over the
    decoded values, rounded to fp32, causal block max) on small inputs with the
    quantizer's own (non-power-of-two) scales;
  * properties of the quantizer over the index rows (the row or block maximum
    maps to +-448).
Source: the atlas record of the report, provenance of section 4.2 (the kernels
handle fp8 as well, no format given); "MiniMax Sparse Attention: let each query
pick its own blocks", section "The mechanism, precisely" (the index scores,
max-pool and top-k).  No GPU is needed.
"""
import numpy as np
import torch

import oracle
import workloads
from parity import quantize_index_cpu
from workloads.configs import small

BLOCK = 32  # small blocks: many key blocks, so many scale rows per sequence


def _case(seed=0, seqs=((5, 300), (17, 17), (40, 260)), hkv=2, d_idx=16):
    cfg = small("fp8idx", seqs, hq=8, hkv=hkv, head_dim=16, d_idx=d_idx, block=BLOCK, topk=4, n_topics=3,
                seed=seed)
    return cfg, workloads.generate(cfg)


def _decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 values of codes by torch's float8_e4m3fn (a library implementation of the format)."""
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _random_codes(rng, shape):
    """Finite E4M3 codes of both signs (the NaN codes 0x7F and 0xFF excluded)."""
    return (rng.integers(0, 0x7F, size=shape) | (rng.integers(0, 2, size=shape) << 7)).astype(np.uint8)


def _block_rows(cu_k, block):
    """Scale row of every key: key blocks of the sequences before it plus its block in the sequence."""
    cu = np.asarray(cu_k, np.int64)
    rows = np.empty(int(cu[-1]), np.int64)
    r0 = 0
    for s in range(len(cu) - 1):
        n = int(cu[s + 1] - cu[s])
        rows[cu[s]:cu[s + 1]] = r0 + np.arange(n) // block
        r0 += -(-n // block)
    return rows


def test_pooled_fp8_equals_bf16_pooled_on_the_fp8_grid():
    cfg, x = _case()
    rng = np.random.default_rng(1)
    total_q, total_k = x.total_q, x.total_k
    q8 = _random_codes(rng, (total_q, cfg.hkv, cfg.d_idx))
    k8 = _random_codes(rng, (total_k, cfg.d_idx))
    nkb = oracle.key_blocks(x.cu_k, BLOCK)
    k_scale = (2.0 ** -(np.arange(nkb) % 5)).astype(np.float32)                     # differs per key block
    q_scale = (2.0 ** ((np.arange(total_q * cfg.hkv) % 4) - 2)).reshape(total_q, cfg.hkv).astype(np.float32)
    kv = _decode(k8) * k_scale[_block_rows(x.cu_k, BLOCK)][:, None]
    qv = _decode(q8) * q_scale[:, :, None]
    kb, qb = torch.from_numpy(kv).to(torch.bfloat16), torch.from_numpy(qv).to(torch.bfloat16)
    assert np.array_equal(kb.double().numpy(), kv) and np.array_equal(qb.double().numpy(), qv)  # exact in bf16
    ref = oracle.pooled(x.cu_q, x.cu_k, qb, kb, BLOCK)
    got = oracle.pooled_fp8(x.cu_q, x.cu_k, q8, q_scale, k8, k_scale, BLOCK)
    assert np.array_equal(got, ref)


def test_pooled_fp8_matches_brute_force_with_quantizer_scales():
    cfg, x = _case(seed=3)
    q8, q_scale, k8, k_scale = oracle.quantize_index_fp8(x.cu_q, x.cu_k, x.q_idx, x.k_idx, BLOCK)
    got = oracle.pooled_fp8(x.cu_q, x.cu_k, q8, q_scale, k8, k_scale, BLOCK)
    kv = _decode(k8) * k_scale.astype(np.float64)[_block_rows(x.cu_k, BLOCK)][:, None]
    qv = _decode(q8) * q_scale.astype(np.float64)[:, :, None]
    pos = oracle.query_positions(x.cu_q, x.cu_k)
    cu_q, cu_k = x.cu_q.numpy(), x.cu_k.numpy()
    nb_stride = got.shape[2]
    ref = np.full(got.shape, -np.inf, np.float32)
    for s in range(len(cu_q) - 1):
        keys = kv[cu_k[s]:cu_k[s + 1]]
        for i in range(cu_q[s], cu_q[s + 1]):
            sc = np.einsum("gd,jd->gj", qv[i], keys[:pos[i] + 1]).astype(np.float32)
            for b in range(pos[i] // BLOCK + 1):
                ref[i, :, b] = sc[:, b * BLOCK:(b + 1) * BLOCK].max(axis=1)
    assert nb_stride == ref.shape[2]
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got))
    # the two float64 sums differ only in order: at most one fp32 unit apart, almost always equal
    ulps = np.abs(got[fin].view(np.int32).astype(np.int64) - ref[fin].view(np.int32).astype(np.int64))
    assert ulps.max() <= 1 and (ulps == 0).mean() > 0.99


def test_index_fp8_is_the_selection_over_pooled_fp8():
    cfg, x = _case(seed=4)
    q8, q_scale, k8, k_scale = oracle.quantize_index_fp8(x.cu_q, x.cu_k, x.q_idx, x.k_idx, BLOCK)
    pooled = oracle.pooled_fp8(x.cu_q, x.cu_k, q8, q_scale, k8, k_scale, BLOCK)
    got = oracle.index_fp8(x.cu_q, x.cu_k, q8, q_scale, k8, k_scale, BLOCK, cfg.topk)
    pos = oracle.query_positions(x.cu_q, x.cu_k)
    for i in range(x.total_q):
        for g in range(cfg.hkv):
            sel, gap = oracle.select(pooled[i, g], pos[i] // BLOCK + 1, cfg.topk)
            assert np.array_equal(got["idx"][i, g], sel) and got["gap"][i, g] == gap


def test_quantize_index_fp8_scales_and_extremes():
    cfg, x = _case(seed=5)
    q8, q_scale, k8, k_scale = oracle.quantize_index_fp8(x.cu_q, x.cu_k, x.q_idx, x.k_idx, BLOCK)
    assert q8.shape == (x.total_q, cfg.hkv, cfg.d_idx) and k8.shape == (x.total_k, cfg.d_idx)
    qf, kf = x.q_idx.float().numpy(), x.k_idx.float().numpy()
    amax_q = np.abs(qf).max(axis=2)
    assert np.array_equal(q_scale, (amax_q / np.float32(448.0)).astype(np.float32))
    rows = _block_rows(x.cu_k, BLOCK)
    for r in range(int(rows.max()) + 1):
        blk = kf[rows == r]
        assert k_scale[r] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))
        j = np.unravel_index(np.abs(blk).argmax(), blk.shape)
        assert k8[rows == r][j] in (0x7E, 0xFE)
    i, g = np.unravel_index(amax_q.argmax(), amax_q.shape)
    assert q8[i, g, np.abs(qf[i, g]).argmax()] in (0x7E, 0xFE)


def test_cpu_quantizer_of_the_tests_matches_the_oracle():
    """The torch-based quantizer that feeds the full-size GPU tests (the oracle's code-by-code search is too
    slow there) gives the oracle quantizer's codes and scales bit for bit."""
    cfg, x = _case(seed=6, seqs=((70, 300), (1, 1), (128, 128), (200, 513)), hkv=4, d_idx=128)
    ref = oracle.quantize_index_fp8(x.cu_q, x.cu_k, x.q_idx, x.k_idx, 128)
    got = quantize_index_cpu(x, block=128, chunk=100)
    for a, b in zip(got, ref):
        assert a.shape == b.shape and np.array_equal(a, b)
