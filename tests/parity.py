"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same inputs (all rows or a sample), compare.

Tolerances (stated for the Main Branch output of the method): selected block
indices bit-exact except rows whose oracle gap between the last selected and
the first unselected non-local pooled score is below 1e-5 relative (near-ties,
counted and reported, exempt together with their O and LSE); O max-abs 1e-2
and mean-abs 1e-3; LSE max-abs 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

NEAR_TIE = 1e-5
O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3


def problem_for(msa, x):
    cfg = x.cfg
    return msa.Problem(x.cu_q, x.cu_k, x.total_q, x.total_k, x.max_q, x.max_k, cfg.hq, cfg.hkv, cfg.d_idx,
                       cfg.topk)


def sample_rows(x, n_random=48, seed=0):
    """Query rows to check: sequence starts and ends, block boundaries, and a seeded random sample."""
    rng = np.random.default_rng(seed)
    cu_q = x.cu_q.cpu().numpy()
    pos = oracle.query_positions(x.cu_q, x.cu_k)
    rows = set()
    for s in range(len(cu_q) - 1):
        a, b = int(cu_q[s]), int(cu_q[s + 1])
        if b > a:
            rows.update({a, b - 1, min(a + 1, b - 1), (a + b) // 2})
            # a query at a block start and one just before it
            for t in range(a, b):
                if pos[t] % 128 == 0 and t > a:
                    rows.update({t, t - 1})
                    break
    if x.total_q:
        rows.update(rng.integers(0, x.total_q, size=min(n_random, x.total_q)).tolist())
    return np.array(sorted(rows), dtype=np.int32)


def compare_indices(idx_gpu: np.ndarray, ref: dict):
    """Returns (tie mask [n, hkv], number of non-exempt mismatching rows); prints the first mismatches."""
    tie = ref["gap"] < NEAR_TIE
    mism = (idx_gpu != ref["idx"]).any(axis=-1) & ~tie
    for r, g in np.argwhere(mism)[:5]:
        print(f"index mismatch row {r} group {g}: gpu {idx_gpu[r, g].tolist()} oracle {ref['idx'][r, g].tolist()} "
              f"gap {ref['gap'][r, g]:.3e}")
    return tie, int(mism.sum())


def compare_attention(o_gpu: np.ndarray, lse_gpu: np.ndarray, ref: dict, group: int, exempt=None):
    """Max/mean abs error of O and max abs error of LSE over the non-exempt rows."""
    ok = np.ones(ref["lse"].shape, dtype=bool)
    if exempt is not None:
        ok = np.repeat(~exempt, group, axis=1)
    err = np.abs(o_gpu.astype(np.float64) - ref["o"])[ok]
    lerr = np.abs(lse_gpu.astype(np.float64) - ref["lse"])[ok]
    if err.size == 0:
        return 0.0, 0.0, 0.0
    return float(err.max()), float(err.mean()), float(lerr.max())


def assert_attention_close(o_gpu, lse_gpu, ref, group, exempt=None, what=""):
    emax, emean, lmax = compare_attention(o_gpu, lse_gpu, ref, group, exempt)
    assert emax < O_MAX, f"{what}: O max abs err {emax:.3e}"
    assert emean < O_MEAN, f"{what}: O mean abs err {emean:.3e}"
    assert lmax < LSE_MAX, f"{what}: LSE max abs err {lmax:.3e}"
    return emax, emean, lmax


def _e4m3_codes(x: np.ndarray) -> np.ndarray:
    """E4M3 codes of fp32 values within +-448 by torch's float8_e4m3fn conversion (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def quantize_index_cpu(x, block: int = 128, chunk: int = 1 << 20):
    """fp8 index inputs of workload x, computed on the CPU with torch's float8_e4m3fn conversion as the rounding
    step, for sizes the oracle's code-by-code quantizer is too slow for: (q8, q_scale, k8, k_scale) in the
    layout of oracle.quantize_index_fp8, which test_oracle_fp8_index_pins checks it against bit for bit.
    Scale = max |x| / 448 in fp32 (1 when 0) per Q_idx row and group and per key block of a sequence;
    code = RNE(x / scale) with the division in fp32 (the quotient never exceeds 448)."""
    qf = x.q_idx.float().cpu().numpy()
    amax = np.abs(qf).max(axis=2)
    q_scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q8 = _e4m3_codes(qf / q_scale[:, :, None])
    cu_k = x.cu_k.cpu().numpy().astype(np.int64)
    n_keys = int(cu_k[-1])
    blk_of_key = np.empty(n_keys, np.int64)
    r0 = 0
    for s in range(len(cu_k) - 1):
        n = int(cu_k[s + 1] - cu_k[s])
        blk_of_key[cu_k[s]:cu_k[s + 1]] = r0 + np.arange(n) // block
        r0 += -(-n // block)
    k_amax = np.zeros(r0, np.float32)
    k_idx = x.k_idx.cpu()
    for a in range(0, n_keys, chunk):
        kf = k_idx[a:a + chunk].float().numpy()
        np.maximum.at(k_amax, blk_of_key[a:a + chunk], np.abs(kf).max(axis=1))
    k_scale = np.where(k_amax > 0, k_amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    k8 = np.empty((n_keys, k_idx.shape[1]), np.uint8)
    for a in range(0, n_keys, chunk):
        kf = k_idx[a:a + chunk].float().numpy()
        k8[a:a + chunk] = _e4m3_codes(kf / k_scale[blk_of_key[a:a + chunk]][:, None])
    return q8, q_scale, k8, k_scale


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()
