"""msa_sparse_attn_decode_static: the decode Main Branch for callers that
cannot allocate device memory.

Some callers of this library run where they may not call cudaMalloc (or an
allocating library routine): a host framework that only hands out its own
pre-allocated tensors, an allocator-free serving loop, a process whose device
memory pool is already fully reserved.  For them the library keeps a fixed
device array as scratch and this entry point takes no workspace.

These tests call it through the C ABI (ctypes on the shared library) and check
that two calls in a row -- on different batches, so the second one starts from
the first one's leftovers in the shared array -- give bit for bit what the
workspace-based msa_sparse_attn_decode gives (the same kernels on the same
inputs; a leftover in the shared array that leaked into a result would show
here), with no device-side error flag raised in either call's scratch.  The
file is named so that pytest collects it after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

from parity import problem_for


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_05_gb300 as m
    return m


def _static_flags(msa):
    """Device-side error flags of the last static-scratch call (msa_read_device_status with no workspace)."""
    flags = ctypes.c_uint32(0xFFFFFFFF)
    st = msa._lib.msa_read_device_status(None, ctypes.byref(flags),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, (st, msa._lib.msa_last_error_detail())
    return flags.value


def _static_call(msa, prob, x, idx):
    """One call of the static-scratch entry point through the C ABI."""
    o = torch.empty_like(x.q)
    lse = torch.empty((x.total_q, x.cfg.hq), dtype=torch.float32, device=x.q.device)
    st = msa._lib.msa_sparse_attn_decode_static(
        ctypes.byref(prob.c()), ctypes.c_void_p(x.q.data_ptr()), ctypes.c_void_p(x.k.data_ptr()),
        ctypes.c_void_p(x.v.data_ptr()), ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, (st, msa._lib.msa_last_error_detail())
    return o, lse


def _decode_batch(msa, n, ctx, seed):
    cfg = workloads.configs.Workload("static_dec", None, seed=seed, decode_batch=n, decode_ctx=ctx, n_topics=16)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    idx = msa.msa_index_topk(prob, x.q_idx, x.k_idx)
    return x, prob, idx


@pytest.mark.gpu
def test_static_scratch_decode_matches_workspace_decode_twice(msa):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    # two batches of different shapes, run back to back through the shared array
    for n, ctx, seed in ((24, 9000, 5), (7, 40000, 6)):
        x, prob, idx = _decode_batch(msa, n, ctx, seed)
        ws = msa.workspace(prob, msa.Op.SPARSE_ATTN_DECODE)
        o_ref, lse_ref = msa.msa_sparse_attn_decode(prob, x.q, x.k, x.v, idx, ws=ws)
        assert msa.msa_read_device_status(ws) == 0
        o, lse = _static_call(msa, prob, x, idx)
        assert _static_flags(msa) == 0
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), "the static scratch changed the output"
        assert torch.equal(lse, lse_ref), "the static scratch changed the LSE"
        assert torch.isfinite(o.float()).all()


@pytest.mark.gpu
def test_static_scratch_rejects_batches_beyond_its_size(msa):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    # 400 decode sequences need more scratch than the fixed array holds: rejected on the host
    prob = msa.problem_from_seqlens([1] * 400, [300] * 400, hq=64, hkv=4, d_idx=128, topk=16)
    q = torch.zeros(400, 64, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(400 * 300, 4, 128, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(400, 4, 16, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(400, 64, dtype=torch.float32, device="cuda")
    st = msa._lib.msa_sparse_attn_decode_static(
        ctypes.byref(prob.c()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kv.data_ptr()),
        ctypes.c_void_p(kv.data_ptr()), ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), None)
    assert st == -4
    assert b"static buffer holds" in msa._lib.msa_last_error_detail()
