"""The C-ABI library without a GPU: it loads, exports every symbol the public
header declares, sizes workspaces, and rejects bad arguments on the host
before any CUDA call (pointers here are never dereferenced)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_05_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:msa_status_t|const char \*|int32_t)\s*\*?\s*(msa_\w+)\s*\(", text,
                                 re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("msa_index_topk", "msa_sparse_attn_prefill", "msa_sparse_attn_decode", "msa_forward",
              "msa_workspace_size", "msa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(msa):
    lib = ctypes.CDLL(msa.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in msa.h but not exported"
    assert msa.abi_version() == 1


FAKE = 0x10000  # aligned, never dereferenced by host-side validation


def base_problem(msa, **kw):
    p = dict(num_seqs=1, cu_seqlens_q=FAKE, cu_seqlens_k=FAKE, total_q=1024, total_k=1024, max_seqlen_q=1024,
             max_seqlen_k=1024, num_q_heads=64, num_kv_heads=4, head_dim=128, index_dim=128, block_size=128,
             topk=16, softmax_scale=0.0)
    p.update(kw)
    return msa.MsaProblem(**p)


def ws_size(msa, prob, op):
    n = ctypes.c_size_t(0)
    st = msa._lib.msa_workspace_size(ctypes.byref(prob), int(op), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("kw,status", [
    (dict(topk=65), -2), (dict(topk=0), -1), (dict(head_dim=64), -2), (dict(block_size=64), -2),
    (dict(index_dim=96), -2), (dict(num_q_heads=62), -1), (dict(num_q_heads=60), -2), (dict(num_q_heads=12, num_kv_heads=4), -2),
    (dict(num_kv_heads=3, num_q_heads=48), -2), (dict(num_seqs=0), -1), (dict(cu_seqlens_q=None), -1),
    (dict(total_q=-1), -1), (dict(max_seqlen_k=2048), -1), (dict(softmax_scale=float("nan")), -1),
])
def test_invalid_problems_are_rejected(msa, kw, status):
    st, _ = ws_size(msa, base_problem(msa, **kw), msa.Op.FORWARD)
    assert st == status


@pytest.mark.parametrize("topk", [1, 16, 17, 32, 64])
def test_topk_range_is_accepted(msa, topk):
    st, n = ws_size(msa, base_problem(msa, topk=topk), msa.Op.FORWARD)
    assert st == 0 and n >= 1024 * 4 * topk * 16 * 128 * 2


def test_workspace_sizes_grow_with_the_problem(msa):
    small = ws_size(msa, base_problem(msa), msa.Op.FORWARD)
    big = ws_size(msa, base_problem(msa, total_q=4096, total_k=4096, max_seqlen_q=4096, max_seqlen_k=4096),
                  msa.Op.FORWARD)
    assert small[0] == 0 and big[0] == 0 and big[1] > small[1] > 0
    # the partial-output buffer dominates prefill: T * Hkv * k * G * 128 * 2 bytes
    assert small[1] >= 1024 * 4 * 16 * 16 * 128 * 2
    dec = ws_size(msa, base_problem(msa, total_q=8, max_seqlen_q=1, num_seqs=8, total_k=8 * 1024,
                                    max_seqlen_k=1024), msa.Op.FORWARD)
    assert dec[0] == 0 and 0 < dec[1] < small[1]


def test_calls_reject_bad_arguments_before_touching_the_device(msa):
    prob = base_problem(msa)
    lib = msa._lib
    p = ctypes.byref(prob)
    # null tensor
    assert lib.msa_forward(p, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == -1
    # misaligned tensor
    assert lib.msa_forward(p, FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == -3
    # workspace too small / missing
    assert lib.msa_forward(p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1024, None) == -4
    assert lib.msa_forward(p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1 << 40, None) == -4
    # misaligned workspace
    _, need = ws_size(msa, prob, msa.Op.FORWARD)
    assert lib.msa_forward(p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 16, need, None) == -3
    # decode-only entry point on a prefill batch
    assert lib.msa_sparse_attn_decode(p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == -1
    # pooled stride too small
    assert lib.msa_index_pool(p, FAKE, FAKE, FAKE, 7, FAKE, 1 << 40, None) == -1
    # decode path with more index heads than the decode scan takes (8)
    dec = base_problem(msa, num_seqs=4, total_q=4, max_seqlen_q=1, num_q_heads=128, num_kv_heads=16)
    assert lib.msa_forward(ctypes.byref(dec), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40,
                           None) == -2


def test_paged_decode_rejects_bad_arguments_on_the_host(msa):
    lib = msa._lib
    dec = base_problem(msa, num_seqs=4, total_q=4, max_seqlen_q=1)
    p = ctypes.byref(dec)
    args = lambda bt=FAKE, mb=16, npg=100: (p, FAKE, FAKE, FAKE, FAKE, FAKE, bt, mb, npg, FAKE, FAKE, FAKE, FAKE,
                                             1 << 40, None)
    assert lib.msa_forward_decode_paged(*args(bt=None)) == -1        # no block table
    assert lib.msa_forward_decode_paged(*args(bt=FAKE + 2)) == -3    # misaligned block table
    assert lib.msa_forward_decode_paged(*args(npg=0)) == -1          # no pages
    assert lib.msa_forward_decode_paged(*args(npg=1 << 24)) == -1    # rows past int32 coordinates
    assert lib.msa_forward_decode_paged(*args(mb=7)) == -1           # a row cannot hold the longest sequence
    pre = base_problem(msa)                                          # a prefill batch
    assert lib.msa_forward_decode_paged(ctypes.byref(pre), *args()[1:]) == -1


def test_paged_fp8_decode_rejects_bad_arguments_on_the_host(msa):
    lib = msa._lib
    dec = base_problem(msa, num_seqs=4, total_q=4, max_seqlen_q=1)
    p = ctypes.byref(dec)
    args = lambda ks=FAKE, bt=FAKE, mb=16, npg=100: (p, FAKE, FAKE, FAKE, ks, FAKE, FAKE, FAKE, bt, mb, npg, FAKE,
                                                      FAKE, FAKE, FAKE, 1 << 40, None)
    assert lib.msa_forward_decode_paged_fp8(*args(ks=None)) == -1     # no K scales
    assert lib.msa_forward_decode_paged_fp8(*args(ks=FAKE + 2)) == -3 # misaligned scales
    assert lib.msa_forward_decode_paged_fp8(*args(bt=None)) == -1     # no block table
    assert lib.msa_forward_decode_paged_fp8(*args(npg=0)) == -1       # no pages
    assert lib.msa_forward_decode_paged_fp8(*args(mb=7)) == -1        # a row cannot hold the longest sequence
    pre = base_problem(msa)                                           # a prefill batch
    assert lib.msa_forward_decode_paged_fp8(ctypes.byref(pre), *args()[1:]) == -1


def test_fp8_index_calls_reject_bad_arguments_on_the_host(msa):
    lib = msa._lib
    pre = base_problem(msa)
    p = ctypes.byref(pre)
    p64 = ctypes.byref(base_problem(msa, index_dim=64))
    quant = lambda prob=p, qi=FAKE, ki=FAKE, q8=FAKE, qs=FAKE, k8=FAKE, ks=FAKE: (prob, qi, ki, q8, qs, k8, ks, FAKE,
                                                                                   1 << 40, None)
    assert lib.msa_quantize_index_fp8(*quant(qi=None, ki=None)) == -1   # nothing to quantize
    assert lib.msa_quantize_index_fp8(*quant(qs=None)) == -1            # a side without its scales
    assert lib.msa_quantize_index_fp8(*quant(k8=FAKE + 8)) == -3        # misaligned codes
    assert lib.msa_quantize_index_fp8(*quant(ks=FAKE + 2)) == -3        # misaligned scales
    assert lib.msa_quantize_index_fp8(*quant(prob=p64)) == -2           # index_dim 64: bf16 index only
    topk = lambda prob=p, qs=FAKE, k8=FAKE: (prob, FAKE, qs, k8, FAKE, FAKE, FAKE, 1 << 40, None)
    assert lib.msa_index_topk_fp8(*topk(qs=None)) == -1
    assert lib.msa_index_topk_fp8(*topk(k8=FAKE + 4)) == -3
    assert lib.msa_index_topk_fp8(*topk(prob=p64)) == -2
    assert lib.msa_index_pool_fp8(p, FAKE, FAKE, FAKE, FAKE, FAKE, 7, FAKE, 1 << 40, None) == -1  # stride < 8 blocks
    fwd = lambda ks=FAKE: (p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ks, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert lib.msa_forward_fp8_index(*fwd(ks=None)) == -1
    assert lib.msa_forward_fp8_index(*fwd(ks=FAKE + 1)) == -3
    st, n = ws_size(msa, pre, msa.Op.QUANTIZE_INDEX_FP8)
    assert st == 0 and n > 0
    dec = base_problem(msa, num_seqs=4, total_q=4, max_seqlen_q=1)
    paged = lambda prob=ctypes.byref(dec), kis=FAKE, bt=FAKE, mb=16, npg=100: (
        prob, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, kis, bt, mb, npg, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert lib.msa_forward_decode_paged_fp8_index(*paged(kis=None)) == -1     # no index-key scales
    assert lib.msa_forward_decode_paged_fp8_index(*paged(bt=FAKE + 2)) == -3  # misaligned block table
    assert lib.msa_forward_decode_paged_fp8_index(*paged(npg=0)) == -1        # no pages
    assert lib.msa_forward_decode_paged_fp8_index(*paged(mb=7)) == -1         # a row cannot hold a sequence
    assert lib.msa_forward_decode_paged_fp8_index(*paged(prob=p)) == -1       # a prefill batch


def test_status_strings(msa):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert msa._lib.msa_status_string(code)
    assert msa._lib.msa_status_string(-99) == b"unknown status"
