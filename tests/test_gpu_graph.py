"""The library's calls inside CUDA graphs.

Each call is captured once with torch.cuda.graph (its workspace and outputs allocated before the capture,
one direct call made first so that one-time set-up stays out of the graph) and replayed.  A replay must give
the outputs of the same call made directly, bit for bit, and must read the inputs' current contents: new
queries are written in place between replays and the replay must follow them.  Covered: the prefill and
decode forward calls, the paged decode, the all-fp8 forward, and the static-scratch decode (whose first
call, made before the capture, looks up its array).  The decode chain's programmatic dependent launches
become programmatic edges of the graph.  The direct calls are themselves checked against the oracle in
test_gpu_parity / test_gpu_fp8_index.
"""
import ctypes

import pytest
import torch

import workloads
from workloads.configs import small

from parity import problem_for
from test_gpu_parity import _paged

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


def _capture(call):
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    return g


def _replay(g, outs):
    """Clears the outputs, replays, returns copies of what the replay wrote."""
    for t in outs:
        t.fill_(-3 if t.dtype == torch.int32 else 7)
    g.replay()
    torch.cuda.synchronize()
    return [t.clone() for t in outs]


def _same(a, b, what):
    for u, v in zip(a, b):
        assert torch.equal(u, v), f"{what}: the replay differs from the direct call"


def _fresh_queries(x, seed):
    """New q and q_idx of the same shapes and distributions, written in place."""
    gen = torch.Generator(device="cuda").manual_seed(seed)
    x.q.copy_(torch.randn(x.q.shape, generator=gen, device="cuda").to(x.q.dtype))
    x.q_idx.copy_((torch.randn(x.q_idx.shape, generator=gen, device="cuda") * 2).to(x.q_idx.dtype))


def _check_forward(msa, x, direct, outs, ws):
    """direct(idx, o, lse) runs the call into the given outputs; the graph captures it into `outs`."""
    g = _capture(lambda: direct(*outs))
    for rep in range(2):
        got = _replay(g, outs)
        ref = [torch.empty_like(t) for t in outs]
        direct(*ref)
        torch.cuda.synchronize()
        _same(got, ref, f"replay {rep}")
        assert msa.msa_read_device_status(ws) == 0
        before = got
        _fresh_queries(x, seed=100 + rep)
        after = _replay(g, outs)
        assert not torch.equal(before[1], after[1]), "the replay did not read the new queries"


def _outs(x, cfg):
    return [torch.empty((x.total_q, cfg.hkv, cfg.topk), dtype=torch.int32, device="cuda"), torch.empty_like(x.q),
            torch.empty((x.total_q, cfg.hq), dtype=torch.float32, device="cuda")]


def test_graph_prefill_forward(msa):
    cfg = small("graph_prefill", ((300, 300), (1000, 1777), (1, 129), (129, 900)), hq=64, hkv=4, d_idx=128,
                topk=16, n_topics=16, seed=41)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    ws = msa.workspace(prob, msa.Op.FORWARD)
    direct = lambda i, o, l: msa.msa_forward(prob, x.q, x.k, x.v, x.q_idx, x.k_idx, idx=i, o=o, lse=l, ws=ws)
    _check_forward(msa, x, direct, _outs(x, cfg), ws)


def test_graph_decode_forward(msa):
    cfg = workloads.configs.Workload("graph_dec", None, seed=42, decode_batch=8, decode_ctx=5000, n_topics=16)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    ws = msa.workspace(prob, msa.Op.FORWARD)
    direct = lambda i, o, l: msa.msa_forward(prob, x.q, x.k, x.v, x.q_idx, x.k_idx, idx=i, o=o, lse=l, ws=ws)
    _check_forward(msa, x, direct, _outs(x, cfg), ws)


def test_graph_decode_paged(msa):
    cfg = workloads.configs.Workload("graph_paged", None, seed=43, decode_batch=6, decode_ctx=9000, n_topics=16)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    k_c, v_c, ki_c, bt = _paged(x, cfg, 43)
    ws = msa.workspace(prob, msa.Op.FORWARD)
    direct = lambda i, o, l: msa.msa_forward_decode_paged(prob, x.q, k_c, v_c, x.q_idx, ki_c, bt, idx=i, o=o, lse=l,
                                                          ws=ws)
    _check_forward(msa, x, direct, _outs(x, cfg), ws)


def test_graph_all_fp8_forward(msa):
    cfg = small("graph_fp8", ((300, 300), (700, 1500), (129, 129)), hq=64, hkv=4, d_idx=128, topk=16,
                n_topics=16, seed=44)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    k8, v8, ks, vs = msa.msa_quantize_kv_fp8(prob, x.k, x.v)
    ki8, kis = msa.msa_quantize_index_fp8(prob, k_idx=x.k_idx)[2:]
    qi8, qis = msa.msa_quantize_index_fp8(prob, q_idx=x.q_idx)[:2]
    ws = msa.workspace(prob, msa.Op.FORWARD_FP8)
    wsq = msa.workspace(prob, msa.Op.QUANTIZE_INDEX_FP8)

    def direct(i, o, l):
        # the queries' index codes are made inside the captured work, so the replay follows new q_idx
        msa.msa_quantize_index_fp8(prob, q_idx=x.q_idx, q_idx8=qi8, q_idx_scale=qis, ws=wsq)
        msa.msa_forward_fp8_index(prob, x.q, k8, v8, ks, vs, qi8, qis, ki8, kis, idx=i, o=o, lse=l, ws=ws)

    _check_forward(msa, x, direct, _outs(x, cfg), ws)


def test_graph_static_scratch_decode(msa):
    cfg = workloads.configs.Workload("graph_static", None, seed=45, decode_batch=12, decode_ctx=7000, n_topics=16)
    x = workloads.generate(cfg, device="cuda")
    prob = problem_for(msa, x)
    idx = msa.msa_index_topk(prob, x.q_idx, x.k_idx)
    o, lse = torch.empty_like(x.q), torch.empty((x.total_q, cfg.hq), dtype=torch.float32, device="cuda")

    def static():
        st = msa._lib.msa_sparse_attn_decode_static(
            ctypes.byref(prob.c()), ctypes.c_void_p(x.q.data_ptr()), ctypes.c_void_p(x.k.data_ptr()),
            ctypes.c_void_p(x.v.data_ptr()), ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(o.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, (st, msa._lib.msa_last_error_detail())

    g = _capture(static)
    ws = msa.workspace(prob, msa.Op.SPARSE_ATTN_DECODE)
    for rep in range(2):
        got = _replay(g, [o, lse])
        o_ref, lse_ref = msa.msa_sparse_attn_decode(prob, x.q, x.k, x.v, idx, ws=ws)
        torch.cuda.synchronize()
        _same(got, [o_ref, lse_ref], f"static replay {rep}")
        _fresh_queries(x, seed=200 + rep)
