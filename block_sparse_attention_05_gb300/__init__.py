"""MiniMax Sparse Attention (MSA) forward pass on GB300 -- Python binding.

A thin ctypes layer over the C ABI in ``include/msa.h`` (library
``_lib/libmsa.so``, built for sm_103a by ``__graft_entry__.build()``).  This
module only marshals torch tensors into pointers and sizes and raises on a
non-OK status; every step of the method runs in the library's CUDA kernels.
There is no CPU fallback: importing without the built library raises.

Entry points (same names as the C functions):
  msa_index_pool, msa_topk_pooled, msa_index_topk,
  msa_sparse_attn_prefill, msa_sparse_attn_decode, msa_forward,
  msa_sparse_attn_decode_static, msa_forward_decode_paged,
  msa_quantize_kv_fp8, msa_sparse_attn_prefill_fp8, msa_sparse_attn_decode_fp8, msa_forward_fp8,
  msa_forward_decode_paged_fp8,
  msa_quantize_index_fp8, msa_index_pool_fp8, msa_index_topk_fp8, msa_forward_fp8_index,
  msa_forward_decode_paged_fp8_index,
  msa_index_prologue,
  msa_workspace_size, msa_read_device_status.
"""
from __future__ import annotations

import ctypes
import dataclasses
import enum
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmsa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first (python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = _lib.msa_last_error_detail().decode() if status == -5 else ""
        super().__init__(f"{where}: {_lib.msa_status_string(status).decode()} (status {status})"
                         + (f" [{detail}]" if detail else ""))


class Op(enum.IntEnum):
    INDEX_PROLOGUE = 11
    INDEX_POOL = 1
    INDEX_TOPK = 2
    SPARSE_ATTN_PREFILL = 3
    SPARSE_ATTN_DECODE = 4
    FORWARD = 5
    TOPK_POOLED = 6
    QUANTIZE_KV_FP8 = 7
    SPARSE_ATTN_PREFILL_FP8 = 8
    SPARSE_ATTN_DECODE_FP8 = 9
    FORWARD_FP8 = 10
    QUANTIZE_INDEX_FP8 = 12


DEVICE_TIMEOUT = 1
DEVICE_BAD_SEQLENS = 2
DEVICE_BAD_INDEX = 4


class MsaProblem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("total_q", ctypes.c_int32),
        ("total_k", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32),
        ("max_seqlen_k", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("index_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
    ]


_P = ctypes.POINTER(MsaProblem)
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t

_lib.msa_status_string.restype = ctypes.c_char_p
_lib.msa_status_string.argtypes = [ctypes.c_int]
_lib.msa_abi_version.restype = ctypes.c_int32
_lib.msa_workspace_size.restype = ctypes.c_int
_lib.msa_workspace_size.argtypes = [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
_lib.msa_index_pool.restype = ctypes.c_int
_lib.msa_index_pool.argtypes = [_P, _vp, _vp, _vp, _i64, _vp, _sz, _vp]
_lib.msa_topk_pooled.restype = ctypes.c_int
_lib.msa_topk_pooled.argtypes = [_P, _vp, _i64, _vp, _vp, _sz, _vp]
_lib.msa_index_topk.restype = ctypes.c_int
_lib.msa_index_topk.argtypes = [_P, _vp, _vp, _vp, _vp, _sz, _vp]
for _fn in (_lib.msa_sparse_attn_prefill, _lib.msa_sparse_attn_decode):
    _fn.restype = ctypes.c_int
    _fn.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.msa_sparse_attn_decode_static.restype = ctypes.c_int
_lib.msa_sparse_attn_decode_static.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.msa_forward.restype = ctypes.c_int
_lib.msa_forward.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.msa_forward_decode_paged.restype = ctypes.c_int
_lib.msa_forward_decode_paged.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32, _i64, _vp, _vp, _vp, _vp,
                                          _sz, _vp]
_lib.msa_quantize_kv_fp8.restype = ctypes.c_int
_lib.msa_quantize_kv_fp8.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
for _fn in (_lib.msa_sparse_attn_prefill_fp8, _lib.msa_sparse_attn_decode_fp8):
    _fn.restype = ctypes.c_int
    _fn.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.msa_forward_fp8.restype = ctypes.c_int
_lib.msa_forward_fp8.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
# problem, q, k8, v8, k_scale, v_scale, q_idx, k_idx cache, block table, stride, pages, idx, o, lse, ws, bytes, stream
_lib.msa_forward_decode_paged_fp8.restype = ctypes.c_int
_lib.msa_forward_decode_paged_fp8.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32, _i64, _vp,
                                              _vp, _vp, _vp, _sz, _vp]
# problem, q_idx, k_idx, q_idx8, q_idx_scale, k_idx8, k_idx_scale, ws, bytes, stream
_lib.msa_quantize_index_fp8.restype = ctypes.c_int
_lib.msa_quantize_index_fp8.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
# problem, q_idx8, q_idx_scale, k_idx8, k_idx_scale, pooled, stride, ws, bytes, stream
_lib.msa_index_pool_fp8.restype = ctypes.c_int
_lib.msa_index_pool_fp8.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _sz, _vp]
_lib.msa_index_topk_fp8.restype = ctypes.c_int
_lib.msa_index_topk_fp8.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
# problem, q, k8, v8, k_scale, v_scale, q_idx8, q_idx_scale, k_idx8, k_idx_scale, idx, o, lse, ws, bytes, stream
_lib.msa_forward_fp8_index.restype = ctypes.c_int
_lib.msa_forward_fp8_index.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
# problem, q, k8, v8, k_scale, v_scale, q_idx8, q_idx_scale, k_idx8 cache, k_idx_scale, block table, stride, pages,
# idx, o, lse, ws, bytes, stream
_lib.msa_forward_decode_paged_fp8_index.restype = ctypes.c_int
_lib.msa_forward_decode_paged_fp8_index.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                                    ctypes.c_int32, _i64, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.msa_index_prologue.restype = ctypes.c_int
_lib.msa_index_prologue.argtypes = [_P, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.msa_read_device_status.restype = ctypes.c_int
_lib.msa_read_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32), _vp]
_lib.msa_set_stage_events.restype = ctypes.c_int
_lib.msa_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
_lib.msa_kernel_launch_count.restype = ctypes.c_int64
_lib.msa_last_error_detail.restype = ctypes.c_char_p

EXPORTED = ("msa_workspace_size", "msa_index_pool", "msa_topk_pooled", "msa_index_topk",
            "msa_sparse_attn_prefill", "msa_sparse_attn_decode", "msa_forward",
            "msa_read_device_status", "msa_status_string", "msa_abi_version", "msa_set_stage_events",
            "msa_kernel_launch_count", "msa_last_error_detail", "msa_sparse_attn_decode_static",
            "msa_forward_decode_paged", "msa_quantize_kv_fp8", "msa_sparse_attn_prefill_fp8",
            "msa_sparse_attn_decode_fp8", "msa_forward_fp8", "msa_index_prologue",
            "msa_forward_decode_paged_fp8", "msa_quantize_index_fp8", "msa_index_pool_fp8", "msa_index_topk_fp8",
            "msa_forward_fp8_index", "msa_forward_decode_paged_fp8_index")

STAGES = ("plan", "index", "topk", "schedule", "attn", "combine")


@dataclasses.dataclass
class Problem:
    """Sizes of one packed batch.  ``cu_q`` / ``cu_k`` are int32 device tensors."""
    cu_q: torch.Tensor
    cu_k: torch.Tensor
    total_q: int
    total_k: int
    max_q: int
    max_k: int
    hq: int
    hkv: int
    d_idx: int
    topk: int
    head_dim: int = 128
    block: int = 128
    scale: float = 0.0

    @property
    def num_seqs(self) -> int:
        return int(self.cu_q.numel()) - 1

    def c(self) -> MsaProblem:
        return MsaProblem(self.num_seqs, _ptr(self.cu_q), _ptr(self.cu_k), self.total_q, self.total_k,
                          self.max_q, self.max_k, self.hq, self.hkv, self.head_dim, self.d_idx, self.block,
                          self.topk, self.scale)


def problem_from_seqlens(q_lens, kv_lens, hq, hkv, d_idx, topk, device="cuda", scale=0.0) -> Problem:
    """Builds the prefix sums from per-sequence lengths (host lists)."""
    cu_q = [0]
    cu_k = [0]
    for a, b in zip(q_lens, kv_lens):
        cu_q.append(cu_q[-1] + int(a))
        cu_k.append(cu_k[-1] + int(b))
    return Problem(torch.tensor(cu_q, dtype=torch.int32, device=device),
                   torch.tensor(cu_k, dtype=torch.int32, device=device), cu_q[-1], cu_k[-1],
                   max(q_lens) if len(q_lens) else 0, max(kv_lens) if len(kv_lens) else 0, hq, hkv, d_idx, topk,
                   scale=scale)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise MsaError(status, where)


def _need(t: torch.Tensor, dtype, name: str):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def msa_workspace_size(problem: Problem, op: Op) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.msa_workspace_size(ctypes.byref(problem.c()), int(op), ctypes.byref(n)), "msa_workspace_size")
    return int(n.value)


def workspace(problem: Problem, op: Op, device=None) -> torch.Tensor:
    """A device buffer large enough for ``op`` (256-byte aligned by the caching allocator)."""
    nbytes = max(msa_workspace_size(problem, op), 256)
    return torch.empty(nbytes, dtype=torch.uint8, device=device or problem.cu_q.device)


def _ws(problem, op, ws):
    if ws is None:
        ws = workspace(problem, op)
    return ws, ctypes.c_size_t(ws.numel())


def max_blocks(problem: Problem) -> int:
    return max(1, (problem.max_k + problem.block - 1) // problem.block)


def msa_index_pool(problem: Problem, q_idx, k_idx, pooled=None, ws=None):
    """Pooled causal index scores, fp32 [total_q * hkv, ceil(max_k / 128)]; entries past a row's causal end
    are left as they were (NaN when ``pooled`` is allocated here)."""
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(k_idx, torch.bfloat16, "k_idx")
    nb = max_blocks(problem)
    if pooled is None:
        pooled = torch.full((problem.total_q * problem.hkv, nb), float("nan"), dtype=torch.float32,
                            device=q_idx.device)
    ws, nws = _ws(problem, Op.INDEX_POOL, ws)
    _check(_lib.msa_index_pool(ctypes.byref(problem.c()), _ptr(q_idx), _ptr(k_idx), _ptr(pooled),
                               pooled.stride(0), _ptr(ws), nws, _stream()), "msa_index_pool")
    return pooled


def msa_topk_pooled(problem: Problem, pooled, idx=None, ws=None):
    _need(pooled, torch.float32, "pooled")
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=pooled.device)
    ws, nws = _ws(problem, Op.TOPK_POOLED, ws)
    _check(_lib.msa_topk_pooled(ctypes.byref(problem.c()), _ptr(pooled), pooled.stride(0), _ptr(idx), _ptr(ws),
                                nws, _stream()), "msa_topk_pooled")
    return idx


def msa_index_topk(problem: Problem, q_idx, k_idx, idx=None, ws=None):
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(k_idx, torch.bfloat16, "k_idx")
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=q_idx.device)
    ws, nws = _ws(problem, Op.INDEX_TOPK, ws)
    _check(_lib.msa_index_topk(ctypes.byref(problem.c()), _ptr(q_idx), _ptr(k_idx), _ptr(idx), _ptr(ws), nws,
                               _stream()), "msa_index_topk")
    return idx


def _attn(fn, op, where, problem, q, k, v, idx, o, lse, ws):
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(idx, torch.int32, "idx")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=q.device)
    ws, nws = _ws(problem, op, ws)
    _check(fn(ctypes.byref(problem.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(o), _ptr(lse), _ptr(ws), nws,
              _stream()), where)
    return o, lse


def msa_sparse_attn_prefill(problem: Problem, q, k, v, idx, o=None, lse=None, ws=None):
    return _attn(_lib.msa_sparse_attn_prefill, Op.SPARSE_ATTN_PREFILL, "msa_sparse_attn_prefill", problem, q, k,
                 v, idx, o, lse, ws)


def msa_sparse_attn_decode(problem: Problem, q, k, v, idx, o=None, lse=None, ws=None):
    return _attn(_lib.msa_sparse_attn_decode, Op.SPARSE_ATTN_DECODE, "msa_sparse_attn_decode", problem, q, k, v,
                 idx, o, lse, ws)


def msa_sparse_attn_decode_static(problem: Problem, q, k, v, idx, o=None, lse=None):
    """The decode Main Branch without a workspace: its scratch is a fixed device array inside the library
    (for callers that cannot allocate device memory; see include/msa.h).  Calls share that array, so calls
    that may overlap on the GPU must be serialised."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(idx, torch.int32, "idx")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=q.device)
    _check(_lib.msa_sparse_attn_decode_static(ctypes.byref(problem.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(idx),
                                              _ptr(o), _ptr(lse), _stream()), "msa_sparse_attn_decode_static")
    return o, lse


def msa_forward(problem: Problem, q, k, v, q_idx, k_idx, idx=None, o=None, lse=None, ws=None):
    """Both branches.  Returns (idx [T, Hkv, k] int32, o [T, Hq, 128] bf16, lse [T, Hq] fp32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (q_idx, "q_idx"), (k_idx, "k_idx")):
        _need(t, torch.bfloat16, n)
    dev = q.device
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=dev)
    ws, nws = _ws(problem, Op.FORWARD, ws)
    _check(_lib.msa_forward(ctypes.byref(problem.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx),
                            _ptr(idx), _ptr(o), _ptr(lse), _ptr(ws), nws, _stream()), "msa_forward")
    return idx, o, lse


def msa_forward_decode_paged(problem: Problem, q, k_cache, v_cache, q_idx, k_idx_cache, block_table, idx=None,
                             o=None, lse=None, ws=None):
    """Decode from paged caches ([num_pages * 128, ...] rows, block_table int32 [num_seqs, max_blocks]).
    Returns (idx, o, lse) as msa_forward."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (q_idx, "q_idx"), (k_idx_cache, "k_idx_cache")):
        _need(t, torch.bfloat16, n)
    _need(block_table, torch.int32, "block_table")
    if block_table.dim() != 2 or k_cache.shape[0] % 128:
        raise ValueError("block_table must be [num_seqs, max_blocks] and the caches whole pages of 128 rows")
    dev = q.device
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=dev)
    ws, nws = _ws(problem, Op.FORWARD, ws)
    _check(_lib.msa_forward_decode_paged(ctypes.byref(problem.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(q_idx), _ptr(k_idx_cache), _ptr(block_table), block_table.shape[1],
                                         k_cache.shape[0] // 128, _ptr(idx), _ptr(o), _ptr(lse), _ptr(ws), nws,
                                         _stream()), "msa_forward_decode_paged")
    return idx, o, lse


# ---------------------------------------------------------------- index prologue
def msa_index_prologue(problem: Problem, x, w_q, w_k, gamma_q, gamma_k, k_idx, q_idx=None, ws=None):
    """Hidden states x [total_q, d_model] -> Q_idx [total_q, Hkv, 128] (returned) and the new tokens' rows
    k_start + pos(i) of the index-key cache k_idx [total_k, 128] (written in place): projection, RMSNorm,
    RoPE on dims 0..63."""
    for t, n in ((x, "x"), (w_q, "w_q"), (w_k, "w_k"), (gamma_q, "gamma_q"), (gamma_k, "gamma_k"), (k_idx, "k_idx")):
        _need(t, torch.bfloat16, n)
    if q_idx is None:
        q_idx = torch.empty((problem.total_q, problem.hkv, problem.d_idx), dtype=torch.bfloat16, device=x.device)
    ws, nws = _ws(problem, Op.INDEX_PROLOGUE, ws)
    _check(_lib.msa_index_prologue(ctypes.byref(problem.c()), _ptr(x), int(x.shape[1]), _ptr(w_q), _ptr(w_k),
                                   _ptr(gamma_q), _ptr(gamma_k), _ptr(q_idx), _ptr(k_idx), _ptr(ws), nws, _stream()),
           "msa_index_prologue")
    return q_idx


# ---------------------------------------------------------------- fp8 K/V
def fp8_scale_rows(problem: Problem) -> int:
    """Rows to allocate for a scale array: total_k / 128 + num_seqs bounds the number of key blocks."""
    return problem.total_k // problem.block + problem.num_seqs


def msa_quantize_kv_fp8(problem: Problem, k, v, k8=None, v8=None, k_scale=None, v_scale=None, ws=None):
    """bf16 K, V -> E4M3 codes (uint8, same shape) and fp32 scales [key blocks, Hkv] (rows past the sequences'
    key blocks are left as they were).  Returns (k8, v8, k_scale, v_scale)."""
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v")
    dev = k.device
    if k8 is None:
        k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    if v8 is None:
        v8 = torch.empty(v.shape, dtype=torch.uint8, device=dev)
    rows = (fp8_scale_rows(problem), problem.hkv)
    if k_scale is None:
        k_scale = torch.zeros(rows, dtype=torch.float32, device=dev)
    if v_scale is None:
        v_scale = torch.zeros(rows, dtype=torch.float32, device=dev)
    ws, nws = _ws(problem, Op.QUANTIZE_KV_FP8, ws)
    _check(_lib.msa_quantize_kv_fp8(ctypes.byref(problem.c()), _ptr(k), _ptr(v), _ptr(k8), _ptr(v8), _ptr(k_scale),
                                    _ptr(v_scale), _ptr(ws), nws, _stream()), "msa_quantize_kv_fp8")
    return k8, v8, k_scale, v_scale


def _attn_fp8(fn, op, where, problem, q, k8, v8, k_scale, v_scale, idx, o, lse, ws):
    _need(q, torch.bfloat16, "q")
    _need(k8, torch.uint8, "k8")
    _need(v8, torch.uint8, "v8")
    _need(k_scale, torch.float32, "k_scale")
    _need(v_scale, torch.float32, "v_scale")
    _need(idx, torch.int32, "idx")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=q.device)
    ws, nws = _ws(problem, op, ws)
    _check(fn(ctypes.byref(problem.c()), _ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale), _ptr(v_scale), _ptr(idx),
              _ptr(o), _ptr(lse), _ptr(ws), nws, _stream()), where)
    return o, lse


def msa_sparse_attn_prefill_fp8(problem: Problem, q, k8, v8, k_scale, v_scale, idx, o=None, lse=None, ws=None):
    return _attn_fp8(_lib.msa_sparse_attn_prefill_fp8, Op.SPARSE_ATTN_PREFILL_FP8, "msa_sparse_attn_prefill_fp8",
                     problem, q, k8, v8, k_scale, v_scale, idx, o, lse, ws)


def msa_sparse_attn_decode_fp8(problem: Problem, q, k8, v8, k_scale, v_scale, idx, o=None, lse=None, ws=None):
    return _attn_fp8(_lib.msa_sparse_attn_decode_fp8, Op.SPARSE_ATTN_DECODE_FP8, "msa_sparse_attn_decode_fp8",
                     problem, q, k8, v8, k_scale, v_scale, idx, o, lse, ws)


def msa_forward_fp8(problem: Problem, q, k8, v8, k_scale, v_scale, q_idx, k_idx, idx=None, o=None, lse=None,
                    ws=None):
    """msa_forward with fp8 K/V for the Main Branch.  Returns (idx, o, lse)."""
    for t, n in ((q, "q"), (q_idx, "q_idx"), (k_idx, "k_idx")):
        _need(t, torch.bfloat16, n)
    for t, n in ((k8, "k8"), (v8, "v8")):
        _need(t, torch.uint8, n)
    _need(k_scale, torch.float32, "k_scale")
    _need(v_scale, torch.float32, "v_scale")
    dev = q.device
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=dev)
    ws, nws = _ws(problem, Op.FORWARD_FP8, ws)
    _check(_lib.msa_forward_fp8(ctypes.byref(problem.c()), _ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale), _ptr(v_scale),
                                _ptr(q_idx), _ptr(k_idx), _ptr(idx), _ptr(o), _ptr(lse), _ptr(ws), nws, _stream()),
           "msa_forward_fp8")
    return idx, o, lse


def msa_forward_decode_paged_fp8(problem: Problem, q, k8_cache, v8_cache, k_scale, v_scale, q_idx, k_idx_cache,
                                 block_table, idx=None, o=None, lse=None, ws=None):
    """Decode from paged fp8 caches: E4M3 codes [num_pages * 128, hkv, 128] with one scale row per page
    (k_scale / v_scale [num_pages, hkv]); bf16 q, q_idx and index-key cache; block_table int32
    [num_seqs, max_blocks].  Returns (idx, o, lse) as msa_forward."""
    for t, n in ((q, "q"), (q_idx, "q_idx"), (k_idx_cache, "k_idx_cache")):
        _need(t, torch.bfloat16, n)
    for t, n in ((k8_cache, "k8_cache"), (v8_cache, "v8_cache")):
        _need(t, torch.uint8, n)
    _need(k_scale, torch.float32, "k_scale")
    _need(v_scale, torch.float32, "v_scale")
    _need(block_table, torch.int32, "block_table")
    if block_table.dim() != 2 or k8_cache.shape[0] % 128:
        raise ValueError("block_table must be [num_seqs, max_blocks] and the caches whole pages of 128 rows")
    n_pages = k8_cache.shape[0] // 128
    if k_scale.numel() < n_pages * problem.hkv or v_scale.numel() < n_pages * problem.hkv:
        raise ValueError("k_scale and v_scale need one row of num_kv_heads scales per page")
    dev = q.device
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=dev)
    ws, nws = _ws(problem, Op.FORWARD_FP8, ws)
    _check(_lib.msa_forward_decode_paged_fp8(ctypes.byref(problem.c()), _ptr(q), _ptr(k8_cache), _ptr(v8_cache),
                                             _ptr(k_scale), _ptr(v_scale), _ptr(q_idx), _ptr(k_idx_cache),
                                             _ptr(block_table), block_table.shape[1], n_pages, _ptr(idx), _ptr(o),
                                             _ptr(lse), _ptr(ws), nws, _stream()), "msa_forward_decode_paged_fp8")
    return idx, o, lse


def msa_quantize_index_fp8(problem: Problem, q_idx=None, k_idx=None, q_idx8=None, q_idx_scale=None, k_idx8=None,
                           k_idx_scale=None, ws=None):
    """bf16 Q_idx [total_q, Hkv, 128] and/or K_idx [total_k, 128] -> E4M3 codes (uint8, same shapes) with fp32
    scales: q_idx_scale [total_q, Hkv] (one per query row and group), k_idx_scale [key blocks] (one per key block
    of a sequence).  Either input may be None (that side is skipped and its outputs returned as None unless given).
    Returns (q_idx8, q_idx_scale, k_idx8, k_idx_scale)."""
    if q_idx is None and k_idx is None:
        raise ValueError("nothing to quantize: q_idx and k_idx are both None")
    if q_idx is not None:
        _need(q_idx, torch.bfloat16, "q_idx")
        dev = q_idx.device
        if q_idx8 is None:
            q_idx8 = torch.empty(q_idx.shape, dtype=torch.uint8, device=dev)
        if q_idx_scale is None:
            q_idx_scale = torch.empty(q_idx.shape[:2], dtype=torch.float32, device=dev)
    if k_idx is not None:
        _need(k_idx, torch.bfloat16, "k_idx")
        dev = k_idx.device
        if k_idx8 is None:
            k_idx8 = torch.empty(k_idx.shape, dtype=torch.uint8, device=dev)
        if k_idx_scale is None:
            k_idx_scale = torch.zeros(fp8_scale_rows(problem), dtype=torch.float32, device=dev)
    ws, nws = _ws(problem, Op.QUANTIZE_INDEX_FP8, ws)
    _check(_lib.msa_quantize_index_fp8(ctypes.byref(problem.c()), _ptr(q_idx), _ptr(k_idx),
                                       _ptr(q_idx8 if q_idx is not None else None),
                                       _ptr(q_idx_scale if q_idx is not None else None),
                                       _ptr(k_idx8 if k_idx is not None else None),
                                       _ptr(k_idx_scale if k_idx is not None else None), _ptr(ws), nws, _stream()),
           "msa_quantize_index_fp8")
    return q_idx8, q_idx_scale, k_idx8, k_idx_scale


def _need_fp8_index(q_idx8, q_idx_scale, k_idx8, k_idx_scale):
    _need(q_idx8, torch.uint8, "q_idx8")
    _need(k_idx8, torch.uint8, "k_idx8")
    _need(q_idx_scale, torch.float32, "q_idx_scale")
    _need(k_idx_scale, torch.float32, "k_idx_scale")


def msa_index_pool_fp8(problem: Problem, q_idx8, q_idx_scale, k_idx8, k_idx_scale, pooled=None, ws=None):
    """msa_index_pool over fp8 index inputs: pooled fp32 [total_q * hkv, ceil(max_k / 128)] (entries past a row's
    causal end are left as they were, NaN when ``pooled`` is allocated here)."""
    _need_fp8_index(q_idx8, q_idx_scale, k_idx8, k_idx_scale)
    if pooled is None:
        pooled = torch.full((problem.total_q * problem.hkv, max_blocks(problem)), float("nan"), dtype=torch.float32,
                            device=q_idx8.device)
    ws, nws = _ws(problem, Op.INDEX_POOL, ws)
    _check(_lib.msa_index_pool_fp8(ctypes.byref(problem.c()), _ptr(q_idx8), _ptr(q_idx_scale), _ptr(k_idx8),
                                   _ptr(k_idx_scale), _ptr(pooled), pooled.stride(0), _ptr(ws), nws, _stream()),
           "msa_index_pool_fp8")
    return pooled


def msa_index_topk_fp8(problem: Problem, q_idx8, q_idx_scale, k_idx8, k_idx_scale, idx=None, ws=None):
    """msa_index_topk over fp8 index inputs.  Returns idx [total_q, Hkv, topk] int32."""
    _need_fp8_index(q_idx8, q_idx_scale, k_idx8, k_idx_scale)
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=q_idx8.device)
    _need(idx, torch.int32, "idx")
    ws, nws = _ws(problem, Op.INDEX_TOPK, ws)
    _check(_lib.msa_index_topk_fp8(ctypes.byref(problem.c()), _ptr(q_idx8), _ptr(q_idx_scale), _ptr(k_idx8),
                                   _ptr(k_idx_scale), _ptr(idx), _ptr(ws), nws, _stream()), "msa_index_topk_fp8")
    return idx


def msa_forward_fp8_index(problem: Problem, q, k8, v8, k_scale, v_scale, q_idx8, q_idx_scale, k_idx8, k_idx_scale,
                          idx=None, o=None, lse=None, ws=None):
    """msa_forward_fp8 with the Index Branch on fp8 inputs too.  Returns (idx, o, lse)."""
    _need(q, torch.bfloat16, "q")
    for t, n in ((k8, "k8"), (v8, "v8")):
        _need(t, torch.uint8, n)
    _need(k_scale, torch.float32, "k_scale")
    _need(v_scale, torch.float32, "v_scale")
    _need_fp8_index(q_idx8, q_idx_scale, k_idx8, k_idx_scale)
    dev = q.device
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=dev)
    ws, nws = _ws(problem, Op.FORWARD_FP8, ws)
    _check(_lib.msa_forward_fp8_index(ctypes.byref(problem.c()), _ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale),
                                      _ptr(v_scale), _ptr(q_idx8), _ptr(q_idx_scale), _ptr(k_idx8), _ptr(k_idx_scale),
                                      _ptr(idx), _ptr(o), _ptr(lse), _ptr(ws), nws, _stream()),
           "msa_forward_fp8_index")
    return idx, o, lse


def msa_forward_decode_paged_fp8_index(problem: Problem, q, k8_cache, v8_cache, k_scale, v_scale, q_idx8,
                                       q_idx_scale, k_idx8_cache, k_idx_scale, block_table, idx=None, o=None,
                                       lse=None, ws=None):
    """Decode from paged fp8 caches with the index keys in fp8 too: K/V codes [num_pages * 128, hkv, 128] with
    scales [num_pages, hkv]; index-key codes [num_pages * 128, 128] with scales [num_pages]; q_idx8 / q_idx_scale
    for the queries; block_table int32 [num_seqs, max_blocks].  Returns (idx, o, lse) as msa_forward."""
    _need(q, torch.bfloat16, "q")
    for t, n in ((k8_cache, "k8_cache"), (v8_cache, "v8_cache")):
        _need(t, torch.uint8, n)
    _need(k_scale, torch.float32, "k_scale")
    _need(v_scale, torch.float32, "v_scale")
    _need_fp8_index(q_idx8, q_idx_scale, k_idx8_cache, k_idx_scale)
    _need(block_table, torch.int32, "block_table")
    if block_table.dim() != 2 or k8_cache.shape[0] % 128 or k_idx8_cache.shape[0] != k8_cache.shape[0]:
        raise ValueError("block_table must be [num_seqs, max_blocks] and the caches whole pages of 128 rows")
    n_pages = k8_cache.shape[0] // 128
    if k_scale.numel() < n_pages * problem.hkv or v_scale.numel() < n_pages * problem.hkv or \
            k_idx_scale.numel() < n_pages:
        raise ValueError("the scale arrays need one row per page")
    dev = q.device
    if idx is None:
        idx = torch.empty((problem.total_q, problem.hkv, problem.topk), dtype=torch.int32, device=dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((problem.total_q, problem.hq), dtype=torch.float32, device=dev)
    ws, nws = _ws(problem, Op.FORWARD_FP8, ws)
    _check(_lib.msa_forward_decode_paged_fp8_index(
        ctypes.byref(problem.c()), _ptr(q), _ptr(k8_cache), _ptr(v8_cache), _ptr(k_scale), _ptr(v_scale), _ptr(q_idx8),
        _ptr(q_idx_scale), _ptr(k_idx8_cache), _ptr(k_idx_scale), _ptr(block_table), block_table.shape[1], n_pages,
        _ptr(idx), _ptr(o), _ptr(lse), _ptr(ws), nws, _stream()), "msa_forward_decode_paged_fp8_index")
    return idx, o, lse


def msa_read_device_status(ws: Optional[torch.Tensor]) -> int:
    """MSA_DEVICE_* flags of the last call on workspace ``ws`` (None: of the last
    msa_sparse_attn_decode_static call on the current device).  Synchronises the stream."""
    flags = ctypes.c_uint32(0)
    _check(_lib.msa_read_device_status(_ptr(ws), ctypes.byref(flags), _stream()), "msa_read_device_status")
    return int(flags.value)


def abi_version() -> int:
    return int(_lib.msa_abi_version())


def kernel_launch_count() -> int:
    """Kernels (and memsets) the library has enqueued in this process."""
    return int(_lib.msa_kernel_launch_count())


class StageTimer:
    """Per-stage CUDA events recorded by the library on the call's stream.

    Use as a context manager around calls; ``elapsed_ms()`` after a
    synchronize gives {stage: ms} for the stages of the last call.
    """

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(STAGES))]
        s = torch.cuda.current_stream()
        for e in self.events:      # materialise the underlying cudaEvent_t handles
            e.record(s)
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self.marks = set()

    def __enter__(self):
        _check(_lib.msa_set_stage_events(self._arr), "msa_set_stage_events")
        return self

    def __exit__(self, *exc):
        _lib.msa_set_stage_events(None)
        return False

    def elapsed_ms(self, stages=STAGES):
        out = {}
        for j, name in enumerate(STAGES):
            if name in stages:
                try:
                    out[name] = self.events[2 * j].elapsed_time(self.events[2 * j + 1])
                except RuntimeError:
                    pass
        return out
