"""CPU oracle of the MiniMax Sparse Attention forward pass (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this package.  The product library never imports it, and it
imports nothing from the product.  The arithmetic lives in ``msa_oracle.c``
(plain C, one loop nest per step of the method); this module only marshals
numpy arrays into it.

Steps and their sources ("MiniMax Sparse Attention: let each query pick its own
blocks", section "The mechanism, precisely", and its Figure 1):
  * ``pooled``    -- index scores Q_idx . K_idx^T, max-pooled per block, causal;
  * ``select``    -- top-k blocks by (score desc, index asc), local block forced;
  * ``attention`` -- exact softmax attention over the selected blocks' tokens;
  * ``index``     -- ``pooled`` then ``select`` (the Index Branch alone);
  * ``forward``   -- the three chained;
  * ``index_prologue`` -- hidden states to index heads: projection, RMSNorm,
    RoPE on the first 64 dims (Figure 1's Index Branch input; the reading is
    stated in ``msa_oracle.c``);
  * ``quantize_fp8``, ``e4m3_value``, ``e4m3_code``, ``attention_fp8`` -- fp8
    (E4M3) K/V with one scale per (key block, KV head), and the Main Branch
    over such K/V (the atlas record of the report: the kernels "also support
    fp8"; the format is a reading, see ``msa_oracle.c``);
  * ``quantize_index_fp8``, ``pooled_fp8``, ``index_fp8`` -- the same codes for
    the index inputs (K_idx: one scale per key block; Q_idx: one per query row
    and group), and the Index Branch over them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def build() -> str:
    """Compile ``msa_oracle.c`` (gcc + OpenMP) if the library is missing or stale."""
    src = os.path.join(_HERE, "msa_oracle.c")
    if (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        subprocess.run(["make", "-s", "-C", _HERE], check=True)
    return _LIB_PATH


def _load(path: str | None = None):
    """Load the oracle library (``path`` overrides the default build, for mutation tests)."""
    global _lib
    with _lock:
        if path is not None:
            _lib = None
        if _lib is None:
            lib = ctypes.CDLL(path or build())
            lib.msa_oracle_pooled.argtypes = [
                ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _u16p, _u16p, ctypes.c_int, _i32p, ctypes.c_int, _f32p]
            lib.msa_oracle_select.argtypes = [ctypes.c_int, _f32p, ctypes.c_int, _i32p, _f64p]
            lib.msa_oracle_attention.argtypes = [
                ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_double, _u16p, _u16p, _u16p, _i32p, ctypes.c_int, _i32p,
                _f64p, _f64p]
            lib.msa_oracle_forward.argtypes = [
                ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, _u16p, _u16p, _u16p, _u16p, _u16p,
                ctypes.c_int, _i32p, _i32p, _f64p, _f64p, _f64p]
            lib.msa_oracle_index.argtypes = [
                ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _u16p, _u16p, ctypes.c_int, _i32p, _i32p, _f64p]
            lib.msa_oracle_pooled_fp8.argtypes = [
                ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _u8p, _f32p, _u8p, _f32p, ctypes.c_int, _i32p, ctypes.c_int, _f32p]
            lib.msa_oracle_index_fp8.argtypes = [
                ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _u8p, _f32p, _u8p, _f32p, ctypes.c_int, _i32p, _i32p, _f64p]
            lib.msa_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.msa_oracle_e4m3_value.restype = ctypes.c_double
            lib.msa_oracle_e4m3_code.argtypes = [ctypes.c_float]
            lib.msa_oracle_e4m3_code.restype = ctypes.c_uint8
            lib.msa_oracle_key_blocks.argtypes = [ctypes.c_int, _i32p, ctypes.c_int]
            lib.msa_oracle_quantize_fp8.argtypes = [ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    _u16p, _u8p, _f32p]
            lib.msa_oracle_attention_fp8.argtypes = [
                ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_double, _u16p, _u8p, _u8p, _f32p, _f32p, _i32p, ctypes.c_int, _i32p,
                _f64p, _f64p]
            lib.msa_oracle_index_prologue.argtypes = [
                ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, _u16p, _u16p, _u16p, _u16p, _u16p, ctypes.c_int, _i32p,
                _f64p, _f64p]
            for fn in (lib.msa_oracle_pooled, lib.msa_oracle_select, lib.msa_oracle_attention,
                       lib.msa_oracle_forward, lib.msa_oracle_index, lib.msa_oracle_key_blocks,
                       lib.msa_oracle_quantize_fp8, lib.msa_oracle_attention_fp8, lib.msa_oracle_index_prologue,
                       lib.msa_oracle_pooled_fp8, lib.msa_oracle_index_fp8):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def use_library(path: str | None):
    """Switch to another build of ``msa_oracle.c`` (None: back to the default one)."""
    global _lib
    with _lock:
        _lib = None
    if path is not None:
        _load(path)


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctype)
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctype)


def _bits(a) -> np.ndarray:
    """bf16 data as raw uint16 bits.  Accepts a torch bf16 tensor or a uint16 array."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # local: only needed when a torch tensor is passed
    assert a.dtype == torch.bfloat16, a.dtype
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    a = np.asarray(a)
    return np.ascontiguousarray(a.astype(np.int32, copy=False))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def max_blocks(cu_k: np.ndarray, block: int) -> int:
    kv = np.diff(_i32(cu_k))
    return int(max(1, ((kv.max() - 1) // block + 1) if kv.size and kv.max() > 0 else 1))


def pooled(cu_q, cu_k, q_idx, k_idx, block: int, rows=None, nb_stride: int | None = None) -> np.ndarray:
    """Block max-pooled causal index scores, fp32 [n_rows, Hkv, nb_stride] (-inf past the causal end)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    qb, kb = _bits(q_idx), _bits(k_idx)
    total_q, hkv, d_idx = qb.shape
    rows_a = None if rows is None else _i32(rows)
    n_rows = total_q if rows_a is None else rows_a.size
    nb_stride = nb_stride or max_blocks(cu_k, block)
    out = np.empty((n_rows, hkv, nb_stride), np.float32)
    rc = _load().msa_oracle_pooled(len(cu_q) - 1, _ptr(cu_q, _i32p), _ptr(cu_k, _i32p), hkv, d_idx,
                                   block, _ptr(qb, _u16p), _ptr(kb, _u16p), n_rows,
                                   _ptr(rows_a, _i32p), nb_stride, _ptr(out, _f32p))
    _check(rc, "pooled")
    return out


def select(pooled_row: np.ndarray, nb: int, k: int):
    """Top-k of one pooled row (local block nb-1 forced).  Returns (idx[k] int32, gap float)."""
    row = np.ascontiguousarray(pooled_row, dtype=np.float32)
    assert row.size >= nb
    sel = np.empty(max(k, 1), np.int32)
    gap = ctypes.c_double(0.0)
    rc = _load().msa_oracle_select(nb, _ptr(row, _f32p), k, _ptr(sel, _i32p), ctypes.byref(gap))
    _check(rc, "select")
    return sel[:k], gap.value


def attention(cu_q, cu_k, q, k, v, idx, block: int, scale: float | None = None, rows=None):
    """Main Branch over given block indices.  Returns (o [n, Hq, D] f64, lse [n, Hq] f64)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    total_q, hq, head_dim = qb.shape
    hkv = kb.shape[1]
    idx_a = _i32(idx)
    topk = idx_a.shape[-1]
    rows_a = None if rows is None else _i32(rows)
    n_rows = total_q if rows_a is None else rows_a.size
    assert idx_a.shape == (n_rows, hkv, topk)
    scale = float(head_dim ** -0.5 if scale is None else scale)
    o = np.empty((n_rows, hq, head_dim), np.float64)
    lse = np.empty((n_rows, hq), np.float64)
    rc = _load().msa_oracle_attention(len(cu_q) - 1, _ptr(cu_q, _i32p), _ptr(cu_k, _i32p), hq, hkv,
                                      head_dim, block, topk, scale, _ptr(qb, _u16p), _ptr(kb, _u16p),
                                      _ptr(vb, _u16p), _ptr(idx_a, _i32p), n_rows,
                                      _ptr(rows_a, _i32p), _ptr(o, _f64p), _ptr(lse, _f64p))
    _check(rc, "attention")
    return o, lse


def index(cu_q, cu_k, q_idx, k_idx, block: int, topk: int, rows=None):
    """Index Branch only (pooled scores, then selection).  Returns dict(idx [n,Hkv,k] i32, gap [n,Hkv] f64)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    qib, kib = _bits(q_idx), _bits(k_idx)
    total_q, hkv, d_idx = qib.shape
    rows_a = None if rows is None else _i32(rows)
    n_rows = total_q if rows_a is None else rows_a.size
    idx = np.empty((n_rows, hkv, topk), np.int32)
    gap = np.empty((n_rows, hkv), np.float64)
    rc = _load().msa_oracle_index(len(cu_q) - 1, _ptr(cu_q, _i32p), _ptr(cu_k, _i32p), hkv, d_idx, block, topk,
                                  _ptr(qib, _u16p), _ptr(kib, _u16p), n_rows, _ptr(rows_a, _i32p),
                                  _ptr(idx, _i32p), _ptr(gap, _f64p))
    _check(rc, "index")
    return {"idx": idx, "gap": gap}


def forward(cu_q, cu_k, q, k, v, q_idx, k_idx, block: int, topk: int, scale: float | None = None,
            rows=None):
    """All three steps.  Returns dict(idx [n,Hkv,k] i32, gap [n,Hkv] f64, o [n,Hq,D] f64, lse [n,Hq] f64)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    qb, kb, vb, qib, kib = _bits(q), _bits(k), _bits(v), _bits(q_idx), _bits(k_idx)
    total_q, hq, head_dim = qb.shape
    hkv = kb.shape[1]
    d_idx = qib.shape[2]
    rows_a = None if rows is None else _i32(rows)
    n_rows = total_q if rows_a is None else rows_a.size
    scale = float(head_dim ** -0.5 if scale is None else scale)
    idx = np.empty((n_rows, hkv, topk), np.int32)
    gap = np.empty((n_rows, hkv), np.float64)
    o = np.empty((n_rows, hq, head_dim), np.float64)
    lse = np.empty((n_rows, hq), np.float64)
    rc = _load().msa_oracle_forward(len(cu_q) - 1, _ptr(cu_q, _i32p), _ptr(cu_k, _i32p), hq, hkv,
                                    head_dim, d_idx, block, topk, scale, _ptr(qb, _u16p),
                                    _ptr(kb, _u16p), _ptr(vb, _u16p), _ptr(qib, _u16p),
                                    _ptr(kib, _u16p), n_rows, _ptr(rows_a, _i32p), _ptr(idx, _i32p),
                                    _ptr(gap, _f64p), _ptr(o, _f64p), _ptr(lse, _f64p))
    _check(rc, "forward")
    return {"idx": idx, "gap": gap, "o": o, "lse": lse}


def index_prologue(cu_q, cu_k, x, wq, wk, gamma_q, gamma_k, rope_dim: int = 64, rope_base: float = 10000.0,
                   eps: float = 1e-6, rows=None):
    """Index query / key heads of the new tokens (query rows) from their hidden states x [total_q, d_model] bf16,
    weights wq [hkv * d_idx, d_model], wk [d_idx, d_model], norm weights gamma_q, gamma_k [d_idx] (all bf16).
    Returns (q_idx [n, hkv, d_idx] f64, k_idx [n, d_idx] f64), unrounded; token i's key row is k_start + pos(i)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    xb, wqb, wkb, gqb, gkb = _bits(x), _bits(wq), _bits(wk), _bits(gamma_q), _bits(gamma_k)
    total_q, d_model = xb.shape
    d_idx = wkb.shape[0]
    hkv = wqb.shape[0] // d_idx
    rows_a = None if rows is None else _i32(rows)
    n_rows = total_q if rows_a is None else rows_a.size
    q_out = np.empty((n_rows, hkv, d_idx), np.float64)
    k_out = np.empty((n_rows, d_idx), np.float64)
    rc = _load().msa_oracle_index_prologue(len(cu_q) - 1, _ptr(cu_q, _i32p), _ptr(cu_k, _i32p), d_model, hkv, d_idx,
                                           rope_dim, float(rope_base), float(eps), _ptr(xb, _u16p), _ptr(wqb, _u16p),
                                           _ptr(wkb, _u16p), _ptr(gqb, _u16p), _ptr(gkb, _u16p), n_rows,
                                           _ptr(rows_a, _i32p), _ptr(q_out, _f64p), _ptr(k_out, _f64p))
    _check(rc, "index_prologue")
    return q_out, k_out


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code (NaN for the NaN codes)."""
    return float(_load().msa_oracle_e4m3_value(int(code)))


def e4m3_code(x: float) -> int:
    """E4M3 code of an fp32 value: nearest, ties to the even code, saturated to +-448."""
    return int(_load().msa_oracle_e4m3_code(float(np.float32(x))))


def key_blocks(cu_k, block: int) -> int:
    cu_k = _i32(cu_k)
    return int(_load().msa_oracle_key_blocks(len(cu_k) - 1, _ptr(cu_k, _i32p), block))


def _u8(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    a = np.asarray(a)
    assert a.dtype == np.uint8, a.dtype
    return np.ascontiguousarray(a)


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def quantize_fp8(cu_k, x, block: int):
    """fp8 copy of K or V ([total_k, Hkv, D] bf16): (codes uint8, same shape; scales fp32 [key blocks, Hkv])."""
    cu_k = _i32(cu_k)
    xb = _bits(x)
    total_k, hkv, head_dim = xb.shape
    codes = np.empty(xb.shape, np.uint8)
    scales = np.empty((key_blocks(cu_k, block), hkv), np.float32)
    rc = _load().msa_oracle_quantize_fp8(len(cu_k) - 1, _ptr(cu_k, _i32p), hkv, head_dim, block, _ptr(xb, _u16p),
                                         _ptr(codes, _u8p), _ptr(scales, _f32p))
    _check(rc, "quantize_fp8")
    return codes, scales


def attention_fp8(cu_q, cu_k, q, k8, v8, k_scale, v_scale, idx, block: int, scale: float | None = None, rows=None):
    """Main Branch over fp8 K/V (codes and per-(key block, KV head) scales).  Returns (o f64, lse f64)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    qb = _bits(q)
    k8a, v8a = _u8(k8), _u8(v8)
    ks, vs = _f32(k_scale), _f32(v_scale)
    total_q, hq, head_dim = qb.shape
    hkv = k8a.shape[1]
    idx_a = _i32(idx)
    topk = idx_a.shape[-1]
    rows_a = None if rows is None else _i32(rows)
    n_rows = total_q if rows_a is None else rows_a.size
    assert idx_a.shape == (n_rows, hkv, topk)
    assert ks.shape[0] >= key_blocks(cu_k, block) and vs.shape == ks.shape
    scale = float(head_dim ** -0.5 if scale is None else scale)
    o = np.empty((n_rows, hq, head_dim), np.float64)
    lse = np.empty((n_rows, hq), np.float64)
    rc = _load().msa_oracle_attention_fp8(len(cu_q) - 1, _ptr(cu_q, _i32p), _ptr(cu_k, _i32p), hq, hkv, head_dim,
                                          block, topk, scale, _ptr(qb, _u16p), _ptr(k8a, _u8p), _ptr(v8a, _u8p),
                                          _ptr(ks, _f32p), _ptr(vs, _f32p), _ptr(idx_a, _i32p), n_rows,
                                          _ptr(rows_a, _i32p), _ptr(o, _f64p), _ptr(lse, _f64p))
    _check(rc, "attention_fp8")
    return o, lse


def quantize_index_fp8(cu_q, cu_k, q_idx, k_idx, block: int):
    """fp8 copies of the index inputs: (q8 [total_q, Hkv, d_idx] uint8, q_scale [total_q, Hkv] fp32,
    k8 [total_k, d_idx] uint8, k_scale [key blocks] fp32).  K_idx is quantized per key block of a sequence,
    Q_idx per (query row, group): the same quantizer, the query rows taken as blocks of one row."""
    qb, kb = _bits(q_idx), _bits(k_idx)
    total_k, d_idx = kb.shape
    k8, k_scale = quantize_fp8(cu_k, kb.reshape(total_k, 1, d_idx), block)
    total_q = qb.shape[0]
    q8, q_scale = quantize_fp8(np.arange(total_q + 1, dtype=np.int32), qb, 1)
    return q8, q_scale, k8.reshape(total_k, d_idx), k_scale.reshape(-1)


def pooled_fp8(cu_q, cu_k, q8, q_scale, k8, k_scale, block: int, rows=None, nb_stride: int | None = None):
    """``pooled`` over E4M3 index inputs (codes and scales as ``quantize_index_fp8`` gives them)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    q8a, k8a, qs, ks = _u8(q8), _u8(k8), _f32(q_scale), _f32(k_scale)
    total_q, hkv, d_idx = q8a.shape
    assert k8a.shape == (int(cu_k[-1]), d_idx) and qs.shape == (total_q, hkv)
    assert ks.size >= key_blocks(cu_k, block)
    rows_a = None if rows is None else _i32(rows)
    n_rows = total_q if rows_a is None else rows_a.size
    nb_stride = nb_stride or max_blocks(cu_k, block)
    out = np.empty((n_rows, hkv, nb_stride), np.float32)
    rc = _load().msa_oracle_pooled_fp8(len(cu_q) - 1, _ptr(cu_q, _i32p), _ptr(cu_k, _i32p), hkv, d_idx, block,
                                       _ptr(q8a, _u8p), _ptr(qs, _f32p), _ptr(k8a, _u8p), _ptr(ks, _f32p), n_rows,
                                       _ptr(rows_a, _i32p), nb_stride, _ptr(out, _f32p))
    _check(rc, "pooled_fp8")
    return out


def index_fp8(cu_q, cu_k, q8, q_scale, k8, k_scale, block: int, topk: int, rows=None):
    """``index`` over E4M3 index inputs.  Returns dict(idx [n,Hkv,k] i32, gap [n,Hkv] f64)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    q8a, k8a, qs, ks = _u8(q8), _u8(k8), _f32(q_scale), _f32(k_scale)
    total_q, hkv, d_idx = q8a.shape
    assert k8a.shape == (int(cu_k[-1]), d_idx) and qs.shape == (total_q, hkv)
    assert ks.size >= key_blocks(cu_k, block)
    rows_a = None if rows is None else _i32(rows)
    n_rows = total_q if rows_a is None else rows_a.size
    idx = np.empty((n_rows, hkv, topk), np.int32)
    gap = np.empty((n_rows, hkv), np.float64)
    rc = _load().msa_oracle_index_fp8(len(cu_q) - 1, _ptr(cu_q, _i32p), _ptr(cu_k, _i32p), hkv, d_idx, block, topk,
                                      _ptr(q8a, _u8p), _ptr(qs, _f32p), _ptr(k8a, _u8p), _ptr(ks, _f32p), n_rows,
                                      _ptr(rows_a, _i32p), _ptr(idx, _i32p), _ptr(gap, _f64p))
    _check(rc, "index_fp8")
    return {"idx": idx, "gap": gap}


def query_positions(cu_q, cu_k) -> np.ndarray:
    """Key position of every packed query row (bottom-right alignment)."""
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    out = np.empty(int(cu_q[-1]), np.int64)
    for s in range(len(cu_q) - 1):
        ql, kl = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        out[cu_q[s]:cu_q[s + 1]] = kl - ql + np.arange(ql)
    return out
