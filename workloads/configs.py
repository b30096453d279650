"""Workload shapes.

Every workload is a packed batch of causal sequences given as (q_len, kv_len)
pairs; the queries of a sequence are its last q_len key positions.  Head
geometry follows the report's testbed (64 query heads, 4 KV heads, head dim
128; "MiniMax Sparse Attention: let each query pick its own blocks", section
"Two design choices"/GQA paragraph, and the atlas record's summary), block 128
and k = 16 ("The mechanism, precisely").  The index head dimension is not given
by the pages; 128 is used (64 for the tiny case).
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Tuple


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seqs: Optional[Tuple[Tuple[int, int], ...]]  # fixed (q_len, kv_len) list, or None -> seq_fn
    hq: int = 64
    hkv: int = 4
    head_dim: int = 128
    d_idx: int = 128
    block: int = 128
    topk: int = 16
    n_topics: int = 64
    seed: int = 1000
    decode_batch: int = 0          # >0: decode batch, kv_len = decode_ctx - block + U{1..block}
    decode_ctx: int = 0
    description: str = ""

    @property
    def is_decode(self) -> bool:
        return self.decode_batch > 0


CONFIGS = {
    "tiny": Workload(
        "tiny", ((2048, 2048),), hq=16, hkv=2, d_idx=64, topk=4, n_topics=8, seed=1000,
        description="T=N=2048 causal, Hq 16 / Hkv 2, d_idx 64, k 4 (incl. local), 8 topics"),
    "prefill_32k": Workload(
        "prefill_32k", ((32768, 32768),), seed=1001,
        description="T=N=32768 causal, Hq 64 / Hkv 4, d_idx 128, k 16, 64 topics"),
    "decode_128k": Workload(
        "decode_128k", None, seed=1002, decode_batch=64, decode_ctx=131072,
        description="64 sequences x 1 query, KV cache 131072-128+U{1..128}, k 16, 64 topics"),
    "varlen": Workload(
        "varlen", ((16384, 16384), (24576, 24576), (40960, 40960), (65536, 65536)), seed=1003,
        description="4 packed causal sequences 16384/24576/40960/65536, k 16, 64 topics"),
    "chunked_1m": Workload(
        "chunked_1m", ((8192, 1048576),), n_topics=256, seed=1004,
        description="last 8192 queries of a 1048576-token causal sequence, k 16, 256 topics"),
    "decode_1m": Workload(
        "decode_1m", None, n_topics=256, seed=1014, decode_batch=8, decode_ctx=1048576,
        description="8 sequences x 1 query, KV cache 1048576-128+U{1..128}, k 16, 256 topics"),
    "prefill_16k": Workload(
        "prefill_16k", ((16384, 16384),), seed=1016,
        description="T=N=16384 causal, Hq 64 / Hkv 4, d_idx 128, k 16, 64 topics (profiling size)"),
    "decode_64k": Workload(
        "decode_64k", None, seed=1017, decode_batch=16, decode_ctx=65536,
        description="16 sequences x 1 query, KV cache 65536-128+U{1..128}, k 16, 64 topics (profiling size)"),
    "prefill_128k": Workload(
        "prefill_128k", ((131072, 131072),), seed=1010,
        description="T=N=131072 causal, Hq 64 / Hkv 4, d_idx 128, k 16, 64 topics"),
}


def get(name: str) -> Workload:
    return CONFIGS[name]


def small(name: str, seqs, **kw) -> Workload:
    """An ad-hoc workload for tests (same recipe, caller-chosen shapes)."""
    return Workload(name, tuple(tuple(s) for s in seqs), **kw)
