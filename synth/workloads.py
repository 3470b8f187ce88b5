"""Seeded synthetic workloads shaped like the ones the pages describe.

Five workloads (W1..W5) mirror the shapes on the pages: Llama-2-7B-like heads
(32 heads, head_dim 128), 2K-32K contexts, page size 16 ("Transformer
推理的内存布局优化" page, section 二; "LLM推理中的KV缓存优化技术与TinyServe实践"
page, section 5.1), outlier channels 10-20x larger than the rest (memory-layout
page, section 二) and pages that differ in relevance (TinyServe page, section 1).
No dataset or trained weights are involved: every value is drawn here.

Every array is a pure function of (workload seed, sequence index, layer, tag),
so one sequence can be regenerated on its own to check a sampled output.
Values are rounded once to the storage dtype (fp16 or bf16, round to nearest
even) and returned both as 16-bit storage and as the exact fp32 widening.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to_dtype(x: np.ndarray, dtype: str) -> Tuple[np.ndarray, np.ndarray]:
    """Round fp32 draws to the storage dtype. Returns (uint16 storage bits, exact fp32 values)."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        h = x.astype(np.float16)
        return h.view(np.uint16), h.astype(np.float32)
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x)
        return bits, bf16_bits_to_f32(bits)
    raise ValueError(f"unknown dtype {dtype}")


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes and value recipe of one synthetic decode workload."""
    name: str
    seed: int
    batch: int
    layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str                      # source dtype of q and of the K/V tokens
    quant: str                      # "none" | "per_token" | "per_group64" | "per_token_u4"
    seq_len: Optional[int]          # fixed context length, or None for a drawn mix
    seq_len_range: Optional[Tuple[int, int]] = None
    pool_pages: Optional[int] = None   # physical pages per layer (None: as needed)
    pool_spare: int = 0                # extra free pages (append workloads)
    outlier_channels: int = 0          # channels per kv head scaled by outlier_scale (K only)
    outlier_scale: float = 1.0
    page_offset_std: float = 0.0       # per-(seq, page, head) K offset, std per channel
    top_k_ratio: Optional[float] = None
    append_steps: int = 0
    description: str = ""

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))


WORKLOADS: Dict[str, Workload] = {
    "w1_tiny_f16": Workload(
        name="w1_tiny_f16", seed=1235, batch=1, layers=1, num_q_heads=4, num_kv_heads=4,
        head_dim=64, page_size=16, dtype="f16", quant="none", seq_len=256, pool_pages=32,
        description="tiny dense fp16: B=1, 4 q = 4 kv heads, d=64, L=256, page 16, "
                    "16 pages drawn from a 32-page pool"),
    "w2_llama7b_bf16": Workload(
        name="w2_llama7b_bf16", seed=1236, batch=4, layers=32, num_q_heads=32, num_kv_heads=32,
        head_dim=128, page_size=16, dtype="bf16", quant="none", seq_len=2048, pool_pages=512,
        description="Llama-2-7B-shaped dense bf16 decode: B=4, 32 layers, 32 = 32 heads, "
                    "d=128, L=2048, page 16, 512-page pool per layer"),
    "w3_gqa_int8_token": Workload(
        name="w3_gqa_int8_token", seed=1237, batch=16, layers=1, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, dtype="f16", quant="per_token", seq_len=None,
        seq_len_range=(1024, 32768), outlier_channels=4, outlier_scale=15.0,
        description="GQA 32/8 per-token INT8: B=16, d=128, L ~ U[1024, 32768], page 16, "
                    "4 of 128 K channels per kv head x15"),
    "w4_long_int8_group": Workload(
        name="w4_long_int8_group", seed=1238, batch=2, layers=1, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=256, dtype="f16", quant="per_group64", seq_len=32768,
        pool_spare=8, outlier_channels=4, outlier_scale=15.0, append_steps=64,
        description="long-context GQA 32/8 per-64-token-group INT8 with append: B=2, d=128, "
                    "L=32768, page 256, 1 token appended per sequence per step"),
    "w5_sparse_f16": Workload(
        name="w5_sparse_f16", seed=1239, batch=8, layers=1, num_q_heads=16, num_kv_heads=16,
        head_dim=64, page_size=16, dtype="f16", quant="none", seq_len=16384, pool_pages=8192,
        page_offset_std=0.5, top_k_ratio=0.3,
        description="query-aware sparse: B=8, 16 = 16 heads, d=64, L=16384, page 16 "
                    "(1024 pages/seq), per-page K offset ~ N(0, 0.5^2), top-K 30%"),
    "w6_gqa_sparse_int8": Workload(
        name="w6_gqa_sparse_int8", seed=1241, batch=8, layers=1, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, dtype="f16", quant="per_token", seq_len=16384,
        outlier_channels=4, outlier_scale=15.0, page_offset_std=0.5, top_k_ratio=0.3,
        description="GQA 32/8 per-token INT8 sparse: B=8, d=128, L=16384, page 16, per-page K "
                    "offset ~ N(0, 0.5^2), top-K 30 % per kv head from the group's summed scores"),
    "w7_gqa_u4_token": Workload(
        name="w7_gqa_u4_token", seed=1242, batch=16, layers=1, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, dtype="f16", quant="per_token_u4", seq_len=None,
        seq_len_range=(1024, 32768), outlier_channels=4, outlier_scale=15.0,
        description="GQA 32/8 per-token 4-bit KV: B=16, d=128, L ~ U[1024, 32768], page 16, "
                    "4 of 128 K channels per kv head x15 (the GQA INT8 workload's shapes)"),
    "dense_32k_bf16": Workload(
        name="dense_32k_bf16", seed=1240, batch=4, layers=1, num_q_heads=32, num_kv_heads=32,
        head_dim=128, page_size=16, dtype="bf16", quant="none", seq_len=32768,
        description="dense bf16 at 32K context: B=4, 32 = 32 heads, d=128, page 16, 1 layer"),
}


def _rng(w: Workload, *tags: int) -> np.random.Generator:
    return np.random.default_rng([w.seed, *tags])


_TAG_LENS, _TAG_OUTLIER, _TAG_K, _TAG_V, _TAG_Q, _TAG_BT, _TAG_OFF, _TAG_APPEND = range(8)


def seq_lens(w: Workload) -> np.ndarray:
    """Context length of every sequence (int32 [B])."""
    if w.seq_len is not None:
        return np.full(w.batch, w.seq_len, dtype=np.int32)
    lo, hi = w.seq_len_range
    return _rng(w, _TAG_LENS).integers(lo, hi, size=w.batch, endpoint=True).astype(np.int32)


def outlier_channels(w: Workload) -> np.ndarray:
    """Outlier channel indices per kv head (int [Hkv][n]); the same for every token."""
    if w.outlier_channels == 0:
        return np.zeros((w.num_kv_heads, 0), dtype=np.int64)
    r = _rng(w, _TAG_OUTLIER)
    return np.stack([np.sort(r.choice(w.head_dim, w.outlier_channels, replace=False))
                     for _ in range(w.num_kv_heads)])


@dataclasses.dataclass
class SeqData:
    """Tokens of one sequence in one layer: storage bits and exact fp32 values."""
    k_bits: np.ndarray   # uint16 [L][Hkv][d]
    v_bits: np.ndarray
    k: np.ndarray        # float32 [L][Hkv][d] (exact widening of the storage values)
    v: np.ndarray


def _draw_kv(w: Workload, n: int, r_k: np.random.Generator, r_v: np.random.Generator,
             first_token: int, offsets: Optional[np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
    H, d = w.num_kv_heads, w.head_dim
    k = r_k.standard_normal((n, H, d), dtype=np.float32)
    v = r_v.standard_normal((n, H, d), dtype=np.float32)
    if w.outlier_channels:
        oc = outlier_channels(w)
        for g in range(H):
            k[:, g, oc[g]] *= np.float32(w.outlier_scale)
    if offsets is not None:
        # offsets: [num_pages][Hkv][d], added to every token of the page
        page = (first_token + np.arange(n)) // w.page_size
        k += offsets[page]
    return k, v


def seq_tokens(w: Workload, b: int, layer: int = 0, length: Optional[int] = None) -> SeqData:
    """The first `length` (default: the context length) tokens of sequence b."""
    L = int(seq_lens(w)[b]) if length is None else int(length)
    offsets = None
    if w.page_offset_std > 0:
        n_pages = -(-L // w.page_size)
        offsets = (_rng(w, _TAG_OFF, b, layer).standard_normal(
            (n_pages, w.num_kv_heads, w.head_dim), dtype=np.float32) * np.float32(w.page_offset_std))
    k, v = _draw_kv(w, L, _rng(w, _TAG_K, b, layer), _rng(w, _TAG_V, b, layer), 0, offsets)
    kb, kf = round_to_dtype(k, w.dtype)
    vb, vf = round_to_dtype(v, w.dtype)
    return SeqData(kb, vb, kf, vf)


def append_tokens(w: Workload, b: int, step: int, layer: int = 0) -> SeqData:
    """The token appended to sequence b at decode step `step` (shape [1][Hkv][d])."""
    k, v = _draw_kv(w, 1, _rng(w, _TAG_APPEND, b, layer, step, 0),
                    _rng(w, _TAG_APPEND, b, layer, step, 1), 0, None)
    kb, kf = round_to_dtype(k, w.dtype)
    vb, vf = round_to_dtype(v, w.dtype)
    return SeqData(kb, vb, kf, vf)


def queries(w: Workload, layer: int = 0, step: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Decode queries [B][Hq][d]: (uint16 storage bits, exact fp32 values)."""
    q = _rng(w, _TAG_Q, layer, step).standard_normal(
        (w.batch, w.num_q_heads, w.head_dim), dtype=np.float32)
    return round_to_dtype(q, w.dtype)


def block_tables(w: Workload, layer: int = 0, extra_pages: int = 0) -> Tuple[np.ndarray, int]:
    """Seeded non-contiguous block tables.

    Returns (int32 [B][max_pages] physical page ids, pool size). Unused entries
    are -1. The pool is a seeded permutation: W1 takes the first 16 ids of a
    permuted 32-page pool, W2 reshapes a permutation of its 512-page pool to
    [4][128], the others permute exactly the pages they need plus any spare.
    `extra_pages` reserves that many more logical pages per sequence (append).
    """
    lens = seq_lens(w)
    ps = w.page_size
    need = [-(-int(L) // ps) + extra_pages for L in lens]
    max_pages = max(need)
    r = _rng(w, _TAG_BT, layer)
    total = sum(need)
    pool = w.pool_pages if w.pool_pages is not None else total + w.pool_spare
    if pool < total:
        raise ValueError("pool too small")
    perm = r.permutation(pool).astype(np.int32)
    bt = np.full((w.batch, max_pages), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    return bt, pool


def make_workload(name: str) -> Workload:
    return WORKLOADS[name]


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


def cache_kind(w: Workload) -> Tuple[str, str]:
    """(storage dtype name, quantisation name) of a workload's cache."""
    if w.quant == "none":
        return w.dtype, "none"
    if w.quant == "per_token_u4":
        return "u4", "per_token"
    return "int8", w.quant
