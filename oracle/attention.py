"""Decode attention over one sequence's cached tokens, in fp64 (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition [KV-practice page, section 2.1]: Attention(Q, K, V) = softmax(Q K^T / sqrt(d)) V.
At decode time Q is the single new token's query, one row per query head, and
K, V are every cached token of the sequence. The paged layout only changes
where a token is stored [HBM-layout page, section 二 layout C]; the oracle
therefore works on tokens in logical order, and the tests gather the GPU pools
through the block table to compare.

GQA grouping (reading): query head h reads kv head h // G with
G = num_q_heads / num_kv_heads, i.e. consecutive query heads share one kv head
[Gemini page, section 3.1 groups query heads per kv head].
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import numpy as np


def decode_attention_tokens(q, k, v, sm_scale: float) -> np.ndarray:
    """One query vector against explicit token rows.

    q: [d]; k, v: [n][d]. Returns [d] (zeros when n == 0).
    x_t = sm_scale * (q . k_t); w = softmax(x) with the maximum subtracted;
    o = sum_t w_t v_t. All fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if k.shape[0] == 0:
        return np.zeros(q.shape[-1], dtype=np.float64)
    x = float(sm_scale) * (k @ q)
    w = np.exp(x - x.max())
    w = w / w.sum()
    return w @ v


def decode_attention(q, k, v, sm_scale: float) -> np.ndarray:
    """Dense decode attention for one sequence.

    q: [Hq][d]; k, v: [L][Hkv][d] (logical token order). Returns [Hq][d] fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    Hq = q.shape[0]
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros(q.shape, dtype=np.float64)
    for h in range(Hq):
        g = h // G
        out[h] = decode_attention_tokens(q[h], k[:, g, :], v[:, g, :], sm_scale)
    return out


def page_token_indices(pages: Sequence[int], page_size: int, length: int) -> np.ndarray:
    """Logical token ids held by the given logical pages (valid tokens only)."""
    idx = [np.arange(p * page_size, min((p + 1) * page_size, length)) for p in pages]
    return np.concatenate(idx) if idx else np.zeros(0, dtype=np.int64)


def sparse_decode_attention(q, k, v, sm_scale: float, selected: Sequence[Sequence[int]],
                            page_size: int) -> np.ndarray:
    """Attention restricted to the tokens of each query head's selected pages.

    selected[h]: logical page ids kept for query head h [TinyServe page,
    section 3.1 phase 3]; the softmax is renormalised over the kept tokens.
    """
    q = np.asarray(q, dtype=np.float64)
    Hq = q.shape[0]
    L, Hkv = k.shape[0], k.shape[1]
    G = Hq // Hkv
    out = np.zeros(q.shape, dtype=np.float64)
    for h in range(Hq):
        g = h // G
        t = page_token_indices(selected[h], page_size, L)
        out[h] = decode_attention_tokens(q[h], k[t, g, :], v[t, g, :], sm_scale)
    return out


def split_partials(q, k, v, sm_scale: float, bounds: Sequence[int]) -> List[Tuple[float, float, np.ndarray]]:
    """Per-split softmax state for one query vector over token rows k, v [n][d].

    bounds: split boundaries 0 = b_0 <= b_1 <= ... <= b_S = n. Split s returns
    (m_s, l_s, acc_s) with m_s = max x over the split, l_s = sum exp(x - m_s),
    acc_s = sum exp(x - m_s) v. An empty split returns (-inf, 0, 0).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            parts.append((-np.inf, 0.0, np.zeros(v.shape[1])))
            continue
        x = float(sm_scale) * (k[a:b] @ q)
        m = float(x.max())
        e = np.exp(x - m)
        parts.append((m, float(e.sum()), e @ v[a:b]))
    return parts


def combine_partials(parts) -> np.ndarray:
    """Merge per-split states: M = max m_s; o = sum e^(m_s - M) acc_s / sum e^(m_s - M) l_s."""
    ms = np.array([p[0] for p in parts], dtype=np.float64)
    if len(parts) == 0 or not np.isfinite(ms).any():
        d = parts[0][2].shape[0] if parts else 0
        return np.zeros(d)
    M = ms.max()
    wsum = 0.0
    acc = np.zeros_like(parts[0][2], dtype=np.float64)
    for m, l, a in parts:
        if not np.isfinite(m):
            continue
        f = np.exp(m - M)
        wsum += f * l
        acc = acc + f * a
    return acc / wsum
