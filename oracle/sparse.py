"""Query-aware page selection with per-page channel bounding boxes (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

[TinyServe page, section 2.1]: for the keys K_j of page j (S tokens x d
channels) the metadata is the direction-aware bounding box
    m_j[i] = min over the page's tokens of K_j[:, i],   M_j[i] = max of the same,
and the relevance of page j to a query q is
    r(q, phi(K_j)) = sum_i ( q_i * M_j[i]  if q_i >= 0  else  q_i * m_j[i] ),
an upper bound on q . k for every key k of the page. The pages keep this
metadata in fp32 [section 5.2] and keep the top-K pages [section 3.1 phase 2,
whose body the page elides; ratio 0.3 in section 5.1].

Readings taken where the pages are silent: the box covers only the valid tokens of a
partially filled page; ties in the score are broken towards the lower logical
page index; the kept pages are returned in ascending page order; K = ceil(0.3 P)
for the 30 % setting and is clipped to the number of pages P.
"""
from __future__ import annotations

import math
from typing import Tuple

import numpy as np


def page_bounding_boxes(keys, page_size: int) -> Tuple[np.ndarray, np.ndarray]:
    """Per-page, per-kv-head channel min and max over valid tokens.

    keys: [L][Hkv][d] values the attention reads (fp32-exact).
    Returns (mn, mx), each float32 [P][Hkv][d] with P = ceil(L / page_size).
    """
    keys = np.asarray(keys, dtype=np.float32)
    L, H, d = keys.shape
    P = -(-L // page_size)
    mn = np.empty((P, H, d), dtype=np.float32)
    mx = np.empty((P, H, d), dtype=np.float32)
    for p in range(P):
        blk = keys[p * page_size:min(L, (p + 1) * page_size)]
        mn[p] = blk.min(axis=0)
        mx[p] = blk.max(axis=0)
    return mn, mx


def page_scores(q, mn, mx, group: int) -> np.ndarray:
    """Relevance score of every page for every query head, fp64.

    q: [Hq][d]; mn, mx: [P][Hkv][d]. Query head h uses kv head h // group.
    Returns r [Hq][P].
    """
    q = np.asarray(q, dtype=np.float64)
    mn = np.asarray(mn, dtype=np.float64)
    mx = np.asarray(mx, dtype=np.float64)
    Hq, d = q.shape
    P = mn.shape[0]
    r = np.zeros((Hq, P), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        pos = q[h] >= 0
        box = np.where(pos[None, :], mx[:, g, :], mn[:, g, :])   # [P][d]
        r[h] = box @ q[h]
    return r


def group_page_scores(r, group: int, mode: str) -> np.ndarray:
    """Page scores of each kv head's query-head group, for a selection shared by
    the group (so the group's K/V pages are read once for its G query heads).

    r: [Hq][P] per-query-head scores (page_scores); query heads g*G .. g*G+G-1
    share kv head g. mode "sum": the sum of the group's G scores; mode "max":
    their maximum. Returns [Hkv][P], fp64.

    The pages score one query per page [TinyServe page, section 2.1] and say
    nothing of query-head groups; these two reductions are the readings taken
    (each is an upper bound of the matching query-key products: "max" bounds
    every head's q . k on the page, "sum" bounds (sum of the heads' q) . k).
    """
    r = np.asarray(r, dtype=np.float64)
    Hq, P = r.shape
    out = np.empty((Hq // group, P), dtype=np.float64)
    for g in range(Hq // group):
        rows = [r[g * group + j] for j in range(group)]
        acc = rows[0].copy()
        for row in rows[1:]:
            if mode == "sum":
                acc = acc + row
            elif mode == "max":
                acc = np.maximum(acc, row)
            else:
                raise ValueError(mode)
        out[g] = acc
    return out


def top_k_count(ratio_or_k, num_pages: int) -> int:
    """Number of pages kept: an int is taken as K, a float as ceil(ratio * P); clipped to P."""
    if isinstance(ratio_or_k, float):
        k = int(math.ceil(ratio_or_k * num_pages))
    else:
        k = int(ratio_or_k)
    return max(0, min(k, num_pages))


def select_top_k(scores, k: int) -> np.ndarray:
    """Indices of the k highest scores, ties to the lower index, returned ascending."""
    scores = np.asarray(scores, dtype=np.float64)
    P = scores.shape[0]
    k = min(int(k), P)
    order = sorted(range(P), key=lambda j: (-scores[j], j))
    return np.array(sorted(order[:k]), dtype=np.int64)
