"""Pins for the oracle's bounding boxes, page scores and top-K (no GPU)."""
import numpy as np
import pytest

import oracle


def test_hand_example_score():
    q = np.array([[1.0, -2.0, 0.0, 0.5]])
    mn = np.array([[[-1.0, 0.5, 5.0, -2.0]]])
    mx = np.array([[[3.0, 4.0, 7.0, 1.0]]])
    # 1*3 + (-2)*0.5 + 0*7 + 0.5*1 = 2.5
    assert oracle.page_scores(q, mn, mx, 1)[0, 0] == 2.5


def test_boxes_brute_force_with_partial_page():
    rng = np.random.default_rng(1)
    L, H, d, ps = 37, 2, 5, 16
    k = rng.standard_normal((L, H, d)).astype(np.float16).astype(np.float32)
    mn, mx = oracle.page_bounding_boxes(k, ps)
    assert mn.shape == (3, H, d)
    for p in range(3):
        toks = range(p * ps, min(L, (p + 1) * ps))
        for h in range(H):
            for i in range(d):
                vals = [float(k[t, h, i]) for t in toks]
                assert mn[p, h, i] == min(vals) and mx[p, h, i] == max(vals)


@pytest.mark.parametrize("ps", [1, 4, 16])
def test_score_never_underestimates(ps):
    # "never underestimates the true attention score" [TinyServe page, section 2.1]
    rng = np.random.default_rng(2 + ps)
    L, H, G, d = 203, 2, 2, 32
    k = rng.standard_normal((L, H, d)).astype(np.float16).astype(np.float32)
    k += rng.standard_normal((1, H, d)).astype(np.float32)
    q = rng.standard_normal((H * G, d))
    q[:, :3] = 0.0
    mn, mx = oracle.page_bounding_boxes(k, ps)
    r = oracle.page_scores(q, mn, mx, G)
    for h in range(H * G):
        g = h // G
        true = k[:, g, :].astype(np.float64) @ q[h]
        for p in range(r.shape[1]):
            seg = true[p * ps:(p + 1) * ps]
            assert r[h, p] >= seg.max()
            if ps == 1:
                assert r[h, p] == pytest.approx(seg.max(), abs=1e-12)


def test_identical_tokens_make_the_bound_exact():
    rng = np.random.default_rng(3)
    row = rng.standard_normal(16).astype(np.float32)
    k = np.tile(row, (16, 1, 1))
    q = rng.standard_normal((1, 16))
    mn, mx = oracle.page_bounding_boxes(k, 16)
    assert oracle.page_scores(q, mn, mx, 1)[0, 0] == pytest.approx(float(row.astype(np.float64) @ q[0]), abs=1e-12)


def brute_top_k(scores, k):
    """Page j is kept iff fewer than k pages beat it (higher score, or equal with lower index)."""
    P = len(scores)
    keep = []
    for j in range(P):
        beaten_by = sum(1 for i in range(P) if scores[i] > scores[j] or (scores[i] == scores[j] and i < j))
        if beaten_by < k:
            keep.append(j)
    return keep


@pytest.mark.parametrize("seed", range(6))
def test_top_k_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(1, 40))
    scores = rng.integers(0, 6, size=P).astype(np.float64)   # many ties
    for k in [1, 2, P // 2, P, P + 3]:
        got = oracle.select_top_k(scores, k).tolist()
        assert got == brute_top_k(scores.tolist(), min(k, P))
        assert got == sorted(got)


def test_top_k_count():
    assert oracle.top_k_count(0.3, 1024) == 308
    assert oracle.top_k_count(0.3, 1) == 1
    assert oracle.top_k_count(1024, 1000) == 1000
    assert oracle.top_k_count(0.3, 0) == 0


def test_group_scores_hand_example():
    # two query heads sharing one kv head
    r = np.array([[1.0, 5.0, -2.0], [3.0, -2.0, -1.0]])
    assert np.array_equal(oracle.group_page_scores(r, 2, "sum"), [[4.0, 3.0, -3.0]])
    assert np.array_equal(oracle.group_page_scores(r, 2, "max"), [[3.0, 5.0, -1.0]])
    # group of one: the per-head scores themselves
    assert np.array_equal(oracle.group_page_scores(r, 1, "sum"), r)
    assert np.array_equal(oracle.group_page_scores(r, 1, "max"), r)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_group_scores_bound_the_group_products(seed):
    # "max" bounds q_h . k for every head of the group and key of the page;
    # "sum" bounds (sum of the group's q) . k, brute force over the keys
    rng = np.random.default_rng(seed)
    G, Hkv, d, ps, L = 4, 2, 8, 4, 23
    keys = rng.standard_normal((L, Hkv, d)).astype(np.float32)
    q = rng.standard_normal((G * Hkv, d))
    mn, mx = oracle.page_bounding_boxes(keys, ps)
    r = oracle.page_scores(q, mn, mx, G)
    smax = oracle.group_page_scores(r, G, "max")
    ssum = oracle.group_page_scores(r, G, "sum")
    P = mn.shape[0]
    for g in range(Hkv):
        qs = q[g * G:(g + 1) * G]
        for p in range(P):
            blk = keys[p * ps:min(L, (p + 1) * ps), g].astype(np.float64)
            assert smax[g, p] >= (qs @ blk.T).max() - 1e-12
            assert ssum[g, p] >= (qs.sum(0) @ blk.T).max() - 1e-12
            # and the sum is never below any single head's bound
            assert ssum[g, p] <= G * smax[g, p] + 1e-12
