"""Query-aware sparse mode on the GPU: page bounding boxes, scores, top-K and
attention over the selected pages, against the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL, gather, load_workload, max_abs_err, oracle_bbox_keys, oracle_dense, queries_dev

pytestmark = pytest.mark.gpu


def check_meta(ld):
    meta = ld.cache.page_meta.cpu().numpy()      # [pages][Hkv][2][d]
    w = ld.w
    for b in range(w.batch):
        L = int(ld.lens[b])
        if L == 0:
            continue
        mn, mx = oracle.page_bounding_boxes(oracle_bbox_keys(w, ld.seqs[b]), w.page_size)
        P = mn.shape[0]
        got = meta[ld.bt[b][:P]]
        assert np.array_equal(got[:, :, 0].view(np.uint32), mn.view(np.uint32))
        assert np.array_equal(got[:, :, 1].view(np.uint32), mx.view(np.uint32))


def check_selection(ld, qf, top_k, sel, cnt, scores):
    """Scores within fp32 tolerance; kept pages bit-exact unless the oracle's K-th and
    (K+1)-th scores tie within 1e-4 relative. Returns the page lists to attend over."""
    w = ld.w
    meta_sel = {}
    for b in range(w.batch):
        L = int(ld.lens[b])
        P = -(-L // w.page_size)
        mn, mx = oracle.page_bounding_boxes(oracle_bbox_keys(w, ld.seqs[b]), w.page_size)
        r = oracle.page_scores(qf[b], mn, mx, w.group)
        for h in range(w.num_q_heads):
            K = min(top_k, P)
            assert cnt[b, h] == K
            slack = 1e-5 * (np.abs(qf[b, h])[None, :] * np.maximum(np.abs(mn[:, h // w.group]),
                                                                 np.abs(mx[:, h // w.group]))).sum(1) + 1e-6
            assert (np.abs(scores[b, h, :P] - r[h]) <= slack).all()
            assert np.isneginf(scores[b, h, P:]).all()
            want = oracle.select_top_k(r[h], K)
            got = sel[b, h, :K]
            assert (sel[b, h, K:] == -1).all()
            assert (np.diff(got) > 0).all()
            if not np.array_equal(got, want):
                srt = np.sort(r[h])[::-1]
                kth, nxt = srt[K - 1], srt[K]
                assert abs(kth - nxt) <= 1e-4 * max(abs(kth), abs(nxt)), (b, h)
                assert (r[h][got] >= nxt - slack[got]).all()
            meta_sel[(b, h)] = got
    return meta_sel


def oracle_sparse(ld, qf, selected, units):
    w = ld.w
    res = {}
    for b, h in units:
        sd = ld.seqs[b]
        o = oracle.sparse_decode_attention(qf[b, h:h + 1], sd.k[:, h // w.group:h // w.group + 1],
                                           sd.v[:, h // w.group:h // w.group + 1], w.sm_scale,
                                           [selected[(b, h)]], w.page_size)
        res[(b, h)] = o[0]
    return res


def run_sparse(ld, q, top_k):
    sel, cnt, scores = ld.cache.score_topk(q, ld.bt_dev, ld.lens_dev, top_k, want_scores=True,
                                           dev_status=ld.status)
    out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=ld.w.sm_scale, sel=sel, sel_count=cnt,
                             dev_status=ld.status)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), cnt.cpu().numpy(), scores.cpu().numpy(), out.cpu().numpy()


@pytest.mark.parametrize("d,Hq,Hkv,ps,top_k", [(64, 4, 4, 16, 5), (128, 8, 2, 32, 3), (64, 8, 4, 64, 2),
                                               (64, 16, 4, 16, 4), (128, 32, 4, 16, 3), (64, 6, 3, 16, 2)])
def test_small_sparse_all_outputs(d, Hq, Hkv, ps, top_k):
    # kv heads are scored 4 (d = 64) or 2 (d = 128) per cluster when they divide
    # the count; 16 query heads per cluster take two select rounds per block
    w = synth.Workload(name="sp", seed=900 + d + ps, batch=4, layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                       head_dim=d, page_size=ps, dtype="f16", quant="none", seq_len=None,
                       seq_len_range=(1, 500), page_offset_std=0.5)
    ld = load_workload(w, lens=np.array([500, 1, 37, 160], dtype=np.int32), with_meta=True)
    check_meta(ld)
    q, qf = queries_dev(w)
    sel, cnt, scores, out = run_sparse(ld, q, top_k)
    chosen = check_selection(ld, qf, top_k, sel, cnt, scores)
    ref = oracle_sparse(ld, qf, chosen, list(chosen))
    assert max_abs_err(out, ref) <= TOL["f16"]
    assert int(ld.status.item()) == 0


def test_w5_full_size_30pct_and_all_pages():
    w = synth.WORKLOADS["w5_sparse_f16"]
    ld = load_workload(w, with_meta=True)
    check_meta(ld)
    q, qf = queries_dev(w)
    P = w.seq_len // w.page_size
    K = oracle.top_k_count(w.top_k_ratio, P)
    assert K == 308
    sel, cnt, scores, out = run_sparse(ld, q, K)
    chosen = check_selection(ld, qf, K, sel, cnt, scores)
    units = [(b, h) for b in range(w.batch) for h in range(w.num_q_heads)]   # every output
    assert max_abs_err(out, oracle_sparse(ld, qf, chosen, units)) <= TOL["f16"]
    # top-K = all pages reproduces dense attention
    sel2, cnt2, scores2, out_all = run_sparse(ld, q, P)
    assert (cnt2 == P).all() and (sel2 == np.arange(P)[None, None, :]).all()
    dense = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale).cpu().numpy()
    assert np.abs(out_all - dense).max() <= 1e-5
    assert max_abs_err(out_all, oracle_dense(ld, qf, units)) <= TOL["f16"]
    assert int(ld.status.item()) == 0


def test_int8_per_token_boxes_and_sparse():
    w = synth.Workload(name="sp8", seed=950, batch=3, layers=1, num_q_heads=8, num_kv_heads=2,
                       head_dim=128, page_size=16, dtype="f16", quant="per_token", seq_len=None,
                       seq_len_range=(1, 300), outlier_channels=4, outlier_scale=15.0, page_offset_std=0.5)
    ld = load_workload(w, lens=np.array([300, 45, 160], dtype=np.int32), with_meta=True)
    check_meta(ld)
    q, qf = queries_dev(w)
    sel, cnt, scores, out = run_sparse(ld, q, 4)
    chosen = check_selection(ld, qf, 4, sel, cnt, scores)
    from helpers import oracle_kv
    for (b, h), pages in chosen.items():
        k, v = oracle_kv(ld, b)
        o = oracle.sparse_decode_attention(qf[b, h:h + 1], k[:, h // 4:h // 4 + 1], v[:, h // 4:h // 4 + 1],
                                           w.sm_scale, [pages], w.page_size)[0]
        assert np.abs(out[b, h] - o).max() <= TOL["int8"]
    assert int(ld.status.item()) == 0


def test_bad_selected_page_is_reported():
    from paged_kv_cache_243_gb300 import binding as B
    w = dataclasses.replace(synth.WORKLOADS["w1_tiny_f16"], batch=1, seq_len=64)
    ld = load_workload(w)
    q, qf = queries_dev(w)
    sel = torch.tensor([[[0, 9]] * 4], dtype=torch.int32, device="cuda")     # page 9 >= 4 pages
    cnt = torch.full((1, 4), 2, dtype=torch.int32, device="cuda")
    ld.status.zero_()
    out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sel=sel, sel_count=cnt, dev_status=ld.status)
    torch.cuda.synchronize()
    assert int(ld.status.item()) & B.DEV_BAD_SELECTED
    out = out.cpu().numpy()
    for h in range(4):
        o = oracle.decode_attention_tokens(qf[0, h], ld.seqs[0].k[:16, h], ld.seqs[0].v[:16, h], w.sm_scale)
        assert np.abs(out[0, h] - o).max() <= TOL["f16"]


def check_group_selection(ld, qf, top_k, mode, sel, cnt, scores, out):
    """One page list per kv head from the sum or max of its group's scores: scores
    within fp32 slack, kept pages bit-exact (ties within 1e-4 relative excepted), and
    every query head's output over its group's list against the oracle."""
    from helpers import oracle_kv
    w = ld.w
    G, Hkv, ps = w.group, w.num_kv_heads, w.page_size
    assert sel.shape == (w.batch, Hkv, top_k)
    tol = TOL["int8"] if w.quant != "none" else TOL[w.dtype]
    for b in range(w.batch):
        L = int(ld.lens[b])
        P = -(-L // ps)
        mn, mx = oracle.page_bounding_boxes(oracle_bbox_keys(w, ld.seqs[b]), ps)
        r = oracle.page_scores(qf[b], mn, mx, G)
        rg = oracle.group_page_scores(r, G, mode)
        k, v = oracle_kv(ld, b)
        for g in range(Hkv):
            K = min(top_k, P)
            assert cnt[b, g] == K
            per_head = [1e-5 * (np.abs(qf[b, h])[None, :] * np.maximum(np.abs(mn[:, g]), np.abs(mx[:, g]))).sum(1)
                        for h in range(g * G, (g + 1) * G)]
            slack = np.sum(per_head, axis=0) + 1e-6
            assert (np.abs(scores[b, g, :P] - rg[g]) <= slack).all()
            assert np.isneginf(scores[b, g, P:]).all()
            want = oracle.select_top_k(rg[g], K)
            got = sel[b, g, :K]
            assert (sel[b, g, K:] == -1).all() and (np.diff(got) > 0).all()
            if not np.array_equal(got, want):
                srt = np.sort(rg[g])[::-1]
                kth, nxt = srt[K - 1], srt[K]
                assert abs(kth - nxt) <= 1e-4 * max(abs(kth), abs(nxt)), (b, g)
                assert (rg[g][got] >= nxt - slack[got]).all()
            for h in range(g * G, (g + 1) * G):
                o = oracle.sparse_decode_attention(qf[b, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], w.sm_scale,
                                                   [got], ps)[0]
                assert np.abs(out[b, h] - o).max() <= tol, (b, h)


def run_group_sparse(ld, q, top_k, mode):
    from paged_kv_cache_243_gb300 import binding as B
    gm = B.SELECT_GROUP_SUM if mode == "sum" else B.SELECT_GROUP_MAX
    sel, cnt, scores = ld.cache.score_topk(q, ld.bt_dev, ld.lens_dev, top_k, want_scores=True,
                                           dev_status=ld.status, group_mode=gm)
    out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=ld.w.sm_scale, sel=sel, sel_count=cnt,
                             sel_shared=True, dev_status=ld.status)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), cnt.cpu().numpy(), scores.cpu().numpy(), out.cpu().numpy()


@pytest.mark.parametrize("mode", ["sum", "max"])
@pytest.mark.parametrize("quant,d,Hq,Hkv,ps,top_k", [("none", 64, 8, 2, 16, 4), ("per_token", 128, 16, 4, 16, 5),
                                                     ("none", 128, 8, 1, 32, 3), ("none", 64, 16, 2, 64, 2)])
def test_group_shared_selection(mode, quant, d, Hq, Hkv, ps, top_k):
    # one page list per kv head, from the sum or max of its group's scores;
    # each query head of the group attends over that list
    w = synth.Workload(name="spg", seed=970 + d + Hq + ps, batch=4, layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                       head_dim=d, page_size=ps, dtype="f16", quant=quant, seq_len=None,
                       seq_len_range=(1, 400), outlier_channels=4 if quant != "none" else 0,
                       outlier_scale=15.0, page_offset_std=0.5)
    ld = load_workload(w, lens=np.array([400, 1, 37, 200], dtype=np.int32), with_meta=True)
    q, qf = queries_dev(w)
    sel, cnt, scores, out = run_group_sparse(ld, q, top_k, mode)
    check_group_selection(ld, qf, top_k, mode, sel, cnt, scores, out)
    assert int(ld.status.item()) == 0


@pytest.mark.slow
def test_w6_full_size_group_sum():
    # GQA 32/8 per-token INT8 with page boxes, B = 8, L = 16384, page 16: one
    # list of 308 pages (30 %) per kv head from the group's summed scores;
    # boxes bit-exact, scores, selections and every output against the oracle
    w = synth.WORKLOADS["w6_gqa_sparse_int8"]
    ld = load_workload(w, with_meta=True)
    check_meta(ld)
    q, qf = queries_dev(w)
    P = w.seq_len // w.page_size
    K = oracle.top_k_count(w.top_k_ratio, P)
    sel, cnt, scores, out = run_group_sparse(ld, q, K, "sum")
    check_group_selection(ld, qf, K, "sum", sel, cnt, scores, out)
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("d,Hq,Hkv,ps", [(128, 16, 4, 128), (64, 8, 2, 64), (128, 32, 8, 256)])
def test_per_group_int8_boxes_and_sparse(d, Hq, Hkv, ps):
    # Per-64-token-group INT8 with page boxes. Every append re-quantises the
    # open group, which changes the restored values of its earlier tokens, so
    # the box of the page holding it must be rebuilt: after chunked prefill and
    # after each of several single-token appends that close a group and open
    # the next, the boxes must equal the oracle's over the restored keys, bit
    # for bit. Then page scoring and sparse attention (lists per query head,
    # and per kv head from group sums and maxima) run over that cache.
    w = synth.Workload(name="spg8", seed=990 + d + Hq + ps, batch=4, layers=1, num_q_heads=Hq,
                       num_kv_heads=Hkv, head_dim=d, page_size=ps, dtype="f16", quant="per_group64",
                       seq_len=None, seq_len_range=(1, 400), outlier_channels=4, outlier_scale=15.0,
                       page_offset_std=0.5)
    lens = np.array([190, 62, 127, 1], dtype=np.int32)
    ld = load_workload(w, lens=lens, with_meta=True, extra_pages=1, chunks=[100, 27, 1, 1, 36, 100])
    check_meta(ld)
    from helpers import bits_to_torch
    from helpers import check_per_group_codes
    K = [s.k for s in ld.seqs]
    V = [s.v for s in ld.seqs]
    cur = lens.copy()
    for step in range(4):       # 190 -> 194 closes group 2; 62 -> 66 closes group 0; 127 -> 131
        toks = [synth.append_tokens(w, b, step) for b in range(w.batch)]
        kb = np.stack([t.k_bits for t in toks])
        vb = np.stack([t.v_bits for t in toks])
        ld.cache.append(bits_to_torch(kb, "f16").cuda(), bits_to_torch(vb, "f16").cuda(), ld.bt_dev,
                        torch.from_numpy(cur.copy()).cuda(), dev_status=ld.status)
        torch.cuda.synchronize()
        cur = cur + 1
        for b in range(w.batch):
            K[b] = np.concatenate([K[b], toks[b].k])
            V[b] = np.concatenate([V[b], toks[b].v])
            ld.seqs[b] = synth.SeqData(None, None, K[b], V[b])
        ld.lens = cur.copy()
        check_meta(ld)
    check_per_group_codes(ld)
    ld.lens_dev = torch.from_numpy(cur.copy()).cuda()
    q, qf = queries_dev(w)
    top_k = 2
    sel, cnt, scores, out = run_sparse(ld, q, top_k)
    chosen = check_selection(ld, qf, top_k, sel, cnt, scores)
    from helpers import oracle_kv
    for (b, h), pages in chosen.items():
        k, v = oracle_kv(ld, b)
        g = h // w.group
        o = oracle.sparse_decode_attention(qf[b, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], w.sm_scale,
                                           [pages], ps)[0]
        assert np.abs(out[b, h] - o).max() <= TOL["int8"], (b, h)
    for mode in ("sum", "max"):
        sel, cnt, scores, out = run_group_sparse(ld, q, top_k, mode)
        check_group_selection(ld, qf, top_k, mode, sel, cnt, scores, out)
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("d,Hkv,patterns", [(64, 4, 1), (64, 4, 3), (128, 2, 1), (128, 2, 5)])
def test_tied_page_scores_keep_the_lowest_pages(d, Hkv, patterns):
    # every page of a head repeats one of `patterns` token blocks, so page scores
    # take at most that many values and tie exactly (same boxes, same arithmetic);
    # one pattern makes every score equal. The top-K must be the pages with the
    # higher values, ties broken by the lower page index, as in the oracle.
    from paged_kv_cache_243_gb300.cache import PagedKVCache
    ps, P, top_k = 16, 40, 13
    rng = np.random.default_rng(1000 + d + patterns)
    blocks = rng.standard_normal((patterns, ps, Hkv, d)).astype(np.float16)
    which = rng.integers(0, patterns, size=P)
    k = np.concatenate([blocks[which[pg]] for pg in range(P)])[None]      # [1][P ps][Hkv][d]
    v = rng.standard_normal(k.shape).astype(np.float16)
    pool = P + 3
    bt = rng.permutation(pool)[:P].astype(np.int32)[None]
    cache = PagedKVCache(pool, ps, Hkv, d, kv_dtype="f16", with_meta=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt_d = torch.from_numpy(bt).cuda()
    cache.append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), bt_d,
                 torch.zeros(1, dtype=torch.int32, device="cuda"), dev_status=status)
    q = torch.from_numpy(rng.standard_normal((1, Hkv, d)).astype(np.float16)).cuda()
    lens = torch.tensor([P * ps], dtype=torch.int32, device="cuda")
    sel, cnt, _ = cache.score_topk(q, bt_d, lens, top_k, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    qf = q.cpu().numpy().astype(np.float64)[0]
    for h in range(Hkv):
        mn, mx = oracle.page_bounding_boxes(k[0][:, h:h + 1].astype(np.float64), ps)
        r = oracle.page_scores(qf[h:h + 1], mn, mx, 1)[0]
        assert cnt[0, h] == top_k
        assert np.array_equal(sel[0, h], oracle.select_top_k(r, top_k)), h


@pytest.mark.parametrize("g1", ["0", "2"])
def test_per_head_lists_on_tensor_cores(monkeypatch, g1):
    # per-query-head page lists (units of one query head) on both consumers
    from helpers import set_knobs
    set_knobs(monkeypatch, PKV_ATTN_MMA_G1=g1)
    w = synth.Workload(name="sph", seed=611, batch=3, layers=1, num_q_heads=8, num_kv_heads=2,
                       head_dim=128, page_size=16, dtype="bf16", quant="none", seq_len=None,
                       seq_len_range=(1, 500))
    ld = load_workload(w, lens=np.array([500, 33, 260], dtype=np.int32), with_meta=True)
    q, qf = queries_dev(w)
    sel, cnt, scores, out = run_sparse(ld, q, 5)
    chosen = check_selection(ld, qf, 5, sel, cnt, scores)
    res = oracle_sparse(ld, qf, chosen, list(chosen))
    for (b, h), o in res.items():
        assert np.abs(out[b, h] - o).max() <= TOL["bf16"], (b, h)
    assert int(ld.status.item()) == 0
