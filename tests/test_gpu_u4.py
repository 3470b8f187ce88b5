"""Per-token 4-bit caches on the GPU: packed codes, scales and zero-points
bit-exact against the oracle's 4-bit quantiser; page boxes bit-exact; dense,
sparse and one-call decode-step attention over the restored values within
tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (TOL, bits_to_torch, check_per_token_u4_codes, gather, load_workload, max_abs_err,
                     oracle_dense, oracle_kv, queries_dev, set_knobs)

pytestmark = pytest.mark.gpu


def small_u4(seed, d=128, Hq=8, Hkv=2, ps=16, batch=4, offsets=0.0):
    return synth.Workload(name="u4", seed=seed, batch=batch, layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                          head_dim=d, page_size=ps, dtype="f16", quant="per_token_u4", seq_len=None,
                          seq_len_range=(1, 400), outlier_channels=4, outlier_scale=15.0,
                          page_offset_std=offsets)


@pytest.mark.parametrize("mma", ["1", "0"])
@pytest.mark.parametrize("d,Hq,Hkv,ps", [(128, 8, 2, 16), (64, 4, 4, 16), (64, 16, 2, 32), (128, 32, 8, 64),
                                          (128, 8, 8, 16), (64, 8, 4, 16)])
def test_u4_small_all_outputs(monkeypatch, d, Hq, Hkv, ps, mma):
    # mma = 1: query-head groups use the tensor-core kernel; 0: the CUDA-core one
    set_knobs(monkeypatch, PKV_ATTN_MMA=mma)
    w = small_u4(800 + d + Hq + ps, d, Hq, Hkv, ps)
    ld = load_workload(w, lens=np.array([1, 400, 17, 250], dtype=np.int32))
    check_per_token_u4_codes(ld)
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    for splits in (0, 1, 5):
        out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, num_splits=splits, dev_status=ld.status)
        assert max_abs_err(out.cpu().numpy(), ref) <= TOL["int8"], splits
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("chunks", [[1] * 40, [3, 61, 70, 1]])
def test_u4_chunked_appends(chunks):
    # per-token codes do not depend on how the tokens are split over calls
    w = small_u4(850, 64, 4, 2, 16, batch=3)
    total = sum(chunks)
    ld = load_workload(w, lens=np.array([total, total - 3, total // 2], dtype=np.int32), chunks=chunks)
    check_per_token_u4_codes(ld)
    assert int(ld.status.item()) == 0


def test_u4_constant_rows():
    # a token whose K (or V) row is constant stores scale 0 and codes 0 and
    # restores the constant exactly
    from paged_kv_cache_243_gb300.cache import PagedKVCache
    d, Hkv, ps, L = 64, 2, 16, 40
    rng = np.random.default_rng(3)
    k = rng.standard_normal((1, L, Hkv, d)).astype(np.float16)
    v = rng.standard_normal((1, L, Hkv, d)).astype(np.float16)
    k[0, 5] = 0.75
    v[0, 9, 1] = -2.0
    cache = PagedKVCache(8, ps, Hkv, d, kv_dtype="u4", quant="per_token", poison=True)
    bt = torch.tensor([[4, 1, 6]], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), bt,
                 torch.zeros(1, dtype=torch.int32, device="cuda"), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kp, vp, sz = cache.k_pages.cpu().numpy(), cache.v_pages.cpu().numpy(), cache.kv_sz.cpu().numpy()
    btn = bt.cpu().numpy()[0]
    gk, gv, gs = gather(kp, btn, L, ps), gather(vp, btn, L, ps), gather(sz, btn, L, ps)
    for x, pool, col in ((k[0].astype(np.float32), gk, 0), (v[0].astype(np.float32), gv, 2)):
        c, s, z = oracle.quantize_per_token_u4(x)
        assert np.array_equal(pool, oracle.pack_u4(c))
        assert np.array_equal(gs[:, :, col].view(np.uint32), s.view(np.uint32))
        assert np.array_equal(gs[:, :, col + 1].view(np.uint32), z.view(np.uint32))
    assert (gk[5] == 0).all() and (gs[5, :, 0] == 0).all() and (gs[5, :, 1] == np.float32(0.75)).all()
    assert (gv[9, 1] == 0).all() and gs[9, 1, 2] == 0 and gs[9, 1, 3] == np.float32(-2.0)


@pytest.mark.parametrize("mma", ["1", "0"])
@pytest.mark.parametrize("big", [0.0, 5000.0])
def test_u4_large_queries(monkeypatch, big, mma):
    # On the tensor-core path a q value beyond 4094 in magnitude switches the
    # unit's q scaling (16 q would overflow fp16). K channels 0 and 1 hold -0.25
    # in every token, each token's minimum, so they restore exactly and only
    # shift all scores of a head by the same amount.
    set_knobs(monkeypatch, PKV_ATTN_MMA=mma)
    from paged_kv_cache_243_gb300.cache import PagedKVCache
    d, Hq, Hkv, ps, L = 128, 8, 2, 16, 200
    rng = np.random.default_rng(17)
    k = np.abs(rng.standard_normal((1, L, Hkv, d))).astype(np.float16)
    k[..., :2] = -0.25
    v = rng.standard_normal((1, L, Hkv, d)).astype(np.float16)
    q = rng.standard_normal((1, Hq, d)).astype(np.float16)
    q[0, :Hq // Hkv, 0] = big          # the first kv head's query group only
    q[0, :Hq // Hkv, 1] = -big / 2
    cache = PagedKVCache(16, ps, Hkv, d, kv_dtype="u4", quant="per_token", poison=True)
    pages = rng.permutation(16)[:(L + ps - 1) // ps].astype(np.int32)
    bt = torch.from_numpy(pages[None, :]).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), bt,
                 torch.zeros(1, dtype=torch.int32, device="cuda"), dev_status=st)
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    sm = 1.0 / np.sqrt(d)
    kr = oracle.per_token_u4_dequant(*oracle.quantize_per_token_u4(k[0].astype(np.float32)))
    vr = oracle.per_token_u4_dequant(*oracle.quantize_per_token_u4(v[0].astype(np.float32)))
    ref = oracle.decode_attention(q[0].astype(np.float64), kr, vr, sm)
    for splits in (0, 3):
        out = cache.attention(torch.from_numpy(q).cuda(), bt, lens, sm_scale=sm, num_splits=splits,
                              dev_status=st).cpu().numpy()[0]
        assert np.isfinite(out).all(), splits
        assert np.abs(out - ref).max() <= TOL["int8"], splits
    assert int(st.item()) == 0


def test_u4_boxes_and_sparse():
    from test_gpu_sparse import check_group_selection, check_meta, check_selection, run_group_sparse, run_sparse
    w = small_u4(870, 128, 8, 2, 16, batch=3, offsets=0.5)
    ld = load_workload(w, lens=np.array([300, 45, 160], dtype=np.int32), with_meta=True)
    check_meta(ld)
    q, qf = queries_dev(w)
    sel, cnt, scores, out = run_sparse(ld, q, 4)
    chosen = check_selection(ld, qf, 4, sel, cnt, scores)
    for (b, h), pages in chosen.items():
        k, v = oracle_kv(ld, b)
        g = h // w.group
        o = oracle.sparse_decode_attention(qf[b, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], w.sm_scale,
                                           [pages], w.page_size)[0]
        assert np.abs(out[b, h] - o).max() <= TOL["int8"], (b, h)
    sel, cnt, scores, out = run_group_sparse(ld, q, 4, "sum")
    check_group_selection(ld, qf, 4, "sum", sel, cnt, scores, out)
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("d,Hq,Hkv", [(128, 16, 4), (64, 4, 4)])
def test_u4_append_attention_steps(d, Hq, Hkv, splits):
    # one-call decode steps: the attention kernel quantises each new token
    # itself; stored rows equal what kv_append would have written
    w = small_u4(890 + d + Hq, d, Hq, Hkv, 16)
    lens = np.array([47, 190, 16, 1], dtype=np.int32)
    steps = 4
    ld = load_workload(w, lens=lens, extra_pages=1)
    K = [s.k for s in ld.seqs]
    V = [s.v for s in ld.seqs]
    cur = lens.copy()
    for step in range(steps):
        toks = [synth.append_tokens(w, b, step) for b in range(w.batch)]
        kb = np.stack([t.k_bits[0] for t in toks])
        vb = np.stack([t.v_bits[0] for t in toks])
        cur = cur + 1
        q, qf = queries_dev(w, step=step)
        out = ld.cache.append_attention(bits_to_torch(kb, "f16").cuda(), bits_to_torch(vb, "f16").cuda(), q,
                                        ld.bt_dev, torch.from_numpy(cur.copy()).cuda(), sm_scale=w.sm_scale,
                                        num_splits=splits, dev_status=ld.status).cpu().numpy()
        for b in range(w.batch):
            K[b] = np.concatenate([K[b], toks[b].k])
            V[b] = np.concatenate([V[b], toks[b].v])
            kd = oracle.per_token_u4_dequant(*oracle.quantize_per_token_u4(K[b]))
            vd = oracle.per_token_u4_dequant(*oracle.quantize_per_token_u4(V[b]))
            for h in range(Hq):
                g = h // w.group
                o = oracle.decode_attention_tokens(qf[b, h], kd[:, g], vd[:, g], w.sm_scale)
                assert np.abs(out[b, h] - o).max() <= TOL["int8"], (step, b, h)
    ld.lens = cur
    for b in range(w.batch):
        ld.seqs[b] = synth.SeqData(None, None, K[b], V[b])
    check_per_token_u4_codes(ld)
    assert int(ld.status.item()) == 0


@pytest.mark.slow
def test_w7_u4_full_size():
    # the GQA 32/8 workload's shapes (B = 16, L ~ U[1K, 32K]) with 4-bit codes:
    # every code and every output, in the benchmark's launch configuration
    w = synth.WORKLOADS["w7_gqa_u4_token"]
    ld = load_workload(w)
    check_per_token_u4_codes(ld)
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    for fresh in (-1, 0):
        out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, dev_status=ld.status, fresh_rows=fresh).cpu().numpy()
        assert max_abs_err(out, ref) <= TOL["int8"], fresh
    assert int(ld.status.item()) == 0
