"""Early start of the attention kernel (fresh_rows >= 0): the launch overlaps
the kernel before it on the stream and reads everything but the rows that
kernel writes before waiting for it. Results must equal the oracle's for
appends of one and several tokens, across 64-token group boundaries of
per-group INT8 caches, and for back-to-back calls sharing output and
workspace."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL, bits_to_torch, load_workload, oracle_dense, queries_dev, set_knobs
from oracle.quant import per_group_dequant, per_token_dequant

pytestmark = pytest.mark.gpu


def _restored(w, k):
    """K or V as attention sees it after quantising every token at once."""
    if w.quant == "none":
        return k.astype(np.float64)
    if w.quant == "per_token":
        return per_token_dequant(*oracle.quantize_per_token(k))
    if w.quant == "per_token_u4":
        return oracle.per_token_u4_dequant(*oracle.quantize_per_token_u4(k))
    return per_group_dequant(*oracle.quantize_per_group(k))


CASES = [
    # name, dtype, quant, d, Hq, Hkv, page
    ("bf16", "bf16", "none", 128, 8, 2, 16),
    ("f16-mha", "f16", "none", 64, 4, 4, 32),
    ("i8-token", "f16", "per_token", 128, 8, 2, 16),
    ("i8-group", "f16", "per_group64", 128, 16, 4, 64),
    ("u4-token", "f16", "per_token_u4", 128, 8, 2, 16),
]


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("name,dt,quant,d,Hq,Hkv,ps", CASES)
def test_append_then_attention_overlapped(name, dt, quant, d, Hq, Hkv, ps, splits):
    _append_then_attention(name, dt, quant, d, Hq, Hkv, ps, splits)


@pytest.mark.parametrize("name,dt,quant,d,Hq,Hkv,ps", [c for c in CASES if c[3] == 128 and c[4] > c[5]])
def test_self_fed_blocks_overlapped(monkeypatch, name, dt, quant, d, Hq, Hkv, ps):
    # the tensor-core blocks without a producer warp (each consumer warp copies
    # its own chunks, the combine released at entry), forced for every
    # early-start call; by default they serve short chains without fresh rows
    set_knobs(monkeypatch, PKV_ATTN_SELF=2)
    _append_then_attention(name, dt, quant, d, Hq, Hkv, ps, 0)


def _append_then_attention(name, dt, quant, d, Hq, Hkv, ps, splits):
    w = synth.Workload(name="early-" + name, seed=610 + d + Hq + ps, batch=3, layers=1,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, page_size=ps, dtype=dt,
                       quant=quant, seq_len=None, seq_len_range=(1, 300),
                       outlier_channels=4 if quant != "none" else 0, outlier_scale=15.0)
    lens = np.array([61, 190, 1], dtype=np.int32)
    steps = [1, 1, 3, 1, 70, 1, 2]               # tokens appended per sequence each step
    ld = load_workload(w, lens=lens, extra_pages=-(-sum(steps) // ps) + 1)
    K = [s.k for s in ld.seqs]
    V = [s.v for s in ld.seqs]
    cur = lens.copy()
    tok = 0
    for i, t_new in enumerate(steps):
        toks = [[synth.append_tokens(w, b, tok + j) for j in range(t_new)] for b in range(w.batch)]
        tok += t_new
        kb = np.stack([np.concatenate([t.k_bits for t in row]) for row in toks])
        vb = np.stack([np.concatenate([t.v_bits for t in row]) for row in toks])
        ld.cache.append(bits_to_torch(kb, dt).cuda(), bits_to_torch(vb, dt).cuda(), ld.bt_dev,
                        torch.from_numpy(cur.copy()).cuda(), dev_status=ld.status)
        for b in range(w.batch):
            K[b] = np.concatenate([K[b]] + [t.k for t in toks[b]])
            V[b] = np.concatenate([V[b]] + [t.v for t in toks[b]])
        cur = cur + t_new
        q, qf = queries_dev(w, step=i)
        out = ld.cache.attention(q, ld.bt_dev, torch.from_numpy(cur.copy()).cuda(), sm_scale=w.sm_scale,
                                 num_splits=splits, dev_status=ld.status, fresh_rows=t_new)
        out = out.cpu().numpy()
        for b in range(w.batch):
            kd, vd = _restored(w, K[b]), _restored(w, V[b])
            for h in range(Hq):
                g = h // w.group
                o = oracle.decode_attention_tokens(qf[b, h], kd[:, g], vd[:, g], w.sm_scale)
                tol = TOL["int8"] if quant != "none" else TOL[dt]
                assert np.abs(out[b, h] - o).max() <= tol, (i, b, h)
    assert int(ld.status.item()) == 0


def test_back_to_back_calls_share_output_and_workspace():
    # each call may start while the previous call's combine still writes the
    # same output buffer and reads the same workspace
    w = synth.Workload(name="early-b2b", seed=640, batch=4, layers=1, num_q_heads=16, num_kv_heads=4,
                       head_dim=128, page_size=16, dtype="bf16", quant="none", seq_len=None,
                       seq_len_range=(1, 600))
    ld = load_workload(w, lens=np.array([600, 33, 257, 1], dtype=np.int32))
    out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    outs = [torch.empty_like(out) for _ in range(4)]
    qs = [queries_dev(w, step=i) for i in range(4)]
    for i, (q, _) in enumerate(qs):            # distinct outputs, one workspace
        ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale, out=outs[i],
                           dev_status=ld.status, fresh_rows=0)
    for q, _ in qs:                            # one output written four times
        ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale, out=out,
                           dev_status=ld.status, fresh_rows=0)
    torch.cuda.synchronize()
    for i, (_, qf) in enumerate(qs):
        ref = oracle_dense(ld, qf)
        got = outs[i].cpu().numpy()
        assert max(float(np.abs(got[b, h] - o).max()) for (b, h), o in ref.items()) <= TOL["bf16"]
    last = out.cpu().numpy()
    assert np.array_equal(last, outs[3].cpu().numpy())
    assert int(ld.status.item()) == 0


FUSED_CASES = [
    # name, dtype, quant, d, Hq, Hkv, page
    ("bf16-gqa", "bf16", "none", 128, 16, 4, 16),
    ("i8-token-mha", "f16", "per_token", 64, 4, 4, 16),
]


@pytest.mark.parametrize("layers,fresh", [(2, 0), (1, 2)])
@pytest.mark.parametrize("name,dt,quant,d,Hq,Hkv,ps", FUSED_CASES)
def test_fused_steps_enqueued_back_to_back(name, dt, quant, d, Hq, Hkv, ps, layers, fresh):
    _fused_steps(name, dt, quant, d, Hq, Hkv, ps, layers, fresh)


@pytest.mark.parametrize("layers,fresh", [(2, 0), (1, 2)])
def test_self_fed_fused_steps(monkeypatch, layers, fresh):
    # one-call steps on GQA per-token INT8 with the self-fed tensor-core blocks
    # forced: each consumer warp writes the new token of the units ending in
    # its lookups before copying their chunks
    set_knobs(monkeypatch, PKV_ATTN_SELF=2)
    _fused_steps("i8-token-gqa", "f16", "per_token", 128, 16, 4, 16, layers, fresh)


def _fused_steps(name, dt, quant, d, Hq, Hkv, ps, layers, fresh):
    # decode steps of one-call append + attention, all enqueued before any
    # synchronisation, so each call may start while the previous call's kernels
    # still run. Two layers: the previous call works on the other cache and
    # writes nothing this one reads (fresh_rows = 0). One layer: the previous
    # step wrote the row just before this step's new row (fresh_rows = 2).
    w = synth.Workload(name="early-fused-" + name, seed=700 + d + Hq, batch=3, layers=layers,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, page_size=ps, dtype=dt, quant=quant,
                       seq_len=None, seq_len_range=(1, 400),
                       outlier_channels=4 if quant != "none" else 0, outlier_scale=15.0)
    lens = np.array([400, 17, 130], dtype=np.int32)
    steps = 4
    lds = [load_workload(w, layer=l, lens=lens, extra_pages=1) for l in range(layers)]
    toks = [[[synth.append_tokens(w, b, 10 * l + s) for b in range(w.batch)] for s in range(steps)]
            for l in range(layers)]
    dev = lambda bits: bits_to_torch(bits, dt).cuda()  # noqa: E731
    k_in = [[dev(np.stack([t.k_bits[0] for t in toks[l][s]])) for s in range(steps)] for l in range(layers)]
    v_in = [[dev(np.stack([t.v_bits[0] for t in toks[l][s]])) for s in range(steps)] for l in range(layers)]
    qs = [[queries_dev(w, step=10 * l + s) for s in range(steps)] for l in range(layers)]
    lens_dev = [torch.from_numpy(lens + s + 1).cuda() for s in range(steps)]
    outs = [[torch.empty((w.batch, Hq, d), dtype=torch.float32, device="cuda") for _ in range(steps)]
            for _ in range(layers)]
    torch.cuda.synchronize()
    for s in range(steps):
        for l in range(layers):
            lds[l].cache.append_attention(k_in[l][s], v_in[l][s], qs[l][s][0], lds[l].bt_dev, lens_dev[s],
                                          sm_scale=w.sm_scale, out=outs[l][s], dev_status=lds[l].status,
                                          fresh_rows=fresh)
    torch.cuda.synchronize()
    for l in range(layers):
        assert int(lds[l].status.item()) == 0
        for b in range(w.batch):
            Kb, Vb = lds[l].seqs[b].k, lds[l].seqs[b].v
            for s in range(steps):
                Kb = np.concatenate([Kb, toks[l][s][b].k])
                Vb = np.concatenate([Vb, toks[l][s][b].v])
                kd, vd = _restored(w, Kb), _restored(w, Vb)
                got = outs[l][s][b].cpu().numpy()
                qf = qs[l][s][1]
                for h in range(Hq):
                    o = oracle.decode_attention_tokens(qf[b, h], kd[:, h // w.group], vd[:, h // w.group],
                                                       w.sm_scale)
                    tol = TOL["int8"] if quant != "none" else TOL[dt]
                    assert np.abs(got[h] - o).max() <= tol, (l, s, b, h)


@pytest.mark.parametrize("group_mode", [0, 1])
@pytest.mark.parametrize("quant,d,Hq,Hkv,ps,top_k", [("none", 64, 8, 8, 16, 7), ("per_token", 128, 16, 4, 16, 5),
                                                     ("none", 128, 8, 2, 32, 3)])
def test_sparse_attention_overlapping_the_scoring(group_mode, quant, d, Hq, Hkv, ps, top_k):
    _sparse_after_scoring(group_mode, quant, d, Hq, Hkv, ps, top_k)


@pytest.mark.parametrize("group_mode", [0, 1])
@pytest.mark.parametrize("quant,d,Hq,Hkv,ps,top_k", [("per_token", 128, 16, 4, 16, 5), ("none", 128, 8, 2, 32, 3)])
def test_self_fed_sparse_after_scoring(monkeypatch, group_mode, quant, d, Hq, Hkv, ps, top_k):
    # the self-fed tensor-core blocks read the page lists in their own warps'
    # lookups, which must wait for the scoring that writes them
    set_knobs(monkeypatch, PKV_ATTN_SELF=2)
    _sparse_after_scoring(group_mode, quant, d, Hq, Hkv, ps, top_k)


def _sparse_after_scoring(group_mode, quant, d, Hq, Hkv, ps, top_k):
    # sparse attention right after the page scoring that writes its lists,
    # started early (fresh_rows = 0): it plans from the lengths and reads the
    # lists only after waiting; results equal the call that waits up front
    import oracle as O
    from helpers import TOL as T, oracle_kv
    w = synth.Workload(name="early-sp", seed=680 + d + Hq + ps + group_mode, batch=4, layers=1,
                       num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, page_size=ps, dtype="f16", quant=quant,
                       seq_len=None, seq_len_range=(1, 500), outlier_channels=4 if quant != "none" else 0,
                       outlier_scale=15.0, page_offset_std=0.5)
    ld = load_workload(w, lens=np.array([500, 1, 70, 33], dtype=np.int32), with_meta=True)
    q, qf = queries_dev(w)
    shared = group_mode != 0
    outs = []
    for fresh in (0, -1):
        sel, cnt, _ = ld.cache.score_topk(q, ld.bt_dev, ld.lens_dev, top_k, dev_status=ld.status,
                                          group_mode=group_mode)
        out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale, sel=sel, sel_count=cnt,
                                 sel_shared=shared, dev_status=ld.status, fresh_rows=fresh)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    assert np.abs(outs[0] - outs[1]).max() <= 1e-6
    tol = T["int8"] if quant != "none" else T["f16"]
    for b in range(w.batch):
        k, v = oracle_kv(ld, b)
        for h in range(Hq):
            g = h // w.group
            r = g if shared else h
            pages = sel[b, r, :cnt[b, r]]
            o = O.sparse_decode_attention(qf[b, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], w.sm_scale, [pages], ps)[0]
            assert np.abs(outs[0][b, h] - o).max() <= tol, (b, h)
    assert int(ld.status.item()) == 0


def test_early_sparse_lists_shorter_than_their_stride():
    # caller-made lists: counts below min(stride, pages), entries past a count
    # hold garbage that must not be read; a zero count gives zeros
    import oracle as O
    from helpers import TOL as T
    w = synth.Workload(name="early-sp2", seed=701, batch=3, layers=1, num_q_heads=4, num_kv_heads=4,
                       head_dim=64, page_size=16, dtype="f16", quant="none", seq_len=None,
                       seq_len_range=(1, 300))
    ld = load_workload(w, lens=np.array([300, 100, 40], dtype=np.int32))
    q, qf = queries_dev(w)
    stride = 6
    rng = np.random.default_rng(9)
    sel = np.full((w.batch, w.num_q_heads, stride), 99999, dtype=np.int32)   # garbage past the counts
    cnt = np.zeros((w.batch, w.num_q_heads), dtype=np.int32)
    for b in range(w.batch):
        P = -(-int(ld.lens[b]) // 16)
        for h in range(w.num_q_heads):
            n = int(rng.integers(0, min(stride, P) + 1)) if (b, h) != (0, 0) else 0
            sel[b, h, :n] = np.sort(rng.choice(P, n, replace=False))
            cnt[b, h] = n
    sel_d, cnt_d = torch.from_numpy(sel).cuda(), torch.from_numpy(cnt).cuda()
    ld.status.zero_()
    out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale, sel=sel_d, sel_count=cnt_d,
                             dev_status=ld.status, fresh_rows=0)
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    assert int(ld.status.item()) == 0
    assert (out[0, 0] == 0).all()
    for b in range(w.batch):
        sd = ld.seqs[b]
        for h in range(w.num_q_heads):
            o = O.sparse_decode_attention(qf[b, h:h + 1], sd.k[:, h:h + 1], sd.v[:, h:h + 1], w.sm_scale,
                                          [sel[b, h, :cnt[b, h]]], 16)[0]
            assert np.abs(out[b, h] - o).max() <= T["f16"], (b, h)


@pytest.mark.parametrize("group_mode", [0, 1])
def test_scoring_started_under_the_previous_attention(group_mode):
    # layers in a row on one set of list buffers: each scoring starts early
    # (early_start) under the previous sparse attention call, which may still
    # read the lists the scoring overwrites; lists and outputs equal those of
    # scorings that wait up front
    w = synth.Workload(name="early-score", seed=720 + group_mode, batch=4, layers=1, num_q_heads=16,
                       num_kv_heads=4, head_dim=128, page_size=16, dtype="f16", quant="per_token",
                       seq_len=None, seq_len_range=(1, 600), outlier_channels=4, outlier_scale=15.0,
                       page_offset_std=0.5)
    ld = load_workload(w, lens=np.array([600, 17, 333, 129], dtype=np.int32), with_meta=True)
    shared = group_mode != 0
    R = w.num_kv_heads if shared else w.num_q_heads
    top_k = 6
    qs = [queries_dev(w, step=s)[0] for s in range(4)]
    res = {}
    for early in (True, False):
        sel = torch.empty((w.batch, R, top_k), dtype=torch.int32, device="cuda")
        cnt = torch.empty((w.batch, R), dtype=torch.int32, device="cuda")
        outs = []
        for s in range(4):
            # (an attention that read lists already overwritten would differ)
            ld.cache.score_topk(qs[s], ld.bt_dev, ld.lens_dev, top_k, dev_status=ld.status, sel=sel, count=cnt,
                                group_mode=group_mode, early_start=early and s > 0)
            outs.append(ld.cache.attention(qs[s], ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale, sel=sel,
                                           sel_count=cnt, sel_shared=shared, dev_status=ld.status, fresh_rows=0))
        torch.cuda.synchronize()
        res[early] = ([o.cpu().numpy() for o in outs], sel.cpu().numpy(), cnt.cpu().numpy())
    assert np.array_equal(res[True][1], res[False][1])
    assert np.array_equal(res[True][2], res[False][2])
    for s in range(4):
        assert np.abs(res[True][0][s] - res[False][0][s]).max() <= 1e-6, s
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("quant,dt", [("per_group64", "f16"), ("none", "bf16")])
def test_self_fed_plan_on_a_long_context_chain(quant, dt):
    # few units of long sequences (the shape for which the plan picks the
    # self-fed blocks by itself: 16-128 chunks per block, a combine of at most
    # one block per SM), attention calls enqueued back to back without fresh
    # rows, each call's merge overlapping the next call
    w = synth.Workload(name="early-self-chain", seed=720, batch=2, layers=1, num_q_heads=32, num_kv_heads=8,
                       head_dim=128, page_size=256, dtype=dt, quant=quant, seq_len=None,
                       seq_len_range=(1, 8192), outlier_channels=4 if quant != "none" else 0,
                       outlier_scale=15.0)
    ld = load_workload(w, lens=np.array([8192, 7000], dtype=np.int32))
    qs = [queries_dev(w, step=i) for i in range(3)]
    outs = [torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda") for _ in qs]
    torch.cuda.synchronize()
    for i, (q, _) in enumerate(qs):
        ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale, out=outs[i],
                           dev_status=ld.status, fresh_rows=0)
    torch.cuda.synchronize()
    tol = TOL["int8"] if quant != "none" else TOL[dt]
    units = [(b, h) for b in range(w.batch) for h in range(0, w.num_q_heads, 3)]
    for i, (_, qf) in enumerate(qs):
        ref = oracle_dense(ld, qf, units)
        got = outs[i].cpu().numpy()
        assert max(float(np.abs(got[b, h] - o).max()) for (b, h), o in ref.items()) <= tol, i
    assert int(ld.status.item()) == 0
