"""One-call decode step (pkv_append_decode_attention): the attention kernel
writes each sequence's new token into its page and attends over it. Outputs
against the oracle over the grown sequences, and the stored rows against the
inputs (bit-exact codes, scales and zero-points for per-token INT8)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL, bits_to_torch, gather, int8_codes, load_workload, queries_dev, set_knobs
from oracle.quant import per_group_dequant, per_token_dequant

pytestmark = pytest.mark.gpu


CASES = [
    # name, dtype, quant, d, Hq, Hkv, page, mma
    ("bf16-mha", "bf16", "none", 128, 8, 8, 16, "1"),
    ("f16-gqa", "f16", "none", 64, 8, 2, 32, "1"),
    ("f16-gqa-cuda-cores", "f16", "none", 128, 16, 4, 16, "0"),
    ("i8-token-gqa", "f16", "per_token", 128, 16, 4, 16, "1"),
    ("i8-token-cuda-cores", "f16", "per_token", 64, 4, 4, 16, "0"),
]


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("name,dt,quant,d,Hq,Hkv,ps,mma", CASES)
def test_append_attention_steps(monkeypatch, name, dt, quant, d, Hq, Hkv, ps, mma, splits):
    set_knobs(monkeypatch, PKV_ATTN_MMA=mma)
    w = synth.Workload(name="fa-" + name, seed=660 + d + Hq + ps, batch=4, layers=1, num_q_heads=Hq,
                       num_kv_heads=Hkv, head_dim=d, page_size=ps, dtype=dt, quant=quant, seq_len=None,
                       seq_len_range=(1, 300), outlier_channels=4 if quant != "none" else 0,
                       outlier_scale=15.0)
    lens = np.array([47, 190, 16, 1], dtype=np.int32)
    steps = 5
    ld = load_workload(w, lens=lens, extra_pages=1)
    K = [s.k for s in ld.seqs]
    V = [s.v for s in ld.seqs]
    cur = lens.copy()
    for step in range(steps):
        toks = [synth.append_tokens(w, b, step) for b in range(w.batch)]
        kb = np.stack([t.k_bits[0] for t in toks])          # [B][Hkv][d]
        vb = np.stack([t.v_bits[0] for t in toks])
        cur = cur + 1
        q, qf = queries_dev(w, step=step)
        out = ld.cache.append_attention(bits_to_torch(kb, dt).cuda(), bits_to_torch(vb, dt).cuda(), q,
                                        ld.bt_dev, torch.from_numpy(cur.copy()).cuda(), sm_scale=w.sm_scale,
                                        num_splits=splits, dev_status=ld.status)
        out = out.cpu().numpy()
        for b in range(w.batch):
            K[b] = np.concatenate([K[b], toks[b].k])
            V[b] = np.concatenate([V[b], toks[b].v])
            if quant == "none":
                kd, vd = K[b].astype(np.float64), V[b].astype(np.float64)
            else:
                kd = per_token_dequant(*oracle.quantize_per_token(K[b]))
                vd = per_token_dequant(*oracle.quantize_per_token(V[b]))
            for h in range(Hq):
                g = h // w.group
                o = oracle.decode_attention_tokens(qf[b, h], kd[:, g], vd[:, g], w.sm_scale)
                tol = TOL["int8"] if quant != "none" else TOL[dt]
                assert np.abs(out[b, h] - o).max() <= tol, (step, b, h)
    # the stored rows equal what kv_append would have written
    c = ld.cache
    for b in range(w.batch):
        L = int(cur[b])
        if quant == "none":
            kp = c.k_pages.view(torch.int16).cpu().numpy().view(np.uint16)
            want = np.concatenate([ld.seqs[b].k_bits] + [synth.append_tokens(w, b, s).k_bits for s in range(steps)])
            assert np.array_equal(gather(kp, ld.bt[b], L, ps), want)
        else:
            kc, ks, kz = oracle.quantize_per_token(K[b])
            vc, vs, vz = oracle.quantize_per_token(V[b])
            sz = gather(c.kv_sz.cpu().numpy(), ld.bt[b], L, ps)
            assert np.array_equal(int8_codes(gather(c.k_pages.cpu().numpy(), ld.bt[b], L, ps)), kc)
            assert np.array_equal(int8_codes(gather(c.v_pages.cpu().numpy(), ld.bt[b], L, ps)), vc)
            assert np.array_equal(sz[:, :, 0].view(np.uint32), ks.view(np.uint32))
            assert np.array_equal(sz[:, :, 1].view(np.uint32), kz.view(np.uint32))
            assert np.array_equal(sz[:, :, 2].view(np.uint32), vs.view(np.uint32))
            assert np.array_equal(sz[:, :, 3].view(np.uint32), vz.view(np.uint32))
    assert int(ld.status.item()) == 0


TWO_LAUNCH_CASES = [
    # name, dtype, quant, d, Hq, Hkv, page, boxes
    ("i8-group-gqa", "f16", "per_group64", 128, 16, 4, 64, False),
    ("i8-group-gqa-boxes", "f16", "per_group64", 64, 8, 2, 128, True),
    ("i8-token-boxes", "f16", "per_token", 128, 16, 4, 16, True),
    ("bf16-boxes", "bf16", "none", 64, 8, 8, 16, True),
]


@pytest.mark.parametrize("splits", [0, 5])
@pytest.mark.parametrize("name,dt,quant,d,Hq,Hkv,ps,boxes", TWO_LAUNCH_CASES)
def test_append_attention_two_launch_caches(name, dt, quant, d, Hq, Hkv, ps, boxes, splits):
    # per-group INT8 and caches with page boxes: the call appends with the
    # kv_append kernels, then attends; codes, scales, boxes and outputs as the
    # two separate calls would give them. The steps cross a 64-token group
    # close (lengths 63 and 64 at the start) and start a new page.
    from helpers import oracle_bbox_keys
    w = synth.Workload(name="fa2-" + name, seed=770 + d + Hq + ps, batch=4, layers=1, num_q_heads=Hq,
                       num_kv_heads=Hkv, head_dim=d, page_size=ps, dtype=dt, quant=quant, seq_len=None,
                       seq_len_range=(1, 300), outlier_channels=4 if quant != "none" else 0,
                       outlier_scale=15.0)
    lens = np.array([63, 190, 64, 1], dtype=np.int32)
    steps = 4
    ld = load_workload(w, lens=lens, extra_pages=1, with_meta=boxes)
    K = [s.k for s in ld.seqs]
    V = [s.v for s in ld.seqs]
    Kb = [s.k_bits for s in ld.seqs]
    Vb = [s.v_bits for s in ld.seqs]
    cur = lens.copy()
    for step in range(steps):
        toks = [synth.append_tokens(w, b, step) for b in range(w.batch)]
        kb = np.stack([t.k_bits[0] for t in toks])
        vb = np.stack([t.v_bits[0] for t in toks])
        cur = cur + 1
        q, qf = queries_dev(w, step=step)
        out = ld.cache.append_attention(bits_to_torch(kb, dt).cuda(), bits_to_torch(vb, dt).cuda(), q,
                                        ld.bt_dev, torch.from_numpy(cur.copy()).cuda(), sm_scale=w.sm_scale,
                                        num_splits=splits, dev_status=ld.status)
        out = out.cpu().numpy()
        for b in range(w.batch):
            K[b] = np.concatenate([K[b], toks[b].k])
            V[b] = np.concatenate([V[b], toks[b].v])
            Kb[b] = np.concatenate([Kb[b], toks[b].k_bits])
            Vb[b] = np.concatenate([Vb[b], toks[b].v_bits])
            if quant == "none":
                kd, vd = K[b].astype(np.float64), V[b].astype(np.float64)
            elif quant == "per_token":
                kd = per_token_dequant(*oracle.quantize_per_token(K[b]))
                vd = per_token_dequant(*oracle.quantize_per_token(V[b]))
            else:
                kd = per_group_dequant(*oracle.quantize_per_group(K[b]))
                vd = per_group_dequant(*oracle.quantize_per_group(V[b]))
            for h in range(Hq):
                g = h // w.group
                o = oracle.decode_attention_tokens(qf[b, h], kd[:, g], vd[:, g], w.sm_scale)
                tol = TOL["int8"] if quant != "none" else TOL[dt]
                assert np.abs(out[b, h] - o).max() <= tol, (step, b, h)
    c = ld.cache
    for b in range(w.batch):
        L = int(cur[b])
        if quant == "none":
            kp = c.k_pages.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(gather(kp, ld.bt[b], L, ps), Kb[b])
        elif quant == "per_token":
            kc, ks, kz = oracle.quantize_per_token(K[b])
            assert np.array_equal(int8_codes(gather(c.k_pages.cpu().numpy(), ld.bt[b], L, ps)), kc)
        else:
            kc, ks, kz = oracle.quantize_per_group(K[b])
            vc, vs, vz = oracle.quantize_per_group(V[b])
            assert np.array_equal(int8_codes(gather(c.k_pages.cpu().numpy(), ld.bt[b], L, ps)), kc)
            assert np.array_equal(int8_codes(gather(c.v_pages.cpu().numpy(), ld.bt[b], L, ps)), vc)
        if boxes:
            sd = synth.SeqData(k_bits=Kb[b], v_bits=Vb[b], k=K[b], v=V[b])
            mn, mx = oracle.page_bounding_boxes(oracle_bbox_keys(w, sd), ps)
            P = mn.shape[0]
            meta = c.page_meta.cpu().numpy()[ld.bt[b][:P]]
            assert np.array_equal(meta[:, :, 0].view(np.uint32), mn.view(np.uint32)), b
            assert np.array_equal(meta[:, :, 1].view(np.uint32), mx.view(np.uint32)), b
    assert int(ld.status.item()) == 0
