"""INT8 caches on the GPU: codes, scales and zero-points bit-exact against the
oracle's quantiser; attention over the restored values within tolerance."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (TOL, bits_to_torch, gather, load_workload, max_abs_err, oracle_dense,
                     queries_dev)

pytestmark = pytest.mark.gpu


def pools(ld):
    c = ld.cache
    return (c.k_pages.cpu().numpy(), c.v_pages.cpu().numpy(), c.kv_sz.cpu().numpy())


def check_per_token_codes(ld):
    kp, vp, sz = pools(ld)
    ps = ld.w.page_size
    for b in range(ld.w.batch):
        L = int(ld.lens[b])
        for x, pool, col in ((ld.seqs[b].k, kp, 0), (ld.seqs[b].v, vp, 2)):
            c, s, z = oracle.quantize_per_token(x)
            assert np.array_equal(gather(pool, ld.bt[b], L, ps), c)
            g = gather(sz, ld.bt[b], L, ps)             # [L][Hkv][4]
            assert np.array_equal(g[:, :, col].view(np.uint32), s.view(np.uint32))
            assert np.array_equal(g[:, :, col + 1].view(np.uint32), z.view(np.uint32))


def check_per_group_codes(ld):
    kp, vp, sz = pools(ld)
    ps = ld.w.page_size
    for b in range(ld.w.batch):
        L = int(ld.lens[b])
        for x, pool, col in ((ld.seqs[b].k, kp, 0), (ld.seqs[b].v, vp, 2)):
            c, s, z = oracle.quantize_per_group(x)
            assert np.array_equal(gather(pool, ld.bt[b], L, ps), c)
            ng = s.shape[0]
            t0 = np.arange(ng) * 64
            gs = sz[ld.bt[b][t0 // ps], :, (t0 % ps) // 64]   # [ng][Hkv][4]
            assert np.array_equal(gs[:, :, col].view(np.uint32), s.view(np.uint32))
            assert np.array_equal(gs[:, :, col + 1].view(np.uint32), z.view(np.uint32))


def small_int8(quant, seed, d=128, Hq=8, Hkv=2, ps=None, batch=4, outliers=4):
    ps = ps or (16 if quant == "per_token" else 128)
    return synth.Workload(name="i8", seed=seed, batch=batch, layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                          head_dim=d, page_size=ps, dtype="f16", quant=quant, seq_len=None,
                          seq_len_range=(1, 400), outlier_channels=outliers, outlier_scale=15.0)


@pytest.mark.parametrize("mma", ["1", "0"])
@pytest.mark.parametrize("d,Hq,Hkv", [(128, 8, 2), (64, 4, 4), (64, 16, 2), (128, 8, 8), (128, 16, 8)])
def test_per_token_small_all_outputs(monkeypatch, d, Hq, Hkv, mma):
    # mma = 1: query-head groups use the tensor-core kernel; 0: the CUDA-core one
    monkeypatch.setenv("PKV_ATTN_MMA", mma)
    w = small_int8("per_token", 300 + d + Hq, d, Hq, Hkv)
    ld = load_workload(w, lens=np.array([1, 400, 17, 250], dtype=np.int32))
    check_per_token_codes(ld)
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    for splits in (0, 1, 5):
        out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, num_splits=splits, dev_status=ld.status)
        assert max_abs_err(out.cpu().numpy(), ref) <= TOL["int8"]
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("mma", ["1", "0"])
@pytest.mark.parametrize("d,Hq,Hkv,ps", [(128, 8, 2, 128), (64, 8, 4, 64), (128, 32, 8, 256), (64, 16, 2, 64)])
def test_per_group_small_all_outputs(monkeypatch, d, Hq, Hkv, ps, mma):
    monkeypatch.setenv("PKV_ATTN_MMA", mma)
    w = small_int8("per_group64", 400 + d + ps, d, Hq, Hkv, ps)
    ld = load_workload(w, lens=np.array([1, 400, 64, 129], dtype=np.int32))
    check_per_group_codes(ld)
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    for splits in (0, 3):
        out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, num_splits=splits, dev_status=ld.status)
        assert max_abs_err(out.cpu().numpy(), ref) <= TOL["int8"]
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("chunks", [[1] * 130, [3, 61, 1, 64, 70, 2, 1], [200, 1, 1]])
def test_per_group_incremental_appends_equal_bulk(chunks):
    # the open 64-token group is re-quantised on every append from its kept
    # originals; the result equals quantising all tokens at once
    w = small_int8("per_group64", 500, 64, 4, 2, 64, batch=3)
    total = sum(chunks)
    ld = load_workload(w, lens=np.array([total, total - 5, total // 2], dtype=np.int32), chunks=chunks)
    check_per_group_codes(ld)
    assert int(ld.status.item()) == 0


def test_w3_full_size():
    w = synth.WORKLOADS["w3_gqa_int8_token"]
    ld = load_workload(w)
    check_per_token_codes(ld)
    q, qf = queries_dev(w)
    out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, dev_status=ld.status).cpu().numpy()
    rng = np.random.default_rng(3)
    units = [(int(b), int(h)) for b, h in zip(rng.integers(0, w.batch, 24), rng.integers(0, w.num_q_heads, 24))]
    units += [(int(np.argmax(ld.lens)), 0), (int(np.argmin(ld.lens)), w.num_q_heads - 1)]
    assert max_abs_err(out, oracle_dense(ld, qf, units)) <= TOL["int8"]
    assert int(ld.status.item()) == 0


def test_w4_full_size_append_steps():
    w = synth.WORKLOADS["w4_long_int8_group"]
    ld = load_workload(w, extra_pages=1)
    q, qf = queries_dev(w)
    lens = ld.lens.copy()
    K = [s.k for s in ld.seqs]
    V = [s.v for s in ld.seqs]
    check_steps = {0, 1, 2, 62, 63}
    for step in range(w.append_steps):
        toks = [synth.append_tokens(w, b, step) for b in range(w.batch)]
        kb = np.stack([t.k_bits for t in toks])
        vb = np.stack([t.v_bits for t in toks])
        pos = torch.from_numpy(lens.copy()).cuda()
        ld.cache.append(bits_to_torch(kb, "f16").cuda(), bits_to_torch(vb, "f16").cuda(), ld.bt_dev, pos,
                        dev_status=ld.status)
        lens += 1
        for b in range(w.batch):
            K[b] = np.concatenate([K[b], toks[b].k])
            V[b] = np.concatenate([V[b], toks[b].v])
        lens_dev = torch.from_numpy(lens.copy()).cuda()
        out = ld.cache.attention(q, ld.bt_dev, lens_dev, dev_status=ld.status)
        if step in check_steps:
            out = out.cpu().numpy()
            for b in range(w.batch):
                kc, ks, kz = oracle.quantize_per_group(K[b])
                vc, vs, vz = oracle.quantize_per_group(V[b])
                from oracle.quant import per_group_dequant
                kd, vd = per_group_dequant(kc, ks, kz), per_group_dequant(vc, vs, vz)
                for h in range(0, w.num_q_heads, 3):
                    g = h // w.group
                    o = oracle.decode_attention_tokens(qf[b, h], kd[:, g], vd[:, g], w.sm_scale)
                    assert np.abs(out[b, h] - o).max() <= TOL["int8"], (step, b, h)
    torch.cuda.synchronize()
    ld.lens = lens
    for b in range(w.batch):
        ld.seqs[b] = synth.SeqData(None, None, K[b], V[b])
    check_per_group_codes(ld)
    assert int(ld.status.item()) == 0
