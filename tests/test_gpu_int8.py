"""INT8 caches on the GPU: codes, scales and zero-points bit-exact against the
oracle's quantiser; attention over the restored values within tolerance."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (TOL, bits_to_torch, check_per_group_codes, check_per_token_codes, gather,
                     load_workload, max_abs_err, oracle_dense, queries_dev, set_knobs)

pytestmark = pytest.mark.gpu


def small_int8(quant, seed, d=128, Hq=8, Hkv=2, ps=None, batch=4, outliers=4):
    ps = ps or (16 if quant == "per_token" else 128)
    return synth.Workload(name="i8", seed=seed, batch=batch, layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                          head_dim=d, page_size=ps, dtype="f16", quant=quant, seq_len=None,
                          seq_len_range=(1, 400), outlier_channels=outliers, outlier_scale=15.0)


@pytest.mark.parametrize("mma", ["1", "0"])
@pytest.mark.parametrize("d,Hq,Hkv", [(128, 8, 2), (64, 4, 4), (64, 16, 2), (128, 8, 8), (128, 16, 8)])
def test_per_token_small_all_outputs(monkeypatch, d, Hq, Hkv, mma):
    # mma = 1: query-head groups use the tensor-core kernel; 0: the CUDA-core one
    set_knobs(monkeypatch, PKV_ATTN_MMA=mma)
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
    set_knobs(monkeypatch, PKV_ATTN_MMA=mma)
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
    # every (sequence, query head) output, in the benchmark's launch
    # configuration (automatic split count; early start after another call)
    ref = oracle_dense(ld, qf)
    for fresh in (-1, 0):
        out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, dev_status=ld.status,
                                 fresh_rows=fresh).cpu().numpy()
        assert max_abs_err(out, ref) <= TOL["int8"], fresh
    assert int(ld.status.item()) == 0


def test_w4_full_size_append_steps():
    w = synth.WORKLOADS["w4_long_int8_group"]
    ld = load_workload(w, extra_pages=1)
    q, qf = queries_dev(w)
    lens = ld.lens.copy()
    K = [s.k for s in ld.seqs]
    V = [s.v for s in ld.seqs]
    check_steps = {0, 1, 2, 62, 63}
    # every step's inputs are on the device before the first launch, so the
    # attention call follows its append directly on the stream and its early
    # start (fresh_rows = 1, as the benchmark's step runs it) overlaps it
    all_toks = [[synth.append_tokens(w, b, step) for b in range(w.batch)] for step in range(w.append_steps)]
    k_dev = [bits_to_torch(np.stack([t.k_bits for t in toks]), "f16").cuda() for toks in all_toks]
    v_dev = [bits_to_torch(np.stack([t.v_bits for t in toks]), "f16").cuda() for toks in all_toks]
    pos_dev = [torch.from_numpy(lens + step).cuda() for step in range(w.append_steps)]
    len_dev = [torch.from_numpy(lens + step + 1).cuda() for step in range(w.append_steps)]
    torch.cuda.synchronize()
    for step in range(w.append_steps):
        toks = all_toks[step]
        ld.cache.append(k_dev[step], v_dev[step], ld.bt_dev, pos_dev[step], dev_status=ld.status)
        lens += 1
        for b in range(w.batch):
            K[b] = np.concatenate([K[b], toks[b].k])
            V[b] = np.concatenate([V[b], toks[b].v])
        out = ld.cache.attention(q, ld.bt_dev, len_dev[step], dev_status=ld.status, fresh_rows=1)
        if step in check_steps:
            out = out.cpu().numpy()
            for b in range(w.batch):
                kc, ks, kz = oracle.quantize_per_group(K[b])
                vc, vs, vz = oracle.quantize_per_group(V[b])
                from oracle.quant import per_group_dequant
                kd, vd = per_group_dequant(kc, ks, kz), per_group_dequant(vc, vs, vz)
                for h in range(w.num_q_heads):
                    g = h // w.group
                    o = oracle.decode_attention_tokens(qf[b, h], kd[:, g], vd[:, g], w.sm_scale)
                    assert np.abs(out[b, h] - o).max() <= TOL["int8"], (step, b, h)
    torch.cuda.synchronize()
    ld.lens = lens
    for b in range(w.batch):
        ld.seqs[b] = synth.SeqData(None, None, K[b], V[b])
    check_per_group_codes(ld)
    assert int(ld.status.item()) == 0
