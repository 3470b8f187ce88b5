"""Dense paged decode attention on the GPU against the oracle (fp16/bf16 caches)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (TOL, bits_to_torch, gather, load_workload, max_abs_err, oracle_dense, queries_dev,
                     set_knobs)

pytestmark = pytest.mark.gpu


def run_attention(ld, q, **kw):
    out = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=ld.w.sm_scale, dev_status=ld.status, **kw)
    torch.cuda.synchronize()
    return out


def test_w1_tiny_all_outputs_and_addressing():
    w = synth.WORKLOADS["w1_tiny_f16"]
    ld = load_workload(w)
    # addressing: the pools read back through the block table give the input bits
    kp = ld.cache.k_pages.view(torch.int16).cpu().numpy().view(np.uint16)
    vp = ld.cache.v_pages.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(w.batch):
        L = int(ld.lens[b])
        assert np.array_equal(gather(kp, ld.bt[b], L, w.page_size), ld.seqs[b].k_bits)
        assert np.array_equal(gather(vp, ld.bt[b], L, w.page_size), ld.seqs[b].v_bits)
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    for splits in (0, 1, 2, 7):
        out = run_attention(ld, q, num_splits=splits).cpu().numpy()
        assert max_abs_err(out, ref) <= TOL["f16"], splits
    assert int(ld.status.item()) == 0


def test_w2_llama_layer_full_size():
    w = synth.WORKLOADS["w2_llama7b_bf16"]
    ld = load_workload(w, layer=0)
    q, qf = queries_dev(w, layer=0)
    out = run_attention(ld, q).cpu().numpy()
    ref = oracle_dense(ld, qf)
    assert max_abs_err(out, ref) <= TOL["bf16"]
    assert int(ld.status.item()) == 0


def test_split_count_invariance():
    w = dataclasses.replace(synth.WORKLOADS["w2_llama7b_bf16"], batch=3, layers=1)
    ld = load_workload(w, lens=np.array([1000, 37, 513], dtype=np.int32))
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    outs = [run_attention(ld, q, num_splits=s).cpu().numpy() for s in (1, 2, 7, 0, 1000)]
    for o in outs:
        assert max_abs_err(o, ref) <= TOL["bf16"]
        assert np.abs(o - outs[0]).max() <= 1e-5


def test_alternating_batch_sizes_on_one_kernel():
    # the kernel's shared-memory size grows with the batch (per-sequence unit
    # table); a smaller call in between must not leave a larger one unlaunchable
    w = dataclasses.replace(synth.WORKLOADS["w2_llama7b_bf16"], batch=8, layers=1)
    ld = load_workload(w, lens=np.array([300, 17, 64, 129, 1, 250, 33, 90], dtype=np.int32))
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    for rows in (8, 1, 8, 3, 8):
        out = ld.cache.attention(q[:rows].contiguous(), ld.bt_dev[:rows].contiguous(),
                                 ld.lens_dev[:rows].contiguous(), sm_scale=w.sm_scale,
                                 dev_status=ld.status)
        torch.cuda.synchronize()
        sub = {k: v for k, v in ref.items() if k[0] < rows}
        assert max_abs_err(out.cpu().numpy(), sub) <= TOL["bf16"], rows
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("stages,per_sm", [("3", "1"), ("4", "1"), ("5", "2"), ("12", "0"), ("32", "0")])
def test_ring_depth_and_blocks_per_sm(monkeypatch, stages, per_sm):
    # the stage count is rounded to a multiple of the consumer warps, so every
    # ring slot has a single reader; results must not depend on these knobs
    set_knobs(monkeypatch, PKV_ATTN_STAGES=stages, PKV_ATTN_CTAS_PER_SM=per_sm)
    w = dataclasses.replace(synth.WORKLOADS["w2_llama7b_bf16"], batch=2, layers=1)
    ld = load_workload(w, lens=np.array([700, 333], dtype=np.int32))
    q, qf = queries_dev(w)
    out = run_attention(ld, q).cpu().numpy()
    assert max_abs_err(out, oracle_dense(ld, qf)) <= TOL["bf16"]
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("mma", ["1", "0"])
@pytest.mark.parametrize("d,Hq,Hkv,ps,dt", [
    (64, 4, 4, 16, "f16"), (64, 8, 4, 32, "bf16"), (64, 16, 4, 16, "f16"), (64, 16, 2, 64, "f16"),
    (128, 8, 8, 16, "bf16"), (128, 8, 4, 48, "f16"), (128, 16, 4, 16, "bf16"), (128, 16, 2, 32, "f16"),
    (128, 32, 4, 16, "bf16"),
])
def test_shapes_ragged_lengths(monkeypatch, d, Hq, Hkv, ps, dt, mma):
    set_knobs(monkeypatch, PKV_ATTN_MMA=mma)
    w = synth.Workload(name="t", seed=77 + d + Hq + ps, batch=5, layers=1, num_q_heads=Hq,
                       num_kv_heads=Hkv, head_dim=d, page_size=ps, dtype=dt, quant="none",
                       seq_len=None, seq_len_range=(1, 300))
    lens = np.array([1, 17, 0, 300, 129], dtype=np.int32)
    ld = load_workload(w, lens=lens)
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    for splits in (0, 3):
        out = run_attention(ld, q, num_splits=splits).cpu().numpy()
        assert max_abs_err(out, ref) <= TOL[dt]
        assert (out[2] == 0).all()          # empty sequence -> zeros
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_q_f32_and_low_precision_out(out_dtype):
    w = dataclasses.replace(synth.WORKLOADS["w1_tiny_f16"], batch=2, seq_len=200)
    ld = load_workload(w)
    _, qf = queries_dev(w)
    q32 = torch.from_numpy(qf).cuda()
    ref = oracle_dense(ld, qf)
    out = run_attention(ld, q32, out_dtype=out_dtype).float().cpu().numpy()
    # compared against the oracle rounded to the output dtype, plus half an ulp
    ulp = 2.0 ** -10 if out_dtype == torch.float16 else 2.0 ** -7
    for (b, h), o in ref.items():
        r = torch.from_numpy(o.astype(np.float32)).to(out_dtype).float().numpy()
        assert np.abs(out[b, h] - r).max() <= TOL["f16"] + 0.5 * ulp * max(1.0, np.abs(o).max())


def test_bad_block_table_entry_is_reported_and_skipped():
    w = dataclasses.replace(synth.WORKLOADS["w1_tiny_f16"], batch=2, seq_len=64)
    ld = load_workload(w)
    q, qf = queries_dev(w)
    bt = ld.bt.copy()
    bt[1, 2] = ld.cache.num_pages + 5      # out of range: must not be read
    ld.bt_dev = torch.from_numpy(bt).cuda()
    ld.status.zero_()
    out = run_attention(ld, q).cpu().numpy()
    from paged_kv_cache_243_gb300 import binding as B
    assert int(ld.status.item()) & B.DEV_BAD_PAGE
    # sequence 0 is untouched; sequence 1 attends over its other 48 tokens
    ref0 = oracle_dense(ld, qf, [(0, h) for h in range(w.num_q_heads)])
    assert max_abs_err(out, ref0) <= TOL["f16"]
    keep = [t for t in range(64) if t // 16 != 2]
    for h in range(w.num_q_heads):
        o = oracle.decode_attention_tokens(qf[1, h], ld.seqs[1].k[keep, h], ld.seqs[1].v[keep, h], w.sm_scale)
        assert np.abs(out[1, h] - o).max() <= TOL["f16"]


def test_seq_len_beyond_block_table_is_clamped_and_reported():
    w = dataclasses.replace(synth.WORKLOADS["w1_tiny_f16"], batch=1, seq_len=64)
    ld = load_workload(w)
    q, qf = queries_dev(w)
    lens = torch.tensor([64 + 10 * 16], dtype=torch.int32, device="cuda")
    ld.status.zero_()
    out = ld.cache.attention(q, ld.bt_dev[:, :4].contiguous(), lens, dev_status=ld.status)
    torch.cuda.synchronize()
    from paged_kv_cache_243_gb300 import binding as B
    assert int(ld.status.item()) & B.DEV_BAD_POSITION
    assert max_abs_err(out.cpu().numpy(), oracle_dense(ld, qf)) <= TOL["f16"]


def test_host_side_errors():
    from paged_kv_cache_243_gb300 import binding as B
    w = dataclasses.replace(synth.WORKLOADS["w1_tiny_f16"], batch=1, seq_len=32)
    ld = load_workload(w)
    q, _ = queries_dev(w)
    with pytest.raises(B.PkvError) as e:
        ld.cache.attention(q[:, :3].contiguous(), ld.bt_dev, ld.lens_dev)   # Hq % Hkv != 0
    assert e.value.status == B.ERR_INVALID_ARG
    desc = ld.cache.descriptor()
    with pytest.raises(B.PkvError) as e:
        B.paged_decode_attention(desc, 1, 4, q.data_ptr(), B.F16, 0.125, ld.bt_dev.data_ptr(), 2,
                                 ld.lens_dev.data_ptr(), 0, 0, 0, q.data_ptr(), B.F32, 0, 0, 0, 0, 0)
    assert e.value.status == B.ERR_WORKSPACE


def _dense_ref_all(ld, qf, k_last=None, v_last=None):
    """Oracle outputs of every (sequence, query head), optionally with the last
    token of each sequence replaced by (k_last[b], v_last[b]) [Hkv][d]."""
    w = ld.w
    res = {}
    for b in range(w.batch):
        k = ld.seqs[b].k
        v = ld.seqs[b].v
        if k_last is not None:
            k = k.copy()
            v = v.copy()
            k[-1] = k_last[b]
            v[-1] = v_last[b]
        for h in range(w.num_q_heads):
            g = h // w.group
            res[(b, h)] = oracle.decode_attention_tokens(qf[b, h], k[:, g, :], v[:, g, :], w.sm_scale)
    return res


@pytest.mark.slow
def test_dense_32k_bf16_all_outputs():
    # The 32K dense bf16 workload (4 sequences x 32768 tokens, 32 = 32 heads,
    # d = 128, page 16) in the launch configuration of the benchmark: automatic
    # split count, early start after the previous call (fresh_rows = 0), and the
    # one-call decode step that writes the token at position 32767 itself.
    # Every one of the 128 outputs is compared with the oracle.
    w = synth.WORKLOADS["dense_32k_bf16"]
    ld = load_workload(w)
    q, qf = queries_dev(w)
    ref = _dense_ref_all(ld, qf)
    for fresh in (-1, 0):
        out = run_attention(ld, q, fresh_rows=fresh).cpu().numpy()
        assert max_abs_err(out, ref) <= TOL["bf16"], fresh
    assert int(ld.status.item()) == 0
    # decode step: the token at position L - 1 is overwritten by the new one
    toks = [synth.append_tokens(w, b, 0) for b in range(w.batch)]
    kb = np.stack([t.k_bits[0] for t in toks])
    vb = np.stack([t.v_bits[0] for t in toks])
    q2, qf2 = queries_dev(w, step=1)
    out = ld.cache.append_attention(bits_to_torch(kb, "bf16").cuda(), bits_to_torch(vb, "bf16").cuda(), q2,
                                    ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale, dev_status=ld.status,
                                    fresh_rows=0)
    torch.cuda.synchronize()
    ref2 = _dense_ref_all(ld, qf2, [t.k[0] for t in toks], [t.v[0] for t in toks])
    assert max_abs_err(out.cpu().numpy(), ref2) <= TOL["bf16"]
    # the stored row is the new token's bits
    kp = ld.cache.k_pages.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(w.batch):
        L = int(ld.lens[b])
        t = L - 1
        assert np.array_equal(kp[ld.bt[b][t // w.page_size], :, t % w.page_size], kb[b])
    assert int(ld.status.item()) == 0


@pytest.mark.parametrize("g1", ["0", "2"])
@pytest.mark.parametrize("d,dt", [(64, "f16"), (128, "bf16"), (64, "bf16"), (128, "f16")])
def test_single_query_heads_on_tensor_cores(monkeypatch, g1, d, dt):
    # one query head per kv head: the tensor-core consumer (PKV_ATTN_MMA_G1=2,
    # every head_dim) against the CUDA-core one (0) and the oracle, ragged
    # lengths, an empty sequence and split counts from one block per unit to
    # more blocks than chunks
    set_knobs(monkeypatch, PKV_ATTN_MMA_G1=g1)
    w = synth.Workload(name="t", seed=501 + d, batch=5, layers=1, num_q_heads=6, num_kv_heads=6,
                       head_dim=d, page_size=16, dtype=dt, quant="none", seq_len=None,
                       seq_len_range=(1, 700))
    lens = np.array([700, 1, 0, 333, 64], dtype=np.int32)
    ld = load_workload(w, lens=lens)
    q, qf = queries_dev(w)
    ref = oracle_dense(ld, qf)
    for splits in (0, 1, 3, 1000):
        out = run_attention(ld, q, num_splits=splits).cpu().numpy()
        assert max_abs_err(out, ref) <= TOL[dt], splits
        assert (out[2] == 0).all()
    assert int(ld.status.item()) == 0
