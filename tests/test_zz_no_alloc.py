"""The allocation-free attention entry point (pkv_paged_decode_attention_noalloc).

It serves callers that cannot allocate device memory at call time, for example
a program that reserves all device memory up front, or a plugin that only gets
its input and output buffers. It runs on the library's fixed device scratch
instead of a caller workspace. Its results must match the regular entry point
on back-to-back calls: the shared scratch keeps the previous call's contents,
and nothing of it may leak into the next result.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from helpers import TOL, load_workload, max_abs_err, oracle_dense, queries_dev

pytestmark = pytest.mark.gpu


def noalloc_attention(ld, q, out_dtype=torch.float32, num_splits=0, sel=None, cnt=None, sel_shared=0,
                      out=None):
    from paged_kv_cache_243_gb300 import binding as B
    from paged_kv_cache_243_gb300.cache import pkv_dtype
    Bsz, Hq, d = q.shape
    if out is None:
        out = torch.empty((Bsz, Hq, d), dtype=out_dtype, device=q.device)
    B.paged_decode_attention_noalloc(
        ld.cache.descriptor(), Bsz, Hq, q.data_ptr(), pkv_dtype(q), float(ld.w.sm_scale),
        ld.bt_dev.data_ptr(), ld.bt_dev.shape[1], ld.lens_dev.data_ptr(),
        0 if sel is None else sel.data_ptr(), 0 if cnt is None else cnt.data_ptr(),
        0 if sel is None else sel.shape[2], out.data_ptr(), pkv_dtype(out), num_splits,
        ld.status.data_ptr(), torch.cuda.current_stream().cuda_stream, sel_shared=sel_shared)
    return out


def two_calls(ld):
    """Two calls in a row, each with its own queries, against the regular entry point."""
    for step in range(2):
        q, qf = queries_dev(ld.w, step=step)
        got = noalloc_attention(ld, q)
        want = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=ld.w.sm_scale,
                                  dev_status=ld.status)
        torch.cuda.synchronize()
        got, want = got.cpu().numpy(), want.cpu().numpy()
        tol = TOL["int8"] if ld.w.quant != "none" else TOL[ld.w.dtype]
        assert np.abs(got - want).max() <= tol, step
        assert max_abs_err(got, oracle_dense(ld, qf)) <= tol, step
    assert int(ld.status.item()) == 0


def test_noalloc_matches_regular_dense():
    w = dataclasses.replace(synth.WORKLOADS["w2_llama7b_bf16"], batch=3, layers=1)
    two_calls(load_workload(w, lens=np.array([700, 5, 2048], dtype=np.int32)))


def test_noalloc_matches_regular_gqa_int8():
    w = synth.Workload(name="na", seed=610, batch=4, layers=1, num_q_heads=16, num_kv_heads=4,
                       head_dim=128, page_size=16, dtype="f16", quant="per_token", seq_len=None,
                       seq_len_range=(1, 3000), outlier_channels=4, outlier_scale=15.0)
    two_calls(load_workload(w, lens=np.array([3000, 1, 129, 1777], dtype=np.int32)))


def test_noalloc_rejects_oversized_scratch():
    # a split count this large needs far more than the fixed scratch holds
    from paged_kv_cache_243_gb300 import binding as B
    w = dataclasses.replace(synth.WORKLOADS["w1_tiny_f16"], batch=1, seq_len=64)
    ld = load_workload(w)
    q, _ = queries_dev(w)
    with pytest.raises(B.PkvError) as e:
        noalloc_attention(ld, q, num_splits=200000)
    assert e.value.status == B.ERR_WORKSPACE


@pytest.mark.parametrize("group_mode", [0, 1])
def test_noalloc_matches_regular_sparse(group_mode):
    # sparse calls: page lists per query head (group_mode 0), and one list per
    # kv head shared by its query-head group (group_mode 1, sel_shared = 1)
    w = synth.Workload(name="nas", seed=640 + group_mode, batch=3, layers=1, num_q_heads=16, num_kv_heads=4,
                       head_dim=64, page_size=16, dtype="f16", quant="none", seq_len=None,
                       seq_len_range=(1, 900), page_offset_std=0.5)
    ld = load_workload(w, lens=np.array([900, 40, 333], dtype=np.int32), with_meta=True)
    for step in range(2):
        q, _ = queries_dev(w, step=step)
        sel, cnt, _ = ld.cache.score_topk(q, ld.bt_dev, ld.lens_dev, 7, dev_status=ld.status,
                                          group_mode=group_mode)
        got = noalloc_attention(ld, q, sel=sel, cnt=cnt, sel_shared=group_mode)
        want = ld.cache.attention(q, ld.bt_dev, ld.lens_dev, sm_scale=w.sm_scale, sel=sel, sel_count=cnt,
                                  sel_shared=bool(group_mode), dev_status=ld.status)
        torch.cuda.synchronize()
        assert np.abs(got.cpu().numpy() - want.cpu().numpy()).max() <= TOL["f16"], step
    assert int(ld.status.item()) == 0


def test_noalloc_later_calls_take_no_device_memory():
    # the first call on a device loads the library's scratch array; a call
    # after it must leave the device's free memory unchanged
    w = dataclasses.replace(synth.WORKLOADS["w2_llama7b_bf16"], batch=2, layers=1)
    ld = load_workload(w, lens=np.array([1000, 77], dtype=np.int32))
    q, qf = queries_dev(w)
    out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    noalloc_attention(ld, q, out=out)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    noalloc_attention(ld, q, out=out)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0
    assert max_abs_err(out.cpu().numpy(), oracle_dense(ld, qf)) <= TOL["bf16"]
    assert int(ld.status.item()) == 0
