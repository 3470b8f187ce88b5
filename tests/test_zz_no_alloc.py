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


def noalloc_attention(ld, q, out_dtype=torch.float32, num_splits=0):
    from paged_kv_cache_243_gb300 import binding as B
    from paged_kv_cache_243_gb300.cache import pkv_dtype
    Bsz, Hq, d = q.shape
    out = torch.empty((Bsz, Hq, d), dtype=out_dtype, device=q.device)
    B.paged_decode_attention_noalloc(
        ld.cache.descriptor(), Bsz, Hq, q.data_ptr(), pkv_dtype(q), float(ld.w.sm_scale),
        ld.bt_dev.data_ptr(), ld.bt_dev.shape[1], ld.lens_dev.data_ptr(), 0, 0, 0, out.data_ptr(),
        pkv_dtype(out), num_splits, ld.status.data_ptr(), torch.cuda.current_stream().cuda_stream)
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
