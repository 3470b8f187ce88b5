"""The seeded generators are deterministic and round like the hardware does."""
import numpy as np
import torch

import synth


def test_deterministic_and_independent_per_sequence():
    w = synth.WORKLOADS["w3_gqa_int8_token"]
    a = synth.seq_tokens(w, 3, length=100)
    b = synth.seq_tokens(w, 3, length=100)
    assert np.array_equal(a.k_bits, b.k_bits) and np.array_equal(a.v_bits, b.v_bits)
    c = synth.seq_tokens(w, 4, length=100)
    assert not np.array_equal(a.k_bits, c.k_bits)
    lens = synth.seq_lens(w)
    assert lens.min() >= 1024 and lens.max() <= 32768 and len(lens) == 16


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * rng.uniform(0.001, 1000, 100000)).astype(np.float32)
    bits, vals = synth.round_to_dtype(x, "bf16")
    t = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(bits.view(np.int16), t.view(torch.int16).numpy())
    assert np.array_equal(vals, t.float().numpy())


def test_block_tables_are_permutations():
    w = synth.WORKLOADS["w2_llama7b_bf16"]
    bt, pool = synth.block_tables(w, layer=3)
    assert bt.shape == (4, 128) and pool == 512
    assert sorted(bt.ravel().tolist()) == list(range(512))
    w1 = synth.WORKLOADS["w1_tiny_f16"]
    bt1, pool1 = synth.block_tables(w1)
    assert bt1.shape == (1, 16) and pool1 == 32 and len(set(bt1.ravel().tolist())) == 16


def test_outliers_and_page_offsets():
    w = synth.WORKLOADS["w3_gqa_int8_token"]
    oc = synth.outlier_channels(w)
    assert oc.shape == (8, 4)
    sd = synth.seq_tokens(w, 0, length=2000)
    sdv = sd.k.std(axis=0)          # [Hkv][d]
    for g in range(8):
        rest = np.setdiff1d(np.arange(128), oc[g])
        assert sdv[g, oc[g]].min() > 10 * sdv[g, rest].max()
    w5 = synth.WORKLOADS["w5_sparse_f16"]
    s5 = synth.seq_tokens(w5, 0, length=64)
    means = s5.k.reshape(4, 16, 16, 64).mean(axis=1)
    assert means.std() > 0.3
