"""Pins of the oracle's byte/page counting against figures printed on the pages (no GPU)."""
import json
import os

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kv_size_expression():
    g = json.load(open(os.path.join(GOLDEN, "kv_size_example.json")))
    f = g["factors"]
    got = oracle.kv_cache_bytes(f["layers"], f["batch"], f["heads"], f["seq_len"], f["head_dim"], f["bytes_per_elem"])
    assert got == g["product_bytes"] == 8 * 2**30
    # the printed figure is not the product (recorded discrepancy)
    assert abs(got / 1e9 - g["printed_figure_gb"]) > 10


def test_bf16_step_volume_of_llama_shapes():
    # same shapes in bf16: 4.29 GB read per 32-layer decode step
    assert oracle.kv_cache_bytes(32, 4, 32, 2048, 128, 2) == 4294967296


def test_alignment_table():
    g = json.load(open(os.path.join(GOLDEN, "alignment_table.json")))
    for row in g["rows"]:
        per_token_kb = row["unaligned_kb"] / row["tokens"]
        assert per_token_kb == 16
        aligned = oracle.blocks_needed(row["tokens"], 16) * 16 * per_token_kb
        assert aligned == row["aligned_kb"]
        red = 100.0 * (aligned - row["unaligned_kb"]) / row["unaligned_kb"]
        assert round(red, 2) == row["redundancy_pct"]


def test_blocks_needed():
    assert oracle.blocks_needed(0, 16) == 0
    assert oracle.blocks_needed(1, 16) == 1
    assert oracle.blocks_needed(16, 16) == 1
    assert oracle.blocks_needed(17, 16) == 2
