"""Pins for the oracle's 4-bit quantiser (no GPU)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_example_round_half_even():
    # min 0, max 15 -> s = 15/15 = 1 exactly, z = 0; codes = rint(x), with
    # 0.5 -> 0, 1.5 -> 2, 2.5 -> 2 and 14.5 -> 14 (ties to even)
    x = np.array([0.0, 0.5, 1.5, 2.5, 14.5, 15.0, 7.0], dtype=np.float32)
    c, s, z = oracle.quantize_block_u4(x)
    assert s == np.float32(1.0) and z == np.float32(0.0)
    assert c.tolist() == [0, 0, 2, 2, 14, 15, 7]


def test_hand_example_offset_and_scale():
    # min -1, max 2 -> s = fl32(3 / 15), the fp32 number nearest 0.2; z = -1.
    # 0 sits 1.0 above the minimum: 5 steps; 0.55 sits 1.55 above: 7.75 -> 8;
    # 1.0 sits 2.0 above: 10 steps (the quotients are far from half-integers)
    x = np.array([-1.0, 2.0, 0.0, 0.55, 1.0], dtype=np.float32)
    c, s, z = oracle.quantize_block_u4(x)
    assert z == np.float32(-1.0)
    assert s == np.float32(0.2)
    assert c.tolist() == [0, 15, 5, 8, 10]


def test_constant_block():
    x = np.full((5, 9), -2.25, dtype=np.float32)
    c, s, z = oracle.quantize_block_u4(x)
    assert s == 0 and z == np.float32(-2.25)
    assert (c == 0).all()
    assert (oracle.dequantize_u4(c, s, z) == -2.25).all()


def _fp16_values(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16).astype(np.float32)


def test_extremes_map_to_code_ends():
    rng = np.random.default_rng(15)
    for _ in range(200):
        x = _fp16_values(rng, 64, scale=rng.uniform(0.01, 20))
        c, s, z = oracle.quantize_block_u4(x)
        assert c[np.argmin(x)] == 0
        assert c[np.argmax(x)] == 15
        assert c.max() <= 15


def test_round_trip_error_at_most_half_scale():
    # |x - x_hat| <= s/2, up to fp32 rounding: fl(x - z) errs by <= 2^-24 (max -
    # min) = 2^-24 * 15 s and the quotient (<= 15.x levels) by <= 2^-24 * 16
    # levels, i.e. below 2e-6 s in all
    rng = np.random.default_rng(17)
    x = _fp16_values(rng, (300, 8, 128))
    x[:, :, [3, 40, 77, 100]] *= 15
    x = x.astype(np.float16).astype(np.float32)
    c, s, z = oracle.quantize_per_token_u4(x)
    xr = oracle.per_token_u4_dequant(c, s, z)
    bound = s.astype(np.float64)[:, :, None] * (0.5 + 4e-6)
    assert (np.abs(xr - x) <= bound).all()
    assert (np.abs(xr - x) / (s.astype(np.float64)[:, :, None] / 2)).max() > 0.99


def test_rows_match_blocks():
    rng = np.random.default_rng(19)
    x = _fp16_values(rng, (40, 64), scale=3)
    x[7] = 0.5   # a constant row
    c, s, z = oracle.quantize_rows_u4(x)
    for i in range(x.shape[0]):
        cb, sb, zb = oracle.quantize_block_u4(x[i])
        assert np.array_equal(c[i], cb) and s[i] == sb and z[i] == zb


def test_packing_low_nibble_is_the_even_channel():
    codes = np.array([[3, 12, 0, 15, 9, 1]], dtype=np.uint8)
    packed = oracle.pack_u4(codes)
    assert packed.tolist() == [[0xC3, 0xF0, 0x19]]
    rng = np.random.default_rng(21)
    c = rng.integers(0, 16, size=(17, 3, 128)).astype(np.uint8)
    assert np.array_equal(oracle.unpack_u4(oracle.pack_u4(c)), c)


def test_bbox_values_are_the_fp32_restoration():
    # fl32(fl32(u s) + z) against the fp64 restoration: equal to within one
    # fp32 rounding of each step
    rng = np.random.default_rng(23)
    x = _fp16_values(rng, (50, 2, 64), scale=4)
    c, s, z = oracle.quantize_per_token_u4(x)
    b32 = oracle.per_token_u4_bbox_values(c, s, z).astype(np.float64)
    b64 = oracle.per_token_u4_dequant(c, s, z)
    mag = np.abs(c.astype(np.float64) * s[:, :, None]) + np.abs(z[:, :, None])
    assert (np.abs(b32 - b64) <= mag * 2.0 ** -23).all()


def test_saving_table_of_the_pages():
    # the pages' table of savings is 1 - bits / 32 for FP16, INT8 and 4-bit
    g = json.load(open(os.path.join(GOLDEN, "quant_saving_table.json")))
    bits = {"FP16": 16, "INT8": 8, "4-bit": 4}
    full = oracle.kv_cache_bytes(32, 1, 32, 2048, 128, 4)
    for row in g["rows"]:
        stored = oracle.kv_cache_bytes(32, 1, 32, 2048, 128, bits[row["scheme"]] / 8)
        assert abs(100.0 * (1 - stored / full) - row["saving_pct"]) < 1e-9, row
