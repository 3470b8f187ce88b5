"""Pins for the oracle's INT8 quantiser (no GPU)."""
import numpy as np
import pytest

import oracle
from oracle.quant import per_group_dequant, per_token_dequant


def test_hand_example_round_half_even():
    # min 0, max 255 -> s = 255/255 = 1 exactly, z = 0; codes = rint(x) - 128,
    # with 2.5 -> 2 and 3.5 -> 4 and 254.5 -> 254 (ties to even).
    x = np.array([0.0, 255.0, 2.5, 3.5, 1.0, 254.5], dtype=np.float32)
    c, s, z = oracle.quantize_block(x)
    assert s == np.float32(1.0) and z == np.float32(0.0)
    assert c.tolist() == [-128, 127, -126, -124, -127, 126]


def test_hand_example_offset_and_scale():
    # min -1, max 1.55 -> s = 2.55/255 (fp32) = 0.01 (fp32 rounding of the quotient)
    x = np.array([-1.0, 1.55, 0.0], dtype=np.float32)
    c, s, z = oracle.quantize_block(x)
    assert z == np.float32(-1.0)
    assert s == np.float32(np.float32(np.float32(1.55) - np.float32(-1.0)) / np.float32(255.0))
    assert c[0] == -128 and c[1] == 127
    # 0 sits 1.0 above the minimum: 1.0 / 0.01 = 100 levels -> code -28
    assert c[2] == -28


def test_constant_block():
    x = np.full((7, 5), 0.375, dtype=np.float32)
    c, s, z = oracle.quantize_block(x)
    assert s == 0 and z == np.float32(0.375)
    assert (c == -128).all()
    assert (oracle.dequantize(c, s, z) == 0.375).all()


def _fp16_values(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16).astype(np.float32)


def test_extremes_map_to_code_ends():
    rng = np.random.default_rng(5)
    for _ in range(200):
        x = _fp16_values(rng, 128, scale=rng.uniform(0.01, 20))
        c, s, z = oracle.quantize_block(x)
        assert c[np.argmin(x)] == -128
        assert c[np.argmax(x)] == 127


def test_round_trip_error_at_most_half_scale():
    # |x - x_hat| <= s/2 for per-token INT8 [HBM-layout page, section 二], up to
    # fp32 rounding: fl(x - z) errs by <= 2^-24 (max - min) = 2^-24 * 255 s and the
    # quotient (<= 255.x levels) by <= 2^-24 * 256 levels, i.e. <= 3.1e-5 s in all.
    rng = np.random.default_rng(7)
    x = _fp16_values(rng, (300, 8, 128))
    x[:, :, [3, 40, 77, 100]] *= 15
    x = x.astype(np.float16).astype(np.float32)
    c, s, z = oracle.quantize_per_token(x)
    xr = per_token_dequant(c, s, z)
    bound = s.astype(np.float64)[:, :, None] * (0.5 + 4e-5)
    assert (np.abs(xr - x) <= bound).all()
    # and the bound is not vacuous: some element sits close to it
    assert (np.abs(xr - x) / (s.astype(np.float64)[:, :, None] / 2)).max() > 0.99


def test_rows_match_blocks():
    rng = np.random.default_rng(9)
    x = _fp16_values(rng, (64, 96), scale=3)
    x[5] = 1.25  # a constant row
    c, s, z = oracle.quantize_rows(x)
    for i in range(x.shape[0]):
        cb, sb, zb = oracle.quantize_block(x[i])
        assert (cb == c[i]).all() and sb == s[i] and zb == z[i]


def test_group_round_trip_and_shapes():
    rng = np.random.default_rng(11)
    x = _fp16_values(rng, (200, 2, 16))
    c, s, z = oracle.quantize_per_group(x)
    assert s.shape == (4, 2)
    xr = per_group_dequant(c, s, z)
    gidx = np.arange(200) // 64
    bound = s.astype(np.float64)[gidx][:, :, None] * (0.5 + 4e-5)
    assert (np.abs(xr - x) <= bound).all()
    # each group's own min and max map to the code ends
    for gi in range(4):
        blk = x[gi * 64:(gi + 1) * 64, 1]
        cb = c[gi * 64:(gi + 1) * 64, 1]
        assert cb.flat[np.argmin(blk)] == -128 and cb.flat[np.argmax(blk)] == 127


@pytest.mark.parametrize("chunks", [[1] * 130, [3, 61, 1, 64, 70, 2, 1], [64, 64, 1], [200]])
def test_incremental_group_append_equals_bulk(chunks):
    rng = np.random.default_rng(13)
    total = sum(chunks)
    x = _fp16_values(rng, (total, 3, 8))
    model = oracle.GroupAppendModel(3, 8)
    pos = 0
    for n in chunks:
        model.append(x[pos:pos + n])
        pos += n
    c, s, z = oracle.quantize_per_group(x)
    assert (model.codes == c).all()
    assert (model.scale_array() == s).all() and (model.zero_array() == z).all()


def test_open_group_is_requantised():
    # after 1 token the group's scale covers that token only; after 2 it covers both
    x = np.array([[[0.0, 1.0]], [[4.0, -4.0]]], dtype=np.float32)
    m = oracle.GroupAppendModel(1, 2)
    m.append(x[:1])
    assert m.scale_array()[0, 0] == np.float32(1.0 / 255.0)
    m.append(x[1:])
    assert m.scale_array()[0, 0] == np.float32(np.float32(8.0) / np.float32(255.0))
    assert m.zero_array()[0, 0] == np.float32(-4.0)


def test_bbox_value_two_step_rounding():
    # fl32(fl32(u * s) + z): code 127 -> u = 255
    c = np.array([127, -128, 0], dtype=np.int8)
    s = np.float32(0.1)
    z = np.float32(-3.0)
    v = oracle.dequant_f32_two_step(c, s, z)
    assert v[0] == np.float32(np.float32(np.float32(255) * s) + z)
    assert v[1] == z
    assert v[2] == np.float32(np.float32(np.float32(128) * s) + z)
