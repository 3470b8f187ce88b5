"""4-bit KV quantisation as a sequence of IEEE-754 fp32 operations (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix: the KV-practice page, section 3.2 (its quantisation
table), lists a 4-bit scheme beside FP16 and INT8, saving 87.5 % of the
memory (4 bits per value against 32) and needing a dedicated kernel. The
pages define no format for it.

Readings taken (the plainest one the INT8 scheme of the same pages supports):
  * per token: one (scale, zero-point) per (token, kv head) over the head_dim
    channels, as per-token INT8 [HBM-layout page, section 二];
  * asymmetric form with a float zero-point equal to the minimum:
        s = (max - min) / 15        (fp32 subtract, fp32 divide)
        z = min
        u = clamp(rint((x - z) / s), 0, 15)    (fp32 ops, ties to even)
    so |x - x_hat| <= s/2; codes are unsigned 4-bit integers u in [0, 15];
  * a constant row (s == 0) stores s = 0 and all codes 0, restoring z;
  * restoration is x_hat = u * s + z, evaluated in fp64; the page boxes use
    fl32(fl32(u * s) + z), the fp32 value the kernels compute;
  * packing: two codes per byte, channel 2i in the low nibble and channel
    2i + 1 in the high nibble, so a row of d channels is d / 2 bytes.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

F32_15 = np.float32(15.0)


def quantize_block_u4(x) -> Tuple[np.ndarray, np.float32, np.float32]:
    """Quantise one block of values sharing one (scale, zero-point) to 4 bits.

    x: any shape, values exactly representable in fp32.
    Returns (uint8 codes in [0, 15] of x's shape, fp32 scale, fp32 zero-point).
    """
    x = np.asarray(x, dtype=np.float32)
    mn = np.float32(x.min())
    mx = np.float32(x.max())
    s = np.float32(np.float32(mx - mn) / F32_15)
    z = mn
    if s == np.float32(0.0):
        return np.zeros(x.shape, dtype=np.uint8), s, z
    t = (x - z).astype(np.float32)          # fp32 subtract
    t = (t / s).astype(np.float32)          # fp32 divide (IEEE, correctly rounded)
    u = np.clip(np.rint(t), 0.0, 15.0)      # round half to even
    return u.astype(np.uint8), s, z


def quantize_rows_u4(x) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """quantize_block_u4 applied independently to every row of a 2-D array.

    Returns (codes uint8 [n][m], scales fp32 [n], zeros fp32 [n]).
    """
    x = np.asarray(x, dtype=np.float32)
    mn = x.min(axis=1)
    mx = x.max(axis=1)
    s = ((mx - mn).astype(np.float32) / F32_15).astype(np.float32)
    const = s == np.float32(0.0)
    s_safe = np.where(const, np.float32(1.0), s).astype(np.float32)
    t = (x - mn[:, None]).astype(np.float32)
    t = (t / s_safe[:, None]).astype(np.float32)
    u = np.clip(np.rint(t), 0.0, 15.0)
    u[const] = 0.0
    return u.astype(np.uint8), s, mn


def quantize_per_token_u4(x) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Per-token 4-bit codes of one sequence's K or V.

    x: [L][Hkv][d]. Returns (codes uint8 [L][Hkv][d] in [0, 15],
    scales fp32 [L][Hkv], zeros fp32 [L][Hkv]).
    """
    x = np.asarray(x, dtype=np.float32)
    L, H, d = x.shape
    c, s, z = quantize_rows_u4(x.reshape(L * H, d))
    return c.reshape(L, H, d), s.reshape(L, H), z.reshape(L, H)


def pack_u4(codes) -> np.ndarray:
    """Two codes per byte along the last axis: channel 2i low nibble, 2i + 1 high."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_u4(packed) -> np.ndarray:
    """Inverse of pack_u4."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def dequantize_u4(codes, scale, zero) -> np.ndarray:
    """x_hat = u * s + z in fp64 (scale/zero broadcast against codes)."""
    return (np.asarray(codes, dtype=np.float64) * np.asarray(scale, dtype=np.float64)
            + np.asarray(zero, dtype=np.float64))


def per_token_u4_dequant(codes, scales, zeros) -> np.ndarray:
    """fp64 restoration of per-token 4-bit codes [L][Hkv][d] with scales [L][Hkv]."""
    return dequantize_u4(codes, np.asarray(scales)[:, :, None], np.asarray(zeros)[:, :, None])


def per_token_u4_bbox_values(codes, scales, zeros) -> np.ndarray:
    """fp32 restoration fl32(fl32(u * s) + z) of per-token 4-bit codes (page-box input)."""
    u = np.asarray(codes, dtype=np.float32)
    p = (u * np.asarray(scales, dtype=np.float32)[:, :, None]).astype(np.float32)
    return (p + np.asarray(zeros, dtype=np.float32)[:, :, None]).astype(np.float32)
