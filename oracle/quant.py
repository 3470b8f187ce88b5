"""INT8 KV quantisation as a sequence of IEEE-754 fp32 operations (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix:
  * per-token dynamic INT8: every token's K vector is quantised with its own
    min/max and restored before attention [HBM-layout page, section 二];
  * per-group INT8: every 64 tokens share one scale/zero-point [Gemini page,
    第一章 "KV Cache 优化核心策略"], stored as int8 [Gemini page, 第一章 code].

Readings where the pages are silent:
  * asymmetric form with a float zero-point equal to the block minimum:
        s = (max - min) / 255        (fp32 subtract, fp32 divide)
        z = min
        c = clamp(rint((x - z) / s), 0, 255) - 128     (fp32 ops, ties to even)
    so that |x - x_hat| <= s/2 holds; codes are signed int8 with a -128 bias;
  * a constant block (s == 0) stores s = 0 and all codes -128, restoring z;
  * dequantisation is x_hat = (c + 128) * s + z, evaluated in fp64;
  * a 64-token group that is still filling (the open group) is always the
    quantisation of its current members: each append re-quantises it from the
    kept originals, and closed groups never change (GroupAppendModel).
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import numpy as np

F32_255 = np.float32(255.0)


def quantize_block(x) -> Tuple[np.ndarray, np.float32, np.float32]:
    """Quantise one block of values that share a single (scale, zero-point).

    x: any shape, float values exactly representable in fp32.
    Returns (int8 codes of x's shape, fp32 scale, fp32 zero-point).
    Each arithmetic step is one correctly rounded fp32 operation.
    """
    x = np.asarray(x, dtype=np.float32)
    mn = np.float32(x.min())
    mx = np.float32(x.max())
    s = np.float32(np.float32(mx - mn) / F32_255)
    z = mn
    if s == np.float32(0.0):
        return np.full(x.shape, -128, dtype=np.int8), s, z
    t = (x - z).astype(np.float32)          # fp32 subtract
    t = (t / s).astype(np.float32)          # fp32 divide (IEEE, correctly rounded)
    u = np.rint(t)                          # round half to even
    u = np.clip(u, 0.0, 255.0)
    codes = (u - 128.0).astype(np.int8)
    return codes, s, z


def quantize_rows(x) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """quantize_block applied independently to every row of a 2-D array.

    x: [n][m] values exactly representable in fp32.
    Returns (codes int8 [n][m], scales fp32 [n], zeros fp32 [n]).
    """
    x = np.asarray(x, dtype=np.float32)
    mn = x.min(axis=1)
    mx = x.max(axis=1)
    s = ((mx - mn).astype(np.float32) / F32_255).astype(np.float32)
    z = mn
    const = s == np.float32(0.0)
    s_safe = np.where(const, np.float32(1.0), s).astype(np.float32)
    t = (x - z[:, None]).astype(np.float32)
    t = (t / s_safe[:, None]).astype(np.float32)
    u = np.clip(np.rint(t), 0.0, 255.0)
    u[const] = 0.0
    return (u - 128.0).astype(np.int8), s, z


def dequantize(codes, scale, zero) -> np.ndarray:
    """x_hat = (c + 128) * s + z in fp64 (scale/zero broadcast against codes)."""
    c = np.asarray(codes, dtype=np.float64)
    return (c + 128.0) * np.asarray(scale, dtype=np.float64) + np.asarray(zero, dtype=np.float64)


def dequant_f32_two_step(codes, scale, zero) -> np.ndarray:
    """fp32 restoration used for the page bounding boxes of an INT8 cache.

    fl32(fl32((c + 128) * s) + z): one fp32 multiply, then one fp32 add.
    (Reading: the pages keep the box in fp32 [TinyServe page, section 5.2] and
    build it from the keys [section 2.1]; for INT8 keys this is the value the
    box is built from.)
    """
    u = (np.asarray(codes, dtype=np.int16) + 128).astype(np.float32)
    p = (u * np.asarray(scale, dtype=np.float32)).astype(np.float32)
    return (p + np.asarray(zero, dtype=np.float32)).astype(np.float32)


def quantize_per_token(x) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Per-token INT8 of one sequence's K or V.

    x: [L][Hkv][d] fp32-exact values. One (scale, zero) per (token, kv head)
    over the d channels [HBM-layout page, section 二].
    Returns (codes int8 [L][Hkv][d], scales fp32 [L][Hkv], zeros fp32 [L][Hkv]).
    """
    x = np.asarray(x, dtype=np.float32)
    L, H, d = x.shape
    c, s, z = quantize_rows(x.reshape(L * H, d))
    return c.reshape(L, H, d), s.reshape(L, H), z.reshape(L, H)


def quantize_per_group(x, group: int = 64) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Per-group INT8 of one sequence's K or V (bulk: all tokens known).

    x: [L][Hkv][d]. Tokens [64 g, 64 g + 63] of one kv head share one
    (scale, zero) over all their 64 x d values [Gemini page, 第一章]; the last
    group holds the L % 64 remaining tokens when L is not a multiple of 64.
    Returns (codes [L][Hkv][d], scales fp32 [ceil(L/64)][Hkv], zeros fp32 [..][Hkv]).
    """
    x = np.asarray(x, dtype=np.float32)
    L, H, d = x.shape
    ng = -(-L // group)
    codes = np.empty((L, H, d), dtype=np.int8)
    s = np.zeros((ng, H), dtype=np.float32)
    z = np.zeros((ng, H), dtype=np.float32)
    for gi in range(ng):
        t0, t1 = gi * group, min(L, gi * group + group)
        for h in range(H):
            c, s[gi, h], z[gi, h] = quantize_block(x[t0:t1, h, :])
            codes[t0:t1, h, :] = c
    return codes, s, z


class GroupAppendModel:
    """Per-group INT8 state of one sequence under repeated appends.

    Keeps the original values of the open (partially filled) group, and on every
    append re-quantises each group that received tokens from all its members.
    Closed groups are never touched again. The reading is pinned by the
    invariant that any sequence of appends leaves the same codes, scales and
    zeros as quantising all tokens at once.
    """

    def __init__(self, num_kv_heads: int, head_dim: int, group: int = 64):
        self.H, self.d, self.group = num_kv_heads, head_dim, group
        self.codes = np.zeros((0, num_kv_heads, head_dim), dtype=np.int8)
        self.scales: List[np.ndarray] = []
        self.zeros: List[np.ndarray] = []
        self.open_values = np.zeros((0, num_kv_heads, head_dim), dtype=np.float32)

    @property
    def length(self) -> int:
        return self.codes.shape[0]

    def append(self, x) -> None:
        x = np.asarray(x, dtype=np.float32)
        G = self.group
        pos = self.length
        self.codes = np.concatenate([self.codes, np.zeros(x.shape, dtype=np.int8)])
        i = 0
        while i < x.shape[0]:
            gi = (pos + i) // G
            take = min(x.shape[0] - i, G * (gi + 1) - (pos + i))
            first_new = pos + i
            if first_new % G != 0:
                members = np.concatenate([self.open_values, x[i:i + take]])
            else:
                members = x[i:i + take]
            t0 = gi * G
            s = np.zeros(self.H, dtype=np.float32)
            z = np.zeros(self.H, dtype=np.float32)
            for h in range(self.H):
                c, s[h], z[h] = quantize_block(members[:, h, :])
                self.codes[t0:t0 + members.shape[0], h, :] = c
            if gi < len(self.scales):
                self.scales[gi], self.zeros[gi] = s, z
            else:
                self.scales.append(s)
                self.zeros.append(z)
            closed = (first_new + take) % G == 0
            self.open_values = (np.zeros((0, self.H, self.d), dtype=np.float32)
                                if closed else members.copy())
            i += take

    def scale_array(self) -> np.ndarray:
        return np.stack(self.scales) if self.scales else np.zeros((0, self.H), np.float32)

    def zero_array(self) -> np.ndarray:
        return np.stack(self.zeros) if self.zeros else np.zeros((0, self.H), np.float32)


def per_token_dequant(codes, scales, zeros) -> np.ndarray:
    """fp64 restoration of per-token codes [L][Hkv][d] with scales [L][Hkv]."""
    return dequantize(codes, np.asarray(scales)[:, :, None], np.asarray(zeros)[:, :, None])


def per_group_dequant(codes, scales, zeros, group: int = 64) -> np.ndarray:
    """fp64 restoration of per-group codes [L][Hkv][d] with scales [ceil(L/64)][Hkv]."""
    L = codes.shape[0]
    gidx = np.arange(L) // group
    return dequantize(codes, np.asarray(scales)[gidx][:, :, None],
                      np.asarray(zeros)[gidx][:, :, None])


def per_token_bbox_values(codes, scales, zeros) -> np.ndarray:
    """fp32 two-step restoration of per-token codes (bounding-box input)."""
    return dequant_f32_two_step(codes, np.asarray(scales)[:, :, None], np.asarray(zeros)[:, :, None])


def per_group_bbox_values(codes, scales, zeros, group: int = 64) -> np.ndarray:
    L = codes.shape[0]
    gidx = np.arange(L) // group
    return dequant_f32_two_step(codes, np.asarray(scales)[gidx][:, :, None],
                                np.asarray(zeros)[gidx][:, :, None])
