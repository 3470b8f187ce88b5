"""The fp16 bit patterns the 4-bit tensor-core consumer builds its operands from,
read from the kernel header and checked with numpy's IEEE half precision.

A 4-bit code masked into mantissa bits 0-3 of a 16-bit half is the subnormal
u * 2^-24, into bits 4-7 u * 2^-20. K codes enter q.K^T in that form, with the q
values of the first kind scaled by 16 (or, for very large q, the others by 1/16);
V codes enter P.V as (u - 8) * 2^-9 through one fp16 fma of the masked subnormal.
Every one of these values must be exact in fp16, or the 4-bit path would be biased.
"""
import os
import re

import numpy as np

HEADER = os.path.join(os.path.dirname(__file__), "..", "paged_kv_cache_243_gb300", "csrc",
                      "attention_kernel.cuh")


def _constants():
    with open(HEADER) as fh:
        txt = fh.read()
    out = {}
    for name, val in re.findall(r"constexpr uint32_t (k\w+) = (0x[0-9A-Fa-f]+)u;", txt):
        out[name] = int(val, 16)
    return out


def _h2(word):
    """The two fp16 halves of a 32-bit word (low, high) as float64."""
    lo = np.array([word & 0xFFFF], dtype=np.uint16).view(np.float16)[0]
    hi = np.array([word >> 16], dtype=np.uint16).view(np.float16)[0]
    return float(lo), float(hi)


def _pair(word):
    """The value of a word whose two fp16 halves are equal."""
    assert word & 0xFFFF == word >> 16, hex(word)
    return _h2(word)[0]


def test_constants_are_the_intended_fp16_pairs():
    c = _constants()
    assert c["kNibLo"] == 0x000F000F and c["kNibHi"] == 0x00F000F0
    assert _pair(c["kH2x16"]) == 16.0
    assert _pair(c["kH2x1o16"]) == 1.0 / 16.0
    assert _pair(c["kH2x2p15"]) == 2.0 ** 15
    assert _pair(c["kH2x2p11"]) == 2.0 ** 11
    assert _pair(c["kH2m2pm6"]) == -(2.0 ** -6)
    lo, hi = _h2(c["kH2m0"])
    assert lo == 0.0 and np.signbit(lo) and hi == 0.0 and np.signbit(hi)


def test_masked_nibbles_are_exact_subnormals():
    c = _constants()
    for u0 in range(16):
        for u1 in range(16):
            # a word whose low half holds nibbles (u0, u1) at bits 0-3, 4-7 and whose
            # high half holds them swapped, plus set bits the masks must drop
            w = u0 | (u1 << 4) | 0xFF00 | ((u1 | (u0 << 4) | 0xFF00) << 16)
            lo, hi = _h2(w & c["kNibLo"])
            assert (lo, hi) == (u0 * 2.0 ** -24, u1 * 2.0 ** -24)
            lo, hi = _h2(w & c["kNibHi"])
            assert (lo, hi) == (u1 * 2.0 ** -20, u0 * 2.0 ** -20)


def test_v_codes_enter_centred_and_scaled_exactly():
    c = _constants()
    mul_lo, mul_hi, add = _pair(c["kH2x2p15"]), _pair(c["kH2x2p11"]), _pair(c["kH2m2pm6"])
    for u in range(16):
        a = np.float16(u * 2.0 ** -24) * np.float64(mul_lo) + add   # exact: every term is
        b = np.float16(u * 2.0 ** -20) * np.float64(mul_hi) + add   # a short binary fraction
        want = (u - 8) * 2.0 ** -9
        assert a == want and b == want
        # and the result is representable in fp16 (the fma rounds nothing)
        assert float(np.float16(want)) == want


def test_k_products_share_one_factor():
    # q slots meeting the bits-0-3 codes carry 16 q, the others q: every product
    # is q u 2^-20, so one key-scale factor (2^20) takes them all back; with the
    # other scaling (q / 16 on the bits-4-7 slots) every product is q u 2^-24
    c = _constants()
    s16, s1o16 = _pair(c["kH2x16"]), _pair(c["kH2x1o16"])
    rng = np.random.default_rng(5)
    q = rng.standard_normal(64).astype(np.float16).astype(np.float64)
    for u in range(16):
        assert np.array_equal((q * s16) * (u * 2.0 ** -24), q * u * 2.0 ** -20)
        assert np.array_equal(q * (u * 2.0 ** -20), q * u * 2.0 ** -20)
        assert np.array_equal(q * (u * 2.0 ** -24), q * u * 2.0 ** -24)
        assert np.array_equal((q * s1o16) * (u * 2.0 ** -20), q * u * 2.0 ** -24)
    # 16 q stays finite in fp16 up to |q| = 4094, the switch-over bound
    assert np.isfinite(np.float16(4094.0) * np.float16(16.0))
    with np.errstate(over="ignore"):
        assert not np.isfinite(np.float16(4096.0) * np.float16(16.0))
