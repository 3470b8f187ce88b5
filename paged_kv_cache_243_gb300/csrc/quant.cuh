// The INT8 quantiser of the kv_append kernels and of the fused append in the
// attention kernel [HBM-layout page, section 二 per-token; Gemini page, 第一章
// per-64-token group]: s = (max - min) / 255, z = min,
// code = clamp(rint((x - z) / s), 0, 255) - 128, every step a correctly rounded
// fp32 operation, so codes are bit-identical to any IEEE implementation.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

// code = rint((x - z) / s) - 128 with the correctly rounded quotient (the
// quotient is in [0, 255], so the clamp of the definition never acts).
// rs = the correctly rounded 1/s (0 when 1/s would not be finite):
// for quotients in [0, 256), (x - z) * rs is within 255 * 2^-23 of (x - z) / s
// and the correctly rounded quotient within 2^-17, so rint of either agrees
// unless the product lies within 1e-3 of a half-integer; there, and when rs
// is 0, the quotient itself is computed (warp-uniform branch, rarely taken).
// Rounding to nearest even uses the standard magic-number method: adding
// 1.5 * 2^23 leaves rint(q) in the low mantissa bits for 0 <= q < 2^22.
__device__ __forceinline__ float quant_recip(float s) { return s >= 1e-30f ? __frcp_rn(s) : 0.f; }
constexpr float kRoundMagic = 12582912.f;   // 1.5 * 2^23

// Codes of N values as bytes (code + 128 = u in [0, 255], stored as the int8
// u - 128, i.e. u ^ 0x80), packed 4 per word: w[k] holds values 4k .. 4k+3.
// The quotient q lies in [0, 255 (1 + 2^-22)], so rint(q) needs no clamp.
template <int N>
__device__ __forceinline__ void quant_words(const float (&x)[N], float s, float z, float rs,
                                            uint32_t (&w)[N / 4]) {
  if (s == 0.f) {
#pragma unroll
    for (int k = 0; k < N / 4; ++k) w[k] = 0x80808080u;   // every code -128
    return;
  }
  float d[N], m[N];
  bool near = rs == 0.f;
#pragma unroll
  for (int e = 0; e < N; ++e) {
    d[e] = __fsub_rn(x[e], z);
    const float q = __fmul_rn(d[e], rs);
    m[e] = __fadd_rn(q, kRoundMagic);                        // rint(q) in the low bits
    const float diff = __fsub_rn(q, __fsub_rn(m[e], kRoundMagic));
    near |= fabsf(diff) > 0.499f;
  }
  if (__any_sync(__activemask(), near)) {
#pragma unroll
    for (int e = 0; e < N; ++e) m[e] = __fadd_rn(__fdiv_rn(d[e], s), kRoundMagic);
  }
#pragma unroll
  for (int k = 0; k < N / 4; ++k) {
    const uint32_t lo = __byte_perm(__float_as_uint(m[4 * k]), __float_as_uint(m[4 * k + 1]), 0x0040);
    const uint32_t hi = __byte_perm(__float_as_uint(m[4 * k + 2]), __float_as_uint(m[4 * k + 3]), 0x0040);
    w[k] = __byte_perm(lo, hi, 0x5410) ^ 0x80808080u;
  }
}

// 4-bit codes [per-token 4-bit reading of the KV-practice page, section 3.2]:
// s = (max - min) / 15, z = min, u = clamp(rint((x - z) / s), 0, 15), each
// step a correctly rounded fp32 operation, as quant_words: rint through the
// reciprocal rs unless a product lies within 1e-3 of a half-integer (then the
// quotient itself). N values (N even) -> N / 2 bytes, value 2i in the low
// nibble of byte i; w[k] holds bytes 4k .. 4k + 3.
template <int N>
__device__ __forceinline__ void quant_nibbles(const float (&x)[N], float s, float z, float rs,
                                              uint32_t (&w)[(N + 7) / 8]) {
#pragma unroll
  for (int k = 0; k < (N + 7) / 8; ++k) w[k] = 0u;
  if (s == 0.f) return;   // constant row: every code 0
  float d[N], m[N];
  bool near = rs == 0.f;
#pragma unroll
  for (int e = 0; e < N; ++e) {
    d[e] = __fsub_rn(x[e], z);
    const float q = __fmul_rn(d[e], rs);
    m[e] = __fadd_rn(q, kRoundMagic);
    const float diff = __fsub_rn(q, __fsub_rn(m[e], kRoundMagic));
    near |= fabsf(diff) > 0.499f;
  }
  if (__any_sync(__activemask(), near)) {
#pragma unroll
    for (int e = 0; e < N; ++e) m[e] = __fadd_rn(__fdiv_rn(d[e], s), kRoundMagic);
  }
#pragma unroll
  for (int e = 0; e < N; ++e) w[e / 8] |= (__float_as_uint(m[e]) & 0xFu) << (4 * (e % 8));
}

// Four consecutive source values (f16/bf16) widened to fp32; i is a multiple of 4.
__device__ __forceinline__ float4 load_src4(const void* p, int dtype, size_t i) {
  const uint2 w = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p) + i);
  if (dtype == PKV_BF16)
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
  return make_float4(__half2float(__ushort_as_half((unsigned short)(w.x & 0xffffu))),
                     __half2float(__ushort_as_half((unsigned short)(w.x >> 16))),
                     __half2float(__ushort_as_half((unsigned short)(w.y & 0xffffu))),
                     __half2float(__ushort_as_half((unsigned short)(w.y >> 16))));
}

}  // namespace pkv
