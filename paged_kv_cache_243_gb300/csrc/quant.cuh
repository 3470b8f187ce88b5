// The INT8 and 4-bit quantisers of the kv_append kernels and of the fused
// append in the attention kernel [HBM-layout page, section 二 per-token;
// Gemini page, 第一章 per-64-token group; 4-bit: KV-practice page, section
// 3.2]: s = (max - min) / 255 (4-bit: / 15), z = min,
// code = clamp(rint((x - z) / s), 0, 255) - 128, stored as the byte
// u = code + 128 (4-bit: u in [0, 15]), every step a correctly rounded fp32
// operation, so codes are bit-identical to any IEEE implementation.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

// code = rint((x - z) / s) - 128 with the correctly rounded quotient (the
// quotient is in [0, 255], so the clamp of the definition never acts).
// rs = the correctly rounded 1/s (0 when 1/s would not be finite). With q the
// exact quotient (at most 255): rs = (1/s)(1 + e1) and the product
// p = fl((x - z) rs) = q (1 + e1)(1 + e2), |e1|, |e2| <= 2^-24, so
// |p - q| <= 255 * 2^-23 (1 + 2^-24) < 3.1e-5, and the correctly rounded
// quotient q* is within 255 * 2^-24 < 1.6e-5 of q. rint(p) and rint(q*) can
// differ only if a half-integer lies between them, i.e. within 4.7e-5 of p:
// when p lies within 1e-4 of a half-integer (or rs is 0), the quotient itself
// is computed (warp-uniform branch, taken by about one warp in ten).
// Rounding to nearest even uses the standard magic-number method: adding
// 1.5 * 2^23 leaves rint(q) in the low mantissa bits for 0 <= q < 2^22, and
// p - rint(p) is computed exactly (both lie in one binade below 256).
__device__ __forceinline__ float quant_recip(float s) { return s >= 1e-30f ? __frcp_rn(s) : 0.f; }
constexpr float kRoundMagic = 12582912.f;   // 1.5 * 2^23
constexpr float kNearHalf = 0.4999f;         // |p - rint(p)| above this: within 1e-4 of a half-integer

// Shared step of both quantisers: for N values (N even), m[e] = rint(q_e) +
// 1.5 * 2^23 with q_e = fl(fl(x_e - z) / s), the integer in m's low mantissa
// bits. Two values per packed fp32x2 instruction. ptxas may contract the
// packed multiply and the magic add into one fma (it never fuses the scalar
// __fmul_rn / __fadd_rn); m then holds the rounding of the exact product
// (x - z) rs, within 255 * 2^-24 of q, and the near-half test covers that
// case by the same bound.
template <int N>
__device__ __forceinline__ void quant_rint(const float (&x)[N], float s, float z, float rs, float (&m)[N]) {
  const uint64_t z2 = pack2f(z, z), rs2 = pack2f(rs, rs), mg2 = pack2f(kRoundMagic, kRoundMagic);
  uint64_t d2[N / 2];
  bool near = rs == 0.f;
#pragma unroll
  for (int e = 0; e < N; e += 2) {
    d2[e / 2] = fsub2(pack2f(x[e], x[e + 1]), z2);
    const uint64_t q2 = fmul2(d2[e / 2], rs2);
    const uint64_t m2 = fadd2(q2, mg2);                 // rint(q) in the low bits
    const uint64_t df = fsub2(q2, fsub2(m2, mg2));      // q - rint(q), exact
    float f0, f1;
    unpack2f(df, f0, f1);
    near |= fabsf(f0) > kNearHalf || fabsf(f1) > kNearHalf;
    unpack2f(m2, m[e], m[e + 1]);
  }
  if (__any_sync(__activemask(), near)) {
#pragma unroll
    for (int e = 0; e < N; e += 2) {
      float d0, d1;
      unpack2f(d2[e / 2], d0, d1);
      m[e] = __fadd_rn(__fdiv_rn(d0, s), kRoundMagic);
      m[e + 1] = __fadd_rn(__fdiv_rn(d1, s), kRoundMagic);
    }
  }
}

// Codes of N values as the stored bytes u = code + 128 in [0, 255], packed 4
// per word: w[k] holds values 4k .. 4k+3. The quotient q lies in [0, 255 (1 +
// 2^-22)], so rint(q) needs no clamp, and its low mantissa byte is u.
template <int N>
__device__ __forceinline__ void pack_words(const float (&m)[N], uint32_t (&w)[N / 4]) {
#pragma unroll
  for (int k = 0; k < N / 4; ++k) {
    const uint32_t lo = __byte_perm(__float_as_uint(m[4 * k]), __float_as_uint(m[4 * k + 1]), 0x0040);
    const uint32_t hi = __byte_perm(__float_as_uint(m[4 * k + 2]), __float_as_uint(m[4 * k + 3]), 0x0040);
    w[k] = __byte_perm(lo, hi, 0x5410);
  }
}

template <int N>
__device__ __forceinline__ void quant_words(const float (&x)[N], float s, float z, float rs,
                                            uint32_t (&w)[N / 4]) {
  if (s == 0.f) {
#pragma unroll
    for (int k = 0; k < N / 4; ++k) w[k] = 0u;   // every code -128 (stored byte 0)
    return;
  }
  float m[N];
  quant_rint<N>(x, s, z, rs, m);
  pack_words<N>(m, w);
}

// 4-bit codes [per-token 4-bit reading of the KV-practice page, section 3.2]:
// s = (max - min) / 15, z = min, u = clamp(rint((x - z) / s), 0, 15), each
// step a correctly rounded fp32 operation, as quant_words: rint through the
// reciprocal rs unless a product lies within 1e-4 of a half-integer (then the
// quotient itself; the bound of quant_words holds a fortiori for quotients of
// at most 15). N values (N even) -> N / 2 bytes, value 2i in the low
// nibble of byte i; w[k] holds bytes 4k .. 4k + 3.
// Packs quant_rint's results as 4-bit codes, value 2i in the low nibble of byte i.
// The codes sit in the low bytes of m (at most 15); for whole words byte
// permutes gather the even and the odd values' bytes of eight values, and one
// shift and or merges them.
template <int N>
__device__ __forceinline__ void pack_nibbles(const float (&m)[N], uint32_t (&w)[(N + 7) / 8]) {
  if constexpr (N % 8 != 0) {   // a partial word: value by value
#pragma unroll
    for (int k = 0; k < (N + 7) / 8; ++k) w[k] = 0u;
#pragma unroll
    for (int e = 0; e < N; ++e) w[e / 8] |= (__float_as_uint(m[e]) & 0xFu) << (4 * (e % 8));
    return;
  }
#pragma unroll
  for (int k = 0; k < N / 8; ++k) {
    const float* v = m + 8 * k;
    const uint32_t e01 = __byte_perm(__float_as_uint(v[0]), __float_as_uint(v[2]), 0x0040);
    const uint32_t e23 = __byte_perm(__float_as_uint(v[4]), __float_as_uint(v[6]), 0x0040);
    const uint32_t o01 = __byte_perm(__float_as_uint(v[1]), __float_as_uint(v[3]), 0x0040);
    const uint32_t o23 = __byte_perm(__float_as_uint(v[5]), __float_as_uint(v[7]), 0x0040);
    const uint32_t ev = __byte_perm(e01, e23, 0x5410);   // bytes: values 0, 2, 4, 6
    const uint32_t od = __byte_perm(o01, o23, 0x5410);   // bytes: values 1, 3, 5, 7
    w[k] = ev | (od << 4);
  }
}

template <int N>
__device__ __forceinline__ void quant_nibbles(const float (&x)[N], float s, float z, float rs,
                                              uint32_t (&w)[(N + 7) / 8]) {
  if (s == 0.f) {   // constant row: every code 0
#pragma unroll
    for (int k = 0; k < (N + 7) / 8; ++k) w[k] = 0u;
    return;
  }
  float m[N];
  quant_rint<N>(x, s, z, rs, m);
  pack_nibbles<N>(m, w);
}

// Four 16-bit source values (f16/bf16, as loaded) widened to fp32; the
// compile-time form for kernels specialised on the source dtype.
template <bool BF16>
__device__ __forceinline__ float4 widen4_t(uint2 w) {
  if constexpr (BF16)
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
  return make_float4(__half2float(__ushort_as_half((unsigned short)(w.x & 0xffffu))),
                     __half2float(__ushort_as_half((unsigned short)(w.x >> 16))),
                     __half2float(__ushort_as_half((unsigned short)(w.y & 0xffffu))),
                     __half2float(__ushort_as_half((unsigned short)(w.y >> 16))));
}

// Four 16-bit source values (f16/bf16, as loaded) widened to fp32.
__device__ __forceinline__ float4 widen4(uint2 w, int dtype) {
  if (dtype == PKV_BF16)
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
  return make_float4(__half2float(__ushort_as_half((unsigned short)(w.x & 0xffffu))),
                     __half2float(__ushort_as_half((unsigned short)(w.x >> 16))),
                     __half2float(__ushort_as_half((unsigned short)(w.y & 0xffffu))),
                     __half2float(__ushort_as_half((unsigned short)(w.y >> 16))));
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
