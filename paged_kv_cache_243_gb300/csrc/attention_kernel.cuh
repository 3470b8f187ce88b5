// Paged decode attention: one persistent launch that splits the whole batch's
// KV chunks evenly over its thread blocks and streams each chunk into shared
// memory with 1-D bulk copies (TMA engine), then a small second launch that
// merges the partial softmax states.
//
// What it computes [KV-practice page, section 2.1]: for query head h of
// sequence b, out = softmax(sm_scale * q . K^T) V over the sequence's cached
// tokens (dense) or over the tokens of its selected pages [TinyServe page,
// section 3.1 phase 3], with K/V of kv head h / G (GQA) read through the block
// table [HBM-layout page, section 二 layout C] and INT8 codes restored in
// registers [HBM-layout page, section 二; Gemini page, 第一章].
//
// Work decomposition. A "unit" is what shares one key/value stream: (sequence,
// kv head) in dense mode, serving all G query heads of the group from one read
// of K/V [Gemini page, section 3.1], or (sequence, query head) in sparse mode.
// A unit's tokens are cut into 16-token chunks; chunks of all units are laid
// end to end and block c of N takes chunks [c W / N, (c + 1) W / N). A block's
// range thus covers whole or partial units, and every block gets the same
// number of chunks whatever the sequence lengths are.
//
// Inside a block: warp 4 is the producer. Its lanes resolve 32 chunks at a time
// (unit, block-table lookup, addresses) and up to S of them issue
// cp.async.bulk copies of the chunks' K rows, V rows and INT8 scales into a
// ring of S shared-memory stages, each guarded by a "full" and an "empty"
// mbarrier. Warps 0-3 consume chunks round robin; each keeps its own
// online-softmax state (running max m, sum l, accumulator) per query head, in
// the log2 domain, and writes it to a workspace record whenever its chunk
// stream leaves a unit (an empty record for units of the block's range it did
// not see). The block's last unit is the exception: after the stream the four
// warps' states meet in shared memory and the block writes one merged record.
//
// Self-fed tensor-core blocks (SELF) have no producer warp: consumer warp w
// reads the chunks w, w + 4, ... from its own stages (S is a multiple of 4),
// so it resolves their lookups and issues their copies itself. Three of these
// 128-thread blocks per SM leave room for a combine block beside them; the
// host uses them for short chains of attention calls (see its plan).
//
// Merge [TinyServe page, section 3.1 phase 4]: attn_combine_kernel, the next
// launch on the stream, folds for every unit the records of all blocks whose
// ranges overlap it:
//   M = max m_s,  out = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s.
//
// Two consumer variants: CUDA cores (lane layouts below) and, for query-head
// groups, mma.sync tensor-core tiles (see the tensor-core section).
// CUDA-core lane layouts. Scores: lane = 8 r + j handles token 4 it + r of the
// chunk and a D/8-wide slice of channels; the 8 lanes of a token reduce their
// partial dot products with a butterfly that also scatters the G query heads
// over the lanes (lane j ends with the full score of head j / (8 / G)).
// Values: lane owns channels [lane * D / 32, (lane + 1) * D / 32) of every
// token and all G heads. Probabilities move between the two layouts through
// shared memory.
#pragma once

#include <type_traits>

#include "pkv_common.cuh"
#include "quant.cuh"

namespace pkv {

constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
// Threads of a block. The self-fed tensor-core variant has no producer warp
// (its consumer warps copy their own chunks), so three of its blocks, three
// warps per SM sub-partition, leave room for a block of the combine beside
// them.
__host__ __device__ constexpr int attn_threads(bool self_fed) {
  return self_fed ? kConsumerWarps * 32 : kAttnThreads;
}
// Small shared scratch: [8, 8 + warps) the unit prefix scan's warp totals.
constexpr int kMiscInts = 32;
constexpr int kQStageBytes = 2048;   // shared-memory copy of q for a block's first units (small: it must
                                     // not cost a resident block per SM)
constexpr int kMiscAbort = 24;   // misc slot: some consumer warp timed out
constexpr int kSkipSelected = -2;   // producer: a chunk past its unit's page list

struct AttnParams {
  // K and V pools as 2-D tensors [num_pages * Hkv * page_size rows][128 bytes]
  // with 128-byte swizzle, for the tensor-core INT8 variant at head_dim 128
  // (which copies each chunk as two 16-row tiles); unused by the others
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  const uint8_t* k_pages;
  const uint8_t* v_pages;
  const float* kv_sz;
  const void* q;
  void* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* sel_pages;  // NULL: dense
  const int32_t* sel_count;
  // partial records, slot ((block + unit) * 4 + warp); for the block's last
  // unit only slot 0, holding the merge of its four warps
  float* ws_wrec;
  int32_t* ws_prefix; // [num_units + 1] chunk prefix, written by block 0 for the combine
  int32_t* dev_status;
  int num_pages, page_size, num_kv_heads, num_q_heads, group;
  int batch, max_pages, sel_stride;
  int units_per_b, num_units;
  int num_ctas, stages;
  int q_dtype, out_dtype;
  float q_scale;  // sm_scale * log2(e): scores live in the log2 domain
  // < 0: wait for the preceding kernel before reading anything. >= 0: that
  // kernel writes, of this launch's inputs, only K/V rows (and scales) at
  // positions >= seq_len - fresh_rows (for per-group INT8: from the start of
  // the 64-token group holding that position), so everything else is read
  // while it still runs; see the early-start notes in the kernel.
  int fresh_rows;
  int comb_groups;  // record groups of the combine kernel (1, 2, 4 or 8)
  // 1: a unit is (sequence, query head) with its own page list (sparse, per
  // query head); 0: (sequence, kv head) serving the G query heads of its group
  // (dense, or sparse with one page list shared by the group).
  int unit_is_q;
  // Fused append (dense calls; NULL: none): k_new / v_new [batch][Hkv][D] of
  // src_dtype hold each sequence's token at position seq_len - 1, which the
  // block streaming that position writes into its page (quantised per token
  // for INT8 caches) before it copies the chunk.
  const void* k_new;
  const void* v_new;
  int src_dtype;
};

struct ChunkInfo {
  const uint8_t* k;
  const uint8_t* v;
  const float* sz;
  int u;
  int nvalid;
  int valid;
  int fresh;  // overlaps rows the preceding kernel may still be writing
  int last;   // the unit's last chunk (holds position seq_len - 1), dense only
  int row;    // pool row of the chunk's first token (tensor-copy coordinate)
};

template <int D, int KV>
struct AttnGeom {
  static constexpr int ESZ = (KV == KV_I8T || KV == KV_I8G || KV == KV_U4T) ? 1 : 2;
  static constexpr bool PTOK = KV == KV_I8T || KV == KV_U4T;   // per-token scales
  static constexpr int ROW = KV == KV_U4T ? D / 2 : D * ESZ;  // bytes of one token row
  static constexpr int KB = kChunk * ROW;          // bytes of one chunk of K (or V)
  static constexpr int SZB = PTOK ? kChunk * 16 : (KV == KV_I8G ? 16 : 0);
  static constexpr int STAGE = ((2 * KB + SZB) + 127) / 128 * 128;
  static constexpr int QD = D / 8;                 // channels per lane in the score layout
  static constexpr int PD = D / 32;                // channels per lane in the value layout
  // The tensor-core variant of INT8 caches at head_dim 128 stages K and V as
  // tiles of 16 rows x 128 bytes with the 128-byte swizzle (16-byte block j of
  // row r lands at block j ^ (r % 8)), which makes its fragment loads free of
  // bank conflicts; its ring stages hold the two tiles (1024-byte aligned) and
  // the scales sit in a separate array.
  static constexpr bool SWZ_OK = ESZ == 1 && D == 128 && KV != KV_U4T;
  static constexpr int TILE_STAGE = 2 * KB;
};

// Bytes of shared memory per ring stage, and extra alignment slack, of a
// kernel variant (swz: the swizzled tensor-core INT8 variant).
__host__ __device__ constexpr int stage_bytes_of(int kb, int szb, bool swz) {
  return swz ? 2 * kb + szb : ((2 * kb + szb) + 127) / 128 * 128;
}
constexpr int kSwizzleAlign = 1024;

template <int GE>
struct AttnSmem {
  // floats per warp: p[16][GE] and alpha[GE] (CUDA-core path), or p[8][16] (tensor-core path)
  static constexpr int PBUF = kChunk * 8 + 8;
};

// Partial-state record of one (block or warp, unit): m[GE], l[GE] (padded to a
// multiple of 4 floats), then acc[GE][D]. All in the log2 domain.
__host__ __device__ constexpr int rec_hdr(int ge) { return (2 * ge + 3) / 4 * 4; }
__host__ __device__ constexpr int rec_floats(int ge, int d) { return rec_hdr(ge) + ge * d; }

__host__ __device__ inline size_t attn_smem_bytes(int stage_bytes, int stages, int ge, int units,
                                                  int batch) {
  size_t s = (size_t)stage_bytes * stages;
  s += (size_t)stages * 16;                       // hdr int4 per stage
  s += (size_t)stages * 16;                       // full + empty mbarriers
  s += (size_t)kConsumerWarps * (kChunk * 8 + 8) * 4;
  s += 32 * sizeof(ChunkInfo);
  s += kMiscInts * 4;                              // misc
  s += (size_t)(units + 1) * 4 + (size_t)batch * 4;
  s = (s + 15) / 16 * 16 + kQStageBytes;           // q rows of the block's first units
  return s;
}

// Channel index of element e of lane-slot j in the score layout.
template <int D, int KV>
__device__ __forceinline__ int qk_dim(int j, int e) {
  if (AttnGeom<D, KV>::ESZ == 2 && D == 128) return e < 8 ? 8 * j + e : 64 + 8 * j + (e - 8);
  return AttnGeom<D, KV>::QD * j + e;
}

// Load this lane's D/8 channels of token row `row` (score layout) as packed
// fp32 pairs (INT8: the stored byte u = code + 128; 4-bit: u = the code).
template <int D, int KV>
__device__ __forceinline__ void load_k_slice(const uint8_t* row, int j, uint64_t (&k2)[D / 16]) {
  if constexpr (KV == KV_F16 || KV == KV_BF16) {
    if constexpr (D == 128) {
      const uint4 a = *reinterpret_cast<const uint4*>(row + j * 16);
      const uint4 b = *reinterpret_cast<const uint4*>(row + (j + 8) * 16);
      k2[0] = widen2<KV>(a.x); k2[1] = widen2<KV>(a.y); k2[2] = widen2<KV>(a.z); k2[3] = widen2<KV>(a.w);
      k2[4] = widen2<KV>(b.x); k2[5] = widen2<KV>(b.y); k2[6] = widen2<KV>(b.z); k2[7] = widen2<KV>(b.w);
    } else {
      const uint4 a = *reinterpret_cast<const uint4*>(row + j * 16);
      k2[0] = widen2<KV>(a.x); k2[1] = widen2<KV>(a.y); k2[2] = widen2<KV>(a.z); k2[3] = widen2<KV>(a.w);
    }
  } else if constexpr (KV == KV_U4T) {
    // D / 8 channels = D / 16 bytes per lane; pair i = the two nibbles of byte i
    if constexpr (D == 128) {
      const uint2 a = *reinterpret_cast<const uint2*>(row + j * 8);
      uint32_t lo0, hi0, lo1, hi1;
      split_nibbles(a.x, lo0, hi0);
      split_nibbles(a.y, lo1, hi1);
#pragma unroll
      for (int i = 0; i < 4; ++i) k2[i] = u4pair(lo0, hi0, i);
#pragma unroll
      for (int i = 0; i < 4; ++i) k2[4 + i] = u4pair(lo1, hi1, i);
    } else {
      const uint32_t a = *reinterpret_cast<const uint32_t*>(row + j * 4);
      uint32_t lo, hi;
      split_nibbles(a, lo, hi);
#pragma unroll
      for (int i = 0; i < 4; ++i) k2[i] = u4pair(lo, hi, i);
    }
  } else {
    if constexpr (D == 128) {
      const uint4 a = *reinterpret_cast<const uint4*>(row + j * 16);
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) k2[i] = u8pair(w[i >> 1], (i & 1) * 2);
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(row + j * 8);
      const uint32_t w[2] = {a.x, a.y};
#pragma unroll
      for (int i = 0; i < 4; ++i) k2[i] = u8pair(w[i >> 1], (i & 1) * 2);
    }
  }
}

// Load this lane's D/32 channels of token row `row` (value layout) as packed pairs.
template <int D, int KV>
__device__ __forceinline__ void load_v_slice(const uint8_t* row, int lane, uint64_t (&v2)[D / 64]) {
  if constexpr (KV == KV_F16 || KV == KV_BF16) {
    if constexpr (D == 128) {
      const uint2 a = *reinterpret_cast<const uint2*>(row + lane * 8);
      v2[0] = widen2<KV>(a.x);
      v2[1] = widen2<KV>(a.y);
    } else {
      v2[0] = widen2<KV>(*reinterpret_cast<const uint32_t*>(row + lane * 4));
    }
  } else if constexpr (KV == KV_U4T) {
    // D / 32 channels = D / 64 bytes per lane
    uint32_t lo, hi;
    if constexpr (D == 128) {
      split_nibbles((uint32_t)*reinterpret_cast<const uint16_t*>(row + lane * 2), lo, hi);
      v2[0] = u4pair(lo, hi, 0);
      v2[1] = u4pair(lo, hi, 1);
    } else {
      split_nibbles((uint32_t)row[lane], lo, hi);
      v2[0] = u4pair(lo, hi, 0);
    }
  } else {
    if constexpr (D == 128) {
      const uint32_t a = *reinterpret_cast<const uint32_t*>(row + lane * 4);
      v2[0] = u8pair(a, 0);
      v2[1] = u8pair(a, 2);
    } else {
      const uint32_t a = (uint32_t)(*reinterpret_cast<const uint16_t*>(row + lane * 2));
      v2[0] = u8pair(a, 0);
    }
  }
}

// Sum partial values over the 8 lanes of a token (lane bits 0-2) while
// scattering heads: lane j returns the total of head j / (8 / GE).
template <int GE>
__device__ __forceinline__ float reduce_scatter8(const float (&v)[GE], int j) {
  if constexpr (GE == 1) {
    float x = v[0];
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
  } else if constexpr (GE == 2) {
    const bool hi = (j >> 2) & 1;
    float keep = hi ? v[1] : v[0];
    float send = hi ? v[0] : v[1];
    keep += __shfl_xor_sync(0xffffffffu, send, 4);
    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
    keep += __shfl_xor_sync(0xffffffffu, keep, 1);
    return keep;
  } else if constexpr (GE == 4) {
    const bool b2 = (j >> 2) & 1, b1 = (j >> 1) & 1;
    float k0 = b2 ? v[2] : v[0], s0 = b2 ? v[0] : v[2];
    float k1 = b2 ? v[3] : v[1], s1 = b2 ? v[1] : v[3];
    k0 += __shfl_xor_sync(0xffffffffu, s0, 4);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 4);
    float keep = b1 ? k1 : k0, send = b1 ? k0 : k1;
    keep += __shfl_xor_sync(0xffffffffu, send, 2);
    keep += __shfl_xor_sync(0xffffffffu, keep, 1);
    return keep;
  } else {
    const bool b2 = (j >> 2) & 1, b1 = (j >> 1) & 1, b0 = j & 1;
    float k4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float keep = b2 ? v[4 + i] : v[i], send = b2 ? v[i] : v[4 + i];
      k4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float k2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float keep = b1 ? k4[2 + i] : k4[i], send = b1 ? k4[i] : k4[2 + i];
      k2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    float keep = b0 ? k2[1] : k2[0], send = b0 ? k2[0] : k2[1];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
  }
}

// ------------------------------------------------------------ tensor-core path
// Warp-level mma.sync m16n8k16 with fp32 accumulation, for query-head groups
// (G >= 2): q.K^T as [16 tokens] x [8 heads] and P.V as [16 channels] x [8 heads]
// per 16-token chunk. INT8 codes enter as exact fp16 integers.
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Two stored INT8 bytes u of a word (selected by sel: 0x4140 -> bytes 0, 1;
// 0x4342 -> bytes 2, 3) as the centred codes (u0 - 128, u1 - 128) in fp16:
// 0x64xx is the fp16 value 1024 + xx, and subtracting 1152 is exact.
__device__ __forceinline__ uint32_t u8x2_to_h2c(uint32_t w, uint32_t sel) {
  const uint32_t h = __byte_perm(w, 0x64646464u, sel);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
  return r;
}

// Two stored INT8 bytes u of a word (sel as above) as the fp16 pair 1024 + u.
__device__ __forceinline__ uint32_t u8x2_to_h2(uint32_t w, uint32_t sel) {
  return __byte_perm(w, 0x64646464u, sel);
}

// 4-bit codes as fp16 subnormals. A code u masked into mantissa bits 0-3 of a
// 16-bit half is the fp16 value u 2^-24; in bits 4-7 it is u 2^-20. Both are
// exact, and the tensor cores and the half-precision fma take subnormal
// operands as they are, so one mask per pair of codes makes an MMA operand.
constexpr uint32_t kNibLo = 0x000F000Fu;   // nibbles at bit offsets 0 and 16
constexpr uint32_t kNibHi = 0x00F000F0u;   // nibbles at bit offsets 4 and 20
constexpr uint32_t kH2x16 = 0x4C004C00u;   // fp16 pair (16, 16)
constexpr uint32_t kH2x1o16 = 0x2C002C00u; // 1/16
constexpr uint32_t kH2m0 = 0x80008000u;    // -0: an fma addend that keeps a -0
constexpr uint32_t kH2x2p15 = 0x78007800u; // 2^15
constexpr uint32_t kH2x2p11 = 0x68006800u; // 2^11
constexpr uint32_t kH2m2pm6 = 0xA400A400u; // -2^-6 = -8 * 2^-9

// fp16x2 a * b + c, one rounding to nearest even (subnormals kept)
__device__ __forceinline__ uint32_t hfma2_rn(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// fp32 pair -> (hi, lo) 16-bit pairs with hi + lo = x to ~2^-22 (fp16) / 2^-16 (bf16).
template <bool BF16>
__device__ __forceinline__ void split_hi_lo(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  if constexpr (BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
  } else {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
  }
}

__device__ __forceinline__ float h2lo_f(uint32_t w, bool bf) {
  return bf ? __uint_as_float(w << 16) : __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
__device__ __forceinline__ float h2hi_f(uint32_t w, bool bf) {
  return bf ? __uint_as_float(w & 0xffff0000u) : __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

__device__ __forceinline__ int find_unit(const int* prefix, int num_units, int x) {
  int lo = 0, hi = num_units - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// 32-bit division when the operands fit (the common case), 64-bit otherwise.
__device__ __forceinline__ long long div_fast(long long a, long long b) {
  if (((unsigned long long)a | (unsigned long long)b) < (1ull << 32))
    return (long long)((unsigned)a / (unsigned)b);
  return a / b;
}
__device__ __forceinline__ int cta_lo(long long c, long long W, long long N) { return (int)div_fast(c * W, N); }
// Largest block c whose range starts at or before chunk x.
__device__ __forceinline__ int cta_of(long long x, long long W, long long N) {
  return (int)div_fast((x + 1) * N - 1, W);
}

// Fused append of one token row (K and V of one kv head) at row r of the
// chunk whose K, V (and per-token scale) rows start at ck, cv (csz), by the 32
// lanes of a warp: a copy for fp16/bf16 caches (source dtype = cache dtype),
// the per-token quantiser of kv_append for INT8 [HBM-layout page, section 二]
// and 4-bit caches.
template <int D, int KV>
__device__ __forceinline__ void append_token_row(const AttnParams& p, int u, int r, uint8_t* ck, uint8_t* cv,
                                                 float* csz, int lane) {
  const int b = u / p.units_per_b, g = u - b * p.units_per_b;
  const size_t src = ((size_t)b * p.num_kv_heads + g) * D;
  constexpr int PL = D / 32;   // values per lane
  if constexpr (KV == KV_I8T || KV == KV_U4T) {
    constexpr bool U4 = KV == KV_U4T;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const void* sp = kv ? p.v_new : p.k_new;
      float x[4];
      if constexpr (PL == 4) {
        const float4 f = load_src4(sp, p.src_dtype, src + lane * 4);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
      } else {
        const uint32_t w = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(sp) + src)[lane];
        const bool bf = p.src_dtype == PKV_BF16;
        x[0] = bf ? __uint_as_float(w << 16) : __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
        x[1] = bf ? __uint_as_float(w & 0xffff0000u) : __half2float(__ushort_as_half((unsigned short)(w >> 16)));
        x[2] = x[0];
        x[3] = x[1];
      }
      float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      }
      const float s = __fdiv_rn(__fsub_rn(mx, mn), U4 ? 15.f : 255.f);
      const float z = mn;
      uint32_t w[1];
      if constexpr (U4) {
        // 4 values (D = 64: the lane's 2 values twice) -> 2 bytes of nibbles
        quant_nibbles<4>(x, s, z, quant_recip(s), w);
        uint8_t* dst = (kv ? cv : ck) + (size_t)r * (D / 2) + lane * (PL / 2);
        if constexpr (PL == 4)
          *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w[0];
        else
          *dst = (uint8_t)w[0];
      } else {
        quant_words<4>(x, s, z, quant_recip(s), w);
        uint8_t* dst = (kv ? cv : ck) + (size_t)r * D + lane * PL;
        if constexpr (PL == 4)
          *reinterpret_cast<uint32_t*>(dst) = w[0];
        else
          *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w[0];
      }
      if (lane == 0) {
        csz[r * 4 + kv * 2 + 0] = s;
        csz[r * 4 + kv * 2 + 1] = z;
      }
    }
  } else {
    // fp16 / bf16: D * 2 bytes per row, 8 (D = 128) or 4 (D = 64) bytes per lane
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(p.k_new) + src;
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(p.v_new) + src;
    if constexpr (PL == 4) {
      const uint2 a = reinterpret_cast<const uint2*>(ks)[lane];
      const uint2 c = reinterpret_cast<const uint2*>(vs)[lane];
      reinterpret_cast<uint2*>(ck + (size_t)r * D * 2)[lane] = a;
      reinterpret_cast<uint2*>(cv + (size_t)r * D * 2)[lane] = c;
    } else {
      const uint32_t a = reinterpret_cast<const uint32_t*>(ks)[lane];
      const uint32_t c = reinterpret_cast<const uint32_t*>(vs)[lane];
      reinterpret_cast<uint32_t*>(ck + (size_t)r * D * 2)[lane] = a;
      reinterpret_cast<uint32_t*>(cv + (size_t)r * D * 2)[lane] = c;
    }
  }
}

// The tensor-core variant is held to 3 resident blocks per SM (<= 136 registers)
// so that 12 consumer warps hide its per-chunk latency; the self-fed one
// (SELF) to 128 registers.
template <int D, int GE, int KV, bool MMA, bool SELF = false>
__global__ void __launch_bounds__(attn_threads(SELF), SELF ? 4 : (MMA ? 3 : 1))
    paged_attention_kernel(const __grid_constant__ AttnParams p) {
  static_assert(!SELF || MMA, "only the tensor-core consumers copy their own chunks");
  using Geo = AttnGeom<D, KV>;
  constexpr int QD = Geo::QD, PD = Geo::PD, KB = Geo::KB, SZB = Geo::SZB;
  // swizzled K/V tiles (tensor copies), scales in their own array
  constexpr bool SWZ = MMA && Geo::SWZ_OK;
  constexpr int STAGE = SWZ ? Geo::TILE_STAGE : Geo::STAGE;   // ring stride
  constexpr int PBUF = AttnSmem<GE>::PBUF;
  constexpr int DUP = 8 / GE;  // lanes (per token) that hold the same head after the scatter
  constexpr int NW = kConsumerWarps;
  constexpr int NT = attn_threads(SELF);

  extern __shared__ __align__(128) uint8_t smem[];
  const int S = p.stages;
  // the swizzle pattern follows shared-memory address bits 7-9, so swizzled
  // tiles start on a 1024-byte boundary (the host adds that much slack)
  uint8_t* ring = SWZ ? smem + ((kSwizzleAlign - (smem_u32(smem) & (kSwizzleAlign - 1))) & (kSwizzleAlign - 1))
                      : smem;
  uint8_t* szring = ring + (size_t)S * STAGE;               // swizzled variant: S x SZB scale bytes
  int4* hdr = reinterpret_cast<int4*>(szring + (SWZ ? (size_t)S * SZB : 0));
  uint64_t* full = reinterpret_cast<uint64_t*>(hdr + S);
  uint64_t* empty = full + S;
  float* pbuf_all = reinterpret_cast<float*>(empty + S);
  ChunkInfo* info = reinterpret_cast<ChunkInfo*>(pbuf_all + NW * PBUF);
  int* misc = reinterpret_cast<int*>(info + 32);
  int* prefix = misc + kMiscInts;
  int* lens = prefix + p.num_units + 1;
  uint8_t* qstage = smem + ((reinterpret_cast<uintptr_t>(lens + p.batch) - reinterpret_cast<uintptr_t>(smem) + 15) & ~uintptr_t(15));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int U = p.num_units;
  // the host never launches these; refuse rather than race (the ring must also
  // hold the four warps' states of the block's last unit after the stream)
  if (S <= 0 || S % NW != 0 || S > 32 || (size_t)S * STAGE < (size_t)NW * rec_floats(GE, D) * 4) {
    if (tid == 0) flag_status(p.dev_status, PKV_DEV_BAD_CONFIG);
    return;
  }
  const int ps = p.page_size;
  const bool sparse = p.sel_pages != nullptr;

  // Early start (fresh_rows >= 0). The launch may begin while the work
  // enqueued just before it (a kernel, or both kernels of the preceding
  // attention call) still runs. Reads of the lengths, tables, q and of all
  // K/V rows that work does not write go ahead at once, and so does the fused
  // append's write of the new rows, which that work leaves alone by the same
  // promise; griddepcontrol.wait comes before the producer copies a chunk
  // holding fresh rows, before any other global write (the preceding work
  // may still read the output or the workspace), and in every block before
  // it exits, so this grid never completes before the preceding one has.
  // The producer warp lets dependents start only after that wait. The
  // self-fed variant lets them start at once: its dependent is this call's
  // combine, which reads only the call's inputs before its own wait for this
  // grid, and whose blocks then wait beside this grid's.
  const bool early = p.fresh_rows >= 0;
  if (!early) {
    pdl_wait();
    pdl_launch_dependents();
  } else if constexpr (SELF) {
    pdl_launch_dependents();
  }
  // ---- sequence lengths (clamped to the block table) and unit chunk counts
  for (int b = tid; b < p.batch; b += NT) {
    int L = p.seq_lens[b];
    int cap = p.max_pages * ps;
    if (L < 0 || L > cap) {
      flag_status(p.dev_status, PKV_DEV_BAD_POSITION);
      L = L < 0 ? 0 : cap;
    }
    lens[b] = L;
  }
  if (tid < S) {
    mbar_init(smem_u32(&full[tid]), 1);
    mbar_init(smem_u32(&empty[tid]), 1);
  }
  if (tid == 0) misc[kMiscAbort] = 0;
  fence_mbar_init();
  __syncthreads();

  const int per = (U + NT - 1) / NT;
  const int ua0 = min(U, tid * per), ua1 = min(U, ua0 + per);
  int my_sum = 0;
  for (int u = ua0; u < ua1; ++u) {
    const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
    const int L = lens[b];
    int n;
    if (!sparse) {
      n = (L + kChunk - 1) / kChunk;
    } else if (early) {
      // the page lists may still be being written: every unit of sequence b
      // gets min(list stride, pages of b) pages' chunks, a bound on any
      // valid list (distinct pages of the sequence); entries past the
      // unit's count are skipped once the lists are read
      const int P = (L + ps - 1) / ps;
      n = min(p.sel_stride, P) * (ps / kChunk);
    } else {
      int cnt = p.sel_count[b * p.units_per_b + hu];
      cnt = cnt < 0 ? 0 : (cnt > p.sel_stride ? p.sel_stride : cnt);
      // every selected page counts as full: a partial last page only adds
      // chunks past the sequence end, which are skipped, and the count needs
      // no dependent load of the page list
      n = cnt * (ps / kChunk);
    }
    prefix[u] = n;
    my_sum += n;
  }
  int incl = my_sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) misc[8 + warp] = incl;
  __syncthreads();
  int wpre = 0;
  for (int w = 0; w < warp; ++w) wpre += misc[8 + w];
  {
    int run = wpre + incl - my_sum;
    for (int u = ua0; u < ua1; ++u) {
      int n = prefix[u];
      prefix[u] = run;
      run += n;
    }
    if (tid == NT - 1) prefix[U] = wpre + incl;
  }
  __syncthreads();

  const long long W = prefix[U];
  const long long N = p.num_ctas;
  const int c = blockIdx.x;
  const int lo = W > 0 ? cta_lo(c, W, N) : 0;
  const int hi = W > 0 ? cta_lo(c + 1, W, N) : 0;
  const int ua = lo < hi ? find_unit(prefix, U, lo) : 0;
  const int ub = lo < hi ? find_unit(prefix, U, hi - 1) : -1;

  // the unit prefix for the combine: block 0 writes it here when it has no
  // chunks, else in its merge phase (after its wait in early mode)
  if (blockIdx.x == 0 && lo >= hi) {
    if (early) pdl_wait();
    for (int u = tid; u <= U; u += NT) p.ws_prefix[u] = prefix[u];
  }
  // ---- units without any chunk produce zeros (block u mod N writes them)
  if (warp < NW) {
    for (int u = c; u < U; u += (int)N) {
      if (prefix[u] != prefix[u + 1]) continue;
      if (early) pdl_wait();
      const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
      const int qh0 = p.unit_is_q ? hu : hu * p.group;
      for (int i = tid; i < GE * D; i += NW * 32)
        store_out_elem(p.out, p.out_dtype, ((size_t)b * p.num_q_heads + qh0) * D + i, 0.f);
    }
  }
  if (lo >= hi) {
    if (early) pdl_wait();   // the block must not complete before the preceding grid
    return;
  }

  // ---- chunk lookups: chunk x of the block's range -> unit, table entries,
  // addresses (the producer warp's, or each self-fed consumer warp's)
  const uint64_t pol = policy_evict_first();
  const int cpp = ps / kChunk;
  // raw lookup of chunk x: unit, chunk-in-unit, and the loaded table entries
  // (l2: the sparse second-level entry was loaded by lookup2)
  struct Raw {
    int u, k, sp, phys, l2;
  };
  auto fetch = [&](int x, Raw& r) {   // issues the global loads
    r.u = -1; r.k = 0; r.sp = 0; r.phys = -1; r.l2 = 0;
    if (x >= hi) return;
    r.u = find_unit(prefix, U, x);
    r.k = x - prefix[r.u];
    const int b = r.u / p.units_per_b, hu = r.u - b * p.units_per_b;
    if (!sparse) {
      const int lp = (r.k * kChunk) / ps;
      if (r.k * kChunk < lens[b]) r.phys = p.block_table[(size_t)b * p.max_pages + lp];
    } else {
      const size_t row = (size_t)b * p.units_per_b + hu;
      if (early && r.k / cpp >= min(max(p.sel_count[row], 0), p.sel_stride)) {
        r.sp = kSkipSelected;   // past the unit's list: no page, no error
        return;
      }
      r.sp = p.sel_pages[row * p.sel_stride + r.k / cpp];
    }
  };
  auto resolve = [&](const Raw& r, ChunkInfo& ci) {   // consumes the loads
    ci.k = nullptr; ci.v = nullptr; ci.sz = nullptr; ci.u = r.u < 0 ? 0 : r.u;
    ci.nvalid = 0; ci.valid = 0; ci.fresh = 0; ci.last = 0; ci.row = 0;
    if (r.u < 0) return;
    const int b = r.u / p.units_per_b, hu = r.u - b * p.units_per_b;
    const int L = lens[b];
    int t0, g, phys = r.phys;
    if (!sparse) {
      t0 = r.k * kChunk;
      g = hu;
    } else {
      if (r.sp == kSkipSelected) return;
      g = p.unit_is_q ? hu / p.group : hu;
      if (r.sp < 0 || (long long)r.sp * ps >= L) {
        flag_status(p.dev_status, PKV_DEV_BAD_SELECTED);
        return;
      }
      t0 = r.sp * ps + (r.k % cpp) * kChunk;
      if (t0 < L) phys = r.l2 ? r.phys : p.block_table[(size_t)b * p.max_pages + t0 / ps];
    }
    const int nv = min(kChunk, L - t0);
    if (nv <= 0) return;
    if (phys < 0 || phys >= p.num_pages) {
      flag_status(p.dev_status, PKV_DEV_BAD_PAGE);
      return;
    }
    const int off = t0 % ps;
    const size_t row0 = ((size_t)phys * p.num_kv_heads + g) * ps + off;
    ci.k = p.k_pages + row0 * Geo::ROW;
    ci.v = p.v_pages + row0 * Geo::ROW;
    ci.row = (int)row0;   // the host keeps pool rows below 2^31 for tensor copies
    if constexpr (Geo::PTOK) ci.sz = p.kv_sz + row0 * 4;
    if constexpr (KV == KV_I8G)
      ci.sz = p.kv_sz + (((size_t)phys * p.num_kv_heads + g) * (ps / 64) + off / 64) * 4;
    ci.nvalid = nv;
    ci.valid = 1;
    ci.last = !sparse && t0 + nv == L;
    if (early) {
      int bnd = L - p.fresh_rows;   // first row the preceding kernel may write
      if constexpr (KV == KV_I8G) bnd = bnd <= 0 ? 0 : bnd / 64 * 64;
      ci.fresh = t0 + nv > bnd;
    }
  };
  // sparse: the table entry of the selected page (issues the dependent load
  // ahead of resolve; an out-of-range page is left to resolve to report)
  auto lookup2 = [&](Raw& r) {
    if (!sparse || r.u < 0 || r.sp == kSkipSelected) return;
    const int b = r.u / p.units_per_b;
    const int L = lens[b];
    if (r.sp < 0 || (long long)r.sp * ps >= L) return;
    const int t0 = r.sp * ps + (r.k % cpp) * kChunk;
    if (t0 < L) {
      r.phys = p.block_table[(size_t)b * p.max_pages + t0 / ps];
      r.l2 = 1;
    }
  };

  if constexpr (!SELF) {
  if (warp == NW) {
    // ================================================================ producer
    // Lane l resolves chunk base + l of each batch of 32. The table entries of
    // batch k + 1 are loaded right after batch k's copies are issued, so their
    // latency overlaps the streaming of batch k.
    // Copies are issued by up to S lanes at once (one per ring stage): a single
    // issuing thread serialises the bulk-copy instructions and cannot keep the
    // ring full. Lane l owns chunk nbase + l of the batch; it waits for its
    // stage's previous use, which is always the phase just before its own.
    int nbase = 0;
    bool abort = false;
    bool waited = !early;    // warp-uniform
    auto wait_prior = [&]() {
      pdl_wait();
      pdl_launch_dependents();
      waited = true;
    };
    // early sparse calls: the page lists are the preceding kernel's output
    if (sparse && !waited) wait_prior();
    Raw cur;
    fetch(lo + lane, cur);
    for (int base = lo; base < hi && !abort; base += 32) {
      ChunkInfo e;
      resolve(cur, e);
      const int cnt = min(32, hi - base);
      bool my_abort = false;
      for (int k0 = 0; k0 < cnt; k0 += S) {
        const bool mine = lane >= k0 && lane < min(cnt, k0 + S);
        if (!waited && __any_sync(0xffffffffu, mine && e.fresh)) wait_prior();
        if constexpr (KV != KV_I8G) {
          unsigned todo = p.k_new ? __ballot_sync(0xffffffffu, mine && e.valid && e.last) : 0u;
          if (todo) {
            // the new token of each of these units, written by the whole warp;
            // with early start the caller promises that the work still running
            // before this call leaves these rows alone, so no wait is needed
            while (todo) {
              const int src = __ffs(todo) - 1;
              todo &= todo - 1;
              const unsigned long long pk = __shfl_sync(0xffffffffu, (unsigned long long)e.k, src);
              const unsigned long long pv = __shfl_sync(0xffffffffu, (unsigned long long)e.v, src);
              const unsigned long long pz = __shfl_sync(0xffffffffu, (unsigned long long)e.sz, src);
              append_token_row<D, KV>(p, __shfl_sync(0xffffffffu, e.u, src),
                                      __shfl_sync(0xffffffffu, e.nvalid, src) - 1,
                                      reinterpret_cast<uint8_t*>(pk), reinterpret_cast<uint8_t*>(pv),
                                      reinterpret_cast<float*>(pz), lane);
            }
            __syncwarp();
            // the rows were written through the generic proxy; the bulk copies
            // below read them through the async proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
        }
        if (mine) {
          const int n = nbase + lane;
          const int s = n % S, use = n / S;
          if (use > 0 && !mbar_wait_bounded(smem_u32(&empty[s]), (use - 1) & 1)) {
            flag_status(p.dev_status, PKV_DEV_TIMEOUT);
            my_abort = true;
          } else {
            hdr[s] = make_int4(e.u, e.nvalid, e.valid, 0);
            const uint32_t fb = smem_u32(&full[s]);
            if (e.valid) {
              uint8_t* st = ring + (size_t)s * STAGE;
              mbar_arrive_expect_tx(fb, 2 * KB + SZB);
              if constexpr (SWZ) {
                tma_load_2d(smem_u32(st), &p.tmap_k, 0, e.row, fb, pol);
                tma_load_2d(smem_u32(st + KB), &p.tmap_v, 0, e.row, fb, pol);
                bulk_g2s(smem_u32(szring + (size_t)s * SZB), e.sz, SZB, fb, pol);
              } else {
                bulk_g2s(smem_u32(st), e.k, KB, fb, pol);
                bulk_g2s(smem_u32(st + KB), e.v, KB, fb, pol);
                if constexpr (SZB > 0) bulk_g2s(smem_u32(st + 2 * KB), e.sz, SZB, fb, pol);
              }
            } else {
              mbar_arrive(fb);
            }
          }
        }
        __syncwarp();
        if (__any_sync(0xffffffffu, my_abort)) break;
      }
      abort = __any_sync(0xffffffffu, my_abort);
      nbase += cnt;
      // the next batch's table loads overlap the streaming of the stages just issued
      fetch(base + 32 + lane, cur);
      // early start: by the end of the first batch the preceding kernel is
      // normally done; waiting here costs nothing and lets dependents launch
      if (!waited) wait_prior();
    }
    if (!waited) wait_prior();
    const int n = nbase;
    // Let every issued copy land before this warp (and so the block) can exit.
    if (lane == 0) {
      const int first = n > S ? n - S : 0;
      for (int i = first; i < n; ++i) {
        if (!mbar_wait_bounded(smem_u32(&full[i % S]), (i / S) & 1)) {
          flag_status(p.dev_status, PKV_DEV_TIMEOUT);
          break;
        }
      }
    }
    return;
  }
  }

  // q of the block's first units, staged in shared memory by the consumer
  // warps while the first copies are in flight: a unit's start then reads q
  // there instead of waiting on global loads mid-stream (later units, beyond
  // what kQStageBytes holds, load q as before)
  const int q_esz = p.q_dtype == PKV_F32 ? 4 : 2;
  const int q_unit_bytes = GE * D * q_esz;
  const int n_staged = min(ub - ua + 1, kQStageBytes / q_unit_bytes);
  for (int i = tid; i < n_staged * (q_unit_bytes / 16); i += NW * 32) {
    const int k = i / (q_unit_bytes / 16), o = i - k * (q_unit_bytes / 16);
    const int u = ua + k, b = u / p.units_per_b, hu = u - b * p.units_per_b;
    const int qh0 = p.unit_is_q ? hu : hu * p.group;
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const uint8_t*>(p.q) + ((size_t)b * p.num_q_heads + qh0) * D * q_esz);
    reinterpret_cast<uint4*>(qstage + (size_t)k * q_unit_bytes)[o] = __ldg(src + o);
  }
  named_bar_sync(2, NW * 32);
  // q of unit u: the staged copy, or its rows in global memory
  auto q_of = [&](int u) -> const void* {
    if (u - ua < n_staged) return qstage + (size_t)(u - ua) * q_unit_bytes;
    const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
    const int qh0 = p.unit_is_q ? hu : hu * p.group;
    return static_cast<const uint8_t*>(p.q) + ((size_t)b * p.num_q_heads + qh0) * D * q_esz;
  };

  // The block's last unit ub: its four warps' states are merged here into one
  // record at slot (c + ub) * 4 (the other units keep one record per warp), so
  // the combine reads one record from each block but a unit's last. After the
  // stream every copy this block issued has been consumed, so the ring holds
  // the four states; a warp that timed out may leave a copy in flight, and the
  // slot then gets an empty record (the status already reports the failure).
  auto merge_last_unit = [&](bool aborted, bool holds_ub, auto&& stage_state) {
    constexpr int RS = rec_floats(GE, D), HDR = rec_hdr(GE);
    float* staged = reinterpret_cast<float*>(ring);
    if (aborted) misc[kMiscAbort] = 1;
    named_bar_sync(1, NW * 32);               // every consumer is done with the ring
    const bool any_abort = misc[kMiscAbort] != 0;
    if (!any_abort) {
      float* mine = staged + warp * RS;
      if (holds_ub) {
        stage_state(mine);
      } else if (lane < GE) {
        mine[lane] = -INFINITY;
        mine[GE + lane] = 0.f;
      }
    }
    named_bar_sync(1, NW * 32);
    if (early) pdl_wait();
    float* dst = p.ws_wrec + (size_t)(c + ub) * NW * RS;
    if (any_abort) {
      if (tid < GE) {
        dst[tid] = -INFINITY;
        dst[GE + tid] = 0.f;
      }
      return;
    }
    for (int o = tid; o < GE * D; o += NW * 32) {
      const int h = o / D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, staged[w * RS + h]);
      float L = 0.f, A = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float m = staged[w * RS + h];
          if (m == -INFINITY) continue;   // empty state: its acc is not written
          const float f = exp2f(m - M);
          L = fmaf(f, staged[w * RS + GE + h], L);
          A = fmaf(f, staged[w * RS + HDR + o], A);
        }
      }
      dst[HDR + o] = A;
      if (o % D == 0) {
        dst[h] = M;
        dst[GE + h] = L;
      }
    }
  };

  if constexpr (!MMA) {
  // ================================================================== consumers
  const int r = lane >> 3, j = lane & 7;
  const int my_head = j / DUP;  // head this lane holds after the score reduction
  float* pb = pbuf_all + warp * PBUF;

  constexpr int QD2 = QD / 2, PD2 = PD / 2;
  uint64_t q2[GE][QD2];  // q * sm_scale * log2(e), packed pairs (score layout)
  float qsum = 0.f;
  uint64_t acc2[GE][PD2];
  float m_h = -INFINITY, l_h = 0.f, zs = 0.f;
  int u_cur = -1, next_unit = ua;

  constexpr int WRS = rec_floats(GE, D), WHDR = rec_hdr(GE);
  auto rec_of = [&](int u) { return p.ws_wrec + ((size_t)(c + u) * NW + warp) * WRS; };

  auto write_empty = [&](int u) {
    if (early) pdl_wait();
    if (lane < GE) {
      float* rec = rec_of(u);
      rec[lane] = -INFINITY;
      rec[GE + lane] = 0.f;
    }
  };

  auto flush_to = [&](float* rec) {   // global or shared memory
#pragma unroll
    for (int h = 0; h < GE; ++h) {
      const float zh = __shfl_sync(0xffffffffu, zs, h * DUP);
      float* dst = rec + WHDR + h * D + lane * PD;
      float a0, a1;
      unpack2f(acc2[h][0], a0, a1);
      if constexpr (PD == 4) {
        float a2, a3;
        unpack2f(acc2[h][1], a2, a3);
        *reinterpret_cast<float4*>(dst) = make_float4(a0 + zh, a1 + zh, a2 + zh, a3 + zh);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(a0 + zh, a1 + zh);
      }
    }
    if (r == 0 && (j % DUP) == 0) {
      rec[my_head] = m_h;
      rec[GE + my_head] = l_h;
    }
  };
  auto flush = [&](int u) {
    if (early) pdl_wait();
    flush_to(rec_of(u));
  };

  auto start_unit = [&](int u) {
    const void* qu = q_of(u);
    float part[GE];
#pragma unroll
    for (int h = 0; h < GE; ++h) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < QD2; ++e) {
        const size_t idx = (size_t)h * D;
        const float x0 = load_q_elem(qu, p.q_dtype, idx + qk_dim<D, KV>(j, 2 * e)) * p.q_scale;
        const float x1 = load_q_elem(qu, p.q_dtype, idx + qk_dim<D, KV>(j, 2 * e + 1)) * p.q_scale;
        q2[h][e] = pack2f(x0, x1);
        s += x0 + x1;
      }
      part[h] = s;
    }
    qsum = reduce_scatter8<GE>(part, j);
#pragma unroll
    for (int h = 0; h < GE; ++h)
#pragma unroll
      for (int e = 0; e < PD2; ++e) acc2[h][e] = 0ull;
    m_h = -INFINITY;
    l_h = 0.f;
    zs = 0.f;
  };

  bool abort = false;
  // S is a multiple of NW (checked by the host), so stage s is only ever read by
  // warp s % NW, which waits on its phases 0, 1, 2, ... in order.
  // chunk n of the block's range sits in stage n mod S at phase n / S; both
  // are stepped, not divided (S is a multiple of NW, so s wraps exactly)
  for (int n = warp, s = warp, use = 0; lo + n < hi; n += NW, s += NW, use += (s >= S), s -= (s >= S) ? S : 0) {
    if (!mbar_wait_bounded(smem_u32(&full[s]), use & 1)) {
      flag_status(p.dev_status, PKV_DEV_TIMEOUT);
      abort = true;
      break;
    }
    const int4 h4 = hdr[s];
    const uint8_t* st = ring + (size_t)s * STAGE;
    if (h4.x != u_cur) {
      if (u_cur >= 0) {
        flush(u_cur);
        next_unit = u_cur + 1;
      }
      for (int v = next_unit; v < h4.x; ++v) write_empty(v);
      u_cur = h4.x;
      start_unit(u_cur);
    }
    if (h4.z) {
      const int nvalid = h4.y;
      const float* sz = reinterpret_cast<const float*>(st + 2 * KB);
      float ks = 0.f, kz = 0.f, vs = 0.f, vz = 0.f;
      if constexpr (KV == KV_I8G) {
        ks = sz[0]; kz = sz[1]; vs = sz[2]; vz = sz[3];
      }
      // ---- scores
      float sc[4];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int t = 4 * it + r;
        uint64_t k2[QD2];
        load_k_slice<D, KV>(st + t * Geo::ROW, j, k2);
        float part[GE];
#pragma unroll
        for (int h = 0; h < GE; ++h) {
          uint64_t a = ffma2(q2[h][0], k2[0], 0ull);
#pragma unroll
          for (int e = 1; e < QD2; ++e) a = ffma2(q2[h][e], k2[e], a);
          part[h] = hsum2(a);
        }
        float sv = reduce_scatter8<GE>(part, j);
        if constexpr (Geo::PTOK) sv = fmaf(sz[t * 4 + 0], sv, sz[t * 4 + 1] * qsum);
        if constexpr (KV == KV_I8G) sv = fmaf(ks, sv, kz * qsum);
        sc[it] = t < nvalid ? sv : -INFINITY;
      }
      // ---- online softmax update (per head, in the score layout)
      float cmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 8));
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 16));
      const float m_new = fmaxf(m_h, cmax);
      const float alpha = fast_exp2(m_h - m_new);
      float pw[4];
      float psum = 0.f, pz = 0.f;
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const float pe = fast_exp2(sc[it] - m_new);
        psum += pe;
        if constexpr (Geo::PTOK) {
          const int t = 4 * it + r;
          if (t < nvalid) {
            pz = fmaf(pe, sz[t * 4 + 3], pz);
            pw[it] = pe * sz[t * 4 + 2];
          } else {
            pw[it] = 0.f;
          }
        } else if constexpr (KV == KV_I8G) {
          pw[it] = pe * vs;
        } else {
          pw[it] = pe;
        }
      }
      psum += __shfl_xor_sync(0xffffffffu, psum, 8);
      psum += __shfl_xor_sync(0xffffffffu, psum, 16);
      l_h = fmaf(l_h, alpha, psum);
      if constexpr (Geo::PTOK) {
        pz += __shfl_xor_sync(0xffffffffu, pz, 8);
        pz += __shfl_xor_sync(0xffffffffu, pz, 16);
        zs = fmaf(zs, alpha, pz);
      } else if constexpr (KV == KV_I8G) {
        zs = fmaf(zs, alpha, vz * psum);
      }
      m_h = m_new;
      if ((j % DUP) == 0) {
#pragma unroll
        for (int it = 0; it < 4; ++it) pb[(4 * it + r) * GE + my_head] = pw[it];
        if (r == 0) pb[kChunk * GE + my_head] = alpha;
      }
      __syncwarp();
      // ---- values (value layout)
#pragma unroll
      for (int h = 0; h < GE; ++h) {
        const float al = pb[kChunk * GE + h];
        const uint64_t al2 = pack2f(al, al);
#pragma unroll
        for (int e = 0; e < PD2; ++e) acc2[h][e] = fmul2(acc2[h][e], al2);
      }
      const uint8_t* vrow = st + KB;
      auto pv_token = [&](int t) {
        uint64_t v2[PD2];
        load_v_slice<D, KV>(vrow + t * Geo::ROW, lane, v2);
#pragma unroll
        for (int h = 0; h < GE; ++h) {
          const float pv = pb[t * GE + h];
          const uint64_t pv2 = pack2f(pv, pv);
#pragma unroll
          for (int e = 0; e < PD2; ++e) acc2[h][e] = ffma2(pv2, v2[e], acc2[h][e]);
        }
      };
      if (nvalid == kChunk) {
#pragma unroll
        for (int t = 0; t < kChunk; ++t) pv_token(t);
      } else {
        for (int t = 0; t < nvalid; ++t) pv_token(t);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
  }
  if (!abort) {
    if (u_cur >= 0 && u_cur != ub) {
      flush(u_cur);
      next_unit = u_cur + 1;
    }
    for (int v = next_unit; v < ub; ++v) write_empty(v);
  }
  merge_last_unit(abort, u_cur == ub, [&](float* rec) { flush_to(rec); });

  } else {
  // ============================================== consumers, tensor-core path
  // Thread (g = lane / 4, t = lane % 4). Scores: C fragment of the [16 tok] x
  // [8 head] product, i.e. tokens g and g + 8, heads 2t and 2t + 1 (with G = 4
  // the softmax runs on token g + 8 (t >> 1) of heads 2 (t & 1), + 1; with
  // G = 2 on token g + 8 (t & 1) of heads 0 and 1). The channel
  // axis is permuted so that thread t reads whole 16-byte blocks of a row:
  // blocks t, t + 4, ... or, with swizzled tiles, blocks 2t and 2t + 1.
  // Values: O^T [16 channels] x [8 heads] per m-tile; thread (g, t) owns
  // channels [g D/8, (g + 1) D/8) of every output head 2t, 2t + 1, and tokens
  // 4t .. 4t + 3 (swizzled tiles: 2t, 2t + 1, 2t + 8, 2t + 9) of the chunk
  // enter the product's k slots. With swizzled tiles every quarter-warp of a
  // fragment load touches 8 distinct 16-byte blocks: no bank conflicts.
  // INT8 K codes enter q.K^T offset, as 1024 + u (one byte permute per pair,
  // exact in fp16, no subtraction); the offset's product (the offset x the q
  // sum) is common to a head's tokens and leaves with the zero-point term.
  // 4-bit K codes enter as fp16 subnormals (one mask per pair): u 2^-24 for
  // the nibbles at bits 0-3 of a half, u 2^-20 for those at bits 4-7. The q
  // values of the first kind's k slots are multiplied by 16 once per unit
  // (or, where that would overflow fp16, the others by 1/16), so every
  // product carries one factor, which the key scale takes back.
  // 4-bit codes (64-byte rows at D = 128, whose 16-byte fragment loads are
  // already free of conflicts): thread t reads block t of a K row, 32
  // channels; a register pairs channels c and c + 4 of one word (k slots
  // 2t, 2t + 1 of a k-step); V tokens 4 jr + t enter k slots (2t, 2t + 1,
  // 2t + 8, 2t + 9) for jr = 0 .. 3, and a register pairs two tokens' nibbles
  // of one channel (a byte permute and a mask).
  // V codes enter P.V centred (u - 128; 4-bit: (u - 8) 2^-9, the masked
  // subnormal times 2^15 or 2^11 minus 2^-6 in one fp16 fma, all exact, the
  // 2^-9 taken back at flush); see the P.V step for why they are centred.
  //
  // The running P.V state is the MMA accumulator itself: a chunk first scales
  // it by alpha (skipped, warp-wide, while no running maximum moved) and its
  // products then accumulate into it. With centred V codes the tensor cores'
  // fp32 accumulation (not IEEE round-to-nearest) adds no error that grows
  // with the chunks a warp streams.
  constexpr bool BF = (KV == KV_BF16);
  constexpr bool U4 = (KV == KV_U4T);
  // codes enter q.K^T as u - KCEN_K (INT8: 1024 + u, 4-bit: u) and P.V as
  // u - KCEN_V (centred); the scale and zero-point terms take the rest. The
  // offset in q.K^T is common to every token of a head, so it only shifts the
  // products the tensor cores sum; P.V stays centred because a weight that
  // loses bits there would carry the offset into the output.
  constexpr float KCEN_K = U4 ? 0.f : -1024.f;
  constexpr float KCEN_V = U4 ? 8.f : 128.f;
  constexpr int ESZ = Geo::ESZ;
  constexpr int E = 16 / ESZ;                 // channels per 16-byte block
  constexpr int NB = (D / 4) / E;             // 16-byte blocks per thread per row
  constexpr int KS = D / 16;                  // k-steps of q.K^T
  constexpr int MT = D / 16;                  // m-tiles of P.V
  constexpr int DPT = D / 8;                  // channels per thread group in P.V
  // With G <= 4 the hi and lo parts of P fill the 8 columns of one P.V MMA
  // (columns [0, G) hi, [G, 2G) lo), halving the P.V tensor work; the lo
  // columns are added to the hi ones at flush.
  constexpr bool PACK = GE <= 4;
  // With G = 4 the score columns of lanes t = 2, 3 are idle (heads 4 .. 7):
  // those lanes take over the token g + 8 scores of lanes t - 2, so every lane
  // runs the softmax of one token for heads 2 (t & 1), 2 (t & 1) + 1. With
  // G = 2, lane t = 1 takes over those of lane 0 (lanes 2, 3 work on idle rows).
  constexpr bool RED = GE == 4 || GE == 2;
  constexpr int RX = GE == 4 ? 2 : 1;   // lane distance of a token pair's halves
  const int g = lane >> 2, t = lane & 3;
  float* pb = pbuf_all + warp * PBUF;
  // logical 16-byte block m (of NB) of a row that thread t reads, and where a
  // logical block of row r sits in shared memory
  auto kblock = [&](int m) { return SWZ ? 2 * t + m : t + 4 * m; };
  auto phys_block = [&](int r, int blk) { return SWZ ? (blk ^ (r & 7)) : blk; };
  auto chan = [&](int i) { return kblock(i / E) * E + (i % E); };
  // V rows (tokens) of k slots 2t, 2t + 1, 2t + 8, 2t + 9 of this thread
  auto vtok = [&](int jr) {
    return U4 ? 4 * jr + t : (SWZ ? 2 * t + (jr & 1) + 8 * (jr >> 1) : 4 * t + jr);
  };

  uint32_t qb[KS][2];
  float qs[2];
  float kmul = 0x1p20f;   // 4-bit: the key scale's factor for the codes' 2^-20 or 2^-24
  float acc[MT][4];
  float m2[2], l2[2], zs2[2];
  int u_cur = -1, next_unit = ua;
  constexpr int WRS = rec_floats(GE, D), WHDR = rec_hdr(GE);
  auto rec_of = [&](int u) { return p.ws_wrec + ((size_t)(c + u) * NW + warp) * WRS; };
  auto write_empty = [&](int u) {
    if (early) pdl_wait();
    if (lane < GE) {
      float* rec = rec_of(u);
      rec[lane] = -INFINITY;
      rec[GE + lane] = 0.f;
    }
  };
  auto flush_to = [&](float* rec) {   // global or shared memory
    if constexpr (GE == 1) {   // the lo column 1 sits beside the hi column 0
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        acc[mt][0] += acc[mt][1];
        acc[mt][2] += acc[mt][3];
      }
    } else if constexpr (PACK) {   // lo columns (threads t + G/2) into the hi ones
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] += __shfl_down_sync(0xffffffffu, acc[mt][e], GE / 2);
    }
    // l and the zero-point sum are kept per lane (tokens g, g + 8; with G = 4
    // or 2 one of them, the other in lane t ^ RX); sum the lanes of each head
    // here instead of on every chunk
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
      for (int off = RED ? RX : 4; off < 32; off = off == RX ? 4 : off << 1) {
        l2[jj] += __shfl_xor_sync(0xffffffffu, l2[jj], off);
        if constexpr (KV != KV_F16 && KV != KV_BF16) zs2[jj] += __shfl_xor_sync(0xffffffffu, zs2[jj], off);
      }
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int h = 2 * t + jj;
      if (h < GE) {
        float* dst = rec + WHDR + h * D + g * DPT;
#pragma unroll
        for (int mt = 0; mt < MT; mt += 2) {
          constexpr float VS = U4 ? 512.f : 1.f;   // 4-bit V entered as (u - 8) 2^-9
          *reinterpret_cast<float4*>(dst + 2 * mt) =
              make_float4(fmaf(acc[mt][jj], VS, zs2[jj]), fmaf(acc[mt][2 + jj], VS, zs2[jj]),
                          fmaf(acc[mt + 1][jj], VS, zs2[jj]), fmaf(acc[mt + 1][2 + jj], VS, zs2[jj]));
        }
        if (g == 0) {
          rec[h] = m2[jj];
          rec[GE + h] = l2[jj];
        }
      }
    }
  };
  auto flush = [&](int u) {
    if (early) pdl_wait();
    flush_to(rec_of(u));
  };
  auto start_unit = [&](int u) {
    float part = 0.f;   // units are (sequence, kv head) on this path; q is 16-bit
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const uint16_t*>(q_of(u)) + (g < GE ? g : 0) * D);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t w0 = 0u, w1 = 0u;
      if constexpr (U4) {
        // k slots (2t, 2t + 1) = channels (c, c + 4), (2t + 8, 2t + 9) = (c + 1, c + 5)
        const uint16_t* qh = reinterpret_cast<const uint16_t*>(qrow);
        const int c = t * (D / 4) + 8 * (kk >> 1) + 2 * (kk & 1);
        if (g < GE) {
          w0 = (uint32_t)qh[c] | ((uint32_t)qh[c + 4] << 16);
          w1 = (uint32_t)qh[c + 1] | ((uint32_t)qh[c + 5] << 16);
        }
      } else {
        const int ch = chan(4 * kk);
        if (g < GE) {
          w0 = qrow[ch / 2];
          w1 = qrow[ch / 2 + 1];
        }
      }
      part += h2lo_f(w0, BF) + h2hi_f(w0, BF) + h2lo_f(w1, BF) + h2hi_f(w1, BF);
      qb[kk][0] = w0;
      qb[kk][1] = w1;
    }
    if constexpr (U4) {
      // The k slots of qb[.][0] meet the codes at bits 0-3 (u 2^-24), those of
      // qb[.][1] the codes at bits 4-7 (u 2^-20). The first are scaled by 16
      // (exact), so every product is q u 2^-20; where some |q| > 4094 (16 q
      // would overflow fp16) the second are scaled by 1/16 instead, and every
      // product is q u 2^-24.
      float qa = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk)
        qa = fmaxf(qa, fmaxf(fabsf(h2lo_f(qb[kk][0], false)), fabsf(h2hi_f(qb[kk][0], false))));
      const bool wide = __any_sync(0xffffffffu, qa > 4094.f);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        if (wide)
          qb[kk][1] = hfma2_rn(qb[kk][1], kH2x1o16, kH2m0);
        else
          qb[kk][0] = hfma2_rn(qb[kk][0], kH2x16, kH2m0);
      }
      kmul = wide ? 0x1p24f : 0x1p20f;
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);     // q sum of head g
    const int qh = GE == 4 ? 2 * (t & 1) : (GE == 2 ? 2 * (t >> 1) : 2 * t);
    qs[0] = __shfl_sync(0xffffffffu, part, qh * 4);
    qs[1] = __shfl_sync(0xffffffffu, part, (qh + 1) * 4);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
    m2[0] = m2[1] = -INFINITY;
    l2[0] = l2[1] = 0.f;
    zs2[0] = zs2[1] = 0.f;
  };

  // ---- self-fed (SELF): the warp copies its own chunks. Block chunk
  // n = warp + NW j (the warp's chunk j) sits in stage n mod S at phase n / S;
  // S is a multiple of NW, so the warp's stages are its own. Its first S / NW
  // chunks are copied up front, and chunk j + S / NW into chunk j's stage once
  // the warp is done with chunk j. Lane l holds the lookups of the warp's
  // chunk 32 cb + l. The next batch is looked up when the first of its chunks
  // is copied: the host plans these blocks for calls of at most ~128 chunks
  // per block, i.e. one batch per warp, so no lookups are held in flight
  // across the stream.
  const int DW = S / NW;
  const int span = hi - lo;
  const int nown = span > warp ? (span - warp + NW - 1) / NW : 0;
  // pool row of the warp's chunk 32 cb + lane (32 bits for tensor copies,
  // whose rows the host keeps below 2^31), and its unit << 7 | fresh << 6 |
  // valid << 5 | nvalid (units stay below 2^24)
  using RowT = typename std::conditional<SWZ, int, unsigned long long>::type;
  RowT a_row = 0;
  int a_uf = 0;
  int cb = 0;
  bool waited = !early;
  auto own_x = [&](int j) { return j < nown ? lo + warp + NW * j : hi; };
  auto take_batch = [&](const Raw& r) {
    ChunkInfo ci;
    resolve(r, ci);
    a_row = ci.valid ? (RowT)((ci.k - p.k_pages) / Geo::ROW) : (RowT)0;
    a_uf = (ci.u << 7) | (ci.fresh << 6) | (ci.valid << 5) | ci.nvalid;
    if constexpr (KV != KV_I8G) {
      // the new token of each unit ending in the batch (fused append), written
      // by the warp before the chunk holding it is copied; with early start
      // the caller promises that the work still running leaves these rows alone
      unsigned todo = p.k_new ? __ballot_sync(0xffffffffu, ci.valid && ci.last) : 0u;
      if (todo) {
        while (todo) {
          const int src = __ffs(todo) - 1;
          todo &= todo - 1;
          const unsigned long long pk = __shfl_sync(0xffffffffu, (unsigned long long)ci.k, src);
          const unsigned long long pv = __shfl_sync(0xffffffffu, (unsigned long long)ci.v, src);
          const unsigned long long pz = __shfl_sync(0xffffffffu, (unsigned long long)ci.sz, src);
          append_token_row<D, KV>(p, __shfl_sync(0xffffffffu, ci.u, src),
                                  __shfl_sync(0xffffffffu, ci.nvalid, src) - 1,
                                  reinterpret_cast<uint8_t*>(pk), reinterpret_cast<uint8_t*>(pv),
                                  reinterpret_cast<float*>(pz), lane);
        }
        __syncwarp();
        // written through the generic proxy, copied through the async proxy
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
    }
  };
  // copy the warp's chunk j into its stage s (warp-uniform; the warp has used
  // every value it read from the stage's previous chunk)
  auto issue = [&](int j, int s) {
    if ((j >> 5) != cb) {
      cb = j >> 5;
      Raw r;
      fetch(own_x(32 * cb + lane), r);
      lookup2(r);
      take_batch(r);
    }
    // the lane holding chunk j's lookups issues its copies
    if (lane == (j & 31)) {
      const RowT row = a_row;
      const int u = a_uf >> 7, fl = a_uf & 127;
      if (((fl >> 6) & 1) && !waited) {   // fresh rows: the preceding grid may still write them
        pdl_wait();
        waited = true;
      }
      hdr[s] = make_int4(u, fl & 31, (fl >> 5) & 1, 0);
      const uint32_t fb = smem_u32(&full[s]);
      if ((fl >> 5) & 1) {
        uint8_t* st = ring + (size_t)s * STAGE;
        const float* szp = nullptr;
        if constexpr (Geo::PTOK) szp = p.kv_sz + row * 4;
        if constexpr (KV == KV_I8G) szp = p.kv_sz + (row / 64) * 4;   // page_size is a multiple of 64
        mbar_arrive_expect_tx(fb, 2 * KB + SZB);
        if constexpr (SWZ) {
          tma_load_2d(smem_u32(st), &p.tmap_k, 0, (int)row, fb, pol);
          tma_load_2d(smem_u32(st + KB), &p.tmap_v, 0, (int)row, fb, pol);
          bulk_g2s(smem_u32(szring + (size_t)s * SZB), szp, SZB, fb, pol);
        } else {
          bulk_g2s(smem_u32(st), p.k_pages + row * Geo::ROW, KB, fb, pol);
          bulk_g2s(smem_u32(st + KB), p.v_pages + row * Geo::ROW, KB, fb, pol);
          if constexpr (SZB > 0) bulk_g2s(smem_u32(st + 2 * KB), szp, SZB, fb, pol);
        }
      } else {
        mbar_arrive(fb);
      }
    }
  };
  if constexpr (SELF) {
    // early sparse calls: the page lists are the preceding kernel's output
    if (sparse && !waited) {
      pdl_wait();
      waited = true;
    }
    Raw r0;
    fetch(own_x(lane), r0);
    lookup2(r0);
    take_batch(r0);
    for (int j = 0; j < DW && j < nown; ++j) issue(j, warp + NW * j);
  }

  bool abort = false;
  int jstop = 0;   // self-fed: the chunk whose wait gave up
  // chunk n of the block's range sits in stage n mod S at phase n / S; both
  // are stepped, not divided (S is a multiple of NW, so s wraps exactly)
  for (int j = 0, n = warp, s = warp, use = 0; lo + n < hi;
       ++j, n += NW, s += NW, use += (s >= S), s -= (s >= S) ? S : 0) {
    if (!mbar_wait_bounded(smem_u32(&full[s]), use & 1)) {
      flag_status(p.dev_status, PKV_DEV_TIMEOUT);
      abort = true;
      jstop = j;
      break;
    }
    const int4 h4 = hdr[s];
    const uint8_t* st = ring + (size_t)s * STAGE;
    if (h4.x != u_cur) {
      if (u_cur >= 0) {
        flush(u_cur);
        next_unit = u_cur + 1;
      }
      for (int v = next_unit; v < h4.x; ++v) write_empty(v);
      u_cur = h4.x;
      start_unit(u_cur);
    }
    if (h4.z) {
      const int nvalid = h4.y;
      const float* sz = reinterpret_cast<const float*>(SWZ ? szring + (size_t)s * SZB : st + 2 * KB);
      // ---- q.K^T on the tensor cores (even and odd k-steps in two
      // accumulators: two dependent MMA chains of half the length)
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      float sco[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (U4) {
        // block t (D / 8 bytes: D / 4 channels) of rows g and g + 8
        constexpr int NWD = D / 32;   // words per block
        uint32_t kw0[NWD], kw1[NWD];
        if constexpr (NWD == 4) {
          const uint4 a = *reinterpret_cast<const uint4*>(st + g * Geo::ROW + t * 16);
          const uint4 b = *reinterpret_cast<const uint4*>(st + (g + 8) * Geo::ROW + t * 16);
          kw0[0] = a.x; kw0[1] = a.y; kw0[2] = a.z; kw0[3] = a.w;
          kw1[0] = b.x; kw1[1] = b.y; kw1[2] = b.z; kw1[3] = b.w;
        } else {
          const uint2 a = *reinterpret_cast<const uint2*>(st + g * Geo::ROW + t * 8);
          const uint2 b = *reinterpret_cast<const uint2*>(st + (g + 8) * Geo::ROW + t * 8);
          kw0[0] = a.x; kw0[1] = a.y;
          kw1[0] = b.x; kw1[1] = b.y;
        }
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          // k-step 2w + h: channels (c, c + 4) at bits 0-3 of each half of
          // word w >> 8h, (c + 1, c + 5) at bits 4-7
          const int w = kk >> 1, h = kk & 1;
          const uint32_t x0 = h ? kw0[w] >> 8 : kw0[w], x1 = h ? kw1[w] >> 8 : kw1[w];
          const uint32_t a0 = x0 & kNibLo, a2 = x0 & kNibHi;
          const uint32_t a1 = x1 & kNibLo, a3 = x1 & kNibHi;
          if (kk & 1)
            mma16816<BF>(sco, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
          else
            mma16816<BF>(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] += sco[e];
      } else {
        uint4 k0[NB], k1[NB];
#pragma unroll
        for (int m = 0; m < NB; ++m) {
          k0[m] = *reinterpret_cast<const uint4*>(st + g * Geo::ROW + phys_block(g, kblock(m)) * 16);
          k1[m] = *reinterpret_cast<const uint4*>(st + (g + 8) * Geo::ROW + phys_block(g + 8, kblock(m)) * 16);
        }
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int m = (4 * kk) / E;
          const int wi = ((4 * kk) % E) * ESZ / 4;
          uint32_t a0, a1, a2, a3;
          if constexpr (ESZ == 1) {
            const uint32_t w0 = word_of(k0[m], wi);
            const uint32_t w1 = word_of(k1[m], wi);
            a0 = u8x2_to_h2(w0, 0x4140u);
            a2 = u8x2_to_h2(w0, 0x4342u);
            a1 = u8x2_to_h2(w1, 0x4140u);
            a3 = u8x2_to_h2(w1, 0x4342u);
          } else {
            a0 = word_of(k0[m], wi);
            a2 = word_of(k0[m], wi + 1);
            a1 = word_of(k1[m], wi);
            a3 = word_of(k1[m], wi + 1);
          }
          if (kk & 1)
            mma16816<BF>(sco, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
          else
            mma16816<BF>(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] += sco[e];
      }
      float al[2];
      if constexpr (RED) {
        const int hf = GE == 4 ? t >> 1 : t & 1;   // 0: token g, 1: token g + 8 (lane t - RX's)
        const float x2 = __shfl_up_sync(0xffffffffu, sc[2], RX);
        const float x3 = __shfl_up_sync(0xffffffffu, sc[3], RX);
        float s2[2] = {hf ? x2 : sc[0], hf ? x3 : sc[1]};
        const int tok = g + 8 * hf;
        float vs = 0.f, vz = 0.f;
        if constexpr (Geo::PTOK) {
          const float4 z = *reinterpret_cast<const float4*>(sz + tok * 4);
          const float kc = fmaf(KCEN_K, z.x, z.y);   // s (u - KCEN_K) + (z + KCEN_K s)
          const float ks = U4 ? z.x * kmul : z.x;
          s2[0] = fmaf(ks, s2[0], kc * qs[0]);
          s2[1] = fmaf(ks, s2[1], kc * qs[1]);
          vs = z.z;
          vz = fmaf(KCEN_V, z.z, z.w);   // centred V codes
        } else if constexpr (KV == KV_I8G) {
          const float4 z = *reinterpret_cast<const float4*>(sz);
          const float kc = fmaf(KCEN_K, z.x, z.y);
          s2[0] = fmaf(z.x, s2[0], kc * qs[0]);
          s2[1] = fmaf(z.x, s2[1], kc * qs[1]);
          vs = z.z;
          vz = fmaf(KCEN_V, z.z, z.w);
        }
        const bool ok = tok < nvalid;
        s2[0] *= p.q_scale;
        s2[1] *= p.q_scale;
        if (!ok) { s2[0] = -INFINITY; s2[1] = -INFINITY; }
        // ---- online softmax per head, over the 16 tokens of lanes (g, t) and
        // (g, t ^ RX)
        float pw2[2];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          float cm = s2[jj];
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, RX));
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
          const float mn = fmaxf(m2[jj], cm);
          al[jj] = fast_exp2(m2[jj] - mn);
          const float p0 = fast_exp2(s2[jj] - mn);
          l2[jj] = fmaf(l2[jj], al[jj], p0);
          if constexpr (Geo::PTOK) {
            zs2[jj] = fmaf(zs2[jj], al[jj], ok ? p0 * vz : 0.f);
            pw2[jj] = ok ? p0 * vs : 0.f;
          } else if constexpr (KV == KV_I8G) {
            zs2[jj] = fmaf(zs2[jj], al[jj], vz * p0);
            pw2[jj] = p0 * vs;
          } else {
            pw2[jj] = p0;
          }
          m2[jj] = mn;
        }
        const int prow = GE == 4 ? 2 * (t & 1) : 2 * (t >> 1);   // G = 2: lanes 2, 3 on idle rows
        pb[prow * kChunk + tok] = pw2[0];
        pb[(prow + 1) * kChunk + tok] = pw2[1];
      } else {
        // sc: (tok g, head 2t), (tok g, head 2t+1), (tok g+8, head 2t), (tok g+8, head 2t+1)
        float vs0 = 0.f, vz0 = 0.f, vs1 = 0.f, vz1 = 0.f;
        if constexpr (Geo::PTOK) {
          const float4 z0 = *reinterpret_cast<const float4*>(sz + g * 4);
          const float4 z1 = *reinterpret_cast<const float4*>(sz + (g + 8) * 4);
          // s (u - KCEN_K) + (z + KCEN_K s) = s u + z
          const float kc0 = fmaf(KCEN_K, z0.x, z0.y), kc1 = fmaf(KCEN_K, z1.x, z1.y);
          const float ks0 = U4 ? z0.x * kmul : z0.x, ks1 = U4 ? z1.x * kmul : z1.x;
          sc[0] = fmaf(ks0, sc[0], kc0 * qs[0]);
          sc[1] = fmaf(ks0, sc[1], kc0 * qs[1]);
          sc[2] = fmaf(ks1, sc[2], kc1 * qs[0]);
          sc[3] = fmaf(ks1, sc[3], kc1 * qs[1]);
          // V codes enter P.V centred: vs (u - KCEN_V) + (vz + KCEN_V vs) = vs u + vz
          vs0 = z0.z; vz0 = fmaf(KCEN_V, z0.z, z0.w); vs1 = z1.z; vz1 = fmaf(KCEN_V, z1.z, z1.w);
        } else if constexpr (KV == KV_I8G) {
          const float4 z = *reinterpret_cast<const float4*>(sz);
          const float kc = fmaf(KCEN_K, z.x, z.y);   // as for per-token scales
          sc[0] = fmaf(z.x, sc[0], kc * qs[0]);
          sc[1] = fmaf(z.x, sc[1], kc * qs[1]);
          sc[2] = fmaf(z.x, sc[2], kc * qs[0]);
          sc[3] = fmaf(z.x, sc[3], kc * qs[1]);
          vs0 = vs1 = z.z;
          vz0 = vz1 = fmaf(KCEN_V, z.z, z.w);   // centred codes, as for per-token scales
        }
        const bool ok0 = g < nvalid, ok1 = g + 8 < nvalid;
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] *= p.q_scale;
        if (!ok0) { sc[0] = -INFINITY; sc[1] = -INFINITY; }
        if (!ok1) { sc[2] = -INFINITY; sc[3] = -INFINITY; }
        // ---- online softmax per head 2t + jj
        float pw[4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          float cm = fmaxf(sc[jj], sc[2 + jj]);
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
          const float mn = fmaxf(m2[jj], cm);
          al[jj] = fast_exp2(m2[jj] - mn);
          const float p0 = fast_exp2(sc[jj] - mn), p1 = fast_exp2(sc[2 + jj] - mn);
          // lane-local running sums (rescaled like the accumulator; the lanes
          // of a head are summed at flush)
          l2[jj] = fmaf(l2[jj], al[jj], p0 + p1);
          if constexpr (Geo::PTOK) {
            const float pz = (ok0 ? p0 * vz0 : 0.f) + (ok1 ? p1 * vz1 : 0.f);
            zs2[jj] = fmaf(zs2[jj], al[jj], pz);
            pw[jj] = ok0 ? p0 * vs0 : 0.f;
            pw[2 + jj] = ok1 ? p1 * vs1 : 0.f;
          } else if constexpr (KV == KV_I8G) {
            zs2[jj] = fmaf(zs2[jj], al[jj], vz0 * (p0 + p1));
            pw[jj] = p0 * vs0;
            pw[2 + jj] = p1 * vs1;
          } else {
            pw[jj] = p0;
            pw[2 + jj] = p1;
          }
          m2[jj] = mn;
        }
        // P' to [head][token] in shared memory, then as the B operand of P.V
        pb[(2 * t) * kChunk + g] = pw[0];
        pb[(2 * t + 1) * kChunk + g] = pw[1];
        pb[(2 * t) * kChunk + g + 8] = pw[2];
        pb[(2 * t + 1) * kChunk + g + 8] = pw[3];
      }
      __syncwarp();
      // B column g: head g (hi part), or with PACK the lo part of head g - GE;
      // its k slots are the tokens vtok(0 .. 3)
      const int hb = (PACK && g >= GE) ? g - GE : g;
      const float* pbh = pb + (hb < GE ? hb : 0) * kChunk;
      float2 pv01, pv23;
      if constexpr (U4) {
        pv01 = make_float2(pbh[t], pbh[t + 4]);
        pv23 = make_float2(pbh[t + 8], pbh[t + 12]);
      } else if constexpr (SWZ) {
        pv01 = *reinterpret_cast<const float2*>(pbh + 2 * t);
        pv23 = *reinterpret_cast<const float2*>(pbh + 2 * t + 8);
      } else {
        const float4 pv4 = *reinterpret_cast<const float4*>(pbh + 4 * t);
        pv01 = make_float2(pv4.x, pv4.y);
        pv23 = make_float2(pv4.z, pv4.w);
      }
      __syncwarp();
      if (g >= (PACK ? 2 * GE : GE)) {
        pv01 = make_float2(0.f, 0.f);
        pv23 = make_float2(0.f, 0.f);
      }
      uint32_t bh0, bl0, bh1, bl1;
      split_hi_lo<BF>(pv01.x, pv01.y, bh0, bl0);
      split_hi_lo<BF>(pv23.x, pv23.y, bh1, bl1);
      if (PACK && g >= GE) {
        bh0 = bl0;
        bh1 = bl1;
      }
      // ---- P.V on the tensor cores, accumulated into the running state
      float a0s = al[0], a1s = al[1];
      if constexpr (GE == 1) {   // columns 0 and 1: hi and lo parts of head 0
        a1s = al[0];
      } else if constexpr (PACK && !RED) {   // lo columns of heads 2 (t - GE/2) + jj
        const int src = t >= GE / 2 ? lane - GE / 2 : lane;
        a0s = __shfl_sync(0xffffffffu, al[0], src);
        a1s = __shfl_sync(0xffffffffu, al[1], src);
      }
      if (__any_sync(0xffffffffu, a0s != 1.f || a1s != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          acc[mt][0] *= a0s;
          acc[mt][1] *= a1s;
          acc[mt][2] *= a0s;
          acc[mt][3] *= a1s;
        }
      }
      const uint8_t* vrow = st + KB;
      if constexpr (U4) {
        // 4-bit: channels [g DPT, (g+1) DPT) = DPT / 2 bytes of tokens vtok(0 .. 3)
        constexpr int NWV = DPT / 8;   // words per token (2 at D = 128, 1 at 64)
        uint32_t rw[4][NWV];
#pragma unroll
        for (int jr = 0; jr < 4; ++jr) {
          const uint8_t* src = vrow + vtok(jr) * Geo::ROW + g * (DPT / 2);
          if constexpr (NWV == 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(src);
            rw[jr][0] = v.x;
            rw[jr][1] = v.y;
          } else {
            rw[jr][0] = *reinterpret_cast<const uint32_t*>(src);
          }
        }
        // m-tile mt: byte mt of the thread's bytes; rows g / g + 8 = its low /
        // high nibble (channels 16 g + 2 mt, + 1); the permute puts the byte
        // of two tokens at bytes 0 and 2
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int wi = mt >> 2, bsel = mt & 3;
          const uint32_t sel = (uint32_t)(bsel | (bsel << 4) | ((bsel + 4) << 8) | ((bsel + 4) << 12));
          const uint32_t t01 = __byte_perm(rw[0][wi], rw[1][wi], sel);
          const uint32_t t23 = __byte_perm(rw[2][wi], rw[3][wi], sel);
          const uint32_t a0 = hfma2_rn(t01 & kNibLo, kH2x2p15, kH2m2pm6);
          const uint32_t a1 = hfma2_rn(t01 & kNibHi, kH2x2p11, kH2m2pm6);
          const uint32_t a2 = hfma2_rn(t23 & kNibLo, kH2x2p15, kH2m2pm6);
          const uint32_t a3 = hfma2_rn(t23 & kNibHi, kH2x2p11, kH2m2pm6);
          mma16816<BF>(acc[mt], a0, a1, a2, a3, bh0, bh1);
          if constexpr (!PACK) mma16816<BF>(acc[mt], a0, a1, a2, a3, bl0, bl1);
        }
      } else if constexpr (ESZ == 1) {
        // int8: dims [g DPT, (g+1) DPT) of tokens vtok(0 .. 3) (DPT bytes per row)
        uint32_t rw[4][DPT / 4];
#pragma unroll
        for (int jr = 0; jr < 4; ++jr) {
          const int r = vtok(jr);
          const uint8_t* src = vrow + r * Geo::ROW + phys_block(r, g) * DPT;
          if constexpr (DPT == 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(src);
            rw[jr][0] = v.x; rw[jr][1] = v.y; rw[jr][2] = v.z; rw[jr][3] = v.w;
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(src);
            rw[jr][0] = v.x; rw[jr][1] = v.y;
          }
        }
        // Masked tokens (stale codes) need no clearing: every code is a
        // finite u - 128 and their weights are exactly 0. The codes enter
        // centred, not as 1024 + u, because weights p * vs below fp16's range
        // are lost in the hi/lo split: with a 1024 offset each lost weight
        // would drop 1024 p vs from the product while the fp32 zero-point sum
        // still removes it, a bias that grows with the tokens a warp streams.
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int wi = mt / 2;
          const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
          const uint32_t t01 = __byte_perm(rw[0][wi], rw[1][wi], sel);
          const uint32_t t23 = __byte_perm(rw[2][wi], rw[3][wi], sel);
          const uint32_t a0 = u8x2_to_h2c(t01, 0x4140u), a1 = u8x2_to_h2c(t01, 0x4342u);
          const uint32_t a2 = u8x2_to_h2c(t23, 0x4140u), a3 = u8x2_to_h2c(t23, 0x4342u);
          mma16816<BF>(acc[mt], a0, a1, a2, a3, bh0, bh1);
          if constexpr (!PACK) mma16816<BF>(acc[mt], a0, a1, a2, a3, bl0, bl1);
        }
      } else {
        // fp16 / bf16: dims [g DPT, (g+1) DPT) of tokens vtok(0 .. 3) (2 DPT bytes per row)
        uint32_t rw[4][DPT / 2];
#pragma unroll
        for (int jr = 0; jr < 4; ++jr) {
          const uint8_t* src = vrow + vtok(jr) * Geo::ROW + g * DPT * 2;
#pragma unroll
          for (int q4 = 0; q4 < DPT / 8; ++q4) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + q4 * 16);
            rw[jr][4 * q4 + 0] = v.x; rw[jr][4 * q4 + 1] = v.y;
            rw[jr][4 * q4 + 2] = v.z; rw[jr][4 * q4 + 3] = v.w;
          }
        }
        if (nvalid < kChunk) {   // masked tokens may hold NaN; weight 0 would not clear it
#pragma unroll
          for (int jr = 0; jr < 4; ++jr)
            if (vtok(jr) >= nvalid)
#pragma unroll
              for (int i = 0; i < DPT / 2; ++i) rw[jr][i] = 0u;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t a0 = __byte_perm(rw[0][mt], rw[1][mt], 0x5410u);
          const uint32_t a1 = __byte_perm(rw[0][mt], rw[1][mt], 0x7632u);
          const uint32_t a2 = __byte_perm(rw[2][mt], rw[3][mt], 0x5410u);
          const uint32_t a3 = __byte_perm(rw[2][mt], rw[3][mt], 0x7632u);
          mma16816<BF>(acc[mt], a0, a1, a2, a3, bh0, bh1);
          if constexpr (!PACK) mma16816<BF>(acc[mt], a0, a1, a2, a3, bl0, bl1);
        }
      }
    }
    __syncwarp();
    if constexpr (SELF) {
      if (j + DW < nown) issue(j + DW, s);
    } else {
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
  }
  if constexpr (SELF) {
    if (abort) {   // let the copies still in flight land before the block exits
      for (int j = jstop; j < nown && j < jstop + DW; ++j) {
        if (!mbar_wait_bounded(smem_u32(&full[warp + NW * (j % DW)]), (j / DW) & 1)) break;
      }
    }
  }
  if (!abort) {
    if (u_cur >= 0 && u_cur != ub) {
      flush(u_cur);
      next_unit = u_cur + 1;
    }
    for (int v = next_unit; v < ub; ++v) write_empty(v);
  }
  merge_last_unit(abort, u_cur == ub, [&](float* rec) { flush_to(rec); });
  }

  // Block 0 publishes the unit prefix for the combine of sparse calls (dense
  // calls recompute it there from the lengths).
  if (blockIdx.x == 0) {
    if (early) pdl_wait();
    for (int u = tid; u <= U; u += NW * 32) p.ws_prefix[u] = prefix[u];
  }
}

// Merge of every unit's records: those of each block whose range overlaps the
// unit, i.e. blocks c_first .. c_last, whose slots ((c + u) * 4 + w) are
// consecutive: one (slot 0) from each block that ends inside the unit, where
// the unit is the block's last and its four warps were merged in the block,
// and four (one per warp, some empty) from a block that moves on past it:
//   M = max m_r,  out = sum_r 2^(m_r - M) acc_r / sum_r 2^(m_r - M) l_r
// (the log2-domain partial states of the attention kernel). The 128 threads
// of block (u, y) form RG = comb_groups record groups of OB = 128 / RG
// threads; thread (g, i) folds records g, g + RG, ... of output y OB + i of
// unit u, and group 0 merges the RG partials. The host picks RG from the
// expected records per unit (more groups when units span many blocks).
// Dense calls compute the unit's chunk range from the sequence lengths before
// waiting for the attention kernel (the lengths are inputs, not its output),
// so only the record loads follow the wait.
// 128 threads: more of these blocks are resident beside the attention blocks
// than of 256-thread ones (W2 22.5 -> 22.2 us per call in a chain, W4 31.8 ->
// 31.2 us), so the next call's kernel is released sooner.
constexpr int kCombineThreads = 128;
template <int D, int GE>
__global__ void __launch_bounds__(kCombineThreads, 4) attn_combine_kernel(const AttnParams p) {
  constexpr int RS = rec_floats(GE, D), HDR = rec_hdr(GE);
  constexpr int BATCH = 8;    // records in flight per thread
  constexpr int NWC = kCombineThreads / 32;
  __shared__ float part[3][kCombineThreads];
  __shared__ long long red[3][NWC];
  const int u = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int RG = p.comb_groups, OB = kCombineThreads / RG;
  const int grp = tid / OB;
  const int o = blockIdx.y * OB + (tid - grp * OB);   // output of the unit
  const bool active = o < GE * D;
  const bool sparse = p.sel_pages != nullptr;
  // the unit chunk ranges follow from the lengths alone in dense calls and in
  // early-start sparse calls (whose units of sequence b all get min(list
  // stride, pages of b) pages' chunks); other sparse calls read the prefix
  // the attention kernel's block 0 wrote
  const bool from_lens = !sparse || p.fresh_rows >= 0;
  const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
  long long W = 0, s0 = 0, s1 = 0;
  if (from_lens) {
    // chunks of each unit of sequence b' (n_b', as in the attention kernel):
    // W = units_per_b * sum_b' n_b', and unit u starts after all units of
    // sequences b' < b and hu units of sequence b
    const int cap = p.max_pages * p.page_size;
    long long tot = 0, before = 0, nb = 0;
    for (int bb = tid; bb < p.batch; bb += kCombineThreads) {
      int L = p.seq_lens[bb];
      L = L < 0 ? 0 : (L > cap ? cap : L);
      const long long n = !sparse ? (L + kChunk - 1) / kChunk
                                  : (long long)min(p.sel_stride, (L + p.page_size - 1) / p.page_size) *
                                        (p.page_size / kChunk);
      tot += n;
      if (bb < b) before += n;
      if (bb == b) nb = n;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, off);
      before += __shfl_xor_sync(0xffffffffu, before, off);
      nb += __shfl_xor_sync(0xffffffffu, nb, off);
    }
    if (lane == 0) {
      red[0][warp] = tot;
      red[1][warp] = before;
      red[2][warp] = nb;
    }
    __syncthreads();
    tot = 0; before = 0; nb = 0;
#pragma unroll
    for (int w = 0; w < NWC; ++w) {
      tot += red[0][w];
      before += red[1][w];
      nb += red[2][w];
    }
    W = tot * p.units_per_b;
    s0 = before * p.units_per_b + (long long)hu * nb;
    s1 = s0 + nb;
  }
  const long long N = p.num_ctas;
  // the unit's covering blocks (known before the wait for dense calls)
  // Records of the unit: one (slot 0, the block's merged last unit) from each
  // covering block before the last, then the last block's: one if the unit is
  // its last unit too (the unit ends with the block), else four (one per warp).
  auto cover = [&](int& c_first, int& nb1, int& R4) {
    c_first = cta_of(s0, W, N);
    const int c_last = cta_of(s1 - 1, W, N);
    nb1 = c_last - c_first;
    R4 = nb1 + (cta_lo(c_last + 1, W, N) <= s1 ? 1 : kConsumerWarps);
  };
  int c_first = 0, nb1 = 0, R4 = 0;
  if (from_lens && s0 != s1) cover(c_first, nb1, R4);
  // The next kernel may launch now, before this grid's wait: its own wait
  // covers this grid, which completes only after the attention grid it
  // merges. (Triggering at the very start measured slower: W2 25.4 against
  // 22.9 us per call in a 32-call chain.)
  pdl_launch_dependents();
  pdl_wait();
  if (!from_lens) {
    W = __ldcg(p.ws_prefix + p.num_units);
    s0 = __ldcg(p.ws_prefix + u);
    s1 = __ldcg(p.ws_prefix + u + 1);
    if (s0 != s1) cover(c_first, nb1, R4);
  }
  if (s0 == s1) return;   // no chunks: the attention kernel wrote zeros
  // With at least one chunk per block (W >= N) every covering block wrote its
  // records; otherwise blocks with empty ranges are skipped.
  const bool dense_cover = W >= N;
  const int oo = active ? o : 0;
  const int h = oo / D;
  const float* rec0 = p.ws_wrec + (size_t)(c_first + u) * kConsumerWarps * RS;
  // slot of record r relative to rec0: block c_first + r (slot 0) for r < nb1,
  // then slots 0.. of block c_first + nb1
  auto rec_slot = [&](int r) { return r < nb1 ? r * kConsumerWarps : nb1 * kConsumerWarps + (r - nb1); };
  float M = -INFINITY, L = 0.f, A = 0.f;
  // BATCH records per load round, two rounds in flight: the next round's loads
  // are issued before the current one is folded
  auto load = [&](int r0, float (&mc)[BATCH], float (&lc)[BATCH], float (&ac)[BATCH]) {
#pragma unroll
    for (int i = 0; i < BATCH; ++i) {
      const int r = r0 + i * RG;
      const int cc = c_first + (r < nb1 ? r : nb1);
      const bool ok = r < R4 && (dense_cover || cta_lo(cc, W, N) < cta_lo(cc + 1, W, N));
      const float* rr = rec0 + (size_t)(ok ? rec_slot(r) : 0) * RS;
      mc[i] = ok ? __ldcg(rr + h) : -INFINITY;
      lc[i] = __ldcg(rr + GE + h);
      ac[i] = __ldcg(rr + HDR + oo);
    }
  };
  // merge (m, l, a) states: max first, then independent exponentials
  auto fold = [&](const float (&mc)[BATCH], const float (&lc)[BATCH], const float (&ac)[BATCH]) {
    float Mb = M;
#pragma unroll
    for (int i = 0; i < BATCH; ++i) Mb = fmaxf(Mb, mc[i]);
    if (Mb == -INFINITY) return;
    float Lb = M == -INFINITY ? 0.f : L * exp2f(M - Mb);
    float Ab = M == -INFINITY ? 0.f : A * exp2f(M - Mb);
#pragma unroll
    for (int i = 0; i < BATCH; ++i) {
      if (mc[i] == -INFINITY) continue;   // empty record: its acc is not written
      const float f = exp2f(mc[i] - Mb);
      Lb = fmaf(f, lc[i], Lb);
      Ab = fmaf(f, ac[i], Ab);
    }
    M = Mb;
    L = Lb;
    A = Ab;
  };
  {
    const int step = RG * BATCH;
    float m0[BATCH], l0[BATCH], a0[BATCH], m1[BATCH], l1[BATCH], a1[BATCH];
    int r0 = grp;
    if (r0 < R4) load(r0, m0, l0, a0);
    while (r0 < R4) {
      if (r0 + step < R4) load(r0 + step, m1, l1, a1);
      fold(m0, l0, a0);
      r0 += step;
      if (r0 >= R4) break;
      if (r0 + step < R4) load(r0 + step, m0, l0, a0);
      fold(m1, l1, a1);
      r0 += step;
    }
  }
  if (RG > 1) {
    part[0][tid] = M;
    part[1][tid] = L;
    part[2][tid] = A;
    __syncthreads();
    if (grp != 0) return;
    float Mx = M;
    for (int g = 1; g < RG; ++g) Mx = fmaxf(Mx, part[0][g * OB + tid]);
    float Ls = 0.f, As = 0.f;
    if (Mx != -INFINITY) {
      for (int g = 0; g < RG; ++g) {
        const float mw = part[0][g * OB + tid];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - Mx);
        Ls = fmaf(f, part[1][g * OB + tid], Ls);
        As = fmaf(f, part[2][g * OB + tid], As);
      }
    }
    L = Ls;
    A = As;
  }
  if (!active) return;
  const int qh0 = p.unit_is_q ? hu : hu * p.group;
  store_out_elem(p.out, p.out_dtype, ((size_t)b * p.num_q_heads + qh0) * D + o, L > 0.f ? A / L : 0.f);
}

}  // namespace pkv
