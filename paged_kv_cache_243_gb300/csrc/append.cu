// kv_append kernels: write new tokens into their pages [HBM-layout page,
// section 三 append_kv: block = pos / block_size, slot = pos % block_size,
// through the block table], quantising to INT8 when the cache is INT8
// [HBM-layout page, section 二 per-token; Gemini page, 第一章 per-64-token
// group] or to 4-bit codes [KV-practice page, section 3.2; per token], and
// refreshing the per-page channel bounding boxes of the keys [TinyServe page,
// section 2.1].
//
// The quantisers are exact fp32 operation sequences (correctly rounded
// subtract and divide, round half to even), so codes, scales and zero-points
// are bit-identical to any other IEEE implementation of the same sequence:
//   INT8: s = (max - min) / 255, z = min, code = clamp(rint((x - z) / s), 0, 255) - 128,
//   stored as the byte u = code + 128;
//   4-bit: s = (max - min) / 15, z = min, u = clamp(rint((x - z) / s), 0, 15).
#include "pkv_internal.h"
#include "quant.cuh"

namespace pkv {

namespace {

__device__ __forceinline__ float load_src(const void* p, int dtype, size_t i) {
  return dtype == PKV_BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i])
                           : __half2float(reinterpret_cast<const __half*>(p)[i]);
}

__device__ __forceinline__ bool row_window(const AppendParams& p, int b, int& pos, int& n) {
  pos = p.positions[b] + p.pos_bias;
  n = p.new_lens ? p.new_lens[b] : p.t_new;
  if (n > p.t_new || n < 0 || pos < 0 || (long long)pos + n > (long long)p.max_pages * p.page_size) {
    flag_status(p.dev_status, PKV_DEV_BAD_POSITION);
    return false;
  }
  return n > 0;
}

// Position -> (logical page, row in the page): a shift and a mask for the
// usual power-of-two page sizes, else an integer division.
__device__ __forceinline__ int page_div(const AppendParams& p, int x) {
  return p.ps_shift >= 0 ? x >> p.ps_shift : x / p.page_size;
}
__device__ __forceinline__ int page_mod(const AppendParams& p, int x) {
  return p.ps_shift >= 0 ? x & (p.page_size - 1) : x % p.page_size;
}

__device__ __forceinline__ int page_of(const AppendParams& p, int b, int lp) {
  const int phys = p.block_table[(size_t)b * p.max_pages + lp];
  if (phys < 0 || phys >= p.num_pages) {
    flag_status(p.dev_status, PKV_DEV_BAD_PAGE);
    return -1;
  }
  return phys;
}

// fp16/bf16 cache: copy (with conversion when the source dtype differs).
// grid (t_new, batch); each thread moves 8 elements per pass. The source rows
// are loaded before the block-table lookup so the two latencies overlap.
__global__ void append_copy_kernel(const AppendParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x, b = blockIdx.y;
  const int D = p.head_dim, H = p.num_kv_heads;
  const int per_head = D / 8;
  const int total = 2 * H * per_head;
  constexpr int kMaxPer = 4;  // 16-byte vectors per thread held across the lookup
  uint4 vals[kMaxPer];
  auto src_of = [&](int idx, int& kv, int& g, int& e8) {
    kv = idx / (H * per_head);
    const int rem = idx - kv * H * per_head;
    g = rem / per_head;
    e8 = rem - g * per_head;
    return (((size_t)b * p.t_new + t) * H + g) * D + e8 * 8;
  };
#pragma unroll
  for (int k = 0; k < kMaxPer; ++k) {
    const int idx = threadIdx.x + k * blockDim.x;
    if (idx < total) {
      int kv, g, e8;
      const size_t src = src_of(idx, kv, g, e8);
      vals[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(kv ? p.v_new : p.k_new) + src);
    }
  }
  int pos, n;
  if (!row_window(p, b, pos, n) || t >= n) return;
  const int tp = pos + t;
  const int phys = page_of(p, b, page_div(p, tp));
  if (phys < 0) return;
  const int slot = page_mod(p, tp);
  auto put = [&](int idx, uint4 v) {
    int kv, g, e8;
    src_of(idx, kv, g, e8);
    const size_t dst = (((size_t)phys * H + g) * p.page_size + slot) * D + e8 * 8;
    uint16_t* dp = reinterpret_cast<uint16_t*>(kv ? p.v_pages : p.k_pages);
    if (p.src_dtype != p.kv_dtype) {
      uint16_t* h = reinterpret_cast<uint16_t*>(&v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = p.src_dtype == PKV_BF16 ? __bfloat162float(__ushort_as_bfloat16(h[e]))
                                                : __half2float(__ushort_as_half(h[e]));
        h[e] = p.kv_dtype == PKV_BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x))
                                      : __half_as_ushort(__float2half_rn(x));
      }
    }
    *reinterpret_cast<uint4*>(dp + dst) = v;
  };
#pragma unroll
  for (int k = 0; k < kMaxPer; ++k) {
    const int idx = threadIdx.x + k * blockDim.x;
    if (idx < total) put(idx, vals[k]);
  }
  for (int idx = threadIdx.x + kMaxPer * blockDim.x; idx < total; idx += blockDim.x) {
    int kv, g, e8;
    const size_t src = src_of(idx, kv, g, e8);
    put(idx, *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(kv ? p.v_new : p.k_new) + src));
  }
}

// Per-token INT8 (U4: per-token 4-bit codes, two per byte): 8 lanes per
// token, each quantising D/8 consecutive values, so the per-token work
// (min/max across lanes, scale, reciprocal) is shared by 8 lanes, not 32.
// grid (token blocks, kv head * 2 + K|V, row), up to 8 warps per block (fewer
// for short appends): warp w of a block serves tokens 8w .. 8w + 7 of the
// block's as two groups of 4, whose source rows are all loaded before either
// is processed (and before the position and block-table lookups), so a warp
// keeps 2 KB of loads in flight.
constexpr int kTokPerWarp = 8;
template <int D, bool U4, bool SRC_BF16>
__global__ void __launch_bounds__(256) append_per_token_kernel(const AppendParams p) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int EPL = D / 8;   // values per lane: 16 (D = 128) or 8 (D = 64)
  const int lane = threadIdx.x & 31, sub = lane >> 3, part = lane & 7;
  const int H = p.num_kv_heads;
  const int kv = blockIdx.y & 1, g = blockIdx.y >> 1, b = blockIdx.z;
  const int tpb = (blockDim.x >> 5) * kTokPerWarp;
  const int wt = blockIdx.x * tpb + (threadIdx.x >> 5) * kTokPerWarp;   // the warp's first token
  if (wt >= p.t_new) return;   // warp-uniform
  const uint16_t* sp = reinterpret_cast<const uint16_t*>(kv ? p.v_new : p.k_new);
  uint2 raw[2][EPL / 4];
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const int t = wt + 4 * gi + sub;
    const uint16_t* src = sp + (((size_t)b * p.t_new + (t < p.t_new ? t : 0)) * H + g) * D + part * EPL;
#pragma unroll
    for (int e = 0; e < EPL / 4; ++e) raw[gi][e] = reinterpret_cast<const uint2*>(src)[e];
  }
  int pos, n;
  if (!row_window(p, b, pos, n)) return;
  int phys[2];
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const int t = wt + 4 * gi + sub;
    phys[gi] = t < n ? p.block_table[(size_t)b * p.max_pages + page_div(p, pos + t)] : -1;
  }
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const int t = wt + 4 * gi + sub;
    float x[EPL];
#pragma unroll
    for (int e = 0; e < EPL / 4; ++e) {
      const float4 f = widen4_t<SRC_BF16>(raw[gi][e]);
      x[4 * e] = f.x; x[4 * e + 1] = f.y; x[4 * e + 2] = f.z; x[4 * e + 3] = f.w;
    }
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int e = 1; e < EPL; ++e) {
      mn = fminf(mn, x[e]);
      mx = fmaxf(mx, x[e]);
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) {   // the token's 8 lanes
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    if (t >= n) continue;
    const int ph = phys[gi];
    if (ph < 0 || ph >= p.num_pages) {
      if (part == 0) flag_status(p.dev_status, PKV_DEV_BAD_PAGE);
      continue;
    }
    const float s = __fdiv_rn(__fsub_rn(mx, mn), U4 ? 15.f : 255.f);
    const float z = mn;
    const float rs = quant_recip(s);
    const size_t row = ((size_t)ph * H + g) * p.page_size + page_mod(p, pos + t);
    if constexpr (U4) {
      uint32_t w[EPL / 8];
      quant_nibbles<EPL>(x, s, z, rs, w);
      uint8_t* dst = reinterpret_cast<uint8_t*>(kv ? p.v_pages : p.k_pages) + row * (D / 2) + part * (EPL / 2);
      if constexpr (EPL == 16)
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      else
        *reinterpret_cast<uint32_t*>(dst) = w[0];
    } else {
      uint32_t w[EPL / 4];
      quant_words<EPL>(x, s, z, rs, w);
      uint8_t* dst = reinterpret_cast<uint8_t*>(kv ? p.v_pages : p.k_pages) + row * D + part * EPL;
      if constexpr (EPL == 16)
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      else
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    }
    if (part == 0) {
      p.kv_sz[row * 4 + kv * 2 + 0] = s;
      p.kv_sz[row * 4 + kv * 2 + 1] = z;
    }
  }
}

__device__ __forceinline__ float* tail_row(const AppendParams& p, int b, int g, int kv, int parity) {
  return p.tail + ((((size_t)b * p.num_kv_heads + g) * 2 + kv) * 2 + parity) * 64 * p.head_dim;
}

// Per-64-token-group INT8. grid (group slot, kv head * 2 + kv, row); one block
// re-quantises one group that received tokens: its members are the kept
// originals of earlier tokens of the open group (tail) plus the new tokens.
// write_tail: also keep the new members of a group that stays open.
// Each thread holds up to kGroupVec4 float4s of the group in registers; all
// of its loads (tail and new tokens) are issued before the first use, and
// before the block-table lookup, so the block pays about one memory latency.
constexpr int kGroupThreads = 256;
template <int D>
__global__ void __launch_bounds__(kGroupThreads, 4) append_per_group_kernel(const AppendParams p, int write_tail) {
  constexpr int kGroupVec4 = 64 * D / 4 / kGroupThreads;   // float4s of a full group per thread
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red_mn[kGroupThreads / 32], red_mx[kGroupThreads / 32];
  __shared__ int ok_s;
  const int b = blockIdx.z, g = blockIdx.y >> 1, kv = blockIdx.y & 1;
  const int H = p.num_kv_heads;
  int pos, n;
  if (!row_window(p, b, pos, n)) return;
  const int gi = pos / 64 + blockIdx.x;
  if (gi > (pos + n - 1) / 64) return;
  const int t0 = gi * 64;
  const int t_end = min(t0 + 64, pos + n);
  const int nf = (t_end - t0) * D / 4;      // float4s of the group
  const void* sp = kv ? p.v_new : p.k_new;
  const float* tl = tail_row(p, b, g, kv, gi & 1);
  float4 x[kGroupVec4];
#pragma unroll
  for (int k = 0; k < kGroupVec4; ++k) {
    const int f = threadIdx.x + k * kGroupThreads;
    if (f < nf) {
      const int i = 4 * f, tt = i / D, e = i - tt * D, tok = t0 + tt;
      x[k] = tok < pos ? *reinterpret_cast<const float4*>(tl + i)
                       : load_src4(sp, p.src_dtype, (((size_t)b * p.t_new + (tok - pos)) * H + g) * D + e);
    }
  }
  if (threadIdx.x == 0) ok_s = page_of(p, b, page_div(p, t0));
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kGroupVec4; ++k) {
    if (threadIdx.x + k * kGroupThreads < nf) {
      mn = fminf(fminf(mn, x[k].x), fminf(x[k].y, fminf(x[k].z, x[k].w)));
      mx = fmaxf(fmaxf(mx, x[k].x), fmaxf(x[k].y, fmaxf(x[k].z, x[k].w)));
    }
  }
  for (int off = 16; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red_mn[warp] = mn;
    red_mx[warp] = mx;
  }
  __syncthreads();
  const int phys = ok_s;
  if (phys < 0) return;
  mn = red_mn[0];
  mx = red_mx[0];
#pragma unroll
  for (int w = 1; w < kGroupThreads / 32; ++w) {
    mn = fminf(mn, red_mn[w]);
    mx = fmaxf(mx, red_mx[w]);
  }
  const float s = __fdiv_rn(__fsub_rn(mx, mn), 255.f);
  const float z = mn;
  const float rs = quant_recip(s);
  const int off0 = page_mod(p, t0);
  uint8_t* dst = reinterpret_cast<uint8_t*>(kv ? p.v_pages : p.k_pages) +
                (((size_t)phys * H + g) * p.page_size + off0) * D;
  float* tw = tail_row(p, b, g, kv, gi & 1);
  const bool keep = write_tail && t_end - t0 < 64;
#pragma unroll
  for (int k = 0; k < kGroupVec4; ++k) {
    const int f = threadIdx.x + k * kGroupThreads;
    if (f < nf) {
      const int i = 4 * f;
      const float xv[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
      uint32_t wq[1];
      quant_words<4>(xv, s, z, rs, wq);
      *reinterpret_cast<uint32_t*>(dst + i) = wq[0];
      if (keep && t0 + i / D >= pos) *reinterpret_cast<float4*>(tw + i) = x[k];
    }
  }
  if (threadIdx.x == 0) {
    float* szp = p.kv_sz + (((size_t)phys * H + g) * (p.page_size / 64) + off0 / 64) * 4;
    szp[kv * 2 + 0] = s;
    szp[kv * 2 + 1] = z;
  }
}

// Bulk per-64-token-group INT8 for groups made of new tokens only: group
// slots 1, 2, ... of an append longer than one group (slot 0, which may hold
// earlier members of the open group, and the tail copy go to the kernels
// above and below). grid (group slot - 1, kv head, row); one block quantises
// K and V of one group together, holding the source values as 16-bit words
// (2 registers per 4 values), so it keeps 32 KB of loads in flight; both
// tensors' min/max meet in one block reduction.
template <int D>
__global__ void __launch_bounds__(kGroupThreads, 4) append_group_bulk_kernel(const AppendParams p) {
  constexpr int NV = 64 * D / 4 / kGroupThreads;   // 4-value elements per thread and tensor
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[4][kGroupThreads / 32];
  __shared__ int phys_s;
  const int b = blockIdx.z, g = blockIdx.y, H = p.num_kv_heads;
  int pos, n;
  if (!row_window(p, b, pos, n)) return;
  const int gi = pos / 64 + 1 + blockIdx.x;
  if (gi > (pos + n - 1) / 64) return;
  const int t0 = gi * 64;   // > pos: every member is a new token
  const int t_end = min(t0 + 64, pos + n);
  const int nf = (t_end - t0) * D / 4;
  const uint16_t* ks = reinterpret_cast<const uint16_t*>(p.k_new);
  const uint16_t* vs = reinterpret_cast<const uint16_t*>(p.v_new);
  uint2 kr[NV], vr[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int f = threadIdx.x + k * kGroupThreads;
    if (f < nf) {
      const int i = 4 * f, tt = i / D, e = i - tt * D;
      const size_t idx = (((size_t)b * p.t_new + (t0 + tt - pos)) * H + g) * D + e;
      kr[k] = *reinterpret_cast<const uint2*>(ks + idx);
      vr[k] = *reinterpret_cast<const uint2*>(vs + idx);
    }
  }
  if (threadIdx.x == 0) phys_s = page_of(p, b, page_div(p, t0));
  float kmn = INFINITY, kmx = -INFINITY, vmn = INFINITY, vmx = -INFINITY;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (threadIdx.x + k * kGroupThreads < nf) {
      const float4 a = widen4(kr[k], p.src_dtype), c = widen4(vr[k], p.src_dtype);
      kmn = fminf(fminf(kmn, a.x), fminf(a.y, fminf(a.z, a.w)));
      kmx = fmaxf(fmaxf(kmx, a.x), fmaxf(a.y, fmaxf(a.z, a.w)));
      vmn = fminf(fminf(vmn, c.x), fminf(c.y, fminf(c.z, c.w)));
      vmx = fmaxf(fmaxf(vmx, c.x), fmaxf(c.y, fmaxf(c.z, c.w)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    kmn = fminf(kmn, __shfl_xor_sync(0xffffffffu, kmn, off));
    kmx = fmaxf(kmx, __shfl_xor_sync(0xffffffffu, kmx, off));
    vmn = fminf(vmn, __shfl_xor_sync(0xffffffffu, vmn, off));
    vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, off));
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[0][warp] = kmn;
    red[1][warp] = kmx;
    red[2][warp] = vmn;
    red[3][warp] = vmx;
  }
  __syncthreads();
  const int phys = phys_s;
  if (phys < 0) return;
  kmn = red[0][0]; kmx = red[1][0]; vmn = red[2][0]; vmx = red[3][0];
#pragma unroll
  for (int w = 1; w < kGroupThreads / 32; ++w) {
    kmn = fminf(kmn, red[0][w]);
    kmx = fmaxf(kmx, red[1][w]);
    vmn = fminf(vmn, red[2][w]);
    vmx = fmaxf(vmx, red[3][w]);
  }
  const float sk = __fdiv_rn(__fsub_rn(kmx, kmn), 255.f), sv = __fdiv_rn(__fsub_rn(vmx, vmn), 255.f);
  const float rk = quant_recip(sk), rv = quant_recip(sv);
  const int off0 = page_mod(p, t0);
  const size_t base = (((size_t)phys * H + g) * p.page_size + off0) * D;
  uint8_t* kd = reinterpret_cast<uint8_t*>(p.k_pages) + base;
  uint8_t* vd = reinterpret_cast<uint8_t*>(p.v_pages) + base;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int f = threadIdx.x + k * kGroupThreads;
    if (f < nf) {
      const float4 a = widen4(kr[k], p.src_dtype), c = widen4(vr[k], p.src_dtype);
      const float xa[4] = {a.x, a.y, a.z, a.w}, xc[4] = {c.x, c.y, c.z, c.w};
      uint32_t wa[1], wc[1];
      quant_words<4>(xa, sk, kmn, rk, wa);
      quant_words<4>(xc, sv, vmn, rv, wc);
      *reinterpret_cast<uint32_t*>(kd + 4 * f) = wa[0];
      *reinterpret_cast<uint32_t*>(vd + 4 * f) = wc[0];
    }
  }
  if (threadIdx.x == 0) {
    float* szp = p.kv_sz + (((size_t)phys * H + g) * (p.page_size / 64) + off0 / 64) * 4;
    *reinterpret_cast<float4*>(szp) = make_float4(sk, kmn, sv, vmn);
  }
}

// Keeps the new members of each row's open group (appends longer than one
// group, run after the quantise kernel so no block reads a tail row another
// block rewrites). grid (kv head * 2 + kv, row).
__global__ void append_tail_kernel(const AppendParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.y, g = blockIdx.x >> 1, kv = blockIdx.x & 1;
  const int D = p.head_dim, H = p.num_kv_heads;
  int pos, n;
  if (!row_window(p, b, pos, n)) return;
  const int end = pos + n;
  if (end % 64 == 0) return;
  const int gi = (end - 1) / 64, t0 = gi * 64;
  const int first = max(t0, pos);
  const void* sp = kv ? p.v_new : p.k_new;
  float* tw = tail_row(p, b, g, kv, gi & 1);
  for (int i = threadIdx.x; i < (end - first) * D; i += blockDim.x) {
    const int tt = i / D, e = i - tt * D;
    const int tok = first + tt;
    tw[(size_t)(tok - t0) * D + e] =
        load_src(sp, p.src_dtype, (((size_t)b * p.t_new + (tok - pos)) * H + g) * D + e);
  }
}

// Recompute the key bounding box of every page the append touched, over the
// page's valid tokens, from the stored keys (INT8 and 4-bit codes restored as
// fl32(fl32(u * s) + z): a packed multiply, then the scalar __fadd_rn, which is
// never fused with it; ptxas may contract a packed mul.rn.f32x2 / add.rn.f32x2
// pair into one fma, a different rounding). One warp per (page, kv head):
// grid (page slot, kv head block of 4, row), 128 threads. Lane l covers
// channel block l mod 16 (D / 16 channels) of rows l / 16, l / 16 + 2, ...:
// a warp reads two whole rows per load instruction, with sixteen rows' loads
// in flight per pass, folds each channel over its eight rows in min/max
// chains, and merges the two row halves with one shuffle at the end.
template <int D, int KV>
__global__ void __launch_bounds__(128) append_meta_kernel(const AppendParams p) {
  constexpr int C = D / 16;   // channels per lane
  constexpr bool I8 = KV == KV_I8T || KV == KV_I8G;
  constexpr int RB = KV == KV_U4T ? C / 2 : (I8 ? C : 2 * C);   // bytes per lane per row
  constexpr int RW = RB >= 4 ? RB / 4 : 1;                      // 32-bit words per lane per row
  constexpr int ROWB = KV == KV_U4T ? D / 2 : (I8 ? D : 2 * D); // bytes per row
  constexpr int RPL = 8;                                        // rows per lane per pass
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.z, g = blockIdx.y * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int H = p.num_kv_heads, ps = p.page_size;
  if (g >= H) return;
  int pos, n;
  if (!row_window(p, b, pos, n)) return;
  const int lp = page_div(p, pos) + blockIdx.x;
  if (lp > page_div(p, pos + n - 1)) return;
  const int phys = page_of(p, b, lp);
  if (phys < 0) return;
  const int nv = min(ps, pos + n - lp * ps);
  const size_t row0 = ((size_t)phys * H + g) * ps;
  const int part = lane & 15, ro = lane >> 4;
  const uint8_t* kb = reinterpret_cast<const uint8_t*>(p.k_pages) + row0 * ROWB + part * RB;
  float mn[C], mx[C];
#pragma unroll
  for (int c = 0; c < C; ++c) {
    mn[c] = INFINITY;
    mx[c] = -INFINITY;
  }
  for (int r0 = 0; r0 < nv; r0 += 2 * RPL) {
    uint32_t w[RPL][RW];
    float2 sc[RPL];
    // rows of this pass: all valid (the usual case: one base, constant
    // offsets), or clamped to the last valid row (a repeated row leaves the
    // bounds unchanged)
    auto load_rows = [&](auto full_t) {
      constexpr bool FULL = decltype(full_t)::value;
#pragma unroll
      for (int i = 0; i < RPL; ++i) {
        const int t = FULL ? r0 + ro + 2 * i : min(r0 + ro + 2 * i, nv - 1);
        const uint8_t* src = FULL ? kb + (size_t)(r0 + ro) * ROWB + 2 * i * ROWB : kb + (size_t)t * ROWB;
        if constexpr (RB == 16) {
          const uint4 v = *reinterpret_cast<const uint4*>(src);
          w[i][0] = v.x; w[i][1] = v.y; w[i][2] = v.z; w[i][3] = v.w;
        } else if constexpr (RB == 8) {
          const uint2 v = *reinterpret_cast<const uint2*>(src);
          w[i][0] = v.x; w[i][1] = v.y;
        } else if constexpr (RB == 4) {
          w[i][0] = *reinterpret_cast<const uint32_t*>(src);
        } else {
          w[i][0] = *reinterpret_cast<const uint16_t*>(src);
        }
        if constexpr (KV == KV_I8T || KV == KV_U4T)
          sc[i] = *reinterpret_cast<const float2*>(p.kv_sz + (row0 + t) * 4);
        else if constexpr (KV == KV_I8G)
          sc[i] = *reinterpret_cast<const float2*>(p.kv_sz + (((size_t)phys * H + g) * (ps / 64) + t / 64) * 4);
        else
          sc[i] = make_float2(0.f, 0.f);
      }
    };
    if (r0 + 2 * RPL <= nv)
      load_rows(std::true_type{});
    else
      load_rows(std::false_type{});
    // channels (c, c + 1) of every row i: values (a[i], b[i]), then the chains
    auto fold = [&](int c, const float (&a)[RPL], const float (&bb)[RPL]) {
      float l0 = mn[c], h0 = mx[c], l1 = mn[c + 1], h1 = mx[c + 1];
#pragma unroll
      for (int i = 0; i < RPL; i += 2) {
        l0 = fminf(fminf(l0, a[i]), a[i + 1]);
        h0 = fmaxf(fmaxf(h0, a[i]), a[i + 1]);
        l1 = fminf(fminf(l1, bb[i]), bb[i + 1]);
        h1 = fmaxf(fmaxf(h1, bb[i]), bb[i + 1]);
      }
      mn[c] = l0; mx[c] = h0; mn[c + 1] = l1; mx[c + 1] = h1;
    };
    auto deq = [&](int i, uint64_t u2, float& a, float& bv) {   // fl32(fl32(u s) + z)
      float p0, p1;
      unpack2f(fmul2(u2, pack2f(sc[i].x, sc[i].x)), p0, p1);
      a = __fadd_rn(p0, sc[i].y);
      bv = __fadd_rn(p1, sc[i].y);
    };
#pragma unroll
    for (int q = 0; q < RW; ++q) {
      if constexpr (I8) {   // word q: channels 4q .. 4q + 3 of the lane's block
#pragma unroll
        for (int jp = 0; jp < 4 && 4 * q + jp < C; jp += 2) {
          float a[RPL], bv[RPL];
#pragma unroll
          for (int i = 0; i < RPL; ++i) deq(i, u8pair(w[i][q], jp), a[i], bv[i]);
          fold(4 * q + jp, a, bv);
        }
      } else if constexpr (KV == KV_U4T) {   // word q: channels 8q .. 8q + 7
#pragma unroll
        for (int j = 0; j < 4 && 8 * q + 2 * j < C; ++j) {
          float a[RPL], bv[RPL];
#pragma unroll
          for (int i = 0; i < RPL; ++i) {
            uint32_t lo, hi;
            split_nibbles(w[i][q], lo, hi);
            deq(i, u4pair(lo, hi, j), a[i], bv[i]);
          }
          fold(8 * q + 2 * j, a, bv);
        }
      } else {   // word q: channels 2q, 2q + 1
        float a[RPL], bv[RPL];
#pragma unroll
        for (int i = 0; i < RPL; ++i) unpack2<KV>(w[i][q], a[i], bv[i]);
        fold(2 * q, a, bv);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < C; ++c) {
    mn[c] = fminf(mn[c], __shfl_xor_sync(0xffffffffu, mn[c], 16));
    mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], 16));
  }
  if (ro != 0) return;
  float* meta = p.page_meta + (((size_t)phys * H + g) * 2) * D + part * C;
#pragma unroll
  for (int c = 0; c < C; c += 4) {
    *reinterpret_cast<float4*>(meta + c) = make_float4(mn[c], mn[c + 1], mn[c + 2], mn[c + 3]);
    *reinterpret_cast<float4*>(meta + D + c) = make_float4(mx[c], mx[c + 1], mx[c + 2], mx[c + 3]);
  }
}

}  // namespace

pkv_status launch_append(const AppendParams& p, cudaStream_t st) {
  const int H = p.num_kv_heads;
  AppendParams pc = p;
  void* args1[] = {&pc};
  cudaError_t e = cudaSuccess;
  if (p.kv_dtype == PKV_F16 || p.kv_dtype == PKV_BF16) {
    e = launch_pdl(reinterpret_cast<const void*>(&append_copy_kernel), dim3(p.t_new, p.batch), dim3(256), 0,
                   st, args1);
  } else if (p.quant == PKV_QUANT_PER_TOKEN) {
    const int warps = min(8, (p.t_new + kTokPerWarp - 1) / kTokPerWarp);
    const dim3 grid((p.t_new + warps * kTokPerWarp - 1) / (warps * kTokPerWarp), H * 2, p.batch);
    const bool u4 = p.kv_dtype == PKV_U4, bf = p.src_dtype == PKV_BF16;
    const void* fn = nullptr;
#define PKV_PT(d, q4, sb) \
    if (p.head_dim == d && u4 == q4 && bf == sb) fn = reinterpret_cast<const void*>(&append_per_token_kernel<d, q4, sb>);
    PKV_PT(128, false, false) PKV_PT(128, false, true) PKV_PT(128, true, false) PKV_PT(128, true, true)
    PKV_PT(64, false, false) PKV_PT(64, false, true) PKV_PT(64, true, false) PKV_PT(64, true, true)
#undef PKV_PT
    if (!fn) return PKV_ERR_UNSUPPORTED;
    e = launch_pdl(fn, grid, dim3(32 * warps), 0, st, args1);
  } else {
    const int groups = (p.t_new + 63) / 64 + 1;
    int inline_tail = p.t_new <= 64;
    void* args2[] = {&pc, &inline_tail};
    const void* fn = p.head_dim == 128 ? reinterpret_cast<const void*>(&append_per_group_kernel<128>)
                                       : reinterpret_cast<const void*>(&append_per_group_kernel<64>);
    // appends longer than a group: the first group slot (which may hold
    // earlier members of the open group) here, the others, all new tokens,
    // in the bulk kernel; the tail kernel then keeps the open group's members
    e = launch_pdl(fn, dim3(inline_tail ? groups : 1, H * 2, p.batch),
                   dim3(kGroupThreads), 0, st, args2);
    if (e == cudaSuccess && !inline_tail) {
      const void* fb = p.head_dim == 128 ? reinterpret_cast<const void*>(&append_group_bulk_kernel<128>)
                                         : reinterpret_cast<const void*>(&append_group_bulk_kernel<64>);
      e = launch_pdl(fb, dim3(groups - 1, H, p.batch), dim3(kGroupThreads), 0, st, args1);
    }
    if (e == cudaSuccess && !inline_tail)
      e = launch_pdl(reinterpret_cast<const void*>(&append_tail_kernel), dim3(H * 2, p.batch), dim3(256), 0,
                     st, args1);
  }
  if (e == cudaSuccess && p.page_meta) {
    const int pages = (p.t_new + p.page_size - 1) / p.page_size + 1;
    const int kind = p.kv_dtype == PKV_U4 ? KV_U4T
                   : p.kv_dtype == PKV_I8 ? (p.quant == PKV_QUANT_PER_TOKEN ? KV_I8T : KV_I8G)
                   : p.kv_dtype == PKV_BF16 ? KV_BF16 : KV_F16;
    const void* fn = nullptr;
#define PKV_META(d, k) \
    if (p.head_dim == d && kind == k) fn = reinterpret_cast<const void*>(&append_meta_kernel<d, k>);
    PKV_META(64, KV_F16) PKV_META(64, KV_BF16) PKV_META(64, KV_I8T) PKV_META(64, KV_I8G) PKV_META(64, KV_U4T)
    PKV_META(128, KV_F16) PKV_META(128, KV_BF16) PKV_META(128, KV_I8T) PKV_META(128, KV_I8G)
    PKV_META(128, KV_U4T)
#undef PKV_META
    if (!fn) return PKV_ERR_UNSUPPORTED;
    e = launch_pdl(fn, dim3(pages, (H + 3) / 4, p.batch), dim3(128), 0, st, args1);
  }
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
