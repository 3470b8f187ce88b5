// Paged decode attention: one persistent launch that splits the whole batch's
// KV chunks evenly over its thread blocks, streams each chunk into shared
// memory with 1-D bulk copies (TMA engine), and merges the per-block partial
// softmax states in the same launch.
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
// (unit, block-table lookup, addresses) and lane 0 issues cp.async.bulk copies
// of the chunk's K rows, V rows and INT8 scales into a ring of shared-memory
// stages, each guarded by a "full" and an "empty" mbarrier. Warps 0-3 consume
// chunks round robin; each keeps its own online-softmax state (running max m,
// sum l, accumulator) per query head, in the log2 domain. When a warp's chunk
// stream moves to another unit it writes its partial state to the workspace.
//
// Merge. Each unit's partials sit in workspace slots (block + unit) * 4 + warp.
// After its warps finish, a block bumps an arrival counter per unit it touched;
// the block that arrives last merges the unit's partials
//   M = max m_s,  out = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s
// and resets the counter to zero for the next call.
//
// Lane layouts. Scores: lane = 8 r + j handles token 4 it + r of the chunk and
// a D/8-wide slice of channels; the 8 lanes of a token reduce their partial
// dot products with a butterfly that also scatters the G query heads over the
// lanes (lane j ends with the full score of head j / (8 / G)). Values: lane
// owns channels [lane * D / 32, (lane + 1) * D / 32) of every token and all G
// heads. Probabilities move between the two layouts through shared memory.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
// Small shared scratch: [0] [1] merge masks, [4, 4 + 2 * 8) per-head M and L of
// the cross-block merge, [8, 8 + warps) scan totals (used before streaming).
constexpr int kMiscInts = 32;

struct AttnParams {
  const uint8_t* k_pages;
  const uint8_t* v_pages;
  const float* kv_sz;
  const void* q;
  void* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* sel_pages;  // NULL: dense
  const int32_t* sel_count;
  float* ws_wrec;     // per-warp partial records, slot ((block + unit) * 4 + warp)
  float* ws_crec;     // per-block partial records, slot (block + unit)
  int32_t* ws_prefix; // [num_units + 1] chunk prefix, written by block 0 for the combine
  int32_t* dev_status;
  int num_pages, page_size, num_kv_heads, num_q_heads, group;
  int batch, max_pages, sel_stride;
  int units_per_b, num_units;
  int num_ctas, stages;
  int q_dtype, out_dtype;
  float q_scale;  // sm_scale * log2(e): scores live in the log2 domain
};

struct ChunkInfo {
  const uint8_t* k;
  const uint8_t* v;
  const float* sz;
  int u;
  int nvalid;
  int valid;
  int pad;
};

template <int D, int KV>
struct AttnGeom {
  static constexpr int ESZ = (KV == KV_I8T || KV == KV_I8G) ? 1 : 2;
  static constexpr int ROW = D * ESZ;              // bytes of one token row
  static constexpr int KB = kChunk * ROW;          // bytes of one chunk of K (or V)
  static constexpr int SZB = KV == KV_I8T ? kChunk * 16 : (KV == KV_I8G ? 16 : 0);
  static constexpr int STAGE = ((2 * KB + SZB) + 127) / 128 * 128;
  static constexpr int QD = D / 8;                 // channels per lane in the score layout
  static constexpr int PD = D / 32;                // channels per lane in the value layout
};

template <int GE>
struct AttnSmem {
  static constexpr int PBUF = kChunk * GE + 8;     // floats per warp: p[16][GE], alpha[GE]
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
  s += (size_t)kConsumerWarps * (kChunk * ge + 8) * 4;
  s += 32 * sizeof(ChunkInfo);
  s += kMiscInts * 4;                              // misc
  s += (size_t)(units + 1) * 4 + (size_t)batch * 4;
  return (s + 15) / 16 * 16;
}

// Channel index of element e of lane-slot j in the score layout.
template <int D, int KV>
__device__ __forceinline__ int qk_dim(int j, int e) {
  if (AttnGeom<D, KV>::ESZ == 2 && D == 128) return e < 8 ? 8 * j + e : 64 + 8 * j + (e - 8);
  return AttnGeom<D, KV>::QD * j + e;
}

// Load this lane's D/8 channels of token row `row` (score layout) as packed
// fp32 pairs (INT8: u = code + 128).
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
  } else {
    if constexpr (D == 128) {
      const uint4 a = *reinterpret_cast<const uint4*>(row + j * 16);
      const uint32_t w[4] = {a.x ^ 0x80808080u, a.y ^ 0x80808080u, a.z ^ 0x80808080u, a.w ^ 0x80808080u};
#pragma unroll
      for (int i = 0; i < 8; ++i) k2[i] = u8pair(w[i >> 1], (i & 1) * 2);
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(row + j * 8);
      const uint32_t w[2] = {a.x ^ 0x80808080u, a.y ^ 0x80808080u};
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
  } else {
    if constexpr (D == 128) {
      const uint32_t a = *reinterpret_cast<const uint32_t*>(row + lane * 4) ^ 0x80808080u;
      v2[0] = u8pair(a, 0);
      v2[1] = u8pair(a, 2);
    } else {
      const uint32_t a = (uint32_t)(*reinterpret_cast<const uint16_t*>(row + lane * 2)) ^ 0x8080u;
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

__device__ __forceinline__ int find_unit(const int* prefix, int num_units, int x) {
  int lo = 0, hi = num_units - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int cta_lo(long long c, long long W, long long N) { return (int)(c * W / N); }
// Largest block c whose range starts at or before chunk x.
__device__ __forceinline__ int cta_of(long long x, long long W, long long N) {
  return (int)(((x + 1) * N - 1) / W);
}

template <int D, int GE, int KV>
__global__ void __launch_bounds__(kAttnThreads, 1) paged_attention_kernel(const AttnParams p) {
  using Geo = AttnGeom<D, KV>;
  constexpr int QD = Geo::QD, PD = Geo::PD, KB = Geo::KB, SZB = Geo::SZB, STAGE = Geo::STAGE;
  constexpr int PBUF = AttnSmem<GE>::PBUF;
  constexpr int DUP = 8 / GE;  // lanes (per token) that hold the same head after the scatter
  constexpr int NW = kConsumerWarps;

  extern __shared__ __align__(128) uint8_t smem[];
  const int S = p.stages;
  uint8_t* ring = smem;
  int4* hdr = reinterpret_cast<int4*>(smem + (size_t)S * STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(hdr + S);
  uint64_t* empty = full + S;
  float* pbuf_all = reinterpret_cast<float*>(empty + S);
  ChunkInfo* info = reinterpret_cast<ChunkInfo*>(pbuf_all + NW * PBUF);
  int* misc = reinterpret_cast<int*>(info + 32);
  int* prefix = misc + kMiscInts;
  int* lens = prefix + p.num_units + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int U = p.num_units;
  if (S <= 0 || S % NW != 0 || S > 32) {  // the host never launches this; refuse rather than race
    if (tid == 0) flag_status(p.dev_status, PKV_DEV_BAD_CONFIG);
    return;
  }
  const int ps = p.page_size;
  const bool sparse = p.sel_pages != nullptr;

  pdl_wait();
  pdl_launch_dependents();
  // ---- sequence lengths (clamped to the block table) and unit chunk counts
  for (int b = tid; b < p.batch; b += kAttnThreads) {
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
  fence_mbar_init();
  __syncthreads();

  const int per = (U + kAttnThreads - 1) / kAttnThreads;
  const int ua0 = min(U, tid * per), ua1 = min(U, ua0 + per);
  int my_sum = 0;
  for (int u = ua0; u < ua1; ++u) {
    const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
    const int L = lens[b];
    int n;
    if (!sparse) {
      n = (L + kChunk - 1) / kChunk;
    } else {
      int cnt = p.sel_count[b * p.num_q_heads + hu];
      cnt = cnt < 0 ? 0 : (cnt > p.sel_stride ? p.sel_stride : cnt);
      if (cnt == 0) {
        n = 0;
      } else {
        const int cpp = ps / kChunk;
        const int last = p.sel_pages[(size_t)(b * p.num_q_heads + hu) * p.sel_stride + cnt - 1];
        const int P = (L + ps - 1) / ps;
        const int lastc = (last >= 0 && last == P - 1) ? (L - last * ps + kChunk - 1) / kChunk : cpp;
        n = (cnt - 1) * cpp + lastc;
      }
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
    if (tid == kAttnThreads - 1) prefix[U] = wpre + incl;
  }
  __syncthreads();

  if (blockIdx.x == 0)
    for (int u = tid; u <= U; u += kAttnThreads) p.ws_prefix[u] = prefix[u];
  const long long W = prefix[U];
  const long long N = p.num_ctas;
  const int c = blockIdx.x;
  const int lo = W > 0 ? cta_lo(c, W, N) : 0;
  const int hi = W > 0 ? cta_lo(c + 1, W, N) : 0;
  const int ua = lo < hi ? find_unit(prefix, U, lo) : 0;
  const int ub = lo < hi ? find_unit(prefix, U, hi - 1) : -1;

  // ---- units without any chunk produce zeros (block u mod N writes them)
  if (warp < NW) {
    for (int u = c; u < U; u += (int)N) {
      if (prefix[u] != prefix[u + 1]) continue;
      const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
      const int qh0 = sparse ? hu : hu * p.group;
      for (int i = tid; i < GE * D; i += NW * 32)
        store_out_elem(p.out, p.out_dtype, ((size_t)b * p.num_q_heads + qh0) * D + i, 0.f);
    }
  }
  if (lo >= hi) return;

  if (warp == NW) {
    // ================================================================ producer
    // Lane l resolves chunk base + l of each batch of 32. The table entries of
    // batch k + 1 are loaded before lane 0 issues the copies of batch k, so
    // their latency overlaps the streaming of batch k.
    const uint64_t pol = policy_evict_first();
    const int cpp = ps / kChunk;
    // raw lookup of chunk x: unit, chunk-in-unit, and the loaded table entries
    struct Raw {
      int u, k, sp, phys;
    };
    auto fetch = [&](int x, Raw& r) {   // issues the global loads
      r.u = -1; r.k = 0; r.sp = 0; r.phys = -1;
      if (x >= hi) return;
      r.u = find_unit(prefix, U, x);
      r.k = x - prefix[r.u];
      const int b = r.u / p.units_per_b, hu = r.u - b * p.units_per_b;
      if (!sparse) {
        const int lp = (r.k * kChunk) / ps;
        if (r.k * kChunk < lens[b]) r.phys = p.block_table[(size_t)b * p.max_pages + lp];
      } else {
        r.sp = p.sel_pages[(size_t)(b * p.num_q_heads + hu) * p.sel_stride + r.k / cpp];
      }
    };
    auto resolve = [&](const Raw& r, ChunkInfo& ci) {   // consumes the loads
      ci.k = nullptr; ci.v = nullptr; ci.sz = nullptr; ci.u = r.u < 0 ? 0 : r.u;
      ci.nvalid = 0; ci.valid = 0; ci.pad = 0;
      if (r.u < 0) return;
      const int b = r.u / p.units_per_b, hu = r.u - b * p.units_per_b;
      const int L = lens[b];
      int t0, g, phys = r.phys;
      if (!sparse) {
        t0 = r.k * kChunk;
        g = hu;
      } else {
        g = hu / p.group;
        if (r.sp < 0 || (long long)r.sp * ps >= L) {
          flag_status(p.dev_status, PKV_DEV_BAD_SELECTED);
          return;
        }
        t0 = r.sp * ps + (r.k % cpp) * kChunk;
        if (t0 < L) phys = p.block_table[(size_t)b * p.max_pages + t0 / ps];
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
      if constexpr (KV == KV_I8T) ci.sz = p.kv_sz + row0 * 4;
      if constexpr (KV == KV_I8G)
        ci.sz = p.kv_sz + (((size_t)phys * p.num_kv_heads + g) * (ps / 64) + off / 64) * 4;
      ci.nvalid = nv;
      ci.valid = 1;
    };
    int n = 0;
    bool abort = false;
    Raw cur;
    fetch(lo + lane, cur);
    for (int base = lo; base < hi && !abort; base += 32) {
      ChunkInfo ci;
      resolve(cur, ci);
      info[lane] = ci;
      __syncwarp();
      const int cnt = min(32, hi - base);
      if (lane == 0) {
        for (int i = 0; i < cnt; ++i, ++n) {
          const int s = n % S, use = n / S;
          if (use > 0 && !mbar_wait_bounded(smem_u32(&empty[s]), (use - 1) & 1)) {
            flag_status(p.dev_status, PKV_DEV_TIMEOUT);
            abort = true;
            break;
          }
          const ChunkInfo e = info[i];
          hdr[s] = make_int4(e.u, e.nvalid, e.valid, 0);
          const uint32_t fb = smem_u32(&full[s]);
          if (e.valid) {
            uint8_t* st = ring + (size_t)s * STAGE;
            mbar_arrive_expect_tx(fb, 2 * KB + SZB);
            bulk_g2s(smem_u32(st), e.k, KB, fb, pol);
            bulk_g2s(smem_u32(st + KB), e.v, KB, fb, pol);
            if constexpr (SZB > 0) bulk_g2s(smem_u32(st + 2 * KB), e.sz, SZB, fb, pol);
          } else {
            mbar_arrive(fb);
          }
        }
      }
      abort = __shfl_sync(0xffffffffu, abort ? 1 : 0, 0) != 0;
      n = __shfl_sync(0xffffffffu, n, 0);
      __syncwarp();
      // the next batch's table loads overlap the streaming of the stages just issued
      fetch(base + 32 + lane, cur);
    }
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
    if (lane < GE) {
      float* rec = rec_of(u);
      rec[lane] = -INFINITY;
      rec[GE + lane] = 0.f;
    }
  };

  auto flush = [&](int u) {
    float* rec = rec_of(u);
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

  auto start_unit = [&](int u) {
    const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
    const int qh0 = sparse ? hu : hu * p.group;
    float part[GE];
#pragma unroll
    for (int h = 0; h < GE; ++h) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < QD2; ++e) {
        const size_t idx = ((size_t)b * p.num_q_heads + qh0 + h) * D;
        const float x0 = load_q_elem(p.q, p.q_dtype, idx + qk_dim<D, KV>(j, 2 * e)) * p.q_scale;
        const float x1 = load_q_elem(p.q, p.q_dtype, idx + qk_dim<D, KV>(j, 2 * e + 1)) * p.q_scale;
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
  for (int n = warp; lo + n < hi; n += NW) {
    const int s = n % S, use = n / S;
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
        if constexpr (KV == KV_I8T) sv = fmaf(sz[t * 4 + 0], sv, sz[t * 4 + 1] * qsum);
        if constexpr (KV == KV_I8G) sv = fmaf(ks, sv, kz * qsum);
        sc[it] = t < nvalid ? sv : -INFINITY;
      }
      // ---- online softmax update (per head, in the score layout)
      float cmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 8));
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 16));
      const float m_new = fmaxf(m_h, cmax);
      const float alpha = exp2f(m_h - m_new);
      float pw[4];
      float psum = 0.f, pz = 0.f;
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const float pe = exp2f(sc[it] - m_new);
        psum += pe;
        if constexpr (KV == KV_I8T) {
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
      if constexpr (KV == KV_I8T) {
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
    if (u_cur >= 0) {
      flush(u_cur);
      next_unit = u_cur + 1;
    }
    for (int v = next_unit; v <= ub; ++v) write_empty(v);
  }

  // ---- in-block merge. Every unit this block touched gets one block record
  // from its 4 warp records; a unit that lies entirely inside this block is
  // final here and goes to the output. Units shared with other blocks are
  // finished by attn_combine_kernel, the next launch on the stream.
  constexpr int RS = rec_floats(GE, D), HDR = rec_hdr(GE);
  constexpr int OUTS = GE * D;                           // outputs of one unit
  constexpr int OPT = (OUTS + NW * 32 - 1) / (NW * 32);  // outputs per thread
  named_bar_sync(1, NW * 32);
  for (int u = ua; u <= ub; ++u) {
    if (prefix[u] == prefix[u + 1]) continue;
    const bool alone = cta_of(prefix[u], W, N) == cta_of(prefix[u + 1] - 1, W, N);
    const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
    const int qh0 = sparse ? hu : hu * p.group;
    const float* wr = p.ws_wrec + (size_t)(c + u) * NW * RS;
    float* cr = p.ws_crec + (size_t)(c + u) * RS;
#pragma unroll
    for (int k = 0; k < OPT; ++k) {
      const int o = tid + k * NW * 32;
      if (o < OUTS) {
        const int h = o / D, ch = o - h * D;
        float mw[NW], lw[NW], aw[NW];
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          mw[w] = wr[w * RS + h];
          lw[w] = wr[w * RS + GE + h];
          aw[w] = wr[w * RS + HDR + o];
        }
        float M = mw[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) M = fmaxf(M, mw[w]);
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            const float f = mw[w] == -INFINITY ? 0.f : exp2f(mw[w] - M);
            L = fmaf(f, lw[w], L);
            A = f > 0.f ? fmaf(f, aw[w], A) : A;
          }
        }
        if (alone) {
          store_out_elem(p.out, p.out_dtype, ((size_t)b * p.num_q_heads + qh0) * D + o,
                         L > 0.f ? A / L : 0.f);
        } else {
          if (ch == 0) {
            cr[h] = M;
            cr[GE + h] = L;
          }
          cr[HDR + o] = A;
        }
      }
    }
  }
}

// Cross-block merge of the units that several blocks shared: one block per
// unit, over the block records [m[G], l[G], acc[G][D]] of the covering blocks,
//   M = max m_c,  out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c
// (the log2-domain partial states of the attention kernel).
template <int D, int GE>
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnParams p) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int RS = rec_floats(GE, D), HDR = rec_hdr(GE);
  constexpr int OUTS = GE * D, OPT = (OUTS + 127) / 128;
  __shared__ float ML[2 * 8];
  const int u = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int U = p.num_units;
  const long long W = __ldcg(p.ws_prefix + U), N = p.num_ctas;
  const int s0 = __ldcg(p.ws_prefix + u), s1 = __ldcg(p.ws_prefix + u + 1);
  if (s0 == s1) return;
  const int c_first = cta_of(s0, W, N), c_last = cta_of(s1 - 1, W, N);
  if (c_first == c_last) return;                 // finished by the attention kernel
  const bool sparse = p.sel_pages != nullptr;
  const int b = u / p.units_per_b, hu = u - b * p.units_per_b;
  const int qh0 = sparse ? hu : hu * p.group;
  // pass A: per head (warp h % 4), M and L over the covering blocks
  for (int h = warp; h < GE; h += 4) {
    float Mx = -INFINITY, Lx = 0.f;
    for (int cc = c_first + lane; cc <= c_last; cc += 32) {
      if (cta_lo(cc, W, N) >= cta_lo(cc + 1, W, N)) continue;
      const float* rr = p.ws_crec + (size_t)(cc + u) * RS;
      const float mc = __ldcg(rr + h), lc = __ldcg(rr + GE + h);
      if (mc == -INFINITY) continue;
      const float Mn = fmaxf(Mx, mc);
      Lx = Lx * exp2f(Mx - Mn) + lc * exp2f(mc - Mn);
      Mx = Mn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float Mo = __shfl_xor_sync(0xffffffffu, Mx, off);
      const float Lo = __shfl_xor_sync(0xffffffffu, Lx, off);
      const float Mn = fmaxf(Mx, Mo);
      Lx = (Mn == -INFINITY) ? 0.f : Lx * exp2f(Mx - Mn) + Lo * exp2f(Mo - Mn);
      Mx = Mn;
    }
    if (lane == 0) {
      ML[h] = Mx;
      ML[GE + h] = Lx;
    }
  }
  __syncthreads();
  // pass B: this thread's outputs, covering blocks in batches of 8
#pragma unroll
  for (int k = 0; k < OPT; ++k) {
    const int o = tid + k * 128;
    if (o >= OUTS) break;
    const int h = o / D;
    const float M = ML[h], L = ML[GE + h];
    float A = 0.f;
    if (M != -INFINITY) {
      for (int cc0 = c_first; cc0 <= c_last; cc0 += 8) {
        float mc[8], ac[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int cc = cc0 + i;
          const bool ok = cc <= c_last && cta_lo(cc, W, N) < cta_lo(cc + 1, W, N);
          const float* rr = p.ws_crec + (size_t)((ok ? cc : c_first) + u) * RS;
          mc[i] = ok ? __ldcg(rr + h) : -INFINITY;
          ac[i] = __ldcg(rr + HDR + o);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float f = mc[i] == -INFINITY ? 0.f : exp2f(mc[i] - M);
          A = f > 0.f ? fmaf(f, ac[i], A) : A;
        }
      }
    }
    store_out_elem(p.out, p.out_dtype, ((size_t)b * p.num_q_heads + qh0) * D + o,
                   L > 0.f ? A / L : 0.f);
  }
}

}  // namespace pkv
