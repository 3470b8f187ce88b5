// page_score_topk: score every page of a sequence against each query head with
// the direction-aware bounding box, then keep the top-K pages [TinyServe page,
// section 2.1 (metadata, score) and section 3.1 phases 1-2]. A row that selects
// is a query head, or a kv head whose G query heads' scores are summed or
// maxed (one shared page list per group; a reading, the pages score one query).
//
// One cluster of 8 blocks per (sequence, KBH consecutive kv heads), whose
// boxes are one contiguous read per page (details at the kernel). Phase 1:
// block r scores the r-th eighth of the pages for every query head of those
// kv heads into its shared memory. Phase 2: block r gathers row r's scores
// from the cluster through distributed shared memory and runs an exact radix
// select (four 8-bit passes over an order-preserving integer image of the
// scores) for the K-th largest score T; pages above T are kept, and of those
// equal to T the lowest page indices fill the remaining places. Phase 3: a
// block-wide scan in page order writes the kept pages in ascending order.
#include <cooperative_groups.h>

#include "pkv_internal.h"

namespace cg = cooperative_groups;

namespace pkv {

namespace {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCluster = 8;        // blocks per (sequence, kv-head block)

// Larger float -> larger unsigned key; NaN is treated as -inf.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) f = -INFINITY;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive scan of one int per thread over the block; returns the block total.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int pre = 0, tot = 0;
  for (int w = 0; w < kTopkWarps; ++w) {
    const int t = warp_tot[w];
    if (w < warp) pre += t;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return pre + x - v;
}

// Exact top-K of one row's scores keys[0, P) (float bits) into
// sel[0, top_k), ascending page order; ties at the K-th score keep the lower
// page indices. Whole block; keys is overwritten.
__device__ void select_row(uint32_t* keys, int P, int K, int top_k, int32_t* sel, int32_t* count,
                           int* hist, int* warp_tot, int& sel_digit, int& sel_remaining) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) *count = K;
  for (int i = K + tid; i < top_k; i += kTopkThreads) sel[i] = -1;
  if (K == 0) return;
  if (K == P) {
    for (int i = tid; i < P; i += kTopkThreads) sel[i] = i;
    return;
  }
  // keys, and the bits where they all agree (AND == OR): leading bytes that
  // every key shares need no radix pass (scores of one sign and binade share
  // their top byte, and a pass over it would serialise P atomics on one bin)
  uint32_t kand = 0xffffffffu, kor = 0u;
  for (int i = tid; i < P; i += kTopkThreads) {
    const uint32_t k = order_key(__uint_as_float(keys[i]));
    keys[i] = k;
    kand &= k;
    kor |= k;
  }
  kand = __reduce_and_sync(0xffffffffu, kand);
  kor = __reduce_or_sync(0xffffffffu, kor);
  if (lane == 0) {
    warp_tot[warp] = (int)kand;
    hist[warp] = (int)kor;
  }
  __syncthreads();
  kand = 0xffffffffu;
  kor = 0u;
  for (int w = 0; w < kTopkWarps; ++w) {
    kand &= (uint32_t)warp_tot[w];
    kor |= (uint32_t)hist[w];
  }
  __syncthreads();
  const uint32_t diff = kand ^ kor;
  // first pass: the byte holding the highest differing bit (all keys equal:
  // no pass, T is that key and the K lowest pages are kept)
  const int top_shift = diff == 0u ? -8 : (31 - __clz(diff)) / 8 * 8;

  // ---- radix select of the K-th largest key
  uint32_t mask = top_shift >= 24 ? 0u : (0xffffffffu << (top_shift + 8));
  uint32_t prefix = kand & mask;
  int remaining = K;
  for (int shift = top_shift; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < P; i += kTopkThreads) {
      const uint32_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds digits 255 - 8l .. 248 - 8l (descending); a scan over the
      // lanes finds the digit where the running count first reaches `remaining`
      int c8[8], lsum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c8[i] = hist[255 - 8 * lane - i];
        lsum += c8[i];
      }
      int incl = lsum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const int excl = incl - lsum;
      const unsigned mine = __ballot_sync(0xffffffffu, excl < remaining && remaining <= incl);
      if (lane == __ffs(mine) - 1) {
        int cum = excl, dgt = 248 - 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum + c8[i] >= remaining) {
            dgt = 255 - 8 * lane - i;
            break;
          }
          cum += c8[i];
        }
        sel_digit = dgt;
        sel_remaining = remaining - cum;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sel_digit << shift;
    mask |= 255u << shift;
    remaining = sel_remaining;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const int need_eq = remaining;  // how many pages scoring exactly T are kept

  // ---- ordered compaction
  const int per = (P + kTopkThreads - 1) / kTopkThreads;
  const int i0 = min(P, tid * per), i1 = min(P, i0 + per);
  int n_eq = 0;
  for (int i = i0; i < i1; ++i) n_eq += keys[i] == T;
  int tot;
  int eq_before = block_excl_scan(n_eq, warp_tot, tot);
  int n_sel = 0;
  {
    int e = eq_before;
    for (int i = i0; i < i1; ++i) {
      const uint32_t k = keys[i];
      if (k > T) ++n_sel;
      else if (k == T) { if (e < need_eq) ++n_sel; ++e; }
    }
  }
  int out = block_excl_scan(n_sel, warp_tot, tot);
  {
    int e = eq_before;
    for (int i = i0; i < i1; ++i) {
      const uint32_t k = keys[i];
      bool take = false;
      if (k > T) take = true;
      else if (k == T) { take = e < need_eq; ++e; }
      if (take) sel[out++] = i;
    }
  }
  __syncthreads();   // keys is reused by the block's next row
}

// One cluster per (sequence, KBH consecutive kv heads). The boxes of those kv
// heads sit next to each other in a page's metadata ([page][kv head][2][D]), so
// each page is one contiguous read of KBH * 2 * D floats (2 KB at the chosen
// KBH): random 2 KB reads stream near the HBM peak where 512 B reads (one
// head's box) reach about half. The cluster scores its G * KBH query heads and
// selects NR rows: the query heads (per-head lists) or the kv heads (a group's
// sum or max). Block r of the cluster scores the r-th eighth of the pages, a
// warp per page (UNROLL pages in flight), into its shared memory; then block r
// gathers row r's scores (rows r, r + 8, ... when NR > 8) from the cluster
// through distributed shared memory and selects them.
// SUM: rows are group sums (the lane partials of the G heads are added and
// reduced once); otherwise per-head rows or group maxima.
template <int D, int KBH, bool SUM>
__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads, 2)
    score_topk_kernel(const TopkParams p) {
  constexpr int CS = kTopkCluster;
  constexpr int NV = KBH * 2 * D / 128;    // float4 box loads per lane per page
  constexpr int UNROLL = 16 / NV;          // pages in flight per warp (8 KB)
  extern __shared__ __align__(16) uint32_t tk_smem[];
  __shared__ int hist[256];
  __shared__ int warp_tot[kTopkWarps];
  __shared__ int sel_digit, sel_remaining;
  // early start: the caller promises that the preceding work writes nothing
  // read here, so the boxes are read and scored at once; every block waits
  // before its first global write (below), and so before it completes
  if (!p.early) {
    pdl_wait();
    pdl_launch_dependents();
  }

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const bool grouped = p.group_mode != PKV_SELECT_PER_HEAD;
  constexpr bool sum_rows = SUM;
  const int G = p.group;
  const int NQ = KBH * G;                           // query heads scored
  const int NR = grouped ? KBH : NQ;                // rows selected
  const int cpb = p.num_kv_heads / KBH;             // clusters per sequence
  const int cl = blockIdx.x / CS;
  const int b = cl / cpb;
  const int g0 = (cl - b * cpb) * KBH;              // first kv head
  const int h0 = g0 * G;                            // first query head
  const int rows_per_b = grouped ? p.num_kv_heads : p.num_q_heads;
  const int row0 = grouped ? g0 : h0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ps = p.page_size;
  int L = p.seq_lens[b];
  if (L < 0) L = 0;
  int P = (L + ps - 1) / ps;
  if (P > p.max_pages) P = p.max_pages;
  const int K = min(p.top_k, P);
  // shared memory: keys [max_pages], own [NR][span], qsm [NQ][D], each
  // rounded to 4 floats so that qsm takes float4 loads
  const int span = ((p.max_pages + CS - 1) / CS + 3) / 4 * 4;
  uint32_t* keys = tk_smem;
  float* own = reinterpret_cast<float*>(tk_smem + (p.max_pages + 3) / 4 * 4);
  float* qsm = own + (size_t)NR * span;

  for (int i = tid; i < NQ * D; i += kTopkThreads)
    qsm[i] = load_q_elem(p.q, p.q_dtype, ((size_t)b * p.num_q_heads + h0) * D + i);
  const int pg0 = (int)((long long)P * rank / CS);
  const int pg1 = (int)((long long)P * (rank + 1) / CS);
  for (int pg = pg0 + tid; pg < pg1; pg += kTopkThreads)
    keys[pg] = (uint32_t)p.block_table[(size_t)b * p.max_pages + pg];
  __syncthreads();

  // lane l's channels: 4 (l % 16) .. + 3 of the min (l < 16) or max box (d = 64;
  // float4 i is kv head i), or 4 l .. + 3 of both (d = 128; float4 2k is kv
  // head k's min, 2k + 1 its max)
  const int ch = D == 64 ? 4 * (lane & 15) : 4 * lane;
  const bool is_max = D == 64 && lane >= 16;
  for (int base = pg0 + warp * UNROLL; base < pg1; base += kTopkWarps * UNROLL) {
    float4 v[UNROLL][NV];
    bool ok[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int pg = base + k;
      const int ph = pg < pg1 ? (int)keys[pg] : -1;   // staged table entry
      ok[k] = ph >= 0 && ph < p.num_pages;
      const float4* box = reinterpret_cast<const float4*>(
          p.page_meta + ((size_t)(ok[k] ? ph : 0) * p.num_kv_heads + g0) * 2 * D);
#pragma unroll
      for (int i = 0; i < NV; ++i) v[k][i] = ok[k] ? __ldg(box + i * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int kk = 0; kk < KBH; ++kk) {
      float rowv[UNROLL];   // grouped: the kv head's row, over its G heads
      for (int j = 0; j < G; ++j) {
        const float4 q4 = *reinterpret_cast<const float4*>(qsm + (kk * G + j) * D + ch);
        float sc[UNROLL];
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
          float4 lo4, hi4;
          if constexpr (D == 64) {
            lo4 = v[k][0];
#pragma unroll
            for (int i = 1; i < NV; ++i) if (i == kk) lo4 = v[k][i];
            hi4 = lo4;
          } else {
            lo4 = v[k][0];
            hi4 = v[k][1];
#pragma unroll
            for (int i = 1; i < NV / 2; ++i)
              if (i == kk) {
                lo4 = v[k][2 * i];
                hi4 = v[k][2 * i + 1];
              }
          }
          float a = 0.f;
          if constexpr (D == 64) {
            // this lane holds one bound: the max for q_i >= 0, the min for q_i < 0
            auto pick = [&](float qc) { return is_max ? qc >= 0.f : qc < 0.f; };
            a = pick(q4.x) ? q4.x * lo4.x : 0.f;
            a = pick(q4.y) ? fmaf(q4.y, lo4.y, a) : a;
            a = pick(q4.z) ? fmaf(q4.z, lo4.z, a) : a;
            a = pick(q4.w) ? fmaf(q4.w, lo4.w, a) : a;
          } else {
            a = q4.x * (q4.x >= 0.f ? hi4.x : lo4.x);
            a = fmaf(q4.y, q4.y >= 0.f ? hi4.y : lo4.y, a);
            a = fmaf(q4.z, q4.z >= 0.f ? hi4.z : lo4.z, a);
            a = fmaf(q4.w, q4.w >= 0.f ? hi4.w : lo4.w, a);
          }
          sc[k] = a;
        }
        if constexpr (sum_rows) {   // a group's sum: add the lane partials, reduce once below
#pragma unroll
          for (int k = 0; k < UNROLL; ++k) rowv[k] = j == 0 ? sc[k] : rowv[k] + sc[k];
          continue;
        }
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) sc[k] += __shfl_xor_sync(0xffffffffu, sc[k], off);
        }
        if (!grouped) {
          if (lane == 0) {
            const int r = kk * G + j;
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
              const int pg = base + k;
              if (pg < pg1) own[r * span + (pg - pg0)] = ok[k] ? sc[k] : -INFINITY;
            }
          }
        } else {   // a group's max
#pragma unroll
          for (int k = 0; k < UNROLL; ++k) rowv[k] = j == 0 ? sc[k] : fmaxf(rowv[k], sc[k]);
        }
      }
      if constexpr (sum_rows) {
#pragma unroll
        for (int k = 0; k < UNROLL; ++k)
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) rowv[k] += __shfl_xor_sync(0xffffffffu, rowv[k], off);
      }
      if (grouped && lane == 0) {
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
          const int pg = base + k;
          if (pg < pg1) own[kk * span + (pg - pg0)] = ok[k] ? rowv[k] : -INFINITY;
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < UNROLL; ++k)
        if (base + k < pg1 && !ok[k]) flag_status(p.dev_status, PKV_DEV_BAD_PAGE);
    }
  }
  __syncthreads();
  if (p.early) {
    pdl_wait();
    pdl_launch_dependents();
  }
  if (p.scores_out) {
    for (int r = 0; r < NR; ++r) {
      float* so = p.scores_out + ((size_t)b * rows_per_b + row0 + r) * p.max_pages;
      for (int pg = pg0 + tid; pg < pg1; pg += kTopkThreads) so[pg] = own[r * span + (pg - pg0)];
      if (rank == 0)
        for (int pg = P + tid; pg < p.max_pages; pg += kTopkThreads) so[pg] = -INFINITY;
    }
  }
  // every score of the cluster's rows now sits in its blocks' shared memory,
  // which stays resident (and unchanged) until the last cluster.sync
  cluster.sync();
  for (int r = rank; r < NR; r += CS) {
    __syncthreads();   // the previous row's select is done with keys
    // page i sits in block rr = floor(((i + 1) CS - 1) / P) of the cluster, at
    // i - floor(P rr / CS); a thread's remote loads (up to GR pages) are all
    // issued before the first is stored
    constexpr int GR = 4;
    for (int i0 = 0; i0 < P; i0 += GR * kTopkThreads) {
      uint32_t v[GR];
#pragma unroll
      for (int j = 0; j < GR; ++j) {
        const int i = i0 + j * kTopkThreads + tid;
        v[j] = 0u;
        if (i < P) {
          const int rr = (int)(((long long)(i + 1) * CS - 1) / P);
          const int a0 = (int)((long long)P * rr / CS);
          v[j] = __float_as_uint(cluster.map_shared_rank(own, rr)[(size_t)r * span + (i - a0)]);
        }
      }
#pragma unroll
      for (int j = 0; j < GR; ++j) {
        const int i = i0 + j * kTopkThreads + tid;
        if (i < P) keys[i] = v[j];
      }
    }
    __syncthreads();
    const size_t bh = (size_t)b * rows_per_b + row0 + r;
    select_row(keys, P, K, p.top_k, p.sel_pages + bh * p.top_k, p.sel_count + bh, hist, warp_tot, sel_digit,
               sel_remaining);
  }
  cluster.sync();
}

}  // namespace

// kv heads per cluster: 2 KB of boxes per page (4 heads at d = 64, 2 at 128),
// dividing the kv heads; a cluster with per-head rows selects KBH * G rows.
int topk_kv_heads_per_cluster(int D, int num_kv_heads) {
  int kbh = D == 64 ? 4 : 2;
  while (kbh > 1 && num_kv_heads % kbh != 0) kbh /= 2;
  return kbh;
}

pkv_status launch_topk(const TopkParams& p, cudaStream_t st) {
  const bool grouped = p.group_mode != PKV_SELECT_PER_HEAD;
  const int kbh = topk_kv_heads_per_cluster(p.head_dim, p.num_kv_heads);
  const int nq = kbh * p.group, nr = grouped ? kbh : nq;
  const int span = ((p.max_pages + kTopkCluster - 1) / kTopkCluster + 3) / 4 * 4;
  const size_t smem = ((size_t)(p.max_pages + 3) / 4 * 4 + (size_t)nr * span + (size_t)nq * p.head_dim) * 4;
  const bool sum = p.group_mode == PKV_SELECT_GROUP_SUM;
  const void* fn = nullptr;
#define PKV_TOPK(d, k)                                                                   \
  if (p.head_dim == d && kbh == k)                                                       \
    fn = sum ? reinterpret_cast<const void*>(&score_topk_kernel<d, k, true>)             \
             : reinterpret_cast<const void*>(&score_topk_kernel<d, k, false>);
  PKV_TOPK(64, 4) PKV_TOPK(64, 2) PKV_TOPK(64, 1) PKV_TOPK(128, 2) PKV_TOPK(128, 1)
#undef PKV_TOPK
  if (!fn) return PKV_ERR_UNSUPPORTED;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return PKV_ERR_CUDA;
  if (smem + fa.sharedSizeBytes > (size_t)optin) return PKV_ERR_UNSUPPORTED;
  if (smem > 48 * 1024) {
    // always the device's maximum, never a per-call size, so a concurrent or
    // later launch that needs more is never left below its need
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  const unsigned grid = (unsigned)(p.batch * (p.num_kv_heads / kbh) * kTopkCluster);
  TopkParams pc = p;
  void* args[] = {&pc};
  if (launch_pdl(fn, dim3(grid), dim3(kTopkThreads), smem, st, args) != cudaSuccess) return PKV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
