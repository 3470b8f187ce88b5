// page_score_topk: score every page of a sequence against one query head with
// the direction-aware bounding box, then keep the top-K pages [TinyServe page,
// section 2.1 (metadata, score) and section 3.1 phases 1-2]. A row that selects
// is a query head, or a kv head whose G query heads' scores are summed or
// maxed (one shared page list per group; a reading, the pages score one query).
//
// One cluster of CS blocks per (sequence, row): 4 for a query head, 8 for a
// kv head's group (G heads to score per page). Phase 1:
// block r of the cluster scores the r-th quarter of the pages (a warp per
// page, lane-parallel over channels, butterfly sum) into its shared memory;
// the leader then gathers the other blocks' scores through distributed shared
// memory. Scoring is bound by the box bytes, and four blocks per row put every
// SM to work on them. Phase 2 (leader): an exact radix select (four 8-bit
// passes over an order-preserving integer image of the scores) finds the K-th
// largest score T; pages above T are kept, and of those equal to T the lowest
// page indices fill the remaining places. Phase 3: a block-wide scan in page
// order writes the kept pages in ascending order.
#include <cooperative_groups.h>

#include "pkv_internal.h"

namespace cg = cooperative_groups;

namespace pkv {

namespace {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkClusterHead = 4;    // rows of one query head
constexpr int kTopkClusterGroup = 8;   // rows of a query-head group

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

template <int D, int CS>
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(kTopkThreads, D == 64 ? 4 : 3)
    score_topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t keys[];  // [max pages of a sequence]
  __shared__ int hist[256];
  __shared__ int warp_tot[kTopkWarps];
  __shared__ int sel_digit, sel_remaining;
  __shared__ float qsm[8 * D];   // the row's query heads (<= 8)
  pdl_wait();
  pdl_launch_dependents();

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  // a row selects: a query head, or a kv head for its group (sum / max)
  const bool grouped = p.group_mode != PKV_SELECT_PER_HEAD;
  const int rows_per_b = grouped ? p.num_kv_heads : p.num_q_heads;
  const int HR = grouped ? p.group : 1;             // query heads scored per row
  const int bh = blockIdx.x / CS;                   // row index b * rows_per_b + r
  const int b = bh / rows_per_b, hr = bh - b * rows_per_b;
  const int g = grouped ? hr : hr / p.group;        // kv head whose boxes are read
  const int h0 = grouped ? hr * p.group : hr;       // first query head of the row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ps = p.page_size;
  int L = p.seq_lens[b];
  if (L < 0) L = 0;
  int P = (L + ps - 1) / ps;
  if (P > p.max_pages) P = p.max_pages;
  const int K = min(p.top_k, P);

  // ---- phase 1: scores
  constexpr int PL = D / 32;  // channels per lane
  for (int i = tid; i < HR * D; i += kTopkThreads)
    qsm[i] = load_q_elem(p.q, p.q_dtype, ((size_t)b * p.num_q_heads + h0) * D + i);
  // this block's pages [pg0, pg1) of the row
  const int pg0 = (int)((long long)P * rank / CS);
  const int pg1 = (int)((long long)P * (rank + 1) / CS);
  // The block-table entries are staged (coalesced) in the key array first;
  // each page's entry is read before its score overwrites that slot.
  for (int pg = pg0 + tid; pg < pg1; pg += kTopkThreads)
    keys[pg] = (uint32_t)p.block_table[(size_t)b * p.max_pages + pg];
  __syncthreads();
  // pages in flight per warp (box loads issued before use); a group's rows
  // keep fewer pages in flight and score every head of the group from one
  // load of each box
  constexpr bool GROUPED = CS == kTopkClusterGroup;
  constexpr int UNROLL = GROUPED ? 4 : 16;
  for (int base = pg0 + warp * UNROLL; base < pg1; base += kTopkWarps * UNROLL) {
    float part[UNROLL];
    __syncwarp();
    if constexpr (!GROUPED) {
      // one query head: each page's partial right after its box loads
      float qv[PL];
#pragma unroll
      for (int e = 0; e < PL; ++e) qv[e] = qsm[lane * PL + e];
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const int pg = base + k;
        const int ph = pg < pg1 ? (int)keys[pg] : -1;   // staged table entry
        part[k] = 0.f;
        if (ph >= 0 && ph < p.num_pages) {
          const float* mrow = p.page_meta + (((size_t)ph * p.num_kv_heads + g) * 2) * D + lane * PL;
          float mn[PL], mx[PL];
          if constexpr (PL == 4) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(mrow));
            const float4 c = __ldg(reinterpret_cast<const float4*>(mrow + D));
            mn[0] = a.x; mn[1] = a.y; mn[2] = a.z; mn[3] = a.w;
            mx[0] = c.x; mx[1] = c.y; mx[2] = c.z; mx[3] = c.w;
          } else {
            const float2 a = __ldg(reinterpret_cast<const float2*>(mrow));
            const float2 c = __ldg(reinterpret_cast<const float2*>(mrow + D));
            mn[0] = a.x; mn[1] = a.y;
            mx[0] = c.x; mx[1] = c.y;
          }
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < PL; ++e) acc = fmaf(qv[e], qv[e] >= 0.f ? mx[e] : mn[e], acc);
          part[k] = acc;
        }
      }
#pragma unroll
      for (int k = 0; k < UNROLL; ++k)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part[k] += __shfl_xor_sync(0xffffffffu, part[k], off);
    } else {
      float mn[UNROLL][PL], mx[UNROLL][PL];
  #pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const int pg = base + k;
        const int ph = pg < pg1 ? (int)keys[pg] : -1;   // staged table entry
  #pragma unroll
        for (int e = 0; e < PL; ++e) { mn[k][e] = 0.f; mx[k][e] = 0.f; }
        if (ph >= 0 && ph < p.num_pages) {
          const float* mrow = p.page_meta + (((size_t)ph * p.num_kv_heads + g) * 2) * D + lane * PL;
          if constexpr (PL == 4) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(mrow));
            const float4 c = __ldg(reinterpret_cast<const float4*>(mrow + D));
            mn[k][0] = a.x; mn[k][1] = a.y; mn[k][2] = a.z; mn[k][3] = a.w;
            mx[k][0] = c.x; mx[k][1] = c.y; mx[k][2] = c.z; mx[k][3] = c.w;
          } else {
            const float2 a = __ldg(reinterpret_cast<const float2*>(mrow));
            const float2 c = __ldg(reinterpret_cast<const float2*>(mrow + D));
            mn[k][0] = a.x; mn[k][1] = a.y;
            mx[k][0] = c.x; mx[k][1] = c.y;
          }
        }
      }
      // each query head of the row: the pages' lane partials, butterfly sums,
      // then the row's reduction (one head: itself; a group: sum or max)
      for (int j = 0; j < HR; ++j) {
        float qv[PL];
  #pragma unroll
        for (int e = 0; e < PL; ++e) qv[e] = qsm[j * D + lane * PL + e];
        float sj[UNROLL];
  #pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
          float acc = 0.f;
  #pragma unroll
          for (int e = 0; e < PL; ++e) acc = fmaf(qv[e], qv[e] >= 0.f ? mx[k][e] : mn[k][e], acc);
          sj[k] = acc;
        }
  #pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
  #pragma unroll
          for (int off = 16; off > 0; off >>= 1) sj[k] += __shfl_xor_sync(0xffffffffu, sj[k], off);
          part[k] = j == 0 ? sj[k] : (p.group_mode == PKV_SELECT_GROUP_MAX ? fmaxf(part[k], sj[k]) : part[k] + sj[k]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const int pg = base + k;
        if (pg >= pg1) break;
        float s = part[k];
        const int ph = (int)keys[pg];
        if (ph < 0 || ph >= p.num_pages) {
          flag_status(p.dev_status, PKV_DEV_BAD_PAGE);
          s = -INFINITY;
        }
        keys[pg] = __float_as_uint(s);
        if (p.scores_out) p.scores_out[(size_t)bh * p.max_pages + pg] = s;
      }
    }
  }
  if (p.scores_out && rank == 0) {
    for (int pg = P + tid; pg < p.max_pages; pg += kTopkThreads)
      p.scores_out[(size_t)bh * p.max_pages + pg] = -INFINITY;
  }
  // every score of the row now sits in the cluster's shared memory; the leader
  // copies the other blocks' parts, which stay resident until it is done
  cluster.sync();
  if (rank == 0) {
    for (int r = 1; r < CS; ++r) {
      const uint32_t* remote = cluster.map_shared_rank(keys, r);
      const int a0 = (int)((long long)P * r / CS), a1 = (int)((long long)P * (r + 1) / CS);
      for (int i = a0 + tid; i < a1; i += kTopkThreads) keys[i] = remote[i];
    }
  }
  cluster.sync();
  if (rank != 0) return;

  int32_t* sel = p.sel_pages + (size_t)bh * p.top_k;
  if (tid == 0) p.sel_count[bh] = K;
  for (int i = K + tid; i < p.top_k; i += kTopkThreads) sel[i] = -1;
  if (K == 0) return;
  if (K == P) {
    for (int i = tid; i < P; i += kTopkThreads) sel[i] = i;
    return;
  }

  for (int i = tid; i < P; i += kTopkThreads) keys[i] = order_key(__uint_as_float(keys[i]));
  __syncthreads();

  // ---- phase 2: radix select of the K-th largest key
  uint32_t prefix = 0, mask = 0;
  int remaining = K;
  for (int shift = 24; shift >= 0; shift -= 8) {
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

  // ---- phase 3: ordered compaction
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
}

}  // namespace

pkv_status launch_topk(const TopkParams& p, cudaStream_t st) {
  const size_t smem = (size_t)p.max_pages * 4;
  const bool grouped = p.group_mode != PKV_SELECT_PER_HEAD;
  const int cs = grouped ? kTopkClusterGroup : kTopkClusterHead;
  const void* fn;
  if (p.head_dim == 128)
    fn = grouped ? reinterpret_cast<const void*>(&score_topk_kernel<128, kTopkClusterGroup>)
                 : reinterpret_cast<const void*>(&score_topk_kernel<128, kTopkClusterHead>);
  else
    fn = grouped ? reinterpret_cast<const void*>(&score_topk_kernel<64, kTopkClusterGroup>)
                 : reinterpret_cast<const void*>(&score_topk_kernel<64, kTopkClusterHead>);
  if (smem > 48 * 1024) {
    // always the one maximum (16384 pages), never a per-call size, so a
    // concurrent or later launch with more pages is never left below its need
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 4) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  const int rows = p.batch * (grouped ? p.num_kv_heads : p.num_q_heads);
  const unsigned grid = (unsigned)(rows * cs);
  TopkParams pc = p;
  void* args[] = {&pc};
  if (launch_pdl(fn, dim3(grid), dim3(kTopkThreads), smem, st, args) != cudaSuccess) return PKV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
