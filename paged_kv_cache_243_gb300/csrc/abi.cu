// C-ABI entry points: argument checks, workspace sizing and kernel dispatch.
// Every host-detectable error is returned before anything is launched.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <unordered_map>

#include "attention_kernel.cuh"
#include "pkv_internal.h"

namespace pkv {

int attn_stage_bytes(int kv_kind, int D, bool swz) {
  const int row = kv_kind == KV_U4T ? D / 2 : ((kv_kind == KV_I8T || kv_kind == KV_I8G) ? D : 2 * D);
  const int kb = kChunk * row;
  const int szb = (kv_kind == KV_I8T || kv_kind == KV_U4T) ? kChunk * 16 : (kv_kind == KV_I8G ? 16 : 0);
  return stage_bytes_of(kb, szb, swz);
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// log2(page_size) for a power of two, else -1 (the append kernels then divide)
int page_shift(int ps) {
  if (ps <= 0 || (ps & (ps - 1)) != 0) return -1;
  int s = 0;
  while ((1 << s) < ps) ++s;
  return s;
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return std::atoi(v);
}

// Tuning knobs (environment variables; results never depend on them). They
// are read from the environment once, at the first call that plans an
// attention launch, and again only on pkv_tuning_reload(), so a call does no
// getenv and a concurrent setenv cannot race with one.
struct Tuning {
  int mma = 1;            // PKV_ATTN_MMA=0: CUDA-core consumers for query-head groups
  int ring_kb = 64;       // PKV_ATTN_RING_KB: ring size per block
  int stages = 0;         // PKV_ATTN_STAGES: explicit stage count (rounded to a multiple of 4)
  int ctas_per_sm = 0;    // PKV_ATTN_CTAS_PER_SM: cap on resident blocks per SM
  int comb_rg = 0;        // PKV_ATTN_COMB_RG: record groups of the combine (1, 2, 4 or 8)
  int mma_g1 = 0;         // PKV_ATTN_MMA_G1: tensor-core consumers for single query heads on
                          // fp16/bf16 caches: 0 never, 1 at head_dim 64, 2 at every head_dim
  int self_fed = 1;       // PKV_ATTN_SELF: self-fed tensor-core blocks 0 never, 1 where the
                          // plan below picks them, 2 for every early-start call
};

std::mutex g_tuning_mu;
Tuning g_tuning;
bool g_tuning_read = false;

void read_tuning_locked() {
  Tuning t;
  t.mma = env_int("PKV_ATTN_MMA", 1);
  t.ring_kb = env_int("PKV_ATTN_RING_KB", 64);
  t.stages = env_int("PKV_ATTN_STAGES", 0);
  t.ctas_per_sm = env_int("PKV_ATTN_CTAS_PER_SM", 0);
  t.comb_rg = env_int("PKV_ATTN_COMB_RG", 0);
  t.mma_g1 = env_int("PKV_ATTN_MMA_G1", 0);
  t.self_fed = env_int("PKV_ATTN_SELF", 1);
  g_tuning = t;
  g_tuning_read = true;
}

Tuning tuning() {
  std::lock_guard<std::mutex> lk(g_tuning_mu);
  if (!g_tuning_read) read_tuning_locked();
  return g_tuning;
}

struct DeviceInfo {
  int sms = 0;
  int max_smem_optin = 0;
};

pkv_status device_info(DeviceInfo& di) {
  static std::mutex mu;
  static std::unordered_map<int, DeviceInfo> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) {
    di = it->second;
    return PKV_OK;
  }
  DeviceInfo d;
  if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  cache[dev] = d;
  di = d;
  return PKV_OK;
}

// Make sure a kernel may launch with `smem` bytes of dynamic shared memory and
// return how many of its blocks fit on one SM at that size. The shared-memory
// limit is one value per (device, kernel); it is only ever raised, so a launch
// prepared earlier with a larger size stays valid after a smaller request.
// Occupancy is kept per (device, kernel, size).
pkv_status prepare_kernel(const void* fn, int threads, size_t smem, int& blocks_per_sm) {
  static std::mutex mu;
  struct Key {
    int dev;
    const void* fn;
    size_t smem;
    bool operator==(const Key& o) const { return dev == o.dev && fn == o.fn && smem == o.smem; }
  };
  struct Hash {
    size_t operator()(const Key& k) const {
      return std::hash<const void*>()(k.fn) ^ (k.smem * 1315423911u) ^ (size_t)k.dev;
    }
  };
  static std::unordered_map<Key, int, Hash> occupancy;   // (dev, fn, smem) -> blocks per SM
  static std::unordered_map<Key, size_t, Hash> limit;    // (dev, fn, 0) -> smem limit set
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  const Key fkey{dev, fn, 0};
  auto lim = limit.find(fkey);
  if (lim == limit.end() || lim->second < smem) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return PKV_ERR_CUDA;
    limit[fkey] = smem;
  }
  const Key key{dev, fn, smem};
  auto it = occupancy.find(key);
  if (it != occupancy.end()) {
    blocks_per_sm = it->second;
    return PKV_OK;
  }
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (nb < 1) return PKV_ERR_UNSUPPORTED;
  occupancy[key] = nb;
  blocks_per_sm = nb;
  return PKV_OK;
}

pkv_status check_cache(const pkv_cache* c, bool need_pools) {
  if (!c) return PKV_ERR_INVALID_ARG;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0 || c->page_size <= 0) return PKV_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (c->page_size % kChunk != 0) return PKV_ERR_UNSUPPORTED;
  if (c->kv_dtype == PKV_F16 || c->kv_dtype == PKV_BF16) {
    if (c->quant != PKV_QUANT_NONE) return PKV_ERR_INVALID_ARG;
  } else if (c->kv_dtype == PKV_I8) {
    if (c->quant != PKV_QUANT_PER_TOKEN && c->quant != PKV_QUANT_PER_GROUP64) return PKV_ERR_INVALID_ARG;
    if (c->quant == PKV_QUANT_PER_GROUP64 && c->page_size % 64 != 0) return PKV_ERR_UNSUPPORTED;
    if (need_pools && (!c->kv_sz || !aligned16(c->kv_sz))) return PKV_ERR_INVALID_ARG;
  } else if (c->kv_dtype == PKV_U4) {
    if (c->quant == PKV_QUANT_PER_GROUP64) return PKV_ERR_UNSUPPORTED;
    if (c->quant != PKV_QUANT_PER_TOKEN) return PKV_ERR_INVALID_ARG;
    if (need_pools && (!c->kv_sz || !aligned16(c->kv_sz))) return PKV_ERR_INVALID_ARG;
  } else {
    return PKV_ERR_INVALID_ARG;
  }
  if (need_pools) {
    if (!c->k_pages || !c->v_pages || !aligned16(c->k_pages) || !aligned16(c->v_pages))
      return PKV_ERR_INVALID_ARG;
  }
  if (c->page_meta && !aligned16(c->page_meta)) return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

int kv_kind(const pkv_cache* c) {
  if (c->kv_dtype == PKV_F16) return KV_F16;
  if (c->kv_dtype == PKV_BF16) return KV_BF16;
  if (c->kv_dtype == PKV_U4) return KV_U4T;
  return c->quant == PKV_QUANT_PER_TOKEN ? KV_I8T : KV_I8G;
}

const void* attn_combine(int D, int ge) {
#define PKV_COMB(d, g) \
  if (D == d && ge == g) return reinterpret_cast<const void*>(&attn_combine_kernel<d, g>);
  PKV_COMB(64, 1) PKV_COMB(64, 2) PKV_COMB(64, 4) PKV_COMB(64, 8)
  PKV_COMB(128, 1) PKV_COMB(128, 2) PKV_COMB(128, 4) PKV_COMB(128, 8)
#undef PKV_COMB
  return nullptr;
}

const void* attn_kernel(int kind, int D, int ge, bool mma, bool self_fed = false) {
  switch (kind) {
    case KV_F16: return attn_kernel_f16(D, ge, mma, self_fed);
    case KV_BF16: return attn_kernel_bf16(D, ge, mma, self_fed);
    case KV_I8T: return attn_kernel_i8t(D, ge, mma, self_fed);
    case KV_U4T: return attn_kernel_u4t(D, ge, mma, self_fed);
    default: return attn_kernel_i8g(D, ge, mma, self_fed);
  }
}

// The tensor-core variant serves query-head groups (G >= 2) when q has the
// dtype of the products' operands: fp16 for fp16, INT8 and 4-bit caches
// (codes enter as exact fp16 integers), bf16 for bf16 caches. Single query
// heads (MHA, or per-head page lists) on fp16/bf16 caches, whose rows enter
// the products as stored, may take it too (PKV_ATTN_MMA_G1); by default they
// stay on the CUDA-core consumer, which measured faster for them (MHA at
// head_dim 64: 91 against 94 us; at 128: 22.4 against 28.5 us per call).
bool use_mma(int kind, int ge, int D, int q_dtype, const Tuning& tn) {
  if (tn.mma == 0) return false;
  if (ge < 2) {
    if (kind != KV_F16 && kind != KV_BF16) return false;
    if (tn.mma_g1 == 0 || (tn.mma_g1 == 1 && D != 64)) return false;
  }
  return kind == KV_BF16 ? q_dtype == PKV_BF16 : q_dtype == PKV_F16;
}

struct AttnPlan {
  const void* fn = nullptr;
  bool mma = false;
  bool swz = false;   // swizzled tensor-copy staging (tensor-core INT8 at head_dim 128)
  int ge = 1, units = 0, stages = 0, ctas = 0;
  size_t smem = 0;
  size_t off_wrec = 0, ws_bytes = 0;
  int comb_groups = 1;
  bool self_fed = false;   // the tensor-core kernel without a producer warp
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Tensor maps of the K and V pools for the swizzled tensor-core INT8 variant:
// each pool as a 2-D tensor [num_pages * Hkv * page_size rows][128 bytes],
// copied in boxes of 16 rows x 128 bytes with the 128-byte swizzle. The
// encoding is plain data (no context state); it is made once per (pool
// address, rows) through the driver's cuTensorMapEncodeTiled, looked up with
// cudaGetDriverEntryPointByVersion so the library does not link the driver.
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

pkv_status pool_tensor_map(const void* base, uint64_t rows, CUtensorMap& out) {
  static std::mutex mu;
  static std::map<std::pair<const void*, uint64_t>, CUtensorMap> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_pair(base, rows);
  auto it = cache.find(key);
  if (it != cache.end()) {
    out = it->second;
    return PKV_OK;
  }
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return PKV_ERR_CUDA;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, (cuuint32_t)kChunk};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PKV_ERR_CUDA;
  if (cache.size() >= 256) cache.clear();
  cache[key] = m;
  out = m;
  return PKV_OK;
}

// q_dtype < 0: size the workspace for whichever kernel variant a call may use.
// sparse: 0 dense, 1 page lists per query head, 2 one page list per kv head shared by its group.
// max_chunks > 0: an upper bound on the call's chunk count (from the block table's
// width or the page lists' stride), used to give small calls fewer blocks.
pkv_status plan_attention(const pkv_cache* c, int32_t batch, int32_t num_q_heads, int sparse,
                          int32_t num_splits, int q_dtype, AttnPlan& pl, long long max_chunks = 0,
                          int fresh_rows = -1) {
  pkv_status st = check_cache(c, false);
  if (st != PKV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || num_q_heads % c->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (num_splits < 0) return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / c->num_kv_heads;
  pl.ge = sparse == 1 ? 1 : G;
  if (pl.ge != 1 && pl.ge != 2 && pl.ge != 4 && pl.ge != 8) return PKV_ERR_UNSUPPORTED;
  pl.units = batch * (sparse == 1 ? num_q_heads : c->num_kv_heads);
  const int kind = kv_kind(c);
  const Tuning tn = tuning();
  pl.mma = q_dtype >= 0 && use_mma(kind, pl.ge, c->head_dim, q_dtype, tn);
  pl.fn = attn_kernel(kind, c->head_dim, pl.ge, pl.mma);
  if (!pl.fn) return PKV_ERR_UNSUPPORTED;
  DeviceInfo di;
  st = device_info(di);
  if (st != PKV_OK) return st;
  // The stage count is a multiple of the consumer-warp count: consumer warp w
  // takes chunks w, w + 4, ..., so every stage is then read by one warp only and
  // that warp waits on the stage's phases strictly in order. (A parity wait on a
  // phase two ahead of the barrier's current phase would pass at once.)
  pl.swz = pl.mma && (kind == KV_I8T || kind == KV_I8G) && c->head_dim == 128;
  const int stage = attn_stage_bytes(kind, c->head_dim, pl.swz);
  const size_t slack = pl.swz ? kSwizzleAlign : 0;   // the ring is moved to a 1024-byte boundary
  const int ring_kb = tn.ring_kb > 0 ? tn.ring_kb : 64;
  int stages = (ring_kb * 1024) / stage;
  // The tensor-core consumers need three stages per warp in flight: with the
  // 8 KB stages of 16-bit caches that is a 96 KB ring and two blocks per SM
  // (GQA bf16, B = 16, L = 32768: 316 against 383 us per call with 8 stages)
  if (q_dtype >= 0 && pl.mma && stages < 3 * kConsumerWarps) stages = 3 * kConsumerWarps;
  const int forced = tn.stages;
  if (forced > 0) stages = forced;
  stages = stages / kConsumerWarps * kConsumerWarps;
  stages = stages < kConsumerWarps ? kConsumerWarps : (stages > 32 ? 32 : stages);
  // after the stream the ring holds the four consumer warps' states of the
  // block's last unit, merged there into one record
  const size_t staging = (size_t)kConsumerWarps * rec_floats(pl.ge, c->head_dim) * 4;
  int min_stages = (int)((staging + stage - 1) / stage);
  min_stages = (min_stages + kConsumerWarps - 1) / kConsumerWarps * kConsumerWarps;
  if (min_stages < kConsumerWarps) min_stages = kConsumerWarps;
  if (min_stages > 32) return PKV_ERR_UNSUPPORTED;
  if (stages < min_stages) stages = min_stages;
  size_t smem = attn_smem_bytes(stage, stages, pl.ge, pl.units, batch) + slack;
  while (smem > (size_t)di.max_smem_optin && stages > min_stages) {
    stages -= kConsumerWarps;
    smem = attn_smem_bytes(stage, stages, pl.ge, pl.units, batch) + slack;
  }
  if (smem > (size_t)di.max_smem_optin) return PKV_ERR_UNSUPPORTED;
  if (stages % kConsumerWarps != 0) return PKV_ERR_UNSUPPORTED;
  pl.stages = stages;
  pl.smem = smem;
  if (num_splits > 0) {
    pl.ctas = num_splits;
  } else {
    // CUDA-core consumers on 8 KB chunks (fp16/bf16, d = 128) keep the HBM
    // busy with 2 blocks (16 stages) per SM, and fewer blocks mean fewer
    // partial records and a shorter merge (W2: 28.8 -> 28.0 us, dense 32K
    // -2.6 %). Smaller chunks and the tensor-core consumers want 3.
    auto blocks_per_sm = [&](const void* fn, bool mma, int& nb) {
      pkv_status r = prepare_kernel(fn, kAttnThreads, smem, nb);
      int cap = tn.ctas_per_sm;
      if (cap <= 0 && !mma && stage >= 8192) cap = 2;
      if (cap <= 0 && mma) cap = 3;   // three per SM whichever tensor-core form runs
      if (cap > 0 && cap < nb) nb = cap;
      return r;
    };
    int nb = 0;
    st = blocks_per_sm(pl.fn, pl.mma, nb);
    if (st != PKV_OK) return st;
    // sizing for any q dtype: the tensor-core variant, where a call may use
    // it, may fit more blocks
    const int mma_q = kind == KV_BF16 ? PKV_BF16 : PKV_F16;
    if (q_dtype < 0 && (pl.ge >= 2 || use_mma(kind, pl.ge, c->head_dim, mma_q, tn))) {
      int nb2 = 0;
      const void* f2 = attn_kernel(kind, c->head_dim, pl.ge, true);
      if (f2 && blocks_per_sm(f2, true, nb2) == PKV_OK && nb2 > nb) nb = nb2;
    }
    pl.ctas = di.sms * nb;
    // A small call (fewer than 4 chunks per resident block) runs on fewer,
    // fuller blocks, at least one per SM: blocks of one chunk each leave the
    // combine dozens of partial states per unit (GQA 32/8, B = 1, L = 1024:
    // 10.3 -> 7.6 us per call).
    if (max_chunks > 0) {
      const long long want = (max_chunks + 3) / 4;
      const long long n = want > di.sms ? want : di.sms;
      if (n < pl.ctas) pl.ctas = (int)n;
    }
  }
  // Combine layout: about blocks per unit + 4 records per unit (one from each
  // block that ends inside the unit, four from the one that moves on); more
  // record groups per block fold them in fewer rounds (loads of the next
  // round overlap the current fold), fewer give more outputs per block
  // (fewer blocks). Cost ~ waves * (3 + rounds).
  {
    const int outs = pl.ge * c->head_dim;
    const long long units = pl.units > 0 ? pl.units : 1;
    const long long rbar = (pl.ctas + units - 1) / units + kConsumerWarps;
    const long long slots = (long long)di.sms * 2;   // combine blocks resident at once
    long long best = -1;
    for (int rg = 1; rg <= 8; rg *= 2) {
      const int ob = kCombineThreads / rg;
      if (ob > outs && rg < 8) continue;
      const long long blocks = units * ((outs + ob - 1) / ob);
      const long long waves = (blocks + slots - 1) / slots;
      const long long rounds = (rbar + rg * 8 - 1) / (rg * 8);
      // (a grid of at most one block per SM releases the next launch sooner:
      // W4 attention-only chain 34.2 -> 33.35 us with 128 blocks instead of
      // 256, but its slower merge delays the next append: W4 step 37.8 ->
      // 38.2 us, so the cost does not favour it)
      const long long cost = waves * (3 + rounds);
      if (best < 0 || cost < best) {
        best = cost;
        pl.comb_groups = rg;
      }
    }
    // Self-fed tensor-core blocks (no producer warp; three per SM, three warps
    // per SM sub-partition) leave room for one 128-thread combine block per SM.
    // The attention kernel then releases the combine at entry, its blocks wait
    // beside the attention blocks, and where its grid has at most one block per
    // SM (record group 1) the next call of a chain, released once every combine
    // block is resident, streams while this call merges. The self-fed
    // consumers stream ~4 % slower (their copies sit on their own path: W3
    // 94.9 against 91.5 us when forced), which that overlap repays only on
    // short calls: early-start calls with no fresh rows (an attention call
    // after another; after an append, the next append waits for the merge
    // anyway: W4's decode step 41.2 against 33.0 us when forced) of at most
    // ~128 chunks per block (W4's attention chain: 24.6 against 29.6 us), and
    // dense: sparse calls resolve two table levels per chunk in the consumer
    // warps (W6's sparse attention chain 28.6 against 27.3 us, with a combine
    // of two outputs per thread so that its grid fitted beside them).
    const void* self_fn = pl.mma && tn.self_fed ? attn_kernel(kind, c->head_dim, pl.ge, true, true) : nullptr;
    const int ob1 = kCombineThreads;
    const bool fits = units * ((outs + ob1 - 1) / ob1) <= di.sms;
    // 16 .. 128 chunks per block: below, a call is mostly its prologue and the
    // self-fed lookups and copies do not pay (GQA bf16, B = 1, L = 4096: 13.6
    // against 15.3 us per call); above, the slower stream outweighs the overlap
    const bool short_call = max_chunks >= 16LL * pl.ctas && max_chunks <= 128LL * pl.ctas;
    if (self_fn && num_splits == 0 && pl.units < (1 << 24) &&
        ((tn.self_fed == 1 && sparse == 0 && fresh_rows == 0 && fits && short_call) ||
         (tn.self_fed == 2 && fresh_rows >= 0))) {
      pl.self_fed = true;
      pl.fn = self_fn;
      if (fits) {
        // one record group while it folds a unit's records in at most 5 rounds
        // (W4, 28 blocks per unit: 24.7 against 25.1 us with 2 groups); past
        // that, the most groups whose grid still fits one block per SM (GQA
        // INT8, B = 1, L = 16384, 57 blocks per unit: 14.6 us with 4 groups,
        // 17.7 with 1, 16.6 with the producer-warp kernel)
        pl.comb_groups = 1;
        if ((rbar + 7) / 8 > 5) {
          for (int rg = 2; rg <= 8; rg *= 2) {
            const int ob = kCombineThreads / rg;
            if (units * ((outs + ob - 1) / ob) <= di.sms) pl.comb_groups = rg;
          }
        }
      }
    }
    const int forced_rg = tn.comb_rg;
    if (forced_rg == 1 || forced_rg == 2 || forced_rg == 4 || forced_rg == 8) pl.comb_groups = forced_rg;
  }
  const size_t rs = (size_t)rec_floats(pl.ge, c->head_dim);
  const size_t cslots = (size_t)(pl.ctas + pl.units);
  size_t off = align256((size_t)(pl.units + 1) * 4);        // unit chunk prefix
  pl.off_wrec = off;
  off = align256(off + cslots * kConsumerWarps * rs * 4);    // warp records
  pl.ws_bytes = off;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_OUT_OF_PAGES: return "out of pages";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_WORKSPACE: return "workspace too small or misaligned";
  }
  return "unknown status";
}

int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

void pkv_tuning_reload(void) {
  std::lock_guard<std::mutex> lk(g_tuning_mu);
  read_tuning_locked();
}

size_t pkv_attention_workspace_bytes(const pkv_cache* cache, int32_t batch, int32_t num_q_heads,
                                     int32_t sparse, int32_t num_splits) {
  AttnPlan pl;
  if (sparse < 0 || sparse > 2) return 0;
  if (plan_attention(cache, batch, num_q_heads, sparse, num_splits, -1, pl) != PKV_OK) return 0;
  return pl.ws_bytes;
}

}  // extern "C"

namespace pkv {
namespace {

// Both attention entry points; k_new / v_new non-NULL: fused append (dense only).
pkv_status attention_impl(const pkv_cache* cache, int32_t batch, int32_t num_q_heads, const void* q,
                          pkv_dtype q_dtype, float sm_scale, const int32_t* block_table, int32_t max_pages,
                          const int32_t* seq_lens, const int32_t* sel_pages, const int32_t* sel_count,
                          int32_t sel_stride, int32_t sel_shared, void* out, pkv_dtype out_dtype,
                          int32_t num_splits, int32_t fresh_rows, const void* k_new, const void* v_new,
                          pkv_dtype src_dtype, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                          void* stream) {
  pkv_status st = check_cache(cache, true);
  if (st != PKV_OK) return st;
  if (q_dtype != PKV_F16 && q_dtype != PKV_BF16 && q_dtype != PKV_F32) return PKV_ERR_INVALID_ARG;
  if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32) return PKV_ERR_INVALID_ARG;
  if (batch < 0 || max_pages <= 0) return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !out || !block_table || !seq_lens || !aligned16(q) || !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  const bool sparse = sel_pages != nullptr;
  if (sparse && (!sel_count || sel_stride <= 0)) return PKV_ERR_INVALID_ARG;
  if (sel_shared != 0 && sel_shared != 1) return PKV_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !(sm_scale < 1e30f)) return PKV_ERR_INVALID_ARG;
  if (fresh_rows < -1) return PKV_ERR_INVALID_ARG;
  const int mode = !sparse ? 0 : (sel_shared ? 2 : 1);
  AttnPlan pl;
  const long long units_per_b = mode == 1 ? num_q_heads : cache->num_kv_heads;
  const long long max_chunks =
      (long long)batch * units_per_b *
      (sparse ? (long long)sel_stride * (cache->page_size / kChunk)
              : ((long long)max_pages * cache->page_size + kChunk - 1) / kChunk);
  st = plan_attention(cache, batch, num_q_heads, mode, num_splits, q_dtype, pl, max_chunks, fresh_rows);
  if (st != PKV_OK) return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < pl.ws_bytes)
    return PKV_ERR_WORKSPACE;
  int nb = 0;
  st = prepare_kernel(pl.fn, attn_threads(pl.self_fed), pl.smem, nb);
  if (st != PKV_OK) return st;

  AttnParams p = {};
  if (pl.swz) {
    // tensor-copy row coordinates are 32-bit signed
    const uint64_t rows = (uint64_t)cache->num_pages * cache->num_kv_heads * cache->page_size;
    if (rows >= (1ull << 31)) return PKV_ERR_UNSUPPORTED;
    st = pool_tensor_map(cache->k_pages, rows, p.tmap_k);
    if (st == PKV_OK) st = pool_tensor_map(cache->v_pages, rows, p.tmap_v);
    if (st != PKV_OK) return st;
  }
  p.k_pages = static_cast<const uint8_t*>(cache->k_pages);
  p.v_pages = static_cast<const uint8_t*>(cache->v_pages);
  p.kv_sz = cache->kv_sz;
  p.q = q;
  p.out = out;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.sel_pages = sel_pages;
  p.sel_count = sel_count;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws_prefix = reinterpret_cast<int32_t*>(ws);
  p.ws_wrec = reinterpret_cast<float*>(ws + pl.off_wrec);
  p.dev_status = dev_status;
  p.num_pages = cache->num_pages;
  p.page_size = cache->page_size;
  p.num_kv_heads = cache->num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.group = num_q_heads / cache->num_kv_heads;
  p.batch = batch;
  p.max_pages = max_pages;
  p.sel_stride = sparse ? sel_stride : 0;
  p.units_per_b = mode == 1 ? num_q_heads : cache->num_kv_heads;
  p.unit_is_q = mode == 1;
  p.num_units = pl.units;
  p.num_ctas = pl.ctas;
  p.stages = pl.stages;
  p.q_dtype = q_dtype;
  p.out_dtype = out_dtype;
  p.q_scale = sm_scale * 1.4426950408889634f;
  p.fresh_rows = fresh_rows;
  p.comb_groups = pl.comb_groups;
  p.k_new = k_new;
  p.v_new = v_new;
  p.src_dtype = src_dtype;
  void* args[] = {&p};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_pdl(pl.fn, dim3(pl.ctas), dim3(attn_threads(pl.self_fed)), pl.smem, cs, args);
  if (e == cudaSuccess) {
    const void* comb = attn_combine(cache->head_dim, pl.ge);
    const int outs = pl.ge * cache->head_dim;
    const int ob = kCombineThreads / p.comb_groups;
    e = launch_pdl(comb, dim3(pl.units, (outs + ob - 1) / ob), dim3(kCombineThreads), 0, cs, args);
  }
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_paged_decode_attention(const pkv_cache* cache, int32_t batch, int32_t num_q_heads,
                                      const void* q, pkv_dtype q_dtype, float sm_scale,
                                      const int32_t* block_table, int32_t max_pages,
                                      const int32_t* seq_lens, const int32_t* sel_pages,
                                      const int32_t* sel_count, int32_t sel_stride,
                                      int32_t sel_shared, void* out, pkv_dtype out_dtype,
                                      int32_t num_splits, int32_t fresh_rows, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return attention_impl(cache, batch, num_q_heads, q, q_dtype, sm_scale, block_table, max_pages, seq_lens,
                        sel_pages, sel_count, sel_stride, sel_shared, out, out_dtype, num_splits, fresh_rows,
                        nullptr, nullptr, PKV_F16, workspace, workspace_bytes, dev_status, stream);
}

pkv_status pkv_append_decode_attention(const pkv_cache* cache, int32_t batch, int32_t num_q_heads,
                                       const void* k_new, const void* v_new, pkv_dtype src_dtype,
                                       const void* q, pkv_dtype q_dtype, float sm_scale,
                                       const int32_t* block_table, int32_t max_pages,
                                       const int32_t* seq_lens, void* out, pkv_dtype out_dtype,
                                       int32_t num_splits, int32_t fresh_rows, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status, void* stream) {
  pkv_status st = check_cache(cache, true);
  if (st != PKV_OK) return st;
  if (src_dtype != PKV_F16 && src_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (batch > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID_ARG;
  if (cache->quant == PKV_QUANT_PER_GROUP64 || cache->page_meta) {
    // Two launches: the kv_append of each sequence's token at seq_lens[b] - 1
    // (per-group INT8 re-quantises the open group; page boxes are refreshed),
    // then the attention, which starts under the append: that kernel writes
    // only the new rows (and their open group and boxes), and it waits for
    // all earlier work before it touches anything.
    if (batch < 0 || max_pages <= 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!block_table || !seq_lens) return PKV_ERR_INVALID_ARG;
    if (cache->quant == PKV_QUANT_PER_GROUP64 &&
        (!cache->tail || !aligned16(cache->tail) || cache->tail_rows < batch))
      return PKV_ERR_INVALID_ARG;
    if (batch > 65535 || cache->num_kv_heads > 32767) return PKV_ERR_UNSUPPORTED;
    // the attention call's own argument checks and plan come first, so that a
    // call refused for them changes nothing
    AttnPlan pl;
    const long long max_chunks = (long long)batch * cache->num_kv_heads *
                                 (((long long)max_pages * cache->page_size + kChunk - 1) / kChunk);
    st = plan_attention(cache, batch, num_q_heads, 0, num_splits, q_dtype, pl, max_chunks);
    if (st != PKV_OK) return st;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < pl.ws_bytes)
      return PKV_ERR_WORKSPACE;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_F16 && q_dtype != PKV_BF16 && q_dtype != PKV_F32) return PKV_ERR_INVALID_ARG;
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32) return PKV_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || !(sm_scale < 1e30f) || fresh_rows < -1) return PKV_ERR_INVALID_ARG;
    AppendParams ap = {};
    ap.k_pages = cache->k_pages;
    ap.v_pages = cache->v_pages;
    ap.kv_sz = cache->kv_sz;
    ap.tail = cache->tail;
    ap.page_meta = cache->page_meta;
    ap.k_new = k_new;
    ap.v_new = v_new;
    ap.block_table = block_table;
    ap.positions = seq_lens;
    ap.pos_bias = -1;
    ap.new_lens = nullptr;
    ap.dev_status = dev_status;
    ap.num_pages = cache->num_pages;
    ap.page_size = cache->page_size;
    ap.num_kv_heads = cache->num_kv_heads;
    ap.head_dim = cache->head_dim;
    ap.kv_dtype = cache->kv_dtype;
    ap.quant = cache->quant;
    ap.src_dtype = src_dtype;
    ap.batch = batch;
    ap.t_new = 1;
    ap.max_pages = max_pages;
    ap.ps_shift = page_shift(cache->page_size);
    st = launch_append(ap, static_cast<cudaStream_t>(stream));
    if (st != PKV_OK) return st;
    return attention_impl(cache, batch, num_q_heads, q, q_dtype, sm_scale, block_table, max_pages, seq_lens,
                          nullptr, nullptr, 0, 0, out, out_dtype, num_splits, 1, nullptr, nullptr, PKV_F16,
                          workspace, workspace_bytes, dev_status, stream);
  }
  if ((cache->kv_dtype == PKV_F16 || cache->kv_dtype == PKV_BF16) && src_dtype != cache->kv_dtype)
    return PKV_ERR_UNSUPPORTED;
  return attention_impl(cache, batch, num_q_heads, q, q_dtype, sm_scale, block_table, max_pages, seq_lens,
                        nullptr, nullptr, 0, 0, out, out_dtype, num_splits, fresh_rows, k_new, v_new,
                        src_dtype, workspace, workspace_bytes, dev_status, stream);
}

pkv_status pkv_kv_append(const pkv_cache* cache, int32_t batch, int32_t t_new, const void* k_new,
                         const void* v_new, pkv_dtype src_dtype, const int32_t* block_table,
                         int32_t max_pages, const int32_t* positions, const int32_t* new_lens,
                         int32_t* dev_status, void* stream) {
  pkv_status st = check_cache(cache, true);
  if (st != PKV_OK) return st;
  if (src_dtype != PKV_F16 && src_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (batch < 0 || t_new < 0 || max_pages <= 0) return PKV_ERR_INVALID_ARG;
  if (batch == 0 || t_new == 0) return PKV_OK;
  if (!k_new || !v_new || !block_table || !positions || !aligned16(k_new) || !aligned16(v_new))
    return PKV_ERR_INVALID_ARG;
  if (cache->quant == PKV_QUANT_PER_GROUP64 &&
      (!cache->tail || !aligned16(cache->tail) || cache->tail_rows < batch))
    return PKV_ERR_INVALID_ARG;
  if ((long long)t_new > (long long)max_pages * cache->page_size) return PKV_ERR_INVALID_ARG;
  if (batch > 65535 || cache->num_kv_heads > 32767) return PKV_ERR_UNSUPPORTED;   // grid y / z limits
  AppendParams p = {};
  p.k_pages = cache->k_pages;
  p.v_pages = cache->v_pages;
  p.kv_sz = cache->kv_sz;
  p.tail = cache->tail;
  p.page_meta = cache->page_meta;
  p.k_new = k_new;
  p.v_new = v_new;
  p.block_table = block_table;
  p.positions = positions;
  p.new_lens = new_lens;
  p.dev_status = dev_status;
  p.num_pages = cache->num_pages;
  p.page_size = cache->page_size;
  p.num_kv_heads = cache->num_kv_heads;
  p.head_dim = cache->head_dim;
  p.kv_dtype = cache->kv_dtype;
  p.quant = cache->quant;
  p.src_dtype = src_dtype;
  p.batch = batch;
  p.t_new = t_new;
  p.max_pages = max_pages;
  p.pos_bias = 0;
  p.ps_shift = page_shift(cache->page_size);
  return launch_append(p, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_page_score_topk(const pkv_cache* cache, int32_t batch, int32_t num_q_heads,
                               const void* q, pkv_dtype q_dtype, const int32_t* block_table,
                               int32_t max_pages, const int32_t* seq_lens, int32_t top_k,
                               int32_t group_mode, int32_t early_start, int32_t* sel_pages,
                               int32_t* sel_count, float* scores_out, int32_t* dev_status, void* stream) {
  pkv_status st = check_cache(cache, false);
  if (st != PKV_OK) return st;
  if (!cache->page_meta) return PKV_ERR_INVALID_ARG;
  if (q_dtype != PKV_F16 && q_dtype != PKV_BF16 && q_dtype != PKV_F32) return PKV_ERR_INVALID_ARG;
  if (batch < 0 || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (max_pages <= 0 || top_k < 1) return PKV_ERR_INVALID_ARG;
  if (group_mode < PKV_SELECT_PER_HEAD || group_mode > PKV_SELECT_GROUP_MAX) return PKV_ERR_INVALID_ARG;
  if (early_start != 0 && early_start != 1) return PKV_ERR_INVALID_ARG;
  if (max_pages > 16384) return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!q || !block_table || !seq_lens || !sel_pages || !sel_count) return PKV_ERR_INVALID_ARG;
  TopkParams p = {};
  p.page_meta = cache->page_meta;
  p.q = q;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.sel_pages = sel_pages;
  p.sel_count = sel_count;
  p.scores_out = scores_out;
  p.dev_status = dev_status;
  p.num_pages = cache->num_pages;
  p.page_size = cache->page_size;
  p.num_kv_heads = cache->num_kv_heads;
  p.head_dim = cache->head_dim;
  p.num_q_heads = num_q_heads;
  p.group = num_q_heads / cache->num_kv_heads;
  p.batch = batch;
  p.max_pages = max_pages;
  p.top_k = top_k;
  p.q_dtype = q_dtype;
  p.group_mode = group_mode;
  p.early = early_start;
  return launch_topk(p, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
