// Internal declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

struct AppendParams {
  void* k_pages;
  void* v_pages;
  float* kv_sz;
  float* tail;
  float* page_meta;
  const void* k_new;
  const void* v_new;
  const int32_t* block_table;
  const int32_t* positions;
  const int32_t* new_lens;
  int32_t* dev_status;
  int num_pages, page_size, num_kv_heads, head_dim;
  int kv_dtype, quant, src_dtype;
  int batch, t_new, max_pages;
  int pos_bias;   // added to positions[b] (-1: positions are the lengths after the append)
  int ps_shift;   // log2(page_size) when it is a power of two, else -1
};

struct TopkParams {
  const float* page_meta;
  const void* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t* sel_pages;
  int32_t* sel_count;
  float* scores_out;
  int32_t* dev_status;
  int num_pages, page_size, num_kv_heads, head_dim;
  int num_q_heads, group, batch, max_pages, top_k, q_dtype;
  int group_mode;  // PKV_SELECT_*: rows are query heads, or kv heads (group sum / max)
  int early;       // 1: read and score before waiting for the preceding work
};

pkv_status launch_append(const AppendParams& p, cudaStream_t st);
pkv_status launch_topk(const TopkParams& p, cudaStream_t st);

// Attention kernels, one getter per KV kind (each in its own translation unit).
// mma: the tensor-core variant (query-head groups of 2, 4 or 8); self_fed:
// its form without a producer warp (head_dim 128; NULL otherwise).
const void* attn_kernel_f16(int D, int GE, bool mma, bool self_fed);
const void* attn_kernel_bf16(int D, int GE, bool mma, bool self_fed);
const void* attn_kernel_i8t(int D, int GE, bool mma, bool self_fed);
const void* attn_kernel_i8g(int D, int GE, bool mma, bool self_fed);
const void* attn_kernel_u4t(int D, int GE, bool mma, bool self_fed);

// Bytes of one shared-memory stage (a 16-token chunk of K and V plus its INT8
// scales), by KV kind and head_dim; swz: the swizzled tensor-copy staging.
int attn_stage_bytes(int kv_kind, int D, bool swz);

}  // namespace pkv
