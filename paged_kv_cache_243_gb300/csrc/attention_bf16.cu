// Instantiations of the paged attention kernel for one KV storage kind:
// head_dim 64/128 x query heads per unit 1/2/4/8, CUDA-core path, and the
// tensor-core path (for these 16-bit caches also for single query heads).
#include "attention_kernel.cuh"
#include "pkv_internal.h"

namespace pkv {

const void* attn_kernel_bf16(int D, int GE, bool mma, bool self_fed) {
  if (self_fed) {   // tensor cores at head_dim 128, no producer warp
    if (!mma || D != 128) return nullptr;
    if (GE == 2) return reinterpret_cast<const void*>(&paged_attention_kernel<128, 2, KV_BF16, true, true>);
    if (GE == 4) return reinterpret_cast<const void*>(&paged_attention_kernel<128, 4, KV_BF16, true, true>);
    if (GE == 8) return reinterpret_cast<const void*>(&paged_attention_kernel<128, 8, KV_BF16, true, true>);
    return nullptr;
  }
#define PKV_CASE(d, ge, tc) \
  if (D == d && GE == ge && mma == tc) \
    return reinterpret_cast<const void*>(&paged_attention_kernel<d, ge, KV_BF16, tc>);
  PKV_CASE(64, 1, false) PKV_CASE(64, 2, false) PKV_CASE(64, 4, false) PKV_CASE(64, 8, false)
  PKV_CASE(128, 1, false) PKV_CASE(128, 2, false) PKV_CASE(128, 4, false) PKV_CASE(128, 8, false)
  PKV_CASE(64, 1, true) PKV_CASE(64, 2, true) PKV_CASE(64, 4, true) PKV_CASE(64, 8, true)
  PKV_CASE(128, 1, true) PKV_CASE(128, 2, true) PKV_CASE(128, 4, true) PKV_CASE(128, 8, true)
#undef PKV_CASE
  return nullptr;
}

}  // namespace pkv
