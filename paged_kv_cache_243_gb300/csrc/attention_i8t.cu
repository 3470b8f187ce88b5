// Instantiations of the paged attention kernel for one KV storage kind
// (head_dim 64/128 x query heads per unit 1/2/4/8).
#include "attention_kernel.cuh"
#include "pkv_internal.h"

namespace pkv {

const void* attn_kernel_i8t(int D, int GE) {
#define PKV_CASE(d, ge) \
  if (D == d && GE == ge) return reinterpret_cast<const void*>(&paged_attention_kernel<d, ge, KV_I8T>);
  PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
  return nullptr;
}

}  // namespace pkv
