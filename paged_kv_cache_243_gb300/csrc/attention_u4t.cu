// Instantiations of the paged attention kernel for per-token 4-bit caches:
// head_dim 64/128 x query heads per unit 1/2/4/8, CUDA-core consumers (the
// codes are restored to fp32 in registers; there is no tensor-core variant).
#include "attention_kernel.cuh"
#include "pkv_internal.h"

namespace pkv {

const void* attn_kernel_u4t(int D, int GE, bool mma) {
  if (mma) return nullptr;
#define PKV_CASE(d, ge) \
  if (D == d && GE == ge) return reinterpret_cast<const void*>(&paged_attention_kernel<d, ge, KV_U4T, false>);
  PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
  return nullptr;
}

}  // namespace pkv
