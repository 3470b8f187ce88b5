// Shared device helpers of the paged KV-cache kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Tokens per staged chunk: every page size is a multiple of it, so a chunk of
// one (page, kv head) is one contiguous run of 16 * head_dim elements.
constexpr int kChunk = 16;

// KV_U4T: per-token 4-bit codes, two per byte (even channel in the low nibble).
enum KvKind : int { KV_F16 = 0, KV_BF16 = 1, KV_I8T = 2, KV_I8G = 3, KV_U4T = 4 };

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float f16_lo(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// Two 16-bit values of a 32-bit word as floats (exact widening).
template <int KV>
__device__ __forceinline__ void unpack2(uint32_t w, float& a, float& b) {
  if (KV == KV_BF16) {
    a = bf16_lo(w);
    b = bf16_hi(w);
  } else {
    a = f16_lo(w);
    b = f16_hi(w);
  }
}

// Stored INT8 byte i of a word (u = code + 128, in [0, 255]) as float(u),
// exactly: u in the low mantissa byte of 2^23, minus 2^23.
__device__ __forceinline__ float u8_as_float(uint32_t w, int i) {
  return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u + (uint32_t)i)) - 8388608.0f;
}

__device__ __forceinline__ float load_q_elem(const void* q, int dtype, size_t idx) {
  if (dtype == PKV_F16) return __half2float(reinterpret_cast<const __half*>(q)[idx]);
  if (dtype == PKV_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(q)[idx]);
  return reinterpret_cast<const float*>(q)[idx];
}

__device__ __forceinline__ void store_out_elem(void* out, int dtype, size_t idx, float v) {
  if (dtype == PKV_F16)
    reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
  else if (dtype == PKV_BF16)
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(out)[idx] = v;
}

__device__ __forceinline__ void flag_status(int32_t* st, int bit) {
  if (st) atomicOr(st, bit);
}

// 4-bit codes of the four bytes of w (channels 2i in the low nibble, 2i + 1
// in the high one): lo = the low nibbles, hi = the high nibbles, one per byte.
__device__ __forceinline__ void split_nibbles(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = w & 0x0F0F0F0Fu;
  hi = (w >> 4) & 0x0F0F0F0Fu;
}

// ------------------------------------------------- packed fp32 pairs (f32x2)
// Two fp32 values in one 64-bit register pair; the .f32x2 forms of fma / add /
// sub / mul issue both lanes in one instruction (sm_100 and later).
__device__ __forceinline__ uint64_t pack2f(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2f(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float hsum2(uint64_t r) {
  float a, b;
  unpack2f(r, a, b);
  return a + b;
}

// Two 16-bit values of a 32-bit word as a packed fp32 pair (exact widening).
template <int KV>
__device__ __forceinline__ uint64_t widen2(uint32_t w) {
  float a, b;
  unpack2<KV>(w, a, b);
  return pack2f(a, b);
}

// Byte i of the low-nibble word and of the high-nibble word (split_nibbles) as
// the pair (u_2i, u_2i+1) of 4-bit codes.
__device__ __forceinline__ uint64_t u4pair(uint32_t lo, uint32_t hi, int i) {
  const float a = __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u + (uint32_t)i));
  const float b = __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u + (uint32_t)i));
  return fsub2(pack2f(a, b), pack2f(8388608.0f, 8388608.0f));
}

// Stored INT8 bytes i, i+1 of a word as the pair (u_i, u_i+1), u = code + 128.
__device__ __forceinline__ uint64_t u8pair(uint32_t w, int i) {
  const float a = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u + (uint32_t)i));
  const float b = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u + (uint32_t)i + 1));
  return fsub2(pack2f(a, b), pack2f(8388608.0f, 8388608.0f));
}

// ------------------------------------------------------------ mbarrier / TMA
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The thread may sleep in the instruction until the phase completes (or about
// 10 us pass), so a waiting warp does not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(10000u)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~2^31 cycles (about a second) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1ll << 31)) return false;
  }
  return true;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Tiled tensor copy of a 2-D box at coordinates (x, y) (x in elements of the
// innermost dimension, a multiple of 16 bytes; here always 0) into this CTA's
// shared memory, completing on an mbarrier. tmap: a CUtensorMap in kernel
// parameter (__grid_constant__), constant or global memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch. pdl_wait: wait until the preceding kernel on
// the stream has completed and its memory is visible (a no-op when this kernel
// was launched without the attribute); every kernel here calls it before its
// first global access. pdl_launch_dependents: let the next kernel start
// launching (its own pdl_wait still holds it until this grid completes).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization allowed.
inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// 2^x by the SFU's approximate exponential (PTX ex2.approx.ftz.f32: relative
// error about 2^-22, results below 2^-126 flushed to zero, 2^-inf = 0). The
// online softmax only takes it of differences x <= 0 from a running maximum.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace pkv
