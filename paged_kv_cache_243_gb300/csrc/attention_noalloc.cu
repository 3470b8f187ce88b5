// pkv_paged_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// pkv_paged_decode_attention needs a caller-provided workspace for the
// per-block partial softmax states. Some callers have no way to provide one:
// a host program that reserves all device memory up front and forbids any
// later cudaMalloc (a cudaMalloc can synchronise the whole device and stall a
// latency-bound serving loop), or a plugin handed only its input and output
// buffers by a framework that owns the allocator. This entry point takes its
// workspace from a fixed array in the library's own device memory instead.
//
// The array is a file-scope __device__ array of kNoallocScratchBytes. CUDA
// loads the module that holds it lazily by default: its memory is taken on a
// device by the first call made with that device current (the call that looks
// up the array's device address), or when the context is created if the
// process runs with CUDA_MODULE_LOADING=EAGER, and held until the process
// exits. All calls share the one array, so calls that can overlap on the GPU
// (different streams, or different host threads) race and must not be issued.
// The looked-up address is kept per device; after cudaDeviceReset on a device
// it is stale, so no call may follow a reset.
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;   // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device (looked up once per
// device; the host-side symbol itself is not a device address).
pkv_status scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_paged_decode_attention_noalloc(const pkv_cache* cache, int32_t batch,
                                              int32_t num_q_heads, const void* q, pkv_dtype q_dtype,
                                              float sm_scale, const int32_t* block_table,
                                              int32_t max_pages, const int32_t* seq_lens,
                                              const int32_t* sel_pages, const int32_t* sel_count,
                                              int32_t sel_stride, int32_t sel_shared, void* out,
                                              pkv_dtype out_dtype, int32_t num_splits,
                                              int32_t* dev_status, void* stream) {
  void* scratch = nullptr;
  const pkv_status st = pkv::scratch_address(&scratch);
  if (st != PKV_OK) return st;
  // The attention call checks the workspace its own plan needs against the
  // array's size and returns PKV_ERR_WORKSPACE, before launching anything, for
  // a call that needs more. The workspace needs no initial contents, so
  // nothing is cleared here.
  return pkv_paged_decode_attention(cache, batch, num_q_heads, q, q_dtype, sm_scale, block_table,
                                    max_pages, seq_lens, sel_pages, sel_count, sel_stride, sel_shared,
                                    out, out_dtype, num_splits, -1, scratch,
                                    pkv::kNoallocScratchBytes, dev_status, stream);
}

}  // extern "C"
