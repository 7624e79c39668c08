// mla_noalloc.cu -- mla_decode for callers that cannot allocate device memory.
//
// The split-KV decode writes one partial output per (request, split, query row) and merges
// them in a second kernel, so it needs scratch memory.  mla_decode takes that scratch from
// the caller.  Some callers cannot call cudaMalloc: for example a serving engine whose
// memory manager hands every free byte of the device to its KV-cache pool at start-up and
// refuses later allocations, or a plugin loaded into a host program that gives it no
// allocator.  mla_decode_noalloc serves them from a fixed buffer in this library's own
// device data (a file-scope array), which every GPU that loads the library holds until the
// process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mla.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB: the largest plan->workspace_bytes accepted
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code the array's
// name is only a host-side stand-in, never a device address, so the address is looked up
// once per device (with that device current) and remembered.
void* scratch_device_ptr() {
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" int mla_decode_noalloc(const mla_decode_plan_t* plan, const void* q, const void* kv_pages,
                                  const int32_t* page_table, const int32_t* seq_lens, int q_len, int num_heads,
                                  float scale, float kv_scale, void* out, float* lse, void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  if (plan->workspace_bytes > kScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if (plan->workspace_bytes > 0) {
    ws = scratch_device_ptr();
    if (!ws) return MLA_ERR_CUDA;
  }
  return mla_decode(plan, q, kv_pages, page_table, seq_lens, q_len, num_heads, scale, kv_scale, out, lse, ws,
                    ws ? kScratchBytes : 0, stream);
}
