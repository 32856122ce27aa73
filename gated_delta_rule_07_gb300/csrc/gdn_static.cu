// gdn_static.cu -- gdn_forward_static_scratch: the forward pass for callers that cannot
// allocate device memory.
//
// Some callers are not allowed to call cudaMalloc at the point where they run the layer:
// plug-ins whose host framework owns every byte of device memory, serving loops with a
// fixed memory plan that forbids allocations after start-up, and code paths where an
// allocation would synchronise the device.  This entry point needs no workspace from them:
// its scratch (the status word, the segment summaries and the incoming states) lives in the
// file-scope device array below, which every GPU that loads the library holds until the
// process exits.
//
// Limits and sharing:
//   * the scratch is kStaticScratchBytes (64 MiB).  What must fit is the workspace without the
//     optional per-chunk factor tiles (the status word and, with P > 1, the segment summaries
//     and incoming states): on the tensor-core path at K = V = 128 that is N * P * Hv <= 341
//     segment-heads of 192 KiB each.  A problem that needs more is rejected with
//     GDN_ERR_WORKSPACE before anything is enqueued; one whose full gdn_workspace_size() is
//     larger but whose minimum fits runs without the factor tiles (the kernels that compute
//     their own factors);
//   * every call on a device uses the same array, and it keeps the last call's contents;
//     the status word is cleared by each call and nothing else has to start at zero;
//   * calls whose work overlaps on the GPU (different streams, or several host threads
//     without ordering between their streams) race on the array: order them on one stream;
//   * the first call on a device looks up the array's device address (with that device
//     current) and caches it; make that first call before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_lookup_mutex;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_static_scratch on the current device (looked up once per device).
// In host code the symbol itself is only a host-side stand-in, never a device address.
gdn_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_lookup_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
        return GDN_ERR_CUDA;
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_forward_static_scratch(const gdn_problem* p, const void* q, const void* k,
                                      const void* v, const float* g, const float* beta,
                                      const float* h0, const int32_t* cu_seqlens, void* out,
                                      float* h_final, cudaStream_t stream) {
  const gdn_status st = gdn_check_problem(p);
  if (st != GDN_OK) return st;
  const size_t need = gdn::workspace_min_bytes(p);  // the factor records are optional
  if (need > kStaticScratchBytes) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const gdn_status ss = scratch_for_current_device(&scratch);
  if (ss != GDN_OK) return ss;
  return gdn_forward(p, q, k, v, g, beta, h0, cu_seqlens, out, h_final, scratch,
                     kStaticScratchBytes, stream);
}

}  // extern "C"
