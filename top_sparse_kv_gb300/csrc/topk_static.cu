// skv_topk_static: the exact top-k of skv_topk for callers that cannot provide a workspace.
//
// Some callers have no way to allocate device memory at the point where they
// select: a plugin that runs inside another runtime which owns the device
// memory pool and hands it no allocator, or a serving loop that must not call
// cudaMalloc because that call can synchronise the whole device.  This entry
// point keeps the selection's scratch (histograms, tickets, per-row state,
// segment counts) in one fixed array compiled into the library instead.
//
// The array is kStaticScratchBytes (16 MiB) of device memory on every GPU
// where this library's module is loaded, held until the process exits.  The
// host cannot use the array's name as a device address, so on the first call
// on each device (that device current) the entry point asks the runtime for
// the address with cudaGetSymbolAddress and caches it; make that first call
// before any stream capture.  Every call shares the one array: the selection
// clears what must start at zero on the stream before it runs, and two calls
// whose kernels overlap on the GPU (different streams, no ordering) race on
// the array and give wrong results.
#include <mutex>

#include "skv_internal.cuh"

namespace skv {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_topk_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

skv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) return SKV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SKV_OK;
}

}  // namespace
}  // namespace skv

extern "C" skv_status skv_topk_static(const skv_problem* p, const float* scores, int32_t* idx,
                                      int32_t* dev_status, void* stream) {
  size_t unused = 0;
  const skv_status valid = skv_workspace_size(p, &unused);  // validates the problem on the host
  if (valid != SKV_OK) return valid;
  if (!scores || !idx) return SKV_ERR_INVALID_ARGUMENT;
  if (skv::topk_workspace_bytes(*p) > skv::kStaticScratchBytes) return SKV_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  const skv_status got = skv::scratch_address(&ws);
  if (got != SKV_OK) return got;
  return skv::launch_topk(*p, scores, idx, ws, dev_status, (cudaStream_t)stream);
}
