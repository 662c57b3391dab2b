// skv_topk_static: the exact top-k of skv_topk for callers that cannot provide a workspace.
//
// Some callers have no way to allocate device memory at the point where they
// select: a plugin that runs inside another runtime which owns the device
// memory pool and hands it no allocator, or a serving loop that must not call
// cudaMalloc because that call can synchronise the whole device.  This entry
// point keeps the selection's scratch (histograms, tickets, per-row state,
// segment counts, segment winners) in one fixed array compiled into the
// library instead.
//
// The array is kStaticScratchBytes (16 MiB) of device memory in every CUDA
// context where this library's module is loaded, held until the process exits
// (or the context is destroyed).  The host cannot use the array's name as a
// device address, so the entry point asks the runtime for the address with
// cudaGetSymbolAddress, in the caller's current context, and caches it together
// with that context's unique id (current_context_id).  A later call in another
// context -- a new primary context after cudaDeviceReset, or a context the caller
// pushed -- sees a different id and looks the address up again, so a cached
// address never outlives the module it points into.  The first call in each context
// does that look-up; make it before any stream capture.  Every call shares the
// one array: the selection clears what must start at zero on the stream before
// it runs, and two calls whose kernels overlap on the GPU (different streams,
// no ordering) race on the array and give wrong results.
#include <mutex>

#include "skv_internal.cuh"

namespace skv {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_topk_scratch[kStaticScratchBytes];

// One cached address per device ordinal, valid only for the context whose id it carries.
constexpr int kMaxDevices = 64;
struct CachedAddress {
  unsigned long long ctx_id = 0;
  bool valid = false;
  void* ptr = nullptr;
};
std::mutex g_scratch_mu;
CachedAddress g_cached[kMaxDevices];

skv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  CachedAddress& c = g_cached[dev];
  unsigned long long id = 0;
  if (c.valid && current_context_id(&id) && c.ctx_id == id) {
    *out = c.ptr;
    return SKV_OK;
  }
  // first call in this context (or no context bound to the thread yet): the look-up
  // binds the runtime's context if needed and resolves the symbol inside it
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) return SKV_ERR_CUDA;
  if (!current_context_id(&id)) return SKV_ERR_CUDA;
  c.ctx_id = id;
  c.valid = true;
  c.ptr = p;
  *out = p;
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
  const skv_problem r = skv::head_rows(*p);  // per query head: one row a query head
  if (skv::topk_workspace_bytes(r) > skv::kStaticScratchBytes) return SKV_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  const skv_status got = skv::scratch_address(&ws);
  if (got != SKV_OK) return got;
  return skv::launch_topk(r, scores, idx, ws, dev_status, (cudaStream_t)stream);
}
