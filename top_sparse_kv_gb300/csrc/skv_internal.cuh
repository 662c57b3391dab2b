// Internal helpers shared by the sm_103a kernels of libskv (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "skv.h"

namespace skv {

// ------------------------------------------------------------------------------------
// launch bookkeeping (host)
// ------------------------------------------------------------------------------------

void count_launch(int n = 1);
int num_sms();  // SMs of the current device (cached per device)

#define SKV_LAUNCH_CHECK()                                  \
  do {                                                      \
    cudaError_t e_ = cudaGetLastError();                    \
    if (e_ != cudaSuccess) return SKV_ERR_CUDA;             \
    ::skv::count_launch();                                  \
  } while (0)

// ------------------------------------------------------------------------------------
// problem geometry shared by host and device
// ------------------------------------------------------------------------------------

struct Regions {
  int L, s_end, l_start;
};

__host__ __device__ __forceinline__ Regions regions_of(int L, int n_sink, int n_local) {
  Regions r;
  r.L = L;
  r.s_end = L < n_sink ? L : n_sink;
  int ls = L - n_local;
  r.l_start = ls > r.s_end ? ls : r.s_end;
  return r;
}

// history length of request b, clamped to [0, max_len]; flags out-of-range lengths
__device__ __forceinline__ int load_len(const int32_t* seq_lens, int b, int max_len, int32_t* status) {
  int L = seq_lens[b];
  if (L < 0 || L > max_len) {
    if (status) atomicOr(status, SKV_DEV_BAD_LENGTH);
    L = L < 0 ? 0 : max_len;
  }
  return L;
}

__device__ __forceinline__ void flag(int32_t* status, int bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------------------------------------------
// element loads: 16-byte vectors of bf16 or fp32 widened to fp32
// ------------------------------------------------------------------------------------

template <typename T>
struct Vec;

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 u;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "r"(addr));
  return u;
}

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;  // elements per 16 bytes
  __device__ __forceinline__ static void widen(uint4 u, float* out) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static void load(const void* p, float* out) {
    widen(*reinterpret_cast<const uint4*>(p), out);
  }
  __device__ __forceinline__ static void load_shared(uint32_t addr, float* out) { widen(lds128(addr), out); }
};

template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void widen(uint4 u, float* out) {
    out[0] = __uint_as_float(u.x);
    out[1] = __uint_as_float(u.y);
    out[2] = __uint_as_float(u.z);
    out[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static void load(const void* p, float* out) {
    widen(*reinterpret_cast<const uint4*>(p), out);
  }
  __device__ __forceinline__ static void load_shared(uint32_t addr, float* out) { widen(lds128(addr), out); }
};

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ float from_float<float>(float x) {
  return x;
}

// ------------------------------------------------------------------------------------
// order-preserving 32-bit keys of fp32 scores (larger score -> larger key)
//   -0.0 is folded onto +0.0; every NaN maps to 0, below -inf.
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA engine) wrappers, inline PTX
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// named barrier over `count` threads (ids 1..15; 0 is __syncthreads)
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~`limit_cycles` SM clocks, returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_cycles = 4000000000LL) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit_cycles) return false;
  }
  return true;
}

// Bounded wait shared by the threads of one CTA: returns false at once when
// *abort is set, and sets it (and the status bit) when this wait gives up.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              int32_t* status, long long limit_cycles = 4000000000LL) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > limit_cycles) {
      *abort = 1;
      if (status) atomicOr(status, SKV_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// 1-D bulk copy global -> shared through the TMA engine; completion is
// signalled as transaction bytes on `bar`.  dst/src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 eviction policies for cache-hinted accesses: a stream read once goes first, data
// read again soon (by the next kernel of the step) goes last.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy for the source lines
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// fp32 global store with an L2 cache policy
__device__ __forceinline__ void st_f32_hint(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

// Ampere-style 16-byte async copy (used for random-row gathers, host rows included).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// Thread-block clusters.  A kernel launched without a cluster dimension runs as clusters
// of one CTA, so these also hold there.  cluster_sync() is the hardware barrier over every
// thread of the cluster, with release / acquire ordering: shared-memory writes before it
// are visible to all the cluster's CTAs after it.  dsmem_addr() maps a local shared
// address to the same offset in the shared memory of the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch.  A kernel started with launch_dependent() may be
// scheduled while the kernel before it in the stream is still running; it calls
// pdl_wait() before its first access to global memory, which returns once that
// kernel has completed and its writes are visible, so only the launch and the CTA
// placement overlap.  pdl_release() lets the next kernel be scheduled early.
// Both are no-ops for an ordinary launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)na;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ------------------------------------------------------------------------------------
// host-side launchers (defined in the kernel files)

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }  // workspace piece boundaries
// ------------------------------------------------------------------------------------

struct PoolView {
  const void* gpu_k;
  const void* gpu_v;
  long long n_gpu;
  const void* host_k;
  const void* host_v;
  long long n_host;
  const int32_t* table;
  int stride;
  int hdiv;      // rows of the kernel per pool head: the pool head of row head h is h / hdiv (1, or G per query head)
  int per_head;  // 1: one table row per (request, pool head); a GPU block then holds one head's rows
};

// The slot-table row of (request b, pool head ph) among `heads` pool heads, and the first
// row of GPU block e for that head (a shared table: blocks of every head; one table row
// a head: blocks of one head).
__device__ __forceinline__ const int32_t* table_row(const PoolView& p, int b, int ph, int heads) {
  return p.table + ((size_t)b * (p.per_head ? heads : 1) + (p.per_head ? ph : 0)) * p.stride;
}
__device__ __forceinline__ size_t gpu_block_row(const PoolView& p, long long e, int ph, int heads, int bs) {
  return (p.per_head ? (size_t)e : (size_t)e * heads + ph) * bs;
}

// The per-query-head reading (SKV_AGG_HEAD) selects and attends one row per query head:
// the problem with n_kv_heads = n_q_heads (a group of one), whose pool rows are those of
// KV head h / G (PoolView::hdiv = G).  For the other readings, the problem itself.
skv_problem head_rows(const skv_problem& p);

// Block selection's attended list (OasisKV notes, §3.2 "compressed key summaries"): the
// sink and local windows rounded outward to whole 16-token blocks, the candidate blocks
// between them, and the list of a (request, KV head): sink blocks, chosen blocks
// (ascending), local blocks, 16 slots a block; slot j holds token 16 blk + j % 16 of the
// (j / 16)-th listed block, or -1 past the history or the list.
constexpr int kBlockTokens = 16;

struct BlockRegions {
  int nb, s_blk, l_blk;  // blocks holding a token; first candidate block; first local block
};

__device__ __forceinline__ BlockRegions block_regions(int L, int ns, int nl) {
  BlockRegions r;
  r.nb = (L + kBlockTokens - 1) / kBlockTokens;
  const int sb = (ns + kBlockTokens - 1) / kBlockTokens;
  r.s_blk = sb < r.nb ? sb : r.nb;
  if (nl <= 0) {
    r.l_blk = r.nb;
  } else {
    const int lb = (L - nl > 0 ? L - nl : 0) / kBlockTokens;
    r.l_blk = lb > r.s_blk ? lb : r.s_blk;
  }
  return r;
}

// Token in slot j of the attended list, given the row's chosen blocks (K of them
// reserved, -1 past the count); a chosen block outside the candidates flags
// SKV_DEV_BAD_INDEX (once per block) and leaves its slots empty.
__device__ __forceinline__ int block_list_token(const int32_t* chosen, int K, const BlockRegions& rg, int L, int j,
                                                int32_t* status) {
  const int n_cand = rg.l_blk - rg.s_blk;
  const int ksel = K < n_cand ? K : n_cand;
  const int count = rg.s_blk + ksel + (rg.nb - rg.l_blk);
  const int i = j / kBlockTokens, off = j % kBlockTokens;
  int blk = -1;
  if (i < rg.s_blk) {
    blk = i;
  } else if (i < rg.s_blk + ksel) {
    blk = chosen[i - rg.s_blk];
    if (blk < rg.s_blk || blk >= rg.l_blk) {
      if (off == 0) flag(status, SKV_DEV_BAD_INDEX);
      blk = -1;
    }
  } else if (i < count) {
    blk = rg.l_blk + (i - rg.s_blk - ksel);
  }
  const int t = blk * kBlockTokens + off;
  return blk >= 0 && t < L ? t : -1;
}

// The attention's block-list mode: list slots resolved from the chosen blocks directly
// (the attended list is written as it is resolved), instead of read from an index list.
struct BlockListView {
  const int32_t* chosen;  // [B * H, K] chosen blocks, ascending, -1 past the count
  int K;
  int ns, nl;             // the problem's sink and local windows (rounded to blocks here)
  int32_t* att;           // [B * H, n_att]: the attended list, written by the attention
};

// Threshold prefetch of host rows (ECHO-OSDI26 wiki, core methods 3 and 5): while the
// indexer scores, the rows of keys that score above the predicted k-th score move from
// the pinned host pool to a GPU staging area; after the exact selection the gather takes
// staged rows from there and reads every other host row as usual (guaranteed recall).
// The prediction is an EMA over steps of each row's k-th score.
struct PrefetchView {
  float* tau;                // [rows] predicted k-th score (NaN: no prediction yet)
  uint32_t* epoch;           // [1] steps completed; rows staged in a step carry tag epoch + 1
  unsigned long long* map;   // [rows * max_len]: (tag << 32) | staging slot of a staged position
  unsigned char* staging;    // [rows, cap, row bytes]
  uint32_t* count;           // [rows] staging slots used this step
  uint32_t* stats;           // [2] or null: attended host rows found staged / read from the host
  int cap;
  float alpha;               // weight of the newest k-th score in the EMA
};

// The unique id of the calling thread's current CUDA context; false when no context is
// bound yet.  Function attributes, module symbols, streams and events belong to a
// context, so state cached across calls is keyed by this id, never by the device
// ordinal alone (a new primary context after cudaDeviceReset, or a context the caller
// pushed, shares the ordinal but none of the old context's objects).
bool current_context_id(unsigned long long* id);

// Sets a kernel's dynamic shared-memory limit to dyn_smem bytes once per context and,
// when blocks_per_sm is not null, returns its resident CTAs per SM for `threads` threads
// and that much shared memory (at least 1).
skv_status prepare_kernel(const void* kernel, int dyn_smem, int threads = 0, int* blocks_per_sm = nullptr);
// How many clusters of `cluster` CTAs (threads each, dyn_smem bytes of dynamic shared
// memory) the current device holds at once (0: none fit, or the query failed); cached per
// CUDA context.  The kernel's dynamic shared-memory limit must already be set
// (prepare_kernel).
skv_status max_active_clusters(const void* kernel, int dyn_smem, int threads, int cluster, int* clusters);

// pf: optional; scoring then also stages the host rows of keys above the prediction
// (contiguous index keys with a per-token slot map only).
// The bounded-wait check (selftest.cu): a one-CTA wait that gives up after limit_cycles.
skv_status launch_wait_check(long long limit_cycles, int arrive, int32_t* status, cudaStream_t st);

skv_status launch_score(const skv_problem& p, const void* q_score, const skv_index_src& idx,
                        const PoolView& pool, float* scores, int32_t* status, cudaStream_t st,
                        const PrefetchView* pf = nullptr);

size_t topk_workspace_bytes(const skv_problem& p);
// zero_words: optional, one word per (request, KV head) row that the launch sets to
// zero when it can do so without using the workspace (*zeroed tells whether it did).
// row_geom: optional device [rows][2] (first candidate, count) replacing the sink/local regions.
// pf: optional; the selection then folds each row's k-th score into pf->tau.
// pos_map: optional [rows][max_len]: written in place of the selected score columns
// (only where topk_maps_positions(p): the one-CTA and two-stage paths).
bool topk_maps_positions(const skv_problem& p);
skv_status launch_topk(const skv_problem& p, const float* scores, int32_t* idx, void* ws,
                       int32_t* status, cudaStream_t st, uint32_t* zero_words = nullptr, bool* zeroed = nullptr,
                       const int32_t* row_geom = nullptr, const PrefetchView* pf = nullptr,
                       const int32_t* pos_map = nullptr);

size_t attn_workspace_bytes(const skv_problem& p);
int attn_splits(const skv_problem& p);
struct PrefetchView;
// bl: optional, bf16 only; the list comes from the chosen blocks (idx is then the list
// the kernel writes, bl->att).
skv_status launch_attn(const skv_problem& p, const void* q, const PoolView& pool, const int32_t* idx,
                       void* out, float* lse, void* ws, int32_t* status, cudaStream_t st,
                       bool tickets_zeroed = false, const PrefetchView* pf = nullptr,
                       const BlockListView* bl = nullptr);
// the per-unit merge tickets inside the attention workspace (nullptr if the path has none)
uint32_t* attn_tickets(const skv_problem& p, void* ws);

// MLA-style latent rows (d_qk 576, d_v 512 = leading entries of the row, one KV head)
bool latent_shape(const skv_problem& p);
size_t latent_workspace_bytes(const skv_problem& p);
// pf: optional; staged host rows are read from the staging area, and the step's end
// advances the epoch and clears the staging counts.
skv_status launch_attn_latent(const skv_problem& p, const void* q, const PoolView& pool, const int32_t* idx,
                              void* out, float* lse, void* ws, int32_t* status, cudaStream_t st,
                              const PrefetchView* pf = nullptr);

skv_status launch_gather(const skv_problem& p, const PoolView& pool, const int32_t* idx, void* k_out,
                         void* v_out, int32_t* status, cudaStream_t st);

// GPU slot cache over a host pool that backs every token (cache.cu)
// units: the cache's units, requests (latent rows) or (request, KV head) pairs (per-head tables)
size_t cache_workspace_bytes(const skv_problem& p, int n_slots, int budget, int units);
// ParisKV retrieval (paris.cu)
skv_status paris_quantizer(int m, float* levels, float* thresholds);
size_t paris_workspace_bytes(const skv_problem& p, const skv_paris& pr);
void paris_offsets(const skv_problem& p, const skv_paris& pr, int64_t* out);
skv_status launch_paris_encode(const skv_problem& p, const skv_paris& pr, const skv_index_src& src,
                               const PoolView& pool, const skv_paris_index& ix, int32_t* status, cudaStream_t st);
skv_status launch_paris_select(const skv_problem& p, const skv_paris& pr, const void* q_score,
                               const skv_paris_index& ix, int32_t* idx, void* pws, int32_t* status, cudaStream_t st);

// The update in two parts: rank (mark, eviction scores, top-k; reads the table, writes
// priorities) may run beside the step's attention; apply (assign, copy) writes the table
// and the slot rows, so it follows the attention.
skv_status launch_cache_rank(const skv_problem& p, const PoolView& pool, const int32_t* idx, int32_t* table,
                             int32_t* owner, int32_t* prio, int32_t* step, int budget, unsigned long long* stats,
                             void* cws, int32_t* status, cudaStream_t st);
skv_status launch_cache_apply(const skv_problem& p, const PoolView& pool, const int32_t* idx, int32_t* table,
                              void* gpu_rows, int32_t* owner, int32_t* prio, int32_t* step, int budget,
                              unsigned long long* stats, const void* attn_ws, void* cws, int32_t* status,
                              cudaStream_t st);
skv_status launch_cache_update(const skv_problem& p, const PoolView& pool, const int32_t* idx, int32_t* table,
                               void* gpu_rows, int32_t* owner, int32_t* prio, int32_t* step, int budget,
                               unsigned long long* stats, const void* attn_ws, void* cws, int32_t* status,
                               cudaStream_t st);

// block selection from per-block key summaries (blocks.cu)
int block_list_len(const skv_problem& p, int topk_blocks);
size_t block_summary_bytes(const skv_problem& p);
size_t block_workspace_bytes(const skv_problem& p, int topk_blocks);
skv_problem block_attn_problem(const skv_problem& p, int topk_blocks);
void* block_tail_ws(const skv_problem& p, void* ws);
skv_status launch_block_summaries(const skv_problem& p, const PoolView& pool, void* summ, int32_t* status,
                                  cudaStream_t st);
// expand = false leaves the attended list to the attention (block-list mode)
skv_status launch_block_select(const skv_problem& p, int topk_blocks, const void* q, const void* summ,
                               int32_t* bidx, int32_t* att, void* ws, int32_t* status, cudaStream_t st,
                               bool expand = true);

}  // namespace skv
