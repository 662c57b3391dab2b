// C ABI of libskv: argument validation and dispatch to the kernels.
//
// Validation happens on the host before anything is enqueued and touches no
// CUDA API, so a rejected call has no side effect (and can be exercised on a
// machine without a GPU).
#include <cuda.h>  // CUcontext and CUresult (the two context calls are fetched from the driver at run time)

#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include "skv_internal.cuh"

namespace skv {

static std::atomic<uint64_t> g_launches{0};

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

namespace {
struct PreparedKernel {
  const void* kernel;
  unsigned long long ctx;
  int smem, threads, blocks;
  int cluster;  // 0: blocks = resident CTAs a SM; > 0: blocks = co-resident clusters of this size
};
std::mutex g_prepared_mu;
std::vector<PreparedKernel> g_prepared;
}  // namespace

skv_status prepare_kernel(const void* kernel, int dyn_smem, int threads, int* blocks_per_sm) {
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(g_prepared_mu);
  if (have_ctx)
    for (const PreparedKernel& e : g_prepared)
      if (e.kernel == kernel && e.ctx == ctx && e.smem == dyn_smem && e.threads == threads && e.cluster == 0) {
        if (blocks_per_sm) *blocks_per_sm = e.blocks;
        return SKV_OK;
      }
  // first use in this context (the call binds the runtime's context if none was bound)
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem) != cudaSuccess)
    return SKV_ERR_CUDA;
  int blocks = 0;
  if (blocks_per_sm != nullptr) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, dyn_smem) != cudaSuccess)
      return SKV_ERR_CUDA;
    if (blocks < 1) blocks = 1;
    *blocks_per_sm = blocks;
  }
  if (have_ctx || current_context_id(&ctx)) g_prepared.push_back({kernel, ctx, dyn_smem, threads, blocks, 0});
  return SKV_OK;
}

skv_status max_active_clusters(const void* kernel, int dyn_smem, int threads, int cluster, int* clusters) {
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(g_prepared_mu);
  if (have_ctx)
    for (const PreparedKernel& e : g_prepared)
      if (e.kernel == kernel && e.ctx == ctx && e.smem == dyn_smem && e.threads == threads && e.cluster == cluster) {
        *clusters = e.blocks;
        return SKV_OK;
      }
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)cluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)dyn_smem;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    // a device or context that cannot report it is treated as holding no cluster (the
    // caller then launches without one); the error is cleared so no later check sees it
    (void)cudaGetLastError();
    n = 0;
  }
  *clusters = n;
  if (have_ctx || current_context_id(&ctx)) g_prepared.push_back({kernel, ctx, dyn_smem, threads, n, cluster});
  return SKV_OK;
}

skv_problem head_rows(const skv_problem& p) {
  if (p.group_agg != SKV_AGG_HEAD) return p;
  skv_problem r = p;
  r.n_kv_heads = p.n_q_heads;
  r.n_idx_q_heads = p.n_q_heads;
  r.group_agg = SKV_AGG_MEAN;  // a group of one: its mean is the head itself
  return r;
}

int num_sms() {
  static int cached_dev = -1;
  static int cached_sms = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cached_sms = n;
    cached_dev = dev;
  }
  return cached_sms;
}

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// The shapes the kernels are built for.
bool is_latent(const skv_problem& p, const skv_kv_pool* pool) { return pool && pool->gpu_v == nullptr; }

skv_status check_problem(const skv_problem* p) {
  if (!p) return SKV_ERR_INVALID_ARGUMENT;
  if (p->batch < 1 || p->n_kv_heads < 1 || p->n_q_heads < 1) return SKV_ERR_INVALID_ARGUMENT;
  if (p->n_q_heads % p->n_kv_heads) return SKV_ERR_INVALID_ARGUMENT;
  if (p->d_qk < 1 || p->d_v < 1 || p->d_idx < 1) return SKV_ERR_INVALID_ARGUMENT;
  if (p->n_idx_q_heads < 1 || p->n_idx_q_heads % p->n_kv_heads) return SKV_ERR_INVALID_ARGUMENT;
  if (p->max_len < 0 || p->topk < 0 || p->n_sink < 0 || p->n_local < 0) return SKV_ERR_INVALID_ARGUMENT;
  if (p->block_size < 1 || p->n_splits < 0) return SKV_ERR_INVALID_ARGUMENT;
  if (p->dtype != SKV_DTYPE_BF16 && p->dtype != SKV_DTYPE_F32) return SKV_ERR_INVALID_ARGUMENT;
  if (p->group_agg != SKV_AGG_MEAN && p->group_agg != SKV_AGG_MAX && p->group_agg != SKV_AGG_HEAD)
    return SKV_ERR_INVALID_ARGUMENT;
  if (p->group_agg == SKV_AGG_MAX && (p->dtype != SKV_DTYPE_BF16 || p->n_idx_q_heads / p->n_kv_heads > 16))
    return SKV_ERR_UNSUPPORTED;  // max needs the tensor-core scoring tile
  if (p->group_agg == SKV_AGG_HEAD &&  // per query head: the tensor-core tile scores every head of a group
      (p->dtype != SKV_DTYPE_BF16 || p->n_idx_q_heads != p->n_q_heads || p->n_q_heads / p->n_kv_heads > 16 ||
       p->n_q_heads > 65535))
    return SKV_ERR_UNSUPPORTED;
  if (!(p->sm_scale == p->sm_scale)) return SKV_ERR_INVALID_ARGUMENT;  // NaN
  if (!p->seq_lens) return SKV_ERR_INVALID_ARGUMENT;
  const long long sel_heads = p->group_agg == SKV_AGG_HEAD ? p->n_q_heads : p->n_kv_heads;  // score rows
  if ((long long)p->batch * sel_heads * (long long)p->max_len > (1LL << 40)) return SKV_ERR_INVALID_ARGUMENT;
  if (p->batch > 65535 || p->n_kv_heads > 65535) return SKV_ERR_UNSUPPORTED;  // grid y/z extents
  return SKV_OK;
}

skv_status check_pool(const skv_problem& p, const skv_kv_pool* pool) {
  if (!pool || !pool->slot_table || !pool->gpu_k) return SKV_ERR_INVALID_ARGUMENT;
  if (pool->n_gpu_blocks < 0 || pool->n_host_blocks < 0) return SKV_ERR_INVALID_ARGUMENT;
  const long long need = ((long long)p.max_len + p.block_size - 1) / p.block_size;
  if (pool->table_stride < need) return SKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(pool->gpu_k) || !aligned16(pool->gpu_v) || !aligned16(pool->host_k) || !aligned16(pool->host_v))
    return SKV_ERR_INVALID_ARGUMENT;
  if ((pool->host_k == nullptr) != (pool->host_v == nullptr) && pool->gpu_v != nullptr)
    return SKV_ERR_INVALID_ARGUMENT;
  if (pool->gpu_v == nullptr && pool->host_v != nullptr) return SKV_ERR_INVALID_ARGUMENT;
  if (pool->table_heads != 0 && pool->table_heads != 1) return SKV_ERR_INVALID_ARGUMENT;
  if (pool->table_heads == 1 && pool->gpu_v == nullptr) return SKV_ERR_UNSUPPORTED;  // K and V pools only
  if (pool->table_heads == 1 && (long long)p.batch * p.n_kv_heads * pool->table_stride >= (1LL << 40))
    return SKV_ERR_INVALID_ARGUMENT;
  return SKV_OK;
}

// the entry points built for a table row per request only
static skv_status no_head_table(const skv_kv_pool* pool) {
  return pool != nullptr && pool->table_heads != 0 ? SKV_ERR_UNSUPPORTED : SKV_OK;
}

// Shapes of the attention / gather kernels.
skv_status check_attn_shape(const skv_problem& p, const skv_kv_pool* pool) {
  const int G = p.n_q_heads / p.n_kv_heads;
  if (is_latent(p, pool)) {
    if (p.n_kv_heads != 1 || p.d_v > p.d_qk) return SKV_ERR_INVALID_ARGUMENT;
    if (!latent_shape(p)) return SKV_ERR_UNSUPPORTED;  // built for 576/512 bf16, heads a multiple of 64
    const long long n_att = (long long)p.n_sink + p.topk + p.n_local;
    if (n_att < 1 || n_att > 64LL * 256) return SKV_ERR_UNSUPPORTED;  // up to 64 blocks of 256 rows
    return SKV_OK;
  }
  if (p.d_qk != 128 || p.d_v != 128) return SKV_ERR_UNSUPPORTED;
  if (G > 16) return SKV_ERR_UNSUPPORTED;
  // at most 1024 splits of at most 512 attended rows each
  if ((long long)p.n_sink + p.topk + p.n_local > 512LL * 1024) return SKV_ERR_UNSUPPORTED;
  return SKV_OK;
}

skv_status check_score_shape(const skv_problem& p, const skv_index_src* index, const skv_kv_pool* pool) {
  if (!index) return SKV_ERR_INVALID_ARGUMENT;
  if (p.d_idx != 128) return SKV_ERR_UNSUPPORTED;
  if (index->layout == SKV_INDEX_PAGED) {
    if (p.block_size != 16 || p.d_idx != p.d_qk || is_latent(p, pool)) return SKV_ERR_UNSUPPORTED;
    if (!pool) return SKV_ERR_INVALID_ARGUMENT;
  } else if (index->layout == SKV_INDEX_CONTIG) {
    if (!index->keys || !aligned16(index->keys)) return SKV_ERR_INVALID_ARGUMENT;
  } else {
    return SKV_ERR_INVALID_ARGUMENT;
  }
  return SKV_OK;
}

PoolView view(const skv_kv_pool* pool) {
  PoolView v{};
  v.hdiv = 1;
  if (!pool) return v;
  v.gpu_k = pool->gpu_k;
  v.gpu_v = pool->gpu_v;
  v.n_gpu = pool->n_gpu_blocks;
  v.host_k = pool->host_k;
  v.host_v = pool->host_v;
  v.n_host = pool->n_host_blocks;
  v.table = pool->slot_table;
  v.per_head = pool->table_heads != 0 ? 1 : 0;
  v.stride = pool->table_stride;
  return v;
}

size_t workspace_bytes(const skv_problem& p) {
  const skv_problem r = head_rows(p);
  const size_t a = attn_workspace_bytes(r), t = topk_workspace_bytes(r);
  return a > t ? a : t;
}

// the pool as the rows of head_rows(p) see it
PoolView head_view(const skv_problem& p, const skv_kv_pool* pool) {
  PoolView v = view(pool);
  if (p.group_agg == SKV_AGG_HEAD) v.hdiv = p.n_q_heads / p.n_kv_heads;
  return v;
}

// the entry points built for one row per KV head only
skv_status no_head_rows(const skv_problem* p) {
  return p->group_agg == SKV_AGG_HEAD ? SKV_ERR_UNSUPPORTED : SKV_OK;
}

#define SKV_TRY(expr)            \
  do {                           \
    skv_status r_ = (expr);      \
    if (r_ != SKV_OK) return r_; \
  } while (0)

}  // namespace
}  // namespace skv

using namespace skv;

extern "C" {

skv_status skv_workspace_size(const skv_problem* p, size_t* bytes) {
  SKV_TRY(check_problem(p));
  if (!bytes) return SKV_ERR_INVALID_ARGUMENT;
  *bytes = workspace_bytes(*p);
  return SKV_OK;
}

skv_status skv_score(const skv_problem* p, const void* q_score, const skv_index_src* index, const skv_kv_pool* pool,
                     float* scores, int32_t* dev_status, void* stream) {
  SKV_TRY(check_problem(p));
  if (!q_score || !scores || !aligned16(q_score) || !aligned16(scores)) return SKV_ERR_INVALID_ARGUMENT;
  if (index && index->layout == SKV_INDEX_PAGED) SKV_TRY(check_pool(*p, pool));
  SKV_TRY(check_score_shape(*p, index, pool));
  return launch_score(*p, q_score, *index, view(pool), scores, dev_status, (cudaStream_t)stream);
}

skv_status skv_topk(const skv_problem* p, const float* scores, int32_t* idx, void* ws, size_t ws_bytes,
                    int32_t* dev_status, void* stream) {
  SKV_TRY(check_problem(p));
  if (!scores || !idx || !aligned16(scores)) return SKV_ERR_INVALID_ARGUMENT;
  const skv_problem r = head_rows(*p);
  const size_t need = topk_workspace_bytes(r);
  if (ws_bytes < need) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  return launch_topk(r, scores, idx, ws, dev_status, (cudaStream_t)stream);
}

skv_status skv_gather(const skv_problem* p, const skv_kv_pool* pool, const int32_t* idx, void* k_out, void* v_out,
                      int32_t* dev_status, void* stream) {
  SKV_TRY(check_problem(p));
  SKV_TRY(check_pool(*p, pool));
  if (!idx || !k_out || !aligned16(k_out) || !aligned16(v_out)) return SKV_ERR_INVALID_ARGUMENT;
  if ((p->d_qk * (p->dtype == SKV_DTYPE_F32 ? 4 : 2)) % 16 || (p->d_v * (p->dtype == SKV_DTYPE_F32 ? 4 : 2)) % 16)
    return SKV_ERR_UNSUPPORTED;
  if (is_latent(*p, pool) && (p->n_kv_heads != 1 || p->d_v > p->d_qk)) return SKV_ERR_INVALID_ARGUMENT;
  if (is_latent(*p, pool)) SKV_TRY(no_head_rows(p));
  return launch_gather(head_rows(*p), head_view(*p, pool), idx, k_out, v_out, dev_status, (cudaStream_t)stream);
}

skv_status skv_sparse_attn(const skv_problem* p, const void* q, const skv_kv_pool* pool, const int32_t* idx,
                           void* out, float* lse, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  SKV_TRY(check_problem(p));
  SKV_TRY(check_pool(*p, pool));
  if (!q || !idx || !out || !aligned16(q) || !aligned16(out)) return SKV_ERR_INVALID_ARGUMENT;
  if (is_latent(*p, pool)) SKV_TRY(no_head_rows(p));
  const skv_problem r = head_rows(*p);
  SKV_TRY(check_attn_shape(r, pool));
  const size_t need = attn_workspace_bytes(r);
  if (ws_bytes < need) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  return launch_attn(r, q, head_view(*p, pool), idx, out, lse, ws, dev_status, (cudaStream_t)stream);
}

static skv_status check_step(const skv_problem* p, const void* q, const void* q_score, const skv_index_src* index,
                             const skv_kv_pool* pool, float* scores, int32_t* idx, void* out, void* ws,
                             size_t ws_bytes) {
  SKV_TRY(check_problem(p));
  SKV_TRY(check_pool(*p, pool));
  const void* qs = q_score ? q_score : q;
  if (!q || !qs || !scores || !idx || !out) return SKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(qs) || !aligned16(scores) || !aligned16(out)) return SKV_ERR_INVALID_ARGUMENT;
  SKV_TRY(check_score_shape(*p, index, pool));
  if (is_latent(*p, pool)) SKV_TRY(no_head_rows(p));
  SKV_TRY(check_attn_shape(head_rows(*p), pool));
  if (ws_bytes < workspace_bytes(*p)) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  return SKV_OK;
}

skv_status skv_decode_step(const skv_problem* p, const void* q, const void* q_score, const skv_index_src* index,
                           const skv_kv_pool* pool, float* scores, int32_t* idx, void* out, float* lse, void* ws,
                           size_t ws_bytes, int32_t* dev_status, void* stream) {
  SKV_TRY(check_step(p, q, q_score, index, pool, scores, idx, out, ws, ws_bytes));
  const void* qs = q_score ? q_score : q;
  cudaStream_t st = (cudaStream_t)stream;
  SKV_TRY(launch_score(*p, qs, *index, view(pool), scores, dev_status, st));
  // per query head, the selection and the attention run over one row a query head
  const skv_problem r = head_rows(*p);
  // the selection clears the attention's merge tickets when it needs no workspace itself
  bool zeroed = false;
  SKV_TRY(launch_topk(r, scores, idx, ws, dev_status, st, attn_tickets(r, ws), &zeroed));
  return launch_attn(r, q, head_view(*p, pool), idx, out, lse, ws, dev_status, st, zeroed);
}

// ---------------------------------------------------------------- block selection

static skv_status check_block_problem(const skv_problem* p, const skv_kv_pool* pool) {
  SKV_TRY(check_problem(p));
  SKV_TRY(no_head_rows(p));
  if (p->block_size != 16 || p->d_qk != 128 || p->d_idx != 128) return SKV_ERR_UNSUPPORTED;
  if (p->n_idx_q_heads != p->n_q_heads) return SKV_ERR_UNSUPPORTED;  // the attention group scores its blocks
  if (p->group_agg == SKV_AGG_MAX && p->n_q_heads / p->n_kv_heads > 16) return SKV_ERR_UNSUPPORTED;
  if (pool) {
    SKV_TRY(check_pool(*p, pool));
    SKV_TRY(no_head_table(pool));
    if (!pool->gpu_v) return SKV_ERR_UNSUPPORTED;  // latent rows: no block mode
  }
  return SKV_OK;
}

skv_status skv_block_workspace_size(const skv_problem* p, int32_t topk_blocks, size_t* bytes, int32_t* list_len) {
  SKV_TRY(check_block_problem(p, nullptr));
  if (topk_blocks < 0 || !bytes) return SKV_ERR_INVALID_ARGUMENT;
  *bytes = block_workspace_bytes(*p, topk_blocks);
  if (list_len) *list_len = block_list_len(*p, topk_blocks);
  return SKV_OK;
}

skv_status skv_block_summaries(const skv_problem* p, const skv_kv_pool* pool, void* summaries, int32_t* dev_status,
                               void* stream) {
  SKV_TRY(check_block_problem(p, pool));
  if (!summaries || !aligned16(summaries)) return SKV_ERR_INVALID_ARGUMENT;
  return launch_block_summaries(*p, view(pool), summaries, dev_status, (cudaStream_t)stream);
}

skv_status skv_block_select(const skv_problem* p, int32_t topk_blocks, const void* q, const void* summaries,
                            int32_t* block_idx, int32_t* att_idx, void* ws, size_t ws_bytes, int32_t* dev_status,
                            void* stream) {
  SKV_TRY(check_block_problem(p, nullptr));
  if (topk_blocks < 0 || !q || !summaries || !att_idx || (topk_blocks > 0 && !block_idx))
    return SKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(summaries)) return SKV_ERR_INVALID_ARGUMENT;
  if (ws_bytes < block_workspace_bytes(*p, topk_blocks)) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  return launch_block_select(*p, topk_blocks, q, summaries, block_idx, att_idx, ws, dev_status,
                             (cudaStream_t)stream);
}

skv_status skv_block_decode_step(const skv_problem* p, int32_t topk_blocks, const void* q, const void* summaries,
                                 const skv_kv_pool* pool, int32_t* block_idx, int32_t* att_idx, void* out,
                                 float* lse, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  SKV_TRY(check_block_problem(p, pool));
  if (topk_blocks < 0 || !q || !summaries || !att_idx || !out || (topk_blocks > 0 && !block_idx))
    return SKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(summaries) || !aligned16(out)) return SKV_ERR_INVALID_ARGUMENT;
  const skv_problem pa = block_attn_problem(*p, topk_blocks);
  SKV_TRY(check_attn_shape(pa, pool));
  if (ws_bytes < block_workspace_bytes(*p, topk_blocks)) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  cudaStream_t st = (cudaStream_t)stream;
  // bf16: the attention derives its list slots from the chosen blocks and writes att_idx
  // itself, so the expansion kernel is not launched
  const bool fused = p->dtype == SKV_DTYPE_BF16;
  SKV_TRY(launch_block_select(*p, topk_blocks, q, summaries, block_idx, att_idx, ws, dev_status, st, !fused));
  if (!fused) return launch_attn(pa, q, view(pool), att_idx, out, lse, block_tail_ws(*p, ws), dev_status, st);
  const BlockListView bl{block_idx, topk_blocks, p->n_sink, p->n_local, att_idx};
  return launch_attn(pa, q, view(pool), att_idx, out, lse, block_tail_ws(*p, ws), dev_status, st, false, nullptr,
                     &bl);
}

// ---------------------------------------------------------------- threshold prefetch

skv_status skv_decode_step_prefetch(const skv_problem* p, const void* q, const void* q_score,
                                    const skv_index_src* index, const skv_kv_pool* pool, float* scores, int32_t* idx,
                                    void* out, float* lse, void* ws, size_t ws_bytes, const skv_prefetch* pf,
                                    int32_t* dev_status, void* stream) {
  SKV_TRY(check_problem(p));
  SKV_TRY(no_head_rows(p));
  SKV_TRY(check_pool(*p, pool));
  SKV_TRY(no_head_table(pool));
  if (!pf || !q_score || !q || !scores || !idx || !out) return SKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(q_score) || !aligned16(scores) || !aligned16(out)) return SKV_ERR_INVALID_ARGUMENT;
  // the latent layout (a per-token map), or a paged pool of 16-token blocks with K and V rows of 128
  const bool latent = pool->gpu_v == nullptr && p->block_size == 1;
  const bool paged = pool->gpu_v != nullptr && p->block_size == 16 && p->d_qk == 128 && p->d_v == 128;
  if ((!latent && !paged) || !index || index->layout != SKV_INDEX_CONTIG || p->dtype != SKV_DTYPE_BF16 ||
      p->group_agg != SKV_AGG_MEAN)
    return SKV_ERR_UNSUPPORTED;
  if (!pf->tau_ema || !pf->epoch || !pf->map || !pf->count || pf->cap < 0 || !(pf->alpha > 0.f && pf->alpha <= 1.f))
    return SKV_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)pf->map & 7u) != 0 || (pf->cap > 0 && (!pf->staging || !aligned16(pf->staging))))
    return SKV_ERR_INVALID_ARGUMENT;
  if ((p->d_qk + (paged ? p->d_v : 0)) * 2 > 1536 || (p->d_qk * 2) % 16)
    return SKV_ERR_UNSUPPORTED;  // a staged token: up to 96 chunks of 16 bytes
  SKV_TRY(check_score_shape(*p, index, pool));
  SKV_TRY(check_attn_shape(*p, pool));
  if (ws_bytes < workspace_bytes(*p)) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  PrefetchView v{};
  v.tau = pf->tau_ema;
  v.epoch = pf->epoch;
  v.map = (unsigned long long*)pf->map;
  v.staging = (unsigned char*)pf->staging;
  v.count = pf->count;
  v.stats = pf->stats;
  v.cap = pf->cap;
  v.alpha = pf->alpha;
  cudaStream_t st = (cudaStream_t)stream;
  const PoolView pv = view(pool);
  SKV_TRY(launch_score(*p, q_score, *index, pv, scores, dev_status, st, &v));
  SKV_TRY(launch_topk(*p, scores, idx, ws, dev_status, st, nullptr, nullptr, nullptr, &v));
  return launch_attn(*p, q, pv, idx, out, lse, ws, dev_status, st, false, &v);
}

// ---------------------------------------------------------------- GPU slot cache

// One side stream per device, with a fork and a join event: the slot cache's ranking
// runs there beside the step's attention.  Created once; a call holds the mutex while
// it enqueues the fork, the ranking and the join, so the events are never shared by
// two calls at once (a wait, once enqueued, no longer depends on the event's reuse).
struct SideStream {
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  unsigned long long ctx = 0;  // the context they belong to
};
static std::mutex g_side_mu;
static SideStream g_side[64];

static skv_status side_stream(SideStream** out) {  // the caller holds g_side_mu
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SKV_ERR_CUDA;
  SideStream& s = g_side[dev];
  unsigned long long ctx = 0;
  // objects of another context (a reset device, a pushed context) are not reused: the
  // old handles are dropped, not destroyed, since their context may no longer exist
  if (s.st != nullptr && (!current_context_id(&ctx) || ctx != s.ctx)) s = SideStream{};
  if (s.st == nullptr) {
    if (cudaStreamCreateWithFlags(&s.st, cudaStreamNonBlocking) != cudaSuccess) return SKV_ERR_CUDA;
    if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess) return SKV_ERR_CUDA;
    if (cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) return SKV_ERR_CUDA;
    if (!current_context_id(&s.ctx)) return SKV_ERR_CUDA;
  }
  *out = &s;
  return SKV_OK;
}

// the slot cache's units: requests (latent rows), or (request, KV head) pairs (per-head tables)
static int cache_units(const skv_problem& p, const skv_kv_pool* pool) {
  return pool->table_heads == 1 ? p.batch * p.n_kv_heads : p.batch;
}

static skv_status check_cache_problem(const skv_problem* p, const skv_kv_pool* pool, int32_t budget) {
  SKV_TRY(check_problem(p));
  SKV_TRY(no_head_rows(p));
  SKV_TRY(check_pool(*p, pool));
  if (budget < 0) return SKV_ERR_INVALID_ARGUMENT;
  if (pool->table_heads == 1) {  // blocks of one table row per (request, KV head)
    const long long units = (long long)p->batch * p->n_kv_heads, stride = pool->table_stride;
    const int elem = p->dtype == SKV_DTYPE_F32 ? 4 : 2;
    if (units > 1024 || (p->d_qk * elem) % 16 || (p->d_v * elem) % 16) return SKV_ERR_UNSUPPORTED;
    if (pool->n_host_blocks < p->batch * stride || pool->n_gpu_blocks < 1) return SKV_ERR_UNSUPPORTED;
    if (pool->n_gpu_blocks > (1LL << 30) || units * stride >= (1LL << 31)) return SKV_ERR_UNSUPPORTED;
    if ((stride + 31) / 32 * 4 > 32 * 1024) return SKV_ERR_UNSUPPORTED;  // the mark kernel's block bitmap
    return SKV_OK;
  }
  if (pool->gpu_v != nullptr || p->block_size != 1 || p->batch > 64) return SKV_ERR_UNSUPPORTED;
  if (pool->n_host_blocks < (long long)p->batch * p->max_len || pool->n_gpu_blocks < 1) return SKV_ERR_UNSUPPORTED;
  if (pool->n_gpu_blocks > (1LL << 30) || (long long)p->batch * p->max_len >= (1LL << 31)) return SKV_ERR_UNSUPPORTED;
  return SKV_OK;
}

skv_status skv_cache_workspace_size(const skv_problem* p, const skv_kv_pool* pool, int32_t budget, size_t* bytes) {
  SKV_TRY(check_cache_problem(p, pool, budget));
  if (!bytes) return SKV_ERR_INVALID_ARGUMENT;
  *bytes = cache_workspace_bytes(*p, (int)pool->n_gpu_blocks, budget, cache_units(*p, pool));
  return SKV_OK;
}

skv_status skv_cache_prepare(void) {
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* side = nullptr;
  return side_stream(&side);
}

static skv_status check_cache_call(const skv_problem* p, const skv_kv_pool* pool, const skv_slot_cache* cache,
                                   void* cache_ws, size_t cache_ws_bytes) {
  if (!cache) return SKV_ERR_INVALID_ARGUMENT;
  SKV_TRY(check_cache_problem(p, pool, cache->budget));
  if (!cache->owner || !cache->prio || !cache->step) return SKV_ERR_INVALID_ARGUMENT;
  if (cache_ws_bytes < cache_workspace_bytes(*p, (int)pool->n_gpu_blocks, cache->budget, cache_units(*p, pool)))
    return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!cache_ws || !aligned16(cache_ws)) return SKV_ERR_INVALID_ARGUMENT;
  return SKV_OK;
}

static skv_status enqueue_cache_update(const skv_problem* p, const skv_kv_pool* pool, const int32_t* idx,
                                       const void* ws, const skv_slot_cache* cache, void* cache_ws,
                                       int32_t* dev_status, void* stream) {
  return launch_cache_update(*p, view(pool), idx, const_cast<int32_t*>(pool->slot_table),
                             const_cast<void*>(pool->gpu_k), cache->owner, cache->prio, cache->step, cache->budget,
                             (unsigned long long*)cache->stats, ws, cache_ws, dev_status, (cudaStream_t)stream);
}

skv_status skv_cache_update(const skv_problem* p, const skv_kv_pool* pool, const int32_t* idx, const void* ws,
                            size_t ws_bytes, const skv_slot_cache* cache, void* cache_ws, size_t cache_ws_bytes,
                            int32_t* dev_status, void* stream) {
  SKV_TRY(check_cache_call(p, pool, cache, cache_ws, cache_ws_bytes));
  size_t need = 0;
  SKV_TRY(skv_workspace_size(p, &need));
  if (ws_bytes < need) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!idx || !ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  return enqueue_cache_update(p, pool, idx, ws, cache, cache_ws, dev_status, stream);
}

skv_status skv_decode_step_cached(const skv_problem* p, const void* q, const void* q_score,
                                  const skv_index_src* index, const skv_kv_pool* pool, float* scores, int32_t* idx,
                                  void* out, float* lse, void* ws, size_t ws_bytes, const skv_slot_cache* cache,
                                  void* cache_ws, size_t cache_ws_bytes, int32_t* dev_status, void* stream) {
  SKV_TRY(check_cache_call(p, pool, cache, cache_ws, cache_ws_bytes));
  SKV_TRY(check_step(p, q, q_score, index, pool, scores, idx, out, ws, ws_bytes));
  const void* qs = q_score ? q_score : q;
  cudaStream_t st = (cudaStream_t)stream;
  const PoolView v = view(pool);
  int32_t* table = const_cast<int32_t*>(pool->slot_table);
  unsigned long long* stats = (unsigned long long*)cache->stats;
  SKV_TRY(launch_score(*p, qs, *index, v, scores, dev_status, st));
  bool zeroed = false;
  SKV_TRY(launch_topk(*p, scores, idx, ws, dev_status, st, attn_tickets(*p, ws), &zeroed));
  // fork: the ranking reads the selection and the table, writes only priorities and
  // its own workspace -- nothing the attention reads or writes
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* side = nullptr;
  SKV_TRY(side_stream(&side));
  if (cudaEventRecord(side->fork, st) != cudaSuccess || cudaStreamWaitEvent(side->st, side->fork, 0) != cudaSuccess)
    return SKV_ERR_CUDA;
  const skv_status rank = launch_cache_rank(*p, v, idx, table, cache->owner, cache->prio, cache->step, cache->budget,
                                            stats, cache_ws, dev_status, side->st);
  const bool joined = cudaEventRecord(side->join, side->st) == cudaSuccess;  // join whatever was enqueued
  const skv_status att = launch_attn(*p, q, v, idx, out, lse, ws, dev_status, st, zeroed);
  if (!joined || cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return SKV_ERR_CUDA;
  if (rank != SKV_OK) return rank;
  if (att != SKV_OK) return att;
  // the table and the slot rows change only after the attention has read them
  return launch_cache_apply(*p, v, idx, table, const_cast<void*>(pool->gpu_k), cache->owner, cache->prio,
                            cache->step, cache->budget, stats, ws, cache_ws, dev_status, st);
}

// ---------------------------------------------------------------- ParisKV retrieval

static skv_status check_paris(const skv_problem* p, const skv_paris* pr, const skv_index_src* index,
                              const skv_kv_pool* pool) {
  SKV_TRY(check_problem(p));
  SKV_TRY(no_head_rows(p));
  SKV_TRY(check_pool(*p, pool));
  SKV_TRY(no_head_table(pool));
  if (!pr || !index || !pr->signs) return SKV_ERR_INVALID_ARGUMENT;
  if (pr->beta_pm < 1 || pr->beta_pm > 1000 || pr->rho_pm < pr->beta_pm || pr->rho_pm > 1000)
    return SKV_ERR_INVALID_ARGUMENT;
  if (pr->m != 8 || p->dtype != SKV_DTYPE_BF16) return SKV_ERR_UNSUPPORTED;
  if ((long long)p->batch * p->n_kv_heads > 65535) return SKV_ERR_UNSUPPORTED;  // rows index grid.y
  if (index->layout == SKV_INDEX_CONTIG) {
    if (p->d_idx != 128) return SKV_ERR_UNSUPPORTED;
    if (!index->keys || !aligned16(index->keys)) return SKV_ERR_INVALID_ARGUMENT;
  } else if (index->layout == SKV_INDEX_PAGED) {
    if (p->d_qk != 128 || pool->gpu_v == nullptr) return SKV_ERR_UNSUPPORTED;
  } else {
    return SKV_ERR_INVALID_ARGUMENT;
  }
  if (p->n_idx_q_heads % p->n_kv_heads) return SKV_ERR_INVALID_ARGUMENT;
  return SKV_OK;
}

static skv_status check_paris_index(const skv_paris_index* ix) {
  if (!ix || !ix->cent || !ix->rec || !ix->hist) return SKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(ix->cent) || !aligned16(ix->rec)) return SKV_ERR_INVALID_ARGUMENT;
  return SKV_OK;
}

skv_status skv_paris_quantizer(int32_t m, float* levels, float* thresholds) {
  if (!levels || !thresholds) return SKV_ERR_INVALID_ARGUMENT;
  return paris_quantizer(m, levels, thresholds);
}

skv_status skv_paris_encode(const skv_problem* p, const skv_paris* paris, const skv_index_src* index,
                            const skv_kv_pool* pool, const skv_paris_index* out, int32_t* dev_status, void* stream) {
  SKV_TRY(check_paris(p, paris, index, pool));
  SKV_TRY(check_paris_index(out));
  return launch_paris_encode(*p, *paris, *index, view(pool), *out, dev_status, (cudaStream_t)stream);
}

static size_t paris_attn_bytes(const skv_problem& p) { return align256(workspace_bytes(p)); }

skv_status skv_paris_workspace_size(const skv_problem* p, const skv_paris* paris, size_t* bytes) {
  SKV_TRY(check_problem(p));
  SKV_TRY(no_head_rows(p));
  if (!paris || !bytes) return SKV_ERR_INVALID_ARGUMENT;
  if (paris->beta_pm < 1 || paris->beta_pm > 1000) return SKV_ERR_INVALID_ARGUMENT;
  *bytes = paris_attn_bytes(*p) + paris_workspace_bytes(*p, *paris);
  return SKV_OK;
}

skv_status skv_paris_workspace_offsets(const skv_problem* p, const skv_paris* paris, int64_t* out) {
  SKV_TRY(check_problem(p));
  SKV_TRY(no_head_rows(p));
  if (!paris || !out) return SKV_ERR_INVALID_ARGUMENT;
  if (paris->beta_pm < 1 || paris->beta_pm > 1000) return SKV_ERR_INVALID_ARGUMENT;
  paris_offsets(*p, *paris, out);
  const int64_t base = (int64_t)paris_attn_bytes(*p);
  for (int i = 0; i < 7; ++i) out[i] += base;
  out[8] += base;
  return SKV_OK;
}

skv_status skv_paris_select(const skv_problem* p, const skv_paris* paris, const void* q_score,
                            const skv_index_src* index, const skv_paris_index* meta, const skv_kv_pool* pool,
                            int32_t* idx, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  SKV_TRY(check_paris(p, paris, index, pool));
  SKV_TRY(check_paris_index(meta));
  if (!q_score || !idx || !aligned16(q_score)) return SKV_ERR_INVALID_ARGUMENT;
  const size_t attn = paris_attn_bytes(*p);
  if (ws_bytes < attn + paris_workspace_bytes(*p, *paris)) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  return launch_paris_select(*p, *paris, q_score, *meta, idx, (unsigned char*)ws + attn, dev_status,
                             (cudaStream_t)stream);
}

skv_status skv_paris_decode_step(const skv_problem* p, const skv_paris* paris, const void* q, const void* q_score,
                                 const skv_index_src* index, const skv_paris_index* meta, const skv_kv_pool* pool,
                                 int32_t* idx, void* out, float* lse, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, void* stream) {
  SKV_TRY(check_paris(p, paris, index, pool));
  SKV_TRY(check_paris_index(meta));
  SKV_TRY(check_attn_shape(*p, pool));
  const void* qs = q_score ? q_score : q;
  if (!q || !qs || !idx || !out) return SKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(qs) || !aligned16(out)) return SKV_ERR_INVALID_ARGUMENT;
  const size_t attn = paris_attn_bytes(*p);
  if (ws_bytes < attn + paris_workspace_bytes(*p, *paris)) return SKV_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned16(ws)) return SKV_ERR_INVALID_ARGUMENT;
  cudaStream_t st = (cudaStream_t)stream;
  SKV_TRY(launch_paris_select(*p, *paris, qs, *meta, idx, (unsigned char*)ws + attn, dev_status, st));
  return launch_attn(*p, q, view(pool), idx, out, lse, ws, dev_status, st, false);
}

const char* skv_status_string(skv_status s) {
  switch (s) {
    case SKV_OK: return "ok";
    case SKV_ERR_INVALID_ARGUMENT: return "invalid argument";
    case SKV_ERR_UNSUPPORTED: return "unsupported shape";
    case SKV_ERR_CUDA: return "CUDA error";
    case SKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SKV_ERR_DEVICE_FAULT: return "device fault reported in dev_status";
    case SKV_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

uint64_t skv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

skv_status skv_check_wait_timeout(int64_t limit_cycles, int32_t arrive, int32_t* dev_status, void* stream) {
  if (limit_cycles < 1 || limit_cycles > 4000000000LL) return SKV_ERR_INVALID_ARGUMENT;
  if ((arrive != 0 && arrive != 1) || dev_status == nullptr) return SKV_ERR_INVALID_ARGUMENT;
  return launch_wait_check((long long)limit_cycles, arrive, dev_status, (cudaStream_t)stream);
}

}  // extern "C"
