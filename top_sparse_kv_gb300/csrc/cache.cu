// GPU slot cache over a host pool that backs every token (sm_103a).
//
// ECHO-OSDI26 wiki, core method 2: the host pool holds every token's row (token t of
// request b at row b * max_len + t); a pool of GPU slots caches some of them, named by
// the slot table (entry >= 0: a GPU slot; < 0: the host row -e - 1).  Per slot, fixed
// -size device state: its owner (b * max_len + t, -1 when free) and its priority (the
// last step that used it).  After a step's attention every kernel below runs inside
// the captured step, with nothing sized by the host:
//   cache_mark_kernel    one CTA per request: attended tokens in GPU slots mark the
//                        slot used this step; the others (misses) are listed in
//                        (request, list position) order
//   cache_score_kernel   each slot's eviction score: NaN when used this step, +inf
//                        when free, else its age (step - priority)
//   (top-k)              the `budget` best candidates, exactly (ties: lower slot)
//   cache_assign_kernel  one CTA: the chosen slots not used this step take the misses
//                        in ascending slot order; evicted owners return to their host
//                        rows in the table; owners, priorities and table entries set;
//                        the step counter advances
//   cache_copy_kernel    a promoted row moves from the step's gathered rows (already
//                        in HBM) into its slot: no second trip over the host link; the
//                        table entry names the slot once the row is in (data, then map)
//
// With one slot-table row per (request, KV head) (OasisKV notes, §3.5: each head keeps
// its own blocks resident), the unit is a (request, KV head) u = b * H + h, an entry is a
// block of block_size tokens, a slot holds one head's block, and block j of request b is
// backed by host block b * stride + j (every head); owners are u * stride + j:
//   cache_head_mark_kernel    one CTA per unit: its attended positions set bits of a
//                             block bitmap in shared memory; the set blocks, ascending,
//                             protect their slots or are listed as misses
//   (scores and top-k as above)
//   cache_head_assign_kernel  cache_assign_kernel over units and blocks
//   cache_head_copy_kernel    one CTA per promotion: the head's K and V rows of the block
//                             from the host pool into the slot
#include "attn_common.cuh"

namespace skv {
namespace {

constexpr int kMarkThreads = 1024;
constexpr int kAssignThreads = 1024;

struct CacheArgs {
  AttnArgs m;                 // the step: sizes, idx, slot table, status
  int32_t* table;             // the slot table, updated in place
  int stride;                 // its row stride
  int32_t* owner;             // [n_slots]
  int32_t* prio;              // [n_slots]
  int32_t* step;              // [1]
  int n_slots, budget, n_att;
  int2* misses;               // [B, n_att]: (position, list index)
  int32_t* miss_count;        // [B]
  int32_t* hit_count;         // [B]: attended tokens found in GPU slots
  unsigned long long* stats;  // [3] or null: hits, misses, promotions, summed over steps
  float* score;               // [n_slots]
  int32_t* score_len;         // [1]: n_slots, the top-k's row length
  const int32_t* chosen;      // [budget] ascending, -1 past the count
  int2* pairs;                // [budget]: (slot, gathered row b * n_att + j)
  int32_t* n_pairs;           // [1]
  const unsigned char* rows;  // [B, n_att, row bytes] the step's gathered rows
  unsigned char* gpu_rows;    // [n_slots, row bytes] the GPU pool
  int row_bytes;
  // one table row per (request, KV head)
  int H, units, bs;             // pool heads, B * H, tokens a block
  const unsigned char* host_k;  // [n_host, H, bs, row_k_bytes]
  const unsigned char* host_v;
  unsigned char* gpu_k;         // [n_slots, bs, row_k_bytes]
  unsigned char* gpu_v;
  int row_k_bytes, row_v_bytes;
};

// Exclusive scan of one value per thread over a CTA of NT threads; *total gets the sum.
template <int NT>
__device__ __forceinline__ int cta_scan(int v, int* total, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NT / 32 ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < NT / 32) warp_sums[lane] = w;
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[NT / 32 - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kMarkThreads) cache_mark_kernel(const CacheArgs c) {
  __shared__ int warp_sums[32];
  const AttnArgs& a = c.m;
  const int b = blockIdx.x;
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const Regions rg = regions_of(L, a.ns, a.nl);
  const int n_list = rg.s_end + a.k + (L - rg.l_start);
  const int32_t* idx_row = a.idx + (size_t)b * a.k;  // one KV head
  const int stp = *c.step;
  int base = 0, hits = 0;
  for (int j0 = 0; j0 < n_list; j0 += kMarkThreads) {
    const int j = j0 + threadIdx.x;
    const int t = j < n_list ? list_pos(a, idx_row, rg, j, n_list) : -1;
    int miss = 0;
    if (t >= 0) {
      const int e = c.table[(size_t)b * c.stride + t];
      if (e >= 0 && e < c.n_slots) {
        c.prio[e] = stp;  // used this step: protected
        ++hits;
      } else if (e < 0) {
        miss = 1;
      }
    }
    int total;
    const int at = cta_scan<kMarkThreads>(miss, &total, warp_sums);
    if (miss) c.misses[(size_t)b * c.n_att + base + at] = make_int2(t, j);
    base += total;
  }
  if (c.stats != nullptr) {
    hits = __reduce_add_sync(0xffffffffu, (unsigned)hits);
    if ((threadIdx.x & 31) == 0) atomicAdd(&c.hit_count[b], hits);
  }
  if (threadIdx.x == 0) c.miss_count[b] = base;
}

__global__ void __launch_bounds__(256) cache_score_kernel(const CacheArgs c) {
  const int stp = *c.step;
  if (blockIdx.x == 0 && threadIdx.x == 0) c.score_len[0] = c.n_slots;
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < c.n_slots; s += gridDim.x * blockDim.x) {
    const int pr = c.prio[s];
    c.score[s] = pr == stp ? __int_as_float(0x7fc00000) : c.owner[s] < 0 ? INFINITY : (float)(stp - pr);
  }
}

__global__ void __launch_bounds__(kAssignThreads) cache_assign_kernel(const CacheArgs c) {
  constexpr int kU = 4;  // chosen entries a thread takes per round, all loads issued first
  __shared__ int warp_sums[32];
  __shared__ int mpre[65];  // miss prefix over requests (at most 64)
  __shared__ unsigned long long hits_sm;
  const AttnArgs& a = c.m;
  const int tid = threadIdx.x;
  const int stp = *c.step;
  // per-request misses (and hits) loaded in parallel; the prefix by one CTA scan
  const int mc = tid < a.B ? c.miss_count[tid] : 0;
  const int hc = (c.stats != nullptr && tid < a.B) ? c.hit_count[tid] : 0;
  if (tid == 0) hits_sm = 0ull;
  int n_miss;
  const int mp = cta_scan<kAssignThreads>(mc, &n_miss, warp_sums);
  if (tid <= a.B) mpre[tid] = mp;
  if (hc != 0) atomicAdd(&hits_sm, (unsigned long long)hc);
  // the chosen slots not used this step, in ascending slot order (compacted into pairs[].x)
  int nv = 0;
  for (int base = 0; base < c.budget; base += kAssignThreads * kU) {
    int sl[kU], ok[kU], cnt = 0;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = base + tid * kU + u;
      sl[u] = i < c.budget ? c.chosen[i] : -1;
    }
    int pr[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) pr[u] = sl[u] >= 0 ? c.prio[sl[u]] : stp;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      ok[u] = sl[u] >= 0 && pr[u] != stp;
      cnt += ok[u];
    }
    int total;
    int at = nv + cta_scan<kAssignThreads>(cnt, &total, warp_sums);
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (ok[u]) c.pairs[at++].x = sl[u];
    nv += total;
  }
  __syncthreads();  // pairs[].x and mpre complete
  const int np = nv < n_miss ? nv : n_miss;
  for (int i = tid; i < np; i += kAssignThreads) {
    int lo = 0, hi = a.B - 1;  // the request of miss i: the last b with mpre[b] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (mpre[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    const int b = lo;
    const int2 ms = c.misses[(size_t)b * c.n_att + (i - mpre[b])];
    const int s = c.pairs[i].x;
    const int old = c.owner[s];
    if (old >= 0 && old / a.max_len < a.B) c.table[(size_t)(old / a.max_len) * c.stride + old % a.max_len] = -old - 1;
    else if (old >= 0) flag(a.status, SKV_DEV_BAD_SLOT);  // an owner no request can hold: table untouched
    c.owner[s] = b * a.max_len + ms.x;  // the table entry follows the row's copy
    c.prio[s] = stp;
    c.pairs[i].y = b * c.n_att + ms.y;
  }
  if (c.stats != nullptr && tid < a.B) c.hit_count[tid] = 0;  // ready for the next step
  __syncthreads();
  if (tid == 0) {
    c.n_pairs[0] = np;
    *c.step = stp + 1;
    if (c.stats != nullptr) {
      c.stats[0] += hits_sm;
      c.stats[1] += (unsigned)n_miss;
      c.stats[2] += (unsigned)np;
    }
  }
}

__global__ void __launch_bounds__(kMarkThreads) cache_head_mark_kernel(const CacheArgs c) {
  extern __shared__ uint32_t blk_bits[];  // [ceil(blocks / 32)]
  __shared__ int warp_sums[32];
  const AttnArgs& a = c.m;
  const int u = blockIdx.x, b = u / c.H;
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const Regions rg = regions_of(L, a.ns, a.nl);
  const int n_list = rg.s_end + a.k + (L - rg.l_start);
  const int32_t* idx_row = a.idx + (size_t)u * a.k;
  const int words = ((L + c.bs - 1) / c.bs + 31) >> 5;
  for (int w = threadIdx.x; w < words; w += kMarkThreads) blk_bits[w] = 0u;
  __syncthreads();
  for (int j = threadIdx.x; j < n_list; j += kMarkThreads) {
    const int t = list_pos(a, idx_row, rg, j, n_list);
    if (t >= 0) atomicOr(&blk_bits[(t / c.bs) >> 5], 1u << ((t / c.bs) & 31));
  }
  __syncthreads();
  const int stp = *c.step;
  const int32_t* trow = c.table + (size_t)u * c.stride;
  int base = 0, hits = 0;
  for (int w0 = 0; w0 < words; w0 += kMarkThreads) {  // the same trip count in every thread
    const int w = w0 + threadIdx.x;
    uint32_t miss = 0;
    for (uint32_t m = w < words ? blk_bits[w] : 0u; m; m &= m - 1) {
      const int bit = __ffs(m) - 1;
      const int e = trow[(w << 5) + bit];
      if (e >= 0 && e < c.n_slots) {
        c.prio[e] = stp;  // used this step: protected
        ++hits;
      } else if (e < 0) {
        miss |= 1u << bit;
      }
    }
    int total;
    int at = base + cta_scan<kMarkThreads>(__popc(miss), &total, warp_sums);
    for (; miss; miss &= miss - 1) c.misses[(size_t)u * c.n_att + at++] = make_int2((w << 5) + __ffs(miss) - 1, 0);
    base += total;
  }
  if (c.stats != nullptr) {
    hits = __reduce_add_sync(0xffffffffu, (unsigned)hits);
    if ((threadIdx.x & 31) == 0) atomicAdd(&c.hit_count[u], hits);
  }
  if (threadIdx.x == 0) c.miss_count[u] = base;
}

__global__ void __launch_bounds__(kAssignThreads) cache_head_assign_kernel(const CacheArgs c) {
  constexpr int kU = 4;  // chosen entries a thread takes per round, all loads issued first
  __shared__ int warp_sums[32];
  __shared__ int mpre[kAssignThreads];  // miss prefix over units (at most kAssignThreads)
  __shared__ unsigned long long hits_sm;
  const AttnArgs& a = c.m;
  const int tid = threadIdx.x;
  const int stp = *c.step;
  const int mc = tid < c.units ? c.miss_count[tid] : 0;
  const int hc = (c.stats != nullptr && tid < c.units) ? c.hit_count[tid] : 0;
  if (tid == 0) hits_sm = 0ull;
  int n_miss;
  const int mp = cta_scan<kAssignThreads>(mc, &n_miss, warp_sums);
  if (tid < c.units) mpre[tid] = mp;
  if (hc != 0) atomicAdd(&hits_sm, (unsigned long long)hc);
  int nv = 0;  // the chosen slots not used this step, ascending, compacted into pairs[].x
  for (int base = 0; base < c.budget; base += kAssignThreads * kU) {
    int sl[kU], ok[kU], pr[kU], cnt = 0;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = base + tid * kU + u;
      sl[u] = i < c.budget ? c.chosen[i] : -1;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) pr[u] = sl[u] >= 0 ? c.prio[sl[u]] : stp;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      ok[u] = sl[u] >= 0 && pr[u] != stp;
      cnt += ok[u];
    }
    int total;
    int at = nv + cta_scan<kAssignThreads>(cnt, &total, warp_sums);
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (ok[u]) c.pairs[at++].x = sl[u];
    nv += total;
  }
  __syncthreads();  // pairs[].x and mpre complete
  const int np = nv < n_miss ? nv : n_miss;
  for (int i = tid; i < np; i += kAssignThreads) {
    int lo = 0, hi = c.units - 1;  // the unit of miss i: the last u with mpre[u] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (mpre[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    const int u = lo;
    const int j = c.misses[(size_t)u * c.n_att + (i - mpre[u])].x;
    const int s = c.pairs[i].x;
    const int old = c.owner[s];
    if (old >= 0 && old / c.stride < c.units) {  // the evicted block returns to its host block
      const int uo = old / c.stride, jo = old % c.stride;
      c.table[(size_t)uo * c.stride + jo] = -((uo / c.H) * c.stride + jo) - 1;
    } else if (old >= 0) {
      flag(a.status, SKV_DEV_BAD_SLOT);  // an owner no unit can hold: table untouched
    }
    c.owner[s] = u * c.stride + j;  // the table entry follows the block's copy
    c.prio[s] = stp;
    c.pairs[i].y = u * c.stride + j;
  }
  if (c.stats != nullptr && tid < c.units) c.hit_count[tid] = 0;  // ready for the next step
  __syncthreads();
  if (tid == 0) {
    c.n_pairs[0] = np;
    *c.step = stp + 1;
    if (c.stats != nullptr) {
      c.stats[0] += hits_sm;
      c.stats[1] += (unsigned)n_miss;
      c.stats[2] += (unsigned)np;
    }
  }
}

__global__ void __launch_bounds__(256) cache_head_copy_kernel(const CacheArgs c) {
  const int i = blockIdx.x;
  if (i >= c.n_pairs[0]) return;
  const int2 pr = c.pairs[i];  // (slot, owner u * stride + j)
  const int u = pr.y / c.stride, j = pr.y % c.stride;
  // the head's first row in its host block, and in the slot
  const size_t hrow = (((size_t)(u / c.H) * c.stride + j) * c.H + u % c.H) * c.bs;
  const size_t grow = (size_t)pr.x * c.bs;
  const uint4* ks = (const uint4*)(c.host_k + hrow * c.row_k_bytes);
  uint4* kd = (uint4*)(c.gpu_k + grow * c.row_k_bytes);
  for (int q = threadIdx.x; q < c.bs * c.row_k_bytes / 16; q += blockDim.x) kd[q] = ks[q];
  const uint4* vs = (const uint4*)(c.host_v + hrow * c.row_v_bytes);
  uint4* vd = (uint4*)(c.gpu_v + grow * c.row_v_bytes);
  for (int q = threadIdx.x; q < c.bs * c.row_v_bytes / 16; q += blockDim.x) vd[q] = vs[q];
  __syncthreads();  // data, then map
  if (threadIdx.x == 0) {
    __threadfence();
    c.table[pr.y] = pr.x;  // owner u * stride + j is the entry's index in the [units, stride] table
  }
}

// Data, then map (UlaCache article §8): the table names the slot only after its row is in.
__global__ void __launch_bounds__(256) cache_copy_kernel(const CacheArgs c) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= c.n_pairs[0]) return;
  const int2 pr = c.pairs[w];
  const uint4* src = (const uint4*)(c.rows + (size_t)pr.y * c.row_bytes);
  uint4* dst = (uint4*)(c.gpu_rows + (size_t)pr.x * c.row_bytes);
  for (int q = lane; q < c.row_bytes / 16; q += 32) dst[q] = src[q];
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    const int own = c.owner[pr.x];  // b * max_len + t, set by the assignment
    c.table[(size_t)(own / c.m.max_len) * c.stride + own % c.m.max_len] = pr.x;
  }
}

struct CacheLayout {
  size_t misses, miss_count, hit_count, score, score_len, chosen, pairs, n_pairs, topk, total;
};

skv_problem cache_topk_problem(const skv_problem& p, int n_slots, int budget, const int32_t* len) {
  skv_problem r = p;
  r.batch = 1;
  r.n_kv_heads = 1;
  r.n_q_heads = 1;
  r.n_idx_q_heads = 1;
  r.max_len = n_slots;
  r.topk = budget;
  r.n_sink = 0;
  r.n_local = 0;
  r.seq_lens = len;
  return r;
}

CacheLayout cache_layout(const skv_problem& p, int n_slots, int budget, int units) {
  const size_t B = (size_t)units, n = (size_t)max_list(p);
  CacheLayout l;
  l.misses = 0;
  l.miss_count = l.misses + align256(B * n * 8);
  l.hit_count = l.miss_count + align256(B * 4);
  l.score = l.hit_count + align256(B * 4);
  l.score_len = l.score + align256((size_t)n_slots * 4);
  l.chosen = l.score_len + 256;
  l.pairs = l.chosen + align256((size_t)budget * 4);
  l.n_pairs = l.pairs + align256((size_t)budget * 8);
  l.topk = l.n_pairs + 256;
  l.total = l.topk + topk_workspace_bytes(cache_topk_problem(p, n_slots, budget, nullptr));
  return l;
}

}  // namespace

size_t cache_workspace_bytes(const skv_problem& p, int n_slots, int budget, int units) {
  return cache_layout(p, n_slots, budget, units).total;
}

namespace {

CacheArgs cache_args(const skv_problem& p, const PoolView& pool, const int32_t* idx, int32_t* table, void* gpu_rows,
                     int32_t* owner, int32_t* prio, int32_t* step, int budget, unsigned long long* stats,
                     const void* attn_ws, void* cws, int32_t* status, CacheLayout* lay_out) {
  const int n_slots = (int)pool.n_gpu;
  const int units = pool.per_head ? p.batch * p.n_kv_heads : p.batch;
  const CacheLayout lay = cache_layout(p, n_slots, budget, units);
  unsigned char* w = (unsigned char*)cws;
  CacheArgs c{};
  c.m = make_args(p, nullptr, pool, idx, status);
  c.table = table;
  c.stride = pool.stride;
  c.owner = owner;
  c.prio = prio;
  c.step = step;
  c.n_slots = n_slots;
  c.budget = budget;
  c.n_att = max_list(p);
  c.misses = (int2*)(w + lay.misses);
  c.miss_count = (int32_t*)(w + lay.miss_count);
  c.hit_count = (int32_t*)(w + lay.hit_count);
  c.stats = stats;
  c.score = (float*)(w + lay.score);
  c.score_len = (int32_t*)(w + lay.score_len);
  c.chosen = (const int32_t*)(w + lay.chosen);
  c.pairs = (int2*)(w + lay.pairs);
  c.n_pairs = (int32_t*)(w + lay.n_pairs);
  c.rows = (const unsigned char*)attn_ws;  // the latent gather's rows lead the attention workspace
  c.gpu_rows = (unsigned char*)gpu_rows;
  c.row_bytes = p.d_qk * 2;
  c.H = pool.per_head ? p.n_kv_heads : 1;
  c.units = units;
  c.bs = p.block_size;
  const int elem = p.dtype == SKV_DTYPE_F32 ? 4 : 2;
  c.row_k_bytes = p.d_qk * elem;
  c.row_v_bytes = p.d_v * elem;
  c.host_k = (const unsigned char*)pool.host_k;
  c.host_v = (const unsigned char*)pool.host_v;
  c.gpu_k = (unsigned char*)const_cast<void*>(pool.gpu_k);
  c.gpu_v = (unsigned char*)const_cast<void*>(pool.gpu_v);
  *lay_out = lay;
  return c;
}

}  // namespace

skv_status launch_cache_rank(const skv_problem& p, const PoolView& pool, const int32_t* idx, int32_t* table,
                             int32_t* owner, int32_t* prio, int32_t* step, int budget, unsigned long long* stats,
                             void* cws, int32_t* status, cudaStream_t st) {
  CacheLayout lay;
  const CacheArgs c = cache_args(p, pool, idx, table, nullptr, owner, prio, step, budget, stats, nullptr, cws, status,
                                 &lay);
  unsigned char* w = (unsigned char*)cws;
  if (stats != nullptr && cudaMemsetAsync(c.hit_count, 0, (size_t)c.units * 4, st) != cudaSuccess) return SKV_ERR_CUDA;
  if (pool.per_head) {
    const int words = ((p.max_len + p.block_size - 1) / p.block_size + 31) / 32;
    cache_head_mark_kernel<<<c.units, kMarkThreads, (size_t)words * 4, st>>>(c);
  } else {
    cache_mark_kernel<<<p.batch, kMarkThreads, 0, st>>>(c);
  }
  SKV_LAUNCH_CHECK();
  const long long sb = ((long long)c.n_slots + 255) / 256;
  const long long cap = (long long)num_sms() * 8;
  cache_score_kernel<<<(unsigned)(sb < cap ? (sb > 0 ? sb : 1) : cap), 256, 0, st>>>(c);
  SKV_LAUNCH_CHECK();
  return launch_topk(cache_topk_problem(p, c.n_slots, budget, c.score_len), c.score, (int32_t*)(w + lay.chosen),
                     w + lay.topk, status, st);
}

skv_status launch_cache_apply(const skv_problem& p, const PoolView& pool, const int32_t* idx, int32_t* table,
                              void* gpu_rows, int32_t* owner, int32_t* prio, int32_t* step, int budget,
                              unsigned long long* stats, const void* attn_ws, void* cws, int32_t* status,
                              cudaStream_t st) {
  CacheLayout lay;
  const CacheArgs c = cache_args(p, pool, idx, table, gpu_rows, owner, prio, step, budget, stats, attn_ws, cws,
                                 status, &lay);
  // a plain launch: this may follow a join of two streams, which is no kernel-to-kernel edge
  if (pool.per_head) {
    cache_head_assign_kernel<<<1, kAssignThreads, 0, st>>>(c);
    SKV_LAUNCH_CHECK();
    if (budget > 0) {
      cache_head_copy_kernel<<<(unsigned)budget, 256, 0, st>>>(c);
      SKV_LAUNCH_CHECK();
    }
    return SKV_OK;
  }
  cache_assign_kernel<<<1, kAssignThreads, 0, st>>>(c);
  SKV_LAUNCH_CHECK();
  if (budget > 0) {
    cache_copy_kernel<<<(unsigned)(((long long)budget * 32 + 255) / 256), 256, 0, st>>>(c);
    SKV_LAUNCH_CHECK();
  }
  return SKV_OK;
}

skv_status launch_cache_update(const skv_problem& p, const PoolView& pool, const int32_t* idx, int32_t* table,
                               void* gpu_rows, int32_t* owner, int32_t* prio, int32_t* step, int budget,
                               unsigned long long* stats, const void* attn_ws, void* cws, int32_t* status,
                               cudaStream_t st) {
  const skv_status r = launch_cache_rank(p, pool, idx, table, owner, prio, step, budget, stats, cws, status, st);
  if (r != SKV_OK) return r;
  return launch_cache_apply(p, pool, idx, table, gpu_rows, owner, prio, step, budget, stats, attn_ws, cws, status,
                            st);
}

}  // namespace skv
