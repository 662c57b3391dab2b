// Block selection from per-block key summaries (sm_103a).
//
// Every 16-token block of a KV head keeps the per-coordinate minimum and maximum
// of its keys; a KV head ranks blocks from these two rows alone and attends the
// chosen blocks whole (OasisKV notes, §3.2 "compressed key summaries", after
// Quest).  A block's score is the largest <q, k> any key inside its
// per-coordinate box can reach: sum_j max(q_j min_j, q_j max_j), with q the
// group's mean query, or the largest of the heads' own bounds (the max reading).
// Sink and local windows are rounded outward to whole blocks; the candidates are
// the blocks between them.
//
//   block_summary_kernel   min / max rows of every block (maintenance: run when
//                          blocks fill, not per step); one warp per block, the
//                          block's rows read through the slot table (GPU pool or
//                          pinned host pool over UVA)
//   block_score_kernel     the box bound of every candidate block from its two
//                          summary rows (1/8 of the keys' bytes); one warp per run
//                          of 32 blocks of a row, the query loaded once per run;
//                          also writes each row's candidate range
//   (top-k)                the exact top-K blocks, the token top-k kernels run on
//                          the block scores with those ranges
//   block_expand_kernel    sink, chosen and local blocks -> the ascending list of
//                          attended token positions, which the sparse attention
//                          reads with zero-width windows (skv_block_select; the
//                          bf16 decode step instead lets the attention derive each
//                          list slot from the chosen blocks and write the list)
#include "skv_internal.cuh"

namespace skv {
namespace {

constexpr int kBlk = kBlockTokens;  // tokens per block: the paged pool's block size
constexpr int kD = 128;
constexpr int kBlockMaxHeads = 16;  // scoring heads kept apart by the max reading

struct BlockArgs {
  PoolView pool;
  const int32_t* seq_lens;
  int B, H, max_len, nbmax, ns, nl;
  int gi, n_idx_q, agg;
  float inv_gi;
  const unsigned char* q;  // [B, n_idx_q, kD] scoring heads
  unsigned char* summ;     // [B, H, nbmax, 2, kD]: min row, max row
  float* bscore;           // [B * H, nbmax]
  int32_t* geom;           // [B * H][2]: first candidate block, candidate count
  const int32_t* bidx;     // [B * H, K] chosen blocks, ascending, -1 past the count
  int K;
  int32_t* att;            // [B * H, n_att]
  int n_att;
  int32_t* status;
};

// Address of row 0 of (request b, head h, block blk) in its tier, or nullptr (bad slot).
__device__ __forceinline__ const unsigned char* block_rows(const BlockArgs& a, int b, int h, int blk, int row_bytes) {
  const int e = a.pool.table[(size_t)b * a.pool.stride + blk];
  if (e >= 0) {
    if (e < a.pool.n_gpu) return (const unsigned char*)a.pool.gpu_k + ((size_t)e * a.H + h) * kBlk * row_bytes;
  } else {
    const long long hb = -(long long)e - 1;
    if (a.pool.host_k != nullptr && hb < a.pool.n_host)
      return (const unsigned char*)a.pool.host_k + ((size_t)hb * a.H + h) * kBlk * row_bytes;
  }
  return nullptr;
}

// One warp per block.  Lanes split the row into 16-byte chunks (CH per row);
// the 32 / CH lane groups take every (32 / CH)-th token, then fold together.
template <typename T>
__global__ void __launch_bounds__(256) block_summary_kernel(const BlockArgs a) {
  constexpr int kRowB = kD * (int)sizeof(T);
  constexpr int CH = kRowB / 16;     // chunks per row: 16 (bf16) or 32 (fp32)
  constexpr int TG = 32 / CH;        // token groups per warp
  constexpr int EPC = 16 / sizeof(T);
  const int lane = threadIdx.x & 31;
  const int c = lane % CH, tg = lane / CH;
  const long long total = (long long)a.B * a.H * a.nbmax;
  for (long long w = blockIdx.x * (long long)(blockDim.x / 32) + (threadIdx.x >> 5); w < total;
       w += (long long)gridDim.x * (blockDim.x / 32)) {
    const int row = (int)(w / a.nbmax), blk = (int)(w % a.nbmax);
    const int b = row / a.H, h = row % a.H;
    const int L = load_len(a.seq_lens, b, a.max_len, a.status);
    if (blk * kBlk >= L) continue;  // no token of this block exists yet
    const int n = L - blk * kBlk < kBlk ? L - blk * kBlk : kBlk;
    const unsigned char* src = block_rows(a, b, h, blk, kRowB);
    float lo[EPC], hi[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      lo[e] = INFINITY;
      hi[e] = -INFINITY;
    }
    if (src != nullptr) {
      for (int t = tg; t < n; t += TG) {
        float v[EPC];
        Vec<T>::load(src + (size_t)t * kRowB + c * 16, v);
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
          lo[e] = fminf(lo[e], v[e]);
          hi[e] = fmaxf(hi[e], v[e]);
        }
      }
    } else {
      if (lane == 0) flag(a.status, SKV_DEV_BAD_SLOT);
#pragma unroll
      for (int e = 0; e < EPC; ++e) lo[e] = hi[e] = __int_as_float(0x7fc00000);  // NaN: the block ranks last
    }
#pragma unroll
    for (int off = CH; off < 32; off <<= 1)
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        lo[e] = fminf(lo[e], __shfl_xor_sync(0xffffffffu, lo[e], off));
        hi[e] = fmaxf(hi[e], __shfl_xor_sync(0xffffffffu, hi[e], off));
      }
    if (src == nullptr) {
#pragma unroll
      for (int e = 0; e < EPC; ++e) lo[e] = hi[e] = __int_as_float(0x7fc00000);
    }
    unsigned char* dst = a.summ + ((size_t)row * a.nbmax + blk) * 2 * kRowB;
    if (tg == 0) {  // min row; the max row from the next token group (or the same lanes for fp32)
      alignas(16) T o[EPC];
#pragma unroll
      for (int e = 0; e < EPC; ++e) o[e] = from_float<T>(lo[e]);
      *reinterpret_cast<uint4*>(dst + c * 16) = *reinterpret_cast<const uint4*>(o);
    }
    if (tg == TG - 1) {
      alignas(16) T o[EPC];
#pragma unroll
      for (int e = 0; e < EPC; ++e) o[e] = from_float<T>(hi[e]);
      *reinterpret_cast<uint4*>(dst + kRowB + c * 16) = *reinterpret_cast<const uint4*>(o);
    }
  }
}

// One warp per run of kRun consecutive blocks of one row: the group's query (its
// mean, or every head for the max reading) is loaded once per run; CH lanes take
// one block (a 16-byte chunk of its min and of its max row each), 32 / CH blocks
// at a time.  Writes the scores of the candidate blocks and every row's
// candidate range.
constexpr int kRun = 32;
constexpr int kBatch = 8;  // blocks of a run whose summary loads are issued together

template <typename T, int GMAX>
__global__ void __launch_bounds__(256) block_score_kernel(const BlockArgs a) {
  constexpr int kRowB = kD * (int)sizeof(T);
  constexpr int CH = kRowB / 16;
  constexpr int BPW = 32 / CH;  // blocks per warp step
  constexpr int EPC = 16 / sizeof(T);
  pdl_release();
  const int lane = threadIdx.x & 31;
  const int c = lane % CH, sub = lane / CH;
  const int runs_per_row = (a.nbmax + kRun - 1) / kRun;
  const long long runs = (long long)a.B * a.H * runs_per_row;
  for (long long w = blockIdx.x * (long long)(blockDim.x / 32) + (threadIdx.x >> 5); w < runs;
       w += (long long)gridDim.x * (blockDim.x / 32)) {
    const int row = (int)(w / runs_per_row), run = (int)(w % runs_per_row);
    const int b = row / a.H, h = row % a.H;
    const int L = load_len(a.seq_lens, b, a.max_len, a.status);
    const BlockRegions rg = block_regions(L, a.ns, a.nl);
    if (run == 0 && lane == 0) {
      a.geom[2 * row] = rg.s_blk;
      a.geom[2 * row + 1] = rg.l_blk - rg.s_blk;
    }
    const int b0 = run * kRun > rg.s_blk ? run * kRun : rg.s_blk;
    const int b1 = run * kRun + kRun < rg.l_blk ? run * kRun + kRun : rg.l_blk;
    if (b0 >= b1) continue;  // no candidate block in this run (warp-uniform)
    // this lane's dims of the group's scoring heads
    const unsigned char* qp = a.q + ((size_t)b * a.n_idx_q + (size_t)h * a.gi) * kRowB + c * 16;
    float qh[GMAX][EPC];
    const bool by_max = a.agg == SKV_AGG_MAX;
    const int nh = by_max ? a.gi : 1;
    if (by_max) {
#pragma unroll
      for (int g = 0; g < GMAX; ++g)
        if (g < a.gi) Vec<T>::load(qp + (size_t)g * kRowB, qh[g]);
    } else {
#pragma unroll
      for (int e = 0; e < EPC; ++e) qh[0][e] = 0.f;
      for (int g = 0; g < a.gi; ++g) {
        float qv[EPC];
        Vec<T>::load(qp + (size_t)g * kRowB, qv);
#pragma unroll
        for (int e = 0; e < EPC; ++e) qh[0][e] += qv[e];
      }
#pragma unroll
      for (int e = 0; e < EPC; ++e) qh[0][e] *= a.inv_gi;
    }
    constexpr int U = kBatch / BPW;  // steps of a batch: their loads issued before any use
    for (int bb = b0; bb < b1; bb += kBatch) {
      uint4 rl[U], rh[U];  // packed until use: a batch's loads in flight without widened registers
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int blk = bb + i * BPW + sub;
        if (blk < b1) {
          const unsigned char* sp = a.summ + ((size_t)row * a.nbmax + blk) * 2 * kRowB;
          rl[i] = *reinterpret_cast<const uint4*>(sp + c * 16);
          rh[i] = *reinterpret_cast<const uint4*>(sp + kRowB + c * 16);
        } else {
          rl[i] = rh[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int blk = bb + i * BPW + sub;
        float lo[EPC], hi[EPC];
        Vec<T>::widen(rl[i], lo);
        Vec<T>::widen(rh[i], hi);
        float u = -INFINITY;
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
          if (g < nh) {  // uniform across the warp
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < EPC; ++e) part += fmaxf(qh[g][e] * lo[e], qh[g][e] * hi[e]);
#pragma unroll
            for (int off = CH / 2; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            u = g == 0 ? part : fmaxf(u, part);
          }
        }
        if (blk < b1 && c == 0) a.bscore[(size_t)row * a.nbmax + blk] = u;
      }
    }
  }
}

// One CTA per (request, KV head): slot j of the attended list holds token
// 16 i + (j % 16) of the i = j / 16-th attended block (sink blocks, chosen
// blocks, local blocks, ascending); only the last block can be partial.
constexpr int kExpandStage = 4096;  // chosen blocks staged in shared memory (more are read from global)

__global__ void __launch_bounds__(512) block_expand_kernel(const BlockArgs a) {
  __shared__ int32_t chosen[kExpandStage];
  pdl_wait();  // the chosen blocks are complete and visible
  pdl_release();
  const int row = blockIdx.x;
  const int b = row / a.H;
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const BlockRegions rg = block_regions(L, a.ns, a.nl);
  const int n_cand = rg.l_blk - rg.s_blk;
  const int ksel = a.K < n_cand ? a.K : n_cand;
  const int32_t* bg = a.bidx + (size_t)row * a.K;
  for (int i = threadIdx.x; i < ksel && i < kExpandStage; i += blockDim.x) chosen[i] = bg[i];
  __syncthreads();
  const int32_t* bi = ksel <= kExpandStage ? chosen : bg;
  int32_t* out = a.att + (size_t)row * a.n_att;
  for (int j = threadIdx.x; j < a.n_att; j += blockDim.x) out[j] = block_list_token(bi, a.K, rg, L, j, a.status);
}

BlockArgs make_block_args(const skv_problem& p, const PoolView& pool, int32_t* status) {
  BlockArgs a{};
  a.pool = pool;
  a.seq_lens = p.seq_lens;
  a.B = p.batch;
  a.H = p.n_kv_heads;
  a.max_len = p.max_len;
  a.nbmax = (p.max_len + kBlk - 1) / kBlk;
  a.ns = p.n_sink;
  a.nl = p.n_local;
  a.gi = p.n_q_heads / p.n_kv_heads;
  a.n_idx_q = p.n_q_heads;
  a.agg = p.group_agg;
  a.inv_gi = 1.f / (float)a.gi;
  a.status = status;
  return a;
}

unsigned warp_grid(long long warps) {
  const long long cap = (long long)num_sms() * 16;  // 16 CTAs of 8 warps per SM
  const long long need = (warps + 7) / 8;
  return (unsigned)(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace

int block_list_len(const skv_problem& p, int topk_blocks) {
  return kBlk * ((p.n_sink + kBlk - 1) / kBlk + topk_blocks + (p.n_local + kBlk - 1) / kBlk + 1);
}

size_t block_summary_bytes(const skv_problem& p) {
  return (size_t)p.batch * p.n_kv_heads * ((p.max_len + kBlk - 1) / kBlk) * 2 * kD *
         (p.dtype == SKV_DTYPE_F32 ? 4 : 2);
}

skv_status launch_block_summaries(const skv_problem& p, const PoolView& pool, void* summ, int32_t* status,
                                  cudaStream_t st) {
  BlockArgs a = make_block_args(p, pool, status);
  a.summ = (unsigned char*)summ;
  const long long warps = (long long)a.B * a.H * a.nbmax;
  if (warps == 0) return SKV_OK;
  if (p.dtype == SKV_DTYPE_F32)
    block_summary_kernel<float><<<warp_grid(warps), 256, 0, st>>>(a);
  else
    block_summary_kernel<__nv_bfloat16><<<warp_grid(warps), 256, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

// The block-score rows as a top-k problem: one "position" per block.
skv_problem block_rows_problem(const skv_problem& p, int topk_blocks) {
  skv_problem r = p;
  r.max_len = (p.max_len + kBlk - 1) / kBlk;
  r.topk = topk_blocks;
  r.n_sink = 0;
  r.n_local = 0;
  return r;
}

// The attention over the expanded token list: windows of width zero, k = the list length.
skv_problem block_attn_problem(const skv_problem& p, int topk_blocks) {
  skv_problem r = p;
  r.topk = block_list_len(p, topk_blocks);
  r.n_sink = 0;
  r.n_local = 0;
  return r;
}

size_t block_workspace_bytes(const skv_problem& p, int topk_blocks) {
  const size_t rows = (size_t)p.batch * p.n_kv_heads;
  const size_t nbmax = (size_t)(p.max_len + kBlk - 1) / kBlk;
  const size_t t = topk_workspace_bytes(block_rows_problem(p, topk_blocks));
  const size_t at = attn_workspace_bytes(block_attn_problem(p, topk_blocks));
  return align256(rows * nbmax * 4) + align256(rows * 2 * 4) + (t > at ? t : at);
}

void* block_tail_ws(const skv_problem& p, void* ws) {
  const size_t rows = (size_t)p.batch * p.n_kv_heads;
  const size_t nbmax = (size_t)(p.max_len + kBlk - 1) / kBlk;
  return (unsigned char*)ws + align256(rows * nbmax * 4) + align256(rows * 2 * 4);
}

skv_status launch_block_select(const skv_problem& p, int topk_blocks, const void* q, const void* summ,
                               int32_t* bidx, int32_t* att, void* ws, int32_t* status, cudaStream_t st,
                               bool expand) {
  BlockArgs a = make_block_args(p, PoolView{}, status);
  const size_t rows = (size_t)p.batch * p.n_kv_heads;
  unsigned char* w = (unsigned char*)ws;
  a.q = (const unsigned char*)q;
  a.summ = (unsigned char*)summ;
  a.bscore = (float*)w;
  a.geom = (int32_t*)(w + align256(rows * a.nbmax * 4));
  void* tws = w + align256(rows * a.nbmax * 4) + align256(rows * 2 * 4);
  a.bidx = bidx;
  a.K = topk_blocks;
  a.att = att;
  a.n_att = block_list_len(p, topk_blocks);
  const long long warps = (long long)rows * ((a.nbmax + kRun - 1) / kRun);
  if (a.agg == SKV_AGG_MAX && a.gi > kBlockMaxHeads) return SKV_ERR_UNSUPPORTED;
  const bool per_head = a.agg == SKV_AGG_MAX;
  const unsigned grid = warp_grid(warps);
  if (p.dtype == SKV_DTYPE_F32) {
    if (!per_head) block_score_kernel<float, 1><<<grid, 256, 0, st>>>(a);
    else if (a.gi <= 8) block_score_kernel<float, 8><<<grid, 256, 0, st>>>(a);
    else block_score_kernel<float, kBlockMaxHeads><<<grid, 256, 0, st>>>(a);
  } else {
    if (!per_head) block_score_kernel<__nv_bfloat16, 1><<<grid, 256, 0, st>>>(a);
    else if (a.gi <= 8) block_score_kernel<__nv_bfloat16, 8><<<grid, 256, 0, st>>>(a);
    else block_score_kernel<__nv_bfloat16, kBlockMaxHeads><<<grid, 256, 0, st>>>(a);
  }
  SKV_LAUNCH_CHECK();
  const skv_problem pb = block_rows_problem(p, topk_blocks);
  const skv_status r = launch_topk(pb, a.bscore, bidx, tws, status, st, nullptr, nullptr, a.geom);
  if (r != SKV_OK) return r;
  if (!expand) return SKV_OK;  // the attention lists the blocks' tokens as it resolves them
  if (launch_dependent(block_expand_kernel, dim3((unsigned)rows), dim3(512), 0, st, 1, a) != cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace skv
