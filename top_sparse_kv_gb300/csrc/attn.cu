// S3 + S4 + S5: slot-table resolve, split-K sparse flash-decode, log-sum-exp merge.
//
// The attended list of (request b, KV head h) is
//     [0, s_end) ++ idx[b][h][0..topk) ++ [l_start, L)
// (sink and local windows attended densely next to the retrieved set:
// ParisKV notes §2.5).  Every list entry t resolves through the slot table
// (vToken notes §3.4 Eq. (2)): e >= 0 reads the GPU pool from HBM, e < 0 reads
// the pinned host pool in place over UVA (ECHO-OSDI26 wiki, core method 1;
// OasisKV notes §3.3 Algorithm 1) -- no copy is launched by the CPU.
//
// attn_split_kernel: one CTA per (split, KV head, request).  The list is cut
// into n_splits equal chunks; each of the 4 warps walks groups of R rows of the
// chunk.  A lane owns 4 of the 128 dims: it holds the G query heads' slices
// (pre-scaled by sm_scale*log2 e) and the G output accumulators.  The R x G
// partial dot products of a group are reduced with a butterfly that leaves one
// finished logit per lane; an fp32 online softmax (running max m, sum l) per
// head rescales the accumulators; V rows are accumulated with the broadcast
// probabilities.  The warps' states are merged in shared memory and the CTA
// writes one (m, l, acc) partial per query head.
//
// The n_splits partials of each (request, KV head) are merged by log-sum-exp:
// m* = max m_s, l = sum l_s 2^(m_s - m*), out = sum acc_s 2^(m_s - m*) / l,
// lse = ln 2 * (m* + log2 l).  The tensor-core kernel runs a unit's splits as one
// thread-block cluster when there are at most 8 and merges through distributed
// shared memory (cluster_merge); otherwise, and in the fp32 kernel, the last CTA
// of the unit to finish merges the partials it finds in the workspace
// (merge_if_last).
#include "attn_common.cuh"


namespace skv {
namespace {


template <typename T, int GM>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(const AttnArgs a) {
  pdl_wait();  // the selection is complete and visible
  constexpr int R = GM >= 4 ? 32 / GM : 8;  // rows per group
  constexpr int NV = R * GM;                // logits per group (8, 16 or 32)
  constexpr int LG_GM = GM == 1 ? 0 : GM == 2 ? 1 : GM == 4 ? 2 : GM == 8 ? 3 : 4;
  constexpr int LG_NV = NV == 8 ? 3 : NV == 16 ? 4 : 5;
  constexpr int SH = 5 - LG_NV;  // lane >> SH = value index after the butterfly
  constexpr size_t kRowBytes = kD * sizeof(T);

  __shared__ float sm_m[kWarps][GM], sm_l[kWarps][GM];
  __shared__ float sm_acc[kWarps][GM][kD];

  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const Regions rg = regions_of(L, a.ns, a.nl);
  const int n_list = rg.s_end + a.k + (L - rg.l_start);
  const int j0 = s * a.chunk;
  int j1 = j0 + a.chunk;
  j1 = j1 < n_list ? j1 : n_list;
  const int32_t* idx_row = a.idx + ((size_t)b * a.H + h) * a.k;

  // query slices, pre-scaled
  float qr[GM][4];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    if (g < a.G) {
      load4<T>(a.q + ((size_t)b * a.Hq + (size_t)h * a.G + g) * kRowBytes + lane * 4 * sizeof(T), qr[g]);
#pragma unroll
      for (int i = 0; i < 4; ++i) qr[g][i] *= a.scale_log2;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) qr[g][i] = 0.f;
    }
  }
  float acc[GM][4];
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[g][i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // for head (lane >> SH) % GM

  const int vidx = lane >> SH;
  const int my_r = vidx / GM;

  for (int base = j0 + warp * R; base < j1; base += kWarps * R) {
    // lanes < R resolve one row each
    const unsigned char* kp = nullptr;
    const unsigned char* vp = nullptr;
    bool ok = false;
    if (lane < R) {
      const int t = list_pos(a, idx_row, rg, base + lane, j1);
      if (t >= 0) {
        ok = resolve_row<T>(a, b, h, t, &kp, &vp);
        if (!ok) flag(a.status, SKV_DEV_BAD_SLOT);
      }
    }
    const unsigned okmask = __ballot_sync(0xffffffffu, ok);
    float kv[R][4], vv[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const unsigned long long kpr = __shfl_sync(0xffffffffu, (unsigned long long)kp, r);
      const unsigned long long vpr = __shfl_sync(0xffffffffu, (unsigned long long)vp, r);
      if (okmask >> r & 1u) {
        load4<T>((const unsigned char*)kpr + lane * 4 * sizeof(T), kv[r]);
        load4<T>((const unsigned char*)vpr + lane * 4 * sizeof(T), vv[r]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) kv[r][i] = vv[r][i] = 0.f;
      }
    }
    // partial logits, value index v = r * GM + g
    float part[NV];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) d = fmaf(qr[g][i], kv[r][i], d);
        part[r * GM + g] = d;
      }
    // butterfly reduce-scatter: after it, lane holds value (lane >> SH)
#pragma unroll
    for (int step = 0; step < LG_NV; ++step) {
      const int off = 16 >> step;
      const int half = NV >> (step + 1);
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = upper ? part[i] : part[i + half];
        const float keep = upper ? part[i + half] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
#pragma unroll
    for (int off = (1 << SH) >> 1; off >= 1; off >>= 1) part[0] += __shfl_xor_sync(0xffffffffu, part[0], off);
    const float z = (okmask >> my_r & 1u) ? part[0] : -INFINITY;
    // online softmax per head; lanes sharing a head differ in bits [SH+LG_GM, 5)
    float mx = z;
#pragma unroll
    for (int off = 1 << (SH + LG_GM); off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m_run, mx);
    const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
    const float p = z == -INFINITY ? 0.f : exp2f(z - m_new);
    float ps = p;
#pragma unroll
    for (int off = 1 << (SH + LG_GM); off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l_run = l_run * alpha + ps;
    m_run = m_new;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      const float ag = __shfl_sync(0xffffffffu, alpha, g << SH);
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[g][i] *= ag;
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        const float prg = __shfl_sync(0xffffffffu, p, (r * GM + g) << SH);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[g][i] = fmaf(prg, vv[r][i], acc[g][i]);
      }
  }

  // merge the warps of the CTA
  if (lane < GM << SH && (lane & ((1 << SH) - 1)) == 0) {
    const int g = lane >> SH;  // my_r == 0 lanes carry every head once
    sm_m[warp][g] = m_run;
    sm_l[warp][g] = l_run;
  }
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int i = 0; i < 4; ++i) sm_acc[warp][g][lane * 4 + i] = acc[g][i];
  __syncthreads();
  const int d = threadIdx.x;  // kThreads == kD
  for (int g = 0; g < a.G; ++g) {
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) ms = fmaxf(ms, sm_m[w][g]);
    float lsum = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = ms == -INFINITY ? 0.f : exp2f(sm_m[w][g] - ms);
      lsum += sm_l[w][g] * f;
      o += sm_acc[w][g][d] * f;
    }
    const size_t hq = (size_t)b * a.Hq + (size_t)h * a.G + g;
    a.ws_o[(hq * a.n_splits + s) * kD + d] = o;
    if (d == 0) {
      a.ws_ml[(hq * a.n_splits + s) * 2 + 0] = ms;
      a.ws_ml[(hq * a.n_splits + s) * 2 + 1] = lsum;
    }
  }
  merge_if_last(a, b, h, a.n_splits);
}

// ---------------------------------------------------------------------------- tensor-core path (bf16)
//
// attn_mma_kernel: one CTA (4 warps) per (split, KV head, request), bf16 storage.
// The split's list entries are walked in tiles of 64 rows.  All list entries of
// the split (at most kMaxChunk) are resolved through the slot table once, up
// front, into row references in shared memory; the 128 threads then gather the
// K and V rows of each tile (GPU pool, host pool or staging rows) with 16-byte
// cp.async copies (zero-filled for empty entries) into a ring of 2 (shallow) or
// 3 (deep) tile stages, swizzled so that ldmatrix reads are conflict-free.
// Warp w owns rows [16w, 16w+16) of every tile.  Groups of more than 8 heads
// (heads on the MMA's M side):
//   S[16 heads x 16 rows] = Q K^T   mma.m16n8k16 (heads padded to 16, K via ldmatrix)
//   O[16 heads x 128]    += P V     P re-packed from the S accumulators as the A
//                                   operand, V via ldmatrix.trans
// Groups of up to 8 heads (NARROW: the keys on the M side, half the MMAs):
//   S^T[16 rows x 8 heads] = K Q^T  K via ldmatrix as the A operand, Q^T held as B
//   O^T[128 x 8 heads]    += V^T P^T V^T via ldmatrix.trans as A, P^T as B after a
//                                   movmatrix.trans of each 8 x 8 block
// with an fp32 online softmax per head (exp2 units), running sums kept per thread.
// The four warps' (m, l, O) are merged in shared memory into one partial per
// query head, which stays in shared memory for the cluster merge or goes to the
// workspace for merge_if_last.

// The n_splits CTAs of one (request, KV head) as one thread-block cluster (at most
// kClusterMax splits): each CTA leaves its per-head partial (m, l, O) in its own shared
// memory; after a cluster barrier, CTA r merges heads r, r + S, ... by reading the S
// partials through distributed shared memory and writes out and lse; a second barrier
// keeps every CTA resident until the others have read its partial.  No workspace round
// trip, fence or ticket: the tail is two hardware barriers and S shared-memory loads.
// The arithmetic and its order are merge_if_last's.
constexpr int kClusterMax = 8;  // portable cluster size

__device__ __forceinline__ void cluster_merge(const AttnArgs& a, int b, int h, const float* cl_o,
                                              const float* cl_ml) {
  cluster_sync();  // every split's partial is in its CTA's shared memory
  const int S = a.n_splits;
  const uint32_t o_loc = smem_u32(cl_o), ml_loc = smem_u32(cl_ml);
  const int d = threadIdx.x;
  const size_t hq0 = (size_t)b * a.Hq + (size_t)h * a.G;
  for (int head = (int)cluster_rank(); head < a.G; head += S) {
    float m_s[kClusterMax], l_s[kClusterMax], o_s[kClusterMax];
#pragma unroll
    for (int s = 0; s < kClusterMax; ++s)
      if (s < S) {
        const uint32_t ml = dsmem_addr(ml_loc + (uint32_t)head * 8u, (uint32_t)s);
        m_s[s] = ld_dsmem_f32(ml);
        l_s[s] = ld_dsmem_f32(ml + 4u);
        o_s[s] = ld_dsmem_f32(dsmem_addr(o_loc + (uint32_t)(head * kD + d) * 4u, (uint32_t)s));
      }
    float ms = -INFINITY;
#pragma unroll
    for (int s = 0; s < kClusterMax; ++s)
      if (s < S) ms = fmaxf(ms, m_s[s]);
    float tot = 0.f;
#pragma unroll
    for (int s = 0; s < kClusterMax; ++s)
      if (s < S) {
        const float w = (ms == -INFINITY || m_s[s] == -INFINITY) ? 0.f : exp2f(m_s[s] - ms);
        tot += w * l_s[s];
        m_s[s] = w;
      }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    float o = 0.f;
#pragma unroll
    for (int s = 0; s < kClusterMax; ++s)
      if (s < S) o = fmaf(m_s[s], o_s[s], o);
    o *= inv;
    const size_t hq = hq0 + head;
    if (a.out_f32)
      ((float*)a.out)[hq * kD + d] = o;
    else
      ((__nv_bfloat16*)a.out)[hq * kD + d] = __float2bfloat16_rn(o);
    if (d == 0 && a.lse) a.lse[hq] = tot > 0.f ? kLn2 * (ms + log2f(tot)) : -INFINITY;
  }
  cluster_sync();  // the other CTAs have read this CTA's partial
}

template <int STAGES, bool CLUSTER, bool NARROW>
__global__ void __launch_bounds__(kThreads, tc::Ring<STAGES>::kCtasPerSm) attn_mma_kernel(const AttnArgs a) {
  constexpr int kStages = tc::Ring<STAGES>::kStages;
  constexpr int kMaxChunk = tc::Ring<STAGES>::kMaxChunk;
  // Before the selection is visible, only what no kernel of the step writes is read: the
  // lengths and the query (the CTA may already be resident while the selection runs).
  using namespace tc;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stages = smem;
  long long* rowref = (long long*)(smem + kStages * 2 * kTileBytes);  // [kMaxChunk]: row index | host bit, -1 empty
  uint32_t* vmask = (uint32_t*)(rowref + kMaxChunk);                   // [tiles][2]

  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int pool_h = h / a.pool.hdiv, pool_heads = a.H / a.pool.hdiv;  // the pool head of this row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const Regions rg = regions_of(L, a.ns, a.nl);
  const int n_list = rg.s_end + a.k + (L - rg.l_start);
  const int j0 = s * a.chunk;
  int j1 = j0 + a.chunk;
  j1 = j1 < n_list ? j1 : n_list;
  const int ntiles = j1 > j0 ? (j1 - j0 + kTileRows - 1) / kTileRows : 0;
  const int32_t* idx_row = a.idx + ((size_t)b * a.H + h) * a.k;

  // Q as the A operand: 16 heads x 128 dims, heads >= G are zero
  // NARROW (G <= 8): Q^T as the B operand instead, 128 dims x 8 heads, heads >= G zero
  uint32_t qa[NARROW ? 1 : 8][4];
  uint32_t qt[NARROW ? 8 : 1][2];
  {
    const __nv_bfloat16* qb = (const __nv_bfloat16*)a.q + ((size_t)b * a.Hq + (size_t)h * a.G) * kD;
    if constexpr (NARROW) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          qt[ks][r] = g < a.G ? *reinterpret_cast<const uint32_t*>(qb + (size_t)g * kD + 16 * ks + 2 * t4 + 8 * r)
                              : 0u;
    } else {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int head = g + ((r & 1) ? 8 : 0);
          const int col = 16 * ks + 2 * t4 + ((r & 2) ? 8 : 0);
          qa[ks][r] = head < a.G ? *reinterpret_cast<const uint32_t*>(qb + (size_t)head * kD + col) : 0u;
        }
    }
  }
  pdl_wait();  // the selection (and, with prefetch, the staging map) is complete and visible

  // resolve every list entry of this split once: row index in its pool (bit 62 = host pool).
  // Up to kMaxChunk / kThreads entries per thread, loads batched so they overlap.
  constexpr int kPer = kMaxChunk / kThreads;
  const int nres = ntiles * kTileRows;
  int tpos[kPer];
  if (a.bl.att != nullptr) {  // block-list mode: slots from the chosen blocks; the list is written here
    const BlockRegions brg = block_regions(L, a.bl.ns, a.bl.nl);
    const size_t unit_row = (size_t)b * a.H + h;
    const int32_t* chosen = a.bl.chosen + unit_row * a.bl.K;
    int32_t* att = a.bl.att + unit_row * a.k;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int jj = threadIdx.x + kThreads * u;
      tpos[u] = -1;
      if (jj < nres && j0 + jj < j1) {
        tpos[u] = block_list_token(chosen, a.bl.K, brg, L, j0 + jj, a.status);
        att[j0 + jj] = tpos[u];
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int jj = threadIdx.x + kThreads * u;
      tpos[u] = (jj < nres && j0 + jj < j1) ? list_pos(a, idx_row, rg, j0 + jj, j1) : -1;
    }
  }
  int ent[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u)
    ent[u] = tpos[u] >= 0 ? table_row(a.pool, b, pool_h, pool_heads)[tpos[u] / a.bs] : 0;
  // threshold prefetch: a host row the scoring pass staged this step (map tag epoch + 1) is
  // read from the staging rows in HBM instead of over the host link
  __shared__ uint32_t s_staged, s_read;
  const size_t unit = (size_t)b * a.H + h;
  uint32_t tag = 0;
  if (a.pf.map != nullptr) {
    tag = *a.pf.epoch + 1u;
    if (threadIdx.x == 0) s_staged = s_read = 0u;
  }
  unsigned long long mv[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u)
    mv[u] = (a.pf.map != nullptr && tpos[u] >= 0 && ent[u] < 0) ? a.pf.map[unit * a.max_len + tpos[u]] : 0ull;
  uint32_t n_staged = 0, n_read = 0;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int jj = threadIdx.x + kThreads * u;
    if (jj >= nres) break;  // uniform per warp: nres is a multiple of 64
    long long ref = -1;
    if (tpos[u] >= 0) {
      const int e = ent[u];
      const long long off = tpos[u] % a.bs;
      if (e >= 0 && e < a.pool.n_gpu) {
        ref = (long long)gpu_block_row(a.pool, e, pool_h, pool_heads, a.bs) + off;
      } else if (e < 0 && a.pool.host_k != nullptr && -(long long)e - 1 < a.pool.n_host) {
        ref = kHostBit | (((-(long long)e - 1) * pool_heads + pool_h) * a.bs + off);
        if (a.pf.map != nullptr) {
          const uint32_t slot = (uint32_t)(mv[u] & 0xFFFFFFFFull);
          if ((uint32_t)(mv[u] >> 32) == tag && slot < (uint32_t)a.pf.cap) {
            ref = kStageBit | (long long)(unit * a.pf.cap + slot);
            ++n_staged;
          } else {
            ++n_read;
          }
        }
      } else {
        flag(a.status, SKV_DEV_BAD_SLOT);
      }
    }
    rowref[jj] = ref;
    const unsigned m = __ballot_sync(0xffffffffu, ref >= 0);
    if (lane == 0) vmask[(jj / kTileRows) * 2 + ((jj / 32) & 1)] = m;
  }
  if (a.pf.stats != nullptr && a.pf.map != nullptr) {  // one atomic per counter per CTA
    __syncthreads();
    if (n_staged) atomicAdd(&s_staged, n_staged);
    if (n_read) atomicAdd(&s_read, n_read);
    __syncthreads();
    if (threadIdx.x == 0 && s_staged) atomicAdd(&a.pf.stats[0], s_staged);
    if (threadIdx.x == 0 && s_read) atomicAdd(&a.pf.stats[1], s_read);
  }
  __syncthreads();

  auto issue_tile = [&](int tile, int stage) {
    unsigned char* kd = stages + stage * 2 * kTileBytes;
    unsigned char* vd = kd + kTileBytes;
#pragma unroll
    for (int u = 0; u < kTileRows * 16 / kThreads; ++u) {
      const int c = threadIdx.x + kThreads * u;
      const int r = c >> 4, ch = c & 15;
      const long long ref = rowref[tile * kTileRows + r];
      const bool ok = ref >= 0;
      const bool host = (ref & kHostBit) != 0;
      const bool staged = (ref & kStageBit) != 0;
      const size_t row = (size_t)(ref & kRefRowMask);
      const unsigned char* kb = staged ? a.pf.staging : (const unsigned char*)(host ? a.pool.host_k : a.pool.gpu_k);
      const unsigned char* vb =
          staged ? a.pf.staging + a.pf_v_off : (const unsigned char*)(host ? a.pool.host_v : a.pool.gpu_v);
      const unsigned char* ks = ok ? kb + row * kRowBytes + ch * 16 : (const unsigned char*)a.pool.gpu_k;
      const unsigned char* vs = ok ? vb + row * kRowBytes + ch * 16 : (const unsigned char*)a.pool.gpu_k;
      cp_async16_zfill(kd + swz(r, ch), ks, ok);
      cp_async16_zfill(vd + swz(r, ch), vs, ok);
    }
  };

  for (int t = 0; t < kStages - 1; ++t) {
    if (t < ntiles) issue_tile(t, t % kStages);
    cp_async_commit();
  }

  constexpr int kOT = NARROW ? 8 : 16;  // O tiles: 8 dims x 16 heads, or (NARROW) 16 dims x 8 heads
  float o[kOT][4];
#pragma unroll
  for (int nt = 0; nt < kOT; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nt][c] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

  for (int i = 0; i < ntiles; ++i) {
    const int ti = i + kStages - 1;
    if (ti < ntiles) issue_tile(ti, ti % kStages);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncthreads();

    const unsigned char* kd = stages + (i % kStages) * 2 * kTileBytes;
    const unsigned char* vd = kd + kTileBytes;
    const unsigned long long mask = vmask[i * 2] | ((unsigned long long)vmask[i * 2 + 1] << 32);
    const uint32_t kbase = smem_u32(kd), vbase = smem_u32(vd);

    if constexpr (!NARROW) {
      float sacc[2][4];
  #pragma unroll
      for (int j = 0; j < 2; ++j) {
  #pragma unroll
        for (int c = 0; c < 4; ++c) sacc[j][c] = 0.f;
  #pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          const int row = 16 * warp + 8 * j + (lane & 7);
          const int ch = 4 * kp + (lane >> 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + swz(row, ch), b0, b1, b2, b3);
          mma_bf16(sacc[j], qa[2 * kp], b0, b1);
          mma_bf16(sacc[j], qa[2 * kp + 1], b2, b3);
        }
      }
      // online softmax per head row (hr 0: head g, hr 1: head g + 8)
      float p[2][4], mx[2] = {-INFINITY, -INFINITY};
  #pragma unroll
      for (int j = 0; j < 2; ++j)
  #pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int row = 16 * warp + 8 * j + 2 * t4 + (c & 1);
          const float z = ((mask >> row) & 1ull) ? sacc[j][c] * a.scale_log2 : -INFINITY;
          p[j][c] = z;
          mx[c >> 1] = fmaxf(mx[c >> 1], z);
        }
      float alpha[2];
  #pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
        mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
        const float m_new = fmaxf(m_r[hr], mx[hr]);
        alpha[hr] = m_new == -INFINITY ? 1.f : exp2f(m_r[hr] - m_new);
        m_r[hr] = m_new;
      }
      float ps[2] = {0.f, 0.f};
  #pragma unroll
      for (int j = 0; j < 2; ++j)
  #pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float z = p[j][c];
          const float e = z == -INFINITY ? 0.f : exp2f(z - m_r[c >> 1]);
          p[j][c] = e;
          ps[c >> 1] += e;
        }
  #pragma unroll
      for (int hr = 0; hr < 2; ++hr) l_r[hr] = l_r[hr] * alpha[hr] + ps[hr];
  #pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= alpha[0];
        o[nt][1] *= alpha[0];
        o[nt][2] *= alpha[1];
        o[nt][3] *= alpha[1];
      }
      uint32_t pa[4];
      pa[0] = pack_bf16(p[0][0], p[0][1]);
      pa[1] = pack_bf16(p[0][2], p[0][3]);
      pa[2] = pack_bf16(p[1][0], p[1][1]);
      pa[3] = pack_bf16(p[1][2], p[1][3]);
  #pragma unroll
      for (int np = 0; np < 8; ++np) {
        const int mi = lane >> 3;
        const int row = 16 * warp + 8 * (mi & 1) + (lane & 7);
        const int ch = 2 * np + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + swz(row, ch), b0, b1, b2, b3);
        mma_bf16(o[2 * np], pa, b0, b1);
        mma_bf16(o[2 * np + 1], pa, b2, b3);
      }

    } else {
      // S^T [16 keys x 8 heads] = K Q^T: the warp's 16 keys on the M side, the heads on N
      float st[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int mi = lane >> 3;
        const int row = 16 * warp + 8 * (mi & 1) + (lane & 7);
        const int ch = 2 * ks + (mi >> 1);
        uint32_t ka[4];
        ldsm_x4(kbase + swz(row, ch), ka[0], ka[1], ka[2], ka[3]);
        mma_bf16(st, ka, qt[ks][0], qt[ks][1]);
      }
      // online softmax per head column: this lane holds keys g and g + 8 of heads 2 t4
      // and 2 t4 + 1 (hr 0, 1); a head's keys are spread over the lanes of equal t4
      const bool v0 = (mask >> (16 * warp + g)) & 1ull, v1 = (mask >> (16 * warp + g + 8)) & 1ull;
      float z[4];
      z[0] = v0 ? st[0] * a.scale_log2 : -INFINITY;
      z[1] = v0 ? st[1] * a.scale_log2 : -INFINITY;
      z[2] = v1 ? st[2] * a.scale_log2 : -INFINITY;
      z[3] = v1 ? st[3] * a.scale_log2 : -INFINITY;
      float mx[2] = {fmaxf(z[0], z[2]), fmaxf(z[1], z[3])};
      float alpha[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], off));
        const float m_new = fmaxf(m_r[hr], mx[hr]);
        alpha[hr] = m_new == -INFINITY ? 1.f : exp2f(m_r[hr] - m_new);
        m_r[hr] = m_new;
      }
      float pv[4], ps[2] = {0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        pv[c] = z[c] == -INFINITY ? 0.f : exp2f(z[c] - m_r[c & 1]);
        ps[c & 1] += pv[c];
      }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) l_r[hr] = l_r[hr] * alpha[hr] + ps[hr];
#pragma unroll
      for (int mt = 0; mt < kOT; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0];
        o[mt][3] *= alpha[1];
      }
      // P^T [16 keys x 8 heads] as the B operand: each 8 x 8 block transposed in registers
      const uint32_t pb0 = movmatrix_t(pack_bf16(pv[0], pv[1]));  // keys 0-7
      const uint32_t pb1 = movmatrix_t(pack_bf16(pv[2], pv[3]));  // keys 8-15
      // O^T [128 dims x 8 heads] += V^T P^T, V^T via ldmatrix.trans
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int mi = lane >> 3;
        const int row = 16 * warp + 8 * (mi >> 1) + (lane & 7);
        const int ch = 2 * mt + (mi & 1);
        uint32_t va[4];
        ldsm_x4_t(vbase + swz(row, ch), va[0], va[1], va[2], va[3]);
        mma_bf16(o[mt], va, pb0, pb1);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // merge the four warps: smem reused as [4][16][128] O and [4][16][2] (m, l)
  float* sm_o = (float*)smem;
  float* sm_ml = sm_o + kWarps * 16 * kD;
  if constexpr (NARROW) {  // heads 2 t4 + hr; a head's row sums spread over the lanes of equal t4
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
#pragma unroll
      for (int off = 4; off <= 16; off <<= 1) l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], off);
#pragma unroll
    for (int mt = 0; mt < kOT; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        sm_o[(warp * 16 + 2 * t4 + (c & 1)) * kD + 16 * mt + g + ((c >> 1) ? 8 : 0)] = o[mt][c];
    if (g == 0) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        sm_ml[(warp * 16 + 2 * t4 + hr) * 2 + 0] = m_r[hr];
        sm_ml[(warp * 16 + 2 * t4 + hr) * 2 + 1] = l_r[hr];
      }
    }
  } else {  // heads g + 8 hr; a head's row sums spread over its lane quad
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 1);
      l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 2);
    }
#pragma unroll
    for (int nt = 0; nt < kOT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int head = g + ((c >> 1) ? 8 : 0);
        sm_o[(warp * 16 + head) * kD + 8 * nt + 2 * t4 + (c & 1)] = o[nt][c];
      }
    if (t4 == 0) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        sm_ml[(warp * 16 + g + 8 * hr) * 2 + 0] = m_r[hr];
        sm_ml[(warp * 16 + g + 8 * hr) * 2 + 1] = l_r[hr];
      }
    }
  }
  __syncthreads();
  const int d = threadIdx.x;
  float* cl_o = sm_ml + kWarps * 16 * 2;  // [16][kD] this split's partial per head (cluster merge)
  float* cl_ml = cl_o + 16 * kD;          // [16][2]
  for (int head = 0; head < a.G; ++head) {
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) ms = fmaxf(ms, sm_ml[(w * 16 + head) * 2]);
    float lsum = 0.f, ov = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = ms == -INFINITY ? 0.f : exp2f(sm_ml[(w * 16 + head) * 2] - ms);
      lsum += sm_ml[(w * 16 + head) * 2 + 1] * f;
      ov += sm_o[(w * 16 + head) * kD + d] * f;
    }
    if constexpr (CLUSTER) {
      cl_o[head * kD + d] = ov;
      if (d == 0) {
        cl_ml[head * 2 + 0] = ms;
        cl_ml[head * 2 + 1] = lsum;
      }
    } else {
      const size_t hq = (size_t)b * a.Hq + (size_t)h * a.G + head;
      a.ws_o[(hq * a.n_splits + s) * kD + d] = ov;
      if (d == 0) {
        a.ws_ml[(hq * a.n_splits + s) * 2 + 0] = ms;
        a.ws_ml[(hq * a.n_splits + s) * 2 + 1] = lsum;
      }
    }
  }
  if constexpr (CLUSTER)
    cluster_merge(a, b, h, cl_o, cl_ml);
  else
    merge_if_last(a, b, h, a.n_splits);
}

// Ends a step with threshold prefetch (paged path): once the attention has read the map
// and the staging rows, advance the step tag and empty every row's staging slots.
__global__ void __launch_bounds__(256) prefetch_end_kernel(const PrefetchView pf, int rows) {
  pdl_wait();
  if (threadIdx.x == 0) *pf.epoch += 1u;
  for (int r = threadIdx.x; r < rows; r += blockDim.x) pf.count[r] = 0u;
}

// ---------------------------------------------------------------------------- gather

template <typename T>
__global__ void gather_kernel(const AttnArgs a, int n_att, int d_k, int d_v, unsigned char* k_out,
                              unsigned char* v_out) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const long long total = (long long)a.B * a.H * n_att;
  if (warp >= total) return;
  const int j = (int)(warp % n_att);
  const int bh = (int)(warp / n_att);
  const int b = bh / a.H, h = bh % a.H;
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const Regions rg = regions_of(L, a.ns, a.nl);
  const int n_list = rg.s_end + a.k + (L - rg.l_start);
  const int32_t* idx_row = a.idx + ((size_t)b * a.H + h) * a.k;
  const int t = list_pos(a, idx_row, rg, j, n_list);
  const unsigned char* kp = nullptr;
  const unsigned char* vp = nullptr;
  bool ok = false;
  if (t >= 0) {
    const int e = table_row(a.pool, b, h / a.pool.hdiv, a.H / a.pool.hdiv)[t / a.bs];
    const size_t off = (size_t)(t % a.bs);
    const bool latent = a.pool.gpu_v == nullptr;
    if (e >= 0 && e < a.pool.n_gpu) {
      const size_t r = gpu_block_row(a.pool, e, h / a.pool.hdiv, a.H / a.pool.hdiv, a.bs) + off;
      kp = (const unsigned char*)a.pool.gpu_k + r * d_k * sizeof(T);
      vp = latent ? kp : (const unsigned char*)a.pool.gpu_v + r * d_v * sizeof(T);
      ok = true;
    } else if (e < 0 && a.pool.host_k != nullptr && (-(long long)e - 1) < a.pool.n_host) {
      const size_t r = ((size_t)(-(long long)e - 1) * (a.H / a.pool.hdiv) + h / a.pool.hdiv) * a.bs + off;
      kp = (const unsigned char*)a.pool.host_k + r * d_k * sizeof(T);
      vp = latent ? kp : (const unsigned char*)a.pool.host_v + r * d_v * sizeof(T);
      ok = true;
    } else {
      flag(a.status, SKV_DEV_BAD_SLOT);
    }
  }
  const size_t orow = (size_t)warp;
  uint4* kd = (uint4*)(k_out + orow * d_k * sizeof(T));
  const int nk = d_k * (int)sizeof(T) / 16;
  for (int c = lane; c < nk; c += 32) kd[c] = ok ? ((const uint4*)kp)[c] : make_uint4(0, 0, 0, 0);
  if (v_out) {
    uint4* vd = (uint4*)(v_out + orow * d_v * sizeof(T));
    const int nv = d_v * (int)sizeof(T) / 16;
    for (int c = lane; c < nv; c += 32) vd[c] = ok ? ((const uint4*)vp)[c] : make_uint4(0, 0, 0, 0);
  }
}


template <typename T, int GM>
skv_status launch_split(const AttnArgs& a, cudaStream_t st) {
  dim3 grid(a.n_splits, a.H, a.B);
  if (launch_dependent(attn_split_kernel<T, GM>, grid, dim3(kThreads), 0, st, 1, a) != cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

// Whether the tensor-core kernel runs a unit's splits as one cluster.  Clusters are
// placed whole inside a GPC, so fewer CTAs may be resident at once than without them;
// the cluster merge is taken when its launch needs no more waves than the plain one
// (measured on gqa32b: 4-CTA clusters of the deep ring, one wave either way, attention
// 39.7 -> 31.9 us; the shallow ring's 7-CTA clusters spill into a second wave, 44 us).
// A choice per device, not per problem: the workspace keeps the plain path's layout.
template <int STAGES, bool NARROW>
skv_status use_cluster(const AttnArgs& a, bool* cluster) {
  constexpr int kSmem = tc::Ring<STAGES>::kSmemBytes;
  *cluster = false;
  if (a.n_splits > kClusterMax) return SKV_OK;
  int per_sm = 0, clusters = 0;
  skv_status r = prepare_kernel((const void*)attn_mma_kernel<STAGES, false, NARROW>, kSmem, kThreads, &per_sm);
  if (r != SKV_OK) return r;
  r = prepare_kernel((const void*)attn_mma_kernel<STAGES, true, NARROW>, kSmem);
  if (r != SKV_OK) return r;
  r = max_active_clusters((const void*)attn_mma_kernel<STAGES, true, NARROW>, kSmem, kThreads, a.n_splits,
                          &clusters);
  if (r != SKV_OK) return r;
  if (clusters < 1) return SKV_OK;
  const long long units = (long long)a.B * a.H;
  const long long slots = (long long)per_sm * num_sms();
  *cluster = (units + clusters - 1) / clusters <= (units * a.n_splits + slots - 1) / slots;
  return SKV_OK;
}

// The tensor-core kernel, with the splits of a unit as one cluster (CLUSTER) or merged
// by the last CTA through the workspace.
template <int STAGES, bool CLUSTER, bool NARROW>
skv_status launch_mma(const AttnArgs& a, cudaStream_t st) {
  constexpr int kSmem = tc::Ring<STAGES>::kSmemBytes;
  const skv_status prep = prepare_kernel((const void*)attn_mma_kernel<STAGES, CLUSTER, NARROW>, kSmem);
  if (prep != SKV_OK) return prep;
  if (launch_dependent(attn_mma_kernel<STAGES, CLUSTER, NARROW>, dim3(a.n_splits, a.H, a.B), dim3(kThreads), kSmem,
                       st, CLUSTER ? a.n_splits : 1, a) != cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

// The ring, the merge form and the MMA orientation: 2 x 2 x 2 kernels.
template <int STAGES>
skv_status launch_mma_ring(const AttnArgs& a, bool cluster, cudaStream_t st) {
  const bool narrow = a.G <= 8;
  if (cluster) return narrow ? launch_mma<STAGES, true, true>(a, st) : launch_mma<STAGES, true, false>(a, st);
  return narrow ? launch_mma<STAGES, false, true>(a, st) : launch_mma<STAGES, false, false>(a, st);
}

template <typename T>
skv_status launch_split_g(const AttnArgs& a, cudaStream_t st) {
  if (a.G <= 1) return launch_split<T, 1>(a, st);
  if (a.G <= 2) return launch_split<T, 2>(a, st);
  if (a.G <= 4) return launch_split<T, 4>(a, st);
  if (a.G <= 8) return launch_split<T, 8>(a, st);
  return launch_split<T, 16>(a, st);
}

}  // namespace

int attn_splits_requested(const skv_problem& p) {
  const int n = max_list(p);
  if (p.n_splits > 0) {
    int sp = p.n_splits < (n > 0 ? n : 1) ? p.n_splits : (n > 0 ? n : 1);
    return sp < kMergeMax ? sp : kMergeMax;
  }
  // Sized for the 152 SMs of a GB300 from the problem alone (the workspace size
  // must not depend on the device): the tensor-core kernel keeps 2 CTAs per SM,
  // aim at about two waves with at least one 64-row tile per split; the fp32
  // kernel aims at about 8 CTAs per SM.
  const long long units = (long long)p.batch * p.n_kv_heads;
  const long long target = p.dtype == SKV_DTYPE_F32 ? 8LL * 152 : 4LL * 152;
  long long want = (target + units - 1) / units;
  long long cap = (n + 63) / 64;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (int)want;
}

// The tensor-core kernel resolves a split's entries up front, so a split holds at
// most its ring's kMaxChunk entries.  Without a requested count, the split count S is
// the smallest that minimises waves(S) x (tiles per CTA(S) + kCtaOverheadTiles) with the
// ring's resident CTAs (3 or 2) on each of the 152 SMs of a GB300 (a function of the
// problem alone, so the workspace size does not depend on the device).  The overhead term is a CTA's
// fixed cost (resolving its entries, prologue, merge ticket) in tiles: measured near
// 3 on GB300; without it the count drifts to one tile per CTA, 2.5x slower at large k.
constexpr long long kCtaOverheadTiles = 3;

// The deep ring when a unit's list is longer than one shallow CTA holds and the fewest
// splits the deep ring allows fit one wave at its 2 CTAs a SM (measured: gqa32b step
// 131.3 -> 129.9 us; block selection +3 %; B1 x 32K x k4096 and the B4 points with k of
// 1,024 or more +2-8 %; many-unit problems lose when pushed into a second wave, and lists
// that fit one CTA lose about 1-2 %, so both keep the shallow ring).  A function of the
// problem alone, like the split count.
bool attn_deep_ring(const skv_problem& p) {
  const int n = max_list(p);
  const long long units = (long long)p.batch * p.n_kv_heads;
  const long long need = n > 0 ? (n + tc::Ring<3>::kMaxChunk - 1) / tc::Ring<3>::kMaxChunk : 1;
  return p.dtype != SKV_DTYPE_F32 && p.n_splits == 0 && n > tc::Ring<2>::kMaxChunk &&
         units * need <= (long long)tc::Ring<3>::kCtasPerSm * 152;
}

int attn_splits(const skv_problem& p) {
  const int n = max_list(p);
  if (p.dtype == SKV_DTYPE_F32) return attn_splits_requested(p);
  const bool deep = attn_deep_ring(p);
  const int max_chunk = deep ? tc::Ring<3>::kMaxChunk : tc::Ring<2>::kMaxChunk;
  const int need = n > 0 ? (n + max_chunk - 1) / max_chunk : 1;
  if (p.n_splits > 0) {
    int sp = p.n_splits < (n > 0 ? n : 1) ? p.n_splits : (n > 0 ? n : 1);
    sp = sp < kMergeMax ? sp : kMergeMax;
    return sp < need ? need : sp;
  }
  const long long units = (long long)p.batch * p.n_kv_heads;
  const long long slots = (long long)(deep ? tc::Ring<3>::kCtasPerSm : tc::Ring<2>::kCtasPerSm) * 152;
  const int hi = n > 0 ? (n + tc::kTileRows - 1) / tc::kTileRows : 1;
  int best = need;
  long long best_cost = -1;
  for (int sp = need; sp <= hi; ++sp) {
    const long long waves = (units * sp + slots - 1) / slots;
    const long long per = ((n + sp - 1) / sp + tc::kTileRows - 1) / tc::kTileRows;
    const long long cost = waves * (per + kCtaOverheadTiles);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = sp;
    }
  }
  return best;
}

size_t attn_workspace_bytes(const skv_problem& p) {
  if (latent_shape(p)) return latent_workspace_bytes(p);
  const size_t S = (size_t)attn_splits(p);
  const size_t hq = (size_t)p.batch * p.n_q_heads;
  return align256(hq * S * p.d_v * 4) + align256(hq * S * 2 * 4) + align256((size_t)p.batch * p.n_kv_heads * 4);
}

uint32_t* attn_tickets(const skv_problem& p, void* ws) {
  if (latent_shape(p)) return nullptr;  // the latent path merges in a kernel of its own
  const size_t S = (size_t)attn_splits(p);
  const size_t hq = (size_t)p.batch * p.n_q_heads;
  return (uint32_t*)((unsigned char*)ws + align256(hq * S * p.d_v * 4) + align256(hq * S * 2 * 4));
}

skv_status launch_attn(const skv_problem& p, const void* q, const PoolView& pool, const int32_t* idx, void* out,
                       float* lse, void* ws, int32_t* status, cudaStream_t st, bool tickets_zeroed,
                       const PrefetchView* pf, const BlockListView* bl) {
  if (pool.gpu_v == nullptr) return launch_attn_latent(p, q, pool, idx, out, lse, ws, status, st, pf);
  AttnArgs a = make_args(p, q, pool, idx, status);
  if (pf != nullptr) {  // staged host rows (bf16 tensor-core path only): K rows, then V rows, [rows, cap] each
    if (p.dtype != SKV_DTYPE_BF16 || p.d_qk != p.d_v) return SKV_ERR_UNSUPPORTED;
    a.pf = *pf;
    a.pf_v_off = (size_t)p.batch * p.n_kv_heads * (size_t)pf->cap * p.d_qk * 2;
  }
  if (bl != nullptr) {  // block-list mode: the bf16 tensor-core kernel only, no sink / local windows
    if (p.dtype != SKV_DTYPE_BF16 || p.n_sink != 0 || p.n_local != 0 || bl->att == nullptr)
      return SKV_ERR_UNSUPPORTED;
    a.bl = *bl;
  }
  a.n_splits = attn_splits(p);
  const int n = max_list(p);
  a.chunk = n > 0 ? (n + a.n_splits - 1) / a.n_splits : 1;
  const size_t hq = (size_t)p.batch * p.n_q_heads;
  a.ws_o = (float*)ws;
  a.ws_ml = (float*)((unsigned char*)ws + align256(hq * a.n_splits * p.d_v * 4));
  a.tickets = (uint32_t*)((unsigned char*)a.ws_ml + align256(hq * a.n_splits * 2 * 4));
  a.out = out;
  a.lse = lse;
  if (a.tickets != attn_tickets(p, ws)) return SKV_ERR_INVALID_ARGUMENT;  // one layout, two readers
  // the bf16 kernel may merge a unit's splits inside a cluster: then no tickets
  const bool deep = p.dtype != SKV_DTYPE_F32 && attn_deep_ring(p);
  bool cluster = false;
  if (p.dtype != SKV_DTYPE_F32) {
    const bool narrow = a.G <= 8;
    const skv_status r = deep ? (narrow ? use_cluster<3, true>(a, &cluster) : use_cluster<3, false>(a, &cluster))
                              : (narrow ? use_cluster<2, true>(a, &cluster) : use_cluster<2, false>(a, &cluster));
    if (r != SKV_OK) return r;
  }
  if (!cluster && !tickets_zeroed &&
      cudaMemsetAsync(a.tickets, 0, (size_t)p.batch * p.n_kv_heads * 4, st) != cudaSuccess)
    return SKV_ERR_CUDA;
  if (p.dtype == SKV_DTYPE_F32) {
    skv_status r = launch_split_g<float>(a, st);
    if (r != SKV_OK) return r;
  } else {
    const skv_status r = deep ? launch_mma_ring<3>(a, cluster, st) : launch_mma_ring<2>(a, cluster, st);
    if (r != SKV_OK) return r;
    if (pf != nullptr) {  // the step is over: the next one stages under a new tag into empty slots
      if (launch_dependent(prefetch_end_kernel, dim3(1), dim3(256), 0, st, 1, a.pf, p.batch * p.n_kv_heads) !=
          cudaSuccess)
        return SKV_ERR_CUDA;
      SKV_LAUNCH_CHECK();
    }
  }
  return SKV_OK;
}

skv_status launch_gather(const skv_problem& p, const PoolView& pool, const int32_t* idx, void* k_out, void* v_out,
                         int32_t* status, cudaStream_t st) {
  AttnArgs a = make_args(p, nullptr, pool, idx, status);
  const int n_att = max_list(p);
  const long long warps = (long long)p.batch * p.n_kv_heads * n_att;
  if (warps == 0) return SKV_OK;
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  if (p.dtype == SKV_DTYPE_F32)
    gather_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(a, n_att, p.d_qk, p.d_v, (unsigned char*)k_out,
                                                              (unsigned char*)v_out);
  else
    gather_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, st>>>(a, n_att, p.d_qk, p.d_v,
                                                                      (unsigned char*)k_out, (unsigned char*)v_out);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace skv
