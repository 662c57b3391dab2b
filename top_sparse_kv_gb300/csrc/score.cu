// S0 + S1: group-query scoring of every candidate key (sm_103a).
//
// s_t = <q_bar, k_t> with q_bar the mean of the group's scoring-query heads
// (ParisKV notes, §1 Eqs. (1)-(3); ECHO-OSDI26 wiki, core method 3 -- the
// indexer scores every history key; OasisKV notes §3.2 -- one ranking per KV head).
//
// Design: the key stream is the dominant HBM traffic of the whole step, so this
// kernel is a pure bandwidth pump.  Keys are moved in 16-token tiles (4 KB in
// bf16): one paged block of one head, or 16 rows of the contiguous index.  A
// producer warp issues 1-D bulk copies (cp.async.bulk, TMA engine) into a
// 4-stage shared-memory ring guarded by mbarriers (full: transaction bytes,
// empty: one arrival per consuming warp).  One pair of consumer warps takes every
// tile; in the pair, four lanes share each of the tile's 16 rows, read their 64
// bytes of it with 128-bit shared loads, multiply by the fp32 group query held in
// registers and reduce with two shuffles.  The CTA is small so that ten share an
// SM: the read rate of bulk copies follows the number of CTAs issuing them.  Work items are
// 512-token slices of one (request, head) row (shorter, down to 32 tokens, when the
// rows would leave CTA slots idle), distributed over a persistent grid sized to the
// resident-CTA capacity of the device.  Host-resident blocks
// (negative slot entries) are read in place through UVA by the consumers.
//
// The max reading (a key scores its largest logit over the group's heads) keeps
// one dot product per head, G flops per key byte -- a contraction that would
// saturate the CUDA cores at HBM speed -- so its consumers use mma.sync tiles
// instead: 16 keys x 8 heads per instruction, fp32 accumulation (see below).
#include "skv_internal.cuh"

namespace skv {
namespace {

constexpr int kTileTokens = 16;
// A CTA: one producer warp, kConsumerWarps consumer warps, a ring of kStages tiles.  The
// key stream's rate follows the number of CTAs an SM holds more than their ring depth: a
// data-movement probe of random 4 KB tiles read by bulk copies measured 6.0 TB/s with 6
// CTAs of 4 or 8 stages a SM and 7.0 TB/s with 10 CTAs of 4 stages.  So the CTA is kept
// small -- two consumer warps, four stages -- and ten share an SM.
constexpr int kConsumerWarps = 2;
constexpr int kScoreThreads = 32 * (1 + kConsumerWarps);
constexpr int kStages = 4;
constexpr int kPairs = kConsumerWarps / 2;  // CUDA-core consumers: a warp pair scores a tile
constexpr int kTilesPerItem = 32;    // tiles a work item covers when the rows fill the GPU
constexpr int kMinTilesPerItem = 2;  // ... and the fewest when they do not
constexpr int kD = 128;
constexpr int kPfList = 512;                    // staging requests a CTA can hold per launch
constexpr int kPfBatch = 4;                     // rows a prefetch warp moves at a time
// prefetch warps a CTA (the template's PF): request chunk c goes to warp c % PF.  Two for the
// latent layout, whose host rows (1,152 bytes, 75 % of the attended rows) keep the link busy;
// one for paged pools, whose few host rows a step need no second warp, so the CTAs keep more
// of the SM's registers for the key stream.
constexpr int kPfChunks = 96;                   // 16-byte chunks of a staged row, at most (1,536 B)
constexpr long long kPfSpinCycles = 4000000000LL;  // the prefetch warp's idle limit (~2 s)

struct ScoreArgs {
  const unsigned char* q;  // [B, n_idx_q, kD]
  int n_idx_q;
  int gi;  // scoring heads per KV head
  int H;
  int layout;
  const unsigned char* contig;  // [B, H, max_len, kD]
  PoolView pool;
  const int32_t* seq_lens;
  int B, max_len, ns, nl;
  float* scores;  // [B, H, max_len]
  int32_t* status;
  int agg;        // SKV_AGG_MEAN | SKV_AGG_MAX (tensor-core consumers only)
  float inv_gi;   // 1 / gi
  PrefetchView pf;  // threshold prefetch (the PF variant only)
  int pf_row_bytes;
  int pf_v_bytes;     // bytes of a staged V row (paged pools), 0 when V is part of the K row
  size_t pf_v_off;    // byte offset of the V staging rows inside the staging area
  int tiles_per_item;
  int items_per_row;
  int total_items;
};

struct Item {
  int row, b, h, j_lo, j_hi, s_end, l_start;
};

__device__ __forceinline__ Item item_of(const ScoreArgs& a, int w) {
  Item it;
  it.row = w / a.items_per_row;
  int c = w - it.row * a.items_per_row;
  it.b = it.row / a.H;
  it.h = it.row - it.b * a.H;
  int L = load_len(a.seq_lens, it.b, a.max_len, a.status);
  Regions r = regions_of(L, a.ns, a.nl);
  it.s_end = r.s_end;
  it.l_start = r.l_start;
  int lo = c * a.tiles_per_item, hi = lo + a.tiles_per_item;
  int jl = r.s_end / kTileTokens;
  int jh = (r.l_start + kTileTokens - 1) / kTileTokens;
  it.j_lo = lo > jl ? lo : jl;
  it.j_hi = hi < jh ? hi : jh;
  if (r.l_start <= r.s_end) it.j_hi = it.j_lo;  // no candidates
  return it;
}

// four consecutive query elements as fp32 (8 bytes of bf16, or 16 of fp32)
template <typename T>
__device__ __forceinline__ void load_q4(const unsigned char* p, float* v) {
  if constexpr (sizeof(T) == 2) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const float4 f = *reinterpret_cast<const float4*>(p);
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  }
}

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// NTILE = 0: CUDA-core consumers (the mean reading, any group size, bf16 or fp32).
// NTILE = 1, 2: tensor-core consumers for bf16, up to 8 * NTILE scoring heads (both readings;
// used for the max, where each key needs one dot product per head).
// HEADS (per query head, tensor-core consumers): every head's dot product goes to its own
// scores row instead of being combined.
template <typename T, int NTILE, int PF, bool HEADS = false>
__device__ __forceinline__ void score_body(const ScoreArgs& a) {
  constexpr int kRowBytes = kD * (int)sizeof(T);
  constexpr int kTileBytes = kTileTokens * kRowBytes;
  constexpr int kChunks = kRowBytes / 16;    // 16-byte chunks per row
  constexpr int kEpc = Vec<T>::N;            // elements per chunk
  constexpr int kCL = kChunks / 4;           // chunks per lane (4 lanes per row)

  extern __shared__ __align__(128) unsigned char stage_mem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ const unsigned char* stage_src[kStages];
  __shared__ volatile int s_abort;  // set when any wait gives up; later waits return at once
  // the item's group query (CUDA-core consumers), written by the producer warp, two items deep
  __shared__ __align__(16) float q_bar[2][kD];
  __shared__ __align__(8) uint64_t q_full[2];   // the producer warp's 32 lanes arrive
  __shared__ __align__(8) uint64_t q_empty[2];  // the consumer threads arrive
  // threshold prefetch: positions the consumers hand to the prefetch warp
  __shared__ int2 pf_list[PF ? kPfList : 1];
  __shared__ volatile int pf_ready[PF ? kPfList : 1];
  __shared__ unsigned pf_n;
  __shared__ volatile int pf_done;

  pdl_release();  // the selection may be placed on SMs as this grid drains; it waits for completion
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], NTILE ? 1 : 2);  // the consumer warp (pair) that owns this stage
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&q_full[q], 32);
      mbar_init(&q_empty[q], 32 * kConsumerWarps);
    }
    fence_barrier_init();
    s_abort = 0;
    pf_n = 0;
    pf_done = 0;
  }
  if (PF)
    for (int i = threadIdx.x; i < kPfList; i += blockDim.x) pf_ready[i] = 0;
  __syncthreads();

  if (PF && warp >= 1 + kConsumerWarps) {
    // ---------------------------------------------------------- prefetch warp
    // Copies the host rows of the positions the consumers list (keys scoring above
    // the row's predicted threshold) into the row's staging slots and tags the map;
    // stops when every consumer warp is done and the list is drained, or after an
    // idle limit (then it flags a timeout).
    const unsigned long long tag = (unsigned long long)(*a.pf.epoch + 1u) << 32;
    const int kch = a.pf_row_bytes / 16;          // 16-byte chunks of the K row ...
    const int chunks = kch + (PF == 1 ? a.pf_v_bytes / 16 : 0);  // ... then of the V row (paged pools)
    const unsigned pw = (unsigned)(warp - 1 - kConsumerWarps);
    unsigned next = pw * kPfBatch;  // this warp's requests: chunks of kPfBatch, every PF-th
    long long idle_from = -1;
    for (;;) {
      const int consumers_done = pf_done;
      unsigned n = *(volatile unsigned*)&pf_n;
      n = n < (unsigned)kPfList ? n : (unsigned)kPfList;
      // up to kPfBatch ready requests at a time: all their host loads in flight before any store
      const unsigned chunk_end = (next / kPfBatch + 1) * kPfBatch;
      int nb = 0;
      while (next + nb < chunk_end && next + nb < n && pf_ready[next + nb]) ++nb;
      if (nb > 0) {
        idle_from = -1;
        // one prefetch warp serves paged pools of 16-token blocks (a K and a V row a token), two
        // the latent layout (a per-token map; one row a token, whose V is its leading part)
        constexpr bool kPaged = PF == 1;
        constexpr int kBs = kPaged ? kTileTokens : 1;
        // per request: its K row's source and staging copy (null: nothing to copy), the same for
        // its V row (paged pools), its map entry
        const uint4* src[kPfBatch];
        uint4* dst[kPfBatch];
        const uint4* srcv[kPfBatch];
        uint4* dstv[kPfBatch];
        unsigned long long* mp[kPfBatch];
        unsigned slot[kPfBatch];
        // lane i < nb resolves request next + i at once: its table entry and, for a host
        // row, a staging slot (one round trip for the batch's table loads, one for its atomics)
        int row_l = 0, t_l = 0, e_l = 0;
        unsigned sl_l = 0xFFFFFFFFu;  // no slot: not a host row
        if (lane < nb) {
          const int2 req = pf_list[next + lane];
          row_l = req.x;
          t_l = req.y;
          e_l = a.pool.table[(size_t)(row_l / a.H) * a.pool.stride + t_l / kBs];
          const long long hb_l = -(long long)e_l - 1;
          if (e_l < 0 && a.pool.host_k != nullptr && hb_l < a.pool.n_host) sl_l = atomicAdd(&a.pf.count[row_l], 1u);
        }
#pragma unroll
        for (int i = 0; i < kPfBatch; ++i) {
          src[i] = nullptr;
          const int row = __shfl_sync(0xffffffffu, row_l, i);
          const int t = __shfl_sync(0xffffffffu, t_l, i);
          const int e = __shfl_sync(0xffffffffu, e_l, i);
          const unsigned sl = __shfl_sync(0xffffffffu, sl_l, i);
          if (i >= nb || sl == 0xFFFFFFFFu) continue;  // past the batch, or not a host row
          if (sl >= (unsigned)a.pf.cap) continue;       // this row's staging is full: it is read later
          const int b = row / a.H, h = row - b * a.H;
          const long long hb = -(long long)e - 1;
          slot[i] = sl;
          const size_t hrow = ((size_t)hb * a.H + h) * kBs + (size_t)(t % kBs);  // the token's host row
          const size_t srow = (size_t)row * a.pf.cap + sl;                         // its staging row
          src[i] = (const uint4*)((const unsigned char*)a.pool.host_k + hrow * (size_t)a.pf_row_bytes);
          dst[i] = (uint4*)(a.pf.staging + srow * (size_t)a.pf_row_bytes);
          if constexpr (kPaged) {
            srcv[i] = (const uint4*)((const unsigned char*)a.pool.host_v + hrow * (size_t)a.pf_v_bytes);
            dstv[i] = (uint4*)(a.pf.staging + a.pf_v_off + srow * (size_t)a.pf_v_bytes);
          }
          mp[i] = a.pf.map + (size_t)row * a.max_len + t;
        }
        next += nb;
        if (next == chunk_end) next += (PF - 1) * kPfBatch;  // on to this warp's next chunk
        uint4 v[kPfBatch][kPfChunks / 32];
#pragma unroll
        for (int i = 0; i < kPfBatch; ++i)
#pragma unroll
          for (int u = 0; u < kPfChunks / 32; ++u) {
            const int c = lane + 32 * u;
            if (src[i] == nullptr || c >= chunks) continue;
            if constexpr (kPaged) {  // K row chunks, then V row chunks
              v[i][u] = c < kch ? src[i][c] : srcv[i][c - kch];
            } else {
              v[i][u] = src[i][c];
            }
          }
#pragma unroll
        for (int i = 0; i < kPfBatch; ++i) {
          if (src[i] == nullptr) continue;
#pragma unroll
          for (int u = 0; u < kPfChunks / 32; ++u) {
            const int c = lane + 32 * u;
            if (c >= chunks) continue;
            if constexpr (kPaged) {
              if (c < kch)
                dst[i][c] = v[i][u];
              else
                dstv[i][c - kch] = v[i][u];
            } else {
              dst[i][c] = v[i][u];
            }
          }
          if (lane == 0) *mp[i] = tag | slot[i];
        }
        continue;
      }
      if (next >= n && consumers_done == kConsumerWarps) break;  // every request has been seen
      const long long now = clock64();
      if (idle_from < 0) idle_from = now;
      if (now - idle_from > kPfSpinCycles) {
        if (lane == 0) flag(a.status, SKV_DEV_TIMEOUT);
        break;
      }
      __nanosleep(200);
    }
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp prepares an item: lane i resolves tile j_lo + i (one coalesced load
    // of the item's slot-table entries instead of one dependent load per tile) and, for
    // the CUDA-core consumers, the lanes fold the group's query into q_bar in shared
    // memory (double-buffered by item), so neither the copies nor the consumers wait on
    // a load at an item boundary.  Lane 0 then issues the item's copies in order.
    // the key stream is read once: its lines leave L2 before the scores the selection reads next
    const uint64_t stream_pol = l2_evict_first_policy();
    uint32_t it = 0, n_item = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < a.total_items; w += gridDim.x) {
      const Item m = item_of(a, w);
      if (m.j_lo >= m.j_hi) continue;  // no candidates: the consumers skip it too
      const int j = m.j_lo + lane;     // this lane's tile (items hold at most 32)
      const unsigned char* src = nullptr;
      int host = 0;
      uint32_t bytes = kTileBytes;
      if (j < m.j_hi) {
        if (a.layout == SKV_INDEX_CONTIG) {
          const int t0 = j * kTileTokens;
          int rows = a.max_len - t0;
          rows = rows < kTileTokens ? rows : kTileTokens;
          bytes = rows * kRowBytes;
          src = a.contig + ((size_t)(m.b * a.H + m.h) * a.max_len + t0) * kRowBytes;
        } else {
          const int e = table_row(a.pool, m.b, m.h, a.H)[j];
          if (e >= 0) {
            if (e < a.pool.n_gpu)  // a block is one tile: its first row times the tile's rows
              src = (const unsigned char*)a.pool.gpu_k + gpu_block_row(a.pool, e, m.h, a.H, 1) * kTileBytes;
          } else {
            const long long hb = -(long long)e - 1;
            if (a.pool.host_k != nullptr && hb < a.pool.n_host) {
              src = (const unsigned char*)a.pool.host_k + ((size_t)hb * a.H + m.h) * kTileBytes;
              host = 1;
            }
          }
          if (src == nullptr) flag(a.status, SKV_DEV_BAD_SLOT);
        }
      }
      if constexpr (NTILE == 0) {
        // q_bar of this item into slot n_item % 2, once the consumers are done with the
        // item that used the slot before (lane l: dims 4l .. 4l + 3)
        const int qs = (int)(n_item & 1u);
        const uint32_t qph = (n_item >> 1) & 1u;
        int okq = 1;
        if (lane == 0) okq = wait_or_abort(&q_empty[qs], qph ^ 1u, &s_abort, a.status);
        if (!__shfl_sync(0xffffffffu, okq, 0)) {
          ok = false;
          break;
        }
        const unsigned char* qp = a.q + ((size_t)m.b * a.n_idx_q + (size_t)m.h * a.gi) * kRowBytes;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int g = 0; g < a.gi; ++g) {
          float x[4];
          load_q4<T>(qp + (size_t)g * kRowBytes + (size_t)lane * 4 * sizeof(T), x);
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] += x[e];
        }
        const float inv = 1.f / (float)a.gi;
        *reinterpret_cast<float4*>(&q_bar[qs][4 * lane]) = make_float4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
        mbar_arrive(&q_full[qs]);  // every lane, after its own stores
      }
      ++n_item;
      for (int jj = m.j_lo; jj < m.j_hi; ++jj, ++it) {
        const int l = jj - m.j_lo;
        const unsigned char* t_src =
            (const unsigned char*)__shfl_sync(0xffffffffu, (unsigned long long)src, l);
        const int t_host = __shfl_sync(0xffffffffu, host, l);
        const uint32_t t_bytes = __shfl_sync(0xffffffffu, bytes, l);
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        int okw = 1;
        if (lane == 0) okw = wait_or_abort(&empty_bar[s], ph ^ 1u, &s_abort, a.status);
        if (!__shfl_sync(0xffffffffu, okw, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (t_src == nullptr || t_host) {
            stage_src[s] = t_src;  // consumers read host rows in place, or score NaN
            mbar_arrive(&full_bar[s]);
          } else {
            unsigned char* dst = stage_mem + s * kTileBytes;
            stage_src[s] = dst;
            mbar_arrive_expect_tx(&full_bar[s], t_bytes);
            bulk_g2s_hint(dst, t_src, t_bytes, &full_bar[s], stream_pol);
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // gave up: let the copies already issued land before this CTA's shared memory goes away
      const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
      for (uint32_t i = first; i < it; ++i) mbar_wait_bounded(&full_bar[i % kStages], (i / kStages) & 1u);
    }
    return;
  }

  if constexpr (NTILE > 0) {
    // ---------------------------------------------------------- tensor-core consumers
    // Warp cw takes the ring stages it % kConsumerWarps == cw.  A tile's 16 keys are the A
    // operand (keys x dims), the group's scoring heads the B operand (dims x heads,
    // NTILE tiles of 8 heads, zero past gi): mma.sync m16n8k16, fp32 accumulation.
    // Within each pair of 16-dim k-steps the dims are taken in a permuted order --
    // the same for keys and queries, which leaves every dot product unchanged -- so
    // that a lane's A fragments for the pair are one 16-byte chunk of a key row:
    // chunk 4p + t4 holds (step 2p: dims 2t4, 2t4+1, 2t4+8, 2t4+9 of the pair's
    // first 16; step 2p+1: the same of its second 16).
    const int cw = warp - 1, g = lane >> 2, t4 = lane & 3;
    uint2 qb[NTILE][4][2];
    int cur_row = -1;
    uint32_t it = 0;
    for (int w = blockIdx.x; w < a.total_items; w += gridDim.x) {
      Item m = item_of(a, w);
      if (m.j_lo >= m.j_hi) continue;
      if (m.row != cur_row) {
        cur_row = m.row;
        const unsigned char* qp = a.q + ((size_t)m.b * a.n_idx_q + (size_t)m.h * a.gi) * kRowBytes;
#pragma unroll
        for (int nt = 0; nt < NTILE; ++nt) {
          const int head = 8 * nt + g;
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2)
              qb[nt][p][s2] = head < a.gi ? *reinterpret_cast<const uint2*>(qp + (size_t)head * kRowBytes +
                                                                             (8 * (4 * p + t4) + 4 * s2) * 2)
                                          : make_uint2(0u, 0u);
        }
      }
      float* out_row = a.scores + (size_t)m.row * a.max_len;
      for (int j = m.j_lo; j < m.j_hi; ++j, ++it) {
        if ((int)(it % kConsumerWarps) != cw) continue;
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        // on a failed wait the tile scores NaN; the loop still reaches every barrier
        const unsigned char* src = wait_or_abort(&full_bar[s], ph, &s_abort, a.status) ? stage_src[s] : nullptr;
        float v0, v1;  // scores of keys g and g + 8 of the tile
        if (src != nullptr) {
          float d[NTILE][4];
#pragma unroll
          for (int nt = 0; nt < NTILE; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
          const bool in_smem = src == stage_mem + s * kTileBytes;
          const uint32_t sb = smem_u32(stage_mem + s * kTileBytes);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int o0 = g * kRowBytes + (4 * p + t4) * 16, o1 = o0 + 8 * kRowBytes;
            uint4 k0, k1;
            if (in_smem) {
              k0 = lds128(sb + o0);
              k1 = lds128(sb + o1);
            } else {  // a host-resident block, read in place
              k0 = *reinterpret_cast<const uint4*>(src + o0);
              k1 = *reinterpret_cast<const uint4*>(src + o1);
            }
#pragma unroll
            for (int nt = 0; nt < NTILE; ++nt) {
              mma16816(d[nt], k0.x, k1.x, k0.y, k1.y, qb[nt][p][0].x, qb[nt][p][0].y);
              mma16816(d[nt], k0.z, k1.z, k0.w, k1.w, qb[nt][p][1].x, qb[nt][p][1].y);
            }
          }
          // lane (g, t4) holds heads 8nt + 2t4, + 1 of keys g and g + 8
          if constexpr (HEADS) {  // every head's own score into its own row
            const int t0 = j * kTileTokens + g, t1 = t0 + 8;
            const bool in0 = t0 >= m.s_end && t0 < m.l_start, in1 = t1 >= m.s_end && t1 < m.l_start;
            float* head_rows = a.scores + (size_t)m.row * a.gi * a.max_len;
#pragma unroll
            for (int nt = 0; nt < NTILE; ++nt)
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int hd = 8 * nt + 2 * t4 + (c & 1);
                const int t = (c & 2) ? t1 : t0;
                if (hd < a.gi && ((c & 2) ? in1 : in0)) head_rows[(size_t)hd * a.max_len + t] = d[nt][c];
              }
            v0 = v1 = 0.f;
          } else if (a.agg == SKV_AGG_MAX) {  // (not HEADS)
            v0 = v1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < NTILE; ++nt) {
              const int hd = 8 * nt + 2 * t4;
              if (hd < a.gi) {
                v0 = fmaxf(v0, d[nt][0]);
                v1 = fmaxf(v1, d[nt][2]);
              }
              if (hd + 1 < a.gi) {
                v0 = fmaxf(v0, d[nt][1]);
                v1 = fmaxf(v1, d[nt][3]);
              }
            }
            v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, 1));
            v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, 1));
            v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, 2));
            v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, 2));
          } else {  // heads past gi contribute zero
            v0 = v1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < NTILE; ++nt) {
              v0 += d[nt][0] + d[nt][1];
              v1 += d[nt][2] + d[nt][3];
            }
            v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
            v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
            v0 *= a.inv_gi;
            v1 *= a.inv_gi;
          }
        } else {
          v0 = v1 = __int_as_float(0x7fc00000);  // NaN: ranks below every score
          if constexpr (HEADS) {  // ... in every head's row
            const int t0 = j * kTileTokens + g, t1 = t0 + 8;
            float* head_rows = a.scores + (size_t)m.row * a.gi * a.max_len;
            for (int hd = 2 * t4; hd < a.gi; hd += 8)
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                if (hd + u >= a.gi) continue;
                if (t0 >= m.s_end && t0 < m.l_start) head_rows[(size_t)(hd + u) * a.max_len + t0] = v0;
                if (t1 >= m.s_end && t1 < m.l_start) head_rows[(size_t)(hd + u) * a.max_len + t1] = v1;
              }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        const int t0 = j * kTileTokens + g, t1 = t0 + 8;
        if constexpr (!HEADS) {
          if (t4 == 0 && t0 >= m.s_end && t0 < m.l_start) out_row[t0] = v0;
          if (t4 == 1 && t1 >= m.s_end && t1 < m.l_start) out_row[t1] = v1;
        }
      }
    }
    return;
  } else {
    // -------------------------------------------------------------- consumers
    // Consumer warp pair p (warps 2p + 1, 2p + 2) takes the tiles it % kPairs == p.  Four lanes
    // share a row: lane a of a row owns chunks kCL*a .. kCL*a+kCL-1, visited in an
    // order rotated by the row so each 128-bit shared load spreads over all banks.
    const int ct = threadIdx.x - 32;
    const int pair = ct >> 6;
    const int r = (ct & 63) >> 2;
    const int la = ct & 3;
    float qr[kCL][kEpc];  // q_bar chunks in this thread's visiting order
    const uint64_t keep_pol = l2_evict_last_policy();  // the selection reads the scores next
    float pf_tau = NAN;    // the row's predicted threshold (prefetch variant)
    int cur_row = -1;
    uint32_t it = 0, n_item = 0;
    for (int w = blockIdx.x; w < a.total_items; w += gridDim.x) {
      Item m = item_of(a, w);
      if (m.j_lo >= m.j_hi) continue;
      if (m.row != cur_row) {
        cur_row = m.row;
        if (PF) pf_tau = a.pf.tau[m.row];
      }
      {  // this item's q_bar from the producer warp (a failed wait leaves the scores garbage, flagged)
        const int qs = (int)(n_item & 1u);
        wait_or_abort(&q_full[qs], (n_item >> 1) & 1u, &s_abort, a.status);
#pragma unroll
        for (int i = 0; i < kCL; ++i) {
          const int c = kCL * la + ((i + r) & (kCL - 1));
#pragma unroll
          for (int e = 0; e < kEpc; e += 4) {
            const float4 x = *reinterpret_cast<const float4*>(&q_bar[qs][c * kEpc + e]);
            qr[i][e] = x.x;
            qr[i][e + 1] = x.y;
            qr[i][e + 2] = x.z;
            qr[i][e + 3] = x.w;
          }
        }
        mbar_arrive(&q_empty[qs]);  // read into registers: the slot may be refilled
        ++n_item;
      }
      float* out_row = a.scores + (size_t)m.row * a.max_len;
      for (int j = m.j_lo; j < m.j_hi; ++j, ++it) {
        if ((int)(it % kPairs) != pair) continue;
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        // on a failed wait the tile scores NaN; the loop still reaches every barrier
        const unsigned char* src = wait_or_abort(&full_bar[s], ph, &s_abort, a.status) ? stage_src[s] : nullptr;
        float part;
        if (src != nullptr) {
          const unsigned char* rowp = src + r * kRowBytes;
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < kCL; ++i) {
            float kv[kEpc];
            Vec<T>::load(rowp + (kCL * la + ((i + r) & (kCL - 1))) * 16, kv);
#pragma unroll
            for (int e = 0; e < kEpc; ++e) acc = fmaf(qr[i][e], kv[e], acc);
          }
          part = acc;
        } else {
          part = __int_as_float(0x7fc00000);  // NaN: ranks below every score
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        const int t = j * kTileTokens + r;
        if (la == 0 && t >= m.s_end && t < m.l_start) {
          st_f32_hint(out_row + t, part, keep_pol);
          if (PF && part > pf_tau) {  // NaN prediction: never
            const unsigned i = atomicAdd(&pf_n, 1u);
            if (i < (unsigned)kPfList) {
              pf_list[i] = make_int2(m.row, t);
              __threadfence_block();
              pf_ready[i] = 1;
            }
          }
        }
      }
    }
    if (PF) {
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        atomicAdd((int*)&pf_done, 1);
      }
    }
  }
}

template <typename T, int NTILE, bool HEADS = false>
__global__ void __launch_bounds__(kScoreThreads, NTILE == 0 ? 10 : 6) score_kernel(const ScoreArgs a) {
  score_body<T, NTILE, 0, HEADS>(a);
}

// The prefetch variant: PF more warps, which copy host rows over the host link while the
// key stream runs.  Two warps: four CTAs share an SM (the host link, not the key stream,
// sets the latent step's time, and the registers then hold the copy batches); one warp:
// five CTAs.
template <typename T, int PF>
__global__ void __launch_bounds__(kScoreThreads + 32 * PF, PF == 1 ? 5 : 4) score_prefetch_kernel(const ScoreArgs a) {
  score_body<T, 0, PF>(a);
}

template <typename T, int NTILE, int PF, bool HEADS = false>
skv_status launch_typed(const ScoreArgs& a, cudaStream_t st) {
  constexpr int kTileBytes = kTileTokens * kD * (int)sizeof(T);
  constexpr int kThreads = kScoreThreads + 32 * PF;
  void (*kernel)(const ScoreArgs) = nullptr;
  if constexpr (PF > 0)
    kernel = score_prefetch_kernel<T, PF>;
  else
    kernel = score_kernel<T, NTILE, HEADS>;
  const int smem = kStages * kTileBytes;
  int blocks_per_sm = 1;
  const skv_status prep = prepare_kernel((const void*)kernel, smem, kThreads, &blocks_per_sm);
  if (prep != SKV_OK) return prep;
  const long long cap = (long long)num_sms() * blocks_per_sm;
  // items of 32 tiles while the rows fill every CTA slot; smaller items (down to 2
  // tiles) for short or few rows, so that more SMs share the key stream
  ScoreArgs b = a;
  const long long tiles = (a.max_len + kTileTokens - 1) / kTileTokens, rows = (long long)a.B * a.H;
  long long tpi = kTilesPerItem;
  if (rows * ((tiles + tpi - 1) / tpi) < cap) {
    tpi = (rows * tiles + cap - 1) / cap;
    tpi = tpi < kMinTilesPerItem ? kMinTilesPerItem : (tpi > kTilesPerItem ? kTilesPerItem : tpi);
  }
  b.tiles_per_item = (int)tpi;
  b.items_per_row = (int)((tiles + tpi - 1) / tpi);
  b.total_items = (int)(b.items_per_row * rows);
  if (b.total_items == 0) return SKV_OK;
  const int grid = (int)(b.total_items < cap ? b.total_items : cap);
  kernel<<<grid, kThreads, smem, st>>>(b);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace

skv_status launch_score(const skv_problem& p, const void* q_score, const skv_index_src& idx,
                        const PoolView& pool, float* scores, int32_t* status, cudaStream_t st,
                        const PrefetchView* pf) {
  ScoreArgs a;
  a.q = (const unsigned char*)q_score;
  a.n_idx_q = p.n_idx_q_heads;
  a.gi = p.n_idx_q_heads / p.n_kv_heads;
  a.H = p.n_kv_heads;
  a.layout = idx.layout;
  a.contig = (const unsigned char*)idx.keys;
  a.pool = pool;
  a.seq_lens = p.seq_lens;
  a.B = p.batch;
  a.max_len = p.max_len;
  a.ns = p.n_sink;
  a.nl = p.n_local;
  a.scores = scores;
  a.status = status;
  a.agg = p.group_agg;
  a.inv_gi = 1.f / (float)a.gi;
  a.pf = pf ? *pf : PrefetchView{};
  a.pf_row_bytes = p.d_qk * (p.dtype == SKV_DTYPE_F32 ? 4 : 2);
  // paged pools stage the V row beside the K row: K rows [rows, cap], then V rows [rows, cap]
  a.pf_v_bytes = pool.gpu_v != nullptr ? p.d_v * (p.dtype == SKV_DTYPE_F32 ? 4 : 2) : 0;
  a.pf_v_off = pf ? (size_t)p.batch * p.n_kv_heads * (size_t)pf->cap * a.pf_row_bytes : 0;
  if (p.max_len == 0) return SKV_OK;
  if (pf != nullptr) {  // threshold prefetch: bf16, the mean, contiguous index keys
    if (p.dtype != SKV_DTYPE_BF16 || a.agg != SKV_AGG_MEAN || a.layout != SKV_INDEX_CONTIG) return SKV_ERR_UNSUPPORTED;
    if ((a.pf_row_bytes + a.pf_v_bytes) / 16 > kPfChunks) return SKV_ERR_UNSUPPORTED;
    return pool.gpu_v != nullptr ? launch_typed<__nv_bfloat16, 0, 1>(a, st) : launch_typed<__nv_bfloat16, 0, 2>(a, st);
  }
  // the mean folds the group into one query (1 flop per key byte): CUDA cores; the max keeps
  // gi dot products per key, a contraction: tensor cores
  if (p.dtype == SKV_DTYPE_F32) return launch_typed<float, 0, 0>(a, st);
  if (a.agg == SKV_AGG_MEAN) return launch_typed<__nv_bfloat16, 0, 0>(a, st);
  if (a.agg == SKV_AGG_HEAD)  // every head's score kept: the tensor-core tile, one row a head
    return a.gi <= 8 ? launch_typed<__nv_bfloat16, 1, 0, true>(a, st) : launch_typed<__nv_bfloat16, 2, 0, true>(a, st);
  if (a.gi <= 8) return launch_typed<__nv_bfloat16, 1, 0>(a, st);
  if (a.gi <= 16) return launch_typed<__nv_bfloat16, 2, 0>(a, st);
  return launch_typed<__nv_bfloat16, 0, 0>(a, st);
}

}  // namespace skv
