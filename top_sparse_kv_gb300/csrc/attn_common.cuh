// Shared pieces of the attention kernels (not part of the ABI): arguments, the
// attended-list walk, slot-table row resolution, the split merge and the
// mma.sync / cp.async / ldmatrix wrappers.
#pragma once

#include "skv_internal.cuh"

namespace skv {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnArgs {
  const unsigned char* q;  // [B, Hq, kD]
  PoolView pool;
  const int32_t* idx;  // [B, H, k]
  const int32_t* seq_lens;
  int B, H, Hq, G, max_len, ns, nl, k, bs;
  float scale_log2;
  int n_splits, chunk;
  float* ws_o;        // [B, Hq, S, dv]
  float* ws_ml;       // [B, Hq, S, 2]
  uint32_t* tickets;  // [B, H], zeroed before the launch
  void* out;          // [B, Hq, dv] (bf16 or fp32)
  float* lse;         // [B, Hq] or null
  int dv, out_f32;
  int32_t* status;
  PrefetchView pf;   // threshold prefetch (bf16 paged path): staged host rows (pf.map == nullptr: none)
  size_t pf_v_off;   // byte offset of the staged V rows inside pf.staging
  BlockListView bl;  // block-list mode (bf16 kernel) when bl.att != nullptr
};

constexpr int kMergeMax = 1024;  // split partials of one head merged through shared memory (max n_splits)

// Called by every CTA of (request b, KV head h) after it wrote its split
// partials: the last one to arrive (ticket) merges the n_splits partials of the
// G query heads -- m* = max m_s, l = sum l_s 2^(m_s - m*), out = sum acc_s
// 2^(m_s - m*) / l, lse = ln 2 (m* + log2 l) -- and writes the output.  No CTA
// waits for another: the others simply return.  A warp per head reads its
// splits' (m, l) pairs with every load in flight at once, and the output is
// accumulated four dims a thread with four splits' float4 loads in flight, so
// the merge costs a few L2 round trips however many splits there are.

__device__ __forceinline__ void merge_if_last(const AttnArgs& a, int b, int h, int ctas_per_unit) {
  __shared__ int s_last;
  __shared__ float s_w[kMergeMax];  // per (head, split): 2^(m_s - m*)
  __shared__ float s_inv[16];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&a.tickets[b * a.H + h], 1u) == (uint32_t)(ctas_per_unit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int S = a.n_splits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int nv = a.dv / 4;  // output dims in float4 groups (d_v = 128)
  const size_t hq0 = (size_t)b * a.Hq + (size_t)h * a.G;
  for (int g0 = 0; g0 < a.G; g0 += 16) {  // heads in groups whose partial count fits kMergeMax
    const int gn = a.G - g0 < 16 ? a.G - g0 : 16;
    const int gc = gn * S <= kMergeMax ? gn : (kMergeMax / S > 0 ? kMergeMax / S : 1);
    for (int gb = 0; gb < gn; gb += gc) {
      const int cnt = (gn - gb < gc ? gn - gb : gc);
      // one warp per head: the lanes stride over the splits' (m_s, l_s) pairs, so a
      // head's loads are all in flight at once; max and sum by butterfly
      for (int gg = warp; gg < cnt; gg += nwarps) {
        const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + (hq0 + g0 + gb + gg) * S;
        float ms = -INFINITY;
        for (int s = lane; s < S; s += 32) ms = fmaxf(ms, __ldcg(ml + s).x);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, off));
        float tot = 0.f;
        for (int s = lane; s < S; s += 32) {
          const float2 v = __ldcg(ml + s);
          const float w = (ms == -INFINITY || v.x == -INFINITY) ? 0.f : exp2f(v.x - ms);
          tot += w * v.y;
          s_w[gg * S + s] = w;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
        if (lane == 0) {
          s_inv[gg] = tot > 0.f ? 1.f / tot : 0.f;
          if (a.lse) a.lse[hq0 + g0 + gb + gg] = tot > 0.f ? kLn2 * (ms + log2f(tot)) : -INFINITY;
        }
      }
      __syncthreads();
      // four output dims a thread: float4 loads of the partials, four splits in flight
      for (int t = threadIdx.x; t < cnt * nv; t += blockDim.x) {
        const int gg = t / nv, d4 = t - gg * nv;
        const size_t hq = hq0 + g0 + gb + gg;
        const float4* po = reinterpret_cast<const float4*>(a.ws_o + hq * (size_t)S * a.dv) + d4;
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll 4
        for (int s = 0; s < S; ++s) {
          const float w = s_w[gg * S + s];
          const float4 v = __ldcg(po + (size_t)s * nv);
          o0 = fmaf(w, v.x, o0);
          o1 = fmaf(w, v.y, o1);
          o2 = fmaf(w, v.z, o2);
          o3 = fmaf(w, v.w, o3);
        }
        const float inv = s_inv[gg];
        const size_t od = hq * a.dv + 4 * d4;
        if (a.out_f32) {
          *reinterpret_cast<float4*>((float*)a.out + od) = make_float4(o0 * inv, o1 * inv, o2 * inv, o3 * inv);
        } else {
          __nv_bfloat16* ob = (__nv_bfloat16*)a.out + od;
          *reinterpret_cast<__nv_bfloat162*>(ob) = __floats2bfloat162_rn(o0 * inv, o1 * inv);
          *reinterpret_cast<__nv_bfloat162*>(ob + 2) = __floats2bfloat162_rn(o2 * inv, o3 * inv);
        }
      }
      __syncthreads();
    }
  }
}

// Position of list entry j, or -1 when the entry is empty / invalid.
__device__ __forceinline__ int list_pos(const AttnArgs& a, const int32_t* idx_row, const Regions& r, int j,
                                        int n_list) {
  if (j >= n_list) return -1;
  if (j < r.s_end) return j;
  const int u = j - r.s_end;
  if (u < a.k) {
    const int t = idx_row[u];
    if (t < 0) return -1;
    if (t < r.s_end || t >= r.l_start) {
      flag(a.status, SKV_DEV_BAD_INDEX);
      return -1;
    }
    return t;
  }
  return r.l_start + (u - a.k);
}

// Row addresses of position t (K row, V row); false when the slot entry is bad.
template <typename T>
__device__ __forceinline__ bool resolve_row(const AttnArgs& a, int b, int h, int t, const unsigned char** kp,
                                            const unsigned char** vp) {
  constexpr size_t kRow = kD * sizeof(T);
  const int heads = a.H / a.pool.hdiv, ph = h / a.pool.hdiv;  // the pool's heads and this row's
  const int e = table_row(a.pool, b, ph, heads)[t / a.bs];
  const size_t off = (size_t)(t % a.bs);
  if (e >= 0) {
    if (e >= a.pool.n_gpu) return false;
    const size_t r = gpu_block_row(a.pool, e, ph, heads, a.bs) + off;
    *kp = (const unsigned char*)a.pool.gpu_k + r * kRow;
    *vp = (const unsigned char*)a.pool.gpu_v + r * kRow;
    return true;
  }
  const long long hb = -(long long)e - 1;
  if (a.pool.host_k == nullptr || hb >= a.pool.n_host) return false;
  const size_t r = ((size_t)hb * heads + ph) * a.bs + off;
  *kp = (const unsigned char*)a.pool.host_k + r * kRow;
  *vp = (const unsigned char*)a.pool.host_v + r * kRow;
  return true;
}

template <typename T>
__device__ __forceinline__ void load4(const unsigned char* p, float* v) {
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

namespace tc {

constexpr int kTileRows = 64;
constexpr int kRowBytes = kD * 2;
constexpr int kTileBytes = kTileRows * kRowBytes;
// Two shapes of the gather ring.  Shallow: 2 stages (one tile in flight while one is
// computed), at most 512 list entries a CTA, 3 CTAs a SM.  Deep: 3 stages, at most 1,024
// entries, 2 CTAs a SM -- for problems whose splits then fit one wave (the fewer, longer
// CTAs keep two tiles in flight each).
template <int STAGES>
struct Ring {
  static constexpr int kStages = STAGES;
  static constexpr int kMaxChunk = STAGES == 2 ? 512 : 1024;  // list entries per CTA (resolved up front)
  static constexpr int kCtasPerSm = STAGES == 2 ? 3 : 2;
  static constexpr int kSmemBytes = STAGES * 2 * kTileBytes + kMaxChunk * 8 + (kMaxChunk / kTileRows) * 2 * 4;
};
constexpr long long kHostBit = 1LL << 62;
constexpr long long kStageBit = 1LL << 61;  // a host row staged this step: read from pf.staging
constexpr long long kRefRowMask = kStageBit - 1;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Transpose of an 8 x 8 bf16 matrix held one row per lane quad (lane / 4 = row,
// elements 2 (lane % 4) and 2 (lane % 4) + 1), returned in the same distribution.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
// byte offset of 16-byte chunk `c` of row `r` in a swizzled tile
__device__ __forceinline__ int swz(int r, int c) { return r * kRowBytes + ((c ^ (r & 7)) << 4); }

}  // namespace tc

inline AttnArgs make_args(const skv_problem& p, const void* q, const PoolView& pool, const int32_t* idx, int32_t* status) {
  AttnArgs a;
  a.q = (const unsigned char*)q;
  a.pool = pool;
  if (a.pool.hdiv < 1) a.pool.hdiv = 1;
  a.idx = idx;
  a.seq_lens = p.seq_lens;
  a.B = p.batch;
  a.H = p.n_kv_heads;
  a.Hq = p.n_q_heads;
  a.G = p.n_q_heads / p.n_kv_heads;
  a.max_len = p.max_len;
  a.ns = p.n_sink;
  a.nl = p.n_local;
  a.k = p.topk;
  a.bs = p.block_size;
  const float scale = p.sm_scale > 0.f ? p.sm_scale : 1.f / sqrtf((float)p.d_qk);
  a.scale_log2 = scale * kLog2e;
  a.status = status;
  a.ws_o = nullptr;
  a.ws_ml = nullptr;
  a.tickets = nullptr;
  a.out = nullptr;
  a.lse = nullptr;
  a.pf = PrefetchView{};
  a.pf_v_off = 0;
  a.bl = BlockListView{};
  a.dv = p.d_v;
  a.out_f32 = p.dtype == SKV_DTYPE_F32;
  a.n_splits = 1;
  a.chunk = 1;
  return a;
}

inline int max_list(const skv_problem& p) { return p.n_sink + p.topk + p.n_local; }


}  // namespace
}  // namespace skv
