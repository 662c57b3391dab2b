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
// attn_merge_kernel: one CTA per (query head, request); merges the n_splits
// partials:  m* = max m_s, l = sum l_s 2^(m_s - m*), out = sum acc_s 2^(m_s - m*) / l,
// lse = ln 2 * (m* + log2 l).
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
  float* ws_o;   // [B, Hq, S, kD]
  float* ws_ml;  // [B, Hq, S, 2]
  int32_t* status;
};

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
  const int e = a.pool.table[(size_t)b * a.pool.stride + t / a.bs];
  const size_t off = (size_t)(t % a.bs);
  if (e >= 0) {
    if (e >= a.pool.n_gpu) return false;
    const size_t r = ((size_t)e * a.H + h) * a.bs + off;
    *kp = (const unsigned char*)a.pool.gpu_k + r * kRow;
    *vp = (const unsigned char*)a.pool.gpu_v + r * kRow;
    return true;
  }
  const long long hb = -(long long)e - 1;
  if (a.pool.host_k == nullptr || hb >= a.pool.n_host) return false;
  const size_t r = ((size_t)hb * a.H + h) * a.bs + off;
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

template <typename T, int GM>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(const AttnArgs a) {
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
}

template <typename T>
__global__ void __launch_bounds__(kD) attn_merge_kernel(const float* ws_o, const float* ws_ml, int n_splits, int Hq,
                                                      int dv, T* out, float* lse) {
  extern __shared__ float sw[];  // weights per split
  __shared__ float s_tot;
  const int j = blockIdx.x, b = blockIdx.y;
  const size_t hq = (size_t)b * Hq + j;
  const float* ml = ws_ml + hq * n_splits * 2;
  if (threadIdx.x == 0) {
    float ms = -INFINITY;
    for (int s = 0; s < n_splits; ++s) ms = fmaxf(ms, ml[2 * s]);
    float tot = 0.f;
    for (int s = 0; s < n_splits; ++s) {
      const float w = (ms == -INFINITY || ml[2 * s] == -INFINITY) ? 0.f : exp2f(ml[2 * s] - ms);
      sw[s] = w;
      tot += ml[2 * s + 1] * w;
    }
    s_tot = tot;
    if (lse) lse[hq] = tot > 0.f ? kLn2 * (ms + log2f(tot)) : -INFINITY;
  }
  __syncthreads();
  const float inv = s_tot > 0.f ? 1.f / s_tot : 0.f;
  for (int d = threadIdx.x; d < dv; d += blockDim.x) {
    float o = 0.f;
    for (int s = 0; s < n_splits; ++s) o = fmaf(sw[s], ws_o[(hq * n_splits + s) * dv + d], o);
    out[hq * dv + d] = from_float<T>(o * inv);
  }
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
    const int e = a.pool.table[(size_t)b * a.pool.stride + t / a.bs];
    const size_t off = (size_t)(t % a.bs);
    const bool latent = a.pool.gpu_v == nullptr;
    if (e >= 0 && e < a.pool.n_gpu) {
      const size_t r = ((size_t)e * a.H + h) * a.bs + off;
      kp = (const unsigned char*)a.pool.gpu_k + r * d_k * sizeof(T);
      vp = latent ? kp : (const unsigned char*)a.pool.gpu_v + r * d_v * sizeof(T);
      ok = true;
    } else if (e < 0 && a.pool.host_k != nullptr && (-(long long)e - 1) < a.pool.n_host) {
      const size_t r = ((size_t)(-(long long)e - 1) * a.H + h) * a.bs + off;
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

AttnArgs make_args(const skv_problem& p, const void* q, const PoolView& pool, const int32_t* idx, int32_t* status) {
  AttnArgs a;
  a.q = (const unsigned char*)q;
  a.pool = pool;
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
  a.n_splits = 1;
  a.chunk = 1;
  return a;
}

int max_list(const skv_problem& p) { return p.n_sink + p.topk + p.n_local; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <typename T, int GM>
skv_status launch_split(const AttnArgs& a, cudaStream_t st) {
  dim3 grid(a.n_splits, a.H, a.B);
  attn_split_kernel<T, GM><<<grid, kThreads, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
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

int attn_splits(const skv_problem& p) {
  const int n = max_list(p);
  if (p.n_splits > 0) return p.n_splits < (n > 0 ? n : 1) ? p.n_splits : (n > 0 ? n : 1);
  // aim at ~8 CTAs per SM in total, each with at least 64 rows
  const long long units = (long long)p.batch * p.n_kv_heads;
  long long want = (8LL * 152 + units - 1) / units;
  long long cap = (n + 63) / 64;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (int)want;
}

size_t attn_workspace_bytes(const skv_problem& p) {
  const size_t S = (size_t)attn_splits(p);
  const size_t hq = (size_t)p.batch * p.n_q_heads;
  return align256(hq * S * p.d_v * 4) + align256(hq * S * 2 * 4);
}

skv_status launch_attn(const skv_problem& p, const void* q, const PoolView& pool, const int32_t* idx, void* out,
                       float* lse, void* ws, int32_t* status, cudaStream_t st) {
  AttnArgs a = make_args(p, q, pool, idx, status);
  a.n_splits = attn_splits(p);
  const int n = max_list(p);
  a.chunk = n > 0 ? (n + a.n_splits - 1) / a.n_splits : 1;
  const size_t hq = (size_t)p.batch * p.n_q_heads;
  a.ws_o = (float*)ws;
  a.ws_ml = (float*)((unsigned char*)ws + align256(hq * a.n_splits * p.d_v * 4));
  skv_status r = p.dtype == SKV_DTYPE_F32 ? launch_split_g<float>(a, st) : launch_split_g<__nv_bfloat16>(a, st);
  if (r != SKV_OK) return r;
  dim3 mgrid(p.n_q_heads, p.batch);
  const size_t smem = (size_t)a.n_splits * sizeof(float);
  if (p.dtype == SKV_DTYPE_F32)
    attn_merge_kernel<float><<<mgrid, kD, smem, st>>>(a.ws_o, a.ws_ml, a.n_splits, p.n_q_heads, p.d_v, (float*)out,
                                                      lse);
  else
    attn_merge_kernel<__nv_bfloat16><<<mgrid, kD, smem, st>>>(a.ws_o, a.ws_ml, a.n_splits, p.n_q_heads, p.d_v,
                                                              (__nv_bfloat16*)out, lse);
  SKV_LAUNCH_CHECK();
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
