// ParisKV approximate retrieval (sm_103a): an alternative to exact scoring and top-k.
//
// ParisKV notes (cc.laoqi.cc, arXiv 2602.07721), §2.  Each key of a (request, KV head)
// row keeps, in HBM:
//   cent [rows, max_len, 16]  one byte per 8-dim subspace: the fixed centroid (sign
//                             pattern) of the key's rotated direction -- the stream
//                             the collision stage reads, 16 bytes a key
//   rec  [rows, max_len, 32]  the rerank record, one 128-byte line a key: words 0-15 the
//                             4-bit direction codes of the 16 subspaces (8 a word,
//                             sign << 3 | cell), words 16-31 the fp32 weights |k| r / alpha
//   hist [rows, 16, 256]      key counts per centroid over [0, L)
// A decode step runs:
//   paris_query_kernel      one CTA per (subspace, row): group-mean query, its SRHT
//                           rotation, the subspace's 256 centroid similarities ranked by
//                           a bitonic sort, its count histogram over the candidate region
//                           (hist minus sink and local keys), its tier weights
//   paris_collision_kernel  S = sum of W over a key's 16 centroid bytes for every
//                           candidate key, a histogram of S per chunk; the last CTA of a
//                           row (ticket) finds the threshold on S and each chunk's output
//                           offset, as a bucket top-k over small integers
//   paris_compact_kernel    per chunk: the candidates in position order (two CTA scans),
//                           then their rerank scores from codes and weights (a thread a
//                           key, eight 16-byte loads)
//   exact top-k             the existing radix select over the candidate scores; its
//                           one-CTA and two-stage paths write the candidates' positions
//                           directly, the others through
//   paris_map_kernel        candidate slots -> positions (ascending stays ascending)
//   attention               the existing split-K kernels over sink U selected U local
#include <cmath>
#include <mutex>

#include "skv_internal.cuh"

namespace skv {
namespace {

constexpr int kD = 128;                  // head dimension
constexpr int kM = 8;                    // subspace dimension
constexpr int kSub = kD / kM;            // 16 subspaces
constexpr int kCent = 1 << kM;           // 256 centroids per subspace
constexpr int kMaxS = 6 * kSub;          // largest collision score
constexpr int kSBins = 128;              // histogram bins (>= kMaxS + 1)
constexpr int kChunk = 8192;             // candidate keys per collision / compaction CTA
constexpr int kEncKeys = 1024;           // keys per encode CTA
__constant__ int kTierPct[6] = {5, 15, 30, 50, 75, 100};  // cumulative tier cuts, per cent of N

struct Quant {
  float level[8];
  float thr[7];
};

// ---------------------------------------------------------------- Lloyd-Max (host)
//
// The magnitude x = |u_j| of one coordinate of a random unit vector in R^m has density
// proportional to (1 - x^2)^((m-3)/2) on [0, 1] (u_j^2 ~ Beta(1/2, (m-1)/2)).  With
// x = sin(theta) both cell integrals have closed forms:
//   int_0^x (1 - s^2)^((m-3)/2) ds  = C_{m-2}(asin x),  C_n(a) = int_0^a cos^n,
//   int_0^x s (1 - s^2)^((m-3)/2) ds = (1 - (1 - x^2)^((m-1)/2)) / (m - 1),
// with C_n(a) = cos^(n-1)(a) sin(a) / n + (n-1)/n C_{n-2}(a), C_0 = a, C_1 = sin a.
// Lloyd's iteration (cuts at midpoints, levels at cell means) runs on these.

double cos_power_integral(int n, double a) {
  if (n == 0) return a;
  if (n == 1) return std::sin(a);
  return std::pow(std::cos(a), n - 1) * std::sin(a) / n + (double)(n - 1) / n * cos_power_integral(n - 2, a);
}

double mass_below(int m, double x) { return cos_power_integral(m - 2, std::asin(x < 1.0 ? x : 1.0)); }
double moment_below(int m, double x) {
  const double y = 1.0 - x * x;
  return (1.0 - std::pow(y > 0.0 ? y : 0.0, 0.5 * (m - 1))) / (m - 1);
}

void lloyd_max_host(int m, double lv[8], double th[7]) {
  for (int i = 0; i < 8; ++i) lv[i] = (i + 0.5) / 8.0;
  for (int it = 0; it < 200000; ++it) {
    double e[9];
    e[0] = 0.0;
    e[8] = 1.0;
    for (int i = 1; i < 8; ++i) e[i] = 0.5 * (lv[i - 1] + lv[i]);
    double change = 0.0;
    for (int i = 0; i < 8; ++i) {
      const double m0 = mass_below(m, e[i + 1]) - mass_below(m, e[i]);
      const double m1 = moment_below(m, e[i + 1]) - moment_below(m, e[i]);
      const double nv = m0 > 0.0 ? m1 / m0 : 0.5 * (e[i] + e[i + 1]);
      change = std::fmax(change, std::fabs(nv - lv[i]));
      lv[i] = nv;
    }
    if (change < 1e-15) break;
  }
  for (int i = 0; i < 7; ++i) th[i] = 0.5 * (lv[i] + lv[i + 1]);
}

Quant quant_for(int m) {
  static std::mutex mu;
  static bool have[65] = {};
  static Quant cache[65];
  std::lock_guard<std::mutex> lock(mu);
  if (!have[m]) {
    double lv[8], th[7];
    lloyd_max_host(m, lv, th);
    for (int i = 0; i < 8; ++i) cache[m].level[i] = (float)lv[i];
    for (int i = 0; i < 7; ++i) cache[m].thr[i] = (float)th[i];
    have[m] = true;
  }
  return cache[m];
}

// ---------------------------------------------------------------- device helpers

// Walsh-Hadamard transform of 128 values held 4 per lane (lane l: indices 4l .. 4l+3),
// unnormalised: out_i = sum_j (-1)^popcount(i & j) in_j.
__device__ __forceinline__ void fwht128(float v[4]) {
  const int lane = threadIdx.x & 31;
  const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[1] = a1 + a3;
  v[2] = a0 - a2;
  v[3] = a1 - a3;
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const bool upper = (lane >> s) & 1;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float p = __shfl_xor_sync(0xffffffffu, v[e], 1 << s);
      v[e] = upper ? p - v[e] : v[e] + p;
    }
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ void load4_bf16(const void* p, float v[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(u.x << 16);
  v[1] = __uint_as_float(u.x & 0xffff0000u);
  v[2] = __uint_as_float(u.y << 16);
  v[3] = __uint_as_float(u.y & 0xffff0000u);
}

// ---------------------------------------------------------------- encode

struct EncArgs {
  const unsigned char* keys;  // contiguous keys [B, H, max_len, 128] bf16, or null (paged)
  PoolView pool;              // paged source when keys == null
  const int32_t* seq_lens;
  const int8_t* signs;        // [128]
  uint8_t* cent;
  uint32_t* rec;
  int32_t* hist;
  int32_t* status;
  int H, max_len, bs;
  Quant qz;
};

__device__ __forceinline__ const unsigned char* key_row(const EncArgs& a, int b, int h, int t) {
  if (a.keys != nullptr) return a.keys + (((size_t)b * a.H + h) * a.max_len + t) * (kD * 2);
  const int e = a.pool.table[(size_t)b * a.pool.stride + t / a.bs];
  const size_t off = (size_t)(t % a.bs);
  if (e >= 0 && e < a.pool.n_gpu)
    return (const unsigned char*)a.pool.gpu_k + ((((size_t)e * a.H + h) * a.bs) + off) * (kD * 2);
  const long long hb = -(long long)e - 1;
  if (e < 0 && a.pool.host_k != nullptr && hb < a.pool.n_host)
    return (const unsigned char*)a.pool.host_k + ((((size_t)hb * a.H + h) * a.bs) + off) * (kD * 2);
  return nullptr;
}

__global__ void __launch_bounds__(256) paris_encode_kernel(const EncArgs a) {
  __shared__ int hist[kSub][kCent];
  __shared__ float lvl[8];
  const int row = blockIdx.y, b = row / a.H, h = row - b * a.H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kSub * kCent; i += blockDim.x) (&hist[0][0])[i] = 0;
  if (threadIdx.x < 8) lvl[threadIdx.x] = a.qz.level[threadIdx.x];
  __syncthreads();
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const int t0 = blockIdx.x * kEncKeys, t1 = min(t0 + kEncKeys, L);
  float sg[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) sg[e] = (float)a.signs[4 * lane + e];
  const float inv_sqrt_d = 0.08838834764831845f;  // 1 / sqrt(128)
  for (int t = t0 + warp; t < t1; t += 8) {
    const unsigned char* src = key_row(a, b, h, t);
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (src != nullptr) load4_bf16(src + lane * 8, v);
    else if (lane == 0) flag(a.status, SKV_DEV_BAD_SLOT);
    const float kn = sqrtf(warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]));
    const float inv = kn > 0.f ? 1.f / kn : 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = v[e] * inv * sg[e];
    fwht128(v);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] *= inv_sqrt_d;
    // subspace lane >> 1 = 8 coordinates on lanes (2s, 2s + 1)
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    const float r = sqrtf(ss);
    const float ir = r > 0.f ? 1.f / r : 0.f;
    uint32_t bits = 0, nib = 0;
    float al = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float u = v[e] * ir;
      const float au = fabsf(u);
      int cell = 0;
#pragma unroll
      for (int i = 0; i < 7; ++i) cell += au >= a.qz.thr[i] ? 1 : 0;
      const bool neg = u < 0.f;
      const float lv = lvl[cell];
      al += (neg ? -lv : lv) * u;
      bits |= (neg ? 1u : 0u) << e;
      nib |= (((neg ? 8u : 0u) | (uint32_t)cell) << (4 * e));
    }
    al += __shfl_xor_sync(0xffffffffu, al, 1);
    const uint32_t pbits = __shfl_xor_sync(0xffffffffu, bits, 1);
    const uint32_t pnib = __shfl_xor_sync(0xffffffffu, nib, 1);
    if ((lane & 1) == 0) {
      const int s = lane >> 1;
      const uint32_t c = bits | (pbits << 4);
      const size_t key = (size_t)row * a.max_len + t;
      a.cent[key * kSub + s] = (uint8_t)c;
      a.rec[key * 32 + s] = nib | (pnib << 16);
      a.rec[key * 32 + 16 + s] = __float_as_uint((r > 0.f && kn > 0.f && al > 0.f) ? kn * r / al : 0.f);
      atomicAdd(&hist[s][c], 1);
    }
  }
  __syncthreads();
  int32_t* g = a.hist + (size_t)row * kSub * kCent;
  for (int i = threadIdx.x; i < kSub * kCent; i += blockDim.x) {
    const int c = (&hist[0][0])[i];
    if (c) atomicAdd(&g[i], c);
  }
}

// ---------------------------------------------------------------- decode step

struct StepArgs {
  const unsigned char* q;    // scoring queries [B, Hs, 128] bf16
  int Hs, gi;                // scoring heads, scoring heads per KV head
  const int32_t* seq_lens;
  const int8_t* signs;
  const uint8_t* cent;
  const uint32_t* rec;
  const int32_t* hist;
  int32_t* status;
  int B, H, max_len, ns, nl, topk;
  int beta_pm, rho_pm;
  int n_chunks;              // chunk slots per row (max over rows)
  Quant qz;
  // workspace
  float* qt;                 // [rows, 128] rotated unit query
  float* nq;                 // [rows] |q|
  uint8_t* W;                // [rows, 16, 256] tier weights
  float* sim;                // [rows, 16, 256] centroid similarities the tiers were ranked by
  uint8_t* S;                // [rows, max_len] collision scores
  uint32_t* chunk_hist;      // [rows, n_chunks, kSBins]: keys of the chunk scoring >= v
  int2* chunk_info;          // [rows, n_chunks]: (output offset, equal-threshold keys before)
  int2* row_info;            // [rows]: (threshold, keys at the threshold to take)
  uint32_t* ticket;          // [rows]
  uint32_t* row_hist;        // [rows, kSBins] collision-score counts of the row
  int32_t* cand_len;         // [B]
  int32_t* cand;             // [rows, c_cap] candidate positions, ascending
  float* cand_score;         // [rows, c_cap]
  int c_cap;
  const int32_t* sel;        // [rows, topk] selected candidate slots
  int32_t* idx;              // [rows, topk] positions
};

struct RowGeom {
  int L, s_end, l_start, n;
};

__device__ __forceinline__ RowGeom row_geom_of(const StepArgs& a, int b) {
  RowGeom g;
  g.L = load_len(a.seq_lens, b, a.max_len, a.status);
  const Regions r = regions_of(g.L, a.ns, a.nl);
  g.s_end = r.s_end;
  g.l_start = r.l_start;
  g.n = r.l_start - r.s_end;
  return g;
}

__device__ __forceinline__ int ceil_frac(long long n, int per_mille) { return (int)((per_mille * n + 999) / 1000); }

// Exclusive scan of one value per thread over a 256-thread CTA; *total gets the sum.
__device__ __forceinline__ int block_scan256(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int pre = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int w = wsum[i];
    pre += i < warp ? w : 0;
    tot += w;
  }
  __syncthreads();  // wsum may be reused
  *total = tot;
  return pre + x - v;
}

// one CTA per (subspace blockIdx.x, row blockIdx.y); thread tid owns centroid tid
__global__ void __launch_bounds__(256) paris_query_kernel(const StepArgs a) {
  __shared__ float qt[kD];
  __shared__ int cnt[kCent];
  __shared__ unsigned long long key[kCent];
  __shared__ int wsum[8];
  const int s = blockIdx.x, row = blockIdx.y, b = row / a.H, h = row - b * a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowGeom g = row_geom_of(a, b);
  cnt[tid] = a.hist[((size_t)row * kSub + s) * kCent + tid];
  // group-mean query, its norm and rotation (warp 0, 4 values a lane)
  if (warp == 0) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < a.gi; ++j) {
      float x[4];
      load4_bf16(a.q + (((size_t)b * a.Hs + h * a.gi + j) * kD + 4 * lane) * 2, x);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] += x[e];
    }
    const float ig = 1.f / (float)a.gi;
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] *= ig;
    const float n = sqrtf(warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]));
    const float inv = n > 0.f ? 1.f / n : 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = v[e] * inv * (float)a.signs[4 * lane + e];
    fwht128(v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qt[4 * lane + e] = v[e] * 0.08838834764831845f;
      if (s == 0) a.qt[(size_t)row * kD + 4 * lane + e] = qt[4 * lane + e];
    }
    if (s == 0 && lane == 0) a.nq[row] = n;
  }
  __syncthreads();
  // the sink [0, s_end) and local [l_start, L) keys leave the counts
  const int n_out = g.s_end + (g.L - g.l_start);
  for (int j = tid; j < n_out; j += 256) {
    const int t = j < g.s_end ? j : g.l_start + (j - g.s_end);
    atomicSub(&cnt[a.cent[((size_t)row * a.max_len + t) * kSub + s]], 1);
  }
  // similarity of centroid tid: sum_j (bit j ? -1 : 1) qt[8s + j], then / sqrt 8
  float sim = 0.f;
#pragma unroll
  for (int j = 0; j < kM; ++j) sim += ((tid >> j) & 1) ? -qt[kM * s + j] : qt[kM * s + j];
  sim *= 0.35355339059327373f;
  a.sim[((size_t)row * kSub + s) * kCent + tid] = sim;
  // ascending sort key: larger similarity first, then the lower id
  key[tid] = ((unsigned long long)(~order_key(sim)) << 32) | (unsigned)tid;
  __syncthreads();
  for (int k = 2; k <= kCent; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int p = tid ^ j;
      if (p > tid) {
        const unsigned long long x = key[tid], y = key[p];
        if ((x > y) == ((tid & k) == 0)) {
          key[tid] = y;
          key[p] = x;
        }
      }
      __syncthreads();
    }
  }
  // thread tid holds rank tid: keys in better-ranked centroids, then the tier weight
  const int c = (int)(key[tid] & 0xffu);
  int total;
  const int start = block_scan256(cnt[c], wsum, &total);
  const long long N = (long long)ceil_frac(g.n, a.rho_pm);
  int wgt = 0;
  if (start < N) {
    wgt = 1;
#pragma unroll
    for (int i = 4; i >= 0; --i)
      if (start < (int)((kTierPct[i] * N + 99) / 100)) wgt = 6 - i;
  }
  a.W[((size_t)row * kSub + s) * kCent + c] = (uint8_t)wgt;
  if (s == 0 && h == 0 && tid == 0) {
    const int C = ceil_frac(g.n, a.beta_pm);
    a.cand_len[b] = C < g.n ? C : g.n;
  }
}

__global__ void __launch_bounds__(256) paris_collision_kernel(const StepArgs a) {
  // byte weights, 256 a subspace: a lookup is one byte load at (subspace * 256 + centroid),
  // the subspace part an immediate; 64 words over 32 banks conflict at most two ways
  __shared__ __align__(16) uint8_t W[kSub][kCent];
  __shared__ uint32_t sh[kSBins];
  __shared__ bool last;
  __shared__ int tsel[2];
  const int row = blockIdx.y, b = row / a.H;
  const int tid = threadIdx.x;
  const RowGeom g = row_geom_of(a, b);
  const int chunks = (g.n + kChunk - 1) / kChunk;
  if ((int)blockIdx.x >= chunks) return;
  pdl_wait();
  reinterpret_cast<uint4*>(&W[0][0])[tid] =
      reinterpret_cast<const uint4*>(a.W + (size_t)row * kSub * kCent)[tid];  // 4 KB = 256 x 16 bytes
  if (tid < kSBins) sh[tid] = 0;
  __syncthreads();
  const int base = g.s_end + blockIdx.x * kChunk;
  const int end = min(base + kChunk, g.l_start);
  const uint4* crow = reinterpret_cast<const uint4*>(a.cent + (size_t)row * a.max_len * kSub);
  constexpr int kU = 4;  // keys in flight per thread
  for (int w0 = base; w0 < end; w0 += kU * 256) {  // the same rounds for every thread
    uint4 c[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int t = w0 + u * 256 + tid;
      c[u] = t < end ? __ldg(crow + t) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int t = w0 + u * 256 + tid;
      const bool live = t < end;
      const uint32_t wd[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
      int S = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) S += W[4 * i + j][(wd[i] >> (8 * j)) & 0xffu];
      if (live) a.S[(size_t)row * a.max_len + t] = (uint8_t)S;
      // one shared atomic per distinct score in the warp
      const unsigned grp = __match_any_sync(0xffffffffu, live ? S : -1);
      if (live && (tid & 31) == __ffs(grp) - 1) atomicAdd(&sh[S], (uint32_t)__popc(grp));
    }
  }
  __syncthreads();
  // this chunk's counts at or above every score (suffix sums: two loads give the counts
  // above and at any threshold), and the row's totals
  uint32_t* hg = a.chunk_hist + ((size_t)row * a.n_chunks + blockIdx.x) * kSBins;
  __shared__ uint32_t wtot[kSBins / 32];
  uint32_t cum = 0;
  if (tid < kSBins) {  // warps 0-3: suffix sums by shuffles, then the later warps' totals
    const int lane = tid & 31;
    cum = sh[tid];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, cum, o);
      if (lane + o < 32) cum += y;
    }
    if (lane == 0) wtot[tid >> 5] = cum;
  }
  __syncthreads();
  if (tid < kSBins) {
    for (int w2 = (tid >> 5) + 1; w2 < kSBins / 32; ++w2) cum += wtot[w2];
    hg[tid] = cum;
    if (tid <= kMaxS && sh[tid] != 0u) atomicAdd(&a.row_hist[(size_t)row * kSBins + tid], sh[tid]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(&a.ticket[row], 1u) == (unsigned)(chunks - 1);
  __syncthreads();
  if (!last) return;
  // the row's last CTA: bucket top-k over the small integer scores
  __threadfence();
  const uint32_t* hr = a.chunk_hist + (size_t)row * a.n_chunks * kSBins;
  if (tid < kSBins) sh[tid] = __ldcg(a.row_hist + (size_t)row * kSBins + tid);
  __syncthreads();
  if (tid == 0) {
    const int C = min(ceil_frac(g.n, a.beta_pm), g.n);
    int t = kSBins, need = 0;
    long long above = 0;
    if (C > 0) {
      for (int v = kMaxS; v >= 0; --v) {
        if (above + sh[v] >= (long long)C) {
          t = v;
          need = (int)(C - above);
          break;
        }
        above += sh[v];
      }
    }
    tsel[0] = t;
    tsel[1] = need;
    a.row_info[row] = make_int2(t, need);
  }
  __syncthreads();
  const int t = tsel[0], need = tsel[1];
  // per chunk: keys above the threshold, keys at it; exclusive scans over the chunks
  __shared__ int carry[2];
  if (tid == 0) carry[0] = carry[1] = 0;
  __syncthreads();
  for (int j0 = 0; j0 < chunks; j0 += 256) {
    const int j = j0 + tid;
    int gt = 0, eq = 0;
    if (j < chunks && t <= kMaxS) {
      const uint32_t* hj = hr + (size_t)j * kSBins;
      gt = (int)__ldcg(hj + t + 1);
      eq = (int)__ldcg(hj + t) - gt;
    }
    // block-wide exclusive scans of eq, then of gt + take (two passes, same carry scheme)
    __shared__ int ws[8];
    int x = eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if ((tid & 31) >= o) x += y;
    }
    if ((tid & 31) == 31) ws[tid >> 5] = x;
    __syncthreads();
    int wpre = 0;
    for (int i = 0; i < (tid >> 5); ++i) wpre += ws[i];
    const int eq_before = carry[1] + wpre + x - eq;
    int blk_eq = 0;
    for (int i = 0; i < 8; ++i) blk_eq += ws[i];
    __syncthreads();
    int take = need - eq_before;
    take = take < 0 ? 0 : (take > eq ? eq : take);
    const int own = gt + take;
    int y2 = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, y2, o);
      if ((tid & 31) >= o) y2 += y;
    }
    if ((tid & 31) == 31) ws[tid >> 5] = y2;
    __syncthreads();
    int wpre2 = 0;
    for (int i = 0; i < (tid >> 5); ++i) wpre2 += ws[i];
    const int off = carry[0] + wpre2 + y2 - own;
    int blk_own = 0;
    for (int i = 0; i < 8; ++i) blk_own += ws[i];
    if (j < chunks) a.chunk_info[(size_t)row * a.n_chunks + j] = make_int2(off, eq_before);
    __syncthreads();
    if (tid == 0) {
      carry[0] += blk_own;
      carry[1] += blk_eq;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256, 4) paris_compact_kernel(const StepArgs a) {
  __shared__ float qt[kD];
  __shared__ float lvl[8];
  __shared__ int list[kChunk];
  __shared__ int wsum[8];
  const int row = blockIdx.y, b = row / a.H;
  const int tid = threadIdx.x;
  const RowGeom g = row_geom_of(a, b);
  const int chunks = (g.n + kChunk - 1) / kChunk;
  if ((int)blockIdx.x >= chunks) return;
  pdl_wait();
  if (tid < kD) qt[tid] = a.qt[(size_t)row * kD + tid];
  if (tid < 8) lvl[tid] = a.qz.level[tid];
  const int2 ri = a.row_info[row];
  const int2 ci = a.chunk_info[(size_t)row * a.n_chunks + blockIdx.x];
  const int t_thr = ri.x, need = ri.y;
  const int base = g.s_end + blockIdx.x * kChunk;
  const int end = min(base + kChunk, g.l_start);
  // thread tid: the 32 consecutive positions base + 32 tid .. base + 32 tid + 31, their
  // scores packed four a word (255 past the end: never a score, never selected)
  constexpr int kPer = kChunk / 256;
  static_assert(kPer == 32, "one selection bit a position");
  const int p0 = base + kPer * tid;
  const uint8_t* srow = a.S + (size_t)row * a.max_len;
  uint32_t sw[kPer / 4];
  if (p0 + kPer <= end && (((uintptr_t)(srow + p0)) & 15u) == 0) {
    const uint4 u0 = *reinterpret_cast<const uint4*>(srow + p0);
    const uint4 u1 = *reinterpret_cast<const uint4*>(srow + p0 + 16);
    sw[0] = u0.x; sw[1] = u0.y; sw[2] = u0.z; sw[3] = u0.w;
    sw[4] = u1.x; sw[5] = u1.y; sw[6] = u1.z; sw[7] = u1.w;
  } else {
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      uint32_t wv = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int p = p0 + 4 * q + e;
        wv |= (uint32_t)(p < end ? srow[p] : 255u) << (8 * e);
      }
      sw[q] = wv;
    }
  }
  auto score_at = [&](int e) { return (int)((sw[e >> 2] >> (8 * (e & 3))) & 0xffu); };
  int n_eq = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) n_eq += score_at(e) == t_thr ? 1 : 0;
  int tot;
  int tie = ci.y + block_scan256(n_eq, wsum, &tot);  // keys at the threshold before this thread's
  unsigned pick = 0;
  int n_sel = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int sv = score_at(e);
    bool sel = sv > t_thr && sv != 255;
    if (sv == t_thr) sel = tie++ < need;
    pick |= (sel ? 1u : 0u) << e;
    n_sel += sel ? 1 : 0;
  }
  int total;
  int at = block_scan256(n_sel, wsum, &total);
#pragma unroll
  for (int e = 0; e < kPer; ++e)
    if ((pick >> e) & 1u) list[at++] = p0 + e;
  __syncthreads();
  // rerank: one thread a candidate, 64 bytes of codes and 64 of weights in 8 vector loads
  int32_t* cand = a.cand + (size_t)row * a.c_cap + ci.x;
  float* cs = a.cand_score + (size_t)row * a.c_cap + ci.x;
  const float nq = a.nq[row];
  for (int i = tid; i < total; i += 256) {
    const int p = list[i];
    const uint4* rv = reinterpret_cast<const uint4*>(a.rec + ((size_t)row * a.max_len + p) * 32);
    uint4 c4[4];
    float4 w4[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      c4[v] = __ldg(rv + v);
      const uint4 u = __ldg(rv + 4 + v);
      w4[v] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
    }
    float acc = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint32_t cw[4] = {c4[v].x, c4[v].y, c4[v].z, c4[v].w};
      const float ww[4] = {w4[v].x, w4[v].y, w4[v].z, w4[v].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int s = 4 * v + q;
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < kM; ++j) {
          const uint32_t nb = (cw[q] >> (4 * j)) & 15u;
          const float lv = lvl[nb & 7u];
          dot += (nb & 8u ? -lv : lv) * qt[kM * s + j];
        }
        acc += ww[q] * dot;
      }
    }
    cand[i] = p;
    cs[i] = nq * acc;
  }
}

__global__ void __launch_bounds__(256) paris_map_kernel(const StepArgs a) {
  pdl_wait();
  const long long n = (long long)a.B * a.H * a.topk;
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n; i += (long long)gridDim.x * 256) {
    const int row = (int)(i / a.topk);
    const int j = a.sel[i];
    a.idx[i] = j >= 0 ? a.cand[(size_t)row * a.c_cap + j] : -1;
  }
}

// ---------------------------------------------------------------- workspace

struct ParisLayout {
  size_t qt, nq, W, sim, S, chunk_hist, chunk_info, row_info, ticket, row_hist, cand_len, cand, cand_score, topk, sel,
      total;
  int n_chunks, c_cap;
};

skv_problem cand_problem(const skv_problem& p, int c_cap, const int32_t* cand_len) {
  skv_problem r = p;
  r.max_len = c_cap;
  r.n_sink = 0;
  r.n_local = 0;
  r.seq_lens = cand_len;
  return r;
}

ParisLayout paris_layout(const skv_problem& p, const skv_paris& pr) {
  ParisLayout l;
  const size_t rows = (size_t)p.batch * p.n_kv_heads;
  l.n_chunks = (p.max_len + kChunk - 1) / kChunk;
  if (l.n_chunks < 1) l.n_chunks = 1;
  const long long cmax = ((long long)pr.beta_pm * p.max_len + 999) / 1000;
  l.c_cap = (int)(((cmax < 1 ? 1 : cmax) + 15) / 16 * 16);
  l.qt = 0;
  l.nq = l.qt + align256(rows * kD * 4);
  l.W = l.nq + align256(rows * 4);
  l.sim = l.W + align256(rows * kSub * kCent);
  l.S = l.sim + align256(rows * kSub * kCent * 4);
  l.chunk_hist = l.S + align256(rows * (size_t)p.max_len);
  l.chunk_info = l.chunk_hist + align256(rows * l.n_chunks * kSBins * 4);
  l.row_info = l.chunk_info + align256(rows * l.n_chunks * 8);
  l.ticket = l.row_info + align256(rows * 8);  // tickets, then the row histograms: one memset
  l.row_hist = l.ticket + rows * 4;
  l.cand_len = l.ticket + align256(rows * 4 + rows * kSBins * 4);
  l.cand = l.cand_len + align256((size_t)p.batch * 4);
  l.cand_score = l.cand + align256(rows * (size_t)l.c_cap * 4);
  l.topk = l.cand_score + align256(rows * (size_t)l.c_cap * 4);
  l.sel = l.topk + align256(topk_workspace_bytes(cand_problem(p, l.c_cap, nullptr)));
  l.total = l.sel + align256(rows * (size_t)(p.topk > 0 ? p.topk : 1) * 4);
  return l;
}

}  // namespace

skv_status paris_quantizer(int m, float* levels, float* thresholds) {
  if (m < 3 || m > 64) return SKV_ERR_INVALID_ARGUMENT;
  const Quant q = quant_for(m);
  for (int i = 0; i < 8; ++i) levels[i] = q.level[i];
  for (int i = 0; i < 7; ++i) thresholds[i] = q.thr[i];
  return SKV_OK;
}

size_t paris_workspace_bytes(const skv_problem& p, const skv_paris& pr) { return paris_layout(p, pr).total; }

void paris_offsets(const skv_problem& p, const skv_paris& pr, int64_t* out) {
  const ParisLayout l = paris_layout(p, pr);
  out[0] = (int64_t)l.qt;
  out[1] = (int64_t)l.nq;
  out[2] = (int64_t)l.W;
  out[3] = (int64_t)l.S;
  out[4] = (int64_t)l.cand_len;
  out[5] = (int64_t)l.cand;
  out[6] = (int64_t)l.cand_score;
  out[7] = (int64_t)l.c_cap;
  out[8] = (int64_t)l.sim;
}

skv_status launch_paris_encode(const skv_problem& p, const skv_paris& pr, const skv_index_src& src,
                               const PoolView& pool, const skv_paris_index& ix, int32_t* status, cudaStream_t st) {
  const int rows = p.batch * p.n_kv_heads;
  EncArgs a{};
  a.keys = src.layout == SKV_INDEX_CONTIG ? (const unsigned char*)src.keys : nullptr;
  a.pool = pool;
  a.seq_lens = p.seq_lens;
  a.signs = pr.signs;
  a.cent = ix.cent;
  a.rec = ix.rec;
  a.hist = ix.hist;
  a.status = status;
  a.H = p.n_kv_heads;
  a.max_len = p.max_len;
  a.bs = p.block_size;
  a.qz = quant_for(pr.m);
  if (cudaMemsetAsync(ix.hist, 0, (size_t)rows * kSub * kCent * 4, st) != cudaSuccess) return SKV_ERR_CUDA;
  const int gx = (p.max_len + kEncKeys - 1) / kEncKeys;
  if (gx == 0 || rows == 0) return SKV_OK;
  paris_encode_kernel<<<dim3(gx, rows), 256, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

skv_status launch_paris_select(const skv_problem& p, const skv_paris& pr, const void* q_score,
                               const skv_paris_index& ix, int32_t* idx, void* pws, int32_t* status, cudaStream_t st) {
  const int rows = p.batch * p.n_kv_heads;
  if (rows == 0) return SKV_OK;
  const ParisLayout l = paris_layout(p, pr);
  unsigned char* w = (unsigned char*)pws;
  StepArgs a{};
  a.q = (const unsigned char*)q_score;
  a.Hs = p.n_idx_q_heads;
  a.gi = p.n_idx_q_heads / p.n_kv_heads;
  a.seq_lens = p.seq_lens;
  a.signs = pr.signs;
  a.cent = ix.cent;
  a.rec = ix.rec;
  a.hist = ix.hist;
  a.status = status;
  a.B = p.batch;
  a.H = p.n_kv_heads;
  a.max_len = p.max_len;
  a.ns = p.n_sink;
  a.nl = p.n_local;
  a.topk = p.topk;
  a.beta_pm = pr.beta_pm;
  a.rho_pm = pr.rho_pm;
  a.n_chunks = l.n_chunks;
  a.qz = quant_for(pr.m);
  a.qt = (float*)(w + l.qt);
  a.nq = (float*)(w + l.nq);
  a.W = (uint8_t*)(w + l.W);
  a.sim = (float*)(w + l.sim);
  a.S = (uint8_t*)(w + l.S);
  a.chunk_hist = (uint32_t*)(w + l.chunk_hist);
  a.chunk_info = (int2*)(w + l.chunk_info);
  a.row_info = (int2*)(w + l.row_info);
  a.ticket = (uint32_t*)(w + l.ticket);
  a.row_hist = (uint32_t*)(w + l.row_hist);
  a.cand_len = (int32_t*)(w + l.cand_len);
  a.cand = (int32_t*)(w + l.cand);
  a.cand_score = (float*)(w + l.cand_score);
  a.c_cap = l.c_cap;
  a.sel = (const int32_t*)(w + l.sel);
  a.idx = idx;
  if (cudaMemsetAsync(a.ticket, 0, (size_t)rows * 4 * (1 + kSBins), st) != cudaSuccess) return SKV_ERR_CUDA;
  paris_query_kernel<<<dim3(kSub, rows), 256, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  if (launch_dependent(paris_collision_kernel, dim3(l.n_chunks, rows), dim3(256), 0, st, 1, a) != cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  if (launch_dependent(paris_compact_kernel, dim3(l.n_chunks, rows), dim3(256), 0, st, 1, a) != cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  if (p.topk > 0) {
    const skv_problem cp = cand_problem(p, l.c_cap, a.cand_len);
    if (topk_maps_positions(cp))  // the selection writes the candidates' positions itself
      return launch_topk(cp, a.cand_score, idx, w + l.topk, status, st, nullptr, nullptr, nullptr, nullptr, a.cand);
    const skv_status r = launch_topk(cp, a.cand_score, (int32_t*)(w + l.sel), w + l.topk, status, st);
    if (r != SKV_OK) return r;
    const long long n = (long long)rows * p.topk;
    const long long blocks = (n + 255) / 256;
    const unsigned grid = (unsigned)(blocks < 4096 ? blocks : 4096);
    if (launch_dependent(paris_map_kernel, dim3(grid), dim3(256), 0, st, 1, a) != cudaSuccess) return SKV_ERR_CUDA;
    SKV_LAUNCH_CHECK();
  }
  return SKV_OK;
}

}  // namespace skv
