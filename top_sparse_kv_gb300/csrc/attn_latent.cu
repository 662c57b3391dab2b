// S3 + S4 + S5 for the MLA-style latent layout (one shared latent row per token).
//
// Every token has one row of 576 entries (512 latent + 64 rope) shared by all
// query heads; V is the first 512 entries of that row (UlaCache article §3: MLA
// keeps one latent across heads; ECHO-OSDI26 wiki: the DSA indexer picks the
// top-k tokens whose latent rows attention reads).  With 128 absorbed heads the
// attention is a real contraction per request -- Q [128 x 576] against the
// selected rows -- so it runs on tensor cores.
//
// Two kernels:
//   latent_gather_kernel  every attended row is resolved through the per-token
//                         slot map and copied once -- from the GPU slot cache
//                         in HBM, or from the pinned host pool over UVA -- into
//                         a contiguous workspace buffer (plus a validity byte).
//                         Host rows therefore cross the host link exactly once.
//   attn_latent_kernel    one CTA per (row split, 64-head group, request): the
//                         64 heads' queries stay in shared memory; 32-row tiles
//                         of the gathered buffer stream through a 2-stage
//                         cp.async ring.  Warp w owns heads 16*(w%4).. of the
//                         group and half (w/4) of the 512 output dims:
//                           S[16 x 32] = Q K^T over 576 dims   (mma.m16n8k16, ldmatrix)
//                           fp32 online softmax per head (exp2 units)
//                           O[16 x 256] += P V                 (P from the S registers,
//                                                              V via ldmatrix.trans)
//                         Partials (m, l, O) per split; the last CTA of the
//                         request merges them by log-sum-exp.
#include "attn_common.cuh"

namespace skv {
namespace {

namespace lat {
constexpr int kD = 576;
constexpr int kDV = 512;
constexpr int kChunks = kD * 2 / 16;  // 72 16-byte chunks per row
constexpr int kRowB = kD * 2;         // 1152
constexpr int kHeads = 64;            // heads per CTA
constexpr int kRows = 32;             // rows per tile
constexpr int kStages = 2;
constexpr int kThreads = 256;
constexpr int kQBytes = kHeads * kRowB;
constexpr int kTileB = kRows * kRowB;
constexpr int kSmem = kQBytes + kStages * kTileB + kStages * kRows;
// byte offset of chunk c of row r in a swizzled [rows x 72 chunks] tile (the XOR
// stays inside each group of 8 chunks, and 72 is a multiple of 8)
__device__ __forceinline__ int swz(int r, int c) { return r * kRowB + ((c ^ (r & 7)) << 4); }
}  // namespace lat

struct LatentArgs {
  AttnArgs m;                  // sizes, slot table, merge buffers, output
  const unsigned char* rows;   // [B, n_att, 576] bf16 gathered rows
  uint8_t* valid;              // [B, n_att]
  int n_att, n_hgroups;
};

__global__ void latent_gather_kernel(const LatentArgs la) {
  const AttnArgs& a = la.m;
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)a.B * la.n_att) return;
  const int b = (int)(w / la.n_att), j = (int)(w % la.n_att);
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const Regions rg = regions_of(L, a.ns, a.nl);
  const int n_list = rg.s_end + a.k + (L - rg.l_start);
  const int32_t* idx_row = a.idx + (size_t)b * a.k;  // one KV head
  const int t = list_pos(a, idx_row, rg, j, n_list);
  const unsigned char* src = nullptr;
  if (t >= 0) {
    const int e = a.pool.table[(size_t)b * a.pool.stride + t / a.bs];
    const size_t off = (size_t)(t % a.bs);
    if (e >= 0 && e < a.pool.n_gpu) {
      src = (const unsigned char*)a.pool.gpu_k + ((size_t)e * a.bs + off) * lat::kRowB;
    } else if (e < 0 && a.pool.host_k != nullptr && -(long long)e - 1 < a.pool.n_host) {
      src = (const unsigned char*)a.pool.host_k + ((size_t)(-(long long)e - 1) * a.bs + off) * lat::kRowB;
    } else {
      flag(a.status, SKV_DEV_BAD_SLOT);
    }
  }
  uint4* dst = (uint4*)(la.rows + (size_t)w * lat::kRowB);
  for (int c = lane; c < lat::kChunks; c += 32) dst[c] = src ? ((const uint4*)src)[c] : make_uint4(0, 0, 0, 0);
  if (lane == 0) la.valid[w] = src != nullptr;
}

__global__ void __launch_bounds__(lat::kThreads, 1) attn_latent_kernel(const LatentArgs la) {
  const AttnArgs& a = la.m;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* qs = smem;
  unsigned char* ks = smem + lat::kQBytes;
  uint8_t* vm = (uint8_t*)(ks + lat::kStages * lat::kTileB);

  const int s = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int hb = warp & 3, half = warp >> 2;
  const int j0 = s * a.chunk;
  int j1 = j0 + a.chunk;
  j1 = j1 < la.n_att ? j1 : la.n_att;
  const int ntiles = j1 > j0 ? (j1 - j0 + lat::kRows - 1) / lat::kRows : 0;

  // the group's 64 query rows
  const unsigned char* qg = a.q + ((size_t)b * a.Hq + (size_t)hg * lat::kHeads) * lat::kRowB;
  for (int c = threadIdx.x; c < lat::kHeads * lat::kChunks; c += lat::kThreads) {
    const int r = c / lat::kChunks, ch = c - r * lat::kChunks;
    tc::cp_async16_zfill(qs + lat::swz(r, ch), qg + (size_t)r * lat::kRowB + ch * 16, true);
  }
  auto issue = [&](int tile, int st) {
    const int rbase = j0 + tile * lat::kRows;
    unsigned char* kd = ks + st * lat::kTileB;
    for (int c = threadIdx.x; c < lat::kRows * lat::kChunks; c += lat::kThreads) {
      const int r = c / lat::kChunks, ch = c - r * lat::kChunks;
      const int j = rbase + r;
      const bool ok = j < j1;
      const unsigned char* src = ok ? la.rows + ((size_t)b * la.n_att + j) * lat::kRowB + ch * 16 : la.rows;
      tc::cp_async16_zfill(kd + lat::swz(r, ch), src, ok);
    }
    if (threadIdx.x < lat::kRows) {
      const int j = rbase + threadIdx.x;
      vm[st * lat::kRows + threadIdx.x] = j < j1 ? la.valid[(size_t)b * la.n_att + j] : 0;
    }
  };
  if (ntiles > 0) issue(0, 0);
  cp_async_commit();

  float o[32][4];
#pragma unroll
  for (int nt = 0; nt < 32; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nt][c] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  const uint32_t qb = smem_u32(qs);

  for (int i = 0; i < ntiles; ++i) {
    if (i + 1 < ntiles) issue(i + 1, (i + 1) % lat::kStages);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int st = i % lat::kStages;
    const uint32_t kb = smem_u32(ks + st * lat::kTileB);
    const uint8_t* v = vm + st * lat::kRows;

    float sacc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) sacc[j][c] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < lat::kD / 16; ++kk) {
      uint32_t qa[4];
      tc::ldsm_x4(qb + lat::swz(16 * hb + (lane & 15), 2 * kk + (lane >> 4)), qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        uint32_t b0, b1, b2, b3;
        tc::ldsm_x4(kb + lat::swz(16 * jp + 8 * (lane >> 4) + (lane & 7), 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
        tc::mma_bf16(sacc[2 * jp], qa, b0, b1);
        tc::mma_bf16(sacc[2 * jp + 1], qa, b2, b3);
      }
    }
    // online softmax (hr 0: head g, hr 1: head g + 8 of this warp's 16)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int row = 8 * j + 2 * t4 + (c & 1);
        const float z = v[row] ? sacc[j][c] * a.scale_log2 : -INFINITY;
        sacc[j][c] = z;
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
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float z = sacc[j][c];
        const float e = z == -INFINITY ? 0.f : exp2f(z - m_r[c >> 1]);
        sacc[j][c] = e;
        ps[c >> 1] += e;
      }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) l_r[hr] = l_r[hr] * alpha[hr] + ps[hr];
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) {
      o[nt][0] *= alpha[0];
      o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1];
      o[nt][3] *= alpha[1];
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {  // rows 16*kk .. 16*kk+15
      uint32_t pa[4];
      pa[0] = tc::pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
      pa[1] = tc::pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
      pa[2] = tc::pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
      pa[3] = tc::pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
      for (int np = 0; np < 16; ++np) {
        const int mi = lane >> 3;
        const int row = 16 * kk + 8 * (mi & 1) + (lane & 7);
        const int ch = 32 * half + 2 * np + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        tc::ldsm_x4_t(kb + lat::swz(row, ch), b0, b1, b2, b3);
        tc::mma_bf16(o[2 * np], pa, b0, b1);
        tc::mma_bf16(o[2 * np + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // partials: each (head, output dim) is owned by exactly one warp of the CTA
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 1);
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 2);
  }
  const int S = a.n_splits;
#pragma unroll
  for (int nt = 0; nt < 32; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int head = hg * lat::kHeads + 16 * hb + g + ((c >> 1) ? 8 : 0);
      const int d = 256 * half + 8 * nt + 2 * t4 + (c & 1);
      const size_t hq = (size_t)b * a.Hq + head;
      a.ws_o[(hq * S + s) * lat::kDV + d] = o[nt][c];
    }
  if (half == 0 && t4 == 0) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const size_t hq = (size_t)b * a.Hq + hg * lat::kHeads + 16 * hb + g + 8 * hr;
      a.ws_ml[(hq * S + s) * 2 + 0] = m_r[hr];
      a.ws_ml[(hq * S + s) * 2 + 1] = l_r[hr];
    }
  }
  merge_if_last(a, b, 0, S * la.n_hgroups);
}

// Splits of the 2048-class row list: minimise waves x (tiles per CTA + the query
// load) with one resident CTA per SM on the 152 SMs of a GB300.
int latent_splits(const skv_problem& p) {
  const int n = max_list(p);
  const int tiles = n > 0 ? (n + lat::kRows - 1) / lat::kRows : 1;
  if (p.n_splits > 0) return p.n_splits < tiles ? p.n_splits : tiles;
  const long long units = (long long)p.batch * (p.n_q_heads / lat::kHeads);
  int best = 1;
  long long best_cost = -1;
  for (int sp = 1; sp <= tiles && sp <= 64; ++sp) {
    const long long waves = (units * sp + 151) / 152;
    const long long cost = waves * ((tiles + sp - 1) / sp + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = sp;
    }
  }
  return best;
}

struct LatentLayout {
  size_t rows, valid, o, ml, tickets, total;
};

LatentLayout latent_layout(const skv_problem& p) {
  const size_t n = (size_t)max_list(p), B = (size_t)p.batch, S = (size_t)latent_splits(p);
  LatentLayout l;
  l.rows = 0;
  l.valid = l.rows + align256(B * n * lat::kRowB);
  l.o = l.valid + align256(B * n);
  l.ml = l.o + align256(B * p.n_q_heads * S * lat::kDV * 4);
  l.tickets = l.ml + align256(B * p.n_q_heads * S * 2 * 4);
  l.total = l.tickets + align256(B * 4);
  return l;
}

}  // namespace

bool latent_shape(const skv_problem& p) {
  return p.d_qk == lat::kD && p.d_v == lat::kDV && p.n_kv_heads == 1 && p.n_q_heads % lat::kHeads == 0 &&
         p.dtype == SKV_DTYPE_BF16;
}

size_t latent_workspace_bytes(const skv_problem& p) { return latent_layout(p).total; }

skv_status launch_attn_latent(const skv_problem& p, const void* q, const PoolView& pool, const int32_t* idx,
                              void* out, float* lse, void* ws, int32_t* status, cudaStream_t st) {
  const LatentLayout lay = latent_layout(p);
  LatentArgs la;
  la.m = make_args(p, q, pool, idx, status);
  la.n_att = max_list(p);
  la.n_hgroups = p.n_q_heads / lat::kHeads;
  la.m.n_splits = latent_splits(p);
  la.m.chunk = la.n_att > 0 ? (la.n_att + la.m.n_splits - 1) / la.m.n_splits : 1;
  unsigned char* w = (unsigned char*)ws;
  la.rows = w + lay.rows;
  la.valid = (uint8_t*)(w + lay.valid);
  la.m.ws_o = (float*)(w + lay.o);
  la.m.ws_ml = (float*)(w + lay.ml);
  la.m.tickets = (uint32_t*)(w + lay.tickets);
  la.m.out = out;
  la.m.lse = lse;
  if (la.n_att == 0) return SKV_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(la.m.tickets, 0, (size_t)p.batch * 4, st) != cudaSuccess) return SKV_ERR_CUDA;
  const long long warps = (long long)p.batch * la.n_att;
  latent_gather_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(la);
  SKV_LAUNCH_CHECK();
  static int configured = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SKV_ERR_CUDA;
  if (configured != dev) {
    if (cudaFuncSetAttribute(attn_latent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lat::kSmem) !=
        cudaSuccess)
      return SKV_ERR_CUDA;
    configured = dev;
  }
  dim3 grid(la.m.n_splits, la.n_hgroups, p.batch);
  attn_latent_kernel<<<grid, lat::kThreads, lat::kSmem, st>>>(la);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace skv
