// S3 + S4 + S5 for the MLA-style latent layout (one shared latent row per token).
//
// Every token has one row of 576 entries (512 latent + 64 rope) shared by all
// query heads; V is the first 512 entries of that row (UlaCache article §3: MLA
// keeps one latent across heads; ECHO-OSDI26 wiki: the DSA indexer picks the
// top-k tokens whose latent rows attention reads).  With 128 absorbed heads the
// attention is a real contraction per request -- Q [128 x 576] against the
// selected rows -- so it runs on the tcgen05 tensor cores with TMEM accumulators.
//
// Three kernels:
//   latent_gather_kernel   every attended row is resolved through the per-token
//                          slot map and copied once -- from the GPU slot cache
//                          in HBM, or from the pinned host pool over UVA -- into
//                          a contiguous workspace buffer (plus a validity byte).
//                          Host rows therefore cross the host link exactly once.
//   attn_latent_tc_kernel  one CTA per (256-row block, output-dim half, request):
//                          S and O accumulate in TMEM (see the kernel's comment).
//   latent_merge_kernel    log-sum-exp merge of the blocks' partials.
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
  PrefetchView pf;             // staged host rows (pf.map == nullptr: none)
};

__global__ void latent_gather_kernel(const LatentArgs la) {
  __shared__ unsigned s_staged, s_read;  // prefetch statistics of this CTA
  if (threadIdx.x == 0) s_staged = s_read = 0u;
  __syncthreads();
  pdl_wait();  // the selection is complete and visible
  const AttnArgs& a = la.m;
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const bool live = w < (long long)a.B * la.n_att;
  const int b = live ? (int)(w / la.n_att) : 0, j = live ? (int)(w % la.n_att) : 0;
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  const Regions rg = regions_of(L, a.ns, a.nl);
  const int n_list = rg.s_end + a.k + (L - rg.l_start);
  const int32_t* idx_row = a.idx + (size_t)b * a.k;  // one KV head
  const int t = live ? list_pos(a, idx_row, rg, j, n_list) : -1;
  const unsigned char* src = nullptr;
  if (t >= 0) {
    const int e = a.pool.table[(size_t)b * a.pool.stride + t / a.bs];
    const size_t off = (size_t)(t % a.bs);
    if (e >= 0 && e < a.pool.n_gpu) {
      src = (const unsigned char*)a.pool.gpu_k + ((size_t)e * a.bs + off) * lat::kRowB;
    } else if (e < 0 && a.pool.host_k != nullptr && -(long long)e - 1 < a.pool.n_host) {
      src = (const unsigned char*)a.pool.host_k + ((size_t)(-(long long)e - 1) * a.bs + off) * lat::kRowB;
      if (la.pf.map != nullptr) {  // staged this step while the indexer scored: read it from HBM
        const unsigned long long tag = (unsigned long long)(*la.pf.epoch + 1u) << 32;
        const unsigned long long mv = la.pf.map[(size_t)b * a.max_len + t];
        const bool staged = (mv & 0xFFFFFFFF00000000ull) == tag && (mv & 0xFFFFFFFFull) < (unsigned)la.pf.cap;
        if (staged) src = la.pf.staging + ((size_t)b * la.pf.cap + (mv & 0xFFFFFFFFull)) * lat::kRowB;
        if (la.pf.stats != nullptr && lane == 0) atomicAdd(staged ? &s_staged : &s_read, 1u);
      }
    } else {
      flag(a.status, SKV_DEV_BAD_SLOT);
    }
  }
  if (live) {
    uint4* dst = (uint4*)(la.rows + (size_t)w * lat::kRowB);
    for (int c = lane; c < lat::kChunks; c += 32) dst[c] = src ? ((const uint4*)src)[c] : make_uint4(0, 0, 0, 0);
    if (lane == 0) la.valid[w] = src != nullptr;
  }
  if (la.pf.stats != nullptr) {  // one atomic per counter per CTA
    __syncthreads();
    if (threadIdx.x == 0 && s_staged) atomicAdd(&la.pf.stats[0], s_staged);
    if (threadIdx.x == 0 && s_read) atomicAdd(&la.pf.stats[1], s_read);
  }
}

// ---------------------------------------------------------------------------- tcgen05 (TMEM) path
namespace t5 {
constexpr int kRows = 256;               // attended rows per CTA (one block)
constexpr int kHalfDv = 256;             // output dims per CTA
constexpr int kThreads = 128;            // one thread per head = one TMEM lane
constexpr int kAtoms = 9;                // 576 dims = 9 slices of 64
constexpr int kQAtom = 128 * 128;        // 128 heads x 64 dims (bf16), 16 KB
constexpr int kKAtom = kRows * 128;      // 256 rows x 64 dims, 32 KB
constexpr int kStage = kQAtom + kKAtom;  // 48 KB
constexpr int kRegion1 = 4 * kKAtom;     // 128 KB: two atom stages, later V (4 x 64 dims x 256 rows)
constexpr int kRegion2 = 4 * kQAtom;     // 64 KB: P (128 heads x 256 rows)
constexpr int kSmem = kRegion1 + kRegion2 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;      // S: columns [0, 256), O: [256, 512)

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled block of rows
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// SM100 shared-memory matrix descriptor (start, leading / stride byte offsets, 128B swizzle)
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for this architecture
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}
// instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, M x N
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
}  // namespace t5

// One CTA per (256-row block, output-dim half, request); 4 warps, thread t = head t.
//   S[128 x 256] (TMEM cols 0..255) = sum over 9 dim slices of Q_a K_a^T:
//       Q_a [128 heads x 64] and K_a [256 rows x 64] staged by cp.async in a
//       128B-swizzled K-major layout (2 stages), one thread issues
//       tcgen05.mma M128 N256 K16 x 4 per slice and commits to an mbarrier.
//   softmax per head from tcgen05.ld of its TMEM lane: the block's max m and
//       sum l, P = 2^(z - m) written as bf16 into a swizzled K-major [128 x 256] tile.
//   O[128 x 256] (TMEM cols 256..511) = P V with V read as an MN-major operand
//       straight from the rows' layout (no transpose), K = 256 rows.
// The whole block's S is in TMEM at once, so the softmax is exact per block and
// O never needs rescaling; blocks are merged by log-sum-exp afterwards.
__global__ void __launch_bounds__(t5::kThreads, 1) attn_latent_tc_kernel(const LatentArgs la) {
  const AttnArgs& a = la.m;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ uint8_t mask[t5::kRows];
  __shared__ volatile int s_abort;

  const int s = blockIdx.x, h2 = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);  // generic pointer of the aligned base
  const uint32_t r1 = base, r2 = base + t5::kRegion1;
  unsigned char* g1 = gbase;
  unsigned char* g2 = gbase + t5::kRegion1;

  const int j0 = s * t5::kRows;
  const int j1 = j0 + t5::kRows < la.n_att ? j0 + t5::kRows : la.n_att;
  const unsigned char* rows_b = la.rows + (size_t)b * la.n_att * lat::kRowB;
  const unsigned char* qg = a.q + (size_t)b * a.Hq * lat::kRowB;

  if (t == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  for (int r = t; r < t5::kRows; r += t5::kThreads) {
    const int j = j0 + r;
    mask[r] = j < j1 ? la.valid[(size_t)b * la.n_att + j] : 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(t5::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  t5::fence_before();
  __syncthreads();
  t5::fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  auto load_atom = [&](int at, int st) {
    unsigned char* sq = g1 + st * t5::kStage;
    unsigned char* sk = sq + t5::kQAtom;
    for (int c = t; c < 128 * 8; c += t5::kThreads) {  // Q slice: 128 heads x 8 chunks
      const int r = c >> 3, ch = c & 7;
      tc::cp_async16_zfill(sq + t5::sw128(r, ch), qg + (size_t)r * lat::kRowB + at * 128 + ch * 16, true);
    }
    for (int c = t; c < t5::kRows * 8; c += t5::kThreads) {  // K slice: 256 rows x 8 chunks
      const int r = c >> 3, ch = c & 7;
      const bool ok = mask[r] != 0;
      const unsigned char* src = ok ? rows_b + (size_t)(j0 + r) * lat::kRowB + at * 128 + ch * 16 : la.rows;
      tc::cp_async16_zfill(sk + t5::sw128(r, ch), src, ok);
    }
  };

  // ---- S = Q K^T over the 9 dim slices.  Every thread runs every iteration and
  // every barrier; after a failed wait (s_abort) the MMAs are simply not issued.
  uint32_t phase = 0;    // mbarrier phases this thread has waited for
  uint32_t commits = 0;  // phases committed (thread 0)
  const uint32_t idesc_s = t5::idesc_bf16(128, 256, false);
  load_atom(0, 0);
  cp_async_commit();
  for (int at = 0; at < t5::kAtoms; ++at) {
    if (at >= 1) {  // the MMAs of slice at-1 read the stage that slice at+1 overwrites
      if (!s_abort) wait_or_abort(&bar, phase & 1u, &s_abort, a.status);
      ++phase;
    }
    if (at + 1 < t5::kAtoms) load_atom(at + 1, (at + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0 && !s_abort) {
      t5::fence_after();
      const uint32_t sq = r1 + (at & 1) * t5::kStage, sk = sq + t5::kQAtom;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        t5::mma(tm, t5::desc_sw128(sq + kk * 32, 16, 1024), t5::desc_sw128(sk + kk * 32, 16, 1024), idesc_s,
                (at > 0 || kk > 0) ? 1u : 0u);
      t5::commit(&bar);
      ++commits;
    }
  }
  if (!s_abort) wait_or_abort(&bar, phase & 1u, &s_abort, a.status);
  ++phase;
  __syncthreads();
  bool ok = !s_abort;  // the same in every thread
  t5::fence_after();

  // ---- V rows of this half into region 1 (the stages are free now)
  cp_async_wait<0>();
  __syncthreads();
  for (int c = t; c < t5::kRows * 32; c += t5::kThreads) {  // 256 rows x 4 dim slices x 8 chunks
    const int r = c >> 5, jat = (c >> 3) & 3, ch = c & 7;
    const bool okr = mask[r] != 0;
    const unsigned char* src =
        okr ? rows_b + (size_t)(j0 + r) * lat::kRowB + (h2 * t5::kHalfDv + jat * 64) * 2 + ch * 16 : la.rows;
    tc::cp_async16_zfill(g1 + jat * t5::kKAtom + t5::sw128(r, ch), src, okr);
  }
  cp_async_commit();

  // ---- softmax of head t over the block
  float m = -INFINITY, l = 0.f;
  if (ok) {
    uint32_t v[32];
    for (int ch = 0; ch < 8; ++ch) {
      t5::ld32(tm + lane_base + ch * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (mask[ch * 32 + j]) m = fmaxf(m, __uint_as_float(v[j]) * a.scale_log2);
    }
    for (int ch = 0; ch < 8; ++ch) {
      t5::ld32(tm + lane_base + ch * 32, v);
      float pv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float z = __uint_as_float(v[j]) * a.scale_log2;
        pv[j] = (mask[ch * 32 + j] && m != -INFINITY) ? exp2f(z - m) : 0.f;
        l += pv[j];
      }
      // rows 32ch .. 32ch+31 = slice ch/2, chunks (ch%2)*4 .. +3 of head row t
      unsigned char* prow = g2 + (ch >> 1) * t5::kQAtom;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 w;
        w.x = tc::pack_bf16(pv[8 * i + 0], pv[8 * i + 1]);
        w.y = tc::pack_bf16(pv[8 * i + 2], pv[8 * i + 3]);
        w.z = tc::pack_bf16(pv[8 * i + 4], pv[8 * i + 5]);
        w.w = tc::pack_bf16(pv[8 * i + 6], pv[8 * i + 7]);
        *reinterpret_cast<uint4*>(prow + t5::sw128(t, (ch & 1) * 4 + i)) = w;
      }
    }
  }
  cp_async_wait<0>();
  fence_proxy_async_smem();
  t5::fence_before();
  __syncthreads();
  ok = ok && !s_abort;

  // ---- O = P V
  if (t == 0 && ok) {
    t5::fence_after();
    const uint32_t idesc_o = t5::idesc_bf16(128, 256, true);
#pragma unroll 4
    for (int kk = 0; kk < t5::kRows / 16; ++kk) {
      const uint64_t ad = t5::desc_sw128(r2 + (kk >> 2) * t5::kQAtom + (kk & 3) * 32, 16, 1024);
      const uint64_t bd = t5::desc_sw128(r1 + kk * 2048, t5::kKAtom, 1024);
      t5::mma(tm + 256, ad, bd, idesc_o, kk > 0 ? 1u : 0u);
    }
    t5::commit(&bar);
    ++commits;
  }
  if (ok) {
    wait_or_abort(&bar, phase & 1u, &s_abort, a.status);
    ++phase;
  }
  __syncthreads();
  ok = ok && !s_abort;
  t5::fence_after();

  // ---- partials: O row t (unnormalised), m, l
  const int S = a.n_splits;
  const size_t hq = (size_t)b * a.Hq + t;
  if (ok) {
    uint32_t v[32];
    float* po = a.ws_o + (hq * S + s) * lat::kDV + h2 * t5::kHalfDv;
    for (int ch = 0; ch < 8; ++ch) {
      t5::ld32(tm + lane_base + 256 + ch * 32, v);
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(po + ch * 32 + j) = make_float4(
            __uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
    }
  } else {
    float* po = a.ws_o + (hq * S + s) * lat::kDV + h2 * t5::kHalfDv;
    for (int d = 0; d < t5::kHalfDv; ++d) po[d] = 0.f;
    m = -INFINITY;
    l = 0.f;
  }
  if (h2 == 0) {
    a.ws_ml[(hq * S + s) * 2 + 0] = m;
    a.ws_ml[(hq * S + s) * 2 + 1] = l;
  }
  if (!ok && t == 0) {
    // a wait gave up: let every MMA this thread committed finish before TMEM is released
    for (uint32_t ph = phase; ph < commits; ++ph) mbar_wait_bounded(&bar, ph & 1u);
  }
  t5::fence_before();
  __syncthreads();
  if (warp == 0) {
    t5::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(t5::kTmemCols) : "memory");
  }
}

// Log-sum-exp merge of the blocks, one CTA per (query head, request), four
// output dims per thread:  m* = max m_s, l = sum l_s 2^(m_s - m*),
// out = sum acc_s 2^(m_s - m*) / l,  lse = ln 2 (m* + log2 l).
__global__ void __launch_bounds__(128) latent_merge_kernel(const AttnArgs a, const PrefetchView pf) {
  __shared__ float w[64];
  __shared__ float s_inv;
  if (pf.map != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    // the step's end: later steps tag their staged rows anew and start with empty staging
    *pf.epoch += 1u;
    for (int r = 0; r < a.B * a.H; ++r) pf.count[r] = 0u;
  }
  const size_t hq = (size_t)blockIdx.y * a.Hq + blockIdx.x;
  const int S = a.n_splits;
  const float* ml = a.ws_ml + hq * S * 2;
  if (threadIdx.x < 32) {
    float ms = -INFINITY;
    for (int s = threadIdx.x; s < S; s += 32) ms = fmaxf(ms, ml[2 * s]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, off));
    float tot = 0.f;
    for (int s = threadIdx.x; s < S; s += 32) {
      const float m = ml[2 * s];
      const float ws = (ms == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - ms);
      w[s] = ws;
      tot += ws * ml[2 * s + 1];
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    if (threadIdx.x == 0) {
      s_inv = tot > 0.f ? 1.f / tot : 0.f;
      if (a.lse) a.lse[hq] = tot > 0.f ? kLn2 * (ms + log2f(tot)) : -INFINITY;
    }
  }
  __syncthreads();
  const int d = 4 * threadIdx.x;
  const float* po = a.ws_o + hq * (size_t)S * a.dv + d;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < S; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(po + (size_t)s * a.dv);
    o.x = fmaf(w[s], v.x, o.x);
    o.y = fmaf(w[s], v.y, o.y);
    o.z = fmaf(w[s], v.z, o.z);
    o.w = fmaf(w[s], v.w, o.w);
  }
  const float inv = s_inv;
  __nv_bfloat16* out = (__nv_bfloat16*)a.out + hq * a.dv + d;
  out[0] = __float2bfloat16_rn(o.x * inv);
  out[1] = __float2bfloat16_rn(o.y * inv);
  out[2] = __float2bfloat16_rn(o.z * inv);
  out[3] = __float2bfloat16_rn(o.w * inv);
}

// One split per 256-row block of the attended list.
int latent_splits(const skv_problem& p) {
  const int n = max_list(p);
  return n > 0 ? (n + t5::kRows - 1) / t5::kRows : 1;
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
  return p.d_qk == lat::kD && p.d_v == lat::kDV && p.n_kv_heads == 1 && p.n_q_heads == 128 &&
         p.dtype == SKV_DTYPE_BF16;
}

size_t latent_workspace_bytes(const skv_problem& p) { return latent_layout(p).total; }

skv_status launch_attn_latent(const skv_problem& p, const void* q, const PoolView& pool, const int32_t* idx,
                              void* out, float* lse, void* ws, int32_t* status, cudaStream_t st,
                              const PrefetchView* pf) {
  const LatentLayout lay = latent_layout(p);
  LatentArgs la;
  la.m = make_args(p, q, pool, idx, status);
  la.n_att = max_list(p);
  la.n_hgroups = 2;
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
  la.pf = pf ? *pf : PrefetchView{};
  if (la.n_att == 0) return SKV_ERR_UNSUPPORTED;
  const long long warps = (long long)p.batch * la.n_att;
  if (launch_dependent(latent_gather_kernel, dim3((unsigned)((warps * 32 + 255) / 256)), dim3(256), 0, st, 1, la) !=
      cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  static int configured = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SKV_ERR_CUDA;
  if (configured != dev) {
    if (cudaFuncSetAttribute(attn_latent_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, t5::kSmem) !=
        cudaSuccess)
      return SKV_ERR_CUDA;
    configured = dev;
  }
  dim3 grid(la.m.n_splits, 2, p.batch);
  attn_latent_tc_kernel<<<grid, t5::kThreads, t5::kSmem, st>>>(la);
  SKV_LAUNCH_CHECK();
  latent_merge_kernel<<<dim3(p.n_q_heads, p.batch), 128, 0, st>>>(la.m, la.pf);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace skv
