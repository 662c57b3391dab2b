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
//   attn_latent_tc_kernel  one CTA per (256-row block, request): Q, K and V slices
//                          arrive by TMA; S and O accumulate in TMEM (see the
//                          kernel's comment).
//   latent_merge_kernel    log-sum-exp merge of the blocks' partials.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched from the driver at run time)

#include <mutex>

#include "attn_common.cuh"

namespace skv {
namespace {

namespace lat {
constexpr int kD = 576;
constexpr int kDV = 512;
constexpr int kChunks = kD * 2 / 16;  // 72 16-byte chunks per row
constexpr int kRowB = kD * 2;         // 1152
}  // namespace lat

struct LatentArgs {
  AttnArgs m;                  // sizes, slot table, merge buffers, output
  const unsigned char* rows;   // [B, n_att, 576] bf16 gathered rows
  uint8_t* valid;              // [B, n_att]
  int n_att;
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
constexpr int kThreads = 256;            // two threads per head: warps w and w + 4 share TMEM lanes 32 (w % 4) ..
                                         // and split the block's columns
constexpr int kAtoms = 9;                // 576 dims = 9 slices of 64
constexpr int kQAtom = 128 * 128;        // 128 heads x 64 dims (bf16), 16 KB
constexpr int kKAtom = kRows * 128;      // 256 rows x 64 dims, 32 KB
constexpr int kStage = kQAtom + kKAtom;  // 48 KB: one (Q, K) slice pair
constexpr int kStages = 4;               // [0, 192 KB): the ring of slice pairs
constexpr int kVOff = 64 * 1024;         // V slices, 4 slots of 64 dims x 256 rows: [64 KB, 192 KB), over stages 1-3
constexpr int kVSlices = 8;              // 512 output dims = 8 slices of 64
constexpr int kPOff = 0;                 // P, 128 heads x 256 rows: [0, 64 KB), over stages 0-1
constexpr int kSmem = kStages * kStage + 1024;  // + alignment slack
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
// two 32-column loads of this warp's TMEM lanes and their wait, in one statement (the
// registers are written asynchronously until the wait)
__device__ __forceinline__ void ld32x2(uint32_t taddr0, uint32_t taddr1, uint32_t* r, uint32_t* q) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15]), "=r"(q[16]), "=r"(q[17]), "=r"(q[18]), "=r"(q[19]), "=r"(q[20]), "=r"(q[21]), "=r"(q[22]), "=r"(q[23]), "=r"(q[24]), "=r"(q[25]), "=r"(q[26]), "=r"(q[27]), "=r"(q[28]), "=r"(q[29]), "=r"(q[30]), "=r"(q[31])
      : "r"(taddr0), "r"(taddr1)
      : "memory");
}
// one 3-D tile of a tensor map into shared memory; completion as transaction bytes on bar
__device__ __forceinline__ void tma3(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
}  // namespace t5

// One CTA per (256-row block, request); 8 warps: head = 32 (w % 4) + lane, warp w % 4
// owning TMEM lanes 32 (w % 4) .. + 31, and w / 4 the half of the columns it reads.
//   S[128 x 256] (TMEM cols 0..255) = sum over 9 dim slices of Q_a K_a^T:
//       thread 0 streams (Q_a [128 heads x 64], K_a [256 rows x 64]) pairs by TMA
//       (3-D tensor maps, 128-byte swizzle: the K-major layout the MMA reads) into a
//       4-stage ring with full / empty mbarriers, and issues tcgen05.mma M128 N256
//       K16 x 4 per slice, committing each slice to its stage's empty barrier.
//   softmax per head from tcgen05.ld of its TMEM lane (each of the head's two threads
//       takes 128 columns; max and sum meet in shared memory): P = 2^(z - m) as bf16
//       in a swizzled K-major [128 x 256] tile.
//   O[128 x 512] = P V, one 64-dim slice of V at a time: the slices arrive by TMA in a
//       4-slot ring over [64 KB, 192 KB) (the first four as soon as the S slices that
//       used that memory are done), each feeding an M128 N64 MMA over the 256 rows;
//       dims 0..255 accumulate in TMEM cols 256..511, dims 256..511 in cols 0..255
//       (S is dead by then).
// The whole block's S is in TMEM at once, so the softmax is exact per block and O
// never needs rescaling; blocks are merged by log-sum-exp afterwards.  Partials are
// stored head-fastest ([b][block][dim / 4][head][4], and [b][block][m, l][head]), so
// every warp store and every merge load is coalesced.  Rows
// past the request's list are zero-filled by the TMA and masked.  Every wait is
// bounded; after one gives up, the CTA waits (bounded) for the copies and MMAs it
// issued, frees its TMEM and writes an empty partial.
__global__ void __launch_bounds__(t5::kThreads, 1)
    attn_latent_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tr,
                          const LatentArgs la) {
  using namespace t5;
  const AttnArgs& a = la.m;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], vfull[4], vempty[4], sdone, odone, drain;
  __shared__ uint32_t tmem_base;
  __shared__ uint8_t mask[kRows];
  __shared__ float xch[2][128];  // the two column halves' max, then their sums, per head
  __shared__ volatile int s_abort;

  const int s = blockIdx.x, b = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5;
  const int head = 32 * (warp & 3) + (t & 31), half = warp >> 2;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);  // generic pointer of the aligned base
  const int j0 = s * kRows;
  const int j1 = j0 + kRows < la.n_att ? j0 + kRows : la.n_att;

  if (t == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    mbar_init(&sdone, 1);
    mbar_init(&odone, 1);
    mbar_init(&drain, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  for (int r = t; r < kRows; r += t5::kThreads) {
    const int j = j0 + r;
    mask[r] = j < j1 ? la.valid[(size_t)b * la.n_att + j] : 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

  // thread 0's bookkeeping of what it issued (for the drain after a failed wait)
  int loads = 0, landed = 0;    // (Q, K) slice pairs issued / seen complete
  int vloads = 0, vlanded = 0;  // V slices issued / seen complete
  auto load_v = [&](int q) {    // V slice q into slot q % 4
    const int slot = q & 3;
    mbar_arrive_expect_tx(&vfull[slot], kKAtom);
    tma3(base + kVOff + slot * kKAtom, &tr, q * 64, j0, b, &vfull[slot]);
  };

  // ---- thread 0: TMA producer and MMA issuer for S = Q K^T
  if (t == 0) {
    auto load = [&](int at) {
      const int st = at % kStages;
      const uint32_t sq = base + st * kStage;
      mbar_arrive_expect_tx(&full[st], kStage);
      tma3(sq, &tq, at * 64, 0, b, &full[st]);
      tma3(sq + kQAtom, &tr, at * 64, j0, b, &full[st]);
    };
    for (int at = 0; at < kStages; ++at) load(at);
    loads = kStages;
    bool alive = true;
    const uint32_t idesc_s = idesc_bf16(128, 256, false);
    for (int at = 0; at < kAtoms && alive; ++at) {
      const int st = at % kStages;
      if (!mbar_wait_bounded(&full[st], (uint32_t)(at / kStages) & 1u)) {
        alive = false;
        break;
      }
      landed = at + 1;
      fence_after();
      const uint32_t sq = base + st * kStage, sk = sq + kQAtom;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma(tm, desc_sw128(sq + kk * 32, 16, 1024), desc_sw128(sk + kk * 32, 16, 1024), idesc_s,
            (at > 0 || kk > 0) ? 1u : 0u);
      commit(&empty[st]);
      if (at == kAtoms - 1) commit(&sdone);
      // the stage of slice at-1 takes slice at+3 once its MMAs are done
      const int nxt = at - 1 + kStages;
      if (at >= 1 && nxt < kAtoms) {
        if (!mbar_wait_bounded(&empty[(at - 1) % kStages], (uint32_t)((at - 1) / kStages) & 1u)) {
          alive = false;
          break;
        }
        load(nxt);
        loads = nxt + 1;
      }
    }
    // V slices 0-3 over stages 1-3: slice 7 is the last to use them (stage 3, second use)
    if (alive && mbar_wait_bounded(&empty[3], 1u)) {
      for (int q = 0; q < 4; ++q) load_v(q);
      vloads = 4;
    } else {
      alive = false;
    }
    if (!alive) {
      s_abort = 1;
      flag(a.status, SKV_DEV_TIMEOUT);
    }
  }

  // ---- softmax of each head over the block (two threads a head, 128 columns each)
  bool ok = wait_or_abort(&sdone, 0u, &s_abort, a.status);
  __syncthreads();
  ok = ok && !s_abort;  // the same in every thread
  fence_after();
  float m = -INFINITY, l = 0.f;
  if (ok) {
    uint32_t v[32], u[32];
    for (int ch = 4 * half; ch < 4 * half + 4; ch += 2) {
      ld32x2(tm + lane_base + ch * 32, tm + lane_base + (ch + 1) * 32, v, u);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (mask[ch * 32 + j]) m = fmaxf(m, __uint_as_float(v[j]) * a.scale_log2);
        if (mask[(ch + 1) * 32 + j]) m = fmaxf(m, __uint_as_float(u[j]) * a.scale_log2);
      }
    }
  }
  xch[half][head] = m;
  __syncthreads();
  m = fmaxf(xch[0][head], xch[1][head]);  // the block's max for this head
  if (ok) {
    uint32_t v[32];
    for (int ch = 4 * half; ch < 4 * half + 4; ++ch) {
      ld32(tm + lane_base + ch * 32, v);
      float pv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float z = __uint_as_float(v[j]) * a.scale_log2;
        pv[j] = (mask[ch * 32 + j] && m != -INFINITY) ? exp2f(z - m) : 0.f;
        l += pv[j];
      }
      // rows 32ch .. 32ch+31 = slice ch/2, chunks (ch%2)*4 .. +3 of head row
      unsigned char* prow = gbase + kPOff + (ch >> 1) * kQAtom;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 w;
        w.x = tc::pack_bf16(pv[8 * i + 0], pv[8 * i + 1]);
        w.y = tc::pack_bf16(pv[8 * i + 2], pv[8 * i + 3]);
        w.z = tc::pack_bf16(pv[8 * i + 4], pv[8 * i + 5]);
        w.w = tc::pack_bf16(pv[8 * i + 6], pv[8 * i + 7]);
        *reinterpret_cast<uint4*>(prow + sw128(head, (ch & 1) * 4 + i)) = w;
      }
    }
  }
  fence_proxy_async_smem();
  fence_before();
  __syncthreads();  // P complete; xch is free again
  xch[half][head] = l;
  ok = ok && !s_abort;

  // ---- O = P V, one 64-dim slice at a time
  if (t == 0 && ok) {
    bool alive = true;
    const uint32_t idesc_o = idesc_bf16(128, 64, true);
    for (int q = 0; q < kVSlices && alive; ++q) {
      const int slot = q & 3;
      if (!mbar_wait_bounded(&vfull[slot], (uint32_t)(q >> 2) & 1u)) {
        alive = false;
        break;
      }
      vlanded = q + 1;
      fence_after();
      const uint32_t dcol = q < 4 ? 256 + 64 * q : 64 * (q - 4);
#pragma unroll 4
      for (int kk = 0; kk < kRows / 16; ++kk) {
        const uint64_t ad = desc_sw128(base + kPOff + (kk >> 2) * kQAtom + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = desc_sw128(base + kVOff + slot * kKAtom + kk * 2048, kKAtom, 1024);
        mma(tm + dcol, ad, bd, idesc_o, kk > 0 ? 1u : 0u);
      }
      commit(&vempty[slot]);
      // the slot of slice q-1 takes slice q+3 once its MMAs are done
      const int nxt = q - 1 + 4;
      if (q >= 1 && nxt < kVSlices) {
        if (!mbar_wait_bounded(&vempty[(q - 1) & 3], (uint32_t)((q - 1) >> 2) & 1u)) {
          alive = false;
          break;
        }
        load_v(nxt);
        vloads = nxt + 1;
      }
    }
    if (alive) {
      commit(&odone);
    } else {
      s_abort = 1;
      flag(a.status, SKV_DEV_TIMEOUT);
    }
  }
  if (ok) ok = wait_or_abort(&odone, 0u, &s_abort, a.status);
  __syncthreads();
  ok = ok && !s_abort;
  fence_after();
  l = xch[0][head] + xch[1][head];  // the block's sum for this head

  // ---- partials, head-fastest in groups of 4 dims: [b][block][dim / 4][head][4], so a
  // warp's float4 stores cover 512 contiguous bytes
  const int S = a.n_splits;
  float4* po = reinterpret_cast<float4*>(a.ws_o) + ((size_t)b * S + s) * (lat::kDV / 4) * 128 + head;
  const int q0 = 64 * half;  // dims 0..255 sit in TMEM cols 256..511, dims 256..511 in cols 0..255
  if (ok) {
    uint32_t v[32], u[32];
    for (int ch = 0; ch < 8; ch += 2) {
      const uint32_t c0 = tm + lane_base + (half == 0 ? 256 : 0) + ch * 32;
      ld32x2(c0, c0 + 32, v, u);
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        po[(size_t)(q0 + ch * 8 + j / 4) * 128] = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                              __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
        po[(size_t)(q0 + (ch + 1) * 8 + j / 4) * 128] = make_float4(
            __uint_as_float(u[j]), __uint_as_float(u[j + 1]), __uint_as_float(u[j + 2]), __uint_as_float(u[j + 3]));
      }
    }
  } else {
    for (int qd = q0; qd < q0 + 64; ++qd) po[(size_t)qd * 128] = make_float4(0.f, 0.f, 0.f, 0.f);
    m = -INFINITY;
    l = 0.f;
  }
  if (half == 0) {  // head-fastest too: [b][block][m, l][head]
    float* ml = a.ws_ml + (((size_t)b * S + s) * 2) * 128 + head;
    ml[0] = m;
    ml[128] = l;
  }
  if (!ok && t == 0) {
    // a wait gave up: the copies and MMAs this CTA issued finish before its memory goes
    for (int at = landed; at < loads; ++at) mbar_wait_bounded(&full[at % kStages], (uint32_t)(at / kStages) & 1u);
    for (int q = vlanded; q < vloads; ++q) mbar_wait_bounded(&vfull[q & 3], (uint32_t)(q >> 2) & 1u);
    commit(&drain);
    mbar_wait_bounded(&drain, 0u);
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(kTmemCols) : "memory");
  }
}

// Log-sum-exp merge of the blocks, one CTA per (request, 8 output dims), thread = head:
// m* = max m_s, l = sum l_s 2^(m_s - m*), out = sum acc_s 2^(m_s - m*) / l,
// lse = ln 2 (m* + log2 l).  The partials are head-fastest, so every load is coalesced.
constexpr int kMergeDims = 8;  // output dims per merge CTA: 64 CTAs a request

__global__ void __launch_bounds__(128) latent_merge_kernel(const AttnArgs a, const PrefetchView pf) {
  constexpr int kDims = kMergeDims;
  const int b = blockIdx.x, dc = blockIdx.y, head = threadIdx.x;
  if (pf.map != nullptr && b == 0 && dc == 0 && head == 0) {
    // the step's end: later steps tag their staged rows anew and start with empty staging
    *pf.epoch += 1u;
    for (int r = 0; r < a.B * a.H; ++r) pf.count[r] = 0u;
  }
  const int S = a.n_splits;
  const size_t hq = (size_t)b * a.Hq + head;
  const float* ml = a.ws_ml + (size_t)b * S * 2 * 128 + head;  // m of block s at [2 s * 128], l at [(2 s + 1) * 128]
  float ms = -INFINITY;
  for (int s = 0; s < S; ++s) ms = fmaxf(ms, ml[(size_t)2 * s * 128]);
  float tot = 0.f;
  for (int s = 0; s < S; ++s) {
    const float m = ml[(size_t)2 * s * 128];
    tot += (ms == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - ms) * ml[(size_t)(2 * s + 1) * 128];
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  if (dc == 0 && a.lse) a.lse[hq] = tot > 0.f ? kLn2 * (ms + log2f(tot)) : -INFINITY;
  float o[kDims];
#pragma unroll
  for (int i = 0; i < kDims; ++i) o[i] = 0.f;
  for (int s = 0; s < S; ++s) {
    const float m = ml[(size_t)2 * s * 128];
    const float w = (ms == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - ms);
    const float4* po = reinterpret_cast<const float4*>(a.ws_o) + ((size_t)b * S + s) * (lat::kDV / 4) * 128 +
                       (size_t)dc * (kDims / 4) * 128 + head;
#pragma unroll
    for (int i = 0; i < kDims / 4; ++i) {
      const float4 x = po[(size_t)i * 128];
      o[4 * i + 0] = fmaf(w, x.x, o[4 * i + 0]);
      o[4 * i + 1] = fmaf(w, x.y, o[4 * i + 1]);
      o[4 * i + 2] = fmaf(w, x.z, o[4 * i + 2]);
      o[4 * i + 3] = fmaf(w, x.w, o[4 * i + 3]);
    }
  }
  uint4* out = reinterpret_cast<uint4*>((__nv_bfloat16*)a.out + hq * a.dv + dc * kDims);
#pragma unroll
  for (int i = 0; i < kDims / 8; ++i) {
    uint4 w;
    w.x = tc::pack_bf16(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
    w.y = tc::pack_bf16(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
    w.z = tc::pack_bf16(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
    w.w = tc::pack_bf16(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
    out[i] = w;
  }
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

// cuTensorMapEncodeTiled, fetched once from the driver through the runtime
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// A [d2][d1][d0] bf16 tensor (rows of d0 elements, packed) in boxes of 64 x box1 x 1,
// swizzled for the 128-byte K-major layout; loads past d1 read zeros.
bool encode_bf16_3d(CUtensorMap* map, const void* ptr, int d0, int d1, int d2, int box1) {
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr || d1 < 1 || d2 < 1) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  const cuuint64_t strides[2] = {(cuuint64_t)d0 * 2, (cuuint64_t)d0 * 2 * d1};
  const cuuint32_t box[3] = {64, (cuuint32_t)box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  const skv_status prep = prepare_kernel((const void*)attn_latent_tc_kernel, t5::kSmem);
  if (prep != SKV_OK) return prep;
  // tensor maps (3-D, bf16, 128-byte swizzle): q [B, 128, 576] in 128-head x 64-dim
  // boxes, the gathered rows [B, n_att, 576] in 256-row x 64-dim boxes
  CUtensorMap tq, tr;
  if (!encode_bf16_3d(&tq, q, lat::kD, p.n_q_heads, p.batch, 128) ||
      !encode_bf16_3d(&tr, la.rows, lat::kD, la.n_att, p.batch, t5::kRows))
    return SKV_ERR_CUDA;
  dim3 grid(la.m.n_splits, 1, p.batch);
  attn_latent_tc_kernel<<<grid, t5::kThreads, t5::kSmem, st>>>(tq, tr, la);
  SKV_LAUNCH_CHECK();
  latent_merge_kernel<<<dim3(p.batch, lat::kDV / kMergeDims), 128, 0, st>>>(la.m, la.pf);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace skv
