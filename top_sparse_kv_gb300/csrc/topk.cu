// S2: exact top-k of each (request, KV head) score row (sm_103a).
//
// The k-th largest score is a threshold: every score above it is in the top-k,
// and only ties at the threshold need a rule (ECHO-OSDI26 wiki, core method 3).
// The threshold is found exactly by a most-significant-digit radix select over
// order-preserving 32-bit keys -- histograms and prefix scans instead of a sort
// (ECHO-OSDI26 wiki, core method 4: a 256-bin histogram on the top bits;
// ParisKV notes §2.3: small-integer histogram + prefix scan, `bucket_topk`).
// Digits: bits [31:21], [20:10], [9:0]  (2048 / 2048 / 1024 bins).
//
// Rows of up to 32K candidates: `topk_solo_kernel`, one CTA per row (described
// above the kernel); more rows than SMs, of up to 8K candidates: `topk_lean_kernel`,
// three rows an SM.  Rows up to 128K: `topk_row_kernel`,
// one thread-block cluster per row (4 CTAs up to 64K candidates, 8 beyond),
// each CTA holding a contiguous slice of the row's keys in shared memory.  Each digit's histogram is built per CTA
// with shared atomics, its nonzero bins added into the row's histogram in
// global memory, and read back after a cluster barrier.  The digit-2 pass also
// counts, per warp, the keys certainly above the threshold (higher top 21 bits)
// and lists the few sharing the threshold's top 21 bits, which settle the
// counts once the threshold is known.  The ordered output is written warp by
// warp: scans of the counts give the bases (the lower-ranked CTAs' totals are
// read from their shared memory), and a ballot walk places every selected
// position.
//
// Longer rows: every row is cut into `cpr` segments, one CTA each.
//   pass p      histogram of digit p over keys matching the prefix; each CTA
//               folds its shared histogram into the row's global one, takes a
//               ticket, and the last CTA to arrive (it never waits for anyone)
//               fixes the next digit and the number k_rem of threshold-equal
//               keys still to take.
//   count       per segment: keys above the threshold and keys equal to it.
//   write       per segment: stable compaction in position order.
// Either way the output is the same on every run: ascending positions, a key
// equal to the threshold selected only while fewer than k_rem equal keys
// precede it in the row (ties to the lower position).
#include <cooperative_groups.h>

#include "skv_internal.cuh"

namespace cg = cooperative_groups;

namespace skv {
namespace {

constexpr int kThreads = 512;
constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kBins = 2048;
constexpr int kMinSeg = 2048;
constexpr int kSoloThreads = 1024;
constexpr int kRowMax4 = 64 * 1024;   // rows up to this length (and above the one-CTA limit): 4-CTA clusters
constexpr int kRowMax8 = 128 * 1024;  // up to this length: 8-CTA clusters (16K keys per CTA)

struct TopkArgs {
  const float* scores;
  int32_t* idx;
  const int32_t* seq_lens;
  int H, max_len, ns, nl, k, cpr, seg;
  int row_q;         // keys per CTA in the cluster path (a multiple of 32)
  uint32_t* hist;    // [rows][3][kBins]
  uint32_t* ticket;  // [rows][4]
  uint32_t* state;   // [rows][4]: prefix, k_rem
  uint32_t* counts;  // [rows][cpr][2]
  int32_t* status;
  uint32_t* zero;    // optional [rows]: set to zero by the one-CTA path
  int seg_len;       // two-stage path: candidates per segment
  int cand_stride;   // two-stage path: candidate slots per row (a multiple of 4)
  uint32_t* cand_key;  // [rows][cand_stride]: segment winners' keys ...
  int32_t* cand_pos;   // ... and positions, segment s at [s * k, s * k + min(k, segment length))
  const int32_t* row_geom;  // optional [rows][2]: (first candidate, candidate count) instead of the regions
  float* tau_ema;           // optional [rows]: EMA of the k-th score, updated by the final selection
  float ema_alpha;
  const int32_t* pos_map;   // optional [rows][max_len]: the position each score column stands for
                            // (one-CTA and two-stage paths), written instead of the column
};

struct RowGeom {
  int s_end, l_start, n, k_eff, lo, hi;
};

__device__ __forceinline__ RowGeom geom(const TopkArgs& a, int row, int x, int seg) {
  RowGeom g;
  if (a.row_geom != nullptr) {  // explicit candidate ranges (block selection), clamped to the row
    int lo = a.row_geom[2 * row], n = a.row_geom[2 * row + 1];
    lo = lo < 0 ? 0 : lo > a.max_len ? a.max_len : lo;
    n = n < 0 ? 0 : n > a.max_len - lo ? a.max_len - lo : n;
    g.s_end = lo;
    g.l_start = lo + n;
  } else {
    const int b = row / a.H;
    const int L = load_len(a.seq_lens, b, a.max_len, a.status);
    Regions r = regions_of(L, a.ns, a.nl);
    g.s_end = r.s_end;
    g.l_start = r.l_start;
  }
  g.n = g.l_start - g.s_end;
  g.k_eff = a.k < g.n ? a.k : g.n;
  long long lo = (long long)g.s_end + (long long)x * seg;
  long long hi = lo + seg;
  g.lo = (int)(lo < g.l_start ? lo : g.l_start);
  g.hi = (int)(hi < g.l_start ? hi : g.l_start);
  return g;
}

// Exclusive block-wide scan of one uint32 per thread; returns the prefix and
// the block total in *total.  NT threads (a multiple of 32, at most 1024).
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total) {
  constexpr int NW = NT / 32;
  __shared__ uint32_t warp_sums[NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < NW ? warp_sums[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < NW) warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const uint32_t before_warp = warp > 0 ? warp_sums[warp - 1] : 0u;
  *total = warp_sums[NW - 1];
  const uint32_t excl = before_warp + x - v;
  __syncthreads();  // warp_sums reusable after return
  return excl;
}

// Given the histogram sh[0..nb) of the keys tied with the prefix so far, find the
// digit whose bin holds the krem-th largest key.  Writes (digit, krem - count of
// keys in higher bins) to out[0..1] (shared memory) from the one thread that sees it.
template <int NT, int NBMAX = kBins>
__device__ __forceinline__ void select_digit(const uint32_t* sh, int nb, uint32_t krem, uint32_t* out) {
  constexpr int PER = (NBMAX + NT - 1) / NT;  // bins per thread (descending order)
  uint32_t mine = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int r = PER * threadIdx.x + e;
    if (r < nb) mine += sh[nb - 1 - r];
  }
  uint32_t total;
  uint32_t before = block_exclusive_scan<NT>(mine, &total);
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int r = PER * threadIdx.x + e;
    if (r < nb) {
      const uint32_t bin = (uint32_t)(nb - 1 - r);
      const uint32_t c = sh[bin];
      if (before < krem && before + c >= krem) {
        out[0] = bin;
        out[1] = krem - before;
      }
      before += c;
    }
  }
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ---------------------------------------------------------------------------- one cluster per row

constexpr int kAmbMax = 1024;  // keys still ambiguous after digit 1, per CTA

// Fold this CTA's histogram into the row's global one (nonzero bins only).
template <int NT>
__device__ __forceinline__ void push_hist(const uint32_t* local, uint32_t* global, int nb) {
  for (int i = threadIdx.x; i < nb; i += NT) {
    const uint32_t v = local[i];
    if (v) atomicAdd(global + i, v);
  }
}

template <int kCluster, int NT>
__global__ void __launch_bounds__(NT) topk_row_kernel(const TopkArgs a) {
  constexpr int kWarps = NT / 32;
  pdl_release();
  pdl_wait();
  extern __shared__ uint32_t keys[];  // [q]
  __shared__ uint32_t sh[kBins];      // this CTA's histogram, then the row's
  __shared__ uint32_t sel[2];
  __shared__ uint32_t wcount[kWarps][2];
  __shared__ uint32_t cta_count[2];
  __shared__ uint32_t amb_pos[kAmbMax];
  __shared__ uint32_t amb_key[kAmbMax];
  __shared__ uint32_t n_amb;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.x / kCluster;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RowGeom g = geom(a, row, 0, a.max_len);
  int32_t* out = a.idx + (size_t)row * a.k;
  if (rank == 0)
    for (int j = g.k_eff + threadIdx.x; j < a.k; j += NT) out[j] = -1;
  if (g.k_eff == 0) return;  // the same decision in every CTA of the cluster
  uint32_t* gh0 = a.hist + (size_t)row * 3 * kBins;  // the row's histograms (zeroed before the launch)
  uint32_t* gh1 = gh0 + kBins;
  uint32_t* gh2 = gh1 + kBins;
  // this CTA's slice of the candidates: positions s_end + [c0, c1)
  const int q = ((g.n + kCluster - 1) / kCluster + 31) & ~31;
  const int c0 = rank * q < g.n ? rank * q : g.n;
  const int c1 = c0 + q < g.n ? c0 + q : g.n;
  const int n = c1 - c0;
  // warp w owns local keys [w*seg, (w+1)*seg) for the ordered output
  const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int w0 = warp * seg < n ? warp * seg : n;
  const int w1 = w0 + seg < n ? w0 + seg : n;

  for (int i = threadIdx.x; i < kBins; i += NT) sh[i] = 0u;
  if (threadIdx.x == 0) n_amb = 0;
  __syncthreads();
  // scores -> keys (16-byte loads for the aligned body) and the local digit-0 histogram
  const size_t e0 = (size_t)row * a.max_len + g.s_end + c0;  // element index of keys[0]
  const int lead = (int)((4 - (e0 & 3)) & 3);
  const int head = lead < n ? lead : n;
  const int nv4 = (n - head) >> 2;
  const float* src = a.scores + e0;
  for (int i = threadIdx.x; i < head; i += NT) {
    const uint32_t key = order_key(__ldcg(src + i));
    keys[i] = key;
    atomicAdd(&sh[key >> 21], 1u);
  }
  const float4* src4 = reinterpret_cast<const float4*>(src + head);
#pragma unroll 4
  for (int v = threadIdx.x; v < nv4; v += NT) {
    const float4 f = __ldcg(src4 + v);
    const int i = head + 4 * v;
    const uint32_t k0 = order_key(f.x), k1 = order_key(f.y), k2 = order_key(f.z), k3 = order_key(f.w);
    keys[i] = k0;
    keys[i + 1] = k1;
    keys[i + 2] = k2;
    keys[i + 3] = k3;
    atomicAdd(&sh[k0 >> 21], 1u);
    atomicAdd(&sh[k1 >> 21], 1u);
    atomicAdd(&sh[k2 >> 21], 1u);
    atomicAdd(&sh[k3 >> 21], 1u);
  }
  for (int i = head + 4 * nv4 + threadIdx.x; i < n; i += NT) {
    const uint32_t key = order_key(__ldcg(src + i));
    keys[i] = key;
    atomicAdd(&sh[key >> 21], 1u);
  }
  __syncthreads();
  push_hist<NT>(sh, gh0, kBins);
  __threadfence();
  cluster.sync();
  for (int i = threadIdx.x; i < kBins; i += NT) sh[i] = __ldcg(gh0 + i);
  __syncthreads();
  select_digit<NT>(sh, kBins, (uint32_t)g.k_eff, sel);
  __syncthreads();
  uint32_t prefix = sel[0] << 21;
  uint32_t krem = sel[1];
  // digit 1 over the keys tied with the threshold's digit 0
  for (int i = threadIdx.x; i < kBins; i += NT) sh[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t key = keys[i];
    if ((key & 0xFFE00000u) == prefix) atomicAdd(&sh[(key >> 10) & 0x7FFu], 1u);
  }
  __syncthreads();
  push_hist<NT>(sh, gh1, kBins);
  __threadfence();
  cluster.sync();
  for (int i = threadIdx.x; i < kBins; i += NT) sh[i] = __ldcg(gh1 + i);
  __syncthreads();
  select_digit<NT>(sh, kBins, krem, sel);
  __syncthreads();
  prefix |= sel[0] << 10;  // top 21 bits of the threshold
  krem = sel[1];
  // digit 2; at the same time each warp counts its keys certainly above the
  // threshold and lists the few keys that share its top 21 bits
  for (int i = threadIdx.x; i < 1024; i += NT) sh[i] = 0u;
  __syncthreads();
  const uint32_t p21 = prefix >> 10;
  uint32_t cgt = 0;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < w1 ? keys[i] : 0u;
    const bool in = i < w1;
    cgt += __popc(__ballot_sync(0xffffffffu, in && (key >> 10) > p21));
    if (in && (key >> 10) == p21) {
      atomicAdd(&sh[key & 0x3FFu], 1u);
      const uint32_t slot = atomicAdd(&n_amb, 1u);
      if (slot < (uint32_t)kAmbMax) {
        amb_pos[slot] = (uint32_t)i;
        amb_key[slot] = key;
      }
    }
  }
  if (lane == 0) wcount[warp][0] = cgt;
  if (lane == 0) wcount[warp][1] = 0;
  __syncthreads();
  push_hist<NT>(sh, gh2, 1024);
  __threadfence();
  cluster.sync();
  for (int i = threadIdx.x; i < 1024; i += NT) sh[i] = __ldcg(gh2 + i);
  __syncthreads();
  select_digit<NT>(sh, 1024, krem, sel);
  __syncthreads();
  const uint32_t tau = prefix | sel[0];
  const uint32_t ktie = sel[1];
  // finish the per-warp counts with the ambiguous keys (or recount if the list overflowed)
  const uint32_t na = n_amb;
  if (na <= (uint32_t)kAmbMax) {
    for (uint32_t t = threadIdx.x; t < na; t += NT) {
      const uint32_t key = amb_key[t];
      const int w = (int)(amb_pos[t] / (uint32_t)seg);
      if (key > tau) atomicAdd(&wcount[w][0], 1u);
      else if (key == tau) atomicAdd(&wcount[w][1], 1u);
    }
  } else {
    uint32_t xg = 0, xe = 0;
    for (int i0 = w0; i0 < w1; i0 += 32) {
      const int i = i0 + lane;
      const uint32_t key = i < w1 ? keys[i] : 0u;
      xg += __popc(__ballot_sync(0xffffffffu, i < w1 && key > tau));
      xe += __popc(__ballot_sync(0xffffffffu, i < w1 && key == tau));
    }
    __syncthreads();
    if (lane == 0) {
      wcount[warp][0] = xg;
      wcount[warp][1] = xe;
    }
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the per-warp counts; CTA totals for the cluster
    uint32_t xg = lane < kWarps ? wcount[lane][0] : 0u, xt = lane < kWarps ? wcount[lane][1] : 0u;
    const uint32_t vg = xg, vt = xt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t yg = __shfl_up_sync(0xffffffffu, xg, off);
      const uint32_t yt = __shfl_up_sync(0xffffffffu, xt, off);
      if (lane >= off) {
        xg += yg;
        xt += yt;
      }
    }
    if (lane < kWarps) {
      wcount[lane][0] = xg - vg;
      wcount[lane][1] = xt - vt;
    }
    if (lane == kWarps - 1) {
      cta_count[0] = xg;
      cta_count[1] = xt;
    }
  }
  cluster.sync();
  uint32_t bg = 0, bt = 0;  // keys of the lower-ranked CTAs
  for (int r = 0; r < rank; ++r) {
    const uint32_t* rc = cluster.map_shared_rank(cta_count, r);
    bg += rc[0];
    bt += rc[1];
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
  bg += wcount[warp][0];
  bt += wcount[warp][1];
  const uint32_t lt = lanemask_lt();
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < w1 ? keys[i] : 0u;
    const bool gt = i < w1 && key > tau;
    const bool eq = i < w1 && key == tau;
    const uint32_t mg = __ballot_sync(0xffffffffu, gt);
    const uint32_t me = __ballot_sync(0xffffffffu, eq);
    const uint32_t gb = bg + __popc(mg & lt);
    const uint32_t tb = bt + __popc(me & lt);
    if (gt) {
      const uint32_t pos = gb + (tb < ktie ? tb : ktie);
      if (pos < (uint32_t)g.k_eff) out[pos] = g.s_end + c0 + i;  // always true when the passes are consistent
    } else if (eq && tb < ktie && gb + tb < (uint32_t)g.k_eff) {
      out[gb + tb] = g.s_end + c0 + i;
    }
    bg += __popc(mg);
    bt += __popc(me);
  }
}

// ---------------------------------------------------------------------------- one CTA per row
//
// Rows of up to 32K candidates: one 1024-thread CTA holds the row's keys in
// shared memory, and every step after the load stays on chip.  Thread t owns the
// P = ceil(n / 1024) <= 32 consecutive candidates [tP, tP + P) for counting and
// for the ordered output; the key array is padded by one word per 32 so these
// per-thread walks are free of bank conflicts.
//   load     coalesced 16-byte loads, all in flight at once; scores -> keys and
//            the histogram of a 13-bit digit 0 (sign, exponent, 4 mantissa bits:
//            scores spread over many bins, so the shared atomics rarely collide)
//   digit 0  the bucket holding the threshold: every warp searches its own 256
//            bins at once (no serial walk)
//   walk     one pass: each thread marks, in two 32-bit masks, its keys in higher
//            buckets (all selected) and its keys in the threshold's bucket
//   digits 1 (11 bits) and 2 (8 bits) over the marked bucket keys only give the
//            threshold key tau and the number of tau-equal keys to take
//   write    one block scan of the packed (above, equal) counts; each thread
//            visits only its marked keys, in position order.
constexpr int kSoloMax = 32 * 1024;  // candidates per row: P <= 32
constexpr int kSoloBins0 = 8192;     // bucket: key bits [31:19]

__host__ __device__ __forceinline__ int solo_pad(int j) { return j + (j >> 5); }
__host__ __forceinline__ size_t solo_smem_bytes(int max_len) {
  return ((size_t)kSoloBins0 + solo_pad(max_len) + 1) * 4;
}

// For each of R ranks kr[0..R) (1-based, counted from the largest key), the bin
// of h[0..NB) that holds the kr-th largest key; NT threads (NW = NT / 32 warps) and
// NB = NW * G with G a multiple of 32.  Every warp loads its own group of G bins
// (descending, coalesced), reduces it in 32-bin chunks and learns the exclusive
// prefix of its group from a scan of the NW group totals; the warp whose group holds
// a rank finds the chunk from its chunk totals and the bin with one warp scan.  Writes
// (bin, kr - keys in higher bins) to out[2r], out[2r+1]; the caller synchronises
// before reading out and before the next call.  LEAN: the bins and chunk totals are not
// kept in registers; the warp that holds a rank reads its chunks again.
template <int NB, int R, int NT = 1024, bool LEAN = false>
__device__ __forceinline__ void select_bins(const uint32_t* h, const uint32_t (&kr)[R], uint32_t* out) {
  constexpr int NW = NT / 32, G = NB / NW, E = G / 32;
  constexpr int EK = LEAN ? 1 : E;  // chunks kept in registers
  static_assert(G % 32 == 0 && NW * G == NB, "whole 32-bin chunks per warp");
  __shared__ uint32_t gsum[NW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int top = NB - 1 - warp * G;
  uint32_t v[EK], ct[EK];
  uint32_t gt = 0;
  if constexpr (LEAN) {
#pragma unroll 4
    for (int e = 0; e < E; ++e) gt += __reduce_add_sync(0xffffffffu, h[top - (e * 32 + lane)]);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = h[top - (e * 32 + lane)];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      ct[e] = __reduce_add_sync(0xffffffffu, v[e]);
      gt += ct[e];
    }
  }
  if (lane == 0) gsum[warp] = gt;
  __syncthreads();
  const uint32_t gl = lane < NW ? gsum[lane] : 0u;
  uint32_t x = gl;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  const uint32_t gexcl = __shfl_sync(0xffffffffu, x - gl, warp);  // keys in the groups above this one
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!(gexcl < kr[r] && kr[r] <= gexcl + gt)) continue;  // warp-uniform
    uint32_t base = gexcl, c = 0;
    int ec = -1;
    if constexpr (LEAN) {
      for (int e = 0; e < E && ec < 0; ++e) {  // warp-uniform exit
        const uint32_t ve = h[top - (e * 32 + lane)];
        const uint32_t te = __reduce_add_sync(0xffffffffu, ve);
        if (base + te >= kr[r]) {
          ec = e;
          c = ve;
        } else {
          base += te;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (ec < 0) {
          if (base + ct[e] >= kr[r]) {
            ec = e;
            c = v[e];
          } else {
            base += ct[e];
          }
        }
      }
    }
    uint32_t xi = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, xi, off);
      if (lane >= off) xi += y;
    }
    const uint32_t excl = base + xi - c;
    if (excl < kr[r] && kr[r] <= excl + c) {
      out[2 * r] = (uint32_t)(top - (ec * 32 + lane));
      out[2 * r + 1] = kr[r] - excl;
    }
  }
}

// The source and destination of one selection (MODE 0: a whole score row -> the
// positions; MODE 1: one segment of a score row -> (key, position) candidates;
// MODE 2: a row's candidates -> the positions).
template <int MODE>
__global__ void __launch_bounds__(kSoloThreads, 1) topk_solo_kernel(const TopkArgs a) {
  constexpr int NT = kSoloThreads;
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* hist = sm;                 // [kSoloBins0]
  uint32_t* keys = hist + kSoloBins0;  // [solo_pad(n) + 1]
  __shared__ uint32_t sel[2];
  const int tid = threadIdx.x;
  const int row = blockIdx.x;
  pdl_release();
  pdl_wait();
  if (MODE != 1 && a.zero != nullptr && tid == 0) a.zero[row] = 0u;
  const RowGeom g = geom(a, row, 0, a.max_len);
  // this selection's n candidates: keys from `src` (scores, or keys for MODE 2)
  int n, lo = 0;
  size_t e0 = 0;  // element offset of a score row's first candidate (its 16-byte alignment)
  const float* src;
  if (MODE == 0) {
    n = g.n;
    e0 = (size_t)row * a.max_len + g.s_end;
    src = a.scores + e0;
  } else if (MODE == 1) {
    lo = blockIdx.y * a.seg_len;
    if (lo >= g.n) return;
    n = g.n - lo < a.seg_len ? g.n - lo : a.seg_len;
    e0 = (size_t)row * a.max_len + g.s_end + lo;
    src = a.scores + e0;
  } else {
    const int segs = (g.n + a.seg_len - 1) / a.seg_len;
    const int last = g.n - (segs - 1) * a.seg_len;
    n = segs == 0 ? 0 : (segs - 1) * a.k + (last < a.k ? last : a.k);
    src = reinterpret_cast<const float*>(a.cand_key + (size_t)row * a.cand_stride);
  }
  const uint32_t keff = (uint32_t)(a.k < n ? a.k : n);
  int32_t* out = a.idx + (size_t)row * a.k;
  uint32_t* ck = a.cand_key + (size_t)row * a.cand_stride + (size_t)blockIdx.y * a.k;
  int32_t* cp = a.cand_pos + (size_t)row * a.cand_stride + (size_t)blockIdx.y * a.k;
  const int32_t* in_pos = a.cand_pos + (size_t)row * a.cand_stride;
  auto key_of = [&](float x) { return MODE == 2 ? __float_as_uint(x) : order_key(x); };
  // writes selected candidate j (key `key`) at output slot `pos`
  auto emit = [&](uint32_t pos, int j, uint32_t key) {
    if (MODE == 0) out[pos] = a.pos_map ? a.pos_map[(size_t)row * a.max_len + g.s_end + j] : g.s_end + j;
    if (MODE == 1) {
      ck[pos] = key;
      cp[pos] = a.pos_map ? a.pos_map[(size_t)row * a.max_len + g.s_end + lo + j] : g.s_end + lo + j;
    }
    if (MODE == 2) out[pos] = in_pos[j];
  };
  if (MODE != 1)
    for (int j = (int)keff + tid; j < a.k; j += NT) out[j] = -1;
  if (keff == 0) return;
  if (keff == (uint32_t)n) {  // every candidate is selected
    for (int j = tid; j < n; j += NT) emit((uint32_t)j, j, MODE == 1 ? key_of(__ldcg(src + j)) : 0u);
    return;
  }
  for (int i = tid; i < kSoloBins0; i += NT) hist[i] = 0u;
  __syncthreads();
  {  // keys and the digit-0 histogram; the aligned body's loads all issued before any use
    const int lead = (int)((4 - (e0 & 3)) & 3);  // candidate rows (e0 = 0) start 16-byte aligned
    const int head = lead < n ? lead : n;
    const int nv4 = (n - head) >> 2;  // <= kSoloMax / 4: at most 8 per thread
    const float4* src4 = reinterpret_cast<const float4*>(src + head);
    float4 f[kSoloMax / 4 / NT];
#pragma unroll
    for (int u = 0; u < kSoloMax / 4 / NT; ++u) {
      const int v = tid + NT * u;
      if (v < nv4) f[u] = __ldcg(src4 + v);
    }
    auto put = [&](int i, float x) {
      const uint32_t key = key_of(x);
      keys[solo_pad(i)] = key;
      atomicAdd(&hist[key >> 19], 1u);
    };
    for (int i = tid; i < head; i += NT) put(i, __ldcg(src + i));
    for (int i = head + 4 * nv4 + tid; i < n; i += NT) put(i, __ldcg(src + i));
#pragma unroll
    for (int u = 0; u < kSoloMax / 4 / NT; ++u) {
      const int v = tid + NT * u;
      if (v < nv4) {
        const int i = head + 4 * v;
        put(i, f[u].x);
        put(i + 1, f[u].y);
        put(i + 2, f[u].z);
        put(i + 3, f[u].w);
      }
    }
  }
  __syncthreads();
  {
    const uint32_t rk[1] = {keff};
    select_bins<kSoloBins0, 1>(hist, rk, sel);
  }
  __syncthreads();
  const uint32_t d0 = sel[0];
  uint32_t krem = sel[1];
  // walk this thread's P <= 32 consecutive candidates: bit i of `above` marks a key
  // in a higher bucket (selected), bit i of `inb` a key in the threshold's bucket
  const int P = (n + NT - 1) / NT;
  const int j0 = tid * P < n ? tid * P : n;
  const int cnt = (j0 + P < n ? j0 + P : n) - j0;
  const uint32_t lo_key = d0 << 19, span = (1u << 19) - 1u;
  uint32_t above = 0, inb = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (i < cnt) {
      const uint32_t key = keys[solo_pad(j0 + i)];
      above |= (key > lo_key + span ? 1u : 0u) << i;
      inb |= (key - lo_key <= span ? 1u : 0u) << i;
    }
  }
  for (int i = tid; i < kBins; i += NT) hist[i] = 0u;
  __syncthreads();
  // digit 1 (bits [18:8]) and digit 2 (bits [7:0]) over the keys of the threshold's bucket
  for (uint32_t mk = inb; mk; mk &= mk - 1)
    atomicAdd(&hist[(keys[solo_pad(j0 + __ffs(mk) - 1)] >> 8) & 0x7FFu], 1u);
  __syncthreads();
  {
    const uint32_t rk[1] = {krem};
    select_bins<kBins, 1>(hist, rk, sel);
  }
  __syncthreads();
  const uint32_t p24 = (d0 << 11) | sel[0];  // the threshold's key >> 8
  krem = sel[1];
  // When every key whose top 24 bits are p24 is selected (the common case: the bucket's
  // keys spread over 2048 second-digit bins), the last digit is not needed: a threshold
  // just below that bin, with no ties to take, selects the same keys.  Not where the k-th
  // key itself is wanted (the EMA), nor for p24 = 0, whose bin starts at key 0.
  const bool whole_bin = hist[sel[0]] == krem && p24 != 0u && (MODE == 1 || a.tau_ema == nullptr);
  __syncthreads();
  uint32_t tau, ktie;
  if (whole_bin) {
    tau = (p24 << 8) - 1u;
    ktie = 0u;
  } else {
    for (int i = tid; i < 256; i += NT) hist[i] = 0u;
    __syncthreads();
    for (uint32_t mk = inb; mk; mk &= mk - 1) {
      const uint32_t key = keys[solo_pad(j0 + __ffs(mk) - 1)];
      if ((key >> 8) == p24) atomicAdd(&hist[key & 0xFFu], 1u);
    }
    __syncthreads();
    select_digit<NT, 256>(hist, 256, krem, sel);
    __syncthreads();
    tau = (p24 << 8) | sel[0];
    ktie = sel[1];
  }
  if (MODE != 1 && a.tau_ema != nullptr && tid == 0) {  // the row's k-th score into its EMA
    const float kth = __uint_as_float((tau & 0x80000000u) ? (tau & 0x7FFFFFFFu) : ~tau);
    const float old = a.tau_ema[row];
    a.tau_ema[row] = old != old ? kth : a.ema_alpha * kth + (1.f - a.ema_alpha) * old;
  }
  // this thread's keys above tau and equal to tau
  uint32_t gt = (uint32_t)__popc(above), eq = 0;
  for (uint32_t mk = inb; mk; mk &= mk - 1) {
    const uint32_t key = keys[solo_pad(j0 + __ffs(mk) - 1)];
    gt += key > tau ? 1u : 0u;
    eq += key == tau ? 1u : 0u;
  }
  // packed scan: both totals stay below 2^16 (n <= 32K)
  uint32_t total;
  const uint32_t pre = block_exclusive_scan<NT>(gt | (eq << 16), &total);
  uint32_t gb = pre & 0xFFFFu, tb = pre >> 16;
  // ordered write: only the marked keys can be selected
  for (uint32_t mk = above | inb; mk; mk &= mk - 1) {
    const int i = __ffs(mk) - 1;
    const int j = j0 + i;
    const bool hi = (above >> i) & 1u;
    const uint32_t key = hi && MODE != 1 ? 0xFFFFFFFFu : keys[solo_pad(j)];
    if (hi || key > tau) {
      const uint32_t pos = gb + (tb < ktie ? tb : ktie);
      if (pos < keff) emit(pos, j, key);  // always true when the counts are consistent
      ++gb;
    } else if (key == tau) {
      if (tb < ktie && gb + tb < keff) emit(gb + tb, j, key);
      ++tb;
    }
  }
}

// ---------------------------------------------------------------------------- many rows
//
// More rows than SMs, of up to 8K candidates: the one-CTA kernel takes a whole SM a row
// (1,024 threads x 62 registers), so 512 short rows run in 3.4 waves of mostly fixed
// block-wide phases.  `topk_lean_kernel` keeps only the digit-0 histogram (32 KB) in
// shared memory, so three 512-thread CTAs share an SM, and reads the row's scores
// (just written, in L2) again where the one-CTA kernel reads its shared copy:
//   count    coalesced 16-byte loads; the 13-bit digit-0 histogram (shared atomics)
//   digit 0  the threshold's bucket
//   walk     thread t reads its P <= 64 consecutive candidates and marks, in two
//            64-bit masks, its keys above the bucket and its keys inside it
//   digits 1 (11 bits) and 2 (8 bits) over the bucket's keys, read once more; then the
//            packed count scan and the ordered write of the one-CTA kernel.
// Same threshold, tie rule and order as the one-CTA kernel, so the same output.
constexpr int kLeanThreads = 512;
constexpr int kLeanMax = 8 * 1024;  // candidates per row it is used for (it handles up to 32K)

__global__ void __launch_bounds__(kLeanThreads, 3) topk_lean_kernel(const TopkArgs a) {
  constexpr int NT = kLeanThreads;
  __shared__ __align__(16) uint32_t hist[kSoloBins0];
  __shared__ uint32_t sel[2];
  const int tid = threadIdx.x;
  const int row = blockIdx.x;
  pdl_release();
  pdl_wait();
  if (a.zero != nullptr && tid == 0) a.zero[row] = 0u;
  const RowGeom g = geom(a, row, 0, a.max_len);
  const int n = g.n;
  const size_t e0 = (size_t)row * a.max_len + g.s_end;
  const float* src = a.scores + e0;
  const uint32_t keff = (uint32_t)(a.k < n ? a.k : n);
  int32_t* out = a.idx + (size_t)row * a.k;
  auto emit = [&](uint32_t pos, int j) {
    out[pos] = a.pos_map ? a.pos_map[(size_t)row * a.max_len + g.s_end + j] : g.s_end + j;
  };
  for (int j = (int)keff + tid; j < a.k; j += NT) out[j] = -1;
  if (keff == 0) return;
  if (keff == (uint32_t)n) {  // every candidate is selected
    for (int j = tid; j < n; j += NT) emit((uint32_t)j, j);
    return;
  }
  for (int i = tid; i < kSoloBins0; i += NT) hist[i] = 0u;
  __syncthreads();
  {  // the digit-0 histogram: the aligned body in batches of loads issued before any use
    const int lead = (int)((4 - (e0 & 3)) & 3);
    const int head = lead < n ? lead : n;
    const int nv4 = (n - head) >> 2;
    const float4* src4 = reinterpret_cast<const float4*>(src + head);
    for (int i = tid; i < head; i += NT) atomicAdd(&hist[order_key(__ldcg(src + i)) >> 19], 1u);
    for (int i = head + 4 * nv4 + tid; i < n; i += NT) atomicAdd(&hist[order_key(__ldcg(src + i)) >> 19], 1u);
    constexpr int kBatch = 2;
    for (int v0 = 0; v0 < nv4; v0 += kBatch * NT) {
      float4 f[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int v = v0 + tid + NT * u;
        if (v < nv4) f[u] = __ldcg(src4 + v);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int v = v0 + tid + NT * u;
        if (v < nv4) {
          atomicAdd(&hist[order_key(f[u].x) >> 19], 1u);
          atomicAdd(&hist[order_key(f[u].y) >> 19], 1u);
          atomicAdd(&hist[order_key(f[u].z) >> 19], 1u);
          atomicAdd(&hist[order_key(f[u].w) >> 19], 1u);
        }
      }
    }
  }
  __syncthreads();
  {
    const uint32_t rk[1] = {keff};
    select_bins<kSoloBins0, 1, NT, true>(hist, rk, sel);
  }
  __syncthreads();
  const uint32_t d0 = sel[0];
  uint32_t krem = sel[1];
  // walk this thread's P <= 64 consecutive candidates [j0, j0 + cnt)
  const int P = (n + NT - 1) / NT;
  const int j0 = tid * P < n ? tid * P : n;
  const int cnt = (j0 + P < n ? j0 + P : n) - j0;
  const float* mine = src + j0;
  auto key_at = [&](int i) { return order_key(__ldcg(mine + i)); };
  const uint32_t lo_key = d0 << 19, span = (1u << 19) - 1u;
  uint64_t above = 0, inb = 0;
  {
    auto mark = [&](int i, float x) {
      const uint32_t key = order_key(x);
      above |= (uint64_t)(key > lo_key + span ? 1u : 0u) << i;
      inb |= (uint64_t)(key - lo_key <= span ? 1u : 0u) << i;
    };
    int lt = (int)((4 - ((e0 + (size_t)j0) & 3)) & 3);  // scalar keys up to a 16-byte boundary
    lt = lt < cnt ? lt : cnt;
    for (int i = 0; i < lt; ++i) mark(i, __ldcg(mine + i));
    const float4* m4 = reinterpret_cast<const float4*>(mine + lt);
    const int nb4 = (cnt - lt) >> 2;
    constexpr int kWalkBatch = 2;
    for (int v = 0; v < nb4; v += kWalkBatch) {
      float4 f[kWalkBatch];
#pragma unroll
      for (int u = 0; u < kWalkBatch; ++u)
        if (v + u < nb4) f[u] = __ldcg(m4 + v + u);
#pragma unroll
      for (int u = 0; u < kWalkBatch; ++u)
        if (v + u < nb4) {
          const int i = lt + 4 * (v + u);
          mark(i, f[u].x);
          mark(i + 1, f[u].y);
          mark(i + 2, f[u].z);
          mark(i + 3, f[u].w);
        }
    }
    for (int i = lt + 4 * nb4; i < cnt; ++i) mark(i, __ldcg(mine + i));
  }
  for (int i = tid; i < kBins; i += NT) hist[i] = 0u;
  __syncthreads();
  // digit 1 (bits [18:8]) and digit 2 (bits [7:0]) over the keys of the threshold's bucket
  for (uint64_t mk = inb; mk; mk &= mk - 1)
    atomicAdd(&hist[(key_at(__ffsll((long long)mk) - 1) >> 8) & 0x7FFu], 1u);
  __syncthreads();
  {
    const uint32_t rk[1] = {krem};
    select_bins<kBins, 1, NT, true>(hist, rk, sel);
  }
  __syncthreads();
  const uint32_t p24 = (d0 << 11) | sel[0];  // the threshold's key >> 8
  krem = sel[1];
  // as in the one-CTA kernel: when every key of the p24 bin is selected, the last digit
  // is not needed (except where the k-th key itself feeds the EMA, or for p24 = 0)
  const bool whole_bin = hist[sel[0]] == krem && p24 != 0u && a.tau_ema == nullptr;
  __syncthreads();
  uint32_t tau, ktie;
  if (whole_bin) {
    tau = (p24 << 8) - 1u;
    ktie = 0u;
  } else {
    for (int i = tid; i < 256; i += NT) hist[i] = 0u;
    __syncthreads();
    for (uint64_t mk = inb; mk; mk &= mk - 1) {
      const uint32_t key = key_at(__ffsll((long long)mk) - 1);
      if ((key >> 8) == p24) atomicAdd(&hist[key & 0xFFu], 1u);
    }
    __syncthreads();
    select_digit<NT, 256>(hist, 256, krem, sel);
    __syncthreads();
    tau = (p24 << 8) | sel[0];
    ktie = sel[1];
  }
  if (a.tau_ema != nullptr && tid == 0) {  // the row's k-th score into its EMA
    const float kth = __uint_as_float((tau & 0x80000000u) ? (tau & 0x7FFFFFFFu) : ~tau);
    const float old = a.tau_ema[row];
    a.tau_ema[row] = old != old ? kth : a.ema_alpha * kth + (1.f - a.ema_alpha) * old;
  }
  // this thread's keys above tau and equal to tau
  uint32_t gt = (uint32_t)__popcll(above), eq = 0;
  for (uint64_t mk = inb; mk; mk &= mk - 1) {
    const uint32_t key = key_at(__ffsll((long long)mk) - 1);
    gt += key > tau ? 1u : 0u;
    eq += key == tau ? 1u : 0u;
  }
  // packed scan: both totals stay below 2^16 (n <= 32K)
  uint32_t total;
  const uint32_t pre = block_exclusive_scan<NT>(gt | (eq << 16), &total);
  uint32_t gb = pre & 0xFFFFu, tb = pre >> 16;
  // ordered write: only the marked keys can be selected
  for (uint64_t mk = above | inb; mk; mk &= mk - 1) {
    const int i = __ffsll((long long)mk) - 1;
    const bool hi = (above >> i) & 1u;
    const uint32_t key = hi ? 0xFFFFFFFFu : key_at(i);
    if (hi || key > tau) {
      const uint32_t pos = gb + (tb < ktie ? tb : ktie);
      if (pos < keff) emit(pos, j0 + i);  // always true when the counts are consistent
      ++gb;
    } else if (key == tau) {
      if (tb < ktie && gb + tb < keff) emit(gb + tb, j0 + i);
      ++tb;
    }
  }
}

// ---------------------------------------------------------------------------- multi-CTA rows

// Calls fn(i, key) for every position i in [lo, hi) of a score row, reading the
// 16-byte-aligned body with float4 loads (the scores buffer is 16-byte aligned).
template <typename F>
__device__ __forceinline__ void for_each_key(const float* srow_base, size_t row_off, int lo, int hi, F fn) {
  if (lo >= hi) return;
  const size_t e0 = row_off + lo;
  const int lead = (int)((4 - (e0 & 3)) & 3);
  const int head = lead < hi - lo ? lead : hi - lo;
  const int nv4 = (hi - lo - head) >> 2;
  const float* src = srow_base + e0;
  for (int i = threadIdx.x; i < head; i += blockDim.x) fn(lo + i, order_key(__ldcg(src + i)));
  const float4* src4 = reinterpret_cast<const float4*>(src + head);
#pragma unroll 4
  for (int v = threadIdx.x; v < nv4; v += blockDim.x) {
    const float4 f = __ldcg(src4 + v);
    const int i = lo + head + 4 * v;
    fn(i, order_key(f.x));
    fn(i + 1, order_key(f.y));
    fn(i + 2, order_key(f.z));
    fn(i + 3, order_key(f.w));
  }
  for (int i = head + 4 * nv4 + threadIdx.x; i < hi - lo; i += blockDim.x) fn(lo + i, order_key(__ldcg(src + i)));
}

template <int PASS>
__global__ void __launch_bounds__(kThreads) topk_pass_kernel(const TopkArgs a) {
  constexpr int kShift = PASS == 0 ? 21 : (PASS == 1 ? 10 : 0);
  constexpr int kBits = PASS == 2 ? 10 : 11;
  constexpr int kNb = 1 << kBits;
  constexpr uint32_t kDigit = (uint32_t)kNb - 1u;
  constexpr uint32_t kHigh = PASS == 0 ? 0u : (PASS == 1 ? 0xFFE00000u : 0xFFFFFC00u);
  __shared__ uint32_t sh[kBins];
  __shared__ int s_last;
  __shared__ uint32_t sel[2];

  const int row = blockIdx.y, x = blockIdx.x;
  const RowGeom g = geom(a, row, x, a.seg);
  if (g.k_eff == 0) return;  // nothing to select in this row (same decision in every CTA)
  uint32_t prefix = 0, krem = (uint32_t)g.k_eff;
  if (PASS > 0) {
    prefix = __ldcg(&a.state[row * 4 + 0]);
    krem = __ldcg(&a.state[row * 4 + 1]);
  }
  for (int i = threadIdx.x; i < kNb; i += kThreads) sh[i] = 0u;
  __syncthreads();
  for_each_key(a.scores, (size_t)row * a.max_len, g.lo, g.hi, [&](int, uint32_t key) {
    if ((key & kHigh) == prefix) atomicAdd(&sh[(key >> kShift) & kDigit], 1u);
  });
  __syncthreads();
  uint32_t* gh = a.hist + ((size_t)row * 3 + PASS) * kBins;
  for (int i = threadIdx.x; i < kNb; i += kThreads) {
    const uint32_t v = sh[i];
    if (v) atomicAdd(&gh[i], v);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&a.ticket[row * 4 + PASS], 1u) == (uint32_t)(a.cpr - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kNb; i += kThreads) sh[i] = __ldcg(&gh[i]);
  __syncthreads();
  select_digit<kThreads>(sh, kNb, krem, sel);
  __syncthreads();
  if (threadIdx.x == 0) {
    a.state[row * 4 + 0] = prefix | (sel[0] << kShift);
    a.state[row * 4 + 1] = sel[1];
  }
}

__global__ void __launch_bounds__(kThreads) topk_count_kernel(const TopkArgs a) {
  const int row = blockIdx.y, x = blockIdx.x;
  const RowGeom g = geom(a, row, x, a.seg);
  if (g.k_eff == 0) return;
  const uint32_t tau = __ldcg(&a.state[row * 4 + 0]);
  uint32_t gt = 0, eq = 0;
  for_each_key(a.scores, (size_t)row * a.max_len, g.lo, g.hi, [&](int, uint32_t key) {
    gt += key > tau;
    eq += key == tau;
  });
  uint32_t tg, te;
  block_exclusive_scan<kThreads>(gt, &tg);
  block_exclusive_scan<kThreads>(eq, &te);
  if (threadIdx.x == 0) {
    a.counts[((size_t)row * a.cpr + x) * 2 + 0] = tg;
    a.counts[((size_t)row * a.cpr + x) * 2 + 1] = te;
  }
}

__global__ void __launch_bounds__(kThreads) topk_write_kernel(const TopkArgs a) {
  const int row = blockIdx.y, x = blockIdx.x;
  const RowGeom g = geom(a, row, x, a.seg);
  int32_t* out = a.idx + (size_t)row * a.k;
  if (x == 0)
    for (int j = g.k_eff + threadIdx.x; j < a.k; j += kThreads) out[j] = -1;
  if (g.k_eff == 0) return;
  const uint32_t tau = __ldcg(&a.state[row * 4 + 0]);
  const uint32_t ktie = __ldcg(&a.state[row * 4 + 1]);
  // counts of the segments before this one
  uint32_t pg = 0, pt = 0;
  for (int y = threadIdx.x; y < x; y += kThreads) {
    pg += __ldcg(&a.counts[((size_t)row * a.cpr + y) * 2 + 0]);
    pt += __ldcg(&a.counts[((size_t)row * a.cpr + y) * 2 + 1]);
  }
  uint32_t base_g, base_t;
  block_exclusive_scan<kThreads>(pg, &base_g);
  block_exclusive_scan<kThreads>(pt, &base_t);
  const float* srow = a.scores + (size_t)row * a.max_len;
  constexpr int kPer = 4;
  for (int t0 = g.lo; t0 < g.hi; t0 += kThreads * kPer) {
    uint32_t gtm = 0, eqm = 0;  // bit masks of the thread's kPer consecutive keys
    const int i0 = t0 + threadIdx.x * kPer;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i = i0 + e;
      if (i < g.hi) {
        const uint32_t key = order_key(__ldcg(srow + i));
        gtm |= (uint32_t)(key > tau) << e;
        eqm |= (uint32_t)(key == tau) << e;
      }
    }
    const uint32_t packed = ((uint32_t)__popc(eqm) << 16) | (uint32_t)__popc(gtm);
    uint32_t tot;
    const uint32_t pre = block_exclusive_scan<kThreads>(packed, &tot);
    uint32_t gb = base_g + (pre & 0xffffu);
    uint32_t tb = base_t + (pre >> 16);
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      if (gtm >> e & 1u) {
        const uint32_t pos = gb + (tb < ktie ? tb : ktie);
        if (pos < (uint32_t)g.k_eff) out[pos] = i0 + e;  // always true when the passes are consistent
        ++gb;
      } else if (eqm >> e & 1u) {
        if (tb < ktie && gb + tb < (uint32_t)g.k_eff) out[gb + tb] = i0 + e;
        ++tb;
      }
    }
    base_g += tot & 0xffffu;
    base_t += tot >> 16;
  }
}

int choose_cpr(const skv_problem& p) {
  const int rows = p.batch * p.n_kv_heads;
  const int target = 2 * num_sms();
  int cpr = (target + rows - 1) / rows;
  const int max_cpr = (p.max_len + kMinSeg - 1) / kMinSeg;
  if (cpr > max_cpr) cpr = max_cpr;
  if (cpr < 1) cpr = 1;
  return cpr;
}

int max_cpr(const skv_problem& p) {
  int m = (p.max_len + kMinSeg - 1) / kMinSeg;
  return m < 1 ? 1 : m;
}


struct Layout {
  size_t hist, ticket, state, counts, total;
  size_t cand_key, cand_pos, cand_end;  // two-stage path
  int segs, seg_len, cand_stride;
};

constexpr int kSegLen = 16 * 1024;      // two-stage path: candidates per first-stage selection,
constexpr int kSegLenLong = 32 * 1024;  // or twice that where it saves first-stage waves

// Rows too long for one CTA whose segment winners fit one: select each segment's
// top-k, then the top-k of the winners (the row's top-k is among them).  When few rows
// could instead take the 8-CTA clusters (at most about two waves on the 152 SMs of a
// GB300 -- a function of the problem alone, so the workspace size is too), only while
// the winners stay at half a CTA's capacity: a second stage over 32K winners measured
// slower than the clusters there, and faster with many rows.
bool two_stage(const skv_problem& p, int* segs) {
  const long long s = ((long long)p.max_len + kSegLen - 1) / kSegLen;
  const long long rows = (long long)p.batch * p.n_kv_heads;
  const bool few_rows = p.max_len <= kRowMax8 && rows * 8 <= 2LL * 152;
  const long long cap = few_rows ? kSoloMax / 2 : kSoloMax;
  const bool yes = p.max_len > kSoloMax && s * p.topk <= cap;
  *segs = yes ? (int)s : 0;
  return yes;
}

// First-stage segment length of a two-stage problem.  One 1024-thread CTA per SM
// (152 on a GB300; a constant, so that the workspace size is a function of the
// problem alone) runs the first stage in waves, and a 32K-key selection costs about
// 1.2 times a 16K-key one (its block-wide phases do not grow with the keys).  So
// 32K segments pay where they cut the waves: 8 rows of 1M keys (4 -> 2 waves) went
// from 39 to 29 us, 32 rows of 128K (2 -> 1) from 26 to 20 us; within one wave the
// 16K segments stay faster (16 rows of 128K: 20.2 against 21.3 us).
int first_stage_seg_len(const skv_problem& p) {
  const long long rows = (long long)p.batch * p.n_kv_heads;
  const long long w16 = (rows * (((long long)p.max_len + kSegLen - 1) / kSegLen) + 151) / 152;
  const long long w32 = (rows * (((long long)p.max_len + kSegLenLong - 1) / kSegLenLong) + 151) / 152;
  return w32 * 6 < w16 * 5 ? kSegLenLong : kSegLen;
}

Layout layout(const skv_problem& p) {
  const size_t rows = (size_t)p.batch * p.n_kv_heads;
  Layout l;
  l.hist = 0;
  l.ticket = l.hist + align256(rows * 3 * kBins * 4);
  l.state = l.ticket + align256(rows * 4 * 4);
  l.counts = l.state + align256(rows * 4 * 4);
  // what the chosen path needs: nothing (one CTA), the row histograms (clusters), all four (multi-CTA)
  if (p.max_len <= kSoloMax) l.total = 0;
  else if (p.max_len <= kRowMax8) l.total = l.ticket;
  else l.total = l.counts + align256(rows * (size_t)max_cpr(p) * 2 * 4);
  l.segs = 0;
  l.seg_len = kSegLen;
  l.cand_stride = 0;
  l.cand_key = l.cand_pos = l.cand_end = 0;
  if (two_stage(p, &l.segs)) {
    l.seg_len = first_stage_seg_len(p);
    l.segs = (int)(((long long)p.max_len + l.seg_len - 1) / l.seg_len);
    l.cand_stride = (int)((((size_t)l.segs * p.topk) + 3) & ~(size_t)3);
    l.cand_key = 0;
    l.cand_pos = align256(rows * l.cand_stride * 4);
    l.cand_end = l.cand_pos + align256(rows * l.cand_stride * 4);
    l.total = l.cand_end;
  }
  return l;
}

template <int kCluster, int NT>
skv_status launch_row(const skv_problem& p, const TopkArgs& a0, int rows, int max_len, cudaStream_t st) {
  TopkArgs a = a0;
  a.row_q = ((p.max_len + kCluster - 1) / kCluster + 31) & ~31;
  const size_t smem = (size_t)a.row_q * 4;
  const int max_smem = ((max_len + kCluster - 1) / kCluster + 31) / 32 * 32 * 4;
  const skv_status prep = prepare_kernel((const void*)topk_row_kernel<kCluster, NT>, max_smem);
  if (prep != SKV_OK) return prep;
  if (launch_dependent(topk_row_kernel<kCluster, NT>, dim3(rows * kCluster), dim3(NT), smem, st, kCluster, a) !=
      cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

template <int MODE>
skv_status launch_solo(const TopkArgs& a, dim3 grid, int n_max, cudaStream_t st) {
  if (n_max > kSoloMax) return SKV_ERR_UNSUPPORTED;  // more keys than one CTA holds
  const skv_status prep = prepare_kernel((const void*)topk_solo_kernel<MODE>, (int)solo_smem_bytes(kSoloMax));
  if (prep != SKV_OK) return prep;
  if (launch_dependent(topk_solo_kernel<MODE>, grid, dim3(kSoloThreads), solo_smem_bytes(n_max), st, 1, a) !=
      cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

skv_status launch_lean(const TopkArgs& a, int rows, cudaStream_t st) {
  if (launch_dependent(topk_lean_kernel, dim3(rows), dim3(kLeanThreads), 0, st, 1, a) != cudaSuccess)
    return SKV_ERR_CUDA;
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace

size_t topk_workspace_bytes(const skv_problem& p) { return layout(p).total; }

bool topk_maps_positions(const skv_problem& p) {
  int segs = 0;
  return p.max_len <= kSoloMax || two_stage(p, &segs);
}

skv_status launch_topk(const skv_problem& p, const float* scores, int32_t* idx, void* ws, int32_t* status,
                       cudaStream_t st, uint32_t* zero_words, bool* zeroed, const int32_t* row_geom,
                       const PrefetchView* pf, const int32_t* pos_map) {
  if (zeroed != nullptr) *zeroed = false;
  if (pos_map != nullptr && !topk_maps_positions(p)) return SKV_ERR_UNSUPPORTED;
  const int rows = p.batch * p.n_kv_heads;
  if (((uintptr_t)scores & 15u) != 0 || ((uintptr_t)ws & 15u) != 0) return SKV_ERR_INVALID_ARGUMENT;
  if (rows == 0 || p.topk == 0) return SKV_OK;
  const Layout lay = layout(p);
  TopkArgs a;
  a.scores = scores;
  a.idx = idx;
  a.seq_lens = p.seq_lens;
  a.H = p.n_kv_heads;
  a.max_len = p.max_len;
  a.ns = p.n_sink;
  a.nl = p.n_local;
  a.k = p.topk;
  a.cpr = choose_cpr(p);
  a.seg = (p.max_len + a.cpr - 1) / a.cpr;
  a.row_q = 0;
  unsigned char* w = (unsigned char*)ws;
  a.hist = (uint32_t*)(w + lay.hist);
  a.ticket = (uint32_t*)(w + lay.ticket);
  a.state = (uint32_t*)(w + lay.state);
  a.counts = (uint32_t*)(w + lay.counts);
  a.status = status;
  a.zero = nullptr;
  a.row_geom = row_geom;
  a.tau_ema = pf ? pf->tau : nullptr;  // the one-CTA and two-stage paths fold it; the others leave it
  a.pos_map = pos_map;
  a.ema_alpha = pf ? pf->alpha : 0.f;

  a.seg_len = lay.seg_len;
  a.cand_stride = lay.cand_stride;
  a.cand_key = (uint32_t*)(w + lay.cand_key);
  a.cand_pos = (int32_t*)(w + lay.cand_pos);
  if (p.max_len <= kSoloMax) {  // uses no workspace, so it may clear words inside it
    a.zero = zero_words;
    // the one-CTA kernel takes a whole SM a row; more rows than SMs of at most 8K keys go
    // to the lean kernel (longer rows measured faster on the one-CTA kernel, in waves)
    const bool lean = rows > num_sms() && p.max_len <= kLeanMax;
    const skv_status r = lean ? launch_lean(a, rows, st) : launch_solo<0>(a, dim3(rows), p.max_len, st);
    if (r == SKV_OK && zeroed != nullptr) *zeroed = zero_words != nullptr;
    return r;
  }
  if (lay.segs > 0) {  // two stages; the second may clear words that lie past the candidates
    const skv_status r1 = launch_solo<1>(a, dim3(rows, lay.segs), lay.seg_len, st);
    if (r1 != SKV_OK) return r1;
    const bool clear = zero_words != nullptr && (unsigned char*)zero_words >= w + lay.cand_end;
    a.zero = clear ? zero_words : nullptr;
    const skv_status r = launch_solo<2>(a, dim3(rows), lay.segs * p.topk, st);
    if (r == SKV_OK && zeroed != nullptr) *zeroed = clear;
    return r;
  }
  if (p.max_len <= kRowMax8) {
    if (cudaMemsetAsync(a.hist, 0, (size_t)rows * 3 * kBins * 4, st) != cudaSuccess) return SKV_ERR_CUDA;
    return p.max_len <= kRowMax4 ? launch_row<4, kRowThreads>(p, a, rows, kRowMax4, st)
                                 : launch_row<8, kRowThreads>(p, a, rows, kRowMax8, st);
  }
  // multi-CTA rows: clear what the passes accumulate into
  if (cudaMemsetAsync(w, 0, lay.state, st) != cudaSuccess) return SKV_ERR_CUDA;
  dim3 grid(a.cpr, rows);
  topk_pass_kernel<0><<<grid, kThreads, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  topk_pass_kernel<1><<<grid, kThreads, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  topk_pass_kernel<2><<<grid, kThreads, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  topk_count_kernel<<<grid, kThreads, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  topk_write_kernel<<<grid, kThreads, 0, st>>>(a);
  SKV_LAUNCH_CHECK();
  return SKV_OK;
}

}  // namespace skv
