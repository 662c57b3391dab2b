// S2: exact top-k of each (request, KV head) score row (sm_103a).
//
// The k-th largest score is a threshold: every score above it is in the top-k,
// and only ties at the threshold need a rule (ECHO-OSDI26 wiki, core method 3).
// The threshold is found exactly by a most-significant-digit radix select over
// order-preserving 32-bit keys -- histograms and prefix scans instead of a sort
// (ECHO-OSDI26 wiki, core method 4: a 256-bin histogram on the top bits;
// ParisKV notes §2.3: small-integer histogram + prefix scan, `bucket_topk`).
//
//   pass 0/1/2  histogram of key bits [31:21], [20:10], [9:0] over the keys
//               whose higher digits equal the threshold prefix found so far.
//               Every CTA of a row folds its shared-memory histogram into the
//               row's global histogram with atomics, then takes a ticket; the
//               last CTA to arrive (it never waits for anyone) scans the global
//               histogram from the top, fixes the next threshold digit and the
//               number k_rem of threshold-equal keys still to take.
//   count       per CTA segment: keys above the threshold, keys equal to it.
//   write       per CTA segment: stable compaction in position order; a key
//               above the threshold is selected, a key equal to it is selected
//               when fewer than k_rem equal keys precede it in the row.  Output
//               positions come from exclusive scans, so the result is the same
//               on every run: ascending positions, ties to the lower position.
//
// Each row is cut into `cpr` contiguous segments, one CTA each, so the grid
// covers the device even when there are few rows and long histories.
#include "skv_internal.cuh"

namespace skv {
namespace {

constexpr int kThreads = 512;
constexpr int kBins = 2048;
constexpr int kMinSeg = 2048;

struct TopkArgs {
  const float* scores;
  int32_t* idx;
  const int32_t* seq_lens;
  int H, max_len, ns, nl, k, cpr, seg;
  uint32_t* ghist;   // [rows][3][kBins]
  uint32_t* ticket;  // [rows][4]
  uint32_t* state;   // [rows][4]: prefix, k_rem
  uint32_t* counts;  // [rows][cpr][2]
  int32_t* status;
};

struct RowGeom {
  int s_end, l_start, n, k_eff, lo, hi;
};

__device__ __forceinline__ RowGeom geom(const TopkArgs& a, int row, int x) {
  RowGeom g;
  const int b = row / a.H;
  const int L = load_len(a.seq_lens, b, a.max_len, a.status);
  Regions r = regions_of(L, a.ns, a.nl);
  g.s_end = r.s_end;
  g.l_start = r.l_start;
  g.n = r.l_start - r.s_end;
  g.k_eff = a.k < g.n ? a.k : g.n;
  long long lo = (long long)g.s_end + (long long)x * a.seg;
  long long hi = lo + a.seg;
  g.lo = (int)(lo < g.l_start ? lo : g.l_start);
  g.hi = (int)(hi < g.l_start ? hi : g.l_start);
  return g;
}

// Exclusive block-wide scan of one uint32 per thread; returns the prefix, and
// the block total in *total.  kThreads == 512 (16 warps).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total) {
  __shared__ uint32_t warp_sums[kThreads / 32];
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
    uint32_t w = lane < kThreads / 32 ? warp_sums[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < kThreads / 32) warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const uint32_t before_warp = warp > 0 ? warp_sums[warp - 1] : 0u;
  *total = warp_sums[kThreads / 32 - 1];
  const uint32_t excl = before_warp + x - v;
  __syncthreads();  // warp_sums reusable after return
  return excl;
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

  const int row = blockIdx.y, x = blockIdx.x;
  const RowGeom g = geom(a, row, x);
  if (g.k_eff == 0) return;  // nothing to select in this row (same decision in every CTA)
  uint32_t prefix = 0, krem = (uint32_t)g.k_eff;
  if (PASS > 0) {
    prefix = __ldcg(&a.state[row * 4 + 0]);
    krem = __ldcg(&a.state[row * 4 + 1]);
  }
  for (int i = threadIdx.x; i < kNb; i += kThreads) sh[i] = 0u;
  __syncthreads();
  const float* srow = a.scores + (size_t)row * a.max_len;
  for (int i = g.lo + threadIdx.x; i < g.hi; i += kThreads) {
    const uint32_t key = order_key(__ldcg(srow + i));
    if ((key & kHigh) == prefix) atomicAdd(&sh[(key >> kShift) & kDigit], 1u);
  }
  __syncthreads();
  uint32_t* gh = a.ghist + ((size_t)row * 3 + PASS) * kBins;
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
  // descending rank r = 4 * tid + e  <->  bin kNb - 1 - r
  uint32_t mine = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int r = 4 * threadIdx.x + e;
    if (r < kNb) mine += sh[kNb - 1 - r];
  }
  uint32_t total;
  uint32_t before = block_exclusive_scan(mine, &total);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int r = 4 * threadIdx.x + e;
    if (r < kNb) {
      const uint32_t bin = (uint32_t)(kNb - 1 - r);
      const uint32_t c = sh[bin];
      if (before < krem && before + c >= krem) {
        a.state[row * 4 + 0] = prefix | (bin << kShift);
        a.state[row * 4 + 1] = krem - before;
      }
      before += c;
    }
  }
}

__global__ void __launch_bounds__(kThreads) topk_count_kernel(const TopkArgs a) {
  const int row = blockIdx.y, x = blockIdx.x;
  const RowGeom g = geom(a, row, x);
  if (g.k_eff == 0) return;
  const uint32_t tau = __ldcg(&a.state[row * 4 + 0]);
  const float* srow = a.scores + (size_t)row * a.max_len;
  uint32_t gt = 0, eq = 0;
  for (int i = g.lo + threadIdx.x; i < g.hi; i += kThreads) {
    const uint32_t key = order_key(__ldcg(srow + i));
    gt += key > tau;
    eq += key == tau;
  }
  uint32_t tg, te;
  block_exclusive_scan(gt, &tg);
  block_exclusive_scan(eq, &te);
  if (threadIdx.x == 0) {
    a.counts[((size_t)row * a.cpr + x) * 2 + 0] = tg;
    a.counts[((size_t)row * a.cpr + x) * 2 + 1] = te;
  }
}

__global__ void __launch_bounds__(kThreads) topk_write_kernel(const TopkArgs a) {
  const int row = blockIdx.y, x = blockIdx.x;
  const RowGeom g = geom(a, row, x);
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
  block_exclusive_scan(pg, &base_g);
  block_exclusive_scan(pt, &base_t);
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
    const uint32_t pre = block_exclusive_scan(packed, &tot);
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

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t topk_workspace_bytes(const skv_problem& p) {
  const size_t rows = (size_t)p.batch * p.n_kv_heads;
  size_t b = align256(rows * 3 * kBins * 4) + align256(rows * 4 * 4);  // histograms + tickets (zeroed)
  b += align256(rows * 4 * 4);                                        // row state
  b += align256(rows * (size_t)max_cpr(p) * 2 * 4);                   // segment counts
  return b;
}

skv_status launch_topk(const skv_problem& p, const float* scores, int32_t* idx, void* ws,
                       int32_t* status, cudaStream_t st) {
  const int rows = p.batch * p.n_kv_heads;
  if (rows == 0 || p.topk == 0) return SKV_OK;
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
  unsigned char* w = (unsigned char*)ws;
  const size_t hist_bytes = align256((size_t)rows * 3 * kBins * 4);
  const size_t ticket_bytes = align256((size_t)rows * 4 * 4);
  a.ghist = (uint32_t*)w;
  a.ticket = (uint32_t*)(w + hist_bytes);
  a.state = (uint32_t*)(w + hist_bytes + ticket_bytes);
  a.counts = (uint32_t*)(w + hist_bytes + 2 * ticket_bytes);
  a.status = status;
  if (cudaMemsetAsync(w, 0, hist_bytes + ticket_bytes, st) != cudaSuccess) return SKV_ERR_CUDA;
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
