/*
 * skv.h -- C ABI of the GB300 sparse-decode library (libskv.so).
 *
 * One decode step, for every (request b, KV head h):
 *   score   every candidate history key against the group's query      skv_score
 *   select  the exact top-k candidate positions                        skv_topk
 *   resolve the attended positions through the slot table and read
 *           their K/V rows from the GPU pool or the pinned host pool   skv_gather
 *   attend  with split-K flash decoding and a log-sum-exp merge        skv_sparse_attn
 * and all four chained on one stream                                   skv_decode_step
 *
 * Conventions (every entry point):
 *  - The caller owns all memory.  Device buffers, pinned host pools and the
 *    workspace are allocated by the caller; the library allocates nothing,
 *    frees nothing and never synchronises.  Every call enqueues kernels (and,
 *    for skv_topk / skv_decode_step, one cudaMemsetAsync on the workspace) on
 *    `stream` and returns.  `stream` is a cudaStream_t passed as void*; NULL
 *    is the legacy default stream.  The device is the caller's current device.
 *  - Host rows are read by the kernels themselves through unified virtual
 *    addressing: host_k / host_v must be device-accessible pinned memory
 *    (cudaHostAlloc / cudaHostRegister).  The CPU launches no copy.
 *    (ECHO-OSDI26 wiki, core method 1: a GPU kernel reads host addresses
 *    directly; OasisKV notes, §3.3 Algorithm 1: UVA gather.)
 *  - Arguments the host can check are checked before anything is enqueued;
 *    a bad argument returns SKV_ERR_INVALID_ARGUMENT / SKV_ERR_UNSUPPORTED /
 *    SKV_ERR_WORKSPACE_TOO_SMALL and enqueues nothing.
 *  - Faults found on the device (a slot-table entry outside its pool, a
 *    selected position outside the candidate region, a wait that gave up)
 *    never trap: the kernel ORs a SKV_DEV_* bit into *dev_status, skips the
 *    offending row (a skipped key scores NaN and ranks last; a skipped
 *    attended row gets zero weight) and completes.  dev_status is a device
 *    int32 the caller zeroes and reads after the stream has drained; it may
 *    be NULL (no reporting).
 *  - All tensors are dense row-major ("C order") and 16-byte aligned.
 *    Element types: SKV_DTYPE_BF16 (bf16 storage, fp32 arithmetic) or
 *    SKV_DTYPE_F32 (fp32 storage and arithmetic) for q, keys, pools and out;
 *    scores and lse are always fp32; indices and tables int32.
 *
 * Regions of request b with history length L = seq_lens[b] (positions 0..L-1,
 * the current token included at L-1):
 *   sink        [0, s_end)            s_end   = min(n_sink, L)
 *   candidates  [s_end, l_start)      l_start = max(s_end, L - n_local)
 *   local       [l_start, L)
 * Sink and local are always attended; the top-k is taken over the candidates
 * only (ParisKV notes, §2.5: Sink and Local are attended densely on the GPU,
 * the retrieval region is the rest).
 */
#ifndef SKV_H
#define SKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t skv_status;

/* Return codes. */
#define SKV_OK 0
#define SKV_ERR_INVALID_ARGUMENT 1   /* NULL / negative / inconsistent sizes / misaligned */
#define SKV_ERR_UNSUPPORTED 2        /* valid but not built (e.g. d_idx != 128)            */
#define SKV_ERR_CUDA 3               /* a CUDA runtime call or launch failed                */
#define SKV_ERR_WORKSPACE_TOO_SMALL 4
#define SKV_ERR_DEVICE_FAULT 5       /* reserved: used by callers that map dev_status       */
#define SKV_ERR_TIMEOUT 6            /* reserved: used by callers that map dev_status       */

/* Bits of *dev_status (OR-ed by kernels). */
#define SKV_DEV_BAD_SLOT 1           /* slot-table entry names a block outside its pool     */
#define SKV_DEV_BAD_INDEX 2          /* a selected position is outside the candidate region */
#define SKV_DEV_BAD_LENGTH 4         /* seq_lens[b] outside [0, max_len] (clamped)          */
#define SKV_DEV_TIMEOUT 8            /* an internal pipeline wait gave up (never expected)  */

/* Element types. */
#define SKV_DTYPE_BF16 0
#define SKV_DTYPE_F32 1

/* How the scoring heads of one KV head's group combine into one score per key.
 * Each KV head ranks the context on its own (OasisKV notes, §3.2); the pages
 * leave the combination of a group's heads open, so both readings are offered,
 * and a third where every query head ranks on its own. */
#define SKV_AGG_MEAN 0               /* <q_bar, k>, q_bar the mean of the heads (orders keys like the sum) */
#define SKV_AGG_MAX 1                /* max over the heads g of <q_g, k>; bf16 with at most 16 scoring
                                        heads per KV head, else SKV_ERR_UNSUPPORTED */
/* Per query head: every query head j ranks the keys of its KV head j / G with its own
 * query, <q_j, k>, selects its own top-k and attends its own list.  The rows of scores,
 * idx and the gathered rows are then per query head (n_q_heads of them per request
 * instead of n_kv_heads); the keys are read once per KV head while scoring.  bf16,
 * n_idx_q_heads == n_q_heads (the attention query scores), at most 16 query heads per
 * KV head, paged K/V pools; skv_score, skv_topk, skv_topk_static, skv_gather,
 * skv_sparse_attn and skv_decode_step only (the block, prefetch, slot-cache and
 * ParisKV entry points return SKV_ERR_UNSUPPORTED). */
#define SKV_AGG_HEAD 2

/* Where the scored keys live. */
#define SKV_INDEX_PAGED 0            /* the K pool itself, through the slot table (block_size 16) */
#define SKV_INDEX_CONTIG 1           /* separate GPU-resident index keys [batch, n_kv_heads, max_len, d_idx] */

/*
 * Sizes of one decode step.
 *   n_q_heads      query heads; G = n_q_heads / n_kv_heads query heads share a
 *                  KV head (query head j belongs to KV head j / G).
 *   d_qk, d_v      key/query and value widths: 128/128 for paged K/V pools;
 *                  576/512 for the latent layout (gpu_v == NULL), where V is the
 *                  first d_v entries of the shared K row.
 *   d_idx          width of the scored keys and scoring query (128).
 *   n_idx_q_heads  heads of the scoring query; n_idx_q_heads / n_kv_heads of them
 *                  are averaged per KV head.  For SKV_INDEX_PAGED scoring with the
 *                  attention query itself: n_q_heads, with d_idx == d_qk.
 *   max_len        capacity: every seq_lens[b] <= max_len; sizes the scores row.
 *   topk           k: positions selected per (request, KV head) among candidates.
 *   n_sink,n_local window sizes (see regions above).
 *   block_size     tokens per slot-table entry: 16 (paged blocks) or 1 (per-token map).
 *   dtype          SKV_DTYPE_*.
 *   group_agg      SKV_AGG_MEAN, SKV_AGG_MAX or SKV_AGG_HEAD.
 *   sm_scale       softmax scale of the attention logits; <= 0 means 1/sqrt(d_qk).
 *   n_splits       split-K chunks per (request, KV head) for attention; 0 lets
 *                  the library choose from the sizes.
 *   seq_lens       device int32 [batch].
 * batch and n_kv_heads above 65535 (grid extents) return SKV_ERR_UNSUPPORTED.
 */
typedef struct skv_problem {
  int32_t batch;
  int32_t n_kv_heads;
  int32_t n_q_heads;
  int32_t d_qk;
  int32_t d_v;
  int32_t d_idx;
  int32_t n_idx_q_heads;
  int32_t max_len;
  int32_t topk;
  int32_t n_sink;
  int32_t n_local;
  int32_t block_size;
  int32_t dtype;
  int32_t group_agg;
  float sm_scale;
  int32_t n_splits;
  const int32_t *seq_lens;
} skv_problem;

/*
 * The KV pool: logical position t of request b resolves through
 *   e = slot_table[b * table_stride + t / block_size]
 *   e >= 0 : GPU block e,          rows gpu_k[e][h][t % block_size][:]
 *   e <  0 : host block (-e - 1),  rows host_k[-e-1][h][t % block_size][:]
 * (vToken notes, §3.4 Eq. (2): slot = block_id * S + offset; UlaCache article
 * §5: one logical address space, the map names the tier.)
 * Pools are [n_blocks, n_kv_heads, block_size, d] (d = d_qk for K, d_v for V).
 * gpu_v == NULL selects the latent layout: V is the first d_v entries of the K
 * row (n_kv_heads must be 1, host_v must be NULL).  host_* may be NULL when no
 * table entry is negative; n_*_blocks bound the entries (checked on device).
 * table_stride >= ceil(max_len / block_size).
 *
 * table_heads = 1 selects one table row per (request, KV head) instead (OasisKV
 * notes, §3.5, Fig. 9: each KV head keeps its own logical-block map, since different
 * heads select different blocks):
 *   e = slot_table[(b * n_kv_heads + h) * table_stride + t / block_size]
 *   e >= 0 : GPU block e holds this head's block only: gpu_k[e][t % block_size][:]
 *            (GPU pools [n_gpu_blocks, block_size, d])
 *   e <  0 : host block (-e - 1) as above (host pools keep every head).
 * Supported by skv_score, skv_gather, skv_sparse_attn, skv_decode_step and the slot
 * cache (skv_cache_*, skv_decode_step_cached), K and V pools (not the latent layout);
 * the other entry points return SKV_ERR_UNSUPPORTED.
 * table_heads = 0 (the default of a zeroed struct) is the shared table above.
 */
typedef struct skv_kv_pool {
  const void *gpu_k;
  const void *gpu_v;
  int64_t n_gpu_blocks;
  const void *host_k;
  const void *host_v;
  int64_t n_host_blocks;
  const int32_t *slot_table;
  int32_t table_stride;
  int32_t table_heads;            /* 0: one table row per request; 1: one per (request, KV head) */
} skv_kv_pool;

/*
 * What skv_score reads.  SKV_INDEX_PAGED: the K pool through the slot table
 * (keys must be GPU-resident for candidate positions: host-resident blocks are
 * read over UVA, slowly).  SKV_INDEX_CONTIG: `keys` is a GPU-resident
 * [batch, n_kv_heads, max_len, d_idx] tensor (the indexer's key cache, kept on
 * the GPU: ECHO-OSDI26 wiki, core method 1).
 */
typedef struct skv_index_src {
  int32_t layout;
  const void *keys;
} skv_index_src;

/* Bytes of workspace skv_topk, skv_sparse_attn and skv_decode_step need for
 * this problem (the same figure serves all three). */
skv_status skv_workspace_size(const skv_problem *p, size_t *bytes);

/*
 * S0 + S1: scores[b][h][t] = <q_bar(b,h), key(b,h,t)> in fp32 for every
 * candidate t of request b; other positions of the row are left untouched.
 *   q_score  [batch, n_idx_q_heads, d_idx]; q_bar(b,h) is the mean of heads
 *            h*Gi .. h*Gi+Gi-1 with Gi = n_idx_q_heads / n_kv_heads.
 *   scores   device fp32 [batch, n_kv_heads, max_len]; with SKV_AGG_HEAD
 *            [batch, n_q_heads, max_len], row j the scores of query head j.
 * (ParisKV notes, §1 Eqs. (1)-(3): s_i = <k_i, q>; ECHO-OSDI26 wiki, core
 * method 3: the indexer scores every history key; OasisKV notes §3.2: every
 * KV head ranks the whole context on its own.)
 */
skv_status skv_score(const skv_problem *p, const void *q_score, const skv_index_src *index,
                     const skv_kv_pool *pool, float *scores, int32_t *dev_status, void *stream);

/*
 * S2: idx[b][h][0..k_eff) = the k_eff = min(topk, #candidates) candidate
 * positions with the largest scores, ascending; ties go to the lower position;
 * -0.0 equals +0.0; NaN ranks below every number.  idx[b][h][k_eff..topk) = -1.
 * Deterministic.  (ECHO-OSDI26 wiki, core method 3: the k-th score is a
 * threshold -- every key above it is in the exact top-k; core method 4 and
 * ParisKV notes §2.3: radix histograms with prefix scans instead of a sort.)
 *   scores  device fp32 [batch, n_kv_heads, max_len] (candidates read only).
 *   idx     device int32 [batch, n_kv_heads, topk].
 *   (SKV_AGG_HEAD: n_q_heads rows a request in both, one per query head.)
 *   ws      device workspace of at least skv_workspace_size() bytes.
 */
skv_status skv_topk(const skv_problem *p, const float *scores, int32_t *idx, void *ws,
                    size_t ws_bytes, int32_t *dev_status, void *stream);

/*
 * skv_topk without a workspace argument -- the pages have no counterpart; this
 * exists for callers that cannot allocate device memory when they select (a
 * plugin inside a runtime that owns the memory pool and gives it no allocator,
 * or a serving loop that must not call cudaMalloc, which can synchronise the
 * device).  Same arguments and results as skv_topk; the scratch is a fixed
 * 16 MiB device array inside the library (held on every GPU that loads the
 * library's module until the process exits), so this call allocates nothing.
 * Problems whose top-k scratch exceeds 16 MiB return SKV_ERR_WORKSPACE_TOO_SMALL
 * and enqueue nothing.  That scratch, for rows = batch * n_kv_heads (batch *
 * n_q_heads with SKV_AGG_HEAD):
 *   max_len <= 32768: none;
 *   longer rows whose segment winners fit one CTA (two stages): two arrays
 *     (winner keys, winner positions) of rows * round_up(segs * topk, 4) * 4
 *     bytes, each rounded up to 256 bytes; segs = ceil(max_len / seg), with seg
 *     16K keys, or 32K where that cuts the first stage's waves (a function of
 *     the problem alone);
 *   otherwise rows up to 128K keys: rows * 24 KB (digit histograms), 256-byte
 *     rounded; longer rows add tickets, row state and per-CTA counts, about
 *     24.1 KB per row plus 8 bytes per 2K keys of a row.
 * So roughly 680 request x KV-head rows fit when the histograms are needed.
 * The array's device address is looked up with cudaGetSymbolAddress in the
 * caller's current context on the first call in that context (that includes
 * the first call after cudaDeviceReset, which brings up a new context), and
 * cached with the context's id; make that first call before any stream
 * capture.  All calls share the array: calls whose kernels overlap on the GPU
 * race and give wrong results; serialise them (one stream, or events).
 */
skv_status skv_topk_static(const skv_problem *p, const float *scores, int32_t *idx, int32_t *dev_status,
                           void *stream);

/*
 * S3 materialised: the attended rows of every (b, h) in attended order
 *   list(b,h) = [0, s_end) ++ idx[b][h][0..topk) ++ [l_start, L)
 * resolved through the slot table.  k_out [batch, n_kv_heads, n_att, d_qk],
 * v_out [batch, n_kv_heads, n_att, d_v] with n_att = n_sink + topk + n_local
 * (SKV_AGG_HEAD: n_q_heads rows a request, query head j's list from KV head j / G);
 * list entries that are empty (idx < 0, or past the end of a short list) give
 * zero rows.  v_out may be NULL.  (vToken notes §3.4 Eq. (2); ECHO-OSDI26
 * wiki, core method 2: recall through the slot map.)
 */
skv_status skv_gather(const skv_problem *p, const skv_kv_pool *pool, const int32_t *idx,
                      void *k_out, void *v_out, int32_t *dev_status, void *stream);

/*
 * S3 + S4 + S5: for every query head j of KV head h = j / G,
 *   z_t = sm_scale * <q[b][j], K_t>,  out[b][j] = sum_t softmax(z)_t V_t,
 *   lse[b][j] = log sum_t exp(z_t)   (natural log)
 * over t in list(b,h) (idx entries < 0 are skipped; SKV_AGG_HEAD: over query
 * head j's own list(b,j), idx [batch, n_q_heads, topk]), computed as n_splits
 * fp32 online-softmax partials merged by log-sum-exp.  K/V rows are read
 * through the slot table inside the kernel (GPU pool from HBM, host pool over
 * UVA).  (ParisKV notes §2.5 and §1 Eqs. (1)-(3).)
 *   q    [batch, n_q_heads, d_qk];  out [batch, n_q_heads, d_v] (dtype);
 *   lse  fp32 [batch, n_q_heads] or NULL.
 */
skv_status skv_sparse_attn(const skv_problem *p, const void *q, const skv_kv_pool *pool,
                           const int32_t *idx, void *out, float *lse, void *ws, size_t ws_bytes,
                           int32_t *dev_status, void *stream);

/*
 * The whole step on one stream: skv_score (q_score, or q when q_score is NULL),
 * skv_topk, skv_sparse_attn.  scores and idx are outputs too.
 */
skv_status skv_decode_step(const skv_problem *p, const void *q, const void *q_score,
                           const skv_index_src *index, const skv_kv_pool *pool, float *scores,
                           int32_t *idx, void *out, float *lse, void *ws, size_t ws_bytes,
                           int32_t *dev_status, void *stream);

/* Static text of a status code. */
const char *skv_status_string(skv_status s);

/* Kernels this library has launched in this process (monotonic). */
uint64_t skv_launch_count(void);

/*
 * Check of the bounded waits (the library's failure detection; no page passage).
 * Every kernel that waits on an mbarrier gives up after a clock limit (about 2 s),
 * ORs SKV_DEV_TIMEOUT into *dev_status and returns, so a lost arrival never hangs
 * the device.  This call runs that same wait in a one-CTA kernel, on a barrier that
 * nothing completes (arrive = 0) or that one thread completes first (arrive = 1),
 * giving up after limit_cycles SM clocks.  After the stream drains, *dev_status has
 * SKV_DEV_TIMEOUT set (arrive = 0) or nothing added (arrive = 1).
 *   limit_cycles  in [1, 4e9] (4e9 clocks are about 2 s), else SKV_ERR_INVALID_ARGUMENT.
 *   arrive        0 or 1, else SKV_ERR_INVALID_ARGUMENT.
 *   dev_status    device int32, required: NULL returns SKV_ERR_INVALID_ARGUMENT.
 */
skv_status skv_check_wait_timeout(int64_t limit_cycles, int32_t arrive, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------------------
 * Block selection from per-block key summaries (OasisKV notes, §3.2 "compressed
 * key summaries", after Quest): every 16-token block of a KV head keeps the
 * per-coordinate minimum and maximum of its keys; a KV head ranks blocks from
 * those two rows alone and attends the chosen blocks whole.
 *
 * A block's score is the largest <q, k> any key inside its per-coordinate box can
 * reach, sum_j max(q_j min_j, q_j max_j): q the group's mean query (SKV_AGG_MEAN)
 * or the largest of the heads' own bounds (SKV_AGG_MAX).  The sink and local
 * windows are rounded outward to whole blocks: blocks [0, ceil(n_sink / 16)) and
 * the blocks from floor(max(L - n_local, 0) / 16) on (none when n_local == 0);
 * the candidates are the blocks between.  The top topk_blocks candidates are
 * chosen exactly (ties to the lower block), and every token t < L of the sink,
 * chosen and local blocks is attended.
 *
 * Requirements: paged K/V pool (gpu_v != NULL) with block_size 16, d_qk = d_idx =
 * 128, n_idx_q_heads == n_q_heads (the attention group scores its blocks); else
 * SKV_ERR_UNSUPPORTED.  Errors are reported as for the token path above.
 *
 * summaries: device [batch, n_kv_heads, ceil(max_len / 16), 2, 128] of the pool's
 *            element type; per block the min row, then the max row; 16-byte
 *            aligned; caller-owned.  Blocks with no token below seq_lens[b] are
 *            not written.  A bad slot-table entry writes NaN rows (the block
 *            ranks last) and sets SKV_DEV_BAD_SLOT.
 * block_idx: device int32 [batch, n_kv_heads, topk_blocks]: chosen blocks,
 *            ascending, -1 past min(topk_blocks, candidate blocks).
 * att_idx:   device int32 [batch, n_kv_heads, list_len]: attended token
 *            positions, ascending, -1 padded; list_len from
 *            skv_block_workspace_size (16 * (ceil(n_sink/16) + topk_blocks +
 *            ceil(n_local/16) + 1)).
 * ------------------------------------------------------------------------------------ */

/* Workspace bytes for skv_block_select / skv_block_decode_step, and list_len
 * (may be NULL).  Enqueues nothing. */
skv_status skv_block_workspace_size(const skv_problem *p, int32_t topk_blocks, size_t *bytes, int32_t *list_len);

/* Writes the min / max summary rows of every block of every (request, KV head),
 * reading the K rows through the slot table (GPU pool, or the pinned host pool
 * over UVA).  Maintenance: run when blocks fill, not every decode step. */
skv_status skv_block_summaries(const skv_problem *p, const skv_kv_pool *pool, void *summaries, int32_t *dev_status,
                               void *stream);

/* Scores the candidate blocks from the summaries, chooses the top topk_blocks of
 * every (request, KV head) and writes block_idx and the attended token list att_idx. */
skv_status skv_block_select(const skv_problem *p, int32_t topk_blocks, const void *q, const void *summaries,
                            int32_t *block_idx, int32_t *att_idx, void *ws, size_t ws_bytes, int32_t *dev_status,
                            void *stream);

/* skv_block_select followed by skv_sparse_attn over att_idx (windows of width
 * zero); out / lse as for skv_decode_step. */
skv_status skv_block_decode_step(const skv_problem *p, int32_t topk_blocks, const void *q, const void *summaries,
                                 const skv_kv_pool *pool, int32_t *block_idx, int32_t *att_idx, void *out,
                                 float *lse, void *ws, size_t ws_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------------------
 * Threshold prefetch of host rows (ECHO-OSDI26 wiki, core methods 3 and 5).  The
 * k-th largest score is a threshold; an EMA over steps of each (request, KV head)'s
 * k-th score predicts this step's.  While the indexer scores, a prefetch warp copies
 * the host rows of keys scoring above the prediction into a GPU staging area; the
 * exact top-k then runs as always, and the gather reads staged rows from HBM and
 * every other selected host row from the host pool (guaranteed recall).  A wrong
 * prediction costs speed only: the step's results are the same bits as without it.
 *
 * State, caller-owned, persistent across steps (zero-filled except tau_ema):
 *   tau_ema  device float [batch * n_kv_heads]: the EMA; NaN until a first step
 *            has selected (initialise to NaN: the first step prefetches nothing).
 *   epoch    device uint32 [1]: steps completed (initialise to 0).
 *   map      device uint64 [batch * n_kv_heads * max_len], 8-byte aligned,
 *            zero-filled once: (step tag << 32) | staging slot of a staged position.
 *   staging  device, 16-byte aligned, of the pool's element type: latent layout
 *            [batch * n_kv_heads, cap, d_qk]; paged pools [2, batch * n_kv_heads, cap, 128]
 *            (the staged K rows, then the staged V rows).
 *   count    device uint32 [batch * n_kv_heads], zero-filled once (reset by every step).
 *   stats    device uint32 [2] or NULL: running counts of attended host rows found
 *            staged / read from the host pool.
 *   cap      staging rows per (request, KV head) per step; rows past it are read
 *            from the host later.
 *   alpha    weight of the newest k-th score in the EMA, in (0, 1] (the pages: 0.5).
 * Supported, with contiguous index keys (a GPU-resident copy of the keys), bf16 and
 * SKV_AGG_MEAN: the latent layout (pool.gpu_v == NULL, block_size 1), or a paged pool
 * of 16-token blocks with d_qk = d_v = 128 whose host blocks back part of the history
 * (the 1M-context host-pool workload); else SKV_ERR_UNSUPPORTED.  The paged step ends
 * with one small kernel that advances the epoch and empties the staging counts.  One
 * step at a time per state (steps on one stream).
 * ------------------------------------------------------------------------------------ */
typedef struct skv_prefetch {
  float *tau_ema;
  uint32_t *epoch;
  uint64_t *map;
  void *staging;
  uint32_t *count;
  uint32_t *stats;
  int32_t cap;
  float alpha;
} skv_prefetch;

/* skv_decode_step with threshold prefetch of host rows; same results. */
skv_status skv_decode_step_prefetch(const skv_problem *p, const void *q, const void *q_score,
                                    const skv_index_src *index, const skv_kv_pool *pool, float *scores,
                                    int32_t *idx, void *out, float *lse, void *ws, size_t ws_bytes,
                                    const skv_prefetch *pf, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------------------
 * GPU slot cache over a host pool that backs every token (ECHO-OSDI26 wiki, core
 * method 2).  The host pool holds token t of request b at row b * max_len + t (slot
 * table entry -(b * max_len + t) - 1); the GPU pool's rows ("slots") cache some
 * tokens (entry = the slot).  After a step's attention the cache is updated inside
 * the same enqueued work, with fixed-size state only:
 *   - attended tokens in GPU slots mark their slot used this step;
 *   - the attended tokens read from the host (misses), in (request, list position)
 *     order, take the best eviction candidates -- free slots, then the oldest last
 *     use, then the lower slot; the top `budget` of them by the exact top-k -- in
 *     ascending slot order, one each, while both last;
 *   - an evicted token's table entry returns to its host row; the promoted row is
 *     copied into its slot from the step's gathered rows (no second host read), and
 *     only then does its table entry name the slot (data, then map: UlaCache
 *     article, §8).
 * The step's own results are those of skv_decode_step; later steps find the
 * promoted tokens in HBM.
 *
 * cache.owner  device int32 [n_gpu_blocks]: b * max_len + t of the slot's token, or
 *              -1 (free).  Must agree with the slot table at the first call.
 * cache.prio   device int32 [n_gpu_blocks]: the last step that used the slot (start: -1).
 * cache.step   device int32 [1]: this step's number, advanced by every call.
 * cache.budget promotions per step, at most.
 * cache.stats  device uint64 [3] or NULL: every call adds its attended tokens found in
 *              GPU slots, those read from the host, and its promotions.
 * The call updates pool->slot_table and the rows of pool->gpu_k in place (both must be
 * writable and used by no other work meanwhile).  Requirements: the latent layout
 * (pool->gpu_v == NULL, block_size 1), batch <= 64, n_host_blocks >= batch * max_len;
 * else SKV_ERR_UNSUPPORTED.
 *
 * With one table row per (request, KV head) (pool->table_heads = 1; OasisKV notes,
 * §3.5: each head keeps its own blocks resident) the same rule runs per (request, KV
 * head) u = b * n_kv_heads + h on blocks: the host pool backs block j of request b at
 * host block b * table_stride + j (every head; entry -(b * table_stride + j) - 1), a
 * slot holds one head's block, the distinct blocks of u's attended positions protect
 * their slots or miss, the misses are taken in (u, block) order, and owners are
 * u * table_stride + j.  A promoted block's K and V rows are copied from the host pool
 * into gpu_k and gpu_v.  Requirements: K and V pools, batch * n_kv_heads <= 1024,
 * n_host_blocks >= batch * table_stride, table_stride <= 262144.
 * ------------------------------------------------------------------------------------ */
typedef struct skv_slot_cache {
  int32_t *owner;
  int32_t *prio;
  int32_t *step;
  int32_t budget;
  uint64_t *stats;
} skv_slot_cache;

/* Bytes of the cache update's own workspace (cache_ws below).  Enqueues nothing. */
skv_status skv_cache_workspace_size(const skv_problem *p, const skv_kv_pool *pool, int32_t budget, size_t *bytes);

/* Creates, once per device, the library's side stream and its two events, which
 * skv_decode_step_cached uses to rank eviction candidates beside the step's attention
 * (it creates them itself on first use; call this first to keep their creation out of a
 * stream capture).  Acts on the current device. */
skv_status skv_cache_prepare(void);

/* The slot-cache update alone, for the step that skv_decode_step (or
 * skv_decode_step_prefetch) has just enqueued on `stream` with these same p, pool, idx
 * and ws: the update reads that step's selection and its gathered rows from ws, so
 * nothing may touch ws in between. */
skv_status skv_cache_update(const skv_problem *p, const skv_kv_pool *pool, const int32_t *idx, const void *ws,
                            size_t ws_bytes, const skv_slot_cache *cache, void *cache_ws, size_t cache_ws_bytes,
                            int32_t *dev_status, void *stream);

/* skv_decode_step, then the slot-cache update described above.  The ranking half of the
 * update (marking, eviction scores, their top-k) runs on the library's side stream,
 * forked from `stream` after the selection and joined back before the table changes,
 * so it overlaps the step's gather and attention; everything is ordered on `stream` when
 * the call's work there is complete (CUDA graph capture of `stream` captures both). */
skv_status skv_decode_step_cached(const skv_problem *p, const void *q, const void *q_score,
                                  const skv_index_src *index, const skv_kv_pool *pool, float *scores, int32_t *idx,
                                  void *out, float *lse, void *ws, size_t ws_bytes, const skv_slot_cache *cache,
                                  void *cache_ws, size_t cache_ws_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------------------
 * ParisKV approximate retrieval: an alternative to exact scoring and top-k
 * (ParisKV notes, cc.laoqi.cc, arXiv 2602.07721, §2.2-§2.5).
 *
 * Per (request, KV head) row the GPU keeps compressed metadata of every key, built by
 * skv_paris_encode from the keys of the index source (contiguous index keys with
 * d_idx = 128, or the K pool through the slot table with d_qk = 128):
 *   - normalise, rotate by the SRHT R = H_128 diag(signs) / sqrt(128);
 *   - per 8-dim subspace s (16 of them): r = |k_s|, u = k_s / r; the centroid id is the
 *     sign pattern of u (bit j set iff u_j < 0), the argmax over the 256 fixed
 *     centroids (+-1/sqrt 8)^8 (§2.2, Eqs. (5)-(6));
 *   - each coordinate of u gets a 4-bit code, sign << 3 | cell, the cell from an
 *     8-level Lloyd-Max quantiser of |u_j| under u_j^2 ~ Beta(1/2, 7/2) (§2.4,
 *     Prop. 4.1; skv_paris_quantizer gives its levels and cuts); v = the decoded
 *     direction, alpha = <v, u>, w = |k| r / alpha (0 for a zero key or subspace).
 * A decode step (skv_paris_decode_step) then, per row, with n = the candidate
 * region's length:
 *   - q = the mean of the row's scoring query heads, q_t = R q / |q|;
 *   - collision (§2.3, Eq. (15)): in each subspace the centroids are ranked by
 *     <q_t,s, omega> (ties: lower id); with N = ceil(rho n / 1000) a centroid preceded
 *     by `start` keys (counted over the candidate region) earns 6..1 at the first cut
 *     ceil(P N / 100), P = 5, 15, 30, 50, 75, 100, above start, 0 from N on; a key's S
 *     sums its 16 centroids' weights;
 *   - the ceil(beta n / 1000) keys of largest S (ties: lower position) are candidates;
 *   - rerank (§2.4): s_hat = |q| sum_s w_s <v_s, q_t,s>; the exact top-k of s_hat
 *     (ties: lower position) is the selection, ascending, -1 past its end;
 *   - attention over sink U selection U local as in skv_decode_step (§2.5).
 * ------------------------------------------------------------------------------------ */
typedef struct skv_paris {
  int32_t m;            /* subspace dimension: 8 (the only one built) */
  int32_t beta_pm;      /* candidates, per mille of the candidate region: 1..1000 */
  int32_t rho_pm;       /* keys earning collision weight per subspace, per mille: beta_pm..1000 */
  const int8_t *signs;  /* device int8 [128]: the SRHT's random signs, +1 or -1 */
} skv_paris;

/* Device metadata, rows = batch * n_kv_heads, 16 subspaces, position-major: */
typedef struct skv_paris_index {
  uint8_t *cent;   /* [rows, max_len, 16] centroid ids (16-byte aligned) */
  uint32_t *rec;   /* [rows, max_len, 32] a 128-byte rerank record per key: words 0-15 the
                    * codes of subspaces 0-15 (nibble j = coordinate j), words 16-31 the
                    * fp32 weights of subspaces 0-15 (16-byte aligned) */
  int32_t *hist;   /* [rows, 16, 256] keys per centroid over positions [0, seq_len) */
} skv_paris_index;

/* The 8 levels and 7 cuts (ascending) of the magnitude quantiser for subspace dimension m
 * (3 <= m <= 64), computed on the host by Lloyd's iteration.  Enqueues nothing. */
skv_status skv_paris_quantizer(int32_t m, float *levels, float *thresholds);

/* Encodes positions [0, seq_lens[b]) of every row into *index and sets index->hist
 * (overwritten).  Positions past a row's length are left as they are.  A decode step
 * reads metadata for every position below its own seq_lens: encode with the same
 * lengths (or longer ones) first.  Errors as for skv_decode_step. */
skv_status skv_paris_encode(const skv_problem *p, const skv_paris *paris, const skv_index_src *index,
                            const skv_kv_pool *pool, const skv_paris_index *out, int32_t *dev_status, void *stream);

/* Workspace of skv_paris_decode_step (includes skv_decode_step's attention workspace). */
skv_status skv_paris_workspace_size(const skv_problem *p, const skv_paris *paris, size_t *bytes);

/* Byte offsets, inside that workspace, of the step's intermediates (for inspection):
 * out[0] rotated queries fp32 [rows, 128], [1] |q| fp32 [rows], [2] tier weights u8
 * [rows, 16, 256], [3] collision scores u8 [rows, max_len], [4] candidate counts int32
 * [batch], [5] candidate positions int32 [rows, c_cap], [6] their rerank scores fp32
 * [rows, c_cap]; out[7] = c_cap; [8] the fp32 centroid similarities <q_tilde_b, omega_c>
 * the tiers were ranked by [rows, 16, 256].  out holds 9 entries. */
skv_status skv_paris_workspace_offsets(const skv_problem *p, const skv_paris *paris, int64_t *out);

/* The retrieval alone (no attention): idx [batch, n_kv_heads, topk] receives the
 * selection.  Same arguments and requirements as skv_paris_decode_step, which is this
 * call followed by skv_sparse_attn on the same workspace. */
skv_status skv_paris_select(const skv_problem *p, const skv_paris *paris, const void *q_score,
                            const skv_index_src *index, const skv_paris_index *meta, const skv_kv_pool *pool,
                            int32_t *idx, void *ws, size_t ws_bytes, int32_t *dev_status, void *stream);

/* One decode step with ParisKV retrieval in place of S1/S2: q_score as for
 * skv_decode_step (NULL: q), idx [batch, n_kv_heads, topk] receives the selection.
 * Requirements: bf16, m = 8, retrieval dimension 128 (d_idx for contiguous index keys,
 * d_qk otherwise), batch * n_kv_heads <= 65535, and whatever the attention path
 * requires; else SKV_ERR_UNSUPPORTED. */
skv_status skv_paris_decode_step(const skv_problem *p, const skv_paris *paris, const void *q, const void *q_score,
                                 const skv_index_src *index, const skv_paris_index *meta, const skv_kv_pool *pool,
                                 int32_t *idx, void *out, float *lse, void *ws, size_t ws_bytes,
                                 int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SKV_H */
