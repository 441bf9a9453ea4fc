/*
 * mqatopk: fused FP8 MQA-logits + per-row top-k key selection for the prefill
 * path of a sparse-attention indexer, for one GB300 GPU (sm_103a).
 *
 * Operation (vLLM API page `vllm.model_executor.kernels.attention.dsa.
 * fused_mqa_topk`, `fused_mqa_topk_prefill` docstring; relu form of the score
 * from vLLM pull request #60618, "What this PR does"): for every query row r
 * and every key j in the row's visible range [starts[r], ends[r]),
 *
 *     s(r, j) = key_scales[j] * sum_{h<32} weights[r,h] * relu(q[r,h,:] . k[j,:])
 *
 * with q and k in FP8 e4m3fn (OCP "fn" flavour: bias 7, max 448, no inf) and
 * head dimension 128.  out[r, :] receives the indices of the row's top-k keys
 * relative to starts[r] (key - start), in no particular order, followed by -1
 * when fewer than k keys are visible.  Ties at the k-th score may be broken
 * either way.  The [rows, keys] logits matrix is never materialised.
 *
 * Conventions shared by every entry point
 *  - All tensors are dense, contiguous, row-major, and live in DEVICE memory
 *    of the current CUDA device unless stated otherwise.  The caller owns every
 *    buffer, the workspace and the stream; the library never allocates device
 *    memory and never synchronises a stream except in mqa_topk_get_status.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously on it.
 *  - Return value: MQA_OK (0) or an MQA_ERR_* code.  Argument errors are
 *    detected on the host before any work is enqueued.  Nothing throws.
 *  - q, k, key_scales, weights, out (and logits) must be 16-byte aligned;
 *    starts/ends 4-byte aligned.
 *  - A row whose range is empty or reversed (end <= start) sees no key: its
 *    output is all -1.  A non-empty range that leaves [0, keys) is clamped to
 *    it on the device and MQA_DEV_RANGE_CLAMPED is recorded in the workspace
 *    status word (fused path) or the dense path's status word.
 */
#ifndef MQATOPK_H_
#define MQATOPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MQA_HEADS 32
#define MQA_HEAD_DIM 128
#define MQA_MAX_KEYS (1 << 24)

/* Return codes. */
#define MQA_OK 0
#define MQA_ERR_INVALID_ARGUMENT 1 /* null pointer, bad size, bad topk */
#define MQA_ERR_MISALIGNED 2       /* a pointer breaks the alignment rule */
#define MQA_ERR_WORKSPACE_TOO_SMALL 3
#define MQA_ERR_UNSUPPORTED_DEVICE 4 /* not a compute capability 10.3 device */
#define MQA_ERR_CUDA 5               /* a CUDA runtime/driver call failed */
#define MQA_ERR_NO_DEVICE 6          /* no CUDA device is visible */

/* Device-side status bits (read with mqa_topk_get_status). */
#define MQA_DEV_RANGE_CLAMPED 1 /* some row's range left [0, keys) */
#define MQA_DEV_WAIT_TIMEOUT 2  /* a bounded wait expired: outputs are undefined */
#define MQA_DEV_INTERNAL 4

/* Per-call counters kept in the fused workspace (indices into `stats`). */
#define MQA_STAT_STATUS 0
#define MQA_STAT_ROWS_RESCANNED 1 /* rows recomputed by the exact rescan */
#define MQA_STAT_COMPACTIONS 2    /* exact in-place candidate compactions */
#define MQA_STAT_CANDIDATES 3     /* candidate records written by gated scans */
#define MQA_STAT_GATED_ROWS 4     /* rows scanned behind a sampled gate */
#define MQA_STAT_BLOCKS_DONE 5    /* 8-row blocks finished (scans + rescans) */
#define MQA_STAT_SAMPLE_TILES 6   /* 128-key tiles scored for gate sampling */
#define MQA_STAT_OVERFLOW_ROWS 7  /* gated rows whose candidates overflowed */
#define MQA_STAT_UNDERFILL_ROWS 8 /* gated rows left with fewer than top-k */
#define MQA_STAT_SELECT_FALLBACK 9 /* gated rows whose threshold bin outgrew the
                                      selection warp's shared-memory list and
                                      took the slab-pass radix select */
#define MQA_STAT_KERNEL_US 10     /* first CTA start to last CTA end, microseconds */
#define MQA_STAT_END_SPREAD_US 11 /* first to last CTA end, microseconds (tail) */
#define MQA_STAT_SPLIT_BLOCKS 12  /* blocks whose key range several CTAs scanned
                                     (key chunks merged by the last to finish) */
#define MQA_STAT_UNSAFE_ROWS 13   /* rows whose weights the fold could not serve
                                     within its error bound: rescanned exactly
                                     with the direct head sum */
#define MQA_STAT_FOLD_BOUND_PPM 14 /* largest fold error bound over the rows the
                                      fold served, in millionths of the error a
                                      row allows (2^-16 of its largest |score|);
                                      above 1000000 a row is unsafe */
#define MQA_STAT_PAIR_ROWS 15     /* rows selected by a pair of parked epilogue
                                     warps (few-block calls) */
#define MQA_STAT_SKIPPED_TILES 16 /* masked selection: 128-key tiles left
                                     unscored because no row of the block
                                     allows a key in them */
#define MQA_STATS_COUNT 17

/* Test-only knobs for mqa_topk_prefill_debug.  Zero-initialise for defaults. */
typedef struct mqa_topk_debug_options {
  int force_gate;      /* 0: sampled gate; 1: gate at +inf (every non-empty row
                          under-fills and is rescanned); 2: no gate (rows longer
                          than the slab overflow and are rescanned) */
  int slab_capacity;   /* candidate records per row; 0 = default (13312).  Must
                          be a multiple of 128, at least 4 * (topk + 64), and
                          not above the default (the workspace is sized for it) */
  int stall;           /* nonzero: the producer first waits on a barrier that
                          nothing completes; the time limit ends the wait, the
                          kernel unwinds and MQA_DEV_WAIT_TIMEOUT is recorded */
  int wait_timeout_ms; /* bound on every device-side wait; 0 = default (4000) */
  int max_ctas;        /* persistent CTAs; 0 = one per SM */
  int force_unsafe;    /* 1: every row that the fold would serve is classified
                          unsafe (rescanned exactly with the direct head sum) */
  int head_sum;        /* 32-head key selection only: 0 or 2 the direct head
                          sum (8-row blocks); 1 the relu fold on the tensor
                          core (6-row blocks) */
  int masked_scan;     /* masked selection only: 0 gathers each row's allowed
                          blocks and scores only them; 1 scans every tile of
                          each 8-row block's key range and masks the scores */
} mqa_topk_debug_options;

/* Bytes of workspace one mqa_topk_prefill call over `rows` rows needs on
 * `device` (a CUDA device ordinal).  The size depends on the device's SM count
 * and on min(rows, ...), not on keys (workspace layout: pull request #60618,
 * sections "Memory" and the workspace list of `get_fused_mqa_topk_workspaces`
 * on the API page):
 *  - a 256-byte header (claim counter, status, counters);
 *  - one persistent CTA per SM (at most 32 per block of rows), two slabs of
 *    8 rows x 13312 candidate records (8 B each) per CTA;
 *  - the key-range split arrays: for the blocks whose key range several CTAs
 *    scan as chunks (every block when there are fewer blocks than CTAs, else
 *    the last partial wave of blocks), a slab of 8 rows x (13312 + 512)
 *    records (more per block at 4 or more chunks, for fewer blocks), the
 *    per-chunk segment counts, a finished-chunk counter and a merge row
 *    counter per block.
 * 323.8 MB for 16,384 rows on 152 SMs.
 * A workspace below this size but at least the header plus the per-CTA slabs
 * of min(blocks, SMs) CTAs still works: the call then splits no block. 
 * Returns MQA_ERR_NO_DEVICE / MQA_ERR_CUDA when the device cannot be queried. */
int mqa_topk_workspace_bytes(int device, int rows, size_t *bytes);

/* Fused top-k prefill selection (the operation above), one kernel launch.
 *  q          [rows, 32, 128] uint8 e4m3fn codes
 *  k          [keys, 128] uint8 e4m3fn codes
 *  key_scales [keys] fp32 (see mqa_ue8m0_decode)
 *  weights    [rows, 32] fp32
 *  starts, ends [rows] int32
 *  out        [rows, topk] int32 (written)
 *  rows >= 0 (0 is a no-op), 1 <= keys <= MQA_MAX_KEYS, topk in {512, 1024, 2048}
 *  workspace  device buffer of at least mqa_topk_workspace_bytes(dev, rows)
 *             bytes, 256-byte aligned; its header is reset on `stream` by
 *             every call, so it may be reused by consecutive calls on one
 *             stream but not by calls that overlap in time.
 * The result is exact up to ties at the k-th score: a sampled per-row gate
 * filters candidates, and any row the gate cannot serve (too many or too few
 * candidates) is rescanned exactly.
 * The call only enqueues work on `stream` (a memset of the workspace header
 * and one kernel launch), so it may be captured into a CUDA graph once a call
 * outside the capture has run on the device; replays read the buffers'
 * current contents. */
int mqa_topk_prefill(const void *q, const void *k, const float *key_scales, const float *weights,
                     const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys, int topk,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes for mqa_topk_prefill_ex with `heads` index heads (32 or
 * 64) per query row.  Same contents as mqa_topk_workspace_bytes; with 64 heads
 * a block holds 4 rows instead of 8. */
int mqa_topk_workspace_bytes_ex(int device, int rows, int heads, size_t *bytes);

/* mqa_topk_prefill for 32 or 64 index heads per query row (the pages list
 * DeepSeek-V3.2's 64 index heads as not yet supported by their kernel: PR
 * #60618, section "Limitations of this PR -- TODOs").  q is [rows, heads, 128] uint8 e4m3fn, weights
 * [rows, heads] fp32; everything else as mqa_topk_prefill.  A 256-column
 * accumulator tile holds 8 rows of 32 heads or 4 rows of 64, so the kernel is
 * compiled once per head count.  opt (nullable) carries the test-only knobs of
 * mqa_topk_prefill_debug.  heads other than 32 or 64: MQA_ERR_INVALID_ARGUMENT. */
int mqa_topk_prefill_ex(const void *q, const void *k, const float *key_scales, const float *weights,
                        const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys, int topk,
                        int heads, void *workspace, size_t workspace_bytes, void *stream,
                        const mqa_topk_debug_options *opt);

/* Block selection, the first half of the pages' two-level candidate selection
 * (PR #60618, "Limitations of this PR -- TODOs": a candidate-source layer also
 * writes, per row, the top 2,048 blocks of 8 keys ranked by their maximum
 * score).  Block b holds keys [8b, 8b + 8) of k; its score is the largest
 * s(r, j) over the row's visible keys in it.  out_blocks [rows, btopk] int32
 * receives the btopk best blocks of each row as b - floor(starts[r] / 8),
 * unordered, -1 padded when the row's range touches fewer blocks; ties at the
 * btopk-th score are taken in any order.  btopk in {512, 1024, 2048}; 32
 * heads; workspace as for mqa_topk_prefill (mqa_topk_workspace_bytes); opt
 * (nullable) as for mqa_topk_prefill_debug.  Same errors as mqa_topk_prefill. */
int mqa_block_topk_prefill(const void *q, const void *k, const float *key_scales, const float *weights,
                           const int32_t *starts, const int32_t *ends, int32_t *out_blocks, int rows, int keys,
                           int btopk, void *workspace, size_t workspace_bytes, void *stream,
                           const mqa_topk_debug_options *opt);

/* Masked selection, the consumer half of the two-level candidate selection
 * (PR #60618, "Limitations of this PR -- TODOs": consumer layers mask their
 * scores to the source layer's blocks before their top-k).  As
 * mqa_topk_prefill, but key j of row r is visible only if it lies in
 * [starts[r], ends[r]) and bit (j / 8) % 32 of word j / 256 of mask row r is
 * set.
 *  mask       [rows, mask_words] uint32, 16-byte aligned; mask_words a multiple
 *             of 4 and >= ceil(keys / 256)
 *  row_items  [rows] int32: the number of visible keys of each row (it sizes
 *             the row's sampled gate in the scan of opt->masked_scan = 1;
 *             the default path reads the mask alone); mqa_block_mask writes it
 * By default each row's allowed blocks are gathered from k and only their
 * keys are scored (the page's remark that scoring only the candidate blocks
 * speeds the consumers up): the workspace needs only the 256-byte header,
 * the cost follows the allowed keys, and the statistics count rows finished
 * (MQA_STAT_BLOCKS_DONE) and visible keys scored (MQA_STAT_CANDIDATES).  With
 * opt->masked_scan = 1 the fused scan of mqa_topk_prefill runs instead over
 * every tile of each 8-row block's range (tiles no row of the block allows
 * are left out, MQA_STAT_SKIPPED_TILES) with the full workspace.
 * 32 heads; workspace as for mqa_topk_prefill (header only by default). */
int mqa_topk_prefill_masked(const void *q, const void *k, const float *key_scales, const float *weights,
                            const int32_t *starts, const int32_t *ends, const uint32_t *mask, int mask_words,
                            const int32_t *row_items, int32_t *out, int rows, int keys, int topk, void *workspace,
                            size_t workspace_bytes, void *stream, const mqa_topk_debug_options *opt);

/* Build the block mask of mqa_topk_prefill_masked from per-row block lists
 * (block_lists [rows, list_len] int32, entries relative to floor(starts[r] /
 * 8) as mqa_block_topk_prefill writes them, -1 or out-of-range entries
 * ignored), and count each row's visible keys into row_items [rows].  One
 * launch on `stream`; mask and row_items are overwritten. */
int mqa_block_mask(const int32_t *block_lists, const int32_t *starts, const int32_t *ends, int rows, int list_len,
                   int keys, uint32_t *mask, int mask_words, int32_t *row_items, void *stream);

/* mqa_topk_prefill with test-only knobs (opt may be NULL). */
int mqa_topk_prefill_debug(const void *q, const void *k, const float *key_scales, const float *weights,
                           const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys,
                           int topk, void *workspace, size_t workspace_bytes, void *stream,
                           const mqa_topk_debug_options *opt);

/* Allocation-free variant of mqa_topk_prefill (the pages have no counterpart;
 * it exists for callers that cannot allocate device memory: code that runs
 * while a stream is being captured into a CUDA graph in global capture mode,
 * where cudaMalloc is not permitted; plugins whose host framework owns the
 * whole device memory pool; latency-critical paths that must never wait on an
 * allocator).  Same inputs, output and result as mqa_topk_prefill, but no
 * workspace argument: the scratch is a static device array inside the library
 * of 256 B + 8 CTAs x 2 slots x 8 rows x 13312 records x 8 B (13 MiB + 256 B),
 * held by every GPU that loads the library until the process exits.  The call
 * therefore runs on at most 8 persistent CTAs (slower than mqa_topk_prefill on
 * big chunks).  Its scratch need does not grow with rows or keys, so every
 * call that passes the argument checks fits; a need beyond the array would be
 * rejected with MQA_ERR_WORKSPACE_TOO_SMALL.  It calls no cudaMalloc/cudaFree.
 *  - The first call on each device resolves the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture begins.
 *  - Every call shares the one array and resets its header on `stream`.
 *    Calls that overlap on the GPU (other streams, other host threads) race
 *    on the scratch and give wrong results: serialise them.
 *  - Device status and counters: mqa_topk_noalloc_get_status. */
int mqa_topk_prefill_noalloc(const void *q, const void *k, const float *key_scales, const float *weights,
                             const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys,
                             int topk, void *stream);

/* Status word and counters of the last mqa_topk_prefill_noalloc call on the
 * current device, as mqa_topk_get_status reads them from a workspace (the
 * pages have no counterpart).  A status with MQA_DEV_WAIT_TIMEOUT means that
 * call's output is undefined.  Synchronises `stream`; status (host) receives
 * the MQA_DEV_* bits, stats (host, nullable) MQA_STATS_COUNT counters. */
int mqa_topk_noalloc_get_status(int32_t *status, int32_t *stats, void *stream);

/* UE8M0 -> fp32 key-scale decode (API page, `fused_mqa_topk_key_scales`
 * docstring): scales is [keys, 4] uint8 whose first byte per key is the
 * exponent e; out[j] is the fp32 with bit pattern e << 23 (2^(e-127) for
 * 1 <= e <= 254).  keys >= 0. */
int mqa_ue8m0_decode(const uint8_t *scales, float *out, int keys, void *stream);

/* Fold preparation (vLLM pull request #60618, "What this PR does", Scoring
 * bullet: since relu(s) = (s + |s|) / 2, the heads' weighted linear halves
 * sum to one folded query v = sum_h w_h q_h times the key).  Per row:
 *  - v[d] in fp32, one fused multiply-add per head in head order;
 *  - MQA_FOLD_TERMS e4m3 terms with power-of-two scales: term t has exponent
 *    e_t, the smallest integer with max_d |r_t[d]| * 2^-e_t <= 448 (0 for a
 *    zero residual), codes u_t = e4m3 round-to-nearest-even of r_t * 2^-e_t,
 *    and r_{t+1} = r_t - 2^e_t E(u_t) (r_0 = v);
 *  - beta = |r_T|_2, so |v . k - sum_t 2^e_t E(u_t) . k| <= beta |k|_2.
 *  q       [rows, 32, 128] uint8 e4m3fn codes, 16-byte aligned
 *  weights [rows, 32] fp32
 *  codes   [rows, MQA_FOLD_TERMS, 128] uint8 (written), 16-byte aligned
 *  exps    [rows, MQA_FOLD_TERMS] int32 (written)
 *  beta    [rows] fp32 (written)
 * rows >= 0 (0 is a no-op).  The fold compilation of the fused kernel
 * (mqa_topk_prefill_debug / _ex with head_sum = 1) computes the same terms in
 * its per-call preparation and runs them as extra accumulator columns; it
 * classifies a row as unsafe, and rescans it exactly with the direct head
 * sum, when beta times the largest key_scale * |k|_2 over the keys could move
 * a score by more than 2^-16 of the row's largest |score| (MQA_STAT_UNSAFE_ROWS,
 * MQA_STAT_FOLD_BOUND_PPM). */
#define MQA_FOLD_TERMS 4
int mqa_fold_prep(const void *q, const float *weights, uint8_t *codes, int32_t *exps, float *beta, int rows,
                  void *stream);

/* Debug: the scores themselves.  logits is [rows, keys] fp32, row-major;
 * s(r, j) for keys in [starts[r], ends[r]) and -inf elsewhere.  Same inputs
 * and limits as mqa_topk_prefill (topk unused); computed by the same tensor-
 * core pipeline and score arithmetic as the fused path.  Needs no workspace
 * beyond a 256-byte device header passed as `workspace` (counters/status). */
int mqa_logits_debug(const void *q, const void *k, const float *key_scales, const float *weights,
                     const int32_t *starts, const int32_t *ends, float *logits, int rows, int keys,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Comparison baseline (dense path): materialise fp32 logits for as many rows
 * as fit in logits_ws (logits_budget_bytes / (keys * 4) rows per call, as the
 * dense path chunks under its logits budget in pull request #60618,
 * "Motivation"), then select each row's top-k from them.  Same inputs and
 * output convention as mqa_topk_prefill; `workspace` is a 256-byte header as
 * for mqa_logits_debug.  logits_budget_bytes must hold at least one row. */
/* Device staging bytes for mqa_topk_prefill_host with these sizes on `device`:
 * the inputs, the decoded scales, the output and the fused op's workspace. */
int mqa_topk_host_staging_bytes(int device, int rows, int keys, int topk, size_t *bytes);

/* The fused op from host buffers (32 heads): copies q, k, the UE8M0 scale
 * bytes ([keys, 4]), weights, starts and ends host -> device into `staging`
 * (device, 256-byte aligned, mqa_topk_host_staging_bytes long), decodes the
 * scales, runs mqa_topk_prefill and copies the indices device -> host into
 * out_host [rows, topk].  Host buffers as the device-buffer entry lays them
 * out.  Everything is enqueued on `stream` with one plain asynchronous copy
 * per buffer: with pinned host memory the copies overlap other streams'
 * work, and out_host holds the result once the stream has reached this
 * point (the call itself does not synchronise).  The status word and
 * counters of the call: mqa_topk_host_get_status.  The pages have no
 * host-buffer entry: it is the end-to-end form of mqa_topk_prefill. */
int mqa_topk_prefill_host(const void *q_host, const void *k_host, const uint8_t *scales_ue8m0_host,
                          const float *weights_host, const int32_t *starts_host, const int32_t *ends_host,
                          int32_t *out_host, int rows, int keys, int topk, void *staging, size_t staging_bytes,
                          void *stream);

/* mqa_topk_get_status for the workspace inside a staging buffer of
 * mqa_topk_prefill_host (the same rows, keys and topk). */
int mqa_topk_host_get_status(const void *staging, int rows, int keys, int topk, int32_t *status, int32_t *stats,
                             void *stream);

/* Measurement helper with no counterpart in the method: one CTA per SM issues
 * tiles_per_sm back-to-back 128 x 256 x 128 FP8 MMA tiles (e4m3 inputs, fp32
 * accumulation in TMEM, the fused kernel's tile shape) from fixed shared-memory
 * operands, no loads and no epilogue.  The FLOPs it does are sms * tiles_per_sm
 * * 2 * 128 * 256 * 128; timing the launch on `stream` gives the tensor pipe's
 * FP8 ceiling at the clocks the GPU holds.  status (device, int32, zeroed by
 * the caller) receives MQA_DEV_WAIT_TIMEOUT if the final wait ran out.
 * tiles_per_sm in [1, 2^26]. */
int mqa_fp8_mma_probe(long long tiles_per_sm, int32_t *status, void *stream);

int mqa_topk_dense_baseline(const void *q, const void *k, const float *key_scales, const float *weights,
                            const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys,
                            int topk, void *logits_ws, size_t logits_budget_bytes, void *workspace,
                            size_t workspace_bytes, void *stream);

/* Read the status word and counters of the last call that used `workspace`.
 * Synchronises `stream`.  status (host) receives the MQA_DEV_* bits; stats
 * (host, nullable) receives MQA_STATS_COUNT int32 counters. */
int mqa_topk_get_status(const void *workspace, int32_t *status, int32_t *stats, void *stream);

/* Static description of a return code. */
const char *mqa_topk_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MQATOPK_H_ */
