// Internal definitions shared by the library's translation units (not part of
// the public C ABI in include/mqatopk.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mqa {

// The fused kernel is compiled once per supported head count (MQA_HEADS 32
// or 64); a 256-column accumulator tile holds 8 rows of 32 heads or 4 rows of
// 64.  The fold compilation (MQA_FOLD, 32 heads) scores 6-row blocks whose
// tile also carries each row's folded query as 4 e4m3 terms: 6 x 32 head
// columns plus 32 fold columns (24 used), so that two tiles fit the 512 TMEM
// columns.  Host code is compiled with the defaults and passes the block rows
// it needs.
#ifndef MQA_HEADS
#define MQA_HEADS 32
#endif
#ifndef MQA_FOLD
#define MQA_FOLD 0
#endif
constexpr int kHeads = MQA_HEADS;  // index heads per query row
static_assert(kHeads == 32 || kHeads == 64, "index heads: 32 or 64");
constexpr bool kFold = MQA_FOLD != 0;  // weighted linear half of relu on the tensor core
static_assert(!kFold || kHeads == 32, "the fold compilation is built for 32 heads");
constexpr int kDim = 128;       // head dimension (bytes per fp8 row)
constexpr int kFoldRowTerms = 4;  // e4m3 terms of a row's folded query
constexpr int kBlockRows = kFold ? 6 : 256 / kHeads;  // query rows per block
constexpr int kTileKeys = 128;  // keys per tile (UMMA M, one TMEM lane per key)
constexpr int kHeadCols = kBlockRows * kHeads;  // head accumulator columns per tile
// fold accumulator columns per tile: the block's rows x 4 terms, padded to
// the UMMA N granule of 16 (the padding columns are never read)
constexpr int kFoldCols = kFold ? (kBlockRows * kFoldRowTerms + 15) / 16 * 16 : 0;
constexpr int kCols = kHeadCols + kFoldCols;  // UMMA N: 256, or 224 with the fold
constexpr int kTmemBufs = 2;                  // accumulator buffers in TMEM
constexpr int kTmemStride = kCols;            // columns between buffers (a multiple of 32)
static_assert(kTmemBufs * kTmemStride <= 512 && kTmemStride % 32 == 0, "TMEM holds 512 columns");
constexpr int kKStages = 6;     // K-tile ring depth
constexpr int kSStages = 8;     // key-scale ring depth (held until the epilogue has read them)
constexpr int kQBytes = kCols * kDim;       // q (and fold terms) per block: 32 or 28 KiB
constexpr int kKTileBytes = kTileKeys * kDim;  // 16 KiB of k per tile

#ifndef MQA_ROWS_PER_WARP
#define MQA_ROWS_PER_WARP (kFold ? 2 : kBlockRows / 4)
#endif
constexpr int kRowsPerWarp = MQA_ROWS_PER_WARP;  // rows of a block each epilogue warp scores
constexpr int kQuadsC = 4;
constexpr int kEpiWarps = kBlockRows * kQuadsC / kRowsPerWarp;  // per TMEM lane quadrant: kBlockRows / kRowsPerWarp
constexpr int kSelWarps = 2;    // candidate selection warps
constexpr int kThreads = (4 + kEpiWarps) * 32;  // warp 0 producer, 1 MMA, 2-3 selection, then epilogue
constexpr int kEpiWarp0 = 4;
constexpr int kSelWarp0 = 2;
constexpr int kQuads = 4;       // TMEM lane quadrants; each row's slab has one segment per quadrant

constexpr int kDefaultSlabCap = 13312;  // candidate records per row per slot (4 segments)
constexpr int kSlots = 2;               // slab slots per CTA (scan one, select the other)
constexpr int kMaxSortBlocks = 8192;    // heaviest-first order kept in smem up to this many blocks
constexpr int kMaxKeys = 1 << 24;
// Block rows of the fold compilation and the rows of its fold-term TMA box
// (the block's 24 term rows plus 8 of the next block's, which fill the
// padding columns), for host code (compiled with the defaults).
constexpr int kFoldBlockRows = 6;
constexpr int kFoldBoxRows = 32;

constexpr int kSampleBins = 160;        // 129 used, padded for the warp scan

// Workspace header (int32 words), zeroed by the host before each launch.
enum WsWord : int {
  kWsClaim = 0,          // next entry of the heaviest-first block order
  kWsStatus = 1,         // device status bits (MQA_DEV_*)
  kWsRowsRescanned = 2,  // rows that took the exact rescan
  kWsCompactions = 3,    // in-place slab compactions
  kWsCandidates = 4,     // candidate records written by gated scans (sum over rows)
  kWsGatedRows = 5,      // rows that used a sampled gate
  kWsBlocksDone = 6,     // row blocks whose scan finished
  kWsSampleTiles = 7,    // sample tiles scored
  kWsOverflowRows = 8,   // rows whose candidates exceeded the slab
  kWsUnderfillRows = 9,  // rows whose gated count fell below top-k
  kWsSelFallback = 10,   // gated rows selected by the slab-pass radix path
  kWsSplitBlocks = 11,   // blocks whose key range was split across CTAs
  // 64-bit globaltimer stamps (word pairs, 8-byte aligned); minima are kept
  // as UINT64_MAX - t so that every stamp is an atomicMax on a zeroed word
  kWsTStartMinInv = 12,  // first CTA start
  kWsTEndMinInv = 14,    // first CTA end
  kWsTEndMax = 16,       // last CTA end
  kWsKeyNorm = 18,       // fold: largest key_scale * |k|_2 over the keys (fp32 bits, rounded up)
  kWsUnsafeRows = 19,    // fold: rows whose fold error bound was too large (rescanned exactly)
  kWsFoldBound = 20,     // fold: largest error bound over classified rows, ppm of the allowed error
  kWsPairRows = 21,      // rows selected by a pair of parked epilogue warps
  kWsSkippedTiles = 22,  // masked selection: tiles left out (no allowed key in any of the block's rows)
  kWsWords = 64
};
constexpr size_t kWsHeaderBytes = 256;

// Device status bits.
constexpr int kDevRangeClamped = 1;
constexpr int kDevWaitTimeout = 2;
constexpr int kDevInternal = 4;

struct FusedParams {
  const float *scales;   // [keys] fp32
  const float *weights;  // [rows, 32]
  const int32_t *starts; // [rows]
  const int32_t *ends;   // [rows]
  int32_t *out;          // [rows, topk]   (top-k mode)
  float *logits;         // [rows, keys]   (logits mode, row-chunk local)
  int32_t *ws;           // workspace header (int32 words)
  uint32_t *slab;        // slabs: [ctas][slots][rows 8][cap] keys, then same for indices
  // Key-range split of the last blocks in claim order (disabled when split_max == 0):
  uint32_t *split_slab;  // per split block: [rows 8][row capacity] keys, then same for indices
  int32_t *split_cnt;    // per split block: [rows 8][32] records per (chunk, quadrant) segment
  int32_t *split_done;   // per split block: chunks finished (zeroed with the header)
  int32_t *merge_next;   // per split block: next row claimed in a spread merge (zeroed with the header)
  int split_max;         // split blocks the arrays above hold
  long long split_words; // uint32 words of split_slab
  const int32_t *row_items;  // masked selection: allowed keys per row
  const uint32_t *mask;      // masked selection: [rows, mask_words] block-mask words
  int mask_words;
  const int32_t *fold_exps;  // fold: [rows, 4] power-of-two exponents of the folded query's terms
  const float *fold_beta;    // fold: [rows] 2-norm of the folded query's residual
  int rows;              // rows of this call
  int row0;              // first global row (logits mode: chunk offset)
  int keys;
  int topk;
  int nblocks;
  int cap;               // slab capacity per row
  int gate_target;       // expected candidates per gated row
  int gate_min;          // rows seeing more keys than this are gated (2 x gate_target)
  int force_gate;        // 0 normal, 1 gate +inf, 2 gate -inf
  int force_unsafe;      // debug (fold): classify every row that needs the fold as unsafe
  int stall;             // debug: wait on a barrier nobody arrives on
  int key_chunks;        // logits mode: key chunks per block
  long long timeout_ns;  // bound on every wait
};

// Launchers (defined next to their kernels), per compilation.  x_map is the
// extra tensor map a compilation reads: the per-row block mask (masked
// selection) or the folded queries' e4m3 terms (fold); the others ignore it.
namespace h32f {  // key selection with the relu fold on the tensor core (4-row blocks)
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *x_map = nullptr);
}  // namespace h32f
namespace h64 {
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *x_map = nullptr);
}  // namespace h64
namespace h32b {  // block selection: top blocks of 8 keys by their largest score
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *x_map = nullptr);
}  // namespace h32b
namespace h32 {  // key selection, 8-row blocks, the direct head sum
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *x_map = nullptr);
}  // namespace h32
namespace h32p {  // key selection whose parked epilogue warps select rows in pairs (few-block calls)
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *x_map = nullptr);
// the scores themselves from the same pipeline with the direct head sum
cudaError_t launch_logits(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                          const FusedParams &p, int ctas, cudaStream_t stream);
}  // namespace h32p
namespace h32m {  // masked selection: keys restricted to a per-row block mask
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *x_map = nullptr);
}  // namespace h32m
// Masked selection that gathers each row's allowed blocks and scores only
// them (32 heads): one persistent CTA per SM, rows claimed through the
// header's claim word.  q_map: q as [rows * 32, 128] in boxes of 32 rows.
struct GatherParams {
  const uint8_t *k;       // [keys, 128] e4m3 codes, 16-byte aligned
  const float *scales;    // [keys] fp32
  const float *weights;   // [rows, 32]
  const int32_t *starts;  // [rows]
  const int32_t *ends;    // [rows]
  const uint32_t *mask;   // [rows, mask_words] block-mask words
  int mask_words;
  int32_t *out;           // [rows, topk]
  int32_t *ws;            // workspace header (int32 words)
  int rows, keys, topk;
  int stall;              // debug: wait on a barrier nobody arrives on
  long long timeout_ns;   // bound on every wait
};
size_t gather_smem_bytes();
cudaError_t launch_gather_masked(const CUtensorMap &q_map, const GatherParams &p, int ctas, cudaStream_t stream);
// FP8 tensor-pipe probe: one CTA per SM issuing `tiles` back-to-back
// 128 x 256 x 128 MMA tiles; a wait past its bound sets *status bits.
cudaError_t launch_fp8_mma_probe(long long tiles, int32_t *status, cudaStream_t stream);
cudaError_t launch_block_mask(const int32_t *lists, const int32_t *starts, const int32_t *ends, int rows,
                              int list_len, int keys, uint32_t *mask, int mask_words, int32_t *row_items,
                              cudaStream_t stream);
// Per-call preparation of the fold compilation (one launch): each row's folded
// query as 4 e4m3 terms with exponents and residual norm, and the largest
// key_scale * |k|_2 over the keys into *key_norm (fp32 bits, atomic max on a
// zeroed word).
cudaError_t launch_fold_call_prep(const uint8_t *q, const float *w, const uint8_t *k, const float *scales,
                                  uint8_t *codes, int32_t *exps, float *beta, int rows, int keys,
                                  int32_t *key_norm, cudaStream_t stream);
cudaError_t launch_ue8m0_decode(const uint8_t *scales, float *out, int keys, cudaStream_t stream);
cudaError_t launch_dense_topk_rows(const float *logits, int rows, int keys, const int32_t *starts,
                                   const int32_t *ends, int32_t *out, int topk, int32_t *ws_status,
                                   cudaStream_t stream);

// Fused-op workspace layout: header, split-done counters, per-CTA slabs, split
// slab, split counts (split_max == 0: header and slabs only).
struct FusedLayout {
  size_t done_off, slab_off, split_off, cnt_off, reset_bytes, total;
  size_t fold_codes_off, fold_exps_off, fold_beta_off;  // fold compilation only (fold_rows > 0)
  long long split_words;
};
constexpr int kMaxChunks = 32;  // key chunks a split block is cut into (a power of two)
// Records per row a split block needs at `chunks` chunks: 4 * chunks
// segments of max(cap / (4 chunks) + 64, cap / 8) records, so that one chunk
// can hold a row's whole gated candidate set (at most cap / 2).
__host__ __device__ inline long long split_row_capacity(int cap, int chunks) {
  const long long a = cap / (4 * chunks) + 64, b = cap / 8;
  return 4LL * chunks * (a > b ? a : b);
}
FusedLayout fused_layout(int ctas, int cap, int split_max, int block_rows, int fold_rows = 0);

// Allocation-free variant: a static device scratch sized for this many CTAs.
constexpr int kStaticScratchCtas = 8;
constexpr size_t kStaticScratchBytes =
    kWsHeaderBytes + (size_t)kStaticScratchCtas * kSlots * 2 * 8 * kDefaultSlabCap * sizeof(uint32_t);  // 8-row blocks
// Device address of the static scratch on the current device (resolved on first use).
cudaError_t static_scratch_address(void **ptr);

}  // namespace mqa
