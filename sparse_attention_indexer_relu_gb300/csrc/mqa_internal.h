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
// 64.  Host code is compiled for 32 and passes the block rows it needs.
#ifndef MQA_HEADS
#define MQA_HEADS 32
#endif
constexpr int kHeads = MQA_HEADS;  // index heads per query row
static_assert(kHeads == 32 || kHeads == 64, "index heads: 32 or 64");
constexpr int kDim = 128;       // head dimension (bytes per fp8 row)
constexpr int kBlockRows = 256 / kHeads;  // query rows per block (one TMEM accumulator group)
constexpr int kTileKeys = 128;  // keys per tile (UMMA M, one TMEM lane per key)
constexpr int kCols = kBlockRows * kHeads;  // 256 accumulator columns per tile (UMMA N)
constexpr int kKStages = 6;     // K-tile ring depth
constexpr int kSStages = 8;     // key-scale ring depth (held until the epilogue has read them)
constexpr int kQBytes = kCols * kDim;       // 32 KiB of q per block
constexpr int kKTileBytes = kTileKeys * kDim;  // 16 KiB of k per tile

#ifndef MQA_ROWS_PER_WARP
#define MQA_ROWS_PER_WARP (256 / MQA_HEADS / 4)
#endif
constexpr int kRowsPerWarp = MQA_ROWS_PER_WARP;  // rows of a block each epilogue warp scores
constexpr int kQuadsC = 4;
constexpr int kEpiWarps = kBlockRows * kQuadsC / kRowsPerWarp;  // per TMEM lane quadrant: 8 / kRowsPerWarp
constexpr int kSelWarps = 2;    // candidate selection warps
constexpr int kThreads = (4 + kEpiWarps) * 32;  // warp 0 producer, 1 MMA, 2-3 selection, then epilogue
constexpr int kEpiWarp0 = 4;
constexpr int kSelWarp0 = 2;
constexpr int kQuads = 4;       // TMEM lane quadrants; each row's slab has one segment per quadrant

constexpr int kDefaultSlabCap = 16384;  // candidate records per row per slot (4 segments)
constexpr int kSlots = 2;               // slab slots per CTA (scan one, select the other)
constexpr int kMaxSortBlocks = 8192;    // heaviest-first order kept in smem up to this many blocks
constexpr int kMaxKeys = 1 << 24;

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
  int split_max;         // split blocks the arrays above hold
  long long split_words; // uint32 words of split_slab
  const int32_t *row_items;  // masked selection: allowed keys per row
  int rows;              // rows of this call
  int row0;              // first global row (logits mode: chunk offset)
  int keys;
  int topk;
  int nblocks;
  int cap;               // slab capacity per row
  int gate_target;       // expected candidates per gated row
  int gate_min;          // rows seeing more keys than this are gated (2 x gate_target)
  int force_gate;        // 0 normal, 1 gate +inf, 2 gate -inf
  int stall;             // debug: wait on a barrier nobody arrives on
  int key_chunks;        // logits mode: key chunks per block
  long long timeout_ns;  // bound on every wait
};

// Launchers (defined next to their kernels), per head count.
namespace h32 {
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *m_map = nullptr);
cudaError_t launch_logits(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                          const FusedParams &p, int ctas, cudaStream_t stream);
}  // namespace h32
namespace h64 {
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *m_map = nullptr);
}  // namespace h64
namespace h32b {  // block selection: top blocks of 8 keys by their largest score
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *m_map = nullptr);
}  // namespace h32b
namespace h32p {  // key selection whose parked epilogue warps select rows in pairs (few-block calls)
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *m_map = nullptr);
}  // namespace h32p
namespace h32m {  // masked selection: keys restricted to a per-row block mask
cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *m_map = nullptr);
}  // namespace h32m
cudaError_t launch_block_mask(const int32_t *lists, const int32_t *starts, const int32_t *ends, int rows,
                              int list_len, int keys, uint32_t *mask, int mask_words, int32_t *row_items,
                              cudaStream_t stream);
cudaError_t launch_ue8m0_decode(const uint8_t *scales, float *out, int keys, cudaStream_t stream);
cudaError_t launch_dense_topk_rows(const float *logits, int rows, int keys, const int32_t *starts,
                                   const int32_t *ends, int32_t *out, int topk, int32_t *ws_status,
                                   cudaStream_t stream);

// Fused-op workspace layout: header, split-done counters, per-CTA slabs, split
// slab, split counts (split_max == 0: header and slabs only).
struct FusedLayout {
  size_t done_off, slab_off, split_off, cnt_off, reset_bytes, total;
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
FusedLayout fused_layout(int ctas, int cap, int split_max, int block_rows);

// Allocation-free variant: a static device scratch sized for this many CTAs.
constexpr int kStaticScratchCtas = 8;
constexpr size_t kStaticScratchBytes =
    kWsHeaderBytes + (size_t)kStaticScratchCtas * kSlots * 2 * 8 * kDefaultSlabCap * sizeof(uint32_t);  // 8-row blocks
// Device address of the static scratch on the current device (resolved on first use).
cudaError_t static_scratch_address(void **ptr);

}  // namespace mqa
