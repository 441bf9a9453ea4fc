// Fused FP8 MQA-logits + per-row top-k for sm_103a (one persistent CTA per SM).
//
// What it computes (vLLM API page `vllm.model_executor.kernels.attention.dsa.
// fused_mqa_topk`, `fused_mqa_topk_prefill` docstring; vLLM pull request
// #60618, "What this PR does"): for each query row r and visible key j in
// [start_r, end_r),
//     s(r, j) = scale_j * sum_h w[r,h] * relu(q[r,h,:] . k[j,:])
// with 32 heads of dimension 128 in FP8 e4m3, and the row's top-k keys as
// indices relative to start_r (unordered, -1 padded).  The [rows, keys]
// logits matrix never reaches HBM.  A second instantiation of the same
// pipeline writes the logits instead (debug entry and dense baseline).
//
// CTA layout (640 threads with 32 index heads):
//   warp 0      producer: claims row blocks heaviest first (or key chunks of
//               the last blocks), loads q (TMA) and per-row ranges/weights,
//               streams 128-key K tiles (TMA) through a 6-stage ring and the
//               tiles' key scales through an 8-stage ring.
//   warp 1      MMA issuer: per K tile, 4 x tcgen05.mma kind::f8f6f4
//               (M = 128 keys, N = 8 rows x 32 heads, K = 32) into one of two
//               256-column TMEM accumulators.
//   warps 2-3   selection: per finished block, each row's top-k from its
//               candidates (score-binned count and gather, exact radix over
//               the threshold bin), output write or rescan request.
//   warps 4-19  epilogue: warp w reads TMEM lane quadrant w % 4 (32 keys) for
//               2 of the block's rows (16x256b loads: 4 keys x 8 heads per
//               thread), relu-weighted head sum, 4-lane reduce-scatter, key
//               scale, range mask; sampled gate; candidate emission to
//               per-(row, quadrant) slab segments; exact compaction on
//               rescans; selection help once the producer has no block left.
// The same source is compiled for 64 index heads (4-row blocks), for block
// selection (the top blocks of 8 keys), for masked selection (keys limited to
// a per-row block mask) and, for calls with few blocks, with the parked
// epilogue warps selecting each row in pairs.
// Every wait is bounded by a time limit; on expiry the kernel records
// MQA_DEV_WAIT_TIMEOUT in the workspace status word and unwinds.
#include "mqa_internal.h"
#include "ptx.cuh"

#include <cfloat>
#include <climits>
#include <mutex>

#ifndef MQA_BLOCKS
#define MQA_BLOCKS 0
#endif
#ifndef MQA_MASKED
#define MQA_MASKED 0
#endif
#ifndef MQA_PAIR_HELPERS
#define MQA_PAIR_HELPERS 0
#endif
#if MQA_FOLD
#define MQA_KNS h32f
static_assert(MQA_HEADS == 32 && !MQA_BLOCKS && !MQA_MASKED && !MQA_PAIR_HELPERS,
              "the fold build is the 32-head key selection");
#elif MQA_PAIR_HELPERS
#define MQA_KNS h32p
static_assert(MQA_HEADS == 32 && !MQA_BLOCKS && !MQA_MASKED, "the pair-helper build is the 32-head key selection");
#elif MQA_BLOCKS
#define MQA_KNS h32b
static_assert(MQA_HEADS == 32 && !MQA_MASKED, "block selection is built for 32 heads");
#elif MQA_MASKED
#define MQA_KNS h32m
static_assert(MQA_HEADS == 32, "masked selection is built for 32 heads");
#elif MQA_HEADS == 64
#define MQA_KNS h64
#else
#define MQA_KNS h32
#endif

namespace mqa {
namespace MQA_KNS {

// The gate's sample tiles are scored once in the 32-head key and block
// selection compilations (8-row, pair-helper and block: the scores are kept in
// the job's slab slot for the gate's two histogram passes) and twice in the
// others (a coarse pass, then a fine pass that scores them again).  Scoring
// once shortened decode batches by 3-6% and, with the scan loop of gated jobs
// kept free of the rescan code, the 1M-key chunk by 3.3% and the 1M-key block
// selection by 0.7%.
#ifndef MQA_SAMPLE_ONCE
#if MQA_HEADS == 32 && !MQA_MASKED && !MQA_FOLD
#define MQA_SAMPLE_ONCE 1
#else
#define MQA_SAMPLE_ONCE 0
#endif
#endif
// Gated scans skip the per-row ballots of a tile in which no key of the
// warp's rows passes the gate (one vote over both rows).  That measured 2%
// faster at 1M keys in the 8-row compilation and 1.5% slower on decode
// batches in the pair-helper compilation, which leaves it out.
#ifndef MQA_ANY_GATE
#define MQA_ANY_GATE (!MQA_PAIR_HELPERS)
#endif
constexpr bool kAnyGate = MQA_ANY_GATE;
constexpr int kSamplePasses = MQA_SAMPLE_ONCE ? 1 : 2;  // times each sample tile is scored
constexpr uint32_t kIdesc = idesc_f8_e4m3_f32(kTileKeys, kCols);
constexpr uint32_t kTmemAllocCols = 512;  // a power of two holding every accumulator buffer


// Selection items: keys, or (block selection) blocks of 8 keys ranked by
// their largest score.  A block b holds keys [8b, 8b + 8) of the key array.
constexpr bool kBlocks = MQA_BLOCKS != 0;
// Masked selection: a key is visible only if its block of 8 is set in the
// row's block mask (bit (j / 8) % 32 of word j / 256).
constexpr bool kMasked = MQA_MASKED != 0;
constexpr int kSkipTiles = 8192;  // masked selection: longest tile range the skip bitmap covers
// Items a row with visible keys [s, e) selects from.
__host__ __device__ __forceinline__ int row_items(int s, int e) {
  if (e <= s) return 0;
  return kBlocks ? ((e - 1) >> 3) - (s >> 3) + 1 : e - s;
}
// Output index of the item whose (first) key is `key`, in a row starting at `base`.
__device__ __forceinline__ int32_t out_index(int key, int base) {
  return kBlocks ? (key >> 3) - (base >> 3) : key - base;
}
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kEpiBarrier = 1;  // named barrier id for the epilogue warps
constexpr int kGateBins = 288;  // 257 two-sided distance bins, padded to 9 per lane
constexpr int kScoreBins = 128;  // linear score bins per gated row between the gate and the sample maximum
constexpr int kSelList = 1024;   // threshold-bin records a selection warp holds in shared memory

struct JobInfo {
  int block;      // row block (-1: no more work)
  int mode;       // 0 gated scan, 1 exact rescan
  int lo_t, nt;   // main tiles [lo_t, lo_t + nt)
  int ns;         // sample tiles, scored before the main tiles (once, or twice: coarse, then fine gate pass)
  uint32_t mask;  // rows taking part
  int nrows;      // valid rows in the block
  int chunk;      // key chunk of a split block (-1: the whole block)
  int nchunks;    // chunks the block is split into (1: not split)
  int bs;         // split block index (its arrays in the split workspace)
  int s_lo_t, s_nt;  // tiles [s_lo_t, s_lo_t + s_nt) the sample plan spans (the whole block)
  int start[kBlockRows], end[kBlockRows];
  int items[kBlockRows];  // items each row selects from (keys, blocks, or allowed keys)
  alignas(16) float w[kBlockRows][kHeads];
  alignas(16) float fm[kBlockRows][kFoldRowTerms];  // fold: 2^e_t of the row's folded-query terms
  float beta[kBlockRows];                           // fold: 2-norm of the row's fold residual
#if MQA_MASKED
  // Masked selection: main tile i takes part when bit (i + toff) of tbytes is
  // set (some taking-part row has an allowed block in it); every tile takes
  // part when skip == 0 (ranges longer than the bitmap).
  int skip, toff;
  uint8_t tbytes[kSkipTiles / 8 + 8];
#endif
};

struct SelSlot {  // what the selection warps need from a finished scan
  int block, mode;
  uint32_t mask;
  int nrows;
  int start[kBlockRows], n[kBlockRows];
  int gated[kBlockRows];
  float blo[kBlockRows], binv[kBlockRows];  // score-bin origin (the gate) and bins per unit score
  int binned[kBlockRows];                    // mode-0 gated row: selected through score bins
  int unsafe[kBlockRows];                    // fold: the gate found the row's fold error bound too large
  int check[kBlockRows];                     // fold: classify the row in selection (no sampled score)
  float beta[kBlockRows];                    // fold: 2-norm of the row's fold residual
  int split;    // candidates are in the split slab of block bs, nseg segments of seglen per row
  int bs, nseg, seglen;
  int dist;        // a spread merge: the block's rows are claimed from merge_next by every chunk CTA
  int count_done;  // this slot counts the block finished (the block's last chunk)
  int segcnt[kBlockRows][32];  // records per (row, segment): 4 quadrant segments, or one run per key chunk
};

struct Smem {
  alignas(1024) uint8_t kring[kKStages][kKTileBytes];
  alignas(1024) uint8_t q[2][kQBytes];
  alignas(128) float sring[kSStages][kTileKeys];  // key scales of the tiles in flight
  alignas(16) uint32_t mring[kSStages][kBlockRows][4];  // block-mask words of the tiles in flight (masked)
  JobInfo job[2];
  SelSlot sel[2];
  float tau[kBlockRows];
  int segcnt[kBlockRows][kQuads];
  int nsplit, nchunks;  // key-range split plan: nsplit blocks of the order, nchunks chunks each
  int split_first;      // the split blocks are the first nsplit of the order (else the last)
  uint32_t ref[kBlockRows];
  int ref_frozen[kBlockRows];  // two-pass sample: the reference is taken from the first tile
  int msample[kBlockRows];
  // gate refinement: the coarse bin that holds the target sample rank
  int g_on[kBlockRows], g_above[kBlockRows], g_j[kBlockRows];
  uint32_t g_klo[kBlockRows], g_khi[kBlockRows];
  int hist[kBlockRows][kGateBins];
  int selhist[kSelWarps][256];
  uint32_t sel_lk[kSelWarps][kSelList];  // keys of the threshold bin's members
  int32_t sel_li[kSelWarps][kSelList];   // and their key indices
  uint32_t smax[kBlockRows];             // largest sample order key per row (current scan)
  uint32_t smin[kBlockRows];             // fold: smallest sample order key per row (current scan)
  float binv[kBlockRows];                // score bins per unit score (current scan)
  uint16_t order[kMaxSortBlocks];
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t sc_full[kSStages], sc_empty[kSStages];
  uint64_t t_full[kTmemBufs], t_empty[kTmemBufs];
  uint64_t j_full[2], j_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t drain, stall_bar;
  uint32_t tmem_base;
  int abort_flag;
  int fifo_block[8];
  uint32_t fifo_mask[8];
  int fifo_head, fifo_tail;
  int retired;
  int seldone[2];    // rows finished over all uses of the selection slot
  int selnext[2];    // rows claimed over all uses of the selection slot
  uint32_t selfail[2];
  int prod_parked;   // the producer has issued its last job and waits for every job to retire
  int grp_row[2];    // spread merge: the row each epilogue group selects next
  unsigned grp_fails;  // spread merge: rows the groups failed (to rescan)
  float key_norm;    // fold: largest key_scale * |k|_2 over the keys (this call)
  int unsafe[kBlockRows];  // fold: rows of the current scan whose fold error bound is too large
  int classified[kBlockRows];  // fold: rows of the current scan classified at the gate
#if MQA_PAIR_HELPERS
  int pair_cnt[kEpiWarps / 2];  // arrivals at the two-warp syncs of each helper pair (monotonic)
  int pair_row[kEpiWarps / 2];  // the row the pair's leader claimed
  int helping[2];               // 1 + the slot use the parked helper pairs select (selection warps then stop claiming)
#endif
};

size_t fused_smem_bytes() { return sizeof(Smem) + 1024; }
constexpr int kAttrDevices = 64;  // device ordinals the launchers track
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory above the 227 KB opt-in limit");

__device__ __forceinline__ Smem &get_smem(uint8_t *raw) {
  uintptr_t a = reinterpret_cast<uintptr_t>(raw);
  a = (a + 1023) & ~uintptr_t(1023);
  return *reinterpret_cast<Smem *>(a);
}

// ------------------------------------------------------------------ waits
__device__ __forceinline__ bool aborted(Smem &S) { return *(volatile int *)&S.abort_flag != 0; }

__device__ __noinline__ void raise_timeout(Smem &S, const FusedParams &p) {
  *(volatile int *)&S.abort_flag = 1;
  atomicOr(p.ws + kWsStatus, kDevWaitTimeout);
}

#ifndef MQA_BACKOFF_SCALE
#define MQA_BACKOFF_SCALE 2
#endif
// Sleep between polls of a waiting role, so that warps which wait for long
// stretches (producer, selection, MMA issuer) leave issue slots to the
// epilogue warps that share their SM sub-partitions.
constexpr unsigned kBackoffMma = 32 * MQA_BACKOFF_SCALE;
constexpr unsigned kBackoffIdle = 256 * MQA_BACKOFF_SCALE;

// Wait for the phase of `bar` with the given parity; false on abort/timeout.
__device__ __forceinline__ bool wait_bar(Smem &S, uint64_t *bar, uint32_t parity, const FusedParams &p,
                                         unsigned backoff_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (aborted(S)) return false;
    if (backoff_ns) __nanosleep(backoff_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if ((long long)(globaltimer_ns() - t0) > p.timeout_ns) {
      raise_timeout(S, p);
      return false;
    }
  }
}

// Spin until *flag >= target (smem, written by another warp); false on abort/timeout.
__device__ __forceinline__ bool wait_counter(Smem &S, int *flag, int target, const FusedParams &p) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (*(volatile int *)flag >= target) return true;
    if (aborted(S)) return false;
    if ((long long)(globaltimer_ns() - t0) > p.timeout_ns) {
      raise_timeout(S, p);
      return false;
    }
    __nanosleep(64);
  }
}

// Spin until the global counter *addr >= target (written by other CTAs of
// this launch); false on abort/timeout.
__device__ __forceinline__ bool wait_global(Smem &S, const int *addr, int target, const FusedParams &p) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (*(volatile const int *)addr >= target) {
      __threadfence();
      return true;
    }
    if (aborted(S)) return false;
    if ((long long)(globaltimer_ns() - t0) > p.timeout_ns) {
      raise_timeout(S, p);
      return false;
    }
    __nanosleep(64);
  }
}

// Spread merge (pair-helper compilation): when every block of the call is
// split and there are no more key chunks than CTAs, CTA i scans chunk job i
// and nothing else, so each CTA is parked once its chunk is scanned.  Every
// chunk CTA of a block then waits for the block's last chunk and claims the
// block's rows one at a time (merge_next), each row selected by its 16
// epilogue warps together, instead of the last chunk's CTA selecting all 8.
// A CTA waits on other CTAs only after it has no scan work left, and the
// chunks it waits for are all assigned to running CTAs, so the wait ends (it
// is also bounded by the call's time limit).
__device__ __forceinline__ bool spread_merge(const Smem &S, const FusedParams &p) {
#if MQA_PAIR_HELPERS
  return S.nsplit > 0 && S.nsplit == p.nblocks && S.nsplit * S.nchunks <= (int)gridDim.x;
#else
  return false;
#endif
}

// ------------------------------------------------------------------ scoring
// A row's kHeads accumulator columns are read in groups of 32: each epilogue
// thread reads a group with two 16x256b TMEM loads (lanes 0-15 and 16-31 of
// its warp's quadrant) and gets 4 keys (A = g, B = g+8, C = g+16, D = g+24
// with g = lane/4) x 8 heads (8i + 2c, 8i + 2c + 1 for i < 4, c = lane%4) of
// it.  relu(x) is formed as (x + |x|): a packed FP add whose second operand
// carries an absolute-value modifier (FMA pipe); the 1/2 is folded into the
// key scale.  x + |x| is exactly 2x or 0 and the halving is exact.  The 4
// threads of a key group then reduce-scatter their partial head sums so that
// every thread owns the full sum of one key.  The summation order is fixed
// and the fused and logits instantiations share this code, so both produce
// bit-identical scores.
#ifndef MQA_RELU_ALU_CHUNKS
#define MQA_RELU_ALU_CHUNKS 1
#endif
// Of a thread's head-pair chunks per key, the first MQA_RELU_ALU_CHUNKS form
// relu as max(x, 0) on the ALU pipe with pre-doubled weights (2w * max(x, 0));
// the rest use x + |x| on the FMA pipe with w.  Both give 2 * w * relu(x)
// exactly (one rounding of the same product), so the split only balances the
// two pipes and leaves the scores bit-identical.  A packed FFMA2 or FADD2
// holds the FMA pipe for two cycles, so the relu add and the weighted
// accumulate keep that pipe saturated through the head sum; moving one chunk
// of four to the ALU pipe was the fastest split measured (none, a quarter,
// three eighths and a half were compared).
constexpr int kHeadGroups = kHeads / 32;  // 32-column groups per row
struct HeadW {
  float2 w[4 * kHeadGroups];  // weights of this thread's heads of one row, as pairs (doubled for ALU chunks)
};

template <int kChunk>
__device__ __forceinline__ float2 relu2(uint32_t a, uint32_t b) {
  const float2 x = make_float2(__uint_as_float(a), __uint_as_float(b));
  if (kChunk < MQA_RELU_ALU_CHUNKS) return make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f));
  return __fadd2_rn(x, make_float2(fabsf(x.x), fabsf(x.y)));
}

// Accumulate head group G (columns 32G .. 32G + 31) of one row.
template <int G>
__device__ __forceinline__ void head_group(const uint32_t (&lo)[16], const uint32_t (&hi)[16], const HeadW &W,
                                           float2 &aA, float2 &aB, float2 &aC, float2 &aD) {
#define MQA_HEAD_CHUNK(i)                                                             \
  aA = __ffma2_rn(relu2<4 * G + i>(lo[4 * i], lo[4 * i + 1]), W.w[4 * G + i], aA);     \
  aB = __ffma2_rn(relu2<4 * G + i>(lo[4 * i + 2], lo[4 * i + 3]), W.w[4 * G + i], aB); \
  aC = __ffma2_rn(relu2<4 * G + i>(hi[4 * i], hi[4 * i + 1]), W.w[4 * G + i], aC);     \
  aD = __ffma2_rn(relu2<4 * G + i>(hi[4 * i + 2], hi[4 * i + 3]), W.w[4 * G + i], aD);
  MQA_HEAD_CHUNK(0)
  MQA_HEAD_CHUNK(1)
  MQA_HEAD_CHUNK(2)
  MQA_HEAD_CHUNK(3)
#undef MQA_HEAD_CHUNK
}

// Full relu-weighted head sum of the key this thread owns (before scaling),
// from the thread's partial sums of keys A..D.
__device__ __forceinline__ float reduce_keys(float2 aA, float2 aB, float2 aC, float2 aD, int lane) {
  const float pA = aA.x + aA.y, pB = aB.x + aB.y, pC = aC.x + aC.y, pD = aD.x + aD.y;
  // step 1 (partner lane^1): even lanes keep keys A, B; odd lanes keep C, D
  const bool odd = lane & 1;
  const float s0 = odd ? pA : pC, s1 = odd ? pB : pD;
  const float k0 = (odd ? pC : pA) + __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
  const float k1 = (odd ? pD : pB) + __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
  // step 2 (partner lane^2): lanes with bit 1 clear keep the first key
  const bool second = lane & 2;
  const float s = second ? k0 : k1;
  return (second ? k1 : k0) + __shfl_xor_sync(0xFFFFFFFFu, s, 2);
}

// Key (0..31 within the warp's quadrant) whose sum reduce_keys leaves in `lane`.
__device__ __forceinline__ int owned_key(int lane) { return (lane >> 2) + 8 * ((lane >> 1) & 1) + 16 * (lane & 1); }

// Scaled head sums of this lane's key for the warp's kRowsPerWarp rows of one
// tile, read from TMEM at `base` (the warp's quadrant, its first row).  Every
// row is always loaded and summed (every TMEM address here is in the
// allocation), so the code has no per-row branches; the caller masks rows
// that do not take part.  The TMEM buffer is released (t_empty) once the last
// row is in registers.
//
// With 32 heads a row is read by key halves: lanes 0-15 of the quadrant
// (keys A, B), their head sums, then lanes 16-31 (keys C, D), so only 16
// accumulator values are in registers at a time.  That measured 3% faster at
// 1M keys than loading a row's two halves together (the summation order, and
// so every score, is the same).  With 64 heads a row's head groups are loaded
// together.
#if MQA_HEADS == 32
__device__ __forceinline__ void score_rows(uint64_t *t_empty, uint32_t base, const HeadW (&W)[kRowsPerWarp],
                                           float hsc, int lane, float (&out)[kRowsPerWarp]) {
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    float2 aA = make_float2(0.f, 0.f), aB = aA, aC = aA, aD = aA;
    {
      uint32_t v[16];
      tmem_ld_16x256b_x4(base + (uint32_t)(rr * kHeads), v);
      tmem_ld_wait();
#define MQA_HALF_CHUNK(i, X, Y)                                         \
  X = __ffma2_rn(relu2<i>(v[4 * i], v[4 * i + 1]), W[rr].w[i], X);      \
  Y = __ffma2_rn(relu2<i>(v[4 * i + 2], v[4 * i + 3]), W[rr].w[i], Y);
      MQA_HALF_CHUNK(0, aA, aB)
      MQA_HALF_CHUNK(1, aA, aB)
      MQA_HALF_CHUNK(2, aA, aB)
      MQA_HALF_CHUNK(3, aA, aB)
    }
    {
      uint32_t v[16];
      tmem_ld_16x256b_x4(base + (16u << 16) + (uint32_t)(rr * kHeads), v);
      tmem_ld_wait();
      if (rr == kRowsPerWarp - 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(t_empty);
      }
      MQA_HALF_CHUNK(0, aC, aD)
      MQA_HALF_CHUNK(1, aC, aD)
      MQA_HALF_CHUNK(2, aC, aD)
      MQA_HALF_CHUNK(3, aC, aD)
#undef MQA_HALF_CHUNK
    }
    out[rr] = reduce_keys(aA, aB, aC, aD, lane) * hsc;
  }
}
#else
__device__ __forceinline__ void score_rows(uint64_t *t_empty, uint32_t base, const HeadW (&W)[kRowsPerWarp],
                                           float hsc, int lane, float (&out)[kRowsPerWarp]) {
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    uint32_t lo[kHeadGroups][16], hi[kHeadGroups][16];
#pragma unroll
    for (int g = 0; g < kHeadGroups; ++g) {
      const uint32_t col = (uint32_t)(rr * kHeads + 32 * g);
      tmem_ld_16x256b_x4(base + col, lo[g]);
      tmem_ld_16x256b_x4(base + (16u << 16) + col, hi[g]);
    }
    tmem_ld_wait();
    if (rr == kRowsPerWarp - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(t_empty);
    }
    float2 aA = make_float2(0.f, 0.f), aB = aA, aC = aA, aD = aA;
    head_group<0>(lo[0], hi[0], W[rr], aA, aB, aC, aD);
    if constexpr (kHeadGroups > 1) head_group<1>(lo[1], hi[1], W[rr], aA, aB, aC, aD);
    out[rr] = reduce_keys(aA, aB, aC, aD, lane) * hsc;
  }
}
#endif  // MQA_HEADS

#if MQA_FOLD
// ------------------------------------------------------------------ scoring with the fold
// relu(s) = (s + |s|) / 2, so sum_h w_h relu(s_h) = (v . k + sum_h w_h |s_h|) / 2
// with the folded query v = sum_h w_h q_h (vLLM pull request #60618, "What
// this PR does", Scoring bullet).  The tensor core computes v . k from v's
// four e4m3 terms: u_t . k in the row's four fold columns, v . k = sum_t
// 2^e_t u_t . k up to the residual (at most beta |k|_2).  So the head sum is one
// packed FMA with an absolute-value operand per head pair:
//     s(r, j) = (scale_j / 2) * (sum_h w_h |s_h| + sum_t 2^e_t u_t . k_j).
// The direct form (exact rescans) forms 2 relu(s) = s + |s| per head and
// leaves the fold columns out:  s(r, j) = (scale_j / 2) * sum_h w_h 2 relu(s_h).
//
// Thread layout (16x256b loads, as the other compilations): per row, thread
// t holds keys A..D (t/4, +8, +16, +24) x heads 8i + 2c, 8i + 2c + 1 (c = t %
// 4), the 4 lanes of a key group then reduce-scatter.  The fold columns of the
// warp's two rows (rbase even: 8 adjacent columns) arrive with one 16x256b.x1
// load per half of the lanes: lane c holds terms 2(c % 2), 2(c % 2) + 1 of row
// rbase + c / 2 for keys A..D, so it adds 2^e-scaled terms into that row's
// partial sums (the other row's multipliers are zero) before the exchange.
// Both rows are loaded before one wait and the accumulator buffer is released
// before any arithmetic.
static_assert(!kFold || kRowsPerWarp == 2, "the fold layout pairs a warp's rows");
static_assert(!kFold || kFoldCols == kFoldBoxRows, "fold columns match the fold-term TMA box");

struct FoldM {
  float2 m[2];  // per row of the warp: (2^e, 2^e') of this lane's two terms, or zeros
};

__device__ __forceinline__ void tmem_ld_16x256b_x1(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr)
               : "memory");
}

template <bool kDirect>
__device__ __forceinline__ void score_rows_fold(uint64_t *t_empty, uint32_t base, uint32_t fold_addr,
                                                const HeadW (&W)[kRowsPerWarp], const FoldM &M, float hsc, int lane,
                                                float (&out)[kRowsPerWarp]) {
  uint32_t lo[kRowsPerWarp][16], hi[kRowsPerWarp][16], flo[4], fhi[4];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    tmem_ld_16x256b_x4(base + (uint32_t)(rr * kHeads), lo[rr]);
    tmem_ld_16x256b_x4(base + (16u << 16) + (uint32_t)(rr * kHeads), hi[rr]);
  }
  if (!kDirect) {
    tmem_ld_16x256b_x1(fold_addr, flo);
    tmem_ld_16x256b_x1(fold_addr + (16u << 16), fhi);
  }
  tmem_ld_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(t_empty);
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    float2 aA = make_float2(0.f, 0.f), aB = aA, aC = aA, aD = aA;
    if (!kDirect) {
      // this lane's fold terms of keys A, B (low lanes) and C, D (high lanes)
      aA = __fmul2_rn(make_float2(__uint_as_float(flo[0]), __uint_as_float(flo[1])), M.m[rr]);
      aB = __fmul2_rn(make_float2(__uint_as_float(flo[2]), __uint_as_float(flo[3])), M.m[rr]);
      aC = __fmul2_rn(make_float2(__uint_as_float(fhi[0]), __uint_as_float(fhi[1])), M.m[rr]);
      aD = __fmul2_rn(make_float2(__uint_as_float(fhi[2]), __uint_as_float(fhi[3])), M.m[rr]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 xA = make_float2(__uint_as_float(lo[rr][4 * i]), __uint_as_float(lo[rr][4 * i + 1]));
      const float2 xB = make_float2(__uint_as_float(lo[rr][4 * i + 2]), __uint_as_float(lo[rr][4 * i + 3]));
      const float2 xC = make_float2(__uint_as_float(hi[rr][4 * i]), __uint_as_float(hi[rr][4 * i + 1]));
      const float2 xD = make_float2(__uint_as_float(hi[rr][4 * i + 2]), __uint_as_float(hi[rr][4 * i + 3]));
      if (kDirect) {
        aA = __ffma2_rn(__fadd2_rn(xA, make_float2(fabsf(xA.x), fabsf(xA.y))), W[rr].w[i], aA);
        aB = __ffma2_rn(__fadd2_rn(xB, make_float2(fabsf(xB.x), fabsf(xB.y))), W[rr].w[i], aB);
        aC = __ffma2_rn(__fadd2_rn(xC, make_float2(fabsf(xC.x), fabsf(xC.y))), W[rr].w[i], aC);
        aD = __ffma2_rn(__fadd2_rn(xD, make_float2(fabsf(xD.x), fabsf(xD.y))), W[rr].w[i], aD);
      } else {
        aA = __ffma2_rn(make_float2(fabsf(xA.x), fabsf(xA.y)), W[rr].w[i], aA);
        aB = __ffma2_rn(make_float2(fabsf(xB.x), fabsf(xB.y)), W[rr].w[i], aB);
        aC = __ffma2_rn(make_float2(fabsf(xC.x), fabsf(xC.y)), W[rr].w[i], aC);
        aD = __ffma2_rn(make_float2(fabsf(xD.x), fabsf(xD.y)), W[rr].w[i], aD);
      }
    }
    out[rr] = reduce_keys(aA, aB, aC, aD, lane) * hsc;
  }
}
#endif

// ------------------------------------------------------------------ sample gate bins
// Distance d (in order-key units) below the row's reference maximum, binned on
// a log scale with four sub-bins per power of two: bin 0 holds d == 0.
__device__ __forceinline__ int dist_bin(uint32_t d) {
  if (d == 0) return 0;
  const int msb = 31 - __clz(d);
  const uint32_t sub = msb >= 2 ? (d >> (msb - 2)) & 3u : (d << (2 - msb)) & 3u;
  return 1 + 4 * msb + (int)sub;
}
// Smallest distance inside bin b (b >= 1).
__device__ __forceinline__ uint32_t dist_bin_lo(int b) {
  const int msb = (b - 1) >> 2, sub = (b - 1) & 3;
  if (msb >= 2) return (uint32_t)(4 + sub) << (msb - 2);
  return (uint32_t)((4 + sub) >> (2 - msb));
}
// Gate bins are two-sided around the reference key: bins 0..127 hold scores
// above it (farther above = smaller bin), bin 128 the reference itself, bins
// 129..256 scores below it (farther below = larger bin).  Bin order is
// therefore descending score order.
__device__ __forceinline__ int gate_bin(uint32_t key, uint32_t ref) {
  return key > ref ? 128 - dist_bin(key - ref) : 128 + dist_bin(ref - key);
}
// Smallest distance beyond bin b (every d in bins 0..b is below it).
__device__ __forceinline__ uint64_t dist_bin_hi(int b) {
  if (b == 0) return 1;
  const int msb = (b - 1) >> 2, sub = (b - 1) & 3;
  if (msb >= 2) return (uint64_t)(5 + sub) << (msb - 2);
  return (uint64_t)((4 + sub) >> (2 - msb)) + 1;
}

// ------------------------------------------------------------------ warp radix select
#ifdef MQA_SEL_NOINLINE
#define MQA_SEL_FN __noinline__
#else
#define MQA_SEL_FN
#endif
// A row's candidates live in nseg segments of `seg` records each (one per
// TMEM lane quadrant, times the key chunks of a split block); segment q holds
// c[q] valid records (c points to shared memory).
struct RowSlab {
  uint32_t *keys;  // [nseg][seg]
  int32_t *idx;    // [nseg][seg]
  int seg, nseg;
  const int *c;
  __device__ int total() const {
    int t = 0;
    for (int q = 0; q < nseg; ++q) t += c[q];
    return t;
  }
};

// A row's candidates are visited in pieces of 128 records (32 lanes x 4),
// numbered across segment boundaries, so that one batch of loads covers
// several short segments (the key chunks of a split block) as readily as one
// long segment.  Lane q (< nseg) holds segment q's record count and the
// running piece counts; piece t lies in the segment whose inclusive piece
// prefix first exceeds t, found by one ballot.
struct PieceMap {
  int cnt;    // lane q: records in segment q
  int pexcl;  // lane q: pieces before segment q
  int pincl;  // lane q: pieces up to and including segment q (INT_MAX past nseg)
  int total;  // pieces in the row
};
__device__ __forceinline__ PieceMap piece_map(const RowSlab &R, int lane) {
  PieceMap m;
  m.cnt = lane < R.nseg ? R.c[lane] : 0;
  const int np = (m.cnt + 127) >> 7;
  int incl = np;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  m.pexcl = incl - np;
  m.total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  m.pincl = lane < R.nseg ? incl : INT_MAX;
  return m;
}
// Piece t: element offset of its first record in the row's slab and the
// number of valid records in it (0 past the last piece).  Warp-uniform.
__device__ __forceinline__ void piece_at(const RowSlab &R, const PieceMap &m, int t, int &at, int &lim) {
  const int q = min(__popc(__ballot_sync(0xFFFFFFFFu, m.pincl <= t)), 31);
  const int pe = __shfl_sync(0xFFFFFFFFu, m.pexcl, q), c = __shfl_sync(0xFFFFFFFFu, m.cnt, q);
  const int off = (t - pe) << 7;
  at = q * R.seg + off;
  lim = t < m.total ? min(c - off, 128) : 0;
}

// Exact k-th largest order key over the row's candidates (requires total > k
// >= 1), by four 8-bit digit levels.  Returns the key T; *take_eq receives
// how many keys equal to T belong to the top k (the rest of the top k is > T).
__device__ MQA_SEL_FN uint32_t warp_radix_select(const RowSlab &R, int k, int *hist, int lane, int *take_eq) {
  uint32_t prefix = 0;
  int want = k;
#pragma unroll 1
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    const uint32_t hi_mask = level == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
#pragma unroll 1
    for (int q = 0; q < R.nseg; ++q) {
      const uint32_t *keys = R.keys + (size_t)q * R.seg;
      const int n = R.c[q];
#pragma unroll 1
      for (int i0 = 0; i0 < n; i0 += 32 * 8) {
        uint32_t kk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + 32 * j + lane;
          kk[j] = i < n ? __ldcg(keys + i) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + 32 * j + lane;
          if (i < n && (kk[j] & hi_mask) == prefix) atomicAdd(&hist[(kk[j] >> shift) & 255u], 1);
        }
      }
    }
    __syncwarp();
    int c[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[255 - 8 * lane - j];
      tot += c[j];
    }
    int incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += v;
    }
    const int excl = incl - tot;
    const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < want && want <= incl);
    const int src = bm ? __ffs(bm) - 1 : 31;
    int bin = 0, above = 0;
    if (lane == src) {
      int run = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run + c[j] >= want) {
          bin = 255 - 8 * lane - j;
          above = run;
          break;
        }
        run += c[j];
      }
    }
    bin = __shfl_sync(0xFFFFFFFFu, bin, src);
    above = __shfl_sync(0xFFFFFFFFu, above, src);
    want -= above;
    prefix |= (uint32_t)bin << shift;
    __syncwarp();
  }
  *take_eq = want;
  return prefix;
}

// Stream the row's candidates once, keeping every key > T plus the first
// `take_eq` keys equal to T (all keys when take_all).  Kept entries either go
// to `out` as idx - base (the caller pads with -1) or are compacted into
// segment 0 (stable; within segment 0 writes never overtake reads, and the
// other segments are only read).  At most `limit` entries are kept.
template <bool kCompact>
__device__ MQA_SEL_FN int warp_emit(const RowSlab &R, uint32_t T, int take_eq, bool take_all, int32_t *out, int base,
                         int limit, int lane) {
  int outc = 0, eq_seen = 0;
  const uint32_t lt = lanemask_lt();
#pragma unroll 1
  for (int q = 0; q < R.nseg; ++q) {
    const uint32_t *keys = R.keys + (size_t)q * R.seg;
    const int32_t *idx = R.idx + (size_t)q * R.seg;
    const int n = R.c[q];
#pragma unroll 1
    for (int i0 = 0; i0 < n; i0 += 32 * 4) {
      uint32_t kk[4];
      int32_t ii[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + 32 * j + lane;
        kk[j] = i < n ? __ldcg(keys + i) : 0u;
        ii[j] = i < n ? __ldcg(idx + i) : 0;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + 32 * j + lane;
        const bool v = i < n;
        const bool gt = v && (take_all || kk[j] > T);
        const bool eq = v && !take_all && kk[j] == T;
        const uint32_t beq = __ballot_sync(0xFFFFFFFFu, eq);
        const int eq_rank = eq_seen + __popc(beq & lt);
        const bool take = gt || (eq && eq_rank < take_eq);
        const uint32_t bt = __ballot_sync(0xFFFFFFFFu, take);
        if (take) {
          const int pos = outc + __popc(bt & lt);
          if (pos < limit) {
            if (kCompact) {
              R.keys[pos] = kk[j];
              R.idx[pos] = ii[j];
            } else {
              out[pos] = out_index(ii[j], base);
            }
          }
        }
        outc += __popc(bt);
        eq_seen += __popc(beq);
      }
    }
  }
  return outc < limit ? outc : limit;
}

// ------------------------------------------------------------------ selection over a key range
// 16-byte loads in flight per lane in the selection warps' scans.
#ifndef MQA_SEL_DEPTH
#define MQA_SEL_DEPTH 4
#endif
constexpr int kSelDepth = MQA_SEL_DEPTH;

// Smallest and largest order key of the row's candidates (one load-only pass).
__device__ void warp_key_range(const RowSlab &R, int lane, uint32_t *kmin, uint32_t *kmax) {
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  const PieceMap pm = piece_map(R, lane);
#pragma unroll 1
  for (int t0 = 0; t0 < pm.total; t0 += kSelDepth) {
    int at[kSelDepth], lim[kSelDepth];
    uint4 kk[kSelDepth];
#pragma unroll
    for (int j = 0; j < kSelDepth; ++j) piece_at(R, pm, t0 + j, at[j], lim[j]);
#pragma unroll
    for (int j = 0; j < kSelDepth; ++j)
      kk[j] = 4 * lane < lim[j] ? __ldcg(reinterpret_cast<const uint4 *>(R.keys + at[j] + 4 * lane))
                                : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < kSelDepth; ++j) {
      const uint32_t v[4] = {kk[j].x, kk[j].y, kk[j].z, kk[j].w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (4 * lane + t < lim[j]) {
          lo = min(lo, v[t]);
          hi = max(hi, v[t]);
        }
      }
    }
  }
  *kmin = __reduce_min_sync(0xFFFFFFFFu, lo);
  *kmax = __reduce_max_sync(0xFFFFFFFFu, hi);
}

// Exact k-th largest order key of the row's candidates (total > k >= 1).
// The candidates lie in [kmin, kmax] and share the binary prefix of those
// two, so 8-bit radix digits start at the highest bit where they differ
// (usually three levels; no pile-up of all keys in one bin).  Eight 16-byte
// loads per lane are in flight per batch.
__device__ MQA_SEL_FN uint32_t warp_select_range(const RowSlab &R, int k, int *hist, int lane, int *take_eq,
                                                  uint32_t kmin, uint32_t kmax) {
  const uint32_t diff = kmin ^ kmax;
  int hi = diff ? 32 - __clz(diff) : 0;  // bits [0, hi) vary among the candidates
  uint32_t prefix = hi >= 32 ? 0u : (kmax & ~((1u << hi) - 1u));
  int want = k;
#pragma unroll 1
  while (hi > 0) {
    const int bits = hi >= 8 ? 8 : hi;
    const int shift = hi - bits;
    const uint32_t dmask = (1u << bits) - 1u;
    const uint32_t hi_mask = hi >= 32 ? 0u : (0xFFFFFFFFu << hi);
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    const PieceMap pm = piece_map(R, lane);
#pragma unroll 1
    for (int t0 = 0; t0 < pm.total; t0 += kSelDepth) {
      int at[kSelDepth], lim[kSelDepth];
      uint4 kk[kSelDepth];
#pragma unroll
      for (int j = 0; j < kSelDepth; ++j) piece_at(R, pm, t0 + j, at[j], lim[j]);
#pragma unroll
      for (int j = 0; j < kSelDepth; ++j)
        kk[j] = 4 * lane < lim[j] ? __ldcg(reinterpret_cast<const uint4 *>(R.keys + at[j] + 4 * lane))
                                  : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < kSelDepth; ++j) {
        const uint32_t v[4] = {kk[j].x, kk[j].y, kk[j].z, kk[j].w};
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (4 * lane + t < lim[j] && (v[t] & hi_mask) == prefix) atomicAdd(&hist[(v[t] >> shift) & dmask], 1);
      }
    }
    __syncwarp();
    int c[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[255 - 8 * lane - j];
      tot += c[j];
    }
    int incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += v;
    }
    const int excl = incl - tot;
    const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < want && want <= incl);
    const int src = bm ? __ffs(bm) - 1 : 31;
    int bin = 0, above = 0;
    if (lane == src) {
      int run = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run + c[j] >= want) {
          bin = 255 - 8 * lane - j;
          above = run;
          break;
        }
        run += c[j];
      }
    }
    bin = __shfl_sync(0xFFFFFFFFu, bin, src);
    above = __shfl_sync(0xFFFFFFFFu, above, src);
    want -= above;
    prefix |= (uint32_t)bin << shift;
    hi = shift;
    __syncwarp();
  }
  *take_eq = want;
  return prefix;
}
__device__ __forceinline__ uint32_t warp_select_range(const RowSlab &R, int k, int *hist, int lane, int *take_eq) {
  uint32_t kmin, kmax;
  warp_key_range(R, lane, &kmin, &kmax);
  return warp_select_range(R, k, hist, lane, take_eq, kmin, kmax);
}

// Write the row's top-k indices (idx - base) to out: every key > T plus
// `take_eq` of the keys equal to T (all keys when take_all).  Which equal keys
// are taken and the output order are free; 8 records per lane per batch.
// Returns the number written (at most `limit`).
__device__ MQA_SEL_FN int warp_emit_out(const RowSlab &R, uint32_t T, int take_eq, bool take_all, int32_t *out, int base,
                             int limit, int lane) {
  int outc = 0, eq_seen = 0;
  const PieceMap pm = piece_map(R, lane);
#pragma unroll 1
  for (int t0 = 0; t0 < pm.total; t0 += 2) {
    {
      int at[2], lim[2];
      uint32_t kk[8];
      int32_t ii[8];
#pragma unroll
      for (int g = 0; g < 2; ++g) piece_at(R, pm, t0 + g, at[g], lim[g]);
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint4 kv = make_uint4(0, 0, 0, 0);
        int4 iv = make_int4(0, 0, 0, 0);
        if (4 * lane < lim[g]) {
          kv = __ldcg(reinterpret_cast<const uint4 *>(R.keys + at[g] + 4 * lane));
          iv = __ldcg(reinterpret_cast<const int4 *>(R.idx + at[g] + 4 * lane));
        }
        kk[4 * g] = kv.x; kk[4 * g + 1] = kv.y; kk[4 * g + 2] = kv.z; kk[4 * g + 3] = kv.w;
        ii[4 * g] = iv.x; ii[4 * g + 1] = iv.y; ii[4 * g + 2] = iv.z; ii[4 * g + 3] = iv.w;
      }
      bool gt[8], eq[8];
      int neq = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool v = 4 * lane + (j & 3) < lim[j >> 2];
        gt[j] = v && (take_all || kk[j] > T);
        eq[j] = v && !take_all && kk[j] == T;
        neq += eq[j];
      }
      int eq_incl = neq;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, eq_incl, off);
        if (lane >= off) eq_incl += v;
      }
      int eq_rank = eq_seen + eq_incl - neq;
      int ntake = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (eq[j]) {
          eq[j] = eq_rank < take_eq;
          ++eq_rank;
        }
        ntake += gt[j] || eq[j];
      }
      int t_incl = ntake;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, t_incl, off);
        if (lane >= off) t_incl += v;
      }
      int pos = outc + t_incl - ntake;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (gt[j] || eq[j]) {
          if (pos < limit) out[pos] = out_index(ii[j], base);
          ++pos;
        }
      }
      outc += __shfl_sync(0xFFFFFFFFu, t_incl, 31);
      eq_seen += __shfl_sync(0xFFFFFFFFu, eq_incl, 31);
    }
  }
  return outc < limit ? outc : limit;
}

// ------------------------------------------------------------------ binned selection
// A gated row's candidates all score above its gate t.  Their scores are
// counted into kScoreBins linear bins between t and the largest sample score
// (scores above that share the top bin).  The count pass finds the bin B that
// holds the k-th largest score; the order keys where bin B starts and ends
// are then found by bisection (the bin is a monotone function of the key), and
// one more pass writes every candidate above B straight to the output and
// gathers B's members into shared memory, where an exact radix select over
// those few records settles the rest.
__device__ __forceinline__ int score_bin(float s, float lo, float inv) {
  const float x = __fmul_rn(__fsub_rn(s, lo), inv);
  return x >= (float)(kScoreBins - 1) ? kScoreBins - 1 : max(0, __float2int_rz(x));
}

// Smallest order key in [lo_key, kKeyPosInf] whose score bin is >= b
// (kKeyPosInf + 1 when there is none).  Keys above +inf's are NaNs and are
// never searched.
constexpr uint32_t kKeyPosInf = 0xFF800000u;
__device__ uint64_t first_key_of_bin(int b, uint32_t lo_key, float lo, float inv) {
  uint64_t a = lo_key, z = (uint64_t)kKeyPosInf + 1;  // answer in [a, z]
  while (a < z) {
    const uint64_t m = (a + z) >> 1;
    if (score_bin(key2f((uint32_t)m), lo, inv) >= b) z = m;
    else a = m + 1;
  }
  return a;
}

// Count pass: score-bin histogram of the row's candidates into hist[kScoreBins].
#ifndef MQA_HIST_DEPTH
#define MQA_HIST_DEPTH 8
#endif
constexpr int kHistDepth = MQA_HIST_DEPTH;  // pieces (16-byte loads per lane) in flight
__device__ void score_hist(const RowSlab &R, float lo, float inv, int *hist, int lane) {
  for (int b = lane; b < kScoreBins; b += 32) hist[b] = 0;
  __syncwarp();
  const PieceMap pm = piece_map(R, lane);
#pragma unroll 1
  for (int t0 = 0; t0 < pm.total; t0 += kHistDepth) {
    int at[kHistDepth], lim[kHistDepth];
    uint4 kk[kHistDepth];
#pragma unroll
    for (int j = 0; j < kHistDepth; ++j) piece_at(R, pm, t0 + j, at[j], lim[j]);
#pragma unroll
    for (int j = 0; j < kHistDepth; ++j)
      kk[j] = 4 * lane < lim[j] ? __ldcg(reinterpret_cast<const uint4 *>(R.keys + at[j] + 4 * lane))
                                : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < kHistDepth; ++j) {
      const int e = 4 * lane;
      if (e < lim[j]) atomicAdd(&hist[score_bin(key2f(kk[j].x), lo, inv)], 1);
      if (e + 1 < lim[j]) atomicAdd(&hist[score_bin(key2f(kk[j].y), lo, inv)], 1);
      if (e + 2 < lim[j]) atomicAdd(&hist[score_bin(key2f(kk[j].z), lo, inv)], 1);
      if (e + 3 < lim[j]) atomicAdd(&hist[score_bin(key2f(kk[j].w), lo, inv)], 1);
    }
  }
  __syncwarp();
}

// Exact top-k of a gated row (total > k >= 1, every candidate scoring above
// lo) into out[0, k).  Returns the number written, or -1 (nothing written)
// when the threshold bin holds more records than the shared-memory list.
constexpr int kBinsPerLane = kScoreBins / 32;
#ifndef MQA_PASS2_GROUPS
#define MQA_PASS2_GROUPS 4
#endif
constexpr int kPass2Groups = MQA_PASS2_GROUPS;  // 16-byte key and index loads in flight per lane
__device__ MQA_SEL_FN int warp_select_binned(const RowSlab &R, int k, float lo, float inv, int *hist, uint32_t *lk,
                                  int32_t *li, int32_t *out, int base, int lane) {
  score_hist(R, lo, inv, hist, lane);
  // lane l owns bins kScoreBins-1 - kBinsPerLane*l - j: a prefix over lanes counts from the top
  int c[kBinsPerLane], tot = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerLane; ++j) {
    c[j] = hist[kScoreBins - 1 - kBinsPerLane * lane - j];
    tot += c[j];
  }
  int incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  const int excl = incl - tot;
  const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < k && k <= incl);
  const int src = bm ? __ffs(bm) - 1 : 31;
  int B = 0, above = 0, nB = 0;
  if (lane == src) {
    int run = excl;
#pragma unroll
    for (int j = 0; j < kBinsPerLane; ++j) {
      if (run + c[j] >= k) {
        B = kScoreBins - 1 - kBinsPerLane * lane - j;
        above = run;
        nB = c[j];
        break;
      }
      run += c[j];
    }
  }
  B = __shfl_sync(0xFFFFFFFFu, B, src);
  above = __shfl_sync(0xFFFFFFFFu, above, src);
  nB = __shfl_sync(0xFFFFFFFFu, nB, src);
  if (nB > kSelList || nB <= 0) return -1;
  // order-key range [kb_lo, kb_hi) of bin B (kb_hi past every key when B is the top bin)
  const uint32_t lo_key = f2key(lo);
  const uint64_t kb_lo = first_key_of_bin(B, lo_key, lo, inv);
  const uint64_t kb_hi = B == kScoreBins - 1 ? (uint64_t)kKeyPosInf + 1 : first_key_of_bin(B + 1, lo_key, lo, inv);
  // pass 2: keys above B go out; B's members go to the list
  int outc = 0, lc = 0;
  const PieceMap pm = piece_map(R, lane);
#pragma unroll 1
  for (int t0 = 0; t0 < pm.total; t0 += kPass2Groups) {
    int at[kPass2Groups], lim[kPass2Groups];
    uint32_t kk[4 * kPass2Groups];
    int32_t ii[4 * kPass2Groups];
#pragma unroll
    for (int gi = 0; gi < kPass2Groups; ++gi) piece_at(R, pm, t0 + gi, at[gi], lim[gi]);
#pragma unroll
    for (int gi = 0; gi < kPass2Groups; ++gi) {
      uint4 kv = make_uint4(0, 0, 0, 0);
      int4 iv = make_int4(0, 0, 0, 0);
      if (4 * lane < lim[gi]) {
        kv = __ldcg(reinterpret_cast<const uint4 *>(R.keys + at[gi] + 4 * lane));
        iv = __ldcg(reinterpret_cast<const int4 *>(R.idx + at[gi] + 4 * lane));
      }
      kk[4 * gi] = kv.x; kk[4 * gi + 1] = kv.y; kk[4 * gi + 2] = kv.z; kk[4 * gi + 3] = kv.w;
      ii[4 * gi] = iv.x; ii[4 * gi + 1] = iv.y; ii[4 * gi + 2] = iv.z; ii[4 * gi + 3] = iv.w;
    }
    // per-lane counts of (above B) and (in B), packed as up + (in << 16)
    uint32_t up = 0, in = 0;
#pragma unroll
    for (int j = 0; j < 4 * kPass2Groups; ++j) {
      const bool v = 4 * lane + (j & 3) < lim[j >> 2];
      if (v && kk[j] >= kb_hi) up |= 1u << j;
      if (v && kk[j] >= kb_lo && kk[j] < kb_hi) in |= 1u << j;
    }
    const int packed = __popc(up) + (__popc(in) << 16);
    int pincl = packed;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, pincl, off);
      if (lane >= off) pincl += v;
    }
    const int pexcl = pincl - packed;
    int po = outc + (pexcl & 0xFFFF), pl = lc + (pexcl >> 16);
#pragma unroll
    for (int j = 0; j < 4 * kPass2Groups; ++j) {
      if ((up >> j) & 1u) {
        if (po < k) out[po] = out_index(ii[j], base);
        ++po;
      }
      if ((in >> j) & 1u) {
        if (pl < kSelList) {
          lk[pl] = kk[j];
          li[pl] = ii[j];
        }
        ++pl;
      }
    }
    const int ptot = __shfl_sync(0xFFFFFFFFu, pincl, 31);
    outc += ptot & 0xFFFF;
    lc += ptot >> 16;
  }
  __syncwarp();
  lc = min(lc, kSelList);
  // exact threshold among the list: the want-th largest key
  const int want = k - above;
  uint32_t kl = 0xFFFFFFFFu, kh = 0u;
  for (int i = lane; i < lc; i += 32) {
    kl = min(kl, lk[i]);
    kh = max(kh, lk[i]);
  }
  kl = __reduce_min_sync(0xFFFFFFFFu, kl);
  kh = __reduce_max_sync(0xFFFFFFFFu, kh);
  const uint32_t diff = kl ^ kh;
  int hb = diff ? 32 - __clz(diff) : 0;
  uint32_t prefix = hb >= 32 ? 0u : (kh & ~((1u << hb) - 1u));
  int w = want;
#pragma unroll 1
  while (hb > 0) {
    const int bits = hb >= 8 ? 8 : hb;
    const int shift = hb - bits;
    const uint32_t dmask = (1u << bits) - 1u;
    const uint32_t hi_mask = hb >= 32 ? 0u : (0xFFFFFFFFu << hb);
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    for (int i = lane; i < lc; i += 32) {
      const uint32_t v = lk[i];
      if ((v & hi_mask) == prefix) atomicAdd(&hist[(v >> shift) & dmask], 1);
    }
    __syncwarp();
    int cc[8], t8 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cc[j] = hist[255 - 8 * lane - j];
      t8 += cc[j];
    }
    int in8 = t8;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, in8, off);
      if (lane >= off) in8 += v;
    }
    const int ex8 = in8 - t8;
    const uint32_t bm8 = __ballot_sync(0xFFFFFFFFu, ex8 < w && w <= in8);
    const int s8 = bm8 ? __ffs(bm8) - 1 : 31;
    int bin = 0, ab = 0;
    if (lane == s8) {
      int run = ex8;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run + cc[j] >= w) {
          bin = 255 - 8 * lane - j;
          ab = run;
          break;
        }
        run += cc[j];
      }
    }
    bin = __shfl_sync(0xFFFFFFFFu, bin, s8);
    ab = __shfl_sync(0xFFFFFFFFu, ab, s8);
    w -= ab;
    prefix |= (uint32_t)bin << shift;
    hb = shift;
    __syncwarp();
  }
  const uint32_t T = prefix;
  // emit from the list: keys > T, then the first w keys equal to T
  int eq_seen = 0;
  const uint32_t ltm = lanemask_lt();
  for (int i0 = 0; i0 < lc; i0 += 32) {
    const int i = i0 + lane;
    const bool v = i < lc;
    const uint32_t key = v ? lk[i] : 0u;
    const bool gt = v && key > T, eq = v && key == T;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const bool take = gt || (eq && eq_seen + __popc(eqm & ltm) < w);
    const uint32_t tm = __ballot_sync(0xFFFFFFFFu, take);
    const int pos = outc + __popc(tm & ltm);
    if (take && pos < k) out[pos] = out_index(li[i], base);
    outc += __popc(tm);
    eq_seen += __popc(eqm);
  }
  return outc < k ? outc : k;
}

// ------------------------------------------------------------------ heaviest-first order
// Key-range split plan (every CTA computes the same one).  The last blocks of
// the claim order are cut into `nchunks` key chunks when that shortens the
// final rounds: with fewer blocks than CTAs all of them (idle SMs take the
// chunks), else the blocks of the last partial wave (splitting one full wave
// before it as well measured no faster and doubled the split's workspace).  Costs
// are counted in units of the lightest block's scan; each chunk also scores
// the block's whole sample again (fraction sfrac of a block).
// Sample tiles of a block whose rows see `L` keys on average (as the producer
// plans them), times the passes that score them.
__device__ long long plan_sample_tiles(const FusedParams &p, long long L) {
  const long long items = kBlocks ? L / 8 : L;
  const long long nt = (L + kTileKeys - 1) / kTileKeys;
  if (items <= p.gate_min) return 0;
  long long want = (32LL * L + (long long)p.gate_target * kTileKeys - 1) / ((long long)p.gate_target * kTileKeys);
  want = want < 4 ? 4 : (want > 64 ? 64 : want);
  if (MQA_SAMPLE_ONCE && want > p.cap / 64) want = p.cap / 64;
  return (long long)kSamplePasses * (want < nt ? want : nt);
}

// `key` holds the blocks' weights (visible keys summed over the block's rows,
// in the high 32 bits) in heaviest-first order.
__device__ void plan_split(Smem &S, const FusedParams &p, const uint64_t *key) {
  const int nb = p.nblocks, ctas = gridDim.x;
  const long long w_light = (long long)(key[nb - 1] >> 32);
  const int cand = nb < ctas ? nb : nb % ctas;
  if (cand == 0 || cand > p.split_max) return;
  const long long L = w_light / kBlockRows;  // mean visible keys per row of the lightest block
  const long long nt = (L + kTileKeys - 1) / kTileKeys;
  if (nt < 8) return;  // too short to be worth a second sample pass
  const float sfrac = (float)plan_sample_tiles(p, L) / (float)nt;
  const float base = (float)((cand + ctas - 1) / ctas);
  float best = 0.97f * base;
  int best_c = 1;
  for (int c = 2; c <= kMaxChunks; c *= 2) {
    if ((long long)cand * 2 * kBlockRows * split_row_capacity(p.cap, c) > p.split_words) break;
    if (nt / c < 4) break;
    const float cost = (float)(((long long)cand * c + ctas - 1) / ctas) * (1.f / c + sfrac);
    if (cost < best) {
      best = cost;
      best_c = c;
    }
  }
  if (best_c > 1) {
    S.nsplit = cand;
    S.nchunks = best_c;
  }
  if (nb >= ctas) return;
  // Fewer blocks than CTAs, of different lengths (a mixed decode batch): the
  // time is the heaviest block's.  Splitting only the heaviest blocks, into
  // more chunks, can shorten it where one chunk count for every block cannot
  // (the lightest block limits it).  Tiles of the i-th heaviest block, and
  // the one-wave time of a plan, in tiles:
  // (divisions by constants and float arithmetic only: thread 0 runs this
  // while the CTA waits)
  auto tiles = [&](int i) -> float {
    return (float)(((key[i] >> 32) / (uint64_t)kBlockRows + kTileKeys - 1) / (uint64_t)kTileKeys);
  };
  const float gt = (float)p.gate_target;
  auto samp = [&](int i) -> float {
    const float Li = (float)((key[i] >> 32) / (uint64_t)kBlockRows);
    if ((kBlocks ? Li / 8.f : Li) <= (float)p.gate_min) return 0.f;
    const float want = fminf(fmaxf(ceilf(Li / (4.f * gt)), 4.f), MQA_SAMPLE_ONCE ? fminf(64.f, (float)(p.cap / 64)) : 64.f);
    return (float)kSamplePasses * fminf(want, ceilf(Li / (float)kTileKeys));
  };
  const float t0 = tiles(0), s0 = samp(0);
  if (t0 < 1.25f * tiles(nb - 1)) return;  // lengths near uniform: the uniform plan is as good
  const float uniform = best_c > 1 ? base * (t0 / best_c + s0) : t0 + s0;  // base = 1 wave here
  float best_first = 0.9f * uniform;
  int bf_n = 0, bf_c = 1;
  for (int c = 2; c <= kMaxChunks; c *= 2) {
    const long long row_words = 2LL * kBlockRows * split_row_capacity(p.cap, c);
    for (int ns = 1; ns < nb; ++ns) {
      if (nb - ns + ns * c > ctas) break;
      if ((long long)ns * row_words > p.split_words) break;
      if (tiles(ns - 1) / c < 4.f) break;
      const float rest = tiles(ns) + samp(ns);
      const float t = fmaxf(t0 / c + s0, rest);
      if (t < best_first) {
        best_first = t;
        bf_n = ns;
        bf_c = c;
      }
    }
  }
  if (bf_n > 0) {
    S.nsplit = bf_n;
    S.nchunks = bf_c;
    S.split_first = 1;
  }
}

__device__ void build_order(Smem &S, const FusedParams &p) {
  const int nb = p.nblocks;
  if (nb > kMaxSortBlocks) return;  // fall back to descending block index
  uint64_t *key = reinterpret_cast<uint64_t *>(&S.kring[0][0]);
  int npow = 1;
  while (npow < nb) npow <<= 1;
  for (int b = threadIdx.x; b < npow; b += blockDim.x) {
    uint64_t v = 0;
    if (b < nb) {
      long long wsum = 0;
      for (int r = b * kBlockRows; r < min(p.rows, (b + 1) * kBlockRows); ++r) {
        const int s = max(__ldg(p.starts + r), 0), e = min(__ldg(p.ends + r), p.keys);
        wsum += e > s ? e - s : 0;
      }
      v = ((uint64_t)wsum << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)b);
    }
    key[b] = v;
  }
  __syncthreads();
  for (int k = 2; k <= npow; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < npow; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = key[i], b = key[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            key[i] = b;
            key[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int b = threadIdx.x; b < nb; b += blockDim.x) S.order[b] = (uint16_t)(0xFFFFFFFFu - (uint32_t)key[b]);
  if (threadIdx.x == 0 && p.split_max > 0) plan_split(S, p, key);
  __syncthreads();
}

// Masked selection: does main tile i of the job hold an allowed key of some
// taking-part row?  (Always true in the other compilations.)
__device__ __forceinline__ bool tile_on(const JobInfo &J, int i) {
#if MQA_MASKED
  if (!J.skip) return true;
  const int b = i + J.toff;
  return (J.tbytes[b >> 3] >> (b & 7)) & 1u;
#else
  (void)J;
  (void)i;
  return true;
#endif
}

__device__ __forceinline__ int sample_tile(const JobInfo &J, int u) {
  // (2u + 1) * nt < 2^31 for nt <= 2^17 tiles and u < 64
  return J.s_lo_t + (int)((unsigned)((2 * u + 1) * J.s_nt) / (unsigned)(2 * J.ns));
}

// ------------------------------------------------------------------ producer (warp 0)
template <bool kLogits>
__device__ void producer(Smem &S, const CUtensorMap *q_map, const CUtensorMap *k_map, const CUtensorMap *s_map,
                         const CUtensorMap *x_map,
                         const FusedParams &p, int lane) {
  const uint64_t pol_k = policy_evict_last(), pol_q = policy_evict_first();
  // claim order: whole blocks, then nsplit blocks as nchunks consecutive key chunks each
  const int nsplit = kLogits ? 0 : S.nsplit, nchunks = kLogits ? 1 : S.nchunks;
  const bool split_first = !kLogits && S.split_first;
  const int nwhole = p.nblocks - nsplit;
  const int total_jobs = kLogits ? p.nblocks * p.key_chunks : nwhole + nsplit * nchunks;
  const int ktiles_all = (p.keys + kTileKeys - 1) / kTileKeys;
  int job_iter = 0, kcount = 0;
  bool exhausted = false;
  const bool spread = !kLogits && spread_merge(S, p);
  bool claimed = false;  // spread merge: this CTA's one chunk job was taken
  if (p.stall) {  // debug: a wait that nothing satisfies, ended by the time limit
    bool ok = true;
    if (lane == 0) ok = wait_bar(S, &S.stall_bar, 0, p);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) return;
  }
  for (;;) {
    const int slot = job_iter & 1;
    bool ok = true;
    if (lane == 0) ok = wait_bar(S, &S.j_empty[slot], ((job_iter >> 1) & 1) ^ 1, p, kBackoffIdle);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) return;
    int block = -1, mode = 0, chunk = 0, kchunk = -1, bs = 0;
    uint32_t mask = (1u << kBlockRows) - 1u;
    if (lane == 0) {
      if (!kLogits) {
        const int head = *(volatile int *)&S.fifo_head;
        if (head != *(volatile int *)&S.fifo_tail) {
          __threadfence_block();
          block = S.fifo_block[head & 7];
          mask = S.fifo_mask[head & 7];
          mode = 1;
          *(volatile int *)&S.fifo_head = head + 1;
        }
      }
      if (block < 0 && !exhausted) {
        const int i = spread ? (claimed ? total_jobs : (int)blockIdx.x) : atomicAdd(p.ws + kWsClaim, 1);
        claimed = true;
        if (i < total_jobs) {
          if (kLogits) {
            block = i / p.key_chunks;
            chunk = i % p.key_chunks;
          } else {
            int oi = i;
            if (split_first) {  // the heaviest blocks' key chunks first, then the whole blocks
              if (i < nsplit * nchunks) {
                bs = i / nchunks;
                kchunk = i % nchunks;
                oi = bs;
              } else {
                oi = nsplit + (i - nsplit * nchunks);
              }
            } else if (i >= nwhole) {  // a key chunk of a split block
              bs = (i - nwhole) / nchunks;
              kchunk = (i - nwhole) % nchunks;
              oi = nwhole + bs;
            }
            block = p.nblocks <= kMaxSortBlocks ? (int)S.order[oi] : p.nblocks - 1 - oi;
          }
        } else {
          exhausted = true;
        }
      }
      if (!kLogits && block < 0 && exhausted) {
        // Every issued job must retire (selection done) before the rescan
        // queue can be declared empty.
        // Parked: no more claims and, until every issued job has retired, no
        // more TMA writes, so the epilogue warps may use the K ring and q
        // buffers as scratch to help select the last blocks' rows.
        *(volatile int *)&S.prod_parked = 1;
        __threadfence_block();
        if (wait_counter(S, &S.retired, job_iter, p)) {
          __threadfence_block();
          const int head = *(volatile int *)&S.fifo_head;
          if (head != *(volatile int *)&S.fifo_tail) {
            block = S.fifo_block[head & 7];
            mask = S.fifo_mask[head & 7];
            mode = 1;
            *(volatile int *)&S.fifo_head = head + 1;
            *(volatile int *)&S.prod_parked = 0;
            __threadfence_block();
          }
        }
      }
    }
    block = __shfl_sync(0xFFFFFFFFu, block, 0);
    mode = __shfl_sync(0xFFFFFFFFu, mode, 0);
    mask = __shfl_sync(0xFFFFFFFFu, mask, 0);
    chunk = __shfl_sync(0xFFFFFFFFu, chunk, 0);
    kchunk = __shfl_sync(0xFFFFFFFFu, kchunk, 0);
    bs = __shfl_sync(0xFFFFFFFFu, bs, 0);
    JobInfo &J = S.job[slot];
    int ntiles = 0;
    if (block >= 0) {
      const int r0 = block * kBlockRows;
      const int nrows = min(kBlockRows, p.rows - r0);
      // rows and ranges (lanes 0..7), weights (all lanes: head = lane)
      int s = 0, e = 0;
      bool part = false;
      if (lane < kBlockRows && lane < nrows) {
        const int gr = r0 + lane;
        s = __ldg(p.starts + gr);
        e = __ldg(p.ends + gr);
        if ((s < 0 || e > p.keys) && e > s) {
          atomicOr(p.ws + kWsStatus, kDevRangeClamped);
          s = max(s, 0);
          e = min(e, p.keys);
        }
        if (e < s) e = s;
        part = ((mask >> lane) & 1u) != 0;
      }
      const uint32_t pm = __ballot_sync(0xFFFFFFFFu, part);
      if (lane < kBlockRows) {
        J.start[lane] = s;
        J.end[lane] = e;
      }
#pragma unroll
      for (int r = 0; r < kBlockRows; ++r)
#pragma unroll
        for (int h = lane; h < kHeads; h += 32)
          J.w[r][h] = r < nrows ? __ldg(p.weights + (size_t)(r0 + r) * kHeads + h) : 0.f;
      if constexpr (kFold) {
        // the folded query's term scales 2^e_t (exact) and residual norm
        if (lane < kBlockRows * kFoldRowTerms) {
          const int r = lane / kFoldRowTerms, t = lane % kFoldRowTerms;
          J.fm[r][t] = r < nrows ? ldexpf(1.f, __ldg(p.fold_exps + (size_t)(r0 + r) * kFoldRowTerms + t)) : 0.f;
        }
        if (lane < kBlockRows) J.beta[lane] = lane < nrows ? __ldg(p.fold_beta + r0 + lane) : 0.f;
      }
      // key range: the union of the taking-part rows' ranges
      const bool live = part && e > s;
      int items = row_items(s, e);
      if (kMasked && lane < kBlockRows && lane < nrows) items = max(0, min(items, __ldg(p.row_items + r0 + lane)));
      if (lane < kBlockRows) J.items[lane] = items;
      int lo = live ? s : INT_MAX, hi = live ? e : 0, len = live ? items : 0;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
        len = max(len, __shfl_xor_sync(0xFFFFFFFFu, len, off));
      }
      int lo_t = 0, nt = 0, ns = 0;
      if (kLogits) {
        const int tpc = (ktiles_all + p.key_chunks - 1) / p.key_chunks;
        lo_t = chunk * tpc;
        nt = max(0, min(ktiles_all, lo_t + tpc) - lo_t);
      } else if (hi > lo) {
        lo_t = lo / kTileKeys;
        nt = (hi + kTileKeys - 1) / kTileKeys - lo_t;
        if (mode == 0 && p.force_gate == 0 && len > p.gate_min) {
          // sample about 32 gate-passing keys per row: tiles ~ 32 * L / (target * 128)
          const long long L = (long long)(hi - lo);
          long long want = (32LL * L + (long long)p.gate_target * kTileKeys - 1) /
                           ((long long)p.gate_target * kTileKeys);
          want = want < 4 ? 4 : (want > 64 ? 64 : want);
          if (MQA_SAMPLE_ONCE && want > p.cap / 64) want = p.cap / 64;  // the sample scores' room in the slab slot
          ns = (int)(want < nt ? want : nt);
        }
      }
      // samples span the whole block; a key chunk scans its share of the tiles
      const int s_lo_t = lo_t, s_nt = nt;
      if (kchunk >= 0) {
        const int tpc = (nt + nchunks - 1) / nchunks;
        const int a = min(nt, kchunk * tpc), b = min(nt, a + tpc);
        lo_t += a;
        nt = b - a;
      }
      if (lane == 0) {
        J.block = block;
        J.mode = mode;
        J.lo_t = lo_t;
        J.nt = nt;
        J.ns = ns;
        J.mask = kLogits ? ((1u << nrows) - 1u) : pm;
        J.nrows = nrows;
        J.chunk = kchunk;
        J.nchunks = kchunk >= 0 ? nchunks : 1;
        J.bs = bs;
        J.s_lo_t = s_lo_t;
        J.s_nt = s_nt;
      }
#if MQA_MASKED
      {
        // Which main tiles hold an allowed block of a taking-part row: lane
        // l covers 8-tile groups l, l + 32, ... from base (lo_t rounded down
        // to 8), one 16-byte load of 4 mask words (8 tiles) per row and group.
        const int base = lo_t & ~7, ngroups = (lo_t + nt - base + 7) >> 3;
        const bool skip = !kLogits && nt > 0 && nt <= kSkipTiles;
        int skipped = 0;
        if (skip) {
          for (int g = lane; g < ngroups; g += 32) {
            uint32_t on = 0, in = 0;
#pragma unroll
            for (int r = 0; r < kBlockRows; ++r) {
              if (!((pm >> r) & 1u)) continue;
              const uint4 w4 = __ldg(reinterpret_cast<const uint4 *>(p.mask + (size_t)(r0 + r) * p.mask_words +
                                                                     (base >> 1) + 4 * g));
              const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int k = 0; k < 8; ++k)
                if ((wv[k >> 1] >> (16 * (k & 1))) & 0xFFFFu) on |= 1u << k;
            }
            const int t0 = base + 8 * g;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (t0 + k >= lo_t && t0 + k < lo_t + nt) in |= 1u << k;
            J.tbytes[g] = (uint8_t)(on & in);
            skipped += __popc(in) - __popc(on & in);
          }
        }
        skipped = __reduce_add_sync(0xFFFFFFFFu, skipped);
        if (lane == 0) {
          J.skip = skip;
          J.toff = lo_t - base;
          if (skipped) atomicAdd(p.ws + kWsSkippedTiles, skipped);
        }
      }
#endif
      ntiles = kSamplePasses * ns + nt;
    } else if (lane == 0) {
      J.block = -1;
    }
    __syncwarp();
    if (lane == 0 && block >= 0 && ntiles > 0) {
      mbar_arrive_expect_tx(&S.j_full[slot], kQBytes);
      tma_load_2d(&S.q[slot][0], q_map, &S.j_full[slot], 0, block * kHeadCols, pol_q);
      // fold: the block's folded-query terms follow its q rows (B operand rows kHeadCols..kCols-1)
      if (kFold)
        tma_load_2d(&S.q[slot][kHeadCols * kDim], x_map, &S.j_full[slot], 0, block * kBlockRows * kFoldRowTerms, pol_q);
    } else {
      mbar_arrive(&S.j_full[slot]);
    }
    if (block < 0) return;
    if (lane == 0) {
      const JobInfo &Jc = S.job[slot];
      for (int u = 0; u < ntiles; ++u) {
        if (u >= kSamplePasses * Jc.ns && !tile_on(Jc, u - kSamplePasses * Jc.ns)) continue;
        const int tile = u < kSamplePasses * Jc.ns ? sample_tile(Jc, u < Jc.ns ? u : u - Jc.ns)
                                                   : Jc.lo_t + (u - kSamplePasses * Jc.ns);
        const int stage = kcount % kKStages;
        const int sst = kcount % kSStages;
        if (!wait_bar(S, &S.k_empty[stage], ((kcount / kKStages) & 1) ^ 1, p, kBackoffIdle)) break;
        // the tile's key scales (zero past the last key); a slot is released
        // once every epilogue warp has read it
        if (!wait_bar(S, &S.sc_empty[sst], ((kcount / kSStages) & 1) ^ 1, p, kBackoffIdle)) break;
        if constexpr (kMasked) {
          mbar_arrive_expect_tx(&S.k_full[stage], kKTileBytes);
          tma_load_2d(&S.kring[stage][0], k_map, &S.k_full[stage], 0, tile * kTileKeys, pol_k);
          // the tile's 16 blocks are half of mask word tile / 2; the box is the
          // 16-byte-aligned group of 4 words holding it, for the block's rows
          mbar_arrive_expect_tx(&S.sc_full[sst], kTileKeys * sizeof(float) + sizeof(S.mring[0]));
          tma_load_1d(&S.sring[sst][0], s_map, &S.sc_full[sst], tile * kTileKeys, pol_k);
          tma_load_2d(&S.mring[sst][0][0], x_map, &S.sc_full[sst], (tile >> 1) & ~3, Jc.block * kBlockRows, pol_k);
        } else {
          // The scales land on the K slot's barrier: the MMA issuer waits for
          // both before its MMAs, so the accumulator's full barrier, which the
          // epilogue waits for, also covers the scales.  One barrier wait per
          // tile fewer in the epilogue measured 5.7% faster at 1M keys.
          mbar_arrive_expect_tx(&S.k_full[stage], kKTileBytes + kTileKeys * sizeof(float));
          tma_load_2d(&S.kring[stage][0], k_map, &S.k_full[stage], 0, tile * kTileKeys, pol_k);
          tma_load_1d(&S.sring[sst][0], s_map, &S.k_full[stage], tile * kTileKeys, pol_k);
        }
        ++kcount;
      }
    }
    kcount = __shfl_sync(0xFFFFFFFFu, kcount, 0);
    if (aborted(S)) return;
    ++job_iter;
  }
}

// ------------------------------------------------------------------ MMA issuer (warp 1, lane 0)
__device__ void mma_issuer(Smem &S, uint32_t tmem, const FusedParams &p) {
  int job_iter = 0;
  int stage = 0, kphase = 0;  // K ring slot and the parity its full barrier completes with
  int buf = 0, tphase = 0;    // accumulator buffer and the parity of its current use
  int mcount = 0;  // tiles issued so far, over all jobs
  // Descriptors of the first K slot; a slot (and a 32-byte K step) moves the
  // start address field (bits 0-13, in 16-byte units) without carrying out of
  // it, since every shared address is below 2^18.
  const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(&S.kring[0][0]));
  for (;;) {
    const int slot = job_iter & 1;
    if (!wait_bar(S, &S.j_full[slot], (job_iter >> 1) & 1, p, kBackoffMma)) break;
    const JobInfo &J = S.job[slot];
    if (J.block < 0) break;
    const int ntiles = kSamplePasses * J.ns + J.nt;
    const uint64_t b_desc = sw128_kmajor_desc(smem_u32(&S.q[slot][0]));
    bool ok = true;
    for (int u = 0; u < ntiles && ok; ++u) {
      if (u >= kSamplePasses * J.ns && !tile_on(J, u - kSamplePasses * J.ns)) continue;
      ok = wait_bar(S, &S.k_full[stage], kphase, p, kBackoffMma) &&
           wait_bar(S, &S.t_empty[buf], tphase ^ 1, p, kBackoffMma);
      if (!ok) break;
      tc_fence_after();
      const uint64_t a_desc = a_desc0 + (uint64_t)(stage * (kKTileBytes >> 4));
      const uint32_t d = tmem + (uint32_t)(buf * kTmemStride);
#pragma unroll
      for (int kk = 0; kk < kDim / 32; ++kk)
        umma_f8(d, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), kIdesc, kk > 0 ? 1u : 0u);
      umma_commit(&S.k_empty[stage]);
      umma_commit(&S.t_full[buf]);
      // Every epilogue warp released this buffer's previous tile (two tiles
      // back) and had read that tile's key scales before: free their slot
      // here, after the MMAs are issued, instead of one arrival per epilogue
      // warp and tile (1M keys: 0.7% faster with the separate gated-scan
      // loop).  The masked scan's epilogue releases its slots itself.
      if (!kMasked && mcount >= kTmemBufs) mbar_arrive(&S.sc_empty[(mcount - kTmemBufs) % kSStages]);
      ++mcount;
      if (++stage == kKStages) {
        stage = 0;
        kphase ^= 1;
      }
      if (++buf == kTmemBufs) {
        buf = 0;
        tphase ^= 1;
      }
    }
    if (!ok) break;
    umma_commit(&S.j_empty[slot]);
    ++job_iter;
  }
  // Make sure no MMA is still writing TMEM when the CTA releases it.
  umma_commit(&S.drain);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(&S.drain, 0)) {
    if ((long long)(globaltimer_ns() - t0) > p.timeout_ns) {
      raise_timeout(S, p);
      break;
    }
  }
}

// One row of a finished key chunk: move the records of quadrant segments 1..3
// down behind segment 0's, so the chunk's candidates form one run.  Returns
// the run's length, or 4 * seglen + 1 when a quadrant segment overflowed.
// Out of line: it runs once per chunk and keeps its registers out of the
// epilogue's tile loop.
__device__ __noinline__ int pack_chunk_row(uint32_t *keys_r, int32_t *idx_r, const int *segcnt, int seglen,
                                           int lane) {
  int dst = segcnt[0];
  if (dst > seglen) return kQuads * seglen + 1;
  for (int q = 1; q < kQuads; ++q) {
    const int n = segcnt[q];
    if (n > seglen) return kQuads * seglen + 1;
    // 128 records per round, all read before any is written: the run lies
    // below the source, so a round's writes never reach records still unread
    for (int i0 = 0; i0 < n; i0 += 128) {
      uint32_t kv[4];
      int32_t iv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + 32 * j + lane;
        kv[j] = i < n ? __ldcg(keys_r + q * seglen + i) : 0u;
        iv[j] = i < n ? __ldcg(idx_r + q * seglen + i) : 0;
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + 32 * j + lane;
        if (i < n) {
          keys_r[dst + i] = kv[j];
          idx_r[dst + i] = iv[j];
        }
      }
      __syncwarp();
    }
    dst += n;
  }
  return dst;
}

// Selection work shared by the selection warps and, at the end, the epilogue
// warps (defined with the selection below).
__device__ void work_slot_rows(Smem &S, const FusedParams &p, int slot, int use, int *hist, uint32_t *lk,
                               int32_t *li, int lane);
#if MQA_PAIR_HELPERS
__device__ void work_slot_rows_pair(Smem &S, const FusedParams &p, int slot, int use, int m, int member, int *hist,
                                    uint32_t *lk, int32_t *li, int lane);
__device__ void work_slot_rows_group(Smem &S, const FusedParams &p, int slot, int ew, int lane);
#endif
// Scratch of one helping epilogue warp: a 256-bin histogram and the list.
constexpr int kHelperScratchBytes = 1024 + 8 * kSelList;
// The epilogue group of a spread merge: the leader's histogram and list, then
// four histogram copies per warp.
static_assert(kHelperScratchBytes + kEpiWarps * 4 * kScoreBins * (int)sizeof(int) <=
                  (int)(sizeof(Smem::kring) + sizeof(Smem::q)),
              "the group's scratch fits the idle K ring and q buffers");
static_assert(kEpiWarps * kHelperScratchBytes <= (int)(sizeof(Smem::kring) + sizeof(Smem::q)),
              "helper scratch exceeds the K ring and q buffers");

#if MQA_FOLD
// Classification of a row for the fold ("weights unsafe to scale", vLLM pull
// request #60618, "What this PR does", Exact rescan bullet).  The fold's error
// on any of the row's scores is at most (scale_j / 2) beta |k_j|_2 <=
// beta * key_norm / 2 (Cauchy-Schwarz on the folded query's residual).  The
// row is safe when that bound stays below 2^-16 of the row's largest |score|,
// of which `seen` (some computed |score| of the row) less the bound is a lower
// bound.  Non-finite weights or scales make the bound NaN or inf: unsafe.
// Lane 0 records the bound in millionths of the allowed error (the largest
// over rows) and, when `count`, counts unsafe rows.  Warp-uniform result.
__device__ bool fold_safe(const FusedParams &p, float key_norm, float beta, float seen, bool count, int lane) {
  const float bound = 0.5f * beta * key_norm;
  const bool safe = p.force_unsafe == 0 && bound * 65537.f <= seen;
  if (lane == 0) {
    const float rel = bound * 65537.f / seen;
    const int ppm = rel < 2000.f ? (int)ceilf(rel * 1e6f) : INT_MAX;  // inf and NaN: INT_MAX
    atomicMax(p.ws + kWsFoldBound, ppm);
    if (!safe && count) atomicAdd(p.ws + kWsUnsafeRows, 1);
  }
  return safe;
}
#endif

// ------------------------------------------------------------------ epilogue (warps 4 and up)
template <bool kLogits>
__device__ void epilogue(Smem &S, uint32_t tmem, const FusedParams &p, int warp, int lane) {
  const int ew = warp - kEpiWarp0;  // 0 .. kEpiWarps - 1
  const int quad = warp & 3;        // TMEM lane quadrant this warp may access
  const int rbase = kRowsPerWarp * (ew >> 2);  // this warp's rows: rbase .. rbase + kRowsPerWarp - 1
  const bool gate_warp = ew < kBlockRows;        // the first kBlockRows warps also own row ew's gate / compaction
  const bool spread = !kLogits && spread_merge(S, p);
  const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
  const float NEG_INF = -INFINITY;
  const int cap = p.cap, seg = p.cap / kQuads;
  const uint32_t lt = lanemask_lt();
  int job_iter = 0, tcount = 0;
  for (;;) {
    const int slot = job_iter & 1;
    bool ok = true;
    if (lane == 0) ok = wait_bar(S, &S.j_full[slot], (job_iter >> 1) & 1, p);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (bar_or(kEpiBarrier, kEpiThreads, !ok || aborted(S))) break;
    const JobInfo &J = S.job[slot];
    if (J.block < 0) {
      // hand the end marker to the selection warps through the next slot
      if (!kLogits && ew == 0 && lane == 0 && wait_bar(S, &S.s_empty[slot], ((job_iter >> 1) & 1) ^ 1, p)) {
        S.sel[slot].block = -1;
        mbar_arrive(&S.s_full[slot]);
      }
      break;
    }
    if (!kLogits) {
      if (lane == 0) ok = wait_bar(S, &S.s_empty[slot], ((job_iter >> 1) & 1) ^ 1, p);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      // per-row state for this scan: warp ew owns row ew
      if (gate_warp && lane == 0) {
        const int n = J.items[ew];
        float t0 = NEG_INF;
        if (J.ns == 0 && J.mode == 0 && p.force_gate == 1 && n > 0) t0 = INFINITY;
        S.tau[ew] = t0;
        S.ref[ew] = 0;
        S.ref_frozen[ew] = 0;
        S.msample[ew] = 0;
        S.smax[ew] = 0;
        S.smin[ew] = 0xFFFFFFFFu;
        S.binv[ew] = 0.f;
        S.unsafe[ew] = 0;
        S.classified[ew] = 0;
      }
      if (gate_warp)
        for (int b = lane; b < kGateBins; b += 32) S.hist[ew][b] = 0;
    }
    if (bar_or(kEpiBarrier, kEpiThreads, !ok || aborted(S))) break;
    int cnt[kRowsPerWarp];
    // tiles [f_lo, f_hi) lie inside the range of every row of this warp
    // (none when one of its rows does not take part)
    int f_lo = 0, f_hi = INT_MAX;
    bool act[kRowsPerWarp];
    float tau[kRowsPerWarp];
    HeadW W[kRowsPerWarp];
#if MQA_FOLD
    // the scales 2^e of this lane's two fold terms, for the row they belong to
    FoldM FM;
    {
      const int c = lane & 3;
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr)
        FM.m[rr] = (c >> 1) == rr ? *reinterpret_cast<const float2 *>(&J.fm[rbase + rr][2 * (c & 1)])
                                  : make_float2(0.f, 0.f);
    }
#endif
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int r = rbase + rr;
      act[rr] = ((J.mask >> r) & 1u) != 0;
      f_lo = max(f_lo, (J.start[r] + kTileKeys - 1) / kTileKeys);
      f_hi = min(f_hi, act[rr] ? J.end[r] / kTileKeys : 0);
      tau[rr] = kLogits ? NEG_INF : S.tau[r];
      cnt[rr] = 0;
#pragma unroll
      for (int i = 0; i < 4 * kHeadGroups; ++i) {
        const float2 wv = *reinterpret_cast<const float2 *>(&J.w[r][8 * i + 2 * (lane & 3)]);
        W[rr].w[i] = !kFold && i < MQA_RELU_ALU_CHUNKS ? make_float2(2.f * wv.x, 2.f * wv.y) : wv;
      }
    }
    const int ns = J.ns, ns2 = kSamplePasses * J.ns, ntiles = kSamplePasses * J.ns + J.nt, mode = J.mode;
    const int block = J.block;
    // this warp's candidate segment of row rbase; row rbase + rr's is rr * row_stride further.
    // Whole block: the CTA's slab slot, [rows][quadrant segments of seg].  Key
    // chunk c of a split block: the split slab, [rows][chunks][quadrant segments].
    uint32_t *seg_keys;
    int32_t *seg_idx;
    int row_stride, seglen;
    if (J.chunk < 0) {
      uint32_t *base = p.slab + ((size_t)(blockIdx.x * kSlots + slot) * 2 * kBlockRows) * (size_t)cap;
      row_stride = cap;
      seglen = seg;
      seg_keys = base + (size_t)rbase * cap + quad * seg;
      seg_idx = reinterpret_cast<int32_t *>(base + (size_t)kBlockRows * cap) + (size_t)rbase * cap + quad * seg;
    } else {
      const int rcap = (int)split_row_capacity(cap, J.nchunks);
      uint32_t *base = p.split_slab + (size_t)J.bs * 2 * kBlockRows * rcap;
      row_stride = rcap;
      seglen = rcap / (kQuads * J.nchunks);
      const int off = rbase * rcap + (J.chunk * kQuads + quad) * seglen;
      seg_keys = base + off;
      seg_idx = reinterpret_cast<int32_t *>(base + (size_t)kBlockRows * rcap) + off;
    }
    bool bail = false;
    // key of this thread within a tile
    const int kown = quad * 32 + owned_key(lane);
    // One tile: wait for its accumulators and scales, score this lane's key for
    // the warp's rows (masked to each row's range), release TMEM and scales.
    auto score_tile = [&](int tile, float (&sv)[kRowsPerWarp]) -> bool {
      const int buf = tcount % kTmemBufs, sst = tcount % kSStages;
      const int key = tile * kTileKeys + kown;
      bool ok = wait_bar(S, &S.t_full[buf], (tcount / kTmemBufs) & 1, p);
      if constexpr (kMasked) ok = wait_bar(S, &S.sc_full[sst], (tcount / kSStages) & 1, p) && ok;
      tc_fence_after();
      const float hsc = 0.5f * S.sring[sst][kown];
      float raw[kRowsPerWarp];
#if MQA_FOLD
      {
        const uint32_t tb = tmem + lane_addr + (uint32_t)(buf * kTmemStride);
        const uint32_t hb = tb + (uint32_t)(rbase * kHeads), fb = tb + (uint32_t)(kHeadCols + rbase * kFoldRowTerms);
        // exact rescans score directly; every other scan through the fold
        if (mode == 1) score_rows_fold<true>(&S.t_empty[buf], hb, fb, W, FM, hsc, lane, raw);
        else score_rows_fold<false>(&S.t_empty[buf], hb, fb, W, FM, hsc, lane, raw);
      }
#else
      const uint32_t base = tmem + lane_addr + (uint32_t)(buf * kCols + rbase * kHeads);
      score_rows(&S.t_empty[buf], base, W, hsc, lane, raw);
#endif
      uint32_t mw[kRowsPerWarp];
      if constexpr (kMasked) {
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) mw[rr] = S.mring[sst][rbase + rr][(tile >> 1) & 3];
      }
      if (kMasked && lane == 0) mbar_arrive(&S.sc_empty[sst]);
      if (tile >= f_lo && tile < f_hi) {
        // the tile lies inside every row's range: no per-key mask
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) sv[rr] = raw[rr];
      } else {
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const int r = rbase + rr;
          sv[rr] = (act[rr] && key >= J.start[r] && key < J.end[r]) ? raw[rr] : NEG_INF;
        }
      }
      if constexpr (kMasked) {
        // keys of blocks the row's mask leaves out are not visible
        const int bit = ((tile & 1) << 4) + (kown >> 3);
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr)
          if (!((mw[rr] >> bit) & 1u)) sv[rr] = NEG_INF;
      }
      if constexpr (kBlocks) {
        // the 8 keys of a block sit in the lanes with the same lane % 4 (key
        // offset lane / 4 within the block): the block's score is their
        // largest, kept by the lane holding the block's first key (lane < 4)
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          float m = sv[rr];
          m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
          m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
          m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
          sv[rr] = lane < 4 ? m : NEG_INF;
        }
      }
      ++tcount;
      return ok;
    };
#if MQA_SAMPLE_ONCE
    // ---- sample tiles, scored once.  Each thread keeps its key's scores of
    // the warp's rows in the job's slab slot (free until the main scan: the
    // slot's last selection ended before the job began) and re-reads only what
    // it wrote, so the gate's coarse and fine passes need neither a second
    // scoring of the tiles nor a barrier per tile.  Row r's score of key k of
    // sample tile u is word (r * ns + u) * kTileKeys + k; ns <= cap / 64 keeps
    // the 8 rows inside the slot's 16 * cap words.
    do {
      if (ns == 0) break;
      // this thread's words: row rbase + rr, sample tile u at samp[(rr * ns + u) * kTileKeys]
      float *const samp = reinterpret_cast<float *>(p.slab + (size_t)(blockIdx.x * kSlots + slot) * 2 * kBlockRows * (size_t)cap) +
                          (size_t)rbase * ns * kTileKeys + kown;
      for (int u = 0; u < ns; ++u) {
        float sv[kRowsPerWarp];
        score_tile(sample_tile(J, u), sv);
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) samp[(rr * ns + u) * kTileKeys] = sv[rr];
      }
      // coarse pass, step A: each row's reference is its largest sample score
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = rbase + rr;
        float mx = NEG_INF;
        for (int u = 0; u < ns; ++u) mx = fmaxf(mx, samp[(rr * ns + u) * kTileKeys]);
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, mx > NEG_INF ? f2key(mx) : 0u);
        if (act[rr] && lane == 0 && m) atomicMax(&S.ref[r], m);
      }
      if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
      // step B: log-binned histogram of each sample score's distance to the reference
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = rbase + rr;
        const uint32_t ref = S.ref[r];
        int nvis = 0;
        if (act[rr] && ref) {
#pragma unroll 1
          for (int u = 0; u < ns; ++u) {
            const float v = samp[(rr * ns + u) * kTileKeys];
            if (v > NEG_INF) {
              atomicAdd(&S.hist[r][gate_bin(f2key(v), ref)], 1);
              ++nvis;
            }
          }
        }
        nvis = __reduce_add_sync(0xFFFFFFFFu, nvis);
        if (lane == 0 && nvis) atomicAdd(&S.msample[r], nvis);
      }
      if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
      // coarse bin of row ew that holds the target sample rank j
      if (gate_warp) {
        const int r = ew;
        const int n = J.items[r];
        const int m = S.msample[r];
        int on = 0, above = 0, jw = 0;
        uint32_t klo = 0, khi = 0;
        if (((J.mask >> r) & 1u) && n > p.gate_min && m > 0) {
          jw = (int)max(1LL, ((long long)m * p.gate_target + n - 1) / n);
          constexpr int kPer = kGateBins / 32;
          int c[kPer], tot = 0;
#pragma unroll
          for (int j = 0; j < kPer; ++j) {
            c[j] = S.hist[r][kPer * lane + j];
            tot += c[j];
          }
          int incl = tot;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int vv = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += vv;
          }
          const int excl = incl - tot;
          const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < jw && jw <= incl);
          if (bm) {
            const int src = __ffs(bm) - 1;
            int bin = 0, run_before = 0;
            if (lane == src) {
              int run = excl;
#pragma unroll
              for (int j = 0; j < kPer; ++j) {
                if (run + c[j] >= jw) { bin = kPer * lane + j; run_before = run; break; }
                run += c[j];
              }
            }
            bin = __shfl_sync(0xFFFFFFFFu, bin, src);
            above = __shfl_sync(0xFFFFFFFFu, run_before, src);
            const uint32_t ref = S.ref[r];
            if (bin == 128) {
              klo = khi = ref;
            } else if (bin > 128) {  // keys ref - d for d in [lo, hi)
              const uint64_t lo = dist_bin_lo(bin - 128), hi = dist_bin_hi(bin - 128);
              khi = ref - (uint32_t)lo;
              klo = (uint64_t)ref >= hi - 1 ? ref - (uint32_t)(hi - 1) : 0u;
            } else {  // keys ref + d for d in [lo, hi)
              const uint64_t lo = dist_bin_lo(128 - bin), hi = dist_bin_hi(128 - bin);
              klo = ref + (uint32_t)lo;
              khi = (uint64_t)ref + hi - 1 > 0xFFFFFFFFull ? 0xFFFFFFFFu : ref + (uint32_t)(hi - 1);
            }
            on = 1;
          }
        }
        __syncwarp();
        for (int b2 = lane; b2 < kGateBins; b2 += 32) S.hist[r][b2] = 0;
        if (lane == 0) {
          S.g_on[r] = on;
          S.g_above[r] = above;
          S.g_j[r] = jw;
          S.g_klo[r] = klo;
          S.g_khi[r] = khi;
          S.tau[r] = NEG_INF;
        }
      }
      if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
      if (ew == 0 && lane == 0) atomicAdd(p.ws + kWsSampleTiles, ns);
      // fine pass: 256 linear sub-bins of the coarse bin, so the gate lands on
      // the target sample rank
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = rbase + rr;
        if (!act[rr]) continue;
        const bool on = S.g_on[r] != 0;
        const uint32_t klo = S.g_klo[r], khi = S.g_khi[r];
        const uint64_t width = (uint64_t)(khi - klo) + 1;
        uint32_t mx = 0, mn = 0xFFFFFFFFu;
#pragma unroll 1
        for (int u = 0; u < ns; ++u) {
          const float v = samp[(rr * ns + u) * kTileKeys];
          if (v > NEG_INF) {
            const uint32_t kv = f2key(v);
            mx = max(mx, kv);
            mn = min(mn, kv);
            if (on && kv >= klo && kv <= khi) atomicAdd(&S.hist[r][(int)(((uint64_t)(khi - kv) * 256) / width)], 1);
          }
        }
        mx = __reduce_max_sync(0xFFFFFFFFu, mx);
        if (lane == 0 && mx) atomicMax(&S.smax[r], mx);
        if constexpr (kFold) {
          mn = __reduce_min_sync(0xFFFFFFFFu, mn);
          if (lane == 0 && mn != 0xFFFFFFFFu) atomicMin(&S.smin[r], mn);
        }
      }
      if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
      if (gate_warp) {
        const int r = ew;
        float t = NEG_INF;
        if (S.g_on[r]) {
          const int need = S.g_j[r] - S.g_above[r];
          const uint32_t klo = S.g_klo[r], khi = S.g_khi[r];
          int c[8], tot = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            c[j] = S.hist[r][8 * lane + j];
            tot += c[j];
          }
          int incl = tot;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int vv = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += vv;
          }
          const int excl = incl - tot;
          const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < need && need <= incl);
          if (bm) {
            const int src = __ffs(bm) - 1;
            int sub = 0;
            if (lane == src) {
              int run = excl;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                run += c[j];
                if (run >= need) { sub = 8 * lane + j; break; }
              }
            }
            sub = __shfl_sync(0xFFFFFFFFu, sub, src);
            // pass every key inside sub-bins 0..sub (and everything above the coarse bin)
            const uint64_t width = (uint64_t)(khi - klo) + 1;
            const uint64_t drop = ((uint64_t)(sub + 1) * width + 255) / 256;
            t = (uint64_t)khi >= drop ? key2f(khi - (uint32_t)drop) : NEG_INF;
          }
        }
#if MQA_FOLD
        // A row that needs the fold (more visible keys than top-k) is
        // classified from its samples' largest |score|; an unsafe row emits
        // nothing, so it under-fills and is rescanned with the direct sum.
        if (((J.mask >> r) & 1u) && J.mode == 0 && J.items[r] > p.topk && S.smax[r] != 0) {
          // the largest |score| among the samples: at the top or the bottom
          const float seen = fmaxf(fabsf(key2f(S.smax[r])), fabsf(key2f(S.smin[r])));
          const bool safe = fold_safe(p, S.key_norm, J.beta[r], seen, J.chunk <= 0, lane);
          if (!safe) t = INFINITY;
          if (lane == 0) {
            S.unsafe[r] = !safe;
            S.classified[r] = 1;
          }
        }
#endif
        if (lane == 0) {
          S.tau[r] = t;
          // linear score bins from the gate to the largest sample score
          const float smax = S.smax[r] ? key2f(S.smax[r]) : NEG_INF;
          S.binv[r] = (t > NEG_INF && smax > t) ? __fdiv_rn((float)kScoreBins, __fsub_rn(smax, t)) : 0.f;
        }
      }
      if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) tau[rr] = S.tau[rbase + rr];
    } while (0);
#else
    // ---- sample tiles: coarse then fine pass of the gate
    for (int u = 0; u < ns2 && !bail; ++u) {
      const int tile = sample_tile(J, u < ns ? u : u - ns);
      float sv[kRowsPerWarp];
      score_tile(tile, sv);
      if (u < ns) {
        // coarse pass, step A: reference maximum from the row's first sample
        // tile with visible keys
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const int r = rbase + rr;
          if (act[rr] && !S.ref_frozen[r]) {
            const uint32_t kv = sv[rr] > NEG_INF ? f2key(sv[rr]) : 0u;
            const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, kv);
            if (lane == 0 && m) atomicMax(&S.ref[r], m);
          }
        }
        if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
        // step B: log-binned histogram of the position relative to the reference
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const int r = rbase + rr;
          if (act[rr]) {
            const uint32_t ref = S.ref[r];
            const bool vis = sv[rr] > NEG_INF;
            if (ref && vis) atomicAdd(&S.hist[r][gate_bin(f2key(sv[rr]), ref)], 1);
            const uint32_t bv = __ballot_sync(0xFFFFFFFFu, vis && ref != 0);
            if (lane == 0 && bv) atomicAdd(&S.msample[r], __popc(bv));
            if (quad == 0 && lane == 0) S.ref_frozen[r] = ref != 0;
          }
        }
        if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
        if (u == ns - 1) {
          // coarse bin of row ew that holds the target sample rank j
          if (gate_warp) {
          const int r = ew;
          const int n = J.items[r];
          const int m = S.msample[r];
          int on = 0, above = 0, jw = 0;
          uint32_t klo = 0, khi = 0;
          if (((J.mask >> r) & 1u) && n > p.gate_min && m > 0) {
            jw = (int)max(1LL, ((long long)m * p.gate_target + n - 1) / n);
            constexpr int kPer = kGateBins / 32;
            int c[kPer], tot = 0;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
              c[j] = S.hist[r][kPer * lane + j];
              tot += c[j];
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
              const int vv = __shfl_up_sync(0xFFFFFFFFu, incl, off);
              if (lane >= off) incl += vv;
            }
            const int excl = incl - tot;
            const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < jw && jw <= incl);
            if (bm) {
              const int src = __ffs(bm) - 1;
              int bin = 0, run_before = 0;
              if (lane == src) {
                int run = excl;
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                  if (run + c[j] >= jw) { bin = kPer * lane + j; run_before = run; break; }
                  run += c[j];
                }
              }
              bin = __shfl_sync(0xFFFFFFFFu, bin, src);
              above = __shfl_sync(0xFFFFFFFFu, run_before, src);
              const uint32_t ref = S.ref[r];
              if (bin == 128) {
                klo = khi = ref;
              } else if (bin > 128) {  // keys ref - d for d in [lo, hi)
                const uint64_t lo = dist_bin_lo(bin - 128), hi = dist_bin_hi(bin - 128);
                khi = ref - (uint32_t)lo;
                klo = (uint64_t)ref >= hi - 1 ? ref - (uint32_t)(hi - 1) : 0u;
              } else {  // keys ref + d for d in [lo, hi)
                const uint64_t lo = dist_bin_lo(128 - bin), hi = dist_bin_hi(128 - bin);
                klo = ref + (uint32_t)lo;
                khi = (uint64_t)ref + hi - 1 > 0xFFFFFFFFull ? 0xFFFFFFFFu : ref + (uint32_t)(hi - 1);
              }
              on = 1;
            }
          }
          __syncwarp();
          for (int b2 = lane; b2 < kGateBins; b2 += 32) S.hist[r][b2] = 0;
          if (lane == 0) {
            S.g_on[r] = on;
            S.g_above[r] = above;
            S.g_j[r] = jw;
            S.g_klo[r] = klo;
            S.g_khi[r] = khi;
            S.tau[r] = NEG_INF;
          }
          }
          if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
          if (ew == 0 && lane == 0) atomicAdd(p.ws + kWsSampleTiles, ns2);
        }
        continue;
      }
      {
        // fine pass over the same sample tiles: 256 linear sub-bins of the
        // coarse bin, so the gate lands on the target sample rank
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const int r = rbase + rr;
          if (act[rr]) {
            const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, sv[rr] > NEG_INF ? f2key(sv[rr]) : 0u);
            if (lane == 0 && m) atomicMax(&S.smax[r], m);
            if constexpr (kFold) {
              const uint32_t n = __reduce_min_sync(0xFFFFFFFFu, sv[rr] > NEG_INF ? f2key(sv[rr]) : 0xFFFFFFFFu);
              if (lane == 0 && n != 0xFFFFFFFFu) atomicMin(&S.smin[r], n);
            }
          }
          if (act[rr] && S.g_on[r] && sv[rr] > NEG_INF) {
            const uint32_t kv = f2key(sv[rr]), klo = S.g_klo[r], khi = S.g_khi[r];
            if (kv >= klo && kv <= khi) {
              const uint64_t width = (uint64_t)(khi - klo) + 1;
              atomicAdd(&S.hist[r][(int)(((uint64_t)(khi - kv) * 256) / width)], 1);
            }
          }
        }
        if (u == ns2 - 1) {
          if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
          if (gate_warp) {
          const int r = ew;
          float t = NEG_INF;
          if (S.g_on[r]) {
            const int need = S.g_j[r] - S.g_above[r];
            const uint32_t klo = S.g_klo[r], khi = S.g_khi[r];
            int c[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              c[j] = S.hist[r][8 * lane + j];
              tot += c[j];
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
              const int vv = __shfl_up_sync(0xFFFFFFFFu, incl, off);
              if (lane >= off) incl += vv;
            }
            const int excl = incl - tot;
            const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < need && need <= incl);
            if (bm) {
              const int src = __ffs(bm) - 1;
              int sub = 0;
              if (lane == src) {
                int run = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  run += c[j];
                  if (run >= need) { sub = 8 * lane + j; break; }
                }
              }
              sub = __shfl_sync(0xFFFFFFFFu, sub, src);
              // pass every key inside sub-bins 0..sub (and everything above the coarse bin)
              const uint64_t width = (uint64_t)(khi - klo) + 1;
              const uint64_t drop = ((uint64_t)(sub + 1) * width + 255) / 256;
              t = (uint64_t)khi >= drop ? key2f(khi - (uint32_t)drop) : NEG_INF;
            }
          }
#if MQA_FOLD
          // A row that needs the fold (more visible keys than top-k) is
          // classified from its samples' largest |score|; an unsafe row emits
          // nothing, so it under-fills and is rescanned with the direct sum.
          if (((J.mask >> r) & 1u) && J.mode == 0 && J.items[r] > p.topk && S.smax[r] != 0) {
            // the largest |score| among the samples: at the top or the bottom
            const float seen = fmaxf(fabsf(key2f(S.smax[r])), fabsf(key2f(S.smin[r])));
            const bool safe = fold_safe(p, S.key_norm, J.beta[r], seen, J.chunk <= 0, lane);
            if (!safe) t = INFINITY;
            if (lane == 0) {
              S.unsafe[r] = !safe;
              S.classified[r] = 1;
            }
          }
#endif
          if (lane == 0) {
            S.tau[r] = t;
            // linear score bins from the gate to the largest sample score
            const float smax = S.smax[r] ? key2f(S.smax[r]) : NEG_INF;
            S.binv[r] = (t > NEG_INF && smax > t) ? __fdiv_rn((float)kScoreBins, __fsub_rn(smax, t)) : 0.f;
          }
          }
          if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
#pragma unroll
          for (int rr = 0; rr < kRowsPerWarp; ++rr) tau[rr] = S.tau[rbase + rr];
        }
        continue;
      }
    }
#endif
    // ---- main tiles
    const int lo_t = J.lo_t;
    if (!kLogits && mode == 0 && !bail) {
      // Gated or plain scan: a loop of its own, without the rescan's
      // compaction steps and bail-out test (1M keys: 0.7% faster).
      for (int u = ns2; u < ntiles; ++u) {
        if (!tile_on(J, u - ns2)) continue;
        const int tile = lo_t + (u - ns2);
        const int key = tile * kTileKeys + kown;
        float sv[kRowsPerWarp];
        score_tile(tile, sv);
        if constexpr (kAnyGate) {
          bool anyp = false;
#pragma unroll
          for (int rr = 0; rr < kRowsPerWarp; ++rr) anyp |= sv[rr] > tau[rr];
          if (!__any_sync(0xFFFFFFFFu, anyp)) continue;
        }
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const bool pass = sv[rr] > tau[rr];
          const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pass);
          if (bal) {
            const int pos = cnt[rr] + __popc(bal & lt);
            if (pass && pos < seglen) {
              const int o = rr * row_stride + pos;
              __stcg(&seg_keys[o], f2key(sv[rr]));
              __stcg(&seg_idx[o], key);
            }
            cnt[rr] += __popc(bal);
          }
        }
      }
    } else
    for (int u = ns2; u < ntiles && !bail; ++u) {
      if (!tile_on(J, u - ns2)) continue;
      const int tile = lo_t + (u - ns2);
      const int key = tile * kTileKeys + kown;
      float sv[kRowsPerWarp];
      score_tile(tile, sv);
      if (kLogits) {
        if (key < p.keys) {
#pragma unroll
          for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            if (act[rr]) {
              const size_t row = (size_t)block * kBlockRows + rbase + rr;
              p.logits[row * (size_t)p.keys + key] = sv[rr];
            }
          }
        }
        continue;
      }
      // main scan: append keys above the gate to this warp's segment of each row
      // (a private counter per warp: no atomics)
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const bool pass = sv[rr] > tau[rr];
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pass);
        if (bal) {
          const int pos = cnt[rr] + __popc(bal & lt);
          if (pass && pos < seglen) {
            const int o = rr * row_stride + pos;
            __stcg(&seg_keys[o], f2key(sv[rr]));
            __stcg(&seg_idx[o], key);
          }
          cnt[rr] += __popc(bal);
        }
      }
      if (mode == 1) {
        // exact rescan: keep each row's segments bounded by compacting the row
        // to its top-k (into segment 0) before any segment can overflow
        if (lane == 0) {
#pragma unroll
          for (int rr = 0; rr < kRowsPerWarp; ++rr) S.segcnt[rbase + rr][quad] = cnt[rr];
        }
        if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
        if (gate_warp) {
        const int r = ew;
        // rescans are whole-block jobs: the CTA's slab slot
        uint32_t *base = p.slab + ((size_t)(blockIdx.x * kSlots + slot) * 2 * kBlockRows) * (size_t)cap;
        RowSlab R;
        R.keys = base + (size_t)r * cap;
        R.idx = reinterpret_cast<int32_t *>(base + (size_t)kBlockRows * cap) + (size_t)r * cap;
        R.seg = seg;
        R.nseg = kQuads;
        R.c = &S.segcnt[r][0];
        int mx = 0;
#pragma unroll
        for (int q = 0; q < kQuads; ++q) mx = max(mx, S.segcnt[r][q]);
        if (((J.mask >> r) & 1u) && mx + 32 > seg) {
          int take_eq = 0;
          const uint32_t T = warp_radix_select(R, p.topk, &S.hist[r][0], lane, &take_eq);
          warp_emit<true>(R, T, take_eq, false, nullptr, 0, p.topk, lane);
          __syncwarp();
          if (lane == 0) {
            S.segcnt[r][0] = p.topk;
            for (int q = 1; q < kQuads; ++q) S.segcnt[r][q] = 0;
            S.tau[r] = key2f(T);
            atomicAdd(p.ws + kWsCompactions, 1);
          }
        }
        }
        __threadfence_block();
        if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) { bail = true; break; }
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          tau[rr] = S.tau[rbase + rr];
          cnt[rr] = S.segcnt[rbase + rr][quad];
        }
      }
    }
    if (!kLogits && lane == 0) {
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) S.segcnt[rbase + rr][quad] = cnt[rr];
    }
    // slab writes of every epilogue warp precede the hand-over (device scope:
    // another CTA may select a split block's candidates)
    __threadfence();
    if (bar_or(kEpiBarrier, kEpiThreads, bail || aborted(S))) break;
    if (!kLogits && J.chunk >= 0) {
      // A key chunk publishes its rows' segment counts.  Up to 8 chunks keep
      // the four quadrant segments (at most 32 per row); past that each row's
      // quadrant segments are packed into one run per chunk (warp ew packs row
      // ew), and a row whose quadrant segment overflowed publishes a length
      // past the run's room.
      if (J.nchunks <= 8) {
        if (ew == 0 && lane < kBlockRows * kQuads)
          p.split_cnt[((size_t)J.bs * kBlockRows + (lane >> 2)) * 32 + J.chunk * kQuads + (lane & 3)] =
              S.segcnt[lane >> 2][lane & 3];
      } else if (gate_warp) {
        const int r = ew, rcap = row_stride;
        uint32_t *keys_r = p.split_slab + (size_t)J.bs * 2 * kBlockRows * rcap + (size_t)r * rcap +
                           (size_t)J.chunk * kQuads * seglen;
        const int n = pack_chunk_row(keys_r, reinterpret_cast<int32_t *>(keys_r + (size_t)kBlockRows * rcap),
                                     &S.segcnt[r][0], seglen, lane);
        if (lane == 0) p.split_cnt[((size_t)J.bs * kBlockRows + r) * 32 + J.chunk] = n;
      }
      __threadfence();
      if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) break;
    }
    if (!kLogits) {
      if (ew == 0) {
        SelSlot &Q = S.sel[slot];
        // The CTA that finishes a split block's last chunk selects the block
        // over every chunk's run (one segment per chunk); the others hand the
        // selection warps an empty job.
        bool merge = true, have = true;
        const bool packed = J.chunk >= 0 && J.nchunks > 8;
        const int nseg = J.chunk < 0 ? kQuads : (packed ? J.nchunks : kQuads * J.nchunks);
        if (J.chunk >= 0) {
          int32_t *cnt_g = p.split_cnt + (size_t)J.bs * kBlockRows * 32;
          int old = 0;
          if (lane == 0) old = atomicAdd(p.split_done + J.bs, 1);
          old = __shfl_sync(0xFFFFFFFFu, old, 0);
          merge = old == J.nchunks - 1;
          have = merge;
          if (spread && !merge) {
            // a spread merge: this chunk's CTA also selects rows of the block
            // once its last chunk is in
            bool okw = true;
            if (lane == 0) okw = wait_global(S, p.split_done + J.bs, J.nchunks, p);
            have = __shfl_sync(0xFFFFFFFFu, okw, 0) != 0;
          }
          if (have) {
            __threadfence();
            for (int i = lane; i < kBlockRows * nseg; i += 32)
              Q.segcnt[i / nseg][i % nseg] = __ldcg(cnt_g + (i / nseg) * 32 + i % nseg);
          }
        } else {
          if (lane < kBlockRows * kQuads) Q.segcnt[lane >> 2][lane & 3] = S.segcnt[lane >> 2][lane & 3];
        }
        if (lane < kBlockRows) {
          Q.start[lane] = J.start[lane];
          Q.n[lane] = J.items[lane];
          Q.gated[lane] = S.tau[lane] > NEG_INF;
          Q.blo[lane] = S.tau[lane];
          Q.binv[lane] = S.binv[lane];
          Q.binned[lane] = J.mode == 0 && S.tau[lane] > NEG_INF;
          Q.unsafe[lane] = kFold && J.mode == 0 && S.unsafe[lane];
          // rows the gate did not classify that may still need the fold's scores
          Q.check[lane] = kFold && J.mode == 0 && !S.classified[lane] && J.items[lane] > p.topk;
          Q.beta[lane] = kFold ? J.beta[lane] : 0.f;
        }
        if (lane == 0) {
          Q.block = J.block;
          Q.mode = J.mode;
          Q.mask = J.mask;
          Q.nrows = have ? J.nrows : 0;
          Q.split = J.chunk >= 0;
          Q.dist = spread && J.chunk >= 0;
          Q.count_done = merge;
          Q.bs = J.bs;
          Q.nseg = nseg;
          Q.seglen = J.chunk < 0 ? seg : (packed ? kQuads * seglen : seglen);
          if (merge && J.chunk >= 0) atomicAdd(p.ws + kWsSplitBlocks, 1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_full[slot]);
      }
#if MQA_PAIR_HELPERS
      if (spread && J.chunk >= 0) {
        // A spread merge: the producer parks after this CTA's one job (no
        // TMA writes follow), then the epilogue warps select the block's rows
        // as one group, with scratch in the idle K ring and q buffers.
        bool okp = true;
        if (ew == 0 && lane == 0) okp = wait_counter(S, &S.prod_parked, 1, p);
        if (bar_or(kEpiBarrier, kEpiThreads, !okp || aborted(S))) break;
        work_slot_rows_group(S, p, slot, ew, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.j_empty[slot]);
        ++job_iter;
        continue;
      }
#endif
      // Once the producer has parked, the epilogue warps help select the
      // block just handed over, with scratch in the idle K ring and q buffers.
      const bool parked =
          bar_or(kEpiBarrier, kEpiThreads, ew == 0 && lane == 0 && *(volatile int *)&S.prod_parked != 0);
      if (parked) {
#if MQA_PAIR_HELPERS
        // warps (2i, 2i + 1) select each row together, in the leader's scratch
        if (ew == 0 && lane == 0) *(volatile int *)&S.helping[slot] = (job_iter >> 1) + 1;
        uint8_t *scr = &S.kring[0][0] + (size_t)(ew & ~1) * kHelperScratchBytes;
        work_slot_rows_pair(S, p, slot, job_iter >> 1, ew >> 1, ew & 1, reinterpret_cast<int *>(scr),
                            reinterpret_cast<uint32_t *>(scr + 1024),
                            reinterpret_cast<int32_t *>(scr + 1024 + 4 * kSelList), lane);
#else
        uint8_t *scr = &S.kring[0][0] + (size_t)ew * kHelperScratchBytes;
        work_slot_rows(S, p, slot, job_iter >> 1, reinterpret_cast<int *>(scr),
                       reinterpret_cast<uint32_t *>(scr + 1024), reinterpret_cast<int32_t *>(scr + 1024 + 4 * kSelList),
                       lane);
#endif
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.j_empty[slot]);
    ++job_iter;
  }
}

#if MQA_PAIR_HELPERS
// ------------------------------------------------------------------ two-warp row selection
// A pair of warps selects one row together: both count half of the row's
// pieces into one histogram, both gather half of them (output and list slots
// reserved with shared atomics, so the order is free), and the leader finishes
// the list.  The two warps meet at bounded syncs on a shared counter.
__device__ bool pair_sync(Smem &S, int m, const FusedParams &p, int lane) {
  __threadfence_block();
  __syncwarp();
  bool ok = true;
  if (lane == 0) {
    const int v = atomicAdd(&S.pair_cnt[m], 1);
    ok = wait_counter(S, &S.pair_cnt[m], (v / 2 + 1) * 2, p);
    __threadfence_block();
  }
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// score_hist over the pieces of this member's batches (member i of kM takes
// every kM-th batch), into this member's four histogram copies (one per lane
// % 4: candidates crowd into the bins just above the gate), already zeroed
// Pieces per batch of a member: a pair takes deep batches; a 16-warp group
// spreads a row's few dozen pieces over all its warps.
template <int kM>
struct MultiDepth {
  static constexpr int kHist = kM == 2 ? kHistDepth : 4;
  static constexpr int kPass2 = kM == 2 ? kPass2Groups : 3;
};
template <int kM>
__device__ void score_hist_part(const RowSlab &R, float lo, float inv, int *hcopies, int lane, int member) {
  constexpr int kD = MultiDepth<kM>::kHist;
  int *hist = hcopies + (member * 4 + (lane & 3)) * kScoreBins;
  const PieceMap pm = piece_map(R, lane);
#pragma unroll 1
  for (int t0 = member * kD; t0 < pm.total; t0 += kM * kD) {
    int at[kD], lim[kD];
    uint4 kk[kD];
#pragma unroll
    for (int j = 0; j < kD; ++j) piece_at(R, pm, t0 + j, at[j], lim[j]);
#pragma unroll
    for (int j = 0; j < kD; ++j)
      kk[j] = 4 * lane < lim[j] ? __ldcg(reinterpret_cast<const uint4 *>(R.keys + at[j] + 4 * lane))
                                : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < kD; ++j) {
      const int e = 4 * lane;
      if (e < lim[j]) atomicAdd(&hist[score_bin(key2f(kk[j].x), lo, inv)], 1);
      if (e + 1 < lim[j]) atomicAdd(&hist[score_bin(key2f(kk[j].y), lo, inv)], 1);
      if (e + 2 < lim[j]) atomicAdd(&hist[score_bin(key2f(kk[j].z), lo, inv)], 1);
      if (e + 3 < lim[j]) atomicAdd(&hist[score_bin(key2f(kk[j].w), lo, inv)], 1);
    }
  }
}

constexpr int kPairOut = 200, kPairList = 201;  // shared output / list counters in the leader's histogram

// Selection of one row by kM warps (members 0 .. kM - 1; member 0 leads),
// meeting at sync() (false: the call is aborting).  Returns the leader's
// written count, 0 for the other members, -1 (all) when the threshold bin
// does not fit the list, or -2 on abort.
template <int kM, class Sync>
__device__ int multi_select_binned(Sync &&sync, int member, const RowSlab &R, int k, float lo, float inv, int *hist,
                                   uint32_t *lk, int32_t *li, int32_t *out, int base, int lane) {
  // the histogram copies (4 per member) follow the leader's list in the
  // members' scratch (the other members' own scratch is otherwise unused)
  int *hcopies = reinterpret_cast<int *>(li + kSelList);
  for (int b = lane; b < 4 * kScoreBins; b += 32) hcopies[member * 4 * kScoreBins + b] = 0;
  if (member == 0 && lane == 0) {
    hist[kPairOut] = 0;
    hist[kPairList] = 0;
  }
  if (!sync()) return -2;
  score_hist_part<kM>(R, lo, inv, hcopies, lane, member);
  if (!sync()) return -2;
  int c[kBinsPerLane], tot = 0;
  if constexpr (kM == 2) {
    // each member sums the copies itself
#pragma unroll
    for (int j = 0; j < kBinsPerLane; ++j) {
      const int b = kScoreBins - 1 - kBinsPerLane * lane - j;
      int v = 0;
#pragma unroll
      for (int cp = 0; cp < 4 * kM; ++cp) v += hcopies[cp * kScoreBins + b];
      c[j] = v;
      tot += c[j];
    }
  } else {
    // one thread per bin sums the copies into the leader's histogram
    // (its first kScoreBins entries are free until the list radix)
    const int t = member * 32 + lane;
    if (t < kScoreBins) {
      int v = 0;
#pragma unroll 8
      for (int cp = 0; cp < 4 * kM; ++cp) v += hcopies[cp * kScoreBins + t];
      hist[t] = v;
    }
    if (!sync()) return -2;
#pragma unroll
    for (int j = 0; j < kBinsPerLane; ++j) {
      c[j] = hist[kScoreBins - 1 - kBinsPerLane * lane - j];
      tot += c[j];
    }
  }
  int incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  const int excl = incl - tot;
  const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < k && k <= incl);
  const int src = bm ? __ffs(bm) - 1 : 31;
  int B = 0, above = 0, nB = 0;
  if (lane == src) {
    int run = excl;
#pragma unroll
    for (int j = 0; j < kBinsPerLane; ++j) {
      if (run + c[j] >= k) {
        B = kScoreBins - 1 - kBinsPerLane * lane - j;
        above = run;
        nB = c[j];
        break;
      }
      run += c[j];
    }
  }
  B = __shfl_sync(0xFFFFFFFFu, B, src);
  above = __shfl_sync(0xFFFFFFFFu, above, src);
  nB = __shfl_sync(0xFFFFFFFFu, nB, src);
  if (nB > kSelList || nB <= 0) return -1;
  constexpr int kP2 = MultiDepth<kM>::kPass2;
  const PieceMap pm = piece_map(R, lane);
#pragma unroll 1
  for (int t0 = member * kP2; t0 < pm.total; t0 += kM * kP2) {
    int at[kP2], lim[kP2];
    uint32_t kk[4 * kP2];
    int32_t ii[4 * kP2];
#pragma unroll
    for (int gi = 0; gi < kP2; ++gi) piece_at(R, pm, t0 + gi, at[gi], lim[gi]);
#pragma unroll
    for (int gi = 0; gi < kP2; ++gi) {
      uint4 kv = make_uint4(0, 0, 0, 0);
      int4 iv = make_int4(0, 0, 0, 0);
      if (4 * lane < lim[gi]) {
        kv = __ldcg(reinterpret_cast<const uint4 *>(R.keys + at[gi] + 4 * lane));
        iv = __ldcg(reinterpret_cast<const int4 *>(R.idx + at[gi] + 4 * lane));
      }
      kk[4 * gi] = kv.x; kk[4 * gi + 1] = kv.y; kk[4 * gi + 2] = kv.z; kk[4 * gi + 3] = kv.w;
      ii[4 * gi] = iv.x; ii[4 * gi + 1] = iv.y; ii[4 * gi + 2] = iv.z; ii[4 * gi + 3] = iv.w;
    }
    // the bin compared directly (the same monotone function as the count pass)
    uint32_t up = 0, in = 0;
#pragma unroll
    for (int j = 0; j < 4 * kP2; ++j) {
      const bool v = 4 * lane + (j & 3) < lim[j >> 2];
      const int bj = score_bin(key2f(kk[j]), lo, inv);
      if (v && bj > B) up |= 1u << j;
      if (v && bj == B) in |= 1u << j;
    }
    const int packed = __popc(up) + (__popc(in) << 16);
    int pincl = packed;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, pincl, off);
      if (lane >= off) pincl += v;
    }
    const int pexcl = pincl - packed;
    const int ptot = __shfl_sync(0xFFFFFFFFu, pincl, 31);
    int ro = 0, rl = 0;
    if (lane == 0) {
      if (ptot & 0xFFFF) ro = atomicAdd(&hist[kPairOut], ptot & 0xFFFF);
      if (ptot >> 16) rl = atomicAdd(&hist[kPairList], ptot >> 16);
    }
    ro = __shfl_sync(0xFFFFFFFFu, ro, 0);
    rl = __shfl_sync(0xFFFFFFFFu, rl, 0);
    int po = ro + (pexcl & 0xFFFF), pl = rl + (pexcl >> 16);
#pragma unroll
    for (int j = 0; j < 4 * kP2; ++j) {
      if ((up >> j) & 1u) {
        if (po < k) out[po] = out_index(ii[j], base);
        ++po;
      }
      if ((in >> j) & 1u) {
        if (pl < kSelList) {
          lk[pl] = kk[j];
          li[pl] = ii[j];
        }
        ++pl;
      }
    }
  }
  if (!sync()) return -2;
  if (member != 0) return 0;
  int outc = hist[kPairOut];
  const int lc = min(hist[kPairList], kSelList);
  __syncwarp();
  // exact threshold among the list: the want-th largest key (as warp_select_binned)
  const int want = k - above;
  uint32_t kl = 0xFFFFFFFFu, kh = 0u;
  for (int i = lane; i < lc; i += 32) {
    kl = min(kl, lk[i]);
    kh = max(kh, lk[i]);
  }
  kl = __reduce_min_sync(0xFFFFFFFFu, kl);
  kh = __reduce_max_sync(0xFFFFFFFFu, kh);
  const uint32_t diff = kl ^ kh;
  int hb = diff ? 32 - __clz(diff) : 0;
  uint32_t prefix = hb >= 32 ? 0u : (kh & ~((1u << hb) - 1u));
  int w = want;
#pragma unroll 1
  while (hb > 0) {
    const int bits = hb >= 8 ? 8 : hb;
    const int shift = hb - bits;
    const uint32_t dmask = (1u << bits) - 1u;
    const uint32_t hi_mask = hb >= 32 ? 0u : (0xFFFFFFFFu << hb);
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    for (int i = lane; i < lc; i += 32) {
      const uint32_t v = lk[i];
      if ((v & hi_mask) == prefix) atomicAdd(&hist[(v >> shift) & dmask], 1);
    }
    __syncwarp();
    int cc[8], t8 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cc[j] = hist[255 - 8 * lane - j];
      t8 += cc[j];
    }
    int in8 = t8;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, in8, off);
      if (lane >= off) in8 += v;
    }
    const int ex8 = in8 - t8;
    const uint32_t bm8 = __ballot_sync(0xFFFFFFFFu, ex8 < w && w <= in8);
    const int s8 = bm8 ? __ffs(bm8) - 1 : 31;
    int bin = 0, ab = 0;
    if (lane == s8) {
      int run = ex8;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run + cc[j] >= w) {
          bin = 255 - 8 * lane - j;
          ab = run;
          break;
        }
        run += cc[j];
      }
    }
    bin = __shfl_sync(0xFFFFFFFFu, bin, s8);
    ab = __shfl_sync(0xFFFFFFFFu, ab, s8);
    w -= ab;
    prefix |= (uint32_t)bin << shift;
    hb = shift;
    __syncwarp();
  }
  const uint32_t T = prefix;
  int eq_seen = 0;
  const uint32_t ltm = lanemask_lt();
  for (int i0 = 0; i0 < lc; i0 += 32) {
    const int i = i0 + lane;
    const bool v = i < lc;
    const uint32_t key = v ? lk[i] : 0u;
    const bool gt = v && key > T, eq = v && key == T;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const bool take = gt || (eq && eq_seen + __popc(eqm & ltm) < w);
    const uint32_t tm = __ballot_sync(0xFFFFFFFFu, take);
    const int pos = outc + __popc(tm & ltm);
    if (take && pos < k) out[pos] = out_index(li[i], base);
    outc += __popc(tm);
    eq_seen += __popc(eqm);
  }
  return outc < k ? outc : k;
}

#endif

// ------------------------------------------------------------------ per-row selection work
// Row r of the block in selection slot `slot`: its top-k indices go to out,
// or (returns true) the row must be rescanned.  hist (256 ints) and the list
// lk/li (kSelList records) are the calling warp's scratch.
__device__ bool select_row(Smem &S, const FusedParams &p, int slot, int r, int *hist, uint32_t *lk, int32_t *li,
                           int lane) {
  const SelSlot &Q = S.sel[slot];
  if (r >= Q.nrows || !((Q.mask >> r) & 1u)) return false;
  const int cap = p.cap, topk = p.topk, n = Q.n[r];
  // candidates: the CTA's slab slot, or the split slab of a merged split block
  const int rcap = Q.split ? Q.nseg * Q.seglen : cap;
  uint32_t *slab_keys = Q.split ? p.split_slab + (size_t)Q.bs * 2 * kBlockRows * rcap
                                : p.slab + ((size_t)(blockIdx.x * kSlots + slot) * 2 * kBlockRows) * (size_t)cap;
  int32_t *slab_idx = reinterpret_cast<int32_t *>(slab_keys + (size_t)kBlockRows * rcap);
  RowSlab R;
  R.keys = slab_keys + (size_t)r * rcap;
  R.idx = slab_idx + (size_t)r * rcap;
  R.seg = Q.seglen;
  R.nseg = Q.nseg;
  R.c = &Q.segcnt[r][0];
  bool over = false;
  for (int q = 0; q < R.nseg; ++q) over = over || R.c[q] > R.seg;
  const int cnt = R.total();
  if (Q.mode == 0) {
    // a row the fold classified unsafe emitted nothing and is rescanned
    const bool unsafe = kFold && Q.unsafe[r] != 0;
    const bool under = !unsafe && Q.gated[r] && cnt < min(topk, n);
    if (lane == 0) {
      if (Q.gated[r] && !unsafe) atomicAdd(p.ws + kWsGatedRows, 1);
      atomicAdd(p.ws + kWsCandidates, cnt);
      if (over) atomicAdd(p.ws + kWsOverflowRows, 1);
      if (under) atomicAdd(p.ws + kWsUnderfillRows, 1);
    }
    if (over || under || unsafe) return true;
  } else if (lane == 0) {
    atomicAdd(p.ws + kWsRowsRescanned, 1);
  }
  int32_t *out = p.out + (size_t)(Q.block * kBlockRows + r) * topk;
  int wrote;
  if (cnt <= topk) {
    wrote = warp_emit_out(R, 0u, 0, true, out, Q.start[r], topk, lane);
  } else {
    wrote = -1;
    if (Q.binned[r]) wrote = warp_select_binned(R, topk, Q.blo[r], Q.binv[r], hist, lk, li, out, Q.start[r], lane);
    if (wrote < 0) {
      if (Q.binned[r] && lane == 0) atomicAdd(p.ws + kWsSelFallback, 1);
      int take_eq = 0;
#if MQA_FOLD
      uint32_t kmin, kmax;
      warp_key_range(R, lane, &kmin, &kmax);
      // a row the gate did not classify: its candidates are all its visible
      // keys, so the largest of their |scores| is the row's
      if (Q.check[r] && !fold_safe(p, S.key_norm, Q.beta[r], fmaxf(fabsf(key2f(kmin)), fabsf(key2f(kmax))), true, lane))
        return true;
      const uint32_t T = warp_select_range(R, topk, hist, lane, &take_eq, kmin, kmax);
#else
      const uint32_t T = warp_select_range(R, topk, hist, lane, &take_eq);
#endif
      wrote = warp_emit_out(R, T, take_eq, false, out, Q.start[r], topk, lane);
    }
  }
  for (int i = wrote + lane; i < topk; i += 32) out[i] = -1;
  return false;
}

// Work on the rows of selection slot `slot` in its use-th use until none is
// left.  Every warp that helps claims rows one at a time through a bounded
// counter (it never passes this use's last row, so it needs no reset and a
// late claimer can never take a row of a later use); the warp that finishes
// the use's last row queues failed rows for a rescan, retires the job and
// releases the slot.
__device__ void work_slot_rows(Smem &S, const FusedParams &p, int slot, int use, int *hist, uint32_t *lk,
                               int32_t *li, int lane) {
  const int base = use * kBlockRows;
  for (;;) {
    int r = -1;
#if MQA_PAIR_HELPERS
    const bool claim = lane == 0 && *(volatile int *)&S.helping[slot] != use + 1;
#else
    const bool claim = lane == 0;
#endif
    if (claim) {
      int v = *(volatile int *)&S.selnext[slot];
      while (v < base + kBlockRows) {
        const int w = atomicCAS(&S.selnext[slot], v, v + 1);
        if (w == v) {
          r = v - base;
          break;
        }
        v = w;
      }
    }
    r = __shfl_sync(0xFFFFFFFFu, r, 0);
    if (r < 0) break;
    const bool fail = select_row(S, p, slot, r, hist, lk, li, lane);
    __syncwarp();
    if (lane == 0) {
      if (fail) atomicOr(&S.selfail[slot], 1u << r);
      __threadfence_block();
      const int done = atomicAdd(&S.seldone[slot], 1);
      if (done == base + kBlockRows - 1) {
        const SelSlot &Q = S.sel[slot];
        const uint32_t fm = atomicExch(&S.selfail[slot], 0u);
        if (fm) {
          const int tail = S.fifo_tail;
          S.fifo_block[tail & 7] = Q.block;
          S.fifo_mask[tail & 7] = fm;
          __threadfence_block();
          *(volatile int *)&S.fifo_tail = tail + 1;
        }
        __threadfence_block();
        if (Q.nrows > 0) atomicAdd(p.ws + kWsBlocksDone, 1);
        atomicAdd(&S.retired, 1);
        mbar_arrive(&S.s_empty[slot]);
      }
    }
  }
}

// ------------------------------------------------------------------ selection (warps 2-3)
#if MQA_PAIR_HELPERS
// Row r selected by kM warps (member 0 leads); returns true when the row
// must be rescanned.  Every member passes the same syncs on every path.
template <int kM, class Sync>
__device__ bool select_row_multi(Smem &S, const FusedParams &p, int slot, int r, Sync &&sync, int member, int *hist,
                                 uint32_t *lk, int32_t *li, int lane, bool &ok) {
  const SelSlot &Q = S.sel[slot];
  bool fail = false;
  if (r < Q.nrows && ((Q.mask >> r) & 1u)) {
    const int cap = p.cap, topk = p.topk, n = Q.n[r];
    const int rcap = Q.split ? Q.nseg * Q.seglen : cap;
    uint32_t *slab_keys = Q.split ? p.split_slab + (size_t)Q.bs * 2 * kBlockRows * rcap
                                  : p.slab + ((size_t)(blockIdx.x * kSlots + slot) * 2 * kBlockRows) * (size_t)cap;
    int32_t *slab_idx = reinterpret_cast<int32_t *>(slab_keys + (size_t)kBlockRows * rcap);
    RowSlab R;
    R.keys = slab_keys + (size_t)r * rcap;
    R.idx = slab_idx + (size_t)r * rcap;
    R.seg = Q.seglen;
    R.nseg = Q.nseg;
    R.c = &Q.segcnt[r][0];
    bool over = false;
    for (int q = 0; q < R.nseg; ++q) over = over || R.c[q] > R.seg;
    const int cnt = R.total();
    if (Q.mode == 0) {
      const bool under = Q.gated[r] && cnt < min(topk, n);
      if (member == 0 && lane == 0) {
        if (Q.gated[r]) atomicAdd(p.ws + kWsGatedRows, 1);
        atomicAdd(p.ws + kWsCandidates, cnt);
        if (over) atomicAdd(p.ws + kWsOverflowRows, 1);
        if (under) atomicAdd(p.ws + kWsUnderfillRows, 1);
      }
      fail = over || under;
    } else if (member == 0 && lane == 0) {
      atomicAdd(p.ws + kWsRowsRescanned, 1);
    }
    if (!fail) {
      int32_t *out = p.out + (size_t)(Q.block * kBlockRows + r) * topk;
      int wrote = -1;
      if (cnt > topk && Q.binned[r]) {
        wrote = multi_select_binned<kM>(sync, member, R, topk, Q.blo[r], Q.binv[r], hist, lk, li, out, Q.start[r],
                                        lane);
        if (wrote == -2) {
          ok = false;
          return false;
        }
      }
      if (member == 0) {
        if (cnt <= topk) {
          wrote = warp_emit_out(R, 0u, 0, true, out, Q.start[r], topk, lane);
        } else if (wrote < 0) {
          if (Q.binned[r] && lane == 0) atomicAdd(p.ws + kWsSelFallback, 1);
          int take_eq = 0;
          const uint32_t T = warp_select_range(R, topk, hist, lane, &take_eq);
          wrote = warp_emit_out(R, T, take_eq, false, out, Q.start[r], topk, lane);
        }
        for (int i = wrote + lane; i < topk; i += 32) out[i] = -1;
      }
    }
  }
  ok = sync();
  return fail;
}

// The rows of the block in selection slot `slot`, claimed by pair m's leader
// and selected by the pair; the pair's leader counts them done (as work_slot_rows).
__device__ void work_slot_rows_pair(Smem &S, const FusedParams &p, int slot, int use, int m, int member, int *hist,
                                    uint32_t *lk, int32_t *li, int lane) {
  const int base = use * kBlockRows;
  for (;;) {
    if (member == 0 && lane == 0) {
      int r = -1;
      int v = *(volatile int *)&S.selnext[slot];
      while (v < base + kBlockRows) {
        const int w = atomicCAS(&S.selnext[slot], v, v + 1);
        if (w == v) {
          r = v - base;
          break;
        }
        v = w;
      }
      *(volatile int *)&S.pair_row[m] = r;
    }
    if (!pair_sync(S, m, p, lane)) return;
    const int r = *(volatile int *)&S.pair_row[m];
    if (r < 0) {
      // both have read the end marker before the leader may overwrite it
      pair_sync(S, m, p, lane);
      return;
    }
    bool ok = true;
    const bool fail = select_row_multi<2>(S, p, slot, r, [&]() { return pair_sync(S, m, p, lane); }, member, hist, lk,
                                          li, lane, ok);
    if (!ok) return;
    if (member == 0 && lane == 0) {
      if (r < S.sel[slot].nrows && ((S.sel[slot].mask >> r) & 1u)) atomicAdd(p.ws + kWsPairRows, 1);
      if (fail) atomicOr(&S.selfail[slot], 1u << r);
      __threadfence_block();
      const int done = atomicAdd(&S.seldone[slot], 1);
      if (done == base + kBlockRows - 1) {
        const SelSlot &Q = S.sel[slot];
        const uint32_t fm = atomicExch(&S.selfail[slot], 0u);
        if (fm) {
          const int tail = S.fifo_tail;
          S.fifo_block[tail & 7] = Q.block;
          S.fifo_mask[tail & 7] = fm;
          __threadfence_block();
          *(volatile int *)&S.fifo_tail = tail + 1;
        }
        __threadfence_block();
        if (Q.nrows > 0) atomicAdd(p.ws + kWsBlocksDone, 1);
        atomicAdd(&S.retired, 1);
        mbar_arrive(&S.s_empty[slot]);
      }
    }
  }
}


// A spread merge's rows, claimed one at a time from the block's merge_next
// and selected by a group of this CTA's epilogue warps together (the group's
// first warp leads).  With fewer key chunks per block than rows, each chunk's
// CTA has several rows to select, and two groups of 8 warps take two rows side
// by side (32 x 8 rows x 64K keys, 4 chunks per block: 153.5 -> 147.4 us);
// with more chunks than rows all 16 warps take one row (4 x 8 rows x 256K
// keys, 32 chunks: 106.5 us against 112.5 with two groups).  The CTA's first
// warp then releases the slot (rows to rescan go to this CTA's queue).
template <int kGroups>
__device__ void merge_group_rows(Smem &S, const FusedParams &p, int slot, int ew, int lane) {
  constexpr int kGroupWarps = kEpiWarps / kGroups;
  constexpr int kGroupScratch =
      (kHelperScratchBytes + kGroupWarps * 4 * kScoreBins * (int)sizeof(int) + 127) / 128 * 128;
  static_assert(kGroups * kGroupScratch <= (int)(sizeof(Smem::kring) + sizeof(Smem::q)),
                "the groups' scratch fits the idle K ring and q buffers");
  const SelSlot &Q = S.sel[slot];
  const int g = ew / kGroupWarps, gm = ew % kGroupWarps;
  uint8_t *scr = &S.kring[0][0] + (size_t)g * kGroupScratch;
  int *hist = reinterpret_cast<int *>(scr);
  uint32_t *lk = reinterpret_cast<uint32_t *>(scr + 1024);
  int32_t *li = reinterpret_cast<int32_t *>(scr + 1024 + 4 * kSelList);
  auto sync = [&]() {
    if (kGroups == 1) return !bar_or(kEpiBarrier, kEpiThreads, aborted(S));
    return g == 0 ? !bar_or(kEpiBarrier + 1, kGroupWarps * 32, aborted(S))
                  : !bar_or(kEpiBarrier + 2, kGroupWarps * 32, aborted(S));
  };
  uint32_t fails = 0;
  for (;;) {
    if (gm == 0 && lane == 0)
      *(volatile int *)&S.grp_row[g] = Q.nrows > 0 ? atomicAdd(p.merge_next + Q.bs, 1) : kBlockRows;
    if (!sync()) return;
    const int r = *(volatile int *)&S.grp_row[g];
    if (r >= kBlockRows) break;
    bool ok = true;
    const bool fail = select_row_multi<kGroupWarps>(S, p, slot, r, sync, gm, hist, lk, li, lane, ok);
    if (!ok) return;
    if (fail) fails |= 1u << r;
    if (gm == 0 && lane == 0 && r < Q.nrows && ((Q.mask >> r) & 1u)) atomicAdd(p.ws + kWsPairRows, 1);
  }
  if constexpr (kGroups > 1) {
    // both groups are done with the slot before it is released
    if (gm == 0 && lane == 0 && fails) atomicOr(&S.grp_fails, fails);
    if (bar_or(kEpiBarrier, kEpiThreads, aborted(S))) return;
    if (ew == 0 && lane == 0) {
      fails = *(volatile unsigned *)&S.grp_fails;
      S.grp_fails = 0;
    }
  }
  if (ew == 0 && lane == 0) {
    if (fails) {
      const int tail = S.fifo_tail;
      S.fifo_block[tail & 7] = Q.block;
      S.fifo_mask[tail & 7] = fails;
      __threadfence_block();
      *(volatile int *)&S.fifo_tail = tail + 1;
    }
    __threadfence_block();
    if (Q.count_done) atomicAdd(p.ws + kWsBlocksDone, 1);
    atomicAdd(&S.retired, 1);
    mbar_arrive(&S.s_empty[slot]);
  }
}
__device__ void work_slot_rows_group(Smem &S, const FusedParams &p, int slot, int ew, int lane) {
  if (S.nchunks < kBlockRows) merge_group_rows<2>(S, p, slot, ew, lane);
  else merge_group_rows<1>(S, p, slot, ew, lane);
}

#endif

__device__ void selection(Smem &S, const FusedParams &p, int warp, int lane) {
  const int sw = warp - kSelWarp0;
  int job_iter = 0;
  for (;;) {
    const int slot = job_iter & 1;
    bool ok = true;
    if (lane == 0) ok = wait_bar(S, &S.s_full[slot], (job_iter >> 1) & 1, p, kBackoffIdle);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) break;
    if (S.sel[slot].block < 0) break;
    // the epilogue group selects (and releases) a spread merge's slot
    if (!S.sel[slot].dist)
      work_slot_rows(S, p, slot, job_iter >> 1, &S.selhist[sw][0], S.sel_lk[sw], S.sel_li[sw], lane);
    ++job_iter;
  }
}

// ------------------------------------------------------------------ kernel
template <bool kLogits>
__global__ void __launch_bounds__(kThreads, 1)
    mqa_fused_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap s_map, const __grid_constant__ CUtensorMap x_map,
                     const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem &S = get_smem(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0 && !kLogits)
    atomicMax(reinterpret_cast<unsigned long long *>(p.ws + kWsTStartMinInv), ~globaltimer_ns());
  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&S.k_full[i], 1);
      mbar_init(&S.k_empty[i], 1);
    }
    for (int i = 0; i < kSStages; ++i) {
      mbar_init(&S.sc_full[i], 1);
      mbar_init(&S.sc_empty[i], kMasked ? kEpiWarps : 1);
    }
    for (int i = 0; i < kTmemBufs; ++i) {
      mbar_init(&S.t_full[i], 1);
      mbar_init(&S.t_empty[i], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.j_full[i], 32);
      mbar_init(&S.j_empty[i], 1 + kEpiWarps);
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.s_empty[i], 1);  // released by the warp that finishes the slot's last row
      S.seldone[i] = 0;
      S.selnext[i] = 0;
      S.selfail[i] = 0;
    }
    mbar_init(&S.drain, 1);
    mbar_init(&S.stall_bar, 1);
    S.abort_flag = 0;
    S.fifo_head = 0;
    S.fifo_tail = 0;
    S.retired = 0;
    S.grp_fails = 0;
    S.nsplit = 0;
    S.split_first = 0;
    S.nchunks = 1;
    S.prod_parked = 0;
    // fold: the per-call preparation wrote the keys' largest scale * |k|_2
    S.key_norm = kFold && !kLogits ? __int_as_float(__ldcg(p.ws + kWsKeyNorm)) : 0.f;
#if MQA_PAIR_HELPERS
    S.helping[0] = 0;
    S.helping[1] = 0;
    for (int i = 0; i < kEpiWarps / 2; ++i) {
      S.pair_cnt[i] = 0;
      S.pair_row[i] = -1;
    }
#endif
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&q_map);
    tma_prefetch_desc(&k_map);
    tma_prefetch_desc(&s_map);
    if (kMasked || kFold) tma_prefetch_desc(&x_map);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemAllocCols);
    tmem_relinquish();
  }
  if (!kLogits) build_order(S, p);
  // the order scratch shared the K ring with later TMA writes
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    producer<kLogits>(S, &q_map, &k_map, &s_map, &x_map, p, lane);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer(S, tmem, p);
  } else if (warp >= kEpiWarp0) {
    epilogue<kLogits>(S, tmem, p, warp, lane);
  } else if (warp >= kSelWarp0 && warp < kSelWarp0 + kSelWarps) {
    if (!kLogits) selection(S, p, warp, lane);
  }
  __syncthreads();
  if (threadIdx.x == 0 && !kLogits) {
    const uint64_t t = globaltimer_ns();
    atomicMax(reinterpret_cast<unsigned long long *>(p.ws + kWsTEndMinInv), ~t);
    atomicMax(reinterpret_cast<unsigned long long *>(p.ws + kWsTEndMax), t);
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemAllocCols);
  }
}

// The shared-memory opt-in is a per-device function attribute: set it once on
// each device a launch runs on (done[] is the calling kernel's own record).
static cudaError_t set_smem_attr(const void *fn, bool (&done)[kAttrDevices]) {
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  if (dev < 0 || dev >= kAttrDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev]) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fused_smem_bytes());
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

cudaError_t launch_fused_topk(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                              const FusedParams &p, int ctas, cudaStream_t stream, const CUtensorMap *x_map) {
  static bool attr_done[kAttrDevices] = {};
  if ((kMasked || kFold) && !x_map) return cudaErrorInvalidValue;
  const cudaError_t attr = set_smem_attr((const void *)mqa_fused_kernel<false>, attr_done);
  if (attr != cudaSuccess) return attr;
  // the extra map is read only by the masked and fold builds; the others get a placeholder
  const CUtensorMap &xm = x_map ? *x_map : s_map;
  mqa_fused_kernel<false><<<ctas, kThreads, fused_smem_bytes(), stream>>>(q_map, k_map, s_map, xm, p);
  return cudaGetLastError();
}

#if MQA_PAIR_HELPERS
cudaError_t launch_logits(const CUtensorMap &q_map, const CUtensorMap &k_map, const CUtensorMap &s_map,
                          const FusedParams &p, int ctas, cudaStream_t stream) {
  static bool attr_done[kAttrDevices] = {};
  const cudaError_t attr = set_smem_attr((const void *)mqa_fused_kernel<true>, attr_done);
  if (attr != cudaSuccess) return attr;
  mqa_fused_kernel<true><<<ctas, kThreads, fused_smem_bytes(), stream>>>(q_map, k_map, s_map, s_map, p);
  return cudaGetLastError();
}
#endif

}  // namespace MQA_KNS

#if MQA_PAIR_HELPERS
// ------------------------------------------------------------------ allocation-free scratch
// Scratch for mqa_topk_prefill_noalloc: the 256-byte header plus the candidate
// slabs of at most kStaticScratchCtas persistent CTAs, as a file-scope device
// array.  Every GPU that loads the library holds it until the process exits.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

cudaError_t static_scratch_address(void **ptr) {
  // Host code cannot use the array's name as a device address: resolve it once
  // per device, with that device current.
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void *a = nullptr;
    e = cudaGetSymbolAddress(&a, g_static_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = a;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}
#endif

}  // namespace mqa
