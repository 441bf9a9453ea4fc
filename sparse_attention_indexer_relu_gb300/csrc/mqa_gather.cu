// Masked selection that scores only the allowed keys (the consumer layers of
// the two-level candidate selection: "vLLM: fused FP8 MQA top-k indexer" pull
// request #60618, "Limitations of this PR -- TODOs", DeepSeek-V4.1 two-level
// candidate selection; the consumers there mask their scores to the source
// layer's top 2,048 blocks of 8 keys before the top-512, and the page notes
// that scoring only the candidate blocks is what speeds those layers up).
//
// Each row is scored on its own: its allowed blocks of 8 keys, in ascending
// order, are gathered 16 at a time into a 128-key tile (one 1 KiB TMA box per
// block) and multiplied on the tensor core by that row's 32 query heads
// (M = 128 keys, N = 32 heads, FP8 inputs, FP32 accumulation in TMEM).  The
// score of key k is key_scale[k] * sum_h w_h * relu(q_h . k), the same
// definition as every other selection mode; the row's top-k of those scores
// (exact, any order, then -1) is chosen in shared memory.
//
// Roles of one persistent CTA (one per SM, 20 warps):
//  - warps 0-7 gather the job's K blocks into a 5-stage ring of tiles with
//    16-byte asynchronous copies (the copies a warp keeps in flight are
//    bounded, so the gather rate grows with the loader warps: the 16,384-row,
//    128K-key masked top-512 on random block lists took 14.2 ms with two
//    loader warps, 10.9 ms with four, 9.7 ms with six, 7.3 ms with eight
//    or ten);
//  - warps 8-11 (one warp per TMEM lane quadrant) form each key's score and
//    store its order key in the job's score buffer, with the job's key count
//    and order-key range;
//  - warp 12 issues the MMAs into 16 TMEM accumulators of 32 columns;
//  - warp 13 claims rows, turns a row's block-mask words into lists of at
//    most 768 blocks (a "job"; a row with more allowed blocks is several
//    jobs) and loads the row's q;
//  - warps 14-19 select: a value-bin histogram over that range, one pass that
//    emits the keys of the bins above the one holding the k-th largest and
//    copies that bin out, and a radix select over the copy.  With the source
//    stage's own top blocks the selection sets the pace, so six warps select
//    (against four with ten loader warps: 10.2 -> 9.7 ms at 128K keys).
// Three job slots let a job's selection overlap the scoring of the next two
// (128K-key masked top-2048 on the source stage's own top blocks: two slots of
// 1,024 blocks 9.7 ms, three of 768 7.9 ms, three or four of 512 8.0 ms).
#include <mutex>

#include "mqa_internal.h"
#include "ptx.cuh"
#include "mqatopk.h"

namespace mqa {
namespace gather {

constexpr int kBlk = 8;                      // keys per block
constexpr int kTileBlocks = kTileKeys / kBlk;  // 16 blocks per 128-key tile
constexpr int kStages = 5;                   // K ring depth
#ifndef MQA_GATHER_LOADER_WARPS
#define MQA_GATHER_LOADER_WARPS 8
#endif
constexpr int kLoaderWarps = MQA_GATHER_LOADER_WARPS;  // warps 0 .. kLoaderWarps - 1
static_assert(kLoaderWarps % 2 == 0, "two loader warps per block of 8 keys");
constexpr int kLoaderThreads = 32 * kLoaderWarps;
constexpr int kBufs = 16;                    // TMEM accumulators (32 columns each)
constexpr int kN = 32;                       // UMMA N: the row's heads
#ifndef MQA_GATHER_JOB_SLOTS
#define MQA_GATHER_JOB_SLOTS 3
#endif
#ifndef MQA_GATHER_SEG_BLOCKS
#define MQA_GATHER_SEG_BLOCKS 768
#endif
constexpr int kJobSlots = MQA_GATHER_JOB_SLOTS;  // jobs in flight (score buffers, q, counters)
constexpr int kLists = kJobSlots + 1;            // block lists: one more, so the next is built ahead
constexpr int kSegBlocks = MQA_GATHER_SEG_BLOCKS;  // blocks per job
static_assert(kSegBlocks % 16 == 0, "a job is whole 128-key tiles");
constexpr int kSegKeys = kSegBlocks * kBlk;  // score-buffer entries per job
constexpr int kMaxTopk = 2048;
constexpr int kList = 1024;                  // selection: threshold-bin keys copied out
#ifndef MQA_GATHER_EPI_SETS
#define MQA_GATHER_EPI_SETS 1
#endif
#ifndef MQA_GATHER_SEL_WARPS
#define MQA_GATHER_SEL_WARPS 6
#endif
constexpr int kEpiSets = MQA_GATHER_EPI_SETS;
// Warp layout: loaders first; the MMA issuer and the job builder fill the
// gap before the epilogue warps (which must start at a multiple of 4, so that
// warp % 4 is their TMEM lane quadrant) when there is one, else follow them;
// the selection warps come last.
#ifndef MQA_GATHER_LATE_ROLES
#define MQA_GATHER_LATE_ROLES 1
#endif
constexpr bool kLateRoles = MQA_GATHER_LATE_ROLES != 0;
constexpr int kEpiWarps = 4 * kEpiSets;
constexpr int kEpiWarp0 = kLateRoles ? (kLoaderWarps + 3) / 4 * 4 : (kLoaderWarps + 2 + 3) / 4 * 4;
constexpr int kMmaWarp = kLateRoles ? kEpiWarp0 + kEpiWarps : kLoaderWarps;
constexpr int kBuilderWarp = kMmaWarp + 1;
constexpr int kSelWarp0 = kLateRoles ? kBuilderWarp + 1 : kEpiWarp0 + kEpiWarps;
constexpr int kSelWarps = MQA_GATHER_SEL_WARPS;
constexpr int kHistCopies = kSelWarps;  // value-bin histograms, one per selection warp
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kThreads = (kSelWarp0 + kSelWarps) * 32;
constexpr uint32_t kSelBar = 1;  // named barrier of the selection warps
constexpr uint32_t kIdesc = idesc_f8_e4m3_f32(128, kN);
constexpr int kQRowBytes = kN * kDim;    // one row's q: 32 heads x 128 B
constexpr uint32_t kTmemCols = kBufs * kN;
static_assert(kTmemCols == 512, "the accumulators fill the 512 TMEM columns");
static_assert(kBufs % kEpiSets == 0, "a TMEM buffer always goes to the same epilogue set");

struct Job {
  int row;          // -1: no more work
  int lb;           // the job's block list: blist[lb]
  int start, end;   // the row's key range (clamped)
  int nblocks;      // blocks in this job's list
  int first, last;  // the row's first / last job
  alignas(16) float w[kN];
};

struct Smem {
  alignas(1024) uint8_t kring[kStages][kTileKeys * kDim];
  alignas(1024) uint8_t q[kJobSlots][kQRowBytes];
  uint32_t sbuf[kJobSlots][kSegKeys];  // order keys of a job's gathered keys (0: not a visible key)
  int32_t blist[kLists][kSegBlocks];  // job j's blocks (global block index, ascending) in list j % kLists
  uint32_t ckey[2][kMaxTopk];     // the row's running top-k over its earlier jobs (ping-pong)
  int32_t cidx[2][kMaxTopk];
  int whist[kHistCopies][256];   // selection histograms
  int wabove[kSelWarps], win[kSelWarps];  // per selection warp: entries above / in the threshold bin
  uint32_t lkey[kList];           // selection: the keys of the threshold value bin
  int32_t lidx[kList];            // and their key indices
  Job job[kJobSlots];
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t t_full[kBufs], t_empty[kBufs];
  uint64_t j_full[kJobSlots], j_empty[kJobSlots], s_full[kJobSlots];
  uint64_t drain, stall_bar;
  uint32_t tmem_base;
  int abort_flag;
  // selection state (written by the selection warps' first warp)
  uint32_t sel_prefix;
  int sel_want, sel_bin, sel_inbin, sel_hb, list_n;
  int cnt_gt, cnt_eq;
  // a job's visible keys (count, order-key range), gathered by the epilogue
  uint32_t jlo[kJobSlots], jhi[kJobSlots];
  int jcnt[kJobSlots];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory above the 227 KB opt-in limit");

__device__ __forceinline__ Smem &get_smem(uint8_t *raw) {
  uintptr_t a = reinterpret_cast<uintptr_t>(raw);
  a = (a + 1023) & ~uintptr_t(1023);
  return *reinterpret_cast<Smem *>(a);
}

// ------------------------------------------------------------------ waits
__device__ __forceinline__ bool aborted(Smem &S) { return *(volatile int *)&S.abort_flag != 0; }

__device__ __noinline__ void raise_timeout(Smem &S, const GatherParams &p) {
  *(volatile int *)&S.abort_flag = 1;
  atomicOr(p.ws + kWsStatus, kDevWaitTimeout);
}

// Wait for the phase of `bar` with the given parity; false on abort or when
// the call's time limit runs out (which aborts the CTA).
__device__ __forceinline__ bool wait_bar(Smem &S, uint64_t *bar, uint32_t parity, const GatherParams &p,
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

// Bounded wait used while unwinding: gives up after `ns` without raising.
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity, long long ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(globaltimer_ns() - t0) > ns) break;
    __nanosleep(256);
  }
}

// ------------------------------------------------------------------ warp 2: rows -> jobs
// Appends the allowed blocks of the row's mask words [*wpos, wend) to `list`
// (ascending) until the list would pass kSegBlocks; blocks outside
// [blo, bhi] are not visible.  Words are read 4 at a time (16-byte loads from
// a 4-word-aligned index), 512 words per pass.  Returns the list length and
// advances *wpos past the words taken.
__device__ int build_list(const uint32_t *mrow, int *wpos, int wend, int blo, int bhi, int32_t *list, int lane) {
  int n = 0;
  int w0 = *wpos;
  while (w0 < wend) {
    const int base = w0 & ~3;
    uint32_t wv[4][4];
    int cnt[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int wi = base + 128 * g + 4 * lane;  // first word of this lane's group g
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (wi < wend) x = __ldg(reinterpret_cast<const uint4 *>(mrow + wi));
      wv[g][0] = x.x;
      wv[g][1] = x.y;
      wv[g][2] = x.z;
      wv[g][3] = x.w;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      cnt[g] = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int wi = base + 128 * g + 4 * lane + j;
        uint32_t v = wv[g][j];
        if (wi < w0 || wi >= wend) v = 0u;
        // blocks 32 wi + b outside [blo, bhi] are not visible
        const int b_lo = blo - 32 * wi, b_hi = bhi - 32 * wi;
        if (b_lo > 0) v = b_lo >= 32 ? 0u : v & (0xFFFFFFFFu << b_lo);
        if (b_hi < 31) v = b_hi < 0 ? 0u : v & (0xFFFFFFFFu >> (31 - b_hi));
        wv[g][j] = v;
        cnt[g] += __popc(v);
      }
    }
    bool full = false;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (full) break;
      int incl = cnt[g];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
      }
      // lanes whose whole group fits (a prefix of the lanes: incl grows with lane)
      const uint32_t fit = __ballot_sync(0xFFFFFFFFu, n + incl <= kSegBlocks);
      const int f = __popc(fit);
      if (lane < f) {
        int pos = n + incl - cnt[g];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t v = wv[g][j];
          const int wi = base + 128 * g + 4 * lane + j;
          while (v) {
            const int b = __ffs(v) - 1;
            v &= v - 1u;
            list[pos++] = 32 * wi + b;
          }
        }
      }
      const int took = f > 0 ? __shfl_sync(0xFFFFFFFFu, incl, f - 1) : 0;
      n += took;
      if (f < 32) {
        // the list is full: the next job starts at lane f's group
        w0 = max(w0, base + 128 * g + 4 * f);
        full = true;
      }
    }
    if (full) break;
    w0 = base + 512;
  }
  *wpos = w0 < wend ? w0 : wend;
  return n;
}

__device__ void builder(Smem &S, const CUtensorMap *q_map, const GatherParams &p, int lane) {
  const uint64_t pol_q = policy_evict_first();
  if (p.stall) {
    // test hook: a wait that nothing completes; the time limit ends it
    if (!wait_bar(S, &S.stall_bar, 0, p)) return;
  }
  int it = 0;
  for (;;) {
    int row = 0;
    if (lane == 0) row = atomicAdd(p.ws + kWsClaim, 1);
    row = __shfl_sync(0xFFFFFFFFu, row, 0);
    const bool done = row >= p.rows;
    int s = 0, e = 0;
    if (!done) {
      s = __ldg(p.starts + row);
      e = __ldg(p.ends + row);
      if ((s < 0 || e > p.keys) && e > s) {
        if (lane == 0) atomicOr(p.ws + kWsStatus, kDevRangeClamped);
        s = max(s, 0);
        e = min(e, p.keys);
      }
      if (e < s) e = s;
    }
    const int blo = s >> 3, bhi = e > s ? (e - 1) >> 3 : blo - 1;
    int wpos = blo >> 5;
    const int wend = e > s ? (bhi >> 5) + 1 : wpos;
    const uint32_t *mrow = p.mask + (size_t)(done ? 0 : row) * p.mask_words;
    const float wl = done ? 0.f : __ldg(p.weights + (size_t)row * kN + lane);
    bool first = true;
    for (;;) {
      const int slot = it % kJobSlots;
      // The list of job `it` goes to blist[it % kLists], last used by job
      // it - kLists, whose selection ended before job it - 1 was published;
      // so it is built before the wait for job it - kJobSlots's slot, while
      // that job is selected.
      const int lb = it % kLists;
      int n = 0;
      if (!done) n = build_list(mrow, &wpos, wend, blo, bhi, S.blist[lb], lane);
      const bool last = wpos >= wend;
      bool ok = true;
      if (lane == 0) ok = wait_bar(S, &S.j_empty[slot], ((it / kJobSlots) & 1) ^ 1, p, 256);
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
        // unwinding: let the q loads of the last two jobs land before the CTA exits
        if (lane == 0)
          for (int i = 1; i <= kJobSlots && i <= it; ++i)
            drain_bar(&S.j_full[(it - i) % kJobSlots], ((it - i) / kJobSlots) & 1, p.timeout_ns);
        return;
      }
      Job &J = S.job[slot];
      if (done) {
        if (lane == 0) {
          J.row = -1;
          mbar_arrive(&S.j_full[slot]);
        }
        return;
      }
      J.w[lane] = wl;
      if (lane == 0) {
        J.row = row;
        J.lb = lb;
        J.start = s;
        J.end = e;
        J.nblocks = n;
        J.first = first;
        J.last = last;
        S.jlo[slot] = 0xFFFFFFFFu;
        S.jhi[slot] = 0u;
        S.jcnt[slot] = 0;
      }
      __syncwarp();
      if (lane == 0) {
        if (n > 0) {
          mbar_arrive_expect_tx(&S.j_full[slot], kQRowBytes);
          tma_load_2d(&S.q[slot][0], q_map, &S.j_full[slot], 0, row * kN, pol_q);
        } else {
          mbar_arrive(&S.j_full[slot]);
        }
      }
      ++it;
      first = false;
      if (last) break;
    }
  }
}

// ------------------------------------------------------------------ warps 0-9: K gathers
// The blocks of a tile are copied with 16-byte asynchronous copies into the
// 128-byte-swizzled K-major layout the MMA reads (16-byte chunk c of tile row
// r at r * 128 + ((c ^ r % 8) * 16)).  Loader thread lt copies chunk lt % 8
// of row (lt / 8) % 8 of blocks lt / 64, lt / 64 + kLoaderWarps / 2, ... of
// the tile, so each warp instruction reads 512 contiguous bytes of k.  Each
// loader thread's copies of a tile arrive on the tile's k_full barrier when
// they land (one arrival per loader thread completes it); the MMA
// issuer fences the copies into the tensor core's proxy after its wait, so
// the loaders never stall on their own copies.  Keys past the last key are
// not copied (their rows are never read back).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every earlier cp.async of this thread has completed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ void k_loader(Smem &S, const GatherParams &p, int lane, int lt) {
  // 64 threads per block: thread lt copies chunk c of row rr of blocks
  // j0, j0 + kJStep, ... of each tile
  constexpr int kJStep = kLoaderWarps / 2;
  const int rr = (lt >> 3) & 7, c = lt & 7, j0 = lt >> 6;
  const uint32_t row_off = (uint32_t)(rr * kDim + ((c ^ rr) << 4));
  const uint8_t *ksrc = p.k + c * 16;
  int it = 0, kc = 0;
  bool ok = true;
  for (;;) {
    const int slot = it % kJobSlots;
    if (lane == 0) ok = wait_bar(S, &S.j_full[slot], (it / kJobSlots) & 1, p, 128);
    if (!(ok = __shfl_sync(0xFFFFFFFFu, ok, 0))) break;
    const Job &J = S.job[slot];
    if (J.row < 0) break;
    const int n = J.nblocks, ntiles = (n + kTileBlocks - 1) / kTileBlocks;
    const int32_t *list = S.blist[J.lb];
    for (int u = 0; u < ntiles; ++u) {
      const int stage = kc % kStages;
      if (lane == 0) ok = wait_bar(S, &S.k_empty[stage], ((kc / kStages) & 1) ^ 1, p, 64);
      if (!(ok = __shfl_sync(0xFFFFFFFFu, ok, 0))) break;
      const int nb = min(kTileBlocks, n - kTileBlocks * u);
      const uint32_t dst = smem_u32(&S.kring[stage][0]) + row_off;
      for (int j = j0; j < nb; j += kJStep) {
        const int key = list[kTileBlocks * u + j] * kBlk + rr;
        if (key < p.keys) cp_async16(dst + (uint32_t)(j * kBlk * kDim), ksrc + (size_t)key * kDim);
      }
      cp_async_arrive(&S.k_full[stage]);
      ++kc;
    }
    if (!ok) break;
    if (lane == 0) mbar_arrive(&S.j_empty[slot]);
    ++it;
  }
  // unwinding: no copy may still be writing when the CTA exits
  cp_async_wait_all();
}

// ------------------------------------------------------------------ warp 1: MMA
__device__ void mma_issuer(Smem &S, uint32_t tmem, const GatherParams &p) {
  int it = 0, kc = 0;
  const uint64_t a0 = sw128_kmajor_desc(smem_u32(&S.kring[0][0]));
  for (;;) {
    const int slot = it % kJobSlots;
    if (!wait_bar(S, &S.j_full[slot], (it / kJobSlots) & 1, p, 64)) break;
    const Job &J = S.job[slot];
    if (J.row < 0) break;
    const int ntiles = (J.nblocks + kTileBlocks - 1) / kTileBlocks;
    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(&S.q[slot][0]));
    bool ok = true;
    for (int u = 0; u < ntiles; ++u, ++kc) {
      const int stage = kc % kStages, buf = kc % kBufs;
      ok = wait_bar(S, &S.k_full[stage], (kc / kStages) & 1, p, 32) &&
           wait_bar(S, &S.t_empty[buf], ((kc / kBufs) & 1) ^ 1, p, 32);
      if (!ok) break;
      // the tile was written by the loaders' generic-proxy copies
      fence_proxy_async();
      tc_fence_after();
      const uint64_t adesc = a0 + (uint64_t)(stage * (kTileKeys * kDim >> 4));
      const uint32_t d = tmem + (uint32_t)(buf * kN);
#pragma unroll
      for (int kk = 0; kk < kDim / 32; ++kk)
        umma_f8(d, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), kIdesc, kk > 0 ? 1u : 0u);
      umma_commit(&S.k_empty[stage]);
      umma_commit(&S.t_full[buf]);
    }
    if (!ok) break;
    // the job's q slot is free once its MMAs are done
    umma_commit(&S.j_empty[slot]);
    ++it;
  }
  umma_commit(&S.drain);
  drain_bar(&S.drain, 0, p.timeout_ns);
}

// ------------------------------------------------------------------ warps 4-11: scores
__device__ void epilogue(Smem &S, uint32_t tmem, const GatherParams &p, int warp, int lane) {
  const int quad = warp & 3, set = (warp - kEpiWarp0) >> 2;
  const int kq = quad * 32 + lane;  // this thread's key within a tile (its TMEM lane)
  const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
  int it = 0, tc = 0;
  for (;;) {
    const int slot = it % kJobSlots;
    bool ok = wait_bar(S, &S.j_full[slot], (it / kJobSlots) & 1, p, 64);
    if (!__all_sync(0xFFFFFFFFu, ok)) return;
    const Job &J = S.job[slot];
    if (J.row < 0) return;
    const int n = J.nblocks, s = J.start, e = J.end;
    const int ntiles = (n + kTileBlocks - 1) / kTileBlocks;
    float2 w2[kN / 2];
#pragma unroll
    for (int h = 0; h < kN / 2; ++h) w2[h] = make_float2(J.w[2 * h], J.w[2 * h + 1]);
    const int32_t *list = S.blist[J.lb];
    uint32_t *sb = S.sbuf[slot];
    // this set's tiles of the job: u0, u0 + 2, ...; the key and scale of the
    // next one are fetched while the current one is scored
    const int u0 = ((set - tc) % kEpiSets + kEpiSets) % kEpiSets;
    auto key_of = [&](int u, bool &valid) -> int {
      const int bi = kTileBlocks * u + (kq >> 3);
      valid = bi < n;
      const int key = valid ? list[bi] * kBlk + (kq & 7) : 0;
      valid = valid && key >= s && key < e;
      return key;
    };
    bool vnext = false;
    int knext = u0 < ntiles ? key_of(u0, vnext) : 0;
    float snext = vnext ? __ldg(p.scales + knext) : 0.f;
    // the job's visible keys: count and order-key range, for the selection
    uint32_t jlo = 0xFFFFFFFFu, jhi = 0u;
    int jcnt = 0;
    for (int u = u0; u < ntiles; u += kEpiSets) {
      const bool valid = vnext;
      const float sc = snext;
      if (u + kEpiSets < ntiles) {
        knext = key_of(u + kEpiSets, vnext);
        snext = vnext ? __ldg(p.scales + knext) : 0.f;
      }
      const int t = tc + u, buf = t % kBufs;
      ok = wait_bar(S, &S.t_full[buf], (t / kBufs) & 1, p, 32);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem + lane_addr + (uint32_t)(buf * kN), v);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.t_empty[buf]);
      // sum_h w_h relu(s_h) as sum_h w_h (s_h + |s_h|) / 2
      float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
      for (int h = 0; h < kN / 2; h += 2) {
        const float2 x0 = make_float2(__uint_as_float(v[2 * h]), __uint_as_float(v[2 * h + 1]));
        const float2 x1 = make_float2(__uint_as_float(v[2 * h + 2]), __uint_as_float(v[2 * h + 3]));
        a0 = __ffma2_rn(__fadd2_rn(x0, make_float2(fabsf(x0.x), fabsf(x0.y))), w2[h], a0);
        a1 = __ffma2_rn(__fadd2_rn(x1, make_float2(fabsf(x1.x), fabsf(x1.y))), w2[h + 1], a1);
      }
      const float score = ((a0.x + a0.y) + (a1.x + a1.y)) * (0.5f * sc);
      const uint32_t key = valid ? f2key(score) : 0u;
      sb[kTileKeys * u + kq] = key;
      if (valid) {
        jlo = min(jlo, key);
        jhi = max(jhi, key);
        ++jcnt;
      }
    }
    tc += ntiles;
    jlo = __reduce_min_sync(0xFFFFFFFFu, jlo);
    jhi = __reduce_max_sync(0xFFFFFFFFu, jhi);
    jcnt = __reduce_add_sync(0xFFFFFFFFu, jcnt);
    if (lane == 0) {
      if (jcnt) {
        atomicMin(&S.jlo[slot], jlo);
        atomicMax(&S.jhi[slot], jhi);
        atomicAdd(&S.jcnt[slot], jcnt);
      }
      mbar_arrive(&S.s_full[slot]);
    }
    ++it;
  }
}

// ------------------------------------------------------------------ warps 12-15: selection
__device__ __forceinline__ void sel_sync() { asm volatile("bar.sync %0, %1;" ::"r"(kSelBar), "r"(kSelThreads) : "memory"); }

// Entry i of a selection: the row's running top-k first (ck, cn entries),
// then the job's score buffer (sb, nent entries); order key 0 is no key.
struct Entries {
  const uint32_t *ck;
  int cn;
  const uint32_t *sb;
  int nent;
  __device__ __forceinline__ int size() const { return cn + nent; }
  __device__ __forceinline__ uint32_t at(int i) const { return i < cn ? ck[i] : sb[i - cn]; }
};

// Value bin (0..255) of an order key: linear in the score over [smin, smin +
// 256 / inv).  Monotone in the key (every step is a monotone rounding), so a
// key in a higher bin is larger than every key in a lower bin.
__device__ __forceinline__ int score_bin(uint32_t key, float smin, float inv) {
  const float v = (key2f(key) - smin) * inv;
  return v >= 255.f ? 255 : (v > 0.f ? (int)v : 0);
}

// Suffix scan of a 256-bin histogram by one warp: the bin b holding the
// want-th largest entry, the entries above it and in it.  Lane l holds bins
// 255 - 8l - j (j < 8).
__device__ __forceinline__ void pick_bin(const int (&cc)[8], int want, int lane, int *bin, int *above, int *inbin) {
  int t8 = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) t8 += cc[j];
  int in8 = t8;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, in8, off);
    if (lane >= off) in8 += v;
  }
  const int ex8 = in8 - t8;
  const uint32_t bm = __ballot_sync(0xFFFFFFFFu, ex8 < want && want <= in8);
  const int sl = bm ? __ffs(bm) - 1 : 31;
  int b = 0, ab = 0, c = 0;
  if (lane == sl) {
    int run = ex8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (run + cc[j] >= want) {
        b = 255 - 8 * lane - j;
        ab = run;
        c = cc[j];
        break;
      }
      run += cc[j];
    }
  }
  *bin = __shfl_sync(0xFFFFFFFFu, b, sl);
  *above = __shfl_sync(0xFFFFFFFFu, ab, sl);
  *inbin = __shfl_sync(0xFFFFFFFFu, c, sl);
}

// One radix digit: histogram of key bits [hb - bits, hb) over the entries
// whose bits from hb up equal S.sel_prefix's; the first selection warp then
// extends the prefix by the digit holding the S.sel_want-th largest entry and
// leaves in S.sel_want how many of that digit's entries are still wanted.
__device__ void sel_digit(Smem &S, const Entries &E, int hb, int bits, int tid, int lane) {
  for (int b = tid; b < 256; b += kSelThreads) S.whist[0][b] = 0;
  sel_sync();
  const uint32_t prefix = S.sel_prefix;
  const uint32_t hi_mask = hb >= 32 ? 0u : (0xFFFFFFFFu << hb);
  const int shift = hb - bits;
  const uint32_t dmask = (1u << bits) - 1u;
  const int tot = E.size();
  for (int i = tid; i < tot; i += kSelThreads) {
    const uint32_t key = E.at(i);
    if (key != 0u && (key & hi_mask) == prefix) atomicAdd(&S.whist[0][(key >> shift) & dmask], 1);
  }
  sel_sync();
  if (tid < 32) {
    int cc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cc[j] = S.whist[0][255 - 8 * lane - j];
    int bin, above, inbin;
    pick_bin(cc, S.sel_want, lane, &bin, &above, &inbin);
    if (lane == 0) {
      S.sel_prefix = prefix | ((uint32_t)bin << shift);
      S.sel_want -= above;
    }
  }
  sel_sync();
}

// Where a selected entry goes: the row's output (relative index, on its last
// job) or the running top-k carried to its next job.
struct Sink {
  int32_t *orow;
  uint32_t *ckey;
  int32_t *cidx;
  int start;
  bool last;
  __device__ __forceinline__ void put(int pos, uint32_t key, int idx) const {
    if (last) {
      orow[pos] = idx - start;
    } else {
      ckey[pos] = key;
      cidx[pos] = idx;
    }
  }
};

// Emit every entry above T and the first take_eq entries equal to T (of the
// entries of E; positions from base_gt and base_eq on), warp-aggregated.
__device__ void emit_threshold(Smem &S, const Entries &E, const int32_t *ci, const int32_t *list, uint32_t T,
                               int take_eq, int base_gt, int base_eq, bool all, const Sink &K, int tid, int lane) {
  const uint32_t ltm = lanemask_lt();
  const int tot = E.size();
  for (int i0 = 0; i0 < tot; i0 += kSelThreads) {
    const int i = i0 + tid;
    const uint32_t key = i < tot ? E.at(i) : 0u;
    const bool gt = key != 0u && key > T;
    const bool eq = !all && key != 0u && key == T;
    const uint32_t bg = __ballot_sync(0xFFFFFFFFu, gt), be = __ballot_sync(0xFFFFFFFFu, eq);
    int g0 = 0, e0 = 0;
    if (lane == 0) {
      if (bg) g0 = atomicAdd(&S.cnt_gt, __popc(bg));
      if (be) e0 = atomicAdd(&S.cnt_eq, __popc(be));
    }
    g0 = __shfl_sync(0xFFFFFFFFu, g0, 0);
    e0 = __shfl_sync(0xFFFFFFFFu, e0, 0);
    int pos = -1;
    if (gt) pos = base_gt + g0 + __popc(bg & ltm);
    if (eq) {
      const int r = e0 + __popc(be & ltm);
      if (r < take_eq) pos = base_eq + r;
    }
    if (pos >= 0) {
      const int idx = i < E.cn ? ci[i] : list[(i - E.cn) >> 3] * kBlk + ((i - E.cn) & 7);
      K.put(pos, key, idx);
    }
  }
}

// Radix select over S.lkey[0, n) for the S.sel_want-th largest key, from the
// copy's highest differing bit: T in S.sel_prefix, the equal keys wanted in
// S.sel_want.
__device__ void list_threshold(Smem &S, int n, int tid, int lane) {
  if (tid < 32) {
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int i = lane; i < n; i += 32) {
      lo = min(lo, S.lkey[i]);
      hi = max(hi, S.lkey[i]);
    }
    lo = __reduce_min_sync(0xFFFFFFFFu, lo);
    hi = __reduce_max_sync(0xFFFFFFFFu, hi);
    const uint32_t diff = lo ^ hi;
    const int hb = diff ? 32 - __clz(diff) : 0;
    if (lane == 0) {
      S.sel_hb = hb;
      S.sel_prefix = hb >= 32 ? 0u : (hi & ~((1u << hb) - 1u));
    }
  }
  sel_sync();
  const Entries L{S.lkey, n, nullptr, 0};
  for (int hb = S.sel_hb; hb > 0;) {
    const int bits = hb >= 8 ? 8 : hb;
    sel_digit(S, L, hb, bits, tid, lane);
    hb -= bits;
  }
}

// One job's selection: the topk largest of its entries (the row's running
// top-k plus the job's scores) go to the sink.  total entries hold a key, in
// the order-key range [kmin, kmax].  Returns how many were selected.
//  - at most topk entries: all of them;
//  - else a histogram of 256 value bins over [kmin, kmax] locates the bin b
//    that holds the topk-th largest; one pass emits the entries of higher
//    bins and copies b's entries out (at most kList of them), and a radix
//    select over the copy settles the threshold among them;
//  - a bin with more entries (or a degenerate range) runs the radix select
//    over every entry instead.
// Keys below `floor` (the running top-k's smallest key when it is full: no
// such key can be selected) are left out of the histogram and the copy.
__device__ int select_job(Smem &S, const Entries &E, const int32_t *ci, const int32_t *list, int total, uint32_t kmin,
                          uint32_t kmax, uint32_t floor, int topk, const Sink &K, int tid, int lane, uint32_t *tmin) {
  const int tot = E.size();
  if (total <= topk) {
    emit_threshold(S, E, ci, list, 0u, 0, 0, 0, true, K, tid, lane);
    *tmin = kmin;
    return total;
  }
  const int wid = tid >> 5;
  const float smin = key2f(kmin), smax = key2f(kmax);
  const float inv = 256.f / (smax - smin);
  const bool binned = smax > smin && inv > 0.f && inv < 3.0e38f;
  if (binned) {
    for (int b = tid; b < kHistCopies * 256; b += kSelThreads) (&S.whist[0][0])[b] = 0;
    sel_sync();
    // four entries per thread and step, loaded before any is counted
    for (int i0 = tid; i0 < tot; i0 += 4 * kSelThreads) {
      uint32_t kk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) kk[u] = i0 + u * kSelThreads < tot ? E.at(i0 + u * kSelThreads) : 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (kk[u] != 0u && kk[u] >= floor) atomicAdd(&S.whist[wid][score_bin(kk[u], smin, inv)], 1);
    }
    sel_sync();
    if (tid < 32) {
      int cc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int b = 255 - 8 * lane - j;
        int c = 0;
#pragma unroll
        for (int w = 0; w < kHistCopies; ++w) c += S.whist[w][b];
        cc[j] = c;
      }
      int bin, above, inbin;
      pick_bin(cc, topk, lane, &bin, &above, &inbin);
      if (lane == 0) {
        S.sel_bin = bin;
        S.sel_want = topk - above;
        S.sel_inbin = inbin;
        S.list_n = 0;
      }
    }
    sel_sync();
    {
      // this warp's entries above and in the threshold bin (its own histogram)
      const int bstar = S.sel_bin;
      int a = 0;
      for (int b = bstar + 1 + lane; b < 256; b += 32) a += S.whist[wid][b];
      a = __reduce_add_sync(0xFFFFFFFFu, a);
      if (lane == 0) {
        S.wabove[wid] = a;
        S.win[wid] = S.whist[wid][bstar];
      }
    }
    sel_sync();
  }
  if (binned && S.sel_inbin <= kList) {
    // entries of higher bins are selected; the threshold bin's are copied
    // out.  Each warp meets the same entries as in the histogram pass, so its
    // output ranges follow from the warps' counts (no shared counters).
    const int bstar = S.sel_bin, want = S.sel_want, n = S.sel_inbin;
    const int above = topk - want;
    const uint32_t ltm = lanemask_lt();
    int g0 = 0, l0 = 0;
    for (int w = 0; w < wid; ++w) {
      g0 += S.wabove[w];
      l0 += S.win[w];
    }
    // four entries per thread and step (the same entries per warp as the
    // histogram pass), all loaded and binned before any is written
    for (int i00 = 0; i00 < tot; i00 += 4 * kSelThreads) {
      uint32_t kk[4];
      int bb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i00 + u * kSelThreads + tid;
        kk[u] = i < tot ? E.at(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) bb[u] = kk[u] != 0u && kk[u] >= floor ? score_bin(kk[u], smin, inv) : -1;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i00 + u * kSelThreads + tid;
        const bool gt = bb[u] > bstar, in = bb[u] == bstar;
        const uint32_t mg = __ballot_sync(0xFFFFFFFFu, gt), mi = __ballot_sync(0xFFFFFFFFu, in);
        if (gt || in) {
          const int idx = i < E.cn ? ci[i] : list[(i - E.cn) >> 3] * kBlk + ((i - E.cn) & 7);
          if (gt) {
            K.put(g0 + __popc(mg & ltm), kk[u], idx);
          } else {
            const int l = l0 + __popc(mi & ltm);
            S.lkey[l] = kk[u];
            S.lidx[l] = idx;
          }
        }
        g0 += __popc(mg);
        l0 += __popc(mi);
      }
    }
    sel_sync();
    list_threshold(S, n, tid, lane);
    const uint32_t T = S.sel_prefix;
    const int take_eq = S.sel_want;
    if (tid == 0) {
      S.cnt_gt = 0;
      S.cnt_eq = 0;
    }
    sel_sync();
    // the copy's keys above T, then take_eq of those equal to T
    const Entries L{S.lkey, n, nullptr, 0};
    emit_threshold(S, L, S.lidx, list, T, take_eq, above, above + (want - take_eq), false, K, tid, lane);
    *tmin = T;
  } else {
    if (tid == 0) {
      S.sel_prefix = 0u;
      S.sel_want = topk;
    }
    sel_sync();
    for (int hb = 32; hb > 0; hb -= 8) sel_digit(S, E, hb, 8, tid, lane);
    const uint32_t T = S.sel_prefix;
    const int take_eq = S.sel_want;
    emit_threshold(S, E, ci, list, T, take_eq, 0, topk - take_eq, false, K, tid, lane);
    *tmin = T;
  }
  return topk;
}

__device__ void selection(Smem &S, const GatherParams &p, int warp, int lane) {
  const int tid = (warp - kSelWarp0) * 32 + lane;
  int it = 0, cin = 0, cn = 0;
  uint32_t clo = 0u, chi = 0u;  // the running top-k's order-key range
  for (;;) {
    const int slot = it % kJobSlots;
    // the four selection warps leave together (each wait is bounded)
    if (bar_or(kSelBar, kSelThreads, !wait_bar(S, &S.j_full[slot], (it / kJobSlots) & 1, p, 256))) return;
    const Job &J = S.job[slot];
    if (J.row < 0) return;
    if (bar_or(kSelBar, kSelThreads, !wait_bar(S, &S.s_full[slot], (it / kJobSlots) & 1, p, 64))) return;
    if (J.first) cn = 0;
    const int topk = p.topk;
    const int nent = ((J.nblocks + kTileBlocks - 1) / kTileBlocks) * kTileKeys;
    const Entries E{S.ckey[cin], cn, S.sbuf[slot], nent};
    const int jn = S.jcnt[slot];
    const int total = cn + jn;
    uint32_t kmin = jn ? S.jlo[slot] : 0xFFFFFFFFu, kmax = jn ? S.jhi[slot] : 0u;
    if (cn) {
      kmin = min(kmin, clo);
      kmax = max(kmax, chi);
    }
    // a full running top-k bounds every key that can still be selected
    const uint32_t floor = cn == topk ? clo : 0u;
    kmin = max(kmin, floor);
    if (tid == 0) {
      S.cnt_gt = 0;
      S.cnt_eq = 0;
    }
    sel_sync();
    const bool last = J.last != 0;
    const int cout = cin ^ 1;
    const Sink K{p.out + (size_t)J.row * topk, S.ckey[cout], S.cidx[cout], J.start, last};
    uint32_t tmin;
    const int c = select_job(S, E, S.cidx[cin], S.blist[J.lb], total, kmin, kmax, floor, topk, K, tid, lane, &tmin);
    if (last)
      for (int i = c + tid; i < topk; i += kSelThreads) K.orow[i] = -1;
    if (tid == 0) {
      atomicAdd(p.ws + kWsCandidates, jn);
      if (last) atomicAdd(p.ws + kWsBlocksDone, 1);
    }
    // the slot's buffers and the carry read above are free
    sel_sync();
    if (!last) {
      // the carry's range: from the threshold (or the smallest entry when
      // all were taken) to the entries' largest
      cn = c;
      cin = cout;
      chi = kmax;
      clo = tmin;
    }
    if (lane == 0) mbar_arrive(&S.j_empty[slot]);
    ++it;
  }
}

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads, 1)
    mqa_gather_kernel(const __grid_constant__ CUtensorMap q_map, const GatherParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem &S = get_smem(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    atomicMax(reinterpret_cast<unsigned long long *>(p.ws + kWsTStartMinInv), ~globaltimer_ns());
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&S.k_full[i], kLoaderThreads);  // one arrival per loader thread
      mbar_init(&S.k_empty[i], 1);
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(&S.t_full[i], 1);
      mbar_init(&S.t_empty[i], 4);  // the four warps of the set that owns the buffer
    }
    for (int i = 0; i < kJobSlots; ++i) {
      mbar_init(&S.j_full[i], 1);
      // released by the loader warps, the MMA issuer (commit) and the selection warps
      mbar_init(&S.j_empty[i], kLoaderWarps + 1 + kSelWarps);
      mbar_init(&S.s_full[i], kEpiWarps);
    }
    mbar_init(&S.drain, 1);
    mbar_init(&S.stall_bar, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kBuilderWarp && lane == 0) tma_prefetch_desc(&q_map);
  if (warp == kMmaWarp) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp < kLoaderWarps) {
    k_loader(S, p, lane, threadIdx.x);
  } else if (warp == kMmaWarp) {
    if (lane == 0) mma_issuer(S, tmem, p);
  } else if (warp == kBuilderWarp) {
    builder(S, &q_map, p, lane);
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    epilogue(S, tmem, p, warp, lane);
  } else if (warp >= kSelWarp0) {
    selection(S, p, warp, lane);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t = globaltimer_ns();
    atomicMax(reinterpret_cast<unsigned long long *>(p.ws + kWsTEndMinInv), ~t);
    atomicMax(reinterpret_cast<unsigned long long *>(p.ws + kWsTEndMax), t);
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace gather

size_t gather_smem_bytes() { return gather::kSmemBytes; }

cudaError_t launch_gather_masked(const CUtensorMap &q_map, const GatherParams &p, int ctas, cudaStream_t stream) {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!done[dev]) {
      e = cudaFuncSetAttribute((const void *)gather::mqa_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)gather::kSmemBytes);
      if (e != cudaSuccess) return e;
      done[dev] = true;
    }
  }
  gather::mqa_gather_kernel<<<ctas, gather::kThreads, gather::kSmemBytes, stream>>>(q_map, p);
  return cudaGetLastError();
}

}  // namespace mqa

// ------------------------------------------------------------------ tensor-pipe probe
// A measurement helper, not part of the method: every CTA (one per SM) issues
// back-to-back 128 x 256 x 128 FP8 MMA tiles (four K = 32 steps, e4m3 inputs,
// fp32 accumulation, the fused kernel's shape) from fixed shared-memory
// operands into two TMEM accumulators.  Timing it gives the tensor pipe's
// FP8 issue ceiling on this GPU at the clocks it holds.
namespace mqa {
namespace probe {
__global__ void __launch_bounds__(128, 1) fp8_mma_probe(long long tiles, int32_t *status) {
  extern __shared__ uint8_t raw[];
  __shared__ uint32_t tbase;
  __shared__ __align__(8) uint64_t bar;
  uint8_t *A = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t *B = A + 128 * kDim;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (128 + 256) * kDim; i += blockDim.x) A[i] = (uint8_t)(0x30 + (i & 7));
  if (warp == 0) {
    tmem_alloc(&tbase, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = idesc_f8_e4m3_f32(128, 256);
    const uint64_t ad = sw128_kmajor_desc(smem_u32(A)), bd = sw128_kmajor_desc(smem_u32(B));
    for (long long t = 0; t < tiles; ++t) {
      const uint32_t d = tbase + (uint32_t)((t & 1) * 256);
#pragma unroll
      for (int kk = 0; kk < kDim / 32; ++kk)
        umma_f8(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, kk > 0 ? 1u : 0u);
    }
    umma_commit(&bar);
    // bounded: about 2 s of polling at most
    const uint64_t t0 = globaltimer_ns();
    bool done = false;
    while (!(done = mbar_try_wait(&bar, 0)) && globaltimer_ns() - t0 < 2000000000ull) {
    }
    if (!done) atomicOr(status, kDevWaitTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}
}  // namespace probe

cudaError_t launch_fp8_mma_probe(long long tiles, int32_t *status, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int smem = (128 + 256) * kDim + 1024;
  e = cudaFuncSetAttribute((const void *)probe::fp8_mma_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  probe::fp8_mma_probe<<<sms, 128, smem, stream>>>(tiles, status);
  return cudaGetLastError();
}
}  // namespace mqa
