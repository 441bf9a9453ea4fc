// C ABI of the library (include/mqatopk.h): argument checks, workspace sizing,
// TMA descriptor encoding and launches.  Host code only.
#include "../../include/mqatopk.h"
#include "mqa_fold.h"
#include "mqa_internal.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

namespace {

using namespace mqa;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ok = false;
  int sms = 0;
  int major = 0, minor = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int device_info(int dev, DeviceInfo *out) {
  if (dev < 0 || dev >= kMaxDevices) return MQA_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev[dev].ok) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return MQA_ERR_NO_DEVICE;
    }
    if (dev >= n) return MQA_ERR_INVALID_ARGUMENT;
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return MQA_ERR_CUDA;
    }
    d.ok = true;
    g_dev[dev] = d;
  }
  *out = g_dev[dev];
  return MQA_OK;
}

int current_device_info(DeviceInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_NO_DEVICE;
  }
  int rc = device_info(dev, out);
  if (rc != MQA_OK) return rc;
  if (!(out->major == 10 && out->minor == 3)) return MQA_ERR_UNSUPPORTED_DEVICE;
  return MQA_OK;
}

int get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return MQA_OK;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return MQA_OK;
}

// 2-D uint8 tensor [rows_outer, 128] with rows of 128 bytes, 128-byte swizzle.
int encode_rows128(CUtensorMap *map, const void *base, uint64_t nrows, uint32_t box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)nrows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDim};
  const cuuint32_t box[2] = {(cuuint32_t)kDim, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MQA_OK : MQA_ERR_CUDA;
}

// 1-D fp32 tensor [n] read in boxes of 128 elements (out-of-range elements read as 0).
int encode_scales(CUtensorMap *map, const float *base, uint64_t n) {
  const cuuint64_t dims[1] = {(cuuint64_t)n};
  const cuuint64_t strides[1] = {(cuuint64_t)(n * sizeof(float))};  // unused for rank 1
  const cuuint32_t box[1] = {(cuuint32_t)kTileKeys};
  const cuuint32_t estr[1] = {1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, const_cast<float *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MQA_OK : MQA_ERR_CUDA;
}

// 2-D uint32 block mask [rows, words], read in boxes of 4 words x 8 rows
// (out-of-range words read as 0, i.e. no key allowed).
int encode_mask(CUtensorMap *map, const uint32_t *base, uint64_t rows, uint64_t words) {
  const cuuint64_t dims[2] = {(cuuint64_t)words, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(words * sizeof(uint32_t))};
  const cuuint32_t box[2] = {4, (cuuint32_t)kBlockRows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MQA_OK : MQA_ERR_CUDA;
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(const void *q, const void *k, const float *scales, const float *weights, const int32_t *starts,
                 const int32_t *ends, const void *out, int rows, int keys) {
  if (rows < 0 || keys < 1 || keys > MQA_MAX_KEYS) return MQA_ERR_INVALID_ARGUMENT;
  if (rows > 0 && (!q || !k || !scales || !weights || !starts || !ends || !out)) return MQA_ERR_INVALID_ARGUMENT;
  if (rows > 0 && (!aligned(q, 16) || !aligned(k, 16) || !aligned(scales, 16) || !aligned(weights, 16) ||
                   !aligned(out, 16) || !aligned(starts, 4) || !aligned(ends, 4)))
    return MQA_ERR_MISALIGNED;
  return MQA_OK;
}

bool valid_topk(int topk) { return topk == 512 || topk == 1024 || topk == 2048; }

// Rows per block: a 256-column accumulator tile holds 8 rows of 32 heads or 4 of 64.
int block_rows(int heads) { return 256 / heads; }

size_t slab_bytes(int ctas, int cap, int brows) {
  return (size_t)ctas * kSlots * 2 * brows * (size_t)cap * sizeof(uint32_t);
}

int fused_ctas(const DeviceInfo &d, int rows, int brows) {
  const int nb = (rows + brows - 1) / brows;
  return nb < d.sms ? nb : d.sms;
}

// With the key-range split, few-block calls also use idle SMs (one CTA per
// key chunk), and up to two waves' worth of blocks can be split.
int fused_ctas_split(const DeviceInfo &d, int rows, int brows) {
  const long long nb = (rows + brows - 1) / brows;
  return nb * kMaxChunks < d.sms ? (int)(nb * kMaxChunks) : d.sms;
}
int split_max_blocks(int ctas, int rows, int brows) {
  const int nb = (rows + brows - 1) / brows;
  return nb < ctas ? nb : nb % ctas;
}

}  // namespace

FusedLayout mqa::fused_layout(int ctas, int cap, int split_max, int brows, int fold_rows) {
  FusedLayout L;
  L.done_off = kWsHeaderBytes;
  // per split block: finished chunks, then the next row of a spread merge
  L.slab_off = L.done_off + (((size_t)2 * split_max * sizeof(int32_t) + 255) / 256) * 256;
  L.split_off = L.slab_off + slab_bytes(ctas, cap, brows);
  long long rc = 0;
  if (split_max > 0) {
    // the largest split set the device plan may choose (see plan_split)
    const long long c2 = (long long)(split_max < 2 * ctas ? split_max : 2 * ctas) * split_row_capacity(cap, 2);
    const long long c4 = (long long)(split_max < ctas / 4 ? split_max : ctas / 4) * split_row_capacity(cap, 4);
    rc = c2 > c4 ? c2 : c4;
    for (int c = 8; c <= kMaxChunks; c *= 2) {
      const long long cc = (long long)(split_max < ctas / c ? split_max : ctas / c) * split_row_capacity(cap, c);
      rc = rc > cc ? rc : cc;
    }
  }
  L.split_words = 2LL * brows * rc;
  L.cnt_off = L.split_off + (size_t)L.split_words * sizeof(uint32_t);
  const size_t cnt_end = L.cnt_off + (size_t)split_max * brows * 32 * sizeof(int32_t);
  // fold: each row's folded-query terms [rows, 4, 128] (TMA source, 1024-byte
  // aligned), their exponents [rows, 4] and residual norms [rows]
  L.fold_codes_off = (cnt_end + 1023) / 1024 * 1024;
  L.fold_exps_off = L.fold_codes_off + (size_t)fold_rows * kFoldRowTerms * kDim;
  L.fold_beta_off = L.fold_exps_off + ((size_t)fold_rows * kFoldRowTerms * sizeof(int32_t) + 15) / 16 * 16;
  L.total = fold_rows > 0 ? L.fold_beta_off + (size_t)fold_rows * sizeof(float) : cnt_end;
  L.reset_bytes = L.slab_off;
  return L;
}

namespace {

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Which compilation of the fused kernel serves a call, and its block shape.
enum class Build { kDirect, kFold, kPairs, kHeads64, kBlocks, kMasked };

struct Plan {
  Build build;
  int brows;     // rows per block
  int ctas;      // persistent CTAs
  int split_max; // blocks the split arrays hold (0: no key-range split)
  FusedLayout L;
};

// The compilation a call runs on: block selection, masked selection and 64
// heads have their own.  32-head key selection runs the direct head sum with
// 8-row blocks; calls with few blocks per CTA (decode batches, small chunks,
// the allocation-free entry) run its compilation whose parked epilogue warps
// select rows in pairs.  The fold compilation (6-row blocks) runs when the
// caller asks for it (debug option head_sum = 1).
Build pick_build(const DeviceInfo &d, int rows, int heads, bool blocks, bool masked, bool noalloc, int head_sum = 0) {
  if (masked) return Build::kMasked;
  if (blocks) return Build::kBlocks;
  if (heads == 64) return Build::kHeads64;
  if (noalloc) return Build::kPairs;
  if (head_sum == 1) return Build::kFold;
  const int nb8 = (rows + 7) / 8;
  const int ctas8 = fused_ctas_split(d, rows, 8);
  return (long long)nb8 * 4 <= ctas8 ? Build::kPairs : Build::kDirect;
}

int build_rows(Build b) {
  switch (b) {
    case Build::kFold: return kFoldBlockRows;
    case Build::kHeads64: return block_rows(64);
    default: return block_rows(32);
  }
}

// Split plan and workspace layout of a call; max_ctas (0: none) caps the CTAs.
Plan plan_call(const DeviceInfo &d, Build b, int rows, int cap, int max_ctas, bool allow_split) {
  Plan P;
  P.build = b;
  P.brows = build_rows(b);
  const int fold_rows = b == Build::kFold ? rows : 0;
  P.ctas = allow_split ? fused_ctas_split(d, rows, P.brows) : fused_ctas(d, rows, P.brows);
  if (max_ctas && max_ctas < P.ctas) P.ctas = max_ctas;
  P.split_max = allow_split ? split_max_blocks(P.ctas, rows, P.brows) : 0;
  P.L = fused_layout(P.ctas, cap, P.split_max, P.brows, fold_rows);
  return P;
}

// Masked selection through the gathering kernel: the workspace header only.
int run_gather(const DeviceInfo &d, const void *q, const void *k, const float *scales, const float *weights,
               const int32_t *starts, const int32_t *ends, const uint32_t *mask, int mask_words, int32_t *out,
               int rows, int keys, int topk, void *workspace, size_t workspace_bytes, void *stream,
               const mqa_topk_debug_options *opt) {
  if (workspace_bytes < kWsHeaderBytes) return MQA_ERR_WORKSPACE_TOO_SMALL;
  int rc = get_encoder();
  if (rc != MQA_OK) return rc;
  CUtensorMap qm;
  // one query row's 32 heads per box
  if (encode_rows128(&qm, q, (uint64_t)rows * 32, 32) != MQA_OK) return MQA_ERR_CUDA;
  GatherParams p;
  std::memset(&p, 0, sizeof p);
  p.k = reinterpret_cast<const uint8_t *>(k);
  p.scales = scales;
  p.weights = weights;
  p.starts = starts;
  p.ends = ends;
  p.mask = mask;
  p.mask_words = mask_words;
  p.out = out;
  p.ws = reinterpret_cast<int32_t *>(workspace);
  p.rows = rows;
  p.keys = keys;
  p.topk = topk;
  p.stall = opt ? opt->stall : 0;
  p.timeout_ns = (long long)((opt && opt->wait_timeout_ms) ? opt->wait_timeout_ms : 4000) * 1000000LL;
  int ctas = rows < d.sms ? rows : d.sms;
  if (opt && opt->max_ctas && opt->max_ctas < ctas) ctas = opt->max_ctas;
  cudaStream_t st = as_stream(stream);
  if (cudaMemsetAsync(workspace, 0, kWsHeaderBytes, st) != cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  return launch_gather_masked(qm, p, ctas, st) == cudaSuccess ? MQA_OK : MQA_ERR_CUDA;
}

int run_fused(const void *q, const void *k, const float *scales, const float *weights, const int32_t *starts,
              const int32_t *ends, int32_t *out, int rows, int keys, int topk, int heads, void *workspace,
              size_t workspace_bytes, void *stream, const mqa_topk_debug_options *opt, bool blocks = false,
              const uint32_t *mask = nullptr, int mask_words = 0, const int32_t *row_items = nullptr,
              bool noalloc = false) {
  int rc = check_common(q, k, scales, weights, starts, ends, out, rows, keys);
  if (rc != MQA_OK) return rc;
  if (!valid_topk(topk) || (heads != 32 && heads != 64) || (blocks && heads != 32)) return MQA_ERR_INVALID_ARGUMENT;
  if (mask && (heads != 32 || blocks || !row_items || mask_words % 4 != 0 ||
               (long long)mask_words * 256 < (long long)keys))
    return MQA_ERR_INVALID_ARGUMENT;
  if (mask && (!aligned(mask, 16) || !aligned(row_items, 4))) return MQA_ERR_MISALIGNED;
  if (!workspace) return MQA_ERR_INVALID_ARGUMENT;
  if (!aligned(workspace, 256)) return MQA_ERR_MISALIGNED;
  int cap = kDefaultSlabCap;
  if (opt && opt->slab_capacity) {
    cap = opt->slab_capacity;
    // four per-quadrant segments, each able to hold top-k plus one tile's worth
    if (cap % (kQuads * 32) != 0 || cap / kQuads < topk + 64 || cap > kDefaultSlabCap)
      return MQA_ERR_INVALID_ARGUMENT;
  }
  if (opt && (opt->force_gate < 0 || opt->force_gate > 2 || opt->wait_timeout_ms < 0 || opt->max_ctas < 0 ||
              opt->force_unsafe < 0 || opt->force_unsafe > 1 || opt->head_sum < 0 || opt->head_sum > 2 ||
              opt->masked_scan < 0 || opt->masked_scan > 1))
    return MQA_ERR_INVALID_ARGUMENT;
  if (rows == 0) return MQA_OK;
  DeviceInfo d;
  rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  const int max_ctas = opt ? opt->max_ctas : 0;
  // masked selection scores only the allowed blocks unless the caller asks
  // for the scan of every tile in each row block's range
  if (mask && !(opt && opt->masked_scan))
    return run_gather(d, q, k, scales, weights, starts, ends, mask, mask_words, out, rows, keys, topk, workspace,
                      workspace_bytes, stream, opt);
  const Build b = pick_build(d, rows, heads, blocks, mask != nullptr, noalloc, opt ? opt->head_sum : 0);
  // key-range split when the workspace holds its arrays (mqa_topk_workspace_bytes
  // sizes for it), else one CTA per block as far as SMs go
  Plan P = plan_call(d, b, rows, cap, max_ctas, true);
  if (workspace_bytes < P.L.total) {
    P = plan_call(d, b, rows, cap, max_ctas, false);
    if (workspace_bytes < P.L.total) return MQA_ERR_WORKSPACE_TOO_SMALL;
  }
  const FusedLayout &L = P.L;
  const int brows = P.brows;
  rc = get_encoder();
  if (rc != MQA_OK) return rc;
  uint8_t *wsb = reinterpret_cast<uint8_t *>(workspace);
  CUtensorMap qm, km, sm, xm;
  if (mask && encode_mask(&xm, mask, (uint64_t)rows, (uint64_t)mask_words) != MQA_OK) return MQA_ERR_CUDA;
  // the fold compilation's B operand rows: the block's folded-query terms after its q rows
  if (b == Build::kFold &&
      encode_rows128(&xm, wsb + L.fold_codes_off, (uint64_t)rows * kFoldRowTerms, kFoldBoxRows) !=
          MQA_OK)
    return MQA_ERR_CUDA;
  // q is [rows * heads, 128]: a block's (row, head) rows per TMA box
  if (encode_rows128(&qm, q, (uint64_t)rows * heads, (uint32_t)(brows * heads)) != MQA_OK ||
      encode_rows128(&km, k, (uint64_t)keys, kTileKeys) != MQA_OK || encode_scales(&sm, scales, keys) != MQA_OK)
    return MQA_ERR_CUDA;
  FusedParams p;
  std::memset(&p, 0, sizeof p);
  p.scales = scales;
  p.weights = weights;
  p.starts = starts;
  p.ends = ends;
  p.out = out;
  p.ws = reinterpret_cast<int32_t *>(workspace);
  p.slab = reinterpret_cast<uint32_t *>(wsb + L.slab_off);
  p.split_max = P.split_max;
  if (P.split_max > 0) {
    p.split_done = reinterpret_cast<int32_t *>(wsb + L.done_off);
    p.merge_next = p.split_done + P.split_max;
    p.split_slab = reinterpret_cast<uint32_t *>(wsb + L.split_off);
    p.split_cnt = reinterpret_cast<int32_t *>(wsb + L.cnt_off);
    p.split_words = L.split_words;
  }
  if (b == Build::kFold) {
    p.fold_exps = reinterpret_cast<const int32_t *>(wsb + L.fold_exps_off);
    p.fold_beta = reinterpret_cast<const float *>(wsb + L.fold_beta_off);
  }
  p.rows = rows;
  p.keys = keys;
  p.topk = topk;
  p.nblocks = (rows + brows - 1) / brows;
  p.row_items = row_items;
  p.mask = mask;
  p.mask_words = mask_words;
  p.cap = cap;
  // The gate aims at 3k candidates per row, at most half the slab row.  At
  // the default capacity a quadrant segment (cap / 4 = 3,328 records) holds
  // 2.17x its expected share of a top-2048 row's 6,144; a row whose quadrant
  // overflows is rescanned exactly.
  p.gate_target = 3 * topk < cap / 2 ? 3 * topk : cap / 2;
  // Masked rows see few of their range's keys, so a sample of the range holds
  // few gate-passing keys: a larger target keeps about 32 of them in the
  // sample (at most 64 tiles) and the gate's under-fill risk negligible.
  if (mask && p.gate_target < 4096) p.gate_target = 4096 < cap / 2 ? 4096 : cap / 2;
  // gate every row that would otherwise bring more than twice the target
  // candidates to the selection (and every row the slab cannot hold)
  p.gate_min = 2 * p.gate_target;
  p.force_gate = opt ? opt->force_gate : 0;
  p.force_unsafe = opt ? opt->force_unsafe : 0;
  p.stall = opt ? opt->stall : 0;
  p.timeout_ns = (long long)((opt && opt->wait_timeout_ms) ? opt->wait_timeout_ms : 4000) * 1000000LL;
  cudaStream_t st = as_stream(stream);
  if (cudaMemsetAsync(workspace, 0, L.reset_bytes, st) != cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  if (b == Build::kFold &&
      launch_fold_call_prep(reinterpret_cast<const uint8_t *>(q), weights, reinterpret_cast<const uint8_t *>(k), scales,
                            wsb + L.fold_codes_off, reinterpret_cast<int32_t *>(wsb + L.fold_exps_off),
                            reinterpret_cast<float *>(wsb + L.fold_beta_off), rows, keys, p.ws + kWsKeyNorm,
                            st) != cudaSuccess)
    return MQA_ERR_CUDA;
  cudaError_t le = cudaSuccess;
  switch (b) {
    case Build::kMasked: le = h32m::launch_fused_topk(qm, km, sm, p, P.ctas, st, &xm); break;
    case Build::kBlocks: le = h32b::launch_fused_topk(qm, km, sm, p, P.ctas, st); break;
    case Build::kHeads64: le = h64::launch_fused_topk(qm, km, sm, p, P.ctas, st); break;
    case Build::kPairs: le = h32p::launch_fused_topk(qm, km, sm, p, P.ctas, st); break;
    case Build::kFold: le = h32f::launch_fused_topk(qm, km, sm, p, P.ctas, st, &xm); break;
    case Build::kDirect: le = h32::launch_fused_topk(qm, km, sm, p, P.ctas, st); break;
  }
  if (le != cudaSuccess) return MQA_ERR_CUDA;
  return MQA_OK;
}

int run_logits_chunk(const DeviceInfo &d, const uint8_t *q, const void *k, const float *scales,
                     const float *weights, const int32_t *starts, const int32_t *ends, float *logits, int rows,
                     int keys, int32_t *ws, bool reset_header, cudaStream_t st) {
  CUtensorMap qm, km, sm;
  if (encode_rows128(&qm, q, (uint64_t)rows * kHeads, kCols) != MQA_OK ||
      encode_rows128(&km, k, (uint64_t)keys, kTileKeys) != MQA_OK || encode_scales(&sm, scales, keys) != MQA_OK)
    return MQA_ERR_CUDA;
  FusedParams p;
  std::memset(&p, 0, sizeof p);
  p.scales = scales;
  p.weights = weights;
  p.starts = starts;
  p.ends = ends;
  p.logits = logits;
  p.ws = ws;
  p.rows = rows;
  p.keys = keys;
  p.topk = 0;
  p.nblocks = (rows + kBlockRows - 1) / kBlockRows;
  p.cap = 0;
  p.timeout_ns = 4000LL * 1000000LL;
  // split each block's key range so that the grid stays full for few rows
  const int ktiles = (keys + kTileKeys - 1) / kTileKeys;
  int kc = 1;
  while ((long long)p.nblocks * kc < 2LL * d.sms && ktiles / (kc * 2) >= 8) kc *= 2;
  p.key_chunks = kc;
  const long long jobs = (long long)p.nblocks * kc;
  const int ctas = (int)(jobs < d.sms ? jobs : d.sms);
  // the claim counter restarts for every launch; the status word persists
  // across the chunks of one dense call
  if (cudaMemsetAsync(ws, 0, reset_header ? kWsHeaderBytes : sizeof(int32_t), st) != cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  return h32p::launch_logits(qm, km, sm, p, ctas, st) == cudaSuccess ? MQA_OK : MQA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mqa_topk_workspace_bytes_ex(int device, int rows, int heads, size_t *bytes) {
  if (!bytes || rows < 0 || (heads != 32 && heads != 64)) return MQA_ERR_INVALID_ARGUMENT;
  DeviceInfo d;
  int rc = device_info(device, &d);
  if (rc != MQA_OK) return rc;
  if (rows == 0) {
    *bytes = kWsHeaderBytes;
    return MQA_OK;
  }
  const Build b = pick_build(d, rows, heads, false, false, false);
  *bytes = plan_call(d, b, rows, kDefaultSlabCap, 0, true).L.total;
  return MQA_OK;
}

int mqa_topk_workspace_bytes(int device, int rows, size_t *bytes) {
  return mqa_topk_workspace_bytes_ex(device, rows, 32, bytes);
}

int mqa_topk_prefill(const void *q, const void *k, const float *key_scales, const float *weights,
                     const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys, int topk,
                     void *workspace, size_t workspace_bytes, void *stream) {
  return run_fused(q, k, key_scales, weights, starts, ends, out, rows, keys, topk, 32, workspace, workspace_bytes,
                   stream, nullptr);
}

int mqa_topk_prefill_debug(const void *q, const void *k, const float *key_scales, const float *weights,
                           const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys,
                           int topk, void *workspace, size_t workspace_bytes, void *stream,
                           const mqa_topk_debug_options *opt) {
  return run_fused(q, k, key_scales, weights, starts, ends, out, rows, keys, topk, 32, workspace, workspace_bytes,
                   stream, opt);
}

int mqa_block_mask(const int32_t *block_lists, const int32_t *starts, const int32_t *ends, int rows, int list_len,
                   int keys, uint32_t *mask, int mask_words, int32_t *row_items, void *stream) {
  if (rows < 0 || list_len < 0 || keys < 1 || keys > MQA_MAX_KEYS || mask_words % 4 != 0 ||
      (long long)mask_words * 256 < (long long)keys)
    return MQA_ERR_INVALID_ARGUMENT;
  if (rows == 0) return MQA_OK;
  if (!starts || !ends || !mask || !row_items || (list_len > 0 && !block_lists)) return MQA_ERR_INVALID_ARGUMENT;
  if (!aligned(mask, 16)) return MQA_ERR_MISALIGNED;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  return launch_block_mask(block_lists, starts, ends, rows, list_len, keys, mask, mask_words, row_items,
                           as_stream(stream)) == cudaSuccess
             ? MQA_OK
             : MQA_ERR_CUDA;
}

int mqa_topk_prefill_masked(const void *q, const void *k, const float *key_scales, const float *weights,
                            const int32_t *starts, const int32_t *ends, const uint32_t *mask, int mask_words,
                            const int32_t *row_items, int32_t *out, int rows, int keys, int topk, void *workspace,
                            size_t workspace_bytes, void *stream, const mqa_topk_debug_options *opt) {
  if (!mask) return MQA_ERR_INVALID_ARGUMENT;
  return run_fused(q, k, key_scales, weights, starts, ends, out, rows, keys, topk, 32, workspace, workspace_bytes,
                   stream, opt, false, mask, mask_words, row_items);
}

int mqa_block_topk_prefill(const void *q, const void *k, const float *key_scales, const float *weights,
                           const int32_t *starts, const int32_t *ends, int32_t *out_blocks, int rows, int keys,
                           int btopk, void *workspace, size_t workspace_bytes, void *stream,
                           const mqa_topk_debug_options *opt) {
  return run_fused(q, k, key_scales, weights, starts, ends, out_blocks, rows, keys, btopk, 32, workspace,
                   workspace_bytes, stream, opt, true);
}

int mqa_topk_prefill_ex(const void *q, const void *k, const float *key_scales, const float *weights,
                        const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys, int topk,
                        int heads, void *workspace, size_t workspace_bytes, void *stream,
                        const mqa_topk_debug_options *opt) {
  return run_fused(q, k, key_scales, weights, starts, ends, out, rows, keys, topk, heads, workspace,
                   workspace_bytes, stream, opt);
}

int mqa_topk_prefill_noalloc(const void *q, const void *k, const float *key_scales, const float *weights,
                             const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys,
                             int topk, void *stream) {
  int rc = check_common(q, k, key_scales, weights, starts, ends, out, rows, keys);
  if (rc != MQA_OK) return rc;
  if (!valid_topk(topk)) return MQA_ERR_INVALID_ARGUMENT;
  if (rows == 0) return MQA_OK;
  DeviceInfo d;
  rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  // The scratch need is set by the CTA count, which this entry caps: the most
  // CTAs (at most kStaticScratchCtas) whose layout with the key-range split
  // fits the array, else the unsplit layout of up to kStaticScratchCtas CTAs
  // (which always fits).  The call runs the direct head sum (8-row blocks),
  // whose scratch does not grow with rows or keys.
  int ctas = 0;
  for (int c = kStaticScratchCtas; c >= 1 && !ctas; --c) {
    const Plan P = plan_call(d, Build::kPairs, rows, kDefaultSlabCap, c, true);
    if (P.split_max > 0 && P.L.total <= kStaticScratchBytes) ctas = P.ctas;
  }
  if (!ctas) {
    const Plan P = plan_call(d, Build::kPairs, rows, kDefaultSlabCap, kStaticScratchCtas, false);
    if (P.L.total > kStaticScratchBytes) return MQA_ERR_WORKSPACE_TOO_SMALL;
    ctas = P.ctas;
  }
  void *scratch = nullptr;
  if (static_scratch_address(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  mqa_topk_debug_options opt;
  std::memset(&opt, 0, sizeof opt);
  opt.max_ctas = ctas;
  return run_fused(q, k, key_scales, weights, starts, ends, out, rows, keys, topk, 32, scratch,
                   kStaticScratchBytes, stream, &opt, false, nullptr, 0, nullptr, true);
}

int mqa_topk_noalloc_get_status(int32_t *status, int32_t *stats, void *stream) {
  if (!status) return MQA_ERR_INVALID_ARGUMENT;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  void *scratch = nullptr;
  if (static_scratch_address(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  return mqa_topk_get_status(scratch, status, stats, stream);
}

int mqa_ue8m0_decode(const uint8_t *scales, float *out, int keys, void *stream) {
  if (keys < 0 || keys > MQA_MAX_KEYS) return MQA_ERR_INVALID_ARGUMENT;
  if (keys == 0) return MQA_OK;
  if (!scales || !out) return MQA_ERR_INVALID_ARGUMENT;
  if (!aligned(scales, 16) || !aligned(out, 16)) return MQA_ERR_MISALIGNED;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  return launch_ue8m0_decode(scales, out, keys, as_stream(stream)) == cudaSuccess ? MQA_OK : MQA_ERR_CUDA;
}

int mqa_fold_prep(const void *q, const float *weights, uint8_t *codes, int32_t *exps, float *beta, int rows,
                  void *stream) {
  static_assert(MQA_FOLD_TERMS == kFoldTerms, "fold term count");
  if (rows < 0) return MQA_ERR_INVALID_ARGUMENT;
  if (rows == 0) return MQA_OK;
  if (!q || !weights || !codes || !exps || !beta) return MQA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(codes, 16) || !aligned(weights, 4) || !aligned(exps, 4) || !aligned(beta, 4))
    return MQA_ERR_MISALIGNED;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  return launch_fold_prep(reinterpret_cast<const uint8_t *>(q), weights, codes, exps, beta, rows,
                          as_stream(stream)) == cudaSuccess
             ? MQA_OK
             : MQA_ERR_CUDA;
}

int mqa_logits_debug(const void *q, const void *k, const float *key_scales, const float *weights,
                     const int32_t *starts, const int32_t *ends, float *logits, int rows, int keys,
                     void *workspace, size_t workspace_bytes, void *stream) {
  int rc = check_common(q, k, key_scales, weights, starts, ends, logits, rows, keys);
  if (rc != MQA_OK) return rc;
  if (!workspace) return MQA_ERR_INVALID_ARGUMENT;
  if (!aligned(workspace, 256)) return MQA_ERR_MISALIGNED;
  if (workspace_bytes < kWsHeaderBytes) return MQA_ERR_WORKSPACE_TOO_SMALL;
  if (rows == 0) return MQA_OK;
  DeviceInfo d;
  rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  rc = get_encoder();
  if (rc != MQA_OK) return rc;
  return run_logits_chunk(d, reinterpret_cast<const uint8_t *>(q), k, key_scales, weights, starts, ends, logits,
                          rows, keys, reinterpret_cast<int32_t *>(workspace), true, as_stream(stream));
}

int mqa_topk_dense_baseline(const void *q, const void *k, const float *key_scales, const float *weights,
                            const int32_t *starts, const int32_t *ends, int32_t *out, int rows, int keys,
                            int topk, void *logits_ws, size_t logits_budget_bytes, void *workspace,
                            size_t workspace_bytes, void *stream) {
  int rc = check_common(q, k, key_scales, weights, starts, ends, out, rows, keys);
  if (rc != MQA_OK) return rc;
  if (!valid_topk(topk) || !logits_ws || !workspace) return MQA_ERR_INVALID_ARGUMENT;
  if (!aligned(logits_ws, 16)) return MQA_ERR_MISALIGNED;
  if (!aligned(workspace, 256)) return MQA_ERR_MISALIGNED;
  if (workspace_bytes < kWsHeaderBytes) return MQA_ERR_WORKSPACE_TOO_SMALL;
  const size_t row_bytes = (size_t)keys * sizeof(float);
  if (logits_budget_bytes < row_bytes) return MQA_ERR_WORKSPACE_TOO_SMALL;
  if (rows == 0) return MQA_OK;
  DeviceInfo d;
  rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  rc = get_encoder();
  if (rc != MQA_OK) return rc;
  const size_t per_call = logits_budget_bytes / row_bytes;
  const int rows_per_call = per_call > (size_t)rows ? rows : (int)per_call;
  cudaStream_t st = as_stream(stream);
  float *L = reinterpret_cast<float *>(logits_ws);
  int32_t *ws = reinterpret_cast<int32_t *>(workspace);
  const uint8_t *qb = reinterpret_cast<const uint8_t *>(q);
  for (int r0 = 0; r0 < rows; r0 += rows_per_call) {
    const int nr = rows - r0 < rows_per_call ? rows - r0 : rows_per_call;
    rc = run_logits_chunk(d, qb + (size_t)r0 * kHeads * kDim, k, key_scales, weights + (size_t)r0 * kHeads,
                          starts + r0, ends + r0, L, nr, keys, ws, r0 == 0, st);
    if (rc != MQA_OK) return rc;
    if (launch_dense_topk_rows(L, nr, keys, starts + r0, ends + r0, out + (size_t)r0 * topk, topk,
                               ws + kWsStatus, st) != cudaSuccess)
      return MQA_ERR_CUDA;
  }
  return MQA_OK;
}

int mqa_topk_get_status(const void *workspace, int32_t *status, int32_t *stats, void *stream) {
  if (!workspace || !status) return MQA_ERR_INVALID_ARGUMENT;
  int32_t h[kWsWords];
  cudaStream_t st = as_stream(stream);
  if (cudaMemcpyAsync(h, workspace, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  *status = h[kWsStatus];
  if (stats) {
    stats[MQA_STAT_STATUS] = h[kWsStatus];
    stats[MQA_STAT_ROWS_RESCANNED] = h[kWsRowsRescanned];
    stats[MQA_STAT_COMPACTIONS] = h[kWsCompactions];
    stats[MQA_STAT_CANDIDATES] = h[kWsCandidates];
    stats[MQA_STAT_GATED_ROWS] = h[kWsGatedRows];
    stats[MQA_STAT_BLOCKS_DONE] = h[kWsBlocksDone];
    stats[MQA_STAT_SAMPLE_TILES] = h[kWsSampleTiles];
    stats[MQA_STAT_OVERFLOW_ROWS] = h[kWsOverflowRows];
    stats[MQA_STAT_UNDERFILL_ROWS] = h[kWsUnderfillRows];
    stats[MQA_STAT_SELECT_FALLBACK] = h[kWsSelFallback];
    stats[MQA_STAT_SPLIT_BLOCKS] = h[kWsSplitBlocks];
    stats[MQA_STAT_UNSAFE_ROWS] = h[kWsUnsafeRows];
    stats[MQA_STAT_FOLD_BOUND_PPM] = h[kWsFoldBound];
    stats[MQA_STAT_PAIR_ROWS] = h[kWsPairRows];
    stats[MQA_STAT_SKIPPED_TILES] = h[kWsSkippedTiles];
    uint64_t t_start_inv, t_end_inv, t_end;
    memcpy(&t_start_inv, h + kWsTStartMinInv, 8);
    memcpy(&t_end_inv, h + kWsTEndMinInv, 8);
    memcpy(&t_end, h + kWsTEndMax, 8);
    const uint64_t t_start = ~t_start_inv, t_end_min = ~t_end_inv;
    stats[MQA_STAT_KERNEL_US] = (t_end && t_end >= t_start) ? (int32_t)((t_end - t_start) / 1000) : 0;
    stats[MQA_STAT_END_SPREAD_US] = (t_end && t_end >= t_end_min) ? (int32_t)((t_end - t_end_min) / 1000) : 0;
  }
  return MQA_OK;
}

const char *mqa_topk_strerror(int code) {
  switch (code) {
    case MQA_OK: return "ok";
    case MQA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MQA_ERR_MISALIGNED: return "misaligned pointer";
    case MQA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MQA_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case MQA_ERR_CUDA: return "CUDA error";
    case MQA_ERR_NO_DEVICE: return "no CUDA device";
    default: return "unknown error";
  }
}

// Device staging of mqa_topk_prefill_host: q, k, the UE8M0 bytes, the decoded
// scales, weights, starts, ends, out, then the fused op's workspace, each
// 256-byte aligned.
namespace {
struct HostStaging {
  size_t q, k, g, sc, w, s, e, out, ws, total;
};
inline size_t up256(size_t x) { return (x + 255) / 256 * 256; }
HostStaging host_staging(int rows, int keys, int topk, size_t ws_bytes) {
  HostStaging H;
  H.q = 0;
  H.k = H.q + up256((size_t)rows * 32 * kDim);
  H.g = H.k + up256((size_t)keys * kDim);
  H.sc = H.g + up256((size_t)keys * 4);
  H.w = H.sc + up256((size_t)keys * sizeof(float));
  H.s = H.w + up256((size_t)rows * 32 * sizeof(float));
  H.e = H.s + up256((size_t)rows * sizeof(int32_t));
  H.out = H.e + up256((size_t)rows * sizeof(int32_t));
  H.ws = H.out + up256((size_t)rows * topk * sizeof(int32_t));
  H.total = H.ws + up256(ws_bytes);
  return H;
}
}  // namespace

int mqa_topk_host_staging_bytes(int device, int rows, int keys, int topk, size_t *bytes) {
  if (!bytes || rows < 0 || keys < 1 || keys > MQA_MAX_KEYS || !valid_topk(topk)) return MQA_ERR_INVALID_ARGUMENT;
  size_t ws = 0;
  const int rc = mqa_topk_workspace_bytes(device, rows, &ws);
  if (rc != MQA_OK) return rc;
  *bytes = host_staging(rows, keys, topk, ws).total;
  return MQA_OK;
}

int mqa_topk_prefill_host(const void *q_host, const void *k_host, const uint8_t *scales_ue8m0_host,
                          const float *weights_host, const int32_t *starts_host, const int32_t *ends_host,
                          int32_t *out_host, int rows, int keys, int topk, void *staging, size_t staging_bytes,
                          void *stream) {
  if (rows < 0 || keys < 1 || keys > MQA_MAX_KEYS || !valid_topk(topk)) return MQA_ERR_INVALID_ARGUMENT;
  if (rows == 0) return MQA_OK;
  if (!q_host || !k_host || !scales_ue8m0_host || !weights_host || !starts_host || !ends_host || !out_host ||
      !staging)
    return MQA_ERR_INVALID_ARGUMENT;
  if (!aligned(staging, 256)) return MQA_ERR_MISALIGNED;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MQA_ERR_CUDA;
  size_t ws_bytes = 0;
  rc = mqa_topk_workspace_bytes(dev, rows, &ws_bytes);
  if (rc != MQA_OK) return rc;
  const HostStaging H = host_staging(rows, keys, topk, ws_bytes);
  if (staging_bytes < H.total) return MQA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t *b = reinterpret_cast<uint8_t *>(staging);
  cudaStream_t st = as_stream(stream);
  // one plain asynchronous copy per input (pinned host buffers overlap with
  // other streams' work; pageable ones are staged by the runtime)
  const struct { size_t off; const void *src; size_t n; } in[] = {
      {H.q, q_host, (size_t)rows * 32 * kDim},
      {H.k, k_host, (size_t)keys * kDim},
      {H.g, scales_ue8m0_host, (size_t)keys * 4},
      {H.w, weights_host, (size_t)rows * 32 * sizeof(float)},
      {H.s, starts_host, (size_t)rows * sizeof(int32_t)},
      {H.e, ends_host, (size_t)rows * sizeof(int32_t)}};
  for (const auto &c : in) {
    if (cudaMemcpyAsync(b + c.off, c.src, c.n, cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaGetLastError();
      return MQA_ERR_CUDA;
    }
  }
  if (launch_ue8m0_decode(b + H.g, reinterpret_cast<float *>(b + H.sc), keys, st) != cudaSuccess)
    return MQA_ERR_CUDA;
  rc = run_fused(b + H.q, b + H.k, reinterpret_cast<const float *>(b + H.sc),
                 reinterpret_cast<const float *>(b + H.w), reinterpret_cast<const int32_t *>(b + H.s),
                 reinterpret_cast<const int32_t *>(b + H.e), reinterpret_cast<int32_t *>(b + H.out), rows, keys, topk,
                 32, b + H.ws, ws_bytes, stream, nullptr);
  if (rc != MQA_OK) return rc;
  if (cudaMemcpyAsync(out_host, b + H.out, (size_t)rows * topk * sizeof(int32_t), cudaMemcpyDeviceToHost, st) !=
      cudaSuccess) {
    cudaGetLastError();
    return MQA_ERR_CUDA;
  }
  return MQA_OK;
}

int mqa_topk_host_get_status(const void *staging, int rows, int keys, int topk, int32_t *status, int32_t *stats,
                             void *stream) {
  if (!staging || rows < 1 || keys < 1 || keys > MQA_MAX_KEYS || !valid_topk(topk)) return MQA_ERR_INVALID_ARGUMENT;
  const HostStaging H = host_staging(rows, keys, topk, 0);
  return mqa_topk_get_status(reinterpret_cast<const uint8_t *>(staging) + H.ws, status, stats, stream);
}

int mqa_fp8_mma_probe(long long tiles_per_sm, int32_t *status, void *stream) {
  if (tiles_per_sm < 1 || tiles_per_sm > (1LL << 26) || !status) return MQA_ERR_INVALID_ARGUMENT;
  DeviceInfo d;
  const int rc = current_device_info(&d);
  if (rc != MQA_OK) return rc;
  return launch_fp8_mma_probe(tiles_per_sm, status, as_stream(stream)) == cudaSuccess ? MQA_OK : MQA_ERR_CUDA;
}

}  // extern "C"
