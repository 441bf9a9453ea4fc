// Auxiliary kernels: UE8M0 key-scale decode, the dense baseline's per-row
// top-k over materialised logits, the block mask of the two-level selection
// and the fold preparation.
#include "mqa_fold.h"
#include "mqa_internal.h"

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include "ptx.cuh"

namespace mqa {

// Key scales arrive as [keys, 4] uint8 UE8M0 groups (four equal bytes); the
// fp32 scale is the float whose bit pattern is (first byte) << 23 (vLLM API
// page `vllm.model_executor.kernels.attention.dsa.fused_mqa_topk`,
// `fused_mqa_topk_key_scales` docstring).  Read as little-endian uint32 words,
// the first byte is the low byte.
__global__ void __launch_bounds__(256) ue8m0_decode_kernel(const uint32_t *__restrict__ groups,
                                                          float *__restrict__ out, int keys) {
  const int n4 = keys >> 2;
  const int stride = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const uint4 g = __ldg(reinterpret_cast<const uint4 *>(groups) + i);
    float4 f;
    f.x = __uint_as_float((g.x & 0xFFu) << 23);
    f.y = __uint_as_float((g.y & 0xFFu) << 23);
    f.z = __uint_as_float((g.z & 0xFFu) << 23);
    f.w = __uint_as_float((g.w & 0xFFu) << 23);
    reinterpret_cast<float4 *>(out)[i] = f;
  }
  for (int j = (n4 << 2) + blockIdx.x * blockDim.x + threadIdx.x; j < keys; j += stride)
    out[j] = __uint_as_float((__ldg(groups + j) & 0xFFu) << 23);
}

cudaError_t launch_ue8m0_decode(const uint8_t *scales, float *out, int keys, cudaStream_t stream) {
  if (keys <= 0) return cudaSuccess;
  const int threads = 256;
  int blocks = ((keys >> 2) + threads - 1) / threads;
  blocks = blocks < 1 ? 1 : (blocks > 4096 ? 4096 : blocks);
  ue8m0_decode_kernel<<<blocks, threads, 0, stream>>>(reinterpret_cast<const uint32_t *>(scales), out, keys);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ dense top-k
// One CTA per row: exact top-k over logits[row, start:end) by four 8-bit
// radix levels on order keys (per-warp histograms, then a CTA sum), then one
// output pass.  Output matches the fused op: relative indices, unordered, -1
// padded.
constexpr int kDenseThreads = 512;
constexpr int kDenseWarps = kDenseThreads / 32;

__global__ void __launch_bounds__(kDenseThreads) dense_topk_kernel(const float *__restrict__ logits, int keys,
                                                                 const int32_t *__restrict__ starts,
                                                                 const int32_t *__restrict__ ends,
                                                                 int32_t *__restrict__ out, int topk,
                                                                 int32_t *ws_status) {
  __shared__ int whist[kDenseWarps][256];
  __shared__ int hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_want, s_gt, s_eq;
  const int row = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int s = starts[row], e = ends[row];
  if ((s < 0 || e > keys) && e > s) {
    if (tid == 0 && ws_status) atomicOr(ws_status, kDevRangeClamped);
    s = max(s, 0);
    e = min(e, keys);
  }
  const int n = e > s ? e - s : 0;
  const float *L = logits + (size_t)row * keys + s;
  int32_t *o = out + (size_t)row * topk;
  if (n <= topk) {
    for (int i = tid; i < topk; i += kDenseThreads) o[i] = i < n ? i : -1;
    return;
  }
  if (tid == 0) {
    s_prefix = 0;
    s_want = topk;
  }
  __syncthreads();
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    const uint32_t hi_mask = level == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    const uint32_t prefix = s_prefix;
    for (int b = lane; b < 256; b += 32) whist[warp][b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kDenseThreads) {
      const uint32_t k = f2key(__ldcs(L + i));
      if ((k & hi_mask) == prefix) atomicAdd(&whist[warp][(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 256) {
      int c = 0;
#pragma unroll
      for (int w = 0; w < kDenseWarps; ++w) c += whist[w][tid];
      hist[tid] = c;
    }
    __syncthreads();
    if (warp == 0) {
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
      const int want = s_want;
      const uint32_t bm = __ballot_sync(0xFFFFFFFFu, excl < want && want <= incl);
      const int src = bm ? __ffs(bm) - 1 : 31;
      if (lane == src) {
        int run = excl;
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= want) {
            s_prefix = prefix | ((uint32_t)(255 - 8 * lane - j) << shift);
            s_want = want - run;
            break;
          }
          run += c[j];
        }
      }
    }
    __syncthreads();
  }
  const uint32_t T = s_prefix;
  const int take_eq = s_want;
  const int ngt = topk - take_eq;
  if (tid == 0) {
    s_gt = 0;
    s_eq = 0;
  }
  __syncthreads();
  for (int i = tid; i < n; i += kDenseThreads) {
    const uint32_t k = f2key(__ldcs(L + i));
    if (k > T) {
      const int pos = atomicAdd(&s_gt, 1);
      if (pos < ngt) o[pos] = i;
    } else if (k == T) {
      const int q = atomicAdd(&s_eq, 1);
      if (q < take_eq) o[ngt + q] = i;
    }
  }
}

cudaError_t launch_dense_topk_rows(const float *logits, int rows, int keys, const int32_t *starts, const int32_t *ends,
                                   int32_t *out, int topk, int32_t *ws_status, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  dense_topk_kernel<<<rows, kDenseThreads, 0, stream>>>(logits, keys, starts, ends, out, topk, ws_status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ block masks
// Masked selection takes, per row, a bit mask over the blocks of 8 keys of the
// key array (bit b % 32 of word b / 32 allows keys [8b, 8b + 8)).  This kernel
// builds it from the candidate-source layer's block lists (block indices
// relative to floor(start / 8), -1 for none; the consumer layers of the
// two-level selection mask their scores to those blocks: vLLM pull request
// #60618, "Limitations of this PR -- TODOs") and counts each row's allowed
// keys inside [start, end), which sizes the row's gate.  One CTA per row.
__global__ void __launch_bounds__(256) block_mask_kernel(const int32_t *__restrict__ lists,
                                                         const int32_t *__restrict__ starts,
                                                         const int32_t *__restrict__ ends, int list_len, int keys,
                                                         uint32_t *__restrict__ mask, int mask_words,
                                                         int32_t *__restrict__ row_items) {
  __shared__ int partial[8];
  const int r = blockIdx.x;
  uint32_t *m = mask + (size_t)r * mask_words;
  for (int w = threadIdx.x; w < mask_words; w += blockDim.x) m[w] = 0u;
  __syncthreads();
  const int s = max(__ldg(starts + r), 0), e = max(s, min(__ldg(ends + r), keys));
  const int b0 = s >> 3, blast = e > s ? (e - 1) >> 3 : b0 - 1;
  int cnt = 0;
  for (int i = threadIdx.x; i < list_len; i += blockDim.x) {
    const int rel = __ldg(lists + (size_t)r * list_len + i);
    if (rel < 0 || rel > blast - b0) continue;
    const int b = b0 + rel;
    const uint32_t bit = 1u << (b & 31);
    if (!(atomicOr(&m[b >> 5], bit) & bit)) cnt += min(e, 8 * b + 8) - max(s, 8 * b);  // first setter counts
  }
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if ((threadIdx.x & 31) == 0) partial[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += partial[i];
    row_items[r] = t;
  }
}

cudaError_t launch_block_mask(const int32_t *lists, const int32_t *starts, const int32_t *ends, int rows,
                              int list_len, int keys, uint32_t *mask, int mask_words, int32_t *row_items,
                              cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  block_mask_kernel<<<rows, 256, 0, stream>>>(lists, starts, ends, list_len, keys, mask, mask_words, row_items);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- the fold
// Folded query of each row and its split into e4m3 terms (vLLM pull request
// #60618, "What this PR does", Scoring bullet: relu(s) = (s + |s|) / 2, so the
// weighted sum of the heads' linear halves is one query, v = sum_h w_h q_h,
// times the key).  One warp per row, lane l owns dimensions 4l .. 4l + 3:
//  - v[d] is formed in fp32 with one fused multiply-add per head, heads in
//    order;
//  - term t: e_t is the smallest integer with max_d |r_t[d]| * 2^-e_t <= 448
//    (0 for a zero residual), u_t[d] = e4m3 round-to-nearest-even of
//    r_t[d] * 2^-e_t, r_{t+1} = r_t - 2^e_t E(u_t) (exact in fp32);
//  - beta = the 2-norm of the last residual, which bounds the linear half's
//    error by beta * |k|_2 for any key k.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// One warp folds row r (lane l owns dimensions 4l .. 4l + 3).
__device__ __forceinline__ void fold_row(const uint8_t *__restrict__ q, const float *__restrict__ w,
                                         uint8_t *__restrict__ codes, int32_t *__restrict__ exps,
                                         float *__restrict__ beta, int r, int lane) {
  const uint8_t *qr = q + (size_t)r * kFoldHeads * kDim;
  const float *wr = w + (size_t)r * kFoldHeads;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  for (int h = 0; h < kFoldHeads; ++h) {
    const float wh = wr[h];
    const uint32_t c4 = *reinterpret_cast<const uint32_t *>(qr + h * kDim + 4 * lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = fmaf(wh, e4m3_value((c4 >> (8 * i)) & 0xFFu), v[i]);
  }
  for (int t = 0; t < kFoldTerms; ++t) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fabsf(v[i]));
    m = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m)));  // non-negative: bits order as values
    int e = 0;
    if (m > 0.f) {
      int ex;
      const float fm = frexpf(m, &ex);
      e = ex - 9 + (fm > 0.875f ? 1 : 0);
    }
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t c = __nv_cvt_float_to_fp8(ldexpf(v[i], -e), __NV_SATFINITE, __NV_E4M3);
      v[i] = v[i] - ldexpf(e4m3_value(c), e);
      packed |= c << (8 * i);
    }
    *reinterpret_cast<uint32_t *>(codes + ((size_t)r * kFoldTerms + t) * kDim + 4 * lane) = packed;
    if (lane == 0) exps[(size_t)r * kFoldTerms + t] = e;
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  if (lane == 0) beta[r] = sqrtf(ss);
}

__global__ void __launch_bounds__(256) fold_prep_kernel(const uint8_t *__restrict__ q, const float *__restrict__ w,
                                                        uint8_t *__restrict__ codes, int32_t *__restrict__ exps,
                                                        float *__restrict__ beta, int rows) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r < rows) fold_row(q, w, codes, exps, beta, r, threadIdx.x & 31);
}

cudaError_t launch_fold_prep(const uint8_t *q, const float *w, uint8_t *codes, int32_t *exps, float *beta, int rows,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  fold_prep_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(q, w, codes, exps, beta, rows);
  return cudaGetLastError();
}

// Per-call preparation for the fold compilation of the fused kernel.  CTAs
// below row_ctas fold 8 rows each (as fold_prep_kernel); the others bound the
// keys: key_scale_j * |k_j|_2 for every key (one thread per key; squares of
// e4m3 values are exact in fp32, the sum and square root round, so the result
// is scaled up by 2^-15 to stay an upper bound), maximised into *key_norm with
// an unsigned atomic max on the fp32 bits (non-negative values order as their
// bits, and every NaN lies above +inf; a NaN code or an infinite scale gives a
// NaN or inf that every row's bound test rejects).
__global__ void __launch_bounds__(256) fold_call_prep_kernel(const uint8_t *__restrict__ q,
                                                             const float *__restrict__ w,
                                                             const uint8_t *__restrict__ k,
                                                             const float *__restrict__ scales,
                                                             uint8_t *__restrict__ codes, int32_t *__restrict__ exps,
                                                             float *__restrict__ beta, int rows, int keys,
                                                             int row_ctas, int32_t *key_norm) {
  const int lane = threadIdx.x & 31;
  if ((int)blockIdx.x < row_ctas) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r < rows) fold_row(q, w, codes, exps, beta, r, lane);
    return;
  }
  float best = 0.f;
  const int stride = (gridDim.x - row_ctas) * blockDim.x;
  for (int j = (blockIdx.x - row_ctas) * blockDim.x + threadIdx.x; j < keys; j += stride) {
    const uint4 *kr = reinterpret_cast<const uint4 *>(k + (size_t)j * kDim);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kDim / 16; ++c) {
      const uint4 u = __ldcs(kr + c);
      const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wv[i] & 0xFFFFu), __NV_E4M3);
        const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wv[i] >> 16), __NV_E4M3);
        const float2 a = __half22float2(__half2(lo)), b = __half22float2(__half2(hi));
        acc = __ffma2_rn(a, a, acc);
        acc = __ffma2_rn(b, b, acc);
      }
    }
    const float n = sqrtf((acc.x + acc.y) * 1.0000153f) * 1.0000153f * __ldg(scales + j);
    best = (n > best || n != n) ? n : best;
  }
  best = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(best)));
  if (lane == 0 && best != 0.f) atomicMax(reinterpret_cast<unsigned *>(key_norm), __float_as_uint(best));
}

cudaError_t launch_fold_call_prep(const uint8_t *q, const float *w, const uint8_t *k, const float *scales,
                                  uint8_t *codes, int32_t *exps, float *beta, int rows, int keys,
                                  int32_t *key_norm, cudaStream_t stream) {
  if (rows <= 0 || keys <= 0) return cudaSuccess;
  const int row_ctas = (rows + 7) / 8;
  int key_ctas = (keys + 255) / 256;
  key_ctas = key_ctas > 1216 ? 1216 : key_ctas;  // 8 per SM of a 152-SM part, grid-stride beyond
  fold_call_prep_kernel<<<row_ctas + key_ctas, 256, 0, stream>>>(q, w, k, scales, codes, exps, beta, rows, keys,
                                                                 row_ctas, key_norm);
  return cudaGetLastError();
}

}  // namespace mqa
