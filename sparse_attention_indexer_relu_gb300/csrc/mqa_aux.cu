// Auxiliary kernels: UE8M0 key-scale decode and the dense baseline's per-row
// top-k over materialised logits.
#include "mqa_internal.h"
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

}  // namespace mqa
