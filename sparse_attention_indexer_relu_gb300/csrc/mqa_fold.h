// Fold preparation: the folded query v = sum_h w_h q_h of each row written as
// e4m3 terms with power-of-two scales (kernel in mqa_aux.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace mqa {
constexpr int kFoldHeads = 32;  // index heads the fold preparation takes
constexpr int kFoldTerms = 4;   // e4m3 terms of the folded query
cudaError_t launch_fold_prep(const uint8_t *q, const float *w, uint8_t *codes, int32_t *exps, float *beta, int rows,
                             cudaStream_t stream);
}  // namespace mqa
