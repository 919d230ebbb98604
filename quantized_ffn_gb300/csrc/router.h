// router.h -- launcher of the device-side router (router.cu).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace zffn {

// logits fp32 [T][E] -> ids int32 [T][k] (highest logit first, ties to the
// lower index, NaN lowest) and softmax weights fp32 [T][k] over the chosen
// logits.  Requires T >= 1 and 1 <= k <= min(E, 64); returns
// cudaErrorInvalidValue otherwise, without launching.
cudaError_t launch_moe_router(const float *logits, int T, int E, int k, int32_t *ids, float *weights,
                              cudaStream_t s);

}  // namespace zffn
