// formats.h -- other block formats of W_down on the single-token paths
// (formats.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace zffn {

struct MatvecArgs;

// Block formats; the values are the ABI's zffn_format codes.
constexpr int kFmtQ4_K = 0, kFmtQ5_K = 1, kFmtQ6_K = 2, kFmtQ5_1 = 3;

bool fmt_valid(int f);
int64_t fmt_row_bytes(int f, int64_t cols);

// Bit-exact fp32 dequantisation of rows x cols weights in format f.
cudaError_t launch_dequant_fmt(int f, const void *blocks, float *out, int64_t rows, int64_t cols,
                               cudaStream_t s);

// Shared memory of the down kernel for W_down in format f (h of every slot,
// quantised, and the warps' chunk buffers).
size_t down_fmt_smem_bytes(int f, int I, int k);

// One token (a.T == 1): the Q4_K gate/up kernel of the single-token path, then
// the down projection with W_down in format wd_fmt (not Q4_K) as its
// programmatic dependent.  a.h is workspace of k * I floats.
cudaError_t launch_token_fmt(const MatvecArgs &a, int wd_fmt, cudaStream_t s);

// The gate/up kernel of the single-token path (ffn_matvec.cu).
__global__ void ffn_gu_kernel(MatvecArgs a);
size_t gu_smem_total(int H, int I, int k);

}  // namespace zffn
