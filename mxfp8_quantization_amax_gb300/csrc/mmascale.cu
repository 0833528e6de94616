// mmascale.cu -- block scales rearranged for block-scaled tensor-core MMA.
//
// The pages give no layout for the scales that feed Blackwell's
// block-scaled MMA ("Blackwell GPU MXFP8 预训练最佳实践" 3.2 only says its
// tensor cores take MXFP8/MXFP6/MXFP4 natively).  The library follows
// NVIDIA's public description of that layout.  A scale array of rows x
// scale_cols bytes (the rowwise MX scales [rows][cols / 32], a columnwise
// copy's [cols][blocks], or NVFP4's [rows][cols / 16]) is padded to
// multiples of 128 rows and 4 columns and cut into 128 x 4 blocks of 512
// bytes, stored block row by block row.  Inside a block, element (r, c)
// sits at byte (r % 32) * 16 + (r / 32) * 4 + c: 16-byte row j holds the
// four scales of rows j, j + 32, j + 64, j + 96.  Padding bytes are 0.
//
// A thread writes one 4-byte word of the output (the four scales of one
// row of one block), so the stores are contiguous across the warp; the
// gathered reads are 4 bytes each.
#include "fp8q_device.cuh"
#include "internal.h"

namespace fp8q {

constexpr int kMsThreads = 256;

__global__ void __launch_bounds__(kMsThreads) mma_scale_kernel(const uint8_t* s, int64_t rows, int64_t scale_cols,
                                                               int64_t s_ld, uint32_t* out, int64_t nwords,
                                                               int64_t bcols) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * kMsThreads;
  for (int64_t w = (int64_t)blockIdx.x * kMsThreads + threadIdx.x; w < nwords; w += stride) {
    const int64_t block = w >> 7;            // 128 words per block
    const int k = (int)(w & 127);            // word k: row (k / 4) + 32 * (k % 4) of the block
    const int64_t br = block / bcols, bc = block - br * bcols;
    const int64_t r = br * 128 + (k >> 2) + 32 * (k & 3);
    uint32_t v = 0;
    if (r < rows) {
      const uint8_t* src = s + r * s_ld + 4 * bc;
#pragma unroll
      for (int c = 0; c < 4; c++)
        if (4 * bc + c < scale_cols) v |= (uint32_t)__ldg(src + c) << (8 * c);
    }
    out[w] = v;
  }
  pdl_launch_dependents();
}

fp8q_status launch_mma_scale(const uint8_t* s, int64_t rows, int64_t scale_cols, int64_t s_ld, uint8_t* out,
                             cudaStream_t stream) {
  const int64_t R = (rows + 127) / 128 * 128, bcols = (scale_cols + 3) / 4;
  const int64_t nwords = R * bcols;  // R * 4 * bcols bytes
  int64_t grid = (nwords + kMsThreads - 1) / kMsThreads;
  const int64_t cap = (int64_t)8 * sm_count();
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  cudaError_t e = launch_kernel(mma_scale_kernel, dim3((unsigned)grid), dim3(kMsThreads), 0, stream, s, rows,
                                scale_cols, s_ld, (uint32_t*)out, nwords, bcols);
  if (e != cudaSuccess) return cuda_fail(e, "MMA scale layout kernel launch");
  return check_launch("MMA scale layout kernel");
}

}  // namespace fp8q
