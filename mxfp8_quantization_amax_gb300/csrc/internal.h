// internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/fp8q.h"

namespace fp8q {

// Records `msg` as this thread's last error and returns `st`.
fp8q_status fail(fp8q_status st, const char* fmt, ...);
// Maps a CUDA error to FP8Q_ERR_CUDA with a message naming `what`.
fp8q_status cuda_fail(cudaError_t e, const char* what);
// Checks cudaGetLastError() after launches.
fp8q_status check_launch(const char* what);
// Every argument check of fp8q_cast_per_tensor except the workspace's.
fp8q_status check_cast_args(const void* x, int32_t dt, int64_t rows, int64_t cols, const int64_t* group_offsets,
                            int32_t num_groups, int32_t fmt, int32_t margin, const float* scale_in, const uint8_t* q,
                            const float* amax_out, const float* scale_out, const float* scale_inv_out,
                            const unsigned long long* sat_count_out);

int sm_count();

#ifndef FP8Q_PDL
#define FP8Q_PDL 1
#endif

// Launches kernel<<<grid, block, smem, stream>>>(args...) with programmatic
// stream serialization allowed (the kernel calls pdl_wait() before touching
// global memory), so its launch overlaps the end of the previous kernel.
template <typename... P, typename... A>
cudaError_t launch_kernel(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = FP8Q_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Per-tensor workspace layout (bytes from the start of the workspace).
struct CastWorkspace {
  unsigned* counter;              // [1]  last-CTA ticket
  unsigned* acc;                  // [G]  amax accumulators (FP32 bits)
  float* scale;                   // [G]  current-scaling scales
  unsigned long long* sat;        // [G]  saturation counters
};
size_t cast_workspace_bytes(int G);
CastWorkspace cast_workspace_carve(void* ws, int G);

// Scale sources of the cast kernel.
enum ScaleSrc : int { kSrcGiven = 0, kSrcWorkspace = 1, kSrcHistory = 2 };

struct PtLaunch {
  const void* x;
  int dt;
  int64_t rows, cols;
  const int64_t* off;
  int G;
  int fmt;
  int margin;
  // scale source
  int src;
  const float* scale_in;
  const float* hist;
  int hist_count;
  // workspace / state scratch
  unsigned* counter;
  unsigned* acc;                 // amax accumulators or nullptr (no fused amax)
  float* ws_scale;
  unsigned long long* sat_acc;   // nullptr: no counting
  // outputs
  uint8_t* q;
  float* amax_out;
  float* scale_out;
  float* scale_inv_out;
  unsigned long long* sat_out;
  // delayed-scaling bookkeeping: the recorded amax goes to *hist_slot, a
  // non-finite one sets *flag
  float* hist_slot;
  unsigned* flag;
  // L2 policy for reading x: 0 default, 1 keep (a second pass follows),
  // 2 last use; elements [0, keep_n) take l2_hint_pre instead
  int l2_hint;
  int64_t keep_n;
  int l2_hint_pre;
  cudaStream_t stream;
};

// Tensors up to this size stay in L2 between the amax and the cast pass of
// current scaling; of a larger tensor, a prefix of this size does.
constexpr int64_t kL2KeepBytes = 48ll << 20;

// Amax pass.  finalize_scales: the last CTA turns acc[] into ws_scale[] and
// the scale outputs, writes amax_out / hist_slot / flag and zeroes acc[].
// Otherwise amax accumulates into acc[] (which the caller zeroed).
fp8q_status launch_amax(const PtLaunch& p, bool finalize_scales);
// Cast pass (optionally with fused amax into acc[] and saturation counts).
fp8q_status launch_cast(const PtLaunch& p);
// Current scaling in one launch (amax, scale and cast) for an ungrouped
// tensor: one cluster up to 2 MB, else a cooperative grid with on-chip
// slices and a streamed rest, up to 8 times the on-chip capacity; *taken is
// false, and nothing is launched, for any other tensor.
fp8q_status launch_current_fused(const PtLaunch& p, bool* taken);

// Dequantization; kind 0 per-tensor, 1 MX rowwise copy, 2 MX columnwise copy.
fp8q_status launch_dequant(int kind, const uint8_t* q, const uint8_t* s, const float* scale_inv,
                           const int64_t* off, int G, int64_t rows, int64_t cols, int64_t s_ld, int fmt,
                           int out_dt, void* y, cudaStream_t stream);

// Blockwise FP8 (BF16 input; block 1: 1x128 / 128x1 groups, 128: 128x128).
fp8q_status launch_blockwise(const void* x, int64_t rows, int64_t cols, int fmt, int block, int pow2, int dir,
                             uint8_t* q, float* s, uint8_t* q_t, float* s_t, cudaStream_t stream);
fp8q_status bw_device_status(bool clear, unsigned* word);
fp8q_status bw_set_wait_budget(unsigned long long ns);

// NVFP4 quantization pass (the tensor amax, FP32 bits, is already in amax).
fp8q_status launch_nvfp4(const void* x, int dt, int64_t rows, int64_t cols, const unsigned* amax, uint8_t* q,
                         uint8_t* s, float* scale_out, cudaStream_t stream);

// MXFP8.
fp8q_status launch_mx(const void* x, int dt, int64_t rows, int64_t cols, const int64_t* off, int G,
                      int fmt, int dir, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                      uint8_t* s_col, int64_t s_col_ld, int round_up, unsigned long long* sat,
                      int mma_layout, cudaStream_t stream);

// Device failure words of the MXFP8 pipeline (synchronizes `stream`) and
// of the per-tensor pipeline, and their wait budgets.
fp8q_status mx_device_status(cudaStream_t stream, bool clear, unsigned* word);
fp8q_status mx_set_wait_budget(unsigned long long ns);
fp8q_status mx_set_stall_producer(bool on);
fp8q_status launch_scale(const float* amax, int G, int fmt, int margin, float* scale_out, float* scale_inv_out,
                         cudaStream_t s);
fp8q_status pt_device_status(bool clear, unsigned* word);
fp8q_status pt_set_wait_budget(unsigned long long ns);
fp8q_status pt_set_stall_publish(bool on);
// Zeroes `bytes` (a multiple of 4) at p in stream order with a kernel that
// keeps the chain of programmatic launches (a few counters or accumulators).
fp8q_status launch_zero_words(void* p, size_t bytes, cudaStream_t s);

}  // namespace fp8q
