// static_ws.cu -- an allocation-free variant of fp8q_cast_per_tensor.
//
// fp8q_cast_per_tensor needs a small device workspace (amax and saturation
// accumulators, current-scaling scales, a completion counter) that the
// caller allocates.  Some callers cannot allocate device memory at the point
// where they quantize: a plugin running inside a host application whose
// allocator owns all device memory, or a latency-critical step where a
// cudaMalloc / cudaFree would synchronize the device.  For them this file
// keeps the workspace in a fixed array in the library's own device memory.
//
// The array is loaded with the library on every GPU that uses it and stays
// there until the process exits.  Its device address is looked up once per
// device, on that device's first call (so make that first call before any
// stream capture), and kept: a context reset (cudaDeviceReset) is not
// supported, since the array may come back at another address.  Every call
// on a device shares the one array: a call checks its arguments, then
// clears the part it uses, then launches; calls whose work overlaps on the
// GPU (different streams, no ordering between them) race on it.
#include <mutex>

#include "internal.h"

namespace fp8q {

// Largest group count the fixed workspace serves.
constexpr int kStaticWsGroups = 256;
constexpr size_t kStaticWsBytes = 8192;

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

static void* g_static_ws_ptr[64];
static std::mutex g_static_ws_mu;

// Device address of g_static_ws on the current device (looked up once per
// device with that device current).
static fp8q_status static_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(FP8Q_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_static_ws_mu);
  if (g_static_ws_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static workspace)");
    g_static_ws_ptr[dev] = p;
  }
  *out = g_static_ws_ptr[dev];
  return FP8Q_OK;
}

}  // namespace fp8q

using namespace fp8q;

extern "C" fp8q_status fp8q_cast_per_tensor_static_ws(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                                      const int64_t* group_offsets, int32_t num_groups,
                                                      int32_t fmt, int32_t margin, const float* scale_in,
                                                      uint8_t* q, float* amax_out, float* scale_out,
                                                      float* scale_inv_out, unsigned long long* sat_count_out,
                                                      void* stream) {
  if (num_groups < 1 || num_groups > kStaticWsGroups)
    return fail(FP8Q_ERR_INVALID_ARG,
                "fp8q_cast_per_tensor_static_ws serves at most %d groups (got %d); use fp8q_cast_per_tensor "
                "with a caller workspace",
                kStaticWsGroups, num_groups);
  const size_t need = fp8q_cast_workspace_bytes(num_groups);
  if (need > kStaticWsBytes)
    return fail(FP8Q_ERR_INVALID_ARG, "static workspace too small: %zu > %zu bytes", need, kStaticWsBytes);
  // a call that would be rejected must not touch the shared array, which
  // another stream's call may be using
  fp8q_status r = check_cast_args(x, dt, rows, cols, group_offsets, num_groups, fmt, margin, scale_in, q, amax_out,
                                  scale_out, scale_inv_out, sat_count_out);
  if (r != FP8Q_OK) return r;
  void* ws = nullptr;
  r = static_ws_address(&ws);
  if (r != FP8Q_OK) return r;
  // the counters and accumulators must start at zero whatever an earlier call
  // left (a zeroing kernel, which keeps the chain of programmatic launches)
  if ((r = launch_zero_words(ws, need, (cudaStream_t)stream)) != FP8Q_OK) return r;
  return fp8q_cast_per_tensor(x, dt, rows, cols, group_offsets, num_groups, fmt, margin, scale_in, q, amax_out,
                              scale_out, scale_inv_out, sat_count_out, ws, need, stream);
}
