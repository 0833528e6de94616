// delayed.cu -- delayed per-tensor scaling state and step.
//
// "HiFloat8：高性能训练之路" 1.2: the scale of step t comes from the max of
// an amax history buffer (eqs. 3-4, with the safety factor 2^-N); every
// Interval steps the true amax of x_t is computed and appended, the oldest
// entry dropping out once the buffer is full.  Section 3 of that page fixes
// the timing for Interval = 1 (scale with the previous amax, then record the
// current one); 5.2 and "昇腾 950" 3.2: the first step without history uses
// current scaling.  "混合精度与 FP8 训练" 8.2: the amax statistic rides in
// the same pass as the cast.
//
// The host owns step, head and count, so no step synchronizes.  The device
// block holds the history ring plus the step's scratch: the fused amax
// accumulator and the last-CTA ticket (both left at zero after each step),
// the current-scaling scale and the saturation counter.
#include <new>

#include "fp8q_device.cuh"
#include "internal.h"

struct fp8q_delayed_state {
  int device;
  int H, interval, margin, fmt;
  int head, count;
  int64_t step;
  void* dmem;
  float* hist;                 // [H]
  unsigned* acc;               // [1]
  unsigned* counter;           // [1]
  unsigned* flag;              // [1]
  float* scale;                // [1]
  unsigned long long* sat;     // [1]
};

namespace fp8q {

static size_t delayed_bytes(int H) { return (size_t)((H * 4 + 63) / 64) * 64 + 64; }

static void carve(fp8q_delayed_state* st) {
  char* b = (char*)st->dmem;
  const size_t hb = (size_t)((st->H * 4 + 63) / 64) * 64;
  st->hist = (float*)b;
  st->acc = (unsigned*)(b + hb);
  st->counter = (unsigned*)(b + hb + 4);
  st->flag = (unsigned*)(b + hb + 8);
  st->scale = (float*)(b + hb + 12);
  st->sat = (unsigned long long*)(b + hb + 16);
}

// Makes the state's device current for the life of the guard and restores
// the caller's device afterwards, so get / set / destroy synchronize and
// copy on the device that runs the state's steps.
struct DeviceGuard {
  int prev = -1;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Steps and resets are enqueued on the caller's stream, which belongs to
// the current device: it must be the state's.
static fp8q_status delayed_check_device(const fp8q_delayed_state* st) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != st->device)
    return fail(FP8Q_ERR_INVALID_ARG, "the delayed-scaling state lives on device %d but device %d is current",
                st->device, dev);
  return FP8Q_OK;
}

fp8q_status delayed_create(int H, int interval, int margin, int fmt, fp8q_delayed_state** out) {
  fp8q_delayed_state* st = new (std::nothrow) fp8q_delayed_state();
  if (!st) return fail(FP8Q_ERR_CUDA, "out of host memory");
  st->H = H;
  st->interval = interval;
  st->margin = margin;
  st->fmt = fmt;
  cudaError_t e = cudaGetDevice(&st->device);
  if (e != cudaSuccess) {
    delete st;
    return cuda_fail(e, "cudaGetDevice");
  }
  e = cudaMalloc(&st->dmem, delayed_bytes(H));
  if (e != cudaSuccess) {
    delete st;
    return cuda_fail(e, "cudaMalloc(delayed state)");
  }
  e = cudaMemset(st->dmem, 0, delayed_bytes(H));
  if (e != cudaSuccess) {
    cudaFree(st->dmem);
    delete st;
    return cuda_fail(e, "cudaMemset(delayed state)");
  }
  carve(st);
  *out = st;
  return FP8Q_OK;
}

fp8q_status delayed_destroy(fp8q_delayed_state* st) {
  DeviceGuard guard(st->device);
  cudaError_t e = guard.err != cudaSuccess ? guard.err : cudaFree(st->dmem);
  delete st;
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, "cudaFree(delayed state)");
}

fp8q_status delayed_reset(fp8q_delayed_state* st, cudaStream_t s) {
  fp8q_status r0 = delayed_check_device(st);
  if (r0 != FP8Q_OK) return r0;
  cudaError_t e = cudaMemsetAsync(st->dmem, 0, delayed_bytes(st->H), s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(delayed reset)");
  st->head = 0;
  st->count = 0;
  st->step = 0;
  return FP8Q_OK;
}

fp8q_status delayed_step(fp8q_delayed_state* st, const void* x, int dt, int64_t n, uint8_t* q,
                         float* scale_used_out, float* scale_inv_out, float* amax_out,
                         unsigned long long* sat_out, cudaStream_t s) {
  fp8q_status r0 = delayed_check_device(st);
  if (r0 != FP8Q_OK) return r0;
  const bool record = (st->step % st->interval) == 0;
  PtLaunch L{};
  L.x = x;
  L.dt = dt;
  L.rows = 1;
  L.cols = n;
  L.off = nullptr;
  L.G = 1;
  L.fmt = st->fmt;
  L.counter = st->counter;
  L.q = q;
  L.sat_acc = sat_out ? st->sat : nullptr;
  L.sat_out = sat_out;
  L.flag = st->flag;
  L.stream = s;
  fp8q_status r;
  if (st->count == 0) {
    // No history yet: current scaling (margin 0); the amax pass publishes
    // the scale and, on a recording step, the history entry.
    L.margin = 0;
    L.acc = st->acc;
    L.ws_scale = st->scale;
    L.amax_out = record ? amax_out : nullptr;
    L.scale_out = scale_used_out;
    L.scale_inv_out = scale_inv_out;
    L.hist_slot = record ? st->hist + st->head : nullptr;
    if ((r = launch_amax(L, true)) != FP8Q_OK) return r;
    PtLaunch C = L;
    C.src = kSrcWorkspace;
    C.acc = nullptr;
    C.amax_out = nullptr;
    C.hist_slot = nullptr;
    C.flag = nullptr;
    C.scale_out = nullptr;
    C.scale_inv_out = nullptr;
    if ((r = launch_cast(C)) != FP8Q_OK) return r;
  } else {
    L.margin = st->margin;
    L.src = kSrcHistory;
    L.hist = st->hist;
    L.hist_count = st->count;
    L.acc = record ? st->acc : nullptr;
    L.amax_out = record ? amax_out : nullptr;
    L.scale_out = scale_used_out;
    L.scale_inv_out = scale_inv_out;
    L.hist_slot = record ? st->hist + st->head : nullptr;
    if ((r = launch_cast(L)) != FP8Q_OK) return r;
  }
  if (record) {
    st->head = (st->head + 1) % st->H;
    st->count = st->count + 1 < st->H ? st->count + 1 : st->H;
  }
  st->step += 1;
  return FP8Q_OK;
}

int delayed_history_len(const fp8q_delayed_state* st) { return st->H; }

fp8q_status delayed_get(const fp8q_delayed_state* st, float* hist, int32_t* head, int32_t* count,
                        int64_t* step, int32_t* nonfinite) {
  DeviceGuard guard(st->device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice(delayed state)");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  if (hist) {
    e = cudaMemcpy(hist, st->hist, sizeof(float) * st->H, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(history)");
  }
  if (nonfinite) {
    unsigned f = 0;
    e = cudaMemcpy(&f, st->flag, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(flag)");
    *nonfinite = f ? 1 : 0;
  }
  if (head) *head = st->head;
  if (count) *count = st->count;
  if (step) *step = st->step;
  return FP8Q_OK;
}

fp8q_status delayed_set(fp8q_delayed_state* st, const float* hist, int32_t head, int32_t count, int64_t step) {
  DeviceGuard guard(st->device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice(delayed state)");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemset(st->dmem, 0, delayed_bytes(st->H));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(delayed set)");
  if (hist) {
    e = cudaMemcpy(st->hist, hist, sizeof(float) * st->H, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(history)");
  }
  st->head = head;
  st->count = count;
  st->step = step;
  return FP8Q_OK;
}

}  // namespace fp8q
