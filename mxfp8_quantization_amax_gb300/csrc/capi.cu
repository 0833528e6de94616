// capi.cu -- the extern "C" entry points of libfp8q: argument validation,
// error reporting and dispatch to the launchers.  Every check that can be
// made on the host is made here, before anything is launched.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "internal.h"

struct fp8q_delayed_state;

#ifndef FP8Q_PT_KEEP_PREFIX  // current scaling of a tensor larger than L2 keeps a prefix of it there
#define FP8Q_PT_KEEP_PREFIX 1
#endif

namespace fp8q {

fp8q_status delayed_create(int H, int interval, int margin, int fmt, fp8q_delayed_state** out);
fp8q_status delayed_destroy(fp8q_delayed_state* st);
fp8q_status delayed_reset(fp8q_delayed_state* st, cudaStream_t s);
fp8q_status delayed_step(fp8q_delayed_state* st, const void* x, int dt, int64_t n, uint8_t* q,
                         float* scale_used_out, float* scale_inv_out, float* amax_out,
                         unsigned long long* sat_out, cudaStream_t s);
fp8q_status delayed_get(const fp8q_delayed_state* st, float* hist, int32_t* head, int32_t* count,
                        int64_t* step, int32_t* nonfinite);
fp8q_status delayed_set(fp8q_delayed_state* st, const float* hist, int32_t head, int32_t count, int64_t step);
int delayed_history_len(const fp8q_delayed_state* st);

static thread_local char g_err[512];

fp8q_status fail(fp8q_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

fp8q_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FP8Q_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

fp8q_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, what);
}

int sm_count() {
  static int cache[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

size_t cast_workspace_bytes(int G) {
  const size_t a = 64 + (size_t)8 * G;
  return ((a + 7) & ~(size_t)7) + (size_t)8 * G;
}

CastWorkspace cast_workspace_carve(void* ws, int G) {
  char* b = (char*)ws;
  CastWorkspace w;
  w.counter = (unsigned*)b;
  w.acc = (unsigned*)(b + 64);
  w.scale = (float*)(b + 64 + (size_t)4 * G);
  w.sat = (unsigned long long*)(b + ((64 + (size_t)8 * G + 7) & ~(size_t)7));
  return w;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

static fp8q_status check_common(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                const int64_t* off, int32_t G) {
  if (dt != FP8Q_IN_BF16 && dt != FP8Q_IN_FP32) return fail(FP8Q_ERR_INVALID_ARG, "dt must be FP8Q_IN_BF16 or FP8Q_IN_FP32");
  if (rows < 0 || cols < 0) return fail(FP8Q_ERR_INVALID_ARG, "rows and cols must be >= 0");
  if (cols > 0 && rows > (INT64_C(1) << 62) / cols) return fail(FP8Q_ERR_INVALID_ARG, "rows * cols too large");
  if (rows * cols > 0 && x == nullptr) return fail(FP8Q_ERR_INVALID_ARG, "x is NULL");
  if (!aligned(x, 16)) return fail(FP8Q_ERR_INVALID_ARG, "x must be 16-byte aligned");
  if (off == nullptr && G != 1) return fail(FP8Q_ERR_INVALID_ARG, "num_groups must be 1 when group_offsets is NULL");
  if (G < 1 || G > FP8Q_MAX_GROUPS) return fail(FP8Q_ERR_INVALID_ARG, "num_groups must be in [1, %d]", FP8Q_MAX_GROUPS);
  if (off != nullptr && !aligned(off, 8)) return fail(FP8Q_ERR_INVALID_ARG, "group_offsets must be 8-byte aligned");
  return FP8Q_OK;
}

static bool fmt_ok(int32_t fmt) { return fmt == FP8Q_E4M3 || fmt == FP8Q_E5M2; }

// MXFP4 / MXFP6 (mxlow.cu).
fp8q_status low_device_status(bool clear, unsigned* word);
fp8q_status low_set_wait_budget(unsigned long long ns);
fp8q_status launch_mxlow(const void* x, int dt, int64_t rows, int64_t cols, int elem, int dir, int round_up,
                         uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, unsigned long long* sat,
                         cudaStream_t stream);

// Block scales for tensor-core MMA (mmascale.cu).
fp8q_status launch_mma_scale(const uint8_t* s, int64_t rows, int64_t scale_cols, int64_t s_ld, uint8_t* out,
                             cudaStream_t stream);

// Quantization statistics (qstats.cu).
size_t qstats_workspace_bytes();
fp8q_status qs_device_status(bool clear, unsigned* word);
fp8q_status qs_set_wait_budget(unsigned long long ns);
fp8q_status launch_qstats(int kind, const void* x, int dt, const uint8_t* q, const uint8_t* s, const float* scale_inv,
                          const int64_t* off, int G, int64_t rows, int64_t cols, int64_t s_ld, int fmt,
                          fp8q_qstats* out, void* workspace, cudaStream_t stream);

}  // namespace fp8q

using namespace fp8q;

extern "C" {

int32_t fp8q_version(void) { return 10000; }

const char* fp8q_last_error_string(void) { return g_err; }

fp8q_status fp8q_check_device(void* stream) {
  g_err[0] = 0;
  unsigned mx = 0, pt = 0, bw = 0, lo = 0, qs = 0;
  fp8q_status r = mx_device_status((cudaStream_t)stream, true, &mx);
  if (r != FP8Q_OK) return r;
  if ((r = pt_device_status(true, &pt)) != FP8Q_OK) return r;
  if ((r = bw_device_status(true, &bw)) != FP8Q_OK) return r;
  if ((r = low_device_status(true, &lo)) != FP8Q_OK) return r;
  if ((r = qs_device_status(true, &qs)) != FP8Q_OK) return r;
  if ((mx | pt | bw | lo | qs) & 1u)
    return fail(FP8Q_ERR_TIMEOUT, "a bounded device-side wait gave up; the outputs of that call are incomplete");
  return FP8Q_OK;
}

fp8q_status fp8q_set_wait_budget_ns(uint64_t ns) {
  g_err[0] = 0;
  fp8q_status r = mx_set_wait_budget((unsigned long long)ns);
  if (r == FP8Q_OK) r = pt_set_wait_budget((unsigned long long)ns);
  if (r == FP8Q_OK) r = low_set_wait_budget((unsigned long long)ns);
  if (r == FP8Q_OK) r = qs_set_wait_budget((unsigned long long)ns);
  return r != FP8Q_OK ? r : bw_set_wait_budget((unsigned long long)ns);
}

fp8q_status fp8q_debug_stall_mx_producer(int32_t on) {
  g_err[0] = 0;
  return mx_set_stall_producer(on != 0);
}

fp8q_status fp8q_debug_stall_scale_publish(int32_t on) {
  g_err[0] = 0;
  return pt_set_stall_publish(on != 0);
}

fp8q_status fp8q_amax(const void* x, int32_t dt, int64_t rows, int64_t cols, const int64_t* group_offsets,
                      int32_t num_groups, float* amax_out, void* stream) {
  g_err[0] = 0;
  fp8q_status r = check_common(x, dt, rows, cols, group_offsets, num_groups);
  if (r != FP8Q_OK) return r;
  if (!amax_out || !aligned(amax_out, 4)) return fail(FP8Q_ERR_INVALID_ARG, "amax_out must be a 4-byte aligned device pointer");
  cudaStream_t s = (cudaStream_t)stream;
  if ((r = launch_zero_words(amax_out, sizeof(float) * num_groups, s)) != FP8Q_OK) return r;
  if (rows * cols == 0) return FP8Q_OK;
  PtLaunch L{};
  L.x = x;
  L.dt = dt;
  L.rows = rows;
  L.cols = cols;
  L.off = group_offsets;
  L.G = num_groups;
  L.fmt = FP8Q_E4M3;
  L.acc = (unsigned*)amax_out;
  L.stream = s;
  return launch_amax(L, false);
}

fp8q_status fp8q_scale_from_amax(const float* amax, int32_t num_groups, int32_t fmt, int32_t margin,
                                 float* scale_out, float* scale_inv_out, void* stream) {
  g_err[0] = 0;
  if (num_groups < 1 || num_groups > FP8Q_MAX_GROUPS)
    return fail(FP8Q_ERR_INVALID_ARG, "num_groups must be in [1, %d]", FP8Q_MAX_GROUPS);
  if (!fmt_ok(fmt)) return fail(FP8Q_ERR_INVALID_ARG, "fmt must be FP8Q_E4M3 or FP8Q_E5M2");
  if (margin < 0 || margin > 63) return fail(FP8Q_ERR_INVALID_ARG, "margin must be in [0, 63]");
  if (!amax || !scale_out) return fail(FP8Q_ERR_INVALID_ARG, "amax and scale_out must not be NULL");
  if (!aligned(amax, 4) || !aligned(scale_out, 4) || !aligned(scale_inv_out, 4))
    return fail(FP8Q_ERR_INVALID_ARG, "misaligned pointer");
  return launch_scale(amax, num_groups, fmt, margin, scale_out, scale_inv_out, (cudaStream_t)stream);
}

size_t fp8q_cast_workspace_bytes(int32_t num_groups) {
  if (num_groups < 1) num_groups = 1;
  return cast_workspace_bytes(num_groups);
}

}  // extern "C"

namespace fp8q {
fp8q_status check_cast_args(const void* x, int32_t dt, int64_t rows, int64_t cols, const int64_t* group_offsets,
                            int32_t num_groups, int32_t fmt, int32_t margin, const float* scale_in, const uint8_t* q,
                            const float* amax_out, const float* scale_out, const float* scale_inv_out,
                            const unsigned long long* sat_count_out) {
  fp8q_status r = check_common(x, dt, rows, cols, group_offsets, num_groups);
  if (r != FP8Q_OK) return r;
  if (!fmt_ok(fmt)) return fail(FP8Q_ERR_INVALID_ARG, "fmt must be FP8Q_E4M3 or FP8Q_E5M2");
  if (margin < 0 || margin > 63) return fail(FP8Q_ERR_INVALID_ARG, "margin must be in [0, 63]");
  if (rows * cols > 0 && q == nullptr) return fail(FP8Q_ERR_INVALID_ARG, "q is NULL");
  if (!aligned(q, 16)) return fail(FP8Q_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (scale_in && !aligned(scale_in, 4)) return fail(FP8Q_ERR_INVALID_ARG, "scale_in must be 4-byte aligned");
  if (!aligned(amax_out, 4) || !aligned(scale_out, 4) || !aligned(scale_inv_out, 4) || !aligned(sat_count_out, 8))
    return fail(FP8Q_ERR_INVALID_ARG, "misaligned output pointer");
  return FP8Q_OK;
}
}  // namespace fp8q

extern "C" {

fp8q_status fp8q_cast_per_tensor(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                 const int64_t* group_offsets, int32_t num_groups, int32_t fmt,
                                 int32_t margin, const float* scale_in, uint8_t* q, float* amax_out,
                                 float* scale_out, float* scale_inv_out, unsigned long long* sat_count_out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  fp8q_status r = check_cast_args(x, dt, rows, cols, group_offsets, num_groups, fmt, margin, scale_in, q, amax_out,
                                  scale_out, scale_inv_out, sat_count_out);
  if (r != FP8Q_OK) return r;
  if (!workspace || !aligned(workspace, 8)) return fail(FP8Q_ERR_INVALID_ARG, "workspace must be an 8-byte aligned device pointer");
  if (workspace_bytes < cast_workspace_bytes(num_groups))
    return fail(FP8Q_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                cast_workspace_bytes(num_groups));
  const CastWorkspace ws = cast_workspace_carve(workspace, num_groups);
  PtLaunch L{};
  L.x = x;
  L.dt = dt;
  L.rows = rows;
  L.cols = cols;
  L.off = group_offsets;
  L.G = num_groups;
  L.fmt = fmt;
  L.margin = margin;
  L.counter = ws.counter;
  L.ws_scale = ws.scale;
  L.q = q;
  L.sat_acc = sat_count_out ? ws.sat : nullptr;
  L.sat_out = sat_count_out;
  L.stream = (cudaStream_t)stream;
  if (scale_in == nullptr) {
    // current scaling.  A small ungrouped tensor takes one launch that reads
    // x once (launch_current_fused); any other takes the amax pass
    // (publishes scales), then the cast.  The first kL2KeepBytes of x (all of a tensor that small) are kept in L2
    // for the second pass: evict-last in the amax pass, which reads the rest
    // evict-first so that it does not push the prefix out, and evict-first
    // (last use) in the cast.
    const int64_t esz = dt == FP8Q_IN_BF16 ? 2 : 4;
    PtLaunch A = L;
    A.acc = ws.acc;
    A.amax_out = amax_out;
    A.scale_out = scale_out;
    A.scale_inv_out = scale_inv_out;
    bool taken = false;
    if ((r = launch_current_fused(A, &taken)) != FP8Q_OK || taken) return r;
    A.sat_acc = nullptr;
    A.keep_n = FP8Q_PT_KEEP_PREFIX || rows * cols * esz <= kL2KeepBytes ? kL2KeepBytes / esz : 0;
    A.l2_hint_pre = 1;
    A.l2_hint = FP8Q_PT_KEEP_PREFIX ? 2 : 0;
    if ((r = launch_amax(A, true)) != FP8Q_OK) return r;
    L.src = kSrcWorkspace;
    L.keep_n = A.keep_n;
    L.l2_hint_pre = 2;
    L.l2_hint = 0;
    return launch_cast(L);
  }
  L.src = kSrcGiven;
  L.scale_in = scale_in;
  L.acc = amax_out ? ws.acc : nullptr;
  L.amax_out = amax_out;
  L.scale_out = scale_out;
  L.scale_inv_out = scale_inv_out;
  return launch_cast(L);
}

fp8q_status fp8q_delayed_create(int32_t history_len, int32_t interval, int32_t margin, int32_t fmt,
                                fp8q_delayed_state** out) {
  g_err[0] = 0;
  if (!out) return fail(FP8Q_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (history_len < 1 || history_len > 1024) return fail(FP8Q_ERR_INVALID_ARG, "history_len must be in [1, 1024]");
  if (interval < 1) return fail(FP8Q_ERR_INVALID_ARG, "interval must be >= 1");
  if (margin < 0 || margin > 63) return fail(FP8Q_ERR_INVALID_ARG, "margin must be in [0, 63]");
  if (!fmt_ok(fmt)) return fail(FP8Q_ERR_INVALID_ARG, "fmt must be FP8Q_E4M3 or FP8Q_E5M2");
  return delayed_create(history_len, interval, margin, fmt, out);
}

fp8q_status fp8q_delayed_destroy(fp8q_delayed_state* st) {
  g_err[0] = 0;
  if (!st) return FP8Q_OK;
  return delayed_destroy(st);
}

fp8q_status fp8q_delayed_reset(fp8q_delayed_state* st, void* stream) {
  g_err[0] = 0;
  if (!st) return fail(FP8Q_ERR_INVALID_ARG, "state is NULL");
  return delayed_reset(st, (cudaStream_t)stream);
}

fp8q_status fp8q_delayed_step(fp8q_delayed_state* st, const void* x, int32_t dt, int64_t n, uint8_t* q,
                              float* scale_used_out, float* scale_inv_out, float* amax_out,
                              unsigned long long* sat_count_out, void* stream) {
  g_err[0] = 0;
  if (!st) return fail(FP8Q_ERR_INVALID_ARG, "state is NULL");
  fp8q_status r = check_common(x, dt, 1, n, nullptr, 1);
  if (r != FP8Q_OK) return r;
  if (n > 0 && q == nullptr) return fail(FP8Q_ERR_INVALID_ARG, "q is NULL");
  if (!aligned(q, 16)) return fail(FP8Q_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (!aligned(scale_used_out, 4) || !aligned(scale_inv_out, 4) || !aligned(amax_out, 4) || !aligned(sat_count_out, 8))
    return fail(FP8Q_ERR_INVALID_ARG, "misaligned output pointer");
  return delayed_step(st, x, dt, n, q, scale_used_out, scale_inv_out, amax_out, sat_count_out,
                      (cudaStream_t)stream);
}

fp8q_status fp8q_delayed_get(const fp8q_delayed_state* st, float* history_host, int32_t* head, int32_t* count,
                             int64_t* step, int32_t* nonfinite) {
  g_err[0] = 0;
  if (!st) return fail(FP8Q_ERR_INVALID_ARG, "state is NULL");
  return delayed_get(st, history_host, head, count, step, nonfinite);
}

fp8q_status fp8q_delayed_set(fp8q_delayed_state* st, const float* history_host, int32_t head, int32_t count,
                             int64_t step) {
  g_err[0] = 0;
  if (!st) return fail(FP8Q_ERR_INVALID_ARG, "state is NULL");
  const int H = delayed_history_len(st);
  if (head < 0 || head >= H || count < 0 || count > H || step < 0)
    return fail(FP8Q_ERR_INVALID_ARG, "need 0 <= head < %d, 0 <= count <= %d, step >= 0", H, H);
  return delayed_set(st, history_host, head, count, step);
}

int64_t mxfp8_col_blocks(const int64_t* off, int32_t G, int64_t rows) {
  if (rows < 0) return -1;
  if (off == nullptr) return (rows + 31) / 32;
  if (G < 1 || G > FP8Q_MAX_GROUPS || off[0] != 0 || off[G] != rows) return -1;
  int64_t t = 0;
  for (int g = 0; g < G; g++) {
    const int64_t n = off[g + 1] - off[g];
    if (n < 0) return -1;
    t += (n + 31) / 32;
  }
  return t;
}

fp8q_status mxfp8_quantize(const void* x, int32_t dt, int64_t rows, int64_t cols, const int64_t* group_offsets,
                           int32_t num_groups, int32_t fmt, int32_t dir, uint8_t* q_row, uint8_t* s_row,
                           uint8_t* q_col, uint8_t* s_col, int64_t s_col_ld, void* stream) {
  return mxfp8_quantize_rule(x, dt, rows, cols, group_offsets, num_groups, fmt, dir, FP8Q_MX_RULE_UP, q_row,
                             s_row, q_col, s_col, s_col_ld, nullptr, stream);
}

fp8q_status mxfp8_quantize_rule(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                const int64_t* group_offsets, int32_t num_groups, int32_t fmt, int32_t dir,
                                int32_t scale_rule, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                                uint8_t* s_col, int64_t s_col_ld, unsigned long long* sat_count, void* stream) {
  return mxfp8_quantize_ex(x, dt, rows, cols, group_offsets, num_groups, fmt, dir, scale_rule,
                           FP8Q_SCALES_ROW_MAJOR, q_row, s_row, q_col, s_col, s_col_ld, sat_count, stream);
}

int64_t mxfp8_mma_scale_bytes(int64_t rows, int64_t scale_cols) {
  if (rows < 0 || scale_cols < 0) return -1;
  return (rows + 127) / 128 * 128 * ((scale_cols + 3) / 4 * 4);
}

fp8q_status mxfp8_quantize_ex(const void* x, int32_t dt, int64_t rows, int64_t cols, const int64_t* group_offsets,
                              int32_t num_groups, int32_t fmt, int32_t dir, int32_t scale_rule,
                              int32_t scale_layout, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                              int64_t s_col_ld, unsigned long long* sat_count, void* stream) {
  g_err[0] = 0;
  if (scale_layout != FP8Q_SCALES_ROW_MAJOR && scale_layout != FP8Q_SCALES_MMA_128X4)
    return fail(FP8Q_ERR_INVALID_ARG, "scale_layout must be FP8Q_SCALES_ROW_MAJOR or FP8Q_SCALES_MMA_128X4");
  if (scale_rule != FP8Q_MX_RULE_UP && scale_rule != FP8Q_MX_RULE_OCP)
    return fail(FP8Q_ERR_INVALID_ARG, "scale_rule must be FP8Q_MX_RULE_UP or FP8Q_MX_RULE_OCP");
  if (!aligned(sat_count, 8)) return fail(FP8Q_ERR_INVALID_ARG, "sat_count must be 8-byte aligned");
  fp8q_status r = check_common(x, dt, rows, cols, group_offsets, num_groups);
  if (r != FP8Q_OK) return r;
  if (!fmt_ok(fmt)) return fail(FP8Q_ERR_INVALID_ARG, "fmt must be FP8Q_E4M3 or FP8Q_E5M2");
  if (dir != MXFP8_ROW && dir != MXFP8_COL && dir != MXFP8_BOTH)
    return fail(FP8Q_ERR_INVALID_ARG, "dir must be MXFP8_ROW, MXFP8_COL or MXFP8_BOTH");
  if (cols % 32 != 0) return fail(FP8Q_ERR_UNSUPPORTED, "MXFP8 needs cols %% 32 == 0 (cols = %lld)", (long long)cols);
  const bool empty = rows * cols == 0;
  // every check before the first write, so that a rejected call leaves the
  // caller's buffers untouched
  if (!empty) {
    if (rows > INT32_MAX / 2) return fail(FP8Q_ERR_UNSUPPORTED, "rows too large");
    if (dir & MXFP8_ROW) {
      if (!q_row || !s_row) return fail(FP8Q_ERR_INVALID_ARG, "q_row and s_row are required for rowwise output");
      // the rowwise codes of a block leave in one 32-byte store, and every
      // row starts on that alignment since cols % 32 == 0
      if (!aligned(q_row, 32)) return fail(FP8Q_ERR_INVALID_ARG, "q_row must be 32-byte aligned");
    }
    if (dir & MXFP8_COL) {
      if (!q_col || !s_col) return fail(FP8Q_ERR_INVALID_ARG, "q_col and s_col are required for columnwise output");
      if (s_col_ld < (rows + 31) / 32)
        return fail(FP8Q_ERR_INVALID_ARG, "s_col_ld (%lld) is below ceil(rows / 32) = %lld", (long long)s_col_ld,
                    (long long)((rows + 31) / 32));
      if (scale_layout == FP8Q_SCALES_MMA_128X4 && group_offsets == nullptr && s_col_ld != (rows + 31) / 32)
        return fail(FP8Q_ERR_INVALID_ARG, "in the MMA layout s_col_ld is the column block count, ceil(rows / 32)");
    }
  }
  if (sat_count) {  // zeroed even for an empty tensor
    fp8q_status z = launch_zero_words(sat_count, 2 * sizeof(unsigned long long), (cudaStream_t)stream);
    if (z != FP8Q_OK) return z;
  }
  if (empty) return FP8Q_OK;
  if (scale_layout == FP8Q_SCALES_MMA_128X4) {
    // The kernels write every scale; the layout's padding (rows past a
    // multiple of 128, scale columns past a multiple of 4) is cleared here,
    // only for shapes that have some, and for the FP32 path.
    cudaStream_t st = (cudaStream_t)stream;
    if ((dir & MXFP8_ROW) && (rows % 128 != 0 || (cols / 32) % 4 != 0 || dt == FP8Q_IN_FP32)) {
      cudaError_t e = cudaMemsetAsync(s_row, 0, (size_t)mxfp8_mma_scale_bytes(rows, cols / 32), st);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(s_row padding)");
    }
    if ((dir & MXFP8_COL) && (cols % 128 != 0 || s_col_ld % 4 != 0 || dt == FP8Q_IN_FP32)) {
      cudaError_t e = cudaMemsetAsync(s_col, 0, (size_t)mxfp8_mma_scale_bytes(cols, s_col_ld), st);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(s_col padding)");
    }
  }
  return launch_mx(x, dt, rows, cols, group_offsets, num_groups, fmt, dir, q_row, s_row, q_col, s_col, s_col_ld,
                   scale_rule == FP8Q_MX_RULE_UP ? 1 : 0, sat_count, scale_layout == FP8Q_SCALES_MMA_128X4,
                   (cudaStream_t)stream);
}

fp8q_status fp8q_quantize_blockwise(const void* x, int32_t dt, int64_t rows, int64_t cols, int32_t fmt,
                                    int32_t block, int32_t pow2_scales, int32_t dir, uint8_t* q, float* scale_inv,
                                    uint8_t* q_t, float* scale_inv_t, void* stream) {
  g_err[0] = 0;
  if (dt != FP8Q_IN_BF16 && dt != FP8Q_IN_FP32) return fail(FP8Q_ERR_INVALID_ARG, "dt must be FP8Q_IN_BF16 or FP8Q_IN_FP32");
  if (dt != FP8Q_IN_BF16) return fail(FP8Q_ERR_UNSUPPORTED, "blockwise quantization takes BF16 input");
  if (!fmt_ok(fmt)) return fail(FP8Q_ERR_INVALID_ARG, "fmt must be FP8Q_E4M3 or FP8Q_E5M2");
  if (block != FP8Q_BLOCK_1X128 && block != FP8Q_BLOCK_128X128)
    return fail(FP8Q_ERR_INVALID_ARG, "block must be FP8Q_BLOCK_1X128 or FP8Q_BLOCK_128X128");
  if (dir != MXFP8_ROW && dir != MXFP8_COL && dir != MXFP8_BOTH)
    return fail(FP8Q_ERR_INVALID_ARG, "dir must be MXFP8_ROW, MXFP8_COL or MXFP8_BOTH");
  if (rows < 0 || cols < 0) return fail(FP8Q_ERR_INVALID_ARG, "rows and cols must be >= 0");
  if (rows % 16 != 0 || cols % 16 != 0)
    return fail(FP8Q_ERR_UNSUPPORTED, "blockwise quantization needs rows %% 16 == 0 and cols %% 16 == 0");
  if (rows > INT32_MAX / 2 || cols > INT32_MAX / 2) return fail(FP8Q_ERR_UNSUPPORTED, "rows or cols too large");
  if (rows * cols == 0) return FP8Q_OK;
  if (!x || !aligned(x, 16)) return fail(FP8Q_ERR_INVALID_ARG, "x must be a 16-byte aligned device pointer");
  if (dir & MXFP8_ROW) {
    if (!q || !scale_inv) return fail(FP8Q_ERR_INVALID_ARG, "q and scale_inv are required for the rowwise copy");
    if (!aligned(q, 16) || !aligned(scale_inv, 4)) return fail(FP8Q_ERR_INVALID_ARG, "misaligned q or scale_inv");
  }
  if (dir & MXFP8_COL) {
    if (!q_t || !scale_inv_t)
      return fail(FP8Q_ERR_INVALID_ARG, "q_t and scale_inv_t are required for the transposed copy");
    if (!aligned(q_t, 16) || !aligned(scale_inv_t, 4)) return fail(FP8Q_ERR_INVALID_ARG, "misaligned q_t or scale_inv_t");
  }
  return launch_blockwise(x, rows, cols, fmt, block, pow2_scales ? 1 : 0, dir, q, scale_inv, q_t, scale_inv_t,
                          (cudaStream_t)stream);
}

fp8q_status fp8q_quantize_nvfp4(const void* x, int32_t dt, int64_t rows, int64_t cols, uint8_t* q, uint8_t* s,
                                float* amax_out, float* scale_out, void* stream) {
  g_err[0] = 0;
  fp8q_status r = check_common(x, dt, rows, cols, nullptr, 1);
  if (r != FP8Q_OK) return r;
  if (cols % 16 != 0) return fail(FP8Q_ERR_UNSUPPORTED, "NVFP4 needs cols %% 16 == 0 (cols = %lld)", (long long)cols);
  if (!amax_out || !aligned(amax_out, 4)) return fail(FP8Q_ERR_INVALID_ARG, "amax_out must be a 4-byte aligned device pointer");
  if (!aligned(scale_out, 4)) return fail(FP8Q_ERR_INVALID_ARG, "scale_out must be 4-byte aligned");
  if (rows * cols > 0 && (!q || !s)) return fail(FP8Q_ERR_INVALID_ARG, "q and s must not be NULL");
  if (!aligned(q, 8)) return fail(FP8Q_ERR_INVALID_ARG, "q must be 8-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  if ((r = launch_zero_words(amax_out, sizeof(float), st)) != FP8Q_OK) return r;
  if (rows * cols > 0) {
    PtLaunch L{};
    L.x = x;
    L.dt = dt;
    L.rows = rows;
    L.cols = cols;
    L.G = 1;
    L.fmt = FP8Q_E4M3;
    L.acc = (unsigned*)amax_out;
    L.stream = st;
    if ((r = launch_amax(L, false)) != FP8Q_OK) return r;
  }
  return launch_nvfp4(x, dt, rows, cols, (const unsigned*)amax_out, q, s, scale_out, st);
}

size_t fp8q_qstats_workspace_bytes(void) { return qstats_workspace_bytes(); }

static fp8q_status check_qstats_common(const void* x, int32_t dt, int64_t rows, int64_t cols, const int64_t* off,
                                       int32_t G, int32_t fmt, const uint8_t* q, const fp8q_qstats* out,
                                       const void* ws, size_t ws_bytes) {
  fp8q_status r = check_common(x, dt, rows, cols, off, G);
  if (r != FP8Q_OK) return r;
  if (!fmt_ok(fmt)) return fail(FP8Q_ERR_INVALID_ARG, "fmt must be FP8Q_E4M3 or FP8Q_E5M2");
  if (rows * cols > 0 && !q) return fail(FP8Q_ERR_INVALID_ARG, "q must not be NULL");
  if (!out || !aligned(out, 8)) return fail(FP8Q_ERR_INVALID_ARG, "out must be an 8-byte aligned device pointer");
  if (!ws || !aligned(ws, 16)) return fail(FP8Q_ERR_INVALID_ARG, "workspace must be a 16-byte aligned device pointer");
  if (ws_bytes < qstats_workspace_bytes())
    return fail(FP8Q_ERR_INVALID_ARG, "workspace_bytes (%zu) is below fp8q_qstats_workspace_bytes() = %zu", ws_bytes,
                qstats_workspace_bytes());
  return FP8Q_OK;
}

static fp8q_status check_dequant_common(const uint8_t* q, int64_t rows, int64_t cols, const int64_t* off, int G,
                                        int32_t fmt, int32_t out_dt, const void* y) {
  if (rows < 0 || cols < 0) return fail(FP8Q_ERR_INVALID_ARG, "rows and cols must be >= 0");
  if (G < 1 || G > FP8Q_MAX_GROUPS) return fail(FP8Q_ERR_INVALID_ARG, "num_groups must be in [1, %d]", FP8Q_MAX_GROUPS);
  if (off != nullptr && !aligned(off, 8)) return fail(FP8Q_ERR_INVALID_ARG, "group_offsets must be 8-byte aligned");
  if (!fmt_ok(fmt)) return fail(FP8Q_ERR_INVALID_ARG, "fmt must be FP8Q_E4M3 or FP8Q_E5M2");
  if (out_dt != FP8Q_OUT_BF16 && out_dt != FP8Q_OUT_FP32)
    return fail(FP8Q_ERR_INVALID_ARG, "out_dt must be FP8Q_OUT_BF16 or FP8Q_OUT_FP32");
  if (rows * cols > 0 && (!q || !y)) return fail(FP8Q_ERR_INVALID_ARG, "q and y must not be NULL");
  if (!aligned(q, 16) || !aligned(y, 16)) return fail(FP8Q_ERR_INVALID_ARG, "q and y must be 16-byte aligned");
  return FP8Q_OK;
}

fp8q_status fp8q_dequantize_per_tensor(const uint8_t* q, int64_t rows, int64_t cols, const int64_t* group_offsets,
                                       int32_t num_groups, int32_t fmt, const float* scale_inv, int32_t out_dt,
                                       void* y, void* stream) {
  g_err[0] = 0;
  fp8q_status r = check_dequant_common(q, rows, cols, group_offsets, num_groups, fmt, out_dt, y);
  if (r != FP8Q_OK) return r;
  if (!scale_inv || !aligned(scale_inv, 4)) return fail(FP8Q_ERR_INVALID_ARG, "scale_inv must be a 4-byte aligned device pointer");
  if (rows * cols == 0) return FP8Q_OK;
  return launch_dequant(0, q, nullptr, scale_inv, group_offsets, num_groups, rows, cols, 0, fmt, out_dt, y,
                        (cudaStream_t)stream);
}

fp8q_status mxfp8_dequantize(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols,
                             const int64_t* group_offsets, int32_t num_groups, int32_t fmt, int32_t dir,
                             int64_t s_ld, int32_t out_dt, void* y, void* stream) {
  g_err[0] = 0;
  fp8q_status r = check_dequant_common(q, rows, cols, group_offsets, num_groups, fmt, out_dt, y);
  if (r != FP8Q_OK) return r;
  if (dir != MXFP8_ROW && dir != MXFP8_COL) return fail(FP8Q_ERR_INVALID_ARG, "dir must be MXFP8_ROW or MXFP8_COL");
  if (cols % 32 != 0) return fail(FP8Q_ERR_UNSUPPORTED, "MXFP8 needs cols %% 32 == 0 (cols = %lld)", (long long)cols);
  if (rows * cols > 0 && !s) return fail(FP8Q_ERR_INVALID_ARG, "s must not be NULL");
  if (dir == MXFP8_COL && s_ld < (rows + 31) / 32)
    return fail(FP8Q_ERR_INVALID_ARG, "s_ld (%lld) is below ceil(rows / 32) = %lld", (long long)s_ld,
                (long long)((rows + 31) / 32));
  if (rows * cols == 0) return FP8Q_OK;
  return launch_dequant(dir == MXFP8_ROW ? 1 : 2, q, s, nullptr, group_offsets, num_groups, rows, cols, s_ld, fmt,
                        out_dt, y, (cudaStream_t)stream);
}

fp8q_status mx_quantize_fp4_fp6(const void* x, int32_t dt, int64_t rows, int64_t cols, int32_t elem, int32_t dir,
                                int32_t scale_rule, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                unsigned long long* sat_count, void* stream) {
  g_err[0] = 0;
  fp8q_status r = check_common(x, dt, rows, cols, nullptr, 1);
  if (r != FP8Q_OK) return r;
  if (elem != FP8Q_E2M1 && elem != FP8Q_E2M3 && elem != FP8Q_E3M2)
    return fail(FP8Q_ERR_INVALID_ARG, "elem must be FP8Q_E2M1, FP8Q_E2M3 or FP8Q_E3M2");
  if (dir < MXFP8_ROW || dir > MXFP8_BOTH) return fail(FP8Q_ERR_INVALID_ARG, "dir must be MXFP8_ROW, _COL or _BOTH");
  if (scale_rule != FP8Q_MX_RULE_UP && scale_rule != FP8Q_MX_RULE_OCP)
    return fail(FP8Q_ERR_INVALID_ARG, "scale_rule must be FP8Q_MX_RULE_UP or FP8Q_MX_RULE_OCP");
  if (cols % 32 != 0) return fail(FP8Q_ERR_UNSUPPORTED, "MX needs cols %% 32 == 0 (cols = %lld)", (long long)cols);
  if (elem == FP8Q_E2M1 && (dir & MXFP8_COL) && rows % 2 != 0)
    return fail(FP8Q_ERR_UNSUPPORTED, "the packed E2M1 columnwise copy needs an even row count");
  const bool n = rows * cols > 0;
  if ((dir & MXFP8_ROW) && n && (!q_row || !s_row)) return fail(FP8Q_ERR_INVALID_ARG, "q_row and s_row are required");
  if ((dir & MXFP8_COL) && n && (!q_col || !s_col)) return fail(FP8Q_ERR_INVALID_ARG, "q_col and s_col are required");
  if (!aligned(q_row, 16) || !aligned(q_col, 16)) return fail(FP8Q_ERR_INVALID_ARG, "q_row and q_col must be 16-byte aligned");
  if (!aligned(sat_count, 8)) return fail(FP8Q_ERR_INVALID_ARG, "sat_count must be 8-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  if (sat_count) {
    fp8q_status z = launch_zero_words(sat_count, 2 * sizeof(unsigned long long), st);
    if (z != FP8Q_OK) return z;
  }
  if (!n) return FP8Q_OK;
  return launch_mxlow(x, dt, rows, cols, elem, dir, scale_rule == FP8Q_MX_RULE_UP ? 1 : 0, q_row, s_row, q_col, s_col,
                      sat_count, st);
}

fp8q_status mx_scales_to_mma_layout(const uint8_t* s, int64_t rows, int64_t scale_cols, int64_t s_ld, uint8_t* out,
                                    void* stream) {
  g_err[0] = 0;
  if (rows < 0 || scale_cols < 0) return fail(FP8Q_ERR_INVALID_ARG, "rows and scale_cols must be >= 0");
  if (s_ld < scale_cols) return fail(FP8Q_ERR_INVALID_ARG, "s_ld must be >= scale_cols");
  if (scale_cols > 0 && rows > (INT64_C(1) << 40) / (scale_cols + 3))
    return fail(FP8Q_ERR_INVALID_ARG, "rows * scale_cols too large");
  if (rows * scale_cols == 0) return FP8Q_OK;
  if (!s || !out) return fail(FP8Q_ERR_INVALID_ARG, "s and out must not be NULL");
  if (!aligned(out, 4)) return fail(FP8Q_ERR_INVALID_ARG, "out must be 4-byte aligned");
  return launch_mma_scale(s, rows, scale_cols, s_ld, out, (cudaStream_t)stream);
}

fp8q_status fp8q_qstats_per_tensor(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                   const int64_t* group_offsets, int32_t num_groups, int32_t fmt, const uint8_t* q,
                                   const float* scale_inv, fp8q_qstats* out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  fp8q_status r = check_qstats_common(x, dt, rows, cols, group_offsets, num_groups, fmt, q, out, workspace,
                                      workspace_bytes);
  if (r != FP8Q_OK) return r;
  if (!aligned(q, 16)) return fail(FP8Q_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (!scale_inv || !aligned(scale_inv, 4)) return fail(FP8Q_ERR_INVALID_ARG, "scale_inv must be a 4-byte aligned device pointer");
  return launch_qstats(0, x, dt, q, nullptr, scale_inv, group_offsets, num_groups, rows, cols, 0, fmt, out, workspace,
                       (cudaStream_t)stream);
}

fp8q_status mxfp8_qstats(const void* x, int32_t dt, int64_t rows, int64_t cols, const int64_t* group_offsets,
                         int32_t num_groups, int32_t fmt, int32_t dir, const uint8_t* q, const uint8_t* s,
                         int64_t s_ld, fp8q_qstats* out, void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  fp8q_status r = check_qstats_common(x, dt, rows, cols, group_offsets, num_groups, fmt, q, out, workspace,
                                      workspace_bytes);
  if (r != FP8Q_OK) return r;
  if (dir != MXFP8_ROW && dir != MXFP8_COL) return fail(FP8Q_ERR_INVALID_ARG, "dir must be MXFP8_ROW or MXFP8_COL");
  if (cols % 32 != 0) return fail(FP8Q_ERR_UNSUPPORTED, "MXFP8 needs cols %% 32 == 0 (cols = %lld)", (long long)cols);
  if (rows * cols > 0 && !s) return fail(FP8Q_ERR_INVALID_ARG, "s must not be NULL");
  if (dir == MXFP8_ROW && !aligned(q, 16)) return fail(FP8Q_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (dir == MXFP8_COL && s_ld < (rows + 31) / 32)
    return fail(FP8Q_ERR_INVALID_ARG, "s_ld (%lld) is below ceil(rows / 32) = %lld", (long long)s_ld,
                (long long)((rows + 31) / 32));
  return launch_qstats(dir, x, dt, q, s, nullptr, group_offsets, num_groups, rows, cols, s_ld, fmt, out, workspace,
                       (cudaStream_t)stream);
}

}  // extern "C"
