// qstats.cu -- quantization-error statistics of a quantized copy against the
// tensor it was made from: the signal and noise energies behind the SQNR, and
// the counts behind the zero-rate.
//
// "昇腾 Ascend 950 低精度格式", appendix 3.4: weights, activations and KV
// cache are compared between formats by their per-layer SQNR and by their
// zero-rate (how many values quantization set to zero).  The pages define
// neither; the library takes the plain reading.  xh is the FP32 value a code
// stands for: per-tensor fl32(value(q) * scale_inv[g]), MX value(q) * 2^X
// rounded to FP32 (exact unless it reaches 2^128, which gives Inf; scale
// byte 0xFF gives NaN).  Over the elements where x and xh are both finite,
//   signal = sum x^2,   noise = sum (x - xh)^2,   SQNR = 10 log10(signal / noise);
// n_zero counts xh == 0, n_flushed counts xh == 0 with x != 0 (a NaN x is
// not zero) and n_nonfinite the pairs left out of the sums.
//
// Arithmetic.  A thread takes 32 elements at a time (a chunk: one rowwise MX
// block, 32 consecutive per-tensor elements, or a 32-row strip of one column
// of a columnwise copy).  Under one multiplier per chunk it sums x^2 and
// e^2 = (x - xh)^2 in FP32 with fused multiply-adds, two lanes at a time in
// Blackwell's packed f32x2 arithmetic, and adds the chunk sums to FP64
// accumulators.  Each FP32 chunk sum is within 17 units of 2^-24 (relative)
// of the exact sum of its (at most twice rounded) terms when it is finite and
// at least 2^-100 (subnormal roundings then weigh below 2^-45), or is exactly
// a sum of zeros.  Zero values are found on the code words (a code of zero
// magnitude is the only way to a zero value when value * m cannot underflow)
// and counted element by element only in chunks that hold one.  Any other
// chunk -- non-finite or tiny sums, a multiplier that changes inside it (a
// group boundary, the ragged end) -- is summed again element by element in
// FP64, as the oracle does.
//
// Totals.  Each CTA writes its partial sums to the workspace; the last CTA
// to finish (atomic ticket) adds them in a fixed order, so results repeat
// exactly from run to run on one GPU.
#include <cudaTypedefs.h>

#include <mutex>

#include "fp8q_device.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fp8q {

constexpr int kQsThreads = 256;
// The kernels in this file never trigger the next launch early
// (griddepcontrol.launch_dependents): the next grid then starts once this
// one has ended.  Their grids are one wave of resident CTAs with fixed
// shares of the work, and a next grid launched into the slots this one
// frees first was measured to slow both: the three qstats launches of an
// 8192^2 step took 206.8 us with the trigger after the main loop and
// 132.1 us without (38.8 + 57.1 + 39.0 us alone).
constexpr int kQsMaxGrid = 2048;  // partials in the workspace (one per CTA)
constexpr int kQsTileCols = 2 * kQsThreads;  // columnwise: a column pair per thread
#ifndef FP8Q_QS_COL_TMA  // BF16 columnwise copies without groups through the TMA-fed kernel
#define FP8Q_QS_COL_TMA 1
#endif
#ifndef FP8Q_QS_TMA_CTAS_PER_SM  // grid of the TMA-fed kernel: CTAs per SM (its residency is 4)
#define FP8Q_QS_TMA_CTAS_PER_SM 4
#endif
#ifndef FP8Q_QS_CODE_PROMOTION  // L2 promotion of the transposed codes' tensor map
#define FP8Q_QS_CODE_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_128B
#endif

struct QsPartial {
  double signal, noise;
  unsigned long long n, n_zero, n_flushed, n_nonfinite;
};

size_t qstats_workspace_bytes() { return 16 + sizeof(QsPartial) * kQsMaxGrid; }

struct QsParams {
  const void* x;
  const uint8_t* q;
  const uint8_t* s;         // MX scale bytes
  const float* scale_inv;   // per-tensor [G]
  const int64_t* off;       // device row offsets [G + 1] or nullptr
  int G;
  int64_t rows, cols;
  int64_t s_ld;             // columnwise: scale bytes per column
  QsPartial* part;          // [gridDim.x]
  unsigned* counter;        // last-CTA ticket, zero between calls
  fp8q_qstats* out;
};

struct QsAcc {
  double signal = 0.0, noise = 0.0;
  unsigned n = 0, nz = 0, nf = 0, nn = 0;
};

// 2^(byte - 127) as an FP32 value (byte 0: 2^-127, subnormal; 0xFF: NaN).
__device__ __forceinline__ float qs_e8m0(uint32_t byte) {
  if (byte == 0xFFu) return __uint_as_float(0x7FC00000u);
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// Two codes (bits 0-7 and 8-15) -> their exact values.
template <int FMT>
__device__ __forceinline__ void qs_decode2(uint32_t two, float& lo, float& hi) {
  uint32_t h2;
  const unsigned short c = (unsigned short)two;
  if constexpr (FMT == kE4M3)
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  else
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(c));
  asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"((unsigned short)(h2 & 0xFFFFu)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"((unsigned short)(h2 >> 16)));
}

template <int FMT>
__device__ __forceinline__ float qs_value(uint32_t code) {
  float lo, hi;
  qs_decode2<FMT>(code & 0xFFu, lo, hi);
  return lo;
}

template <int DT>
__device__ __forceinline__ float qs_x(const void* x, int64_t i) {
  if constexpr (DT == kBF16)
    return __uint_as_float((uint32_t)__ldg((const unsigned short*)x + i) << 16);
  else
    return __ldg((const float*)x + i);
}

// One element in FP64 (the oracle's own arithmetic); the caller counts n.
__device__ __forceinline__ void qs_elem(QsAcc& a, float x, float xh) {
  if (xh == 0.0f) {
    a.nz++;
    if (!(x == 0.0f)) a.nf++;
  }
  if (!isfinite(x) || !isfinite(xh)) {
    a.nn++;
    return;
  }
  const double e = (double)x - (double)xh;
  a.signal = fma((double)x, (double)x, a.signal);
  a.noise = fma(e, e, a.noise);
}

// Two FP32 lanes in one 64-bit register (Blackwell's packed f32x2 ops).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(f32x2 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(f32x2 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// One pair step: x = X, codes decode to V, multiplier M; S += x^2, N += e^2
// lane by lane, e = x - fl32(v * m).
__device__ __forceinline__ void qs_pair(f32x2 X, f32x2 V, f32x2 M, f32x2& S, f32x2& N) {
  const f32x2 E = f2_sub(X, f2_mul(V, M));
  S = f2_fma(X, X, S);
  N = f2_fma(E, E, N);
}

// Bit 7 of each byte of the result: that code's magnitude bits are nonzero.
__device__ __forceinline__ uint32_t qs_nonzero_codes(uint32_t w) { return (w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu; }

constexpr float kQsSmall = 7.88860905221011805e-31f;  // 2^-100

// Bit 7 + 8k of the result: element k of four has a nonzero magnitude.
// BF16: w0 holds elements 0 and 1, w1 elements 2 and 3 (low half first).
__device__ __forceinline__ uint32_t qs_nonzero_bf16x4(uint32_t w0, uint32_t w1) {
  const uint32_t t0 = (w0 & 0x7FFF7FFFu) + 0x7FFF7FFFu, t1 = (w1 & 0x7FFF7FFFu) + 0x7FFF7FFFu;
  return __byte_perm(t0, t1, 0x7531);
}
// FP32: one element per word.
__device__ __forceinline__ uint32_t qs_nonzero_f32x4(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  const uint32_t t0 = (w0 & 0x7FFFFFFFu) + 0x7FFFFFFFu, t1 = (w1 & 0x7FFFFFFFu) + 0x7FFFFFFFu;
  const uint32_t t2 = (w2 & 0x7FFFFFFFu) + 0x7FFFFFFFu, t3 = (w3 & 0x7FFFFFFFu) + 0x7FFFFFFFu;
  return __byte_perm(__byte_perm(t0, t1, 0x0073), __byte_perm(t2, t3, 0x0073), 0x5410);
}

// Zero counts of four elements: code_nz from qs_nonzero_codes (bit 7 of a
// byte: that code is nonzero), x_nz from qs_nonzero_* (the input is).
__device__ __forceinline__ void qs_count4(QsAcc& a, uint32_t code_nz, uint32_t x_nz) {
  a.nz += __popc(~code_nz & 0x80808080u);
  a.nf += __popc(~code_nz & x_nz & 0x80808080u);
}

// Settles one chunk of 32 elements whose FP32 sums s and n the caller took
// under the single multiplier m, from its registers:
//   code_nz       AND of qs_nonzero_codes over the chunk's code words;
//   x_zero        every x of the chunk is +-0;  codes_zero  every code is;
//   m_exact_zero  xh == 0 exactly when the code is +-0 (value * m cannot
//                 underflow): always for MX scales, and for a finite
//                 per-tensor multiplier of magnitude at least 2^-100;
//   count(a)      adds the chunk's zero counts (qs_count4 per code word).
// The FP32 sums are kept when they are finite (then every pair is finite)
// and each is either at least 2^-100 or exactly a sum of zeros; otherwise
// the chunk is summed again in FP64 from memory (xat(i), code(i)).
template <int FMT, class XF, class CF, class KF>
__device__ __forceinline__ void qs_settle(QsAcc& a, float s, float n, uint32_t code_nz, bool x_zero, bool codes_zero,
                                          bool m_exact_zero, float m, XF xat, CF code, KF count) {
  a.n += 32;
  const bool ok = isfinite(s) && isfinite(n) && m_exact_zero && (s >= kQsSmall || x_zero) &&
                  (n >= kQsSmall || (x_zero && codes_zero));
  if (!ok) {
    for (int i = 0; i < 32; i++) qs_elem(a, xat(i), __fmul_rn(qs_value<FMT>(code(i)), m));
    return;
  }
  a.signal += (double)s;
  a.noise += (double)n;
  if ((code_nz & 0x80808080u) != 0x80808080u) count(a);
}

// Group boundary g, clamped into [0, rows].
__device__ __forceinline__ int64_t qs_row(const QsParams& p, int g) {
  if (p.off == nullptr) return g == 0 ? 0 : p.rows;
  const int64_t v = __ldg(p.off + g);
  return v < 0 ? 0 : (v > p.rows ? p.rows : v);
}

// Last group g with (clamped) off[g] <= r.
__device__ __forceinline__ int qs_group(const QsParams& p, int64_t r) {
  if (p.off == nullptr || p.G <= 1) return 0;
  int lo = 0, hi = p.G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (qs_row(p, mid) <= r) lo = mid; else hi = mid;
  }
  return lo;
}

// Per-tensor: the multiplier of row r, or false for a row in no group.
__device__ __forceinline__ bool qs_tensor_scale(const QsParams& p, int64_t r, float& si) {
  const int g = qs_group(p, r);
  if (r < qs_row(p, g) || r >= qs_row(p, g + 1)) return false;
  si = __ldg(p.scale_inv + g);
  return true;
}

// Columnwise: index of the column block holding row r (blocks of 32 rows
// from each group's first row, numbered over the groups in order), or -1
// for a row in no group.  blk[g]: blocks before group g.
__device__ __forceinline__ int64_t qs_col_block(const QsParams& p, const int* blk, int64_t r) {
  if (p.off == nullptr || p.G <= 1) return r / 32;
  const int g = qs_group(p, r);
  const int64_t r0 = qs_row(p, g);
  if (r < r0 || r >= qs_row(p, g + 1)) return -1;
  return blk[g] + (r - r0) / 32;
}

// blk[g] = sum over h < g of ceil(n_h / 32) (clamped group sizes), g <= G.
__device__ void qs_build_blk(const QsParams& p, int* blk) {
  __shared__ int tot[kQsThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (p.G + kQsThreads - 1) / kQsThreads;
  const int g_lo = tid * per, g_hi = min(p.G, g_lo + per);
  int sum = 0;
  for (int g = g_lo; g < g_hi; g++) {
    const int64_t n = qs_row(p, g + 1) - qs_row(p, g);
    sum += n > 0 ? (int)((n + 31) / 32) : 0;
  }
  int inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) tot[warp] = inc;
  __syncthreads();
  int run = inc - sum;
  for (int w = 0; w < warp; w++) run += tot[w];
  for (int g = g_lo; g < g_hi; g++) {
    blk[g] = run;
    const int64_t n = qs_row(p, g + 1) - qs_row(p, g);
    run += n > 0 ? (int)((n + 31) / 32) : 0;
  }
  if (tid == kQsThreads - 1) blk[p.G] = run;
  __syncthreads();
}

// Block sum of the six totals over NT threads; thread 0 gets the result.
template <int NT = kQsThreads>
__device__ __forceinline__ void qs_block_sum(double& s, double& n, unsigned long long (&c)[4]) {
  __shared__ double sd[2][NT / 32];
  __shared__ unsigned long long sc[4][NT / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
#pragma unroll
    for (int j = 0; j < 4; j++) c[j] += __shfl_xor_sync(0xFFFFFFFFu, c[j], o);
  }
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sd[0][w] = s;
    sd[1][w] = n;
#pragma unroll
    for (int j = 0; j < 4; j++) sc[j][w] = c[j];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    s = n = 0.0;
    for (int j = 0; j < 4; j++) c[j] = 0;
    for (int i = 0; i < NT / 32; i++) {
      s += sd[0][i];
      n += sd[1][i];
      for (int j = 0; j < 4; j++) c[j] += sc[j][i];
    }
  }
}

// The CTA's partial into the workspace; the last CTA adds all partials in
// index order, writes the result and re-arms the ticket.  Every one of the
// CTA's NT threads calls it.
template <int NT = kQsThreads>
__device__ void qs_finish(const QsParams& p, const QsAcc& a) {
  double s = a.signal, n = a.noise;
  unsigned long long c[4] = {a.n, a.nz, a.nf, a.nn};
  qs_block_sum<NT>(s, n, c);
  if (threadIdx.x == 0) {
    QsPartial& d = p.part[blockIdx.x];
    d.signal = s;
    d.noise = n;
    d.n = c[0];
    d.n_zero = c[1];
    d.n_flushed = c[2];
    d.n_nonfinite = c[3];
  }
  __shared__ bool last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(p.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  s = n = 0.0;
  for (int j = 0; j < 4; j++) c[j] = 0;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += NT) {
    const QsPartial* d = p.part + i;
    s += __ldcg(&d->signal);
    n += __ldcg(&d->noise);
    c[0] += __ldcg(&d->n);
    c[1] += __ldcg(&d->n_zero);
    c[2] += __ldcg(&d->n_flushed);
    c[3] += __ldcg(&d->n_nonfinite);
  }
  qs_block_sum<NT>(s, n, c);
  if (threadIdx.x == 0) {
    p.out->signal = s;
    p.out->noise = n;
    p.out->n = c[0];
    p.out->n_zero = c[1];
    p.out->n_flushed = c[2];
    p.out->n_nonfinite = c[3];
    p.out->sqnr_db = n == 0.0 ? (s > 0.0 ? (double)INFINITY : (double)NAN) : 10.0 * log10(s / n);
    p.out->zero_rate = c[0] ? (double)c[2] / (double)c[0] : 0.0;
    *p.counter = 0;
  }
}

// Rowwise MX copy (MX = true: q [rows][cols], s [rows][cols / 32]) or
// per-tensor copy (q [rows][cols], scale_inv [G]), in x's own order.
template <int DT, int FMT, bool MX>
__global__ void __launch_bounds__(kQsThreads) qstats_lin_kernel(QsParams p) {
  pdl_wait();
  QsAcc a;
  const int64_t n = p.rows * p.cols;
  const int64_t nchunk = n / 32;
  const int64_t stride = (int64_t)gridDim.x * kQsThreads;
  const int64_t tid = (int64_t)blockIdx.x * kQsThreads + threadIdx.x;
  constexpr int kXw = DT == kBF16 ? 16 : 32;
  const bool one_scale = MX || p.off == nullptr || p.G <= 1;
  for (int64_t b = tid; b < nchunk; b += stride) {
    uint32_t xw[kXw];
    const char* xp = (const char*)p.x + b * (32 * (DT == kBF16 ? 2 : 4));
#pragma unroll
    for (int j = 0; j < kXw / 4; j++) {
      const uint4 v = ld_stream(xp + 16 * j);
      xw[4 * j] = v.x;
      xw[4 * j + 1] = v.y;
      xw[4 * j + 2] = v.z;
      xw[4 * j + 3] = v.w;
    }
    const uint4 q0 = ld_stream(p.q + 32 * b), q1 = ld_stream(p.q + 32 * b + 16);
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float m;
    bool uniform = true;
    if constexpr (MX) {
      m = qs_e8m0(__ldg(p.s + b));
    } else if (one_scale) {
      m = __ldg(p.scale_inv);
    } else {
      const int64_t r0 = 32 * b / p.cols, r1 = (32 * b + 31) / p.cols;
      const int g = qs_group(p, r0);
      uniform = r0 >= qs_row(p, g) && r1 < qs_row(p, g + 1);
      m = __ldg(p.scale_inv + g);
    }
    const int64_t e0 = 32 * b;
    auto xg = [&](int i) { return qs_x<DT>(p.x, e0 + i); };
    auto cg = [&](int i) { return (uint32_t)__ldg(p.q + e0 + i); };
    if (uniform) {
      // four independent accumulation chains (pairs k % 4), added at the end
      const f32x2 zero2 = f2_make(0.0f, 0.0f);
      f32x2 Sc[4] = {zero2, zero2, zero2, zero2}, Nc[4] = {zero2, zero2, zero2, zero2};
      const f32x2 M = f2_make(m, m);
#pragma unroll
      for (int k = 0; k < 16; k++) {
        float v0, v1;
        qs_decode2<FMT>(qw[k >> 1] >> (16 * (k & 1)), v0, v1);
        f32x2 X;
        if constexpr (DT == kBF16) X = f2_make(bf16_lo(xw[k]), bf16_hi(xw[k]));
        else X = f2_make(__uint_as_float(xw[2 * k]), __uint_as_float(xw[2 * k + 1]));
        qs_pair(X, f2_make(v0, v1), M, Sc[k & 3], Nc[k & 3]);
      }
      const f32x2 S = f2_add(f2_add(Sc[0], Sc[1]), f2_add(Sc[2], Sc[3]));
      const f32x2 N = f2_add(f2_add(Nc[0], Nc[1]), f2_add(Nc[2], Nc[3]));
      uint32_t nzc = 0xFFFFFFFFu, cor = 0u, xor_ = 0u;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        nzc &= qs_nonzero_codes(qw[j]);
        cor |= qw[j] & 0x7F7F7F7Fu;
      }
#pragma unroll
      for (int j = 0; j < kXw; j++) xor_ |= xw[j] & (DT == kBF16 ? 0x7FFF7FFFu : 0x7FFFFFFFu);
      const bool m_exact_zero = MX || (isfinite(m) && fabsf(m) >= kQsSmall);
      auto count = [&](QsAcc& acc) {
#pragma unroll
        for (int j = 0; j < 8; j++) {
          const uint32_t xnz = DT == kBF16 ? qs_nonzero_bf16x4(xw[2 * j], xw[2 * j + 1])
                                           : qs_nonzero_f32x4(xw[4 * j], xw[4 * j + 1], xw[4 * j + 2], xw[4 * j + 3]);
          qs_count4(acc, qs_nonzero_codes(qw[j]), xnz);
        }
      };
      qs_settle<FMT>(a, __fadd_rn(f2_lo(S), f2_hi(S)), __fadd_rn(f2_lo(N), f2_hi(N)), nzc, xor_ == 0u, cor == 0u,
                     m_exact_zero, m, xg, cg, count);
    } else {
      for (int i = 0; i < 32; i++) {
        float si;
        if (qs_tensor_scale(p, (e0 + i) / p.cols, si)) {
          a.n++;
          qs_elem(a, xg(i), __fmul_rn(qs_value<FMT>(cg(i)), si));
        }
      }
    }
  }
  if (tid == 0) {  // the ragged end (per-tensor only: MX rows are whole blocks)
    for (int64_t e = 32 * nchunk; e < n; e++) {
      float si;
      if (qs_tensor_scale(p, e / p.cols, si)) {
        a.n++;
        qs_elem(a, qs_x<DT>(p.x, e), __fmul_rn(qs_value<FMT>(__ldg(p.q + e)), si));
      }
    }
  }
  qs_finish(p, a);
}

// Columnwise MX copy: q [cols][rows], s [cols][s_ld].  Tiles of 32 rows x
// 512 columns, a thread per column pair (c, c + 1): the two columns' codes
// are contiguous in q, the warp's x reads are contiguous along each row,
// and the pair rides the two lanes of the packed FP32 arithmetic.
template <int DT, int FMT>
__global__ void __launch_bounds__(kQsThreads) qstats_col_kernel(QsParams p) {
  extern __shared__ int blk[];  // [G + 1], grouped tensors only
  pdl_wait();
  if (p.off != nullptr && p.G > 1) qs_build_blk(p, blk);
  QsAcc a;
  const int64_t ntr = (p.rows + 31) / 32, ntc = (p.cols + kQsTileCols - 1) / kQsTileCols;
  const int64_t ntiles = ntr * ntc;
  const bool qvec = (p.rows % 16) == 0 && ((uintptr_t)p.q & 15) == 0;
  // tile t = tr * ntc + tc, stepped by the grid size without a division per step
  const int64_t G = gridDim.x, dr = G / ntc, dc = G - dr * ntc;
  int64_t tr = (int64_t)blockIdx.x / ntc, tc = (int64_t)blockIdx.x - tr * ntc;
  for (int64_t t = blockIdx.x; t < ntiles; t += G, tr += dr, tc += dc, (tc >= ntc ? (tc -= ntc, tr++) : 0)) {
    const int64_t c = tc * kQsTileCols + 2 * threadIdx.x;  // cols % 32 == 0: c + 1 < cols too
    if (c >= p.cols) continue;
    const int64_t r0 = tr * 32;
    const int nr = (int)min(p.rows - r0, (int64_t)32);
    const int64_t sb0 = qs_col_block(p, blk, r0);
    const int64_t sb1 = nr == 32 ? qs_col_block(p, blk, r0 + 31) : -2;
    const uint8_t* qa = p.q + c * p.rows + r0;
    const uint8_t* qb = qa + p.rows;
    if (sb0 >= 0 && sb0 == sb1) {  // 32 rows under one scale per column
      const float nan = __uint_as_float(0x7FC00000u);
      const float ma = sb0 < p.s_ld ? qs_e8m0(__ldg(p.s + c * p.s_ld + sb0)) : nan;
      const float mb = sb0 < p.s_ld ? qs_e8m0(__ldg(p.s + (c + 1) * p.s_ld + sb0)) : nan;
      uint32_t wa[8], wb[8];
      if (qvec) {
        const uint4 a0 = ld_stream(qa), a1 = ld_stream(qa + 16), b0 = ld_stream(qb), b1 = ld_stream(qb + 16);
        wa[0] = a0.x; wa[1] = a0.y; wa[2] = a0.z; wa[3] = a0.w; wa[4] = a1.x; wa[5] = a1.y; wa[6] = a1.z; wa[7] = a1.w;
        wb[0] = b0.x; wb[1] = b0.y; wb[2] = b0.z; wb[3] = b0.w; wb[4] = b1.x; wb[5] = b1.y; wb[6] = b1.z; wb[7] = b1.w;
      } else {
#pragma unroll
        for (int j = 0; j < 8; j++) {
          wa[j] = (uint32_t)__ldg(qa + 4 * j) | ((uint32_t)__ldg(qa + 4 * j + 1) << 8) |
                  ((uint32_t)__ldg(qa + 4 * j + 2) << 16) | ((uint32_t)__ldg(qa + 4 * j + 3) << 24);
          wb[j] = (uint32_t)__ldg(qb + 4 * j) | ((uint32_t)__ldg(qb + 4 * j + 1) << 8) |
                  ((uint32_t)__ldg(qb + 4 * j + 2) << 16) | ((uint32_t)__ldg(qb + 4 * j + 3) << 24);
        }
      }
      f32x2 S = f2_make(0.0f, 0.0f), N = S;
      const f32x2 M = f2_make(ma, mb);
      // row i of the pair: BF16 one word (column c low), FP32 two words
      uint32_t xv[DT == kBF16 ? 32 : 64];
#pragma unroll
      for (int i = 0; i < 32; i++) {
        if constexpr (DT == kBF16) {
          xv[i] = __ldg((const unsigned*)((const uint16_t*)p.x + (r0 + i) * p.cols + c));
        } else {
          const float2 w = __ldg((const float2*)((const float*)p.x + (r0 + i) * p.cols + c));
          xv[2 * i] = __float_as_uint(w.x);
          xv[2 * i + 1] = __float_as_uint(w.y);
        }
      }
#pragma unroll
      for (int i = 0; i < 32; i++) {
        const f32x2 X = DT == kBF16 ? f2_make(bf16_lo(xv[i]), bf16_hi(xv[i]))
                                    : f2_make(__uint_as_float(xv[2 * i]), __uint_as_float(xv[2 * i + 1]));
        const int j = i & 3;
        float va, vb;  // row i's code of column c (low byte) and of column c + 1
        qs_decode2<FMT>(__byte_perm(wa[i >> 2], wb[i >> 2], j | ((4 + j) << 4)), va, vb);
        qs_pair(X, f2_make(va, vb), M, S, N);
      }
      uint32_t za = 0xFFFFFFFFu, zb = 0xFFFFFFFFu, ca = 0u, cb = 0u, xa = 0u, xb = 0u;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        za &= qs_nonzero_codes(wa[j]);
        zb &= qs_nonzero_codes(wb[j]);
        ca |= wa[j] & 0x7F7F7F7Fu;
        cb |= wb[j] & 0x7F7F7F7Fu;
      }
#pragma unroll
      for (int i = 0; i < 32; i++) {
        if constexpr (DT == kBF16) {
          xa |= xv[i] & 0x7FFFu;
          xb |= xv[i] & 0x7FFF0000u;
        } else {
          xa |= xv[2 * i] & 0x7FFFFFFFu;
          xb |= xv[2 * i + 1] & 0x7FFFFFFFu;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int64_t cc = c + h;
        const uint8_t* qc = h ? qb : qa;
        auto xg = [&](int i) { return qs_x<DT>(p.x, (r0 + i) * p.cols + cc); };
        auto cg = [&](int i) { return (uint32_t)__ldg(qc + i); };
        auto count = [&](QsAcc& acc) {
#pragma unroll
          for (int j = 0; j < 8; j++) {
            uint32_t t[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
              const int i = 4 * j + k;
              t[k] = DT == kBF16 ? (xv[i] & 0x7FFF7FFFu) + 0x7FFF7FFFu
                                 : (xv[2 * i + h] & 0x7FFFFFFFu) + 0x7FFFFFFFu;
            }
            // bit 15 (column c) or bit 31 (column c + 1, and FP32) of each row
            const uint32_t sel = (DT == kBF16 && h == 0) ? 0x0051u : 0x0073u;
            const uint32_t xnz = __byte_perm(__byte_perm(t[0], t[1], sel), __byte_perm(t[2], t[3], sel), 0x5410);
            qs_count4(acc, qs_nonzero_codes(h ? wb[j] : wa[j]), xnz);
          }
        };
        qs_settle<FMT>(a, h ? f2_hi(S) : f2_lo(S), h ? f2_hi(N) : f2_lo(N), h ? zb : za, (h ? xb : xa) == 0u,
                       (h ? cb : ca) == 0u, true, h ? mb : ma, xg, cg, count);
      }
    } else {
      for (int h = 0; h < 2; h++) {
        const int64_t cc = c + h;
        const uint8_t* qc = h ? qb : qa;
        for (int i = 0; i < nr; i++) {
          const int64_t sb = qs_col_block(p, blk, r0 + i);
          if (sb < 0) continue;
          const float m = sb < p.s_ld ? qs_e8m0(__ldg(p.s + cc * p.s_ld + sb)) : __uint_as_float(0x7FC00000u);
          a.n++;
          qs_elem(a, qs_x<DT>(p.x, (r0 + i) * p.cols + cc), __fmul_rn(qs_value<FMT>(__ldg(qc + i)), m));
        }
      }
    }
  }
  qs_finish(p, a);
}

// ---------------------------------------------------------------------------
// Columnwise MX copy of a BF16 tensor without groups, rows % 32 == 0: TMA-fed
// ---------------------------------------------------------------------------
// A producer warp streams, per block of 32 rows x 256 columns, the x tile
// (four 64-column boxes, 128-byte swizzle: 16 KB) and the block's codes from
// the transposed copy (one box of 32 codes x 256 columns: 8 KB) into a
// two-stage mbarrier ring; four consumer warps take a column pair per thread
// as the kernel above does, reading both from shared memory.  A unit is up
// to 4 blocks of one 256-column strip, so a column's scale bytes of the unit
// are one 4-byte load; each CTA takes a contiguous range of units.  Waits
// are bounded: on expiry the failure word is set, the rest is skipped, and
// the CTA still adds its (then meaningless) partial so that the ticket
// re-arms.
constexpr int kQtCons = 128;
constexpr int kQtThreads = kQtCons + 32;
constexpr int kQtCols = 256;
constexpr int kQtSubCols = 64;
constexpr int kQtSubBytes = 32 * 128;
constexpr int kQtXBytes = 32 * kQtCols * 2;
constexpr int kQtCodeBytes = 32 * kQtCols;
constexpr int kQtStageBytes = kQtXBytes + kQtCodeBytes;
constexpr int kQtStages = 2;
#ifndef FP8Q_QS_TMA_UNIT  // blocks per unit (1..4)
#define FP8Q_QS_TMA_UNIT 4
#endif
constexpr int kQtUnit = FP8Q_QS_TMA_UNIT;
static_assert(kQtUnit >= 1 && kQtUnit <= 4, "a unit's scale bytes of a column fill one word");

__device__ unsigned int g_qs_error;
__device__ unsigned long long g_qs_budget_ns = 1000000000ull;

#ifndef FP8Q_QS_BLOCK_SPLIT  // 1: CTAs take equal ranges of blocks, 0: of whole units
#define FP8Q_QS_BLOCK_SPLIT 1
#endif

// Blocks are numbered unit by unit: row group ti (kQtUnit row blocks, fewer
// in a ragged last group), strip by strip, and within a unit by row block.
// A run is the part of one unit that lies in a CTA's range of blocks.
struct QtRun {
  int64_t ti;    // row group
  int64_t c0;    // first column of the strip
  int j0, j1;    // row blocks [j0, j1) of the unit
  int nblk;      // row blocks in the whole unit
};

__device__ __forceinline__ QtRun qt_run(int b, int b_end, int nbr, int strips) {
  QtRun r;
  const int ti = b / (kQtUnit * strips);
  const int rem = b - ti * kQtUnit * strips;
  r.ti = ti;
  r.nblk = min(kQtUnit, nbr - ti * kQtUnit);
  const int strip = rem / r.nblk;
  r.c0 = (int64_t)strip * kQtCols;
  r.j0 = rem - strip * r.nblk;
  r.j1 = min(r.nblk, r.j0 + (b_end - b));
  return r;
}

template <int FMT>
__global__ void __launch_bounds__(kQtThreads, 4)
    qstats_col_tma_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap qmap,
                          QsParams p) {
  extern __shared__ unsigned char qt_smem[];
  __shared__ uint64_t full[kQtStages], empty[kQtStages];
  __shared__ volatile int abort_flag;
  unsigned char* stages = qt_smem + ((1024 - (smem_u32(qt_smem) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kQtStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kQtCons / 32);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (tid == kQtCons) {
    prefetch_tensormap(&xmap);
    prefetch_tensormap(&qmap);
  }
  pdl_wait();
  __syncthreads();
  const int nbr = (int)(p.rows / 32);
  const int strips = (int)((p.cols + kQtCols - 1) / kQtCols);
  // this CTA's blocks [b_begin, b_end): equal shares of blocks, or of units
  // (block indices fit 32 bits: the launcher checks)
  int b_begin, b_end;
  if (FP8Q_QS_BLOCK_SPLIT) {
    const int64_t blocks = (int64_t)nbr * strips;
    b_begin = (int)(blocks * blockIdx.x / gridDim.x);
    b_end = (int)(blocks * (blockIdx.x + 1) / gridDim.x);
  } else {
    const int64_t units = (nbr + kQtUnit - 1) / kQtUnit * strips;
    const int64_t u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
    // unit u starts at block u * kQtUnit, except in a ragged last row group
    const int64_t full = nbr / kQtUnit * strips;
    b_begin = (int)(u0 <= full ? u0 * kQtUnit : full * kQtUnit + (u0 - full) * (nbr % kQtUnit));
    b_end = (int)(u1 <= full ? u1 * kQtUnit : full * kQtUnit + (u1 - full) * (nbr % kQtUnit));
  }
  const uint64_t budget = g_qs_budget_ns;
  QsAcc a;

  if (warp == kQtCons / 32) {
    // ---------------- producer (lane 0; the warp then joins the finish) ----------------
    if (lane == 0) {
      int64_t k = 0;
      bool stop = false;
      for (int b = b_begin; b < b_end && !abort_flag && !stop;) {
        const QtRun run = qt_run(b, b_end, nbr, strips);
        b += run.j1 - run.j0;
        const int c0 = (int)run.c0;
        const int64_t rb0 = run.ti * kQtUnit;
        for (int j = run.j0; j < run.j1; j++, ++k) {
          const int s = (int)(k % kQtStages);
          const uint32_t round = (uint32_t)(k / kQtStages);
          if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1u, budget)) {
            atomicOr(&g_qs_error, 1u);
            abort_flag = 1;
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(&full[s], kQtStageBytes);
          unsigned char* dst = stages + s * kQtStageBytes;
          const int row = (int)((rb0 + j) * 32);
#pragma unroll
          for (int q = 0; q < kQtCols / kQtSubCols; q++)
            tma_load_2d(dst + q * kQtSubBytes, &xmap, c0 + q * kQtSubCols, row, &full[s]);
          tma_load_2d(dst + kQtXBytes, &qmap, row, c0, &full[s]);
        }
      }
      const int64_t first = k > kQtStages ? k - kQtStages : 0;  // every issued copy lands before the finish
      for (int64_t j = first; j < k; j++)
        mbar_wait(&full[j % kQtStages], (uint32_t)((j / kQtStages) & 1), 2000000000ull);
    }
  } else {
    // ---------------- consumers ----------------
    const float nan = __uint_as_float(0x7FC00000u);
    int64_t k = 0;
    for (int b = b_begin; b < b_end && !abort_flag;) {
      const QtRun run = qt_run(b, b_end, nbr, strips);
      b += run.j1 - run.j0;
      const int64_t c0 = run.c0;
      const int64_t rb0 = run.ti * kQtUnit;
      const int64_t c = c0 + 2 * tid;  // this thread's columns c, c + 1
      const bool col_ok = c < p.cols;
      // the two columns' scale bytes of the run's blocks (byte j of the unit)
      uint32_t sa = 0, sb = 0;
      if (col_ok) {
        const uint8_t* ea = p.s + c * p.s_ld + rb0;
        const uint8_t* eb = ea + p.s_ld;
        if (run.j0 == 0 && run.j1 == kQtUnit && rb0 + kQtUnit <= p.s_ld &&
            (((uintptr_t)ea | (uintptr_t)eb) & 3u) == 0) {
          sa = __ldg((const unsigned*)ea);
          sb = __ldg((const unsigned*)eb);
        } else {
          for (int j = run.j0; j < run.j1 && rb0 + j < p.s_ld; j++) {
            sa |= (uint32_t)__ldg(ea + j) << (8 * j);
            sb |= (uint32_t)__ldg(eb + j) << (8 * j);
          }
        }
      }
      bool gave_up = false;
      for (int j = run.j0; j < run.j1; j++, ++k) {
        const int s = (int)(k % kQtStages);
        const uint32_t round = (uint32_t)(k / kQtStages);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], round & 1u, budget))) {
          atomicOr(&g_qs_error, 1u);
          abort_flag = 1;
          gave_up = true;
          break;
        }
        const unsigned char* stage = stages + s * kQtStageBytes;
        if (col_ok) {
          const int64_t r0 = (rb0 + j) * 32;
          const bool in_ld = rb0 + j < p.s_ld;
          const float ma = in_ld ? qs_e8m0((sa >> (8 * j)) & 0xFFu) : nan;
          const float mb = in_ld ? qs_e8m0((sb >> (8 * j)) & 0xFFu) : nan;
          // x: row i's word holds columns c (low half) and c + 1
          const unsigned char* xs = stage + (tid >> 5) * kQtSubBytes + 4 * (tid & 3);
          const int ch = (tid & 31) >> 2;
          uint32_t xv[32];
#pragma unroll
          for (int i = 0; i < 32; i++) xv[i] = *(const uint32_t*)(xs + i * 128 + ((ch ^ (i & 7)) << 4));
          // codes: column c's 32 bytes, then column c + 1's
          const uint4* qs = (const uint4*)(stage + kQtXBytes + 64 * tid);
          const uint4 a0 = qs[0], a1 = qs[1], b0 = qs[2], b1 = qs[3];
          const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
          // four independent accumulation chains (rows i % 4), added at the end
          const f32x2 zero2 = f2_make(0.0f, 0.0f);
          f32x2 Sc[4] = {zero2, zero2, zero2, zero2}, Nc[4] = {zero2, zero2, zero2, zero2};
          const f32x2 M = f2_make(ma, mb);
#pragma unroll
          for (int i = 0; i < 32; i++) {
            const int jj = i & 3;
            float va, vb;
            qs_decode2<FMT>(__byte_perm(wa[i >> 2], wb[i >> 2], jj | ((4 + jj) << 4)), va, vb);
            qs_pair(f2_make(bf16_lo(xv[i]), bf16_hi(xv[i])), f2_make(va, vb), M, Sc[jj], Nc[jj]);
          }
          const f32x2 S = f2_add(f2_add(Sc[0], Sc[1]), f2_add(Sc[2], Sc[3]));
          const f32x2 N = f2_add(f2_add(Nc[0], Nc[1]), f2_add(Nc[2], Nc[3]));
          uint32_t za = 0xFFFFFFFFu, zb = 0xFFFFFFFFu;
#pragma unroll
          for (int w = 0; w < 8; w++) {
            za &= qs_nonzero_codes(wa[w]);
            zb &= qs_nonzero_codes(wb[w]);
          }
          // whether every x / every code of a column is +-0: settling needs
          // it only for a chunk whose sums fall below 2^-100
          const bool small = !(fminf(fminf(f2_lo(S), f2_hi(S)), fminf(f2_lo(N), f2_hi(N))) >= kQsSmall);
          uint32_t ca = 1u, cb = 1u, xa = 1u, xb = 1u;
          if (small) {
            ca = cb = xa = xb = 0u;
#pragma unroll
            for (int w = 0; w < 8; w++) {
              ca |= wa[w] & 0x7F7F7F7Fu;
              cb |= wb[w] & 0x7F7F7F7Fu;
            }
#pragma unroll
            for (int i = 0; i < 32; i++) {
              xa |= xv[i] & 0x7FFFu;
              xb |= xv[i] & 0x7FFF0000u;
            }
          }
#pragma unroll
          for (int h = 0; h < 2; h++) {
            const int64_t cc = c + h;
            const uint8_t* qc = p.q + cc * p.rows + r0;
            auto xg = [&](int i) { return qs_x<kBF16>(p.x, (r0 + i) * p.cols + cc); };
            auto cg = [&](int i) { return (uint32_t)__ldg(qc + i); };
            auto count = [&](QsAcc& acc) {
#pragma unroll
              for (int w = 0; w < 8; w++) {
                uint32_t t[4];
#pragma unroll
                for (int q = 0; q < 4; q++) t[q] = (xv[4 * w + q] & 0x7FFF7FFFu) + 0x7FFF7FFFu;
                // bit 15 (column c) or bit 31 (column c + 1) of each row
                const uint32_t sel = h == 0 ? 0x0051u : 0x0073u;
                const uint32_t xnz = __byte_perm(__byte_perm(t[0], t[1], sel), __byte_perm(t[2], t[3], sel), 0x5410);
                qs_count4(acc, qs_nonzero_codes(h ? wb[w] : wa[w]), xnz);
              }
            };
            qs_settle<FMT>(a, h ? f2_hi(S) : f2_lo(S), h ? f2_hi(N) : f2_lo(N), h ? zb : za, (h ? xb : xa) == 0u,
                           (h ? cb : ca) == 0u, true, h ? mb : ma, xg, cg, count);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (gave_up) break;
    }
  }
  qs_finish<kQtThreads>(p, a);
}

static PFN_cuTensorMapEncodeTiled_v12000 qs_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}

// Launches the TMA-fed columnwise kernel; *used = false when the call does
// not qualify (grouped, FP32, ragged rows, unaligned buffers) or no tensor
// map could be encoded, and the caller takes the kernel above.
template <int FMT>
static cudaError_t qs_col_tma(const QsParams& p, cudaStream_t stream, bool* used) {
  *used = false;
  if (!(p.off == nullptr || p.G <= 1) || p.rows % 32 != 0 || p.rows <= 0 || p.cols <= 0 ||
      ((uintptr_t)p.x & 15u) != 0 || ((uintptr_t)p.q & 15u) != 0)
    return cudaSuccess;
  auto enc = qs_encode_fn();
  if (!enc) return cudaSuccess;
  CUtensorMap xmap, qmap;
  {
    cuuint64_t dims[2] = {(cuuint64_t)p.cols, (cuuint64_t)p.rows};
    cuuint64_t strides[1] = {(cuuint64_t)p.cols * 2};
    cuuint32_t box[2] = {kQtSubCols, 32};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaSuccess;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)p.rows, (cuuint64_t)p.cols};
    cuuint64_t strides[1] = {(cuuint64_t)p.rows};
    cuuint32_t box[2] = {32, kQtCols};
    cuuint32_t estr[2] = {1, 1};
    // 128-byte L2 promotion: a unit's codes of a column are 4 x 32 bytes, and
    // a 256-byte fill also fetches the next unit's, which another CTA reads
    // much later (measured with 256: 1.10x the algorithmic DRAM reads, and
    // 161.2 against 148.8 us at 16384 x 14336)
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, FP8Q_QS_CODE_PROMOTION,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaSuccess;
  }
  auto kernel = qstats_col_tma_kernel<FMT>;
  constexpr size_t smem = 1024 + (size_t)kQtStages * kQtStageBytes;
  static bool attr = false;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr = true;
    }
  }
  const int64_t blocks = p.rows / 32 * ((p.cols + kQtCols - 1) / kQtCols);
  if (blocks >= INT32_MAX) return cudaSuccess;  // block indices are 32-bit in the kernel
  // each CTA a contiguous range of blocks: one wave of resident CTAs (every
  // CTA ends with a block reduction and a ticket, which many small CTAs
  // would repeat), at most one CTA per block
  int64_t grid = (int64_t)FP8Q_QS_TMA_CTAS_PER_SM * sm_count();
  if (grid > blocks) grid = blocks;
  if (grid > kQsMaxGrid) grid = kQsMaxGrid;
  *used = true;
  return launch_kernel(kernel, dim3((unsigned)grid), dim3(kQtThreads), smem, stream, xmap, qmap, p);
}

fp8q_status qs_device_status(bool clear, unsigned* word) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_qs_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (clear && v) {
    const unsigned z = 0;
    e = cudaMemcpyToSymbol(g_qs_error, &z, sizeof(z));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
  }
  *word = v;
  return FP8Q_OK;
}

fp8q_status qs_set_wait_budget(unsigned long long ns) {
  cudaError_t e = cudaMemcpyToSymbol(g_qs_budget_ns, &ns, sizeof(ns));
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, "cudaMemcpyToSymbol(wait budget)");
}

template <class K>
static int qs_grid(K kernel, size_t smem, int64_t units) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kQsThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  int64_t g = (int64_t)per_sm * sm_count();
  if (g > kQsMaxGrid) g = kQsMaxGrid;
  if (units < g) g = units;
  return g < 1 ? 1 : (int)g;
}

template <int DT, int FMT>
static fp8q_status qs_launch_typed(int kind, QsParams p, cudaStream_t stream) {
  cudaError_t e;
  if (kind == 2) {
    if constexpr (DT == kBF16 && FP8Q_QS_COL_TMA) {
      bool used = false;
      e = qs_col_tma<FMT>(p, stream, &used);
      if (e != cudaSuccess) return cuda_fail(e, "quantization statistics kernel launch");
      if (used) return check_launch("quantization statistics kernel");
    }
    const size_t smem = (p.off != nullptr && p.G > 1) ? sizeof(int) * (size_t)(p.G + 1) : 0;
    const int64_t tiles = ((p.rows + 31) / 32) * ((p.cols + kQsTileCols - 1) / kQsTileCols);
    const int grid = qs_grid(qstats_col_kernel<DT, FMT>, smem, tiles);
    e = launch_kernel(qstats_col_kernel<DT, FMT>, dim3(grid), dim3(kQsThreads), smem, stream, p);
  } else {
    const int64_t chunks = (p.rows * p.cols / 32 + kQsThreads - 1) / kQsThreads;
    if (kind == 1) {
      const int grid = qs_grid(qstats_lin_kernel<DT, FMT, true>, 0, chunks);
      e = launch_kernel(qstats_lin_kernel<DT, FMT, true>, dim3(grid), dim3(kQsThreads), 0, stream, p);
    } else {
      const int grid = qs_grid(qstats_lin_kernel<DT, FMT, false>, 0, chunks);
      e = launch_kernel(qstats_lin_kernel<DT, FMT, false>, dim3(grid), dim3(kQsThreads), 0, stream, p);
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "quantization statistics kernel launch");
  return check_launch("quantization statistics kernel");
}

fp8q_status launch_qstats(int kind, const void* x, int dt, const uint8_t* q, const uint8_t* s, const float* scale_inv,
                          const int64_t* off, int G, int64_t rows, int64_t cols, int64_t s_ld, int fmt,
                          fp8q_qstats* out, void* workspace, cudaStream_t stream) {
  QsParams p{};
  p.x = x;
  p.q = q;
  p.s = s;
  p.scale_inv = scale_inv;
  p.off = off;
  p.G = G;
  p.rows = rows;
  p.cols = cols;
  p.s_ld = s_ld;
  p.counter = (unsigned*)workspace;
  p.part = (QsPartial*)((char*)workspace + 16);
  p.out = out;
  if (dt == kBF16)
    return fmt == kE4M3 ? qs_launch_typed<kBF16, kE4M3>(kind, p, stream) : qs_launch_typed<kBF16, kE5M2>(kind, p, stream);
  return fmt == kE4M3 ? qs_launch_typed<kFP32, kE4M3>(kind, p, stream) : qs_launch_typed<kFP32, kE5M2>(kind, p, stream);
}

}  // namespace fp8q
