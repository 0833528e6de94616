// dequant.cu -- FP8 codes back to BF16 or FP32: per-tensor (per-group) and
// MXFP8 (rowwise copy, or the columnwise copy in its own transposed layout).
//
// "HiFloat8：高性能训练之路" 1.1-1.2: a quantized tensor is de-scaled by
// scale_inv = 1 / Scale.  "Blackwell GPU MXFP8 预训练最佳实践" 4.1 and 4.3:
// an MX element stands for value * 2^X (X = scale byte - 127, byte 0xFF is
// NaN); without MX hardware the blocks are dequantized to BF16 and an
// ordinary BF16 matmul runs.
//
// Arithmetic.  A code is decoded exactly (packed e4m3x2 / e5m2x2 -> f16x2
// conversion, then f16 -> f32).  Per-tensor: y = fl32(value * scale_inv),
// then the output rounding.  MX: value * 2^X is exact in FP32 except for
// overflow to Inf.  BF16 output rounds to nearest, ties to even; every NaN
// result is written as the canonical quiet NaN (BF16 0x7FC0, FP32
// 0x7FC00000).
//
// Work split.  A thread converts 16 codes (one 16-byte load) per vector and
// keeps kDqUnroll vectors in flight; the grid strides over the vectors.  A
// vector whose 16 elements share one scale (the common case) takes the
// packed path; one that crosses a group or block boundary looks its scale up
// per run of elements.  A ragged tail (n % 16 codes) goes element by element.
#include "fp8q_device.cuh"
#include "internal.h"

namespace fp8q {

constexpr int kDqThreads = 256;
constexpr int kDqUnroll = 4;

enum DqKind : int { kDqTensor = 0, kDqMxRow = 1, kDqMxCol = 2 };

struct DqParams {
  const uint8_t* q;
  const uint8_t* s;         // MX scale bytes
  const float* scale_inv;   // per-tensor [G]
  const int64_t* off;       // device row offsets [G + 1] or nullptr
  int G;
  int64_t rows, cols;       // of the original tensor
  int64_t s_ld;             // columnwise: scale bytes per column
  int64_t n;                // codes
  void* y;
};

// Clamped group boundary (offsets outside [0, rows] are pulled back in).
__device__ __forceinline__ int64_t dq_grp_row(const DqParams& p, int g) {
  if (p.off == nullptr) return g == 0 ? 0 : p.rows;
  const int64_t v = __ldg(p.off + g);
  return v < 0 ? 0 : (v > p.rows ? p.rows : v);
}

// Last group g with off[g] <= r.
__device__ __forceinline__ int dq_group(const DqParams& p, int64_t r) {
  if (p.off == nullptr || p.G <= 1) return 0;
  int lo = 0, hi = p.G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (dq_grp_row(p, mid) <= r) lo = mid; else hi = mid;
  }
  return lo;
}

// 2^(byte - 127) as an FP32 multiplier (byte 0: 2^-127, subnormal; 0xFF: NaN).
__device__ __forceinline__ float e8m0_value(uint32_t byte) {
  if (byte == 0xFFu) return __uint_as_float(0x7FC00000u);
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// The multiplier of flat element e, and the flat index where it stops
// applying (the end of e's run of equal scale).
template <int KIND>
__device__ __forceinline__ float dq_scale(const DqParams& p, const int* blk, int64_t e, int64_t& run_end) {
  if constexpr (KIND == kDqMxRow) {
    run_end = (e / 32 + 1) * 32;
    return e8m0_value(__ldg(p.s + e / 32));
  } else if constexpr (KIND == kDqTensor) {
    const int64_t row = e / p.cols;
    const int g = dq_group(p, row);
    run_end = dq_grp_row(p, g + 1) * p.cols;
    if (run_end <= e) run_end = (row + 1) * p.cols;  // clamped (empty) groups: one row at a time
    return __ldg(p.scale_inv + g);
  } else {
    const int64_t c = e / p.rows, r = e - c * p.rows;
    const int g = dq_group(p, r);
    const int64_t r0 = dq_grp_row(p, g), r1 = dq_grp_row(p, g + 1);
    if (r < r0 || r >= r1) {  // a row in no group (offsets not covering [0, rows)): NaN
      run_end = e + 1;
      return __uint_as_float(0x7FC00000u);
    }
    const int64_t b = (r - r0) / 32;
    const int64_t end_r = min(r0 + 32 * (b + 1), r1);  // > r
    run_end = c * p.rows + end_r;
    const int64_t sb = blk[g] + b;
    return sb < p.s_ld ? e8m0_value(__ldg(p.s + c * p.s_ld + sb)) : __uint_as_float(0x7FC00000u);
  }
}

// Two codes (bits 0-7 and 8-15 of `two`) -> two exact floats.
template <int FMT>
__device__ __forceinline__ void decode2(uint32_t two, float& lo, float& hi) {
  uint32_t h2;
  const unsigned short c = (unsigned short)two;
  if constexpr (FMT == kE4M3)
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  else
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(c));
  asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"((unsigned short)(h2 & 0xFFFFu)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"((unsigned short)(h2 >> 16)));
}

// Two floats -> packed BF16 (a in bits 0-15), ties to even, canonical NaN.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(b), "f"(a));
  const uint32_t nan = __vcmpgtu2(w & 0x7FFF7FFFu, 0x7F807F80u);
  return (w & ~nan) | (0x7FC07FC0u & nan);
}

__device__ __forceinline__ uint32_t f32_bits(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC00000u : b;
}

// 16 codes of one vector times their multipliers, written at element e.
template <int FMT, int OUT>
__device__ __forceinline__ void emit16(const DqParams& p, int64_t e, const uint4& c, const float (&m)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  float v[16];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    decode2<FMT>(w[k] & 0xFFFFu, v[4 * k], v[4 * k + 1]);
    decode2<FMT>(w[k] >> 16, v[4 * k + 2], v[4 * k + 3]);
  }
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __fmul_rn(v[i], m[i]);
  if constexpr (OUT == kBF16) {
    uint16_t* y = (uint16_t*)p.y + e;
    st_stream(y, make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                            pack_bf16(v[6], v[7])));
    st_stream(y + 8, make_uint4(pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]), pack_bf16(v[12], v[13]),
                                pack_bf16(v[14], v[15])));
  } else {
    uint32_t* y = (uint32_t*)p.y + e;
#pragma unroll
    for (int k = 0; k < 4; k++)
      st_stream(y + 4 * k, make_uint4(f32_bits(v[4 * k]), f32_bits(v[4 * k + 1]), f32_bits(v[4 * k + 2]),
                                      f32_bits(v[4 * k + 3])));
  }
}

// Block-wide exclusive scan of the column-block counts ceil(n_g / 32):
// blk[g] = first s_col block of group g (G + 1 entries).
template <int NT>
__device__ void dq_build_blk(const DqParams& p, int* blk) {
  __shared__ int tot[NT / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (p.G + NT - 1) / NT;
  const int g_lo = tid * per, g_hi = min(p.G, g_lo + per);
  int sum = 0;
  for (int g = g_lo; g < g_hi; g++) {
    const int64_t n = dq_grp_row(p, g + 1) - dq_grp_row(p, g);
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
  int before = 0;
  for (int w = 0; w < warp; w++) before += tot[w];
  int run = before + inc - sum;
  for (int g = g_lo; g < g_hi; g++) {
    blk[g] = run;
    const int64_t n = dq_grp_row(p, g + 1) - dq_grp_row(p, g);
    run += n > 0 ? (int)((n + 31) / 32) : 0;
  }
  if (tid == NT - 1) blk[p.G] = run;
  __syncthreads();
}

template <int KIND, int FMT, int OUT>
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(DqParams p) {
  extern __shared__ int blk[];  // columnwise: [G + 1]
  pdl_wait();
  if constexpr (KIND == kDqMxCol) dq_build_blk<kDqThreads>(p, blk);

  const int64_t nvec = p.n / 16;
  const int64_t stride = (int64_t)gridDim.x * kDqThreads;
  for (int64_t v0 = (int64_t)blockIdx.x * kDqThreads + threadIdx.x; v0 < nvec; v0 += stride * kDqUnroll) {
    uint4 c[kDqUnroll];
#pragma unroll
    for (int k = 0; k < kDqUnroll; k++) {
      const int64_t v = v0 + k * stride;
      c[k] = v < nvec ? ld_stream(p.q + 16 * v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kDqUnroll; k++) {
      const int64_t v = v0 + k * stride;
      if (v >= nvec) break;
      const int64_t e = 16 * v;
      float m[16];
      int64_t run_end;
      const float m0 = dq_scale<KIND>(p, blk, e, run_end);
      if (run_end >= e + 16) {
#pragma unroll
        for (int i = 0; i < 16; i++) m[i] = m0;
      } else {  // the vector crosses a group or block boundary
        int64_t cur = e, end = run_end;
        float mc = m0;
#pragma unroll
        for (int i = 0; i < 16; i++) {
          if (e + i >= end) {
            cur = e + i;
            mc = dq_scale<KIND>(p, blk, cur, end);
          }
          m[i] = mc;
        }
      }
      emit16<FMT, OUT>(p, e, c[k], m);
    }
  }

  // ragged tail: the last n % 16 codes, one per thread
  const int64_t t0 = nvec * 16;
  const int64_t i = t0 + (int64_t)blockIdx.x * kDqThreads + threadIdx.x;
  if (i < p.n) {
    int64_t run_end;
    const float m = dq_scale<KIND>(p, blk, i, run_end);
    float lo, hi;
    decode2<FMT>(__ldg(p.q + i), lo, hi);
    lo = __fmul_rn(lo, m);
    if constexpr (OUT == kBF16) ((uint16_t*)p.y)[i] = (uint16_t)(pack_bf16(lo, 0.0f) & 0xFFFFu);
    else ((uint32_t*)p.y)[i] = f32_bits(lo);
  }
  pdl_launch_dependents();
}

template <int KIND, int FMT, int OUT>
static cudaError_t launch_dq_t(const DqParams& p, cudaStream_t s) {
  const size_t smem = KIND == kDqMxCol ? sizeof(int) * (size_t)(p.G + 1) : 0;
  static int per_sm = [] {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, dequant_kernel<KIND, FMT, OUT>, kDqThreads,
                                                      sizeof(int) * (FP8Q_MAX_GROUPS + 1)) != cudaSuccess || v < 1)
      v = 1;
    return v;
  }();
  const int64_t nvec = p.n / 16;
  int64_t grid = (nvec + (int64_t)kDqThreads * kDqUnroll - 1) / ((int64_t)kDqThreads * kDqUnroll);
  const int64_t cap = (int64_t)per_sm * sm_count();
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_kernel(dequant_kernel<KIND, FMT, OUT>, dim3((unsigned)grid), dim3(kDqThreads), smem, s, p);
}

template <int KIND>
static cudaError_t launch_dq_kind(const DqParams& p, int fmt, int out_dt, cudaStream_t s) {
  if (fmt == kE4M3) return out_dt == kBF16 ? launch_dq_t<KIND, kE4M3, kBF16>(p, s) : launch_dq_t<KIND, kE4M3, kFP32>(p, s);
  return out_dt == kBF16 ? launch_dq_t<KIND, kE5M2, kBF16>(p, s) : launch_dq_t<KIND, kE5M2, kFP32>(p, s);
}

fp8q_status launch_dequant(int kind, const uint8_t* q, const uint8_t* s, const float* scale_inv,
                           const int64_t* off, int G, int64_t rows, int64_t cols, int64_t s_ld, int fmt,
                           int out_dt, void* y, cudaStream_t stream) {
  DqParams p{};
  p.q = q;
  p.s = s;
  p.scale_inv = scale_inv;
  p.off = off;
  p.G = off ? G : 1;
  p.rows = rows;
  p.cols = cols;
  p.s_ld = s_ld;
  p.n = rows * cols;
  p.y = y;
  cudaError_t e;
  if (kind == kDqTensor) e = launch_dq_kind<kDqTensor>(p, fmt, out_dt, stream);
  else if (kind == kDqMxRow) e = launch_dq_kind<kDqMxRow>(p, fmt, out_dt, stream);
  else e = launch_dq_kind<kDqMxCol>(p, fmt, out_dt, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize kernel launch");
  return check_launch("dequantize kernel");
}

}  // namespace fp8q
