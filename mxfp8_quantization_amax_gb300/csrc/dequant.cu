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

#ifndef FP8Q_DQ_UNROLL  // 16-code vectors in flight per thread
#define FP8Q_DQ_UNROLL 2
#endif
constexpr int kDqThreads = 256;
constexpr int kDqUnroll = FP8Q_DQ_UNROLL;

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
  int use_tab;              // columnwise: per-row-vector scale table in shared memory
};

// Columnwise scale table: for the 16 rows starting at 16 * vr (the same in
// every column), up to three runs of rows under one s_col block each: rows
// [0, t0) under sb0, [t0, t1) under sb1, [t1, 16) under sb2 (t0 = 16: one
// run).  A block of -1 is a row in no group.  Bit 16 of t marks 16 rows
// with more than three runs.
struct ColTab {
  int sb0, sb1, sb2, t;  // t = t0 | t1 << 8 | multi << 16
};
constexpr int kDqMaxTabBytes = 96 * 1024;

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
    if (p.off == nullptr || p.G <= 1) {
      run_end = p.n;
      return __ldg(p.scale_inv);
    }
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

// Multipliers of the 16-element vector at flat element e, as up to three
// runs (see VecScale); multi is set when it holds more than two boundaries
// (it then takes the out-of-line path).  The lookup is shared by the
// warp: its 32 vectors are consecutive, so lane 0 locates the group of the
// first one (the only division and search) and each lane derives its own
// scale from that; a lane outside that group does the full lookup.  Every
// lane of the warp must call (valid: this lane's vector exists).
struct VecScale {
  float m0, m1, m2;
  int t0, t1;  // elements below t0 take m0, below t1 m1, the rest m2
  bool multi;
};

template <int KIND>
__device__ __forceinline__ VecScale dq_vec_scale(const DqParams& p, const int* blk, const ColTab* tab, int64_t e,
                                                 bool valid) {
  VecScale r{0.0f, 0.0f, 0.0f, 16, 16, false};
  const unsigned kAll = 0xFFFFFFFFu;
  if constexpr (KIND == kDqTensor) {
    if (p.off == nullptr || p.G <= 1) {
      r.m0 = r.m1 = r.m2 = __ldg(p.scale_inv);
      return r;
    }
    const int lane = threadIdx.x & 31;
    const int64_t e0 = __shfl_sync(kAll, e, 0);
    int g = 0;
    long long gs = 0, ge = 0;
    if (lane == 0) {
      g = dq_group(p, e0 / p.cols);
      gs = dq_grp_row(p, g) * p.cols;
      ge = dq_grp_row(p, g + 1) * p.cols;
    }
    g = __shfl_sync(kAll, g, 0);
    gs = __shfl_sync(kAll, gs, 0);
    ge = __shfl_sync(kAll, ge, 0);
    if (valid && e >= gs && e + 16 <= ge) {
      r.m0 = r.m1 = r.m2 = __ldg(p.scale_inv + g);
      return r;
    }
  } else if constexpr (KIND == kDqMxCol) {
    if (p.use_tab || ((p.off == nullptr || p.G <= 1) && p.rows % 16 == 0)) {
      const int lane = threadIdx.x & 31;
      const int64_t e0 = __shfl_sync(kAll, e, 0);
      long long c0 = 0, rw = 0;
      if (lane == 0) {
        if (p.n <= 0xFFFFFFFFll) {  // 32-bit division where the sizes allow
          c0 = (uint32_t)e0 / (uint32_t)p.rows;
        } else {
          c0 = e0 / p.rows;
        }
        rw = e0 - c0 * p.rows;
      }
      c0 = __shfl_sync(kAll, c0, 0);
      rw = __shfl_sync(kAll, rw, 0);
      int64_t row = rw + 16 * lane, col = c0;
      if (row >= p.rows) {  // the warp's vectors run into the next column
        row -= p.rows;
        col += 1;
      }
      if (valid && row < p.rows && (p.off == nullptr || p.G <= 1)) {  // one group: block = row / 32
        const int64_t sb = row >> 5;
        r.m0 = r.m1 = r.m2 = sb < p.s_ld ? e8m0_value(__ldg(p.s + col * p.s_ld + sb)) : __uint_as_float(0x7FC00000u);
        return r;
      }
      if (valid && row < p.rows) {
        const ColTab te = tab[row >> 4];
        const uint8_t* scol = p.s + col * p.s_ld;
        const float nan = __uint_as_float(0x7FC00000u);
        r.m0 = te.sb0 >= 0 && te.sb0 < p.s_ld ? e8m0_value(__ldg(scol + te.sb0)) : nan;
        r.t0 = te.t & 0xFF;
        r.t1 = (te.t >> 8) & 0xFF;
        r.multi = (te.t >> 16) != 0;
        r.m1 = r.t0 == 16 ? r.m0 : (te.sb1 >= 0 && te.sb1 < p.s_ld ? e8m0_value(__ldg(scol + te.sb1)) : nan);
        r.m2 = r.t1 == 16 ? r.m1 : (te.sb2 >= 0 && te.sb2 < p.s_ld ? e8m0_value(__ldg(scol + te.sb2)) : nan);
        return r;
      }
    }
  }
  if (!valid) return r;
  // the full lookup (always for rowwise MX, where it is one byte load)
  int64_t end1 = e + 16;
  r.m0 = dq_scale<KIND>(p, blk, e, end1);
  r.t0 = (int)min(end1 - e, (int64_t)16);
  r.m1 = r.m2 = r.m0;
  if (r.t0 < 16) {
    int64_t end2;
    r.m1 = r.m2 = dq_scale<KIND>(p, blk, e + r.t0, end2);
    r.t1 = (int)min(end2 - e, (int64_t)16);
    if (r.t1 < 16) {
      int64_t end3;
      r.m2 = dq_scale<KIND>(p, blk, e + r.t1, end3);
      r.multi = end3 < e + 16;
    }
  }
  return r;
}

// 8 codes (two words) times their multipliers -- elements i < t0 take m0,
// those below t1 m1, the rest m2 -- written at element e (e % 8 == 0).
template <int FMT, int OUT>
__device__ __forceinline__ void emit8(const DqParams& p, int64_t e, uint32_t w0, uint32_t w1, float m0, float m1,
                                      float m2, int t0, int t1) {
  float v[8];
  decode2<FMT>(w0 & 0xFFFFu, v[0], v[1]);
  decode2<FMT>(w0 >> 16, v[2], v[3]);
  decode2<FMT>(w1 & 0xFFFFu, v[4], v[5]);
  decode2<FMT>(w1 >> 16, v[6], v[7]);
#pragma unroll
  for (int i = 0; i < 8; i++) v[i] = __fmul_rn(v[i], i < t0 ? m0 : (i < t1 ? m1 : m2));
  if constexpr (OUT == kBF16) {
    st_stream((uint16_t*)p.y + e, make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                                             pack_bf16(v[6], v[7])));
  } else {
    uint32_t* y = (uint32_t*)p.y + e;
    st_stream(y, make_uint4(f32_bits(v[0]), f32_bits(v[1]), f32_bits(v[2]), f32_bits(v[3])));
    st_stream(y + 4, make_uint4(f32_bits(v[4]), f32_bits(v[5]), f32_bits(v[6]), f32_bits(v[7])));
  }
}

// A vector that holds more than one group or block boundary (groups of
// fewer than 16 rows): one lookup per run of equal scale, then the packed
// emit.  Kept out of line: it is rare, and a lane that takes it holds up its
// warp, so it must stay short.
template <int KIND, int FMT, int OUT>
__device__ __noinline__ void emit16_runs(const DqParams& p, const int* blk, int64_t e, uint4 c) {
  float m[16];
  int i = 0;
  while (i < 16) {
    int64_t end;
    const float mi = dq_scale<KIND>(p, blk, e + i, end);
    const int n = (int)min(end - (e + i), (int64_t)(16 - i));
#pragma unroll 1
    for (int j = 0; j < n; j++) m[i + j] = mi;
    i += n;
  }
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int h = 0; h < 2; h++) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 2; k++) {
      decode2<FMT>(w[2 * h + k] & 0xFFFFu, v[4 * k], v[4 * k + 1]);
      decode2<FMT>(w[2 * h + k] >> 16, v[4 * k + 2], v[4 * k + 3]);
    }
#pragma unroll
    for (int j = 0; j < 8; j++) v[j] = __fmul_rn(v[j], m[8 * h + j]);
    if constexpr (OUT == kBF16) {
      st_stream((uint16_t*)p.y + e + 8 * h, make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
                                                       pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7])));
    } else {
      uint32_t* y = (uint32_t*)p.y + e + 8 * h;
      st_stream(y, make_uint4(f32_bits(v[0]), f32_bits(v[1]), f32_bits(v[2]), f32_bits(v[3])));
      st_stream(y + 4, make_uint4(f32_bits(v[4]), f32_bits(v[5]), f32_bits(v[6]), f32_bits(v[7])));
    }
  }
}

// One element (any position): the ragged tail.
template <int KIND, int FMT, int OUT>
__device__ __noinline__ void emit1(const DqParams& p, const int* blk, int64_t i, uint32_t code) {
  int64_t run_end;
  const float m = dq_scale<KIND>(p, blk, i, run_end);
  float lo, hi;
  decode2<FMT>(code, lo, hi);
  lo = __fmul_rn(lo, m);
  if constexpr (OUT == kBF16) ((uint16_t*)p.y)[i] = (uint16_t)(pack_bf16(lo, 0.0f) & 0xFFFFu);
  else ((uint32_t*)p.y)[i] = f32_bits(lo);
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

// Fills the columnwise scale table for rows / 16 row-vectors.  Each thread
// takes a contiguous range: one binary search, then it walks forward.
template <int NT>
__device__ void dq_build_tab(const DqParams& p, const int* blk, ColTab* tab) {
  const int nvr = (int)(p.rows / 16);
  const int per = (nvr + NT - 1) / NT;
  const int lo = threadIdx.x * per, hi = min(nvr, lo + per);
  if (lo < hi) {
    int g = dq_group(p, 16LL * lo);
    for (int vr = lo; vr < hi; vr++) {
      const int64_t r = 16LL * vr;
      while (g + 1 < p.G && dq_grp_row(p, g + 1) <= r) g++;
      // walk the runs of [r, r + 16): block of row x, and where it ends
      int sb[3] = {-1, -1, -1}, ends[3] = {16, 16, 16};
      int nrun = 0;
      int gx = g;
      int64_t x = r;
      while (x < r + 16 && nrun < 4) {
        while (gx + 1 < p.G && dq_grp_row(p, gx + 1) <= x) gx++;
        const int64_t r0 = dq_grp_row(p, gx), r1 = dq_grp_row(p, gx + 1);
        int blk_x = -1;
        int64_t end;
        if (x >= r0 && x < r1) {
          const int64_t b = (x - r0) >> 5;
          blk_x = (int)(blk[gx] + b);
          end = min(r0 + 32 * (b + 1), r1);
        } else {  // a row in no group: its own run
          end = x + 1;
        }
        end = min(end, r + 16);
        if (nrun < 3) {
          sb[nrun] = blk_x;
          ends[nrun] = (int)(end - r);
        }
        nrun++;
        x = end;
      }
      ColTab e;
      e.sb0 = sb[0];
      e.sb1 = nrun > 1 ? sb[1] : sb[0];
      e.sb2 = nrun > 2 ? sb[2] : e.sb1;
      e.t = ends[0] | ((nrun > 1 ? ends[1] : 16) << 8) | (nrun > 3 ? 1 << 16 : 0);
      tab[vr] = e;
    }
  }
  __syncthreads();
}

template <int KIND, int FMT, int OUT>
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(DqParams p) {
  extern __shared__ int blk[];  // columnwise: [G + 1], then the scale table
  ColTab* tab = (ColTab*)(blk + ((p.G + 4) & ~3));
  pdl_wait();
  if constexpr (KIND == kDqMxCol) {
    dq_build_blk<kDqThreads>(p, blk);
    if (p.use_tab) dq_build_tab<kDqThreads>(p, blk, tab);
  }

  const int64_t nvec = p.n / 16;
  const int64_t stride = (int64_t)gridDim.x * kDqThreads;
  const int lane = threadIdx.x & 31;
  // the condition is the warp's first vector, so whole warps iterate together
  // (the scale lookup shuffles across the warp)
  for (int64_t v0 = (int64_t)blockIdx.x * kDqThreads + threadIdx.x; v0 - lane < nvec; v0 += stride * kDqUnroll) {
    // every load of the round first (codes, then each vector's scales), so
    // they are in flight together
    uint4 c[kDqUnroll];
    VecScale sc[kDqUnroll];
#pragma unroll
    for (int k = 0; k < kDqUnroll; k++) {
      const int64_t v = v0 + k * stride;
      c[k] = v < nvec ? ld_stream(p.q + 16 * v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kDqUnroll; k++) {
      const int64_t v = v0 + k * stride;
      sc[k] = dq_vec_scale<KIND>(p, blk, tab, 16 * v, v < nvec);
    }
#pragma unroll
    for (int k = 0; k < kDqUnroll; k++) {
      const int64_t v = v0 + k * stride;
      if (v >= nvec) break;
      const int64_t e = 16 * v;
      if (!sc[k].multi) {
        emit8<FMT, OUT>(p, e, c[k].x, c[k].y, sc[k].m0, sc[k].m1, sc[k].m2, sc[k].t0, sc[k].t1);
        emit8<FMT, OUT>(p, e + 8, c[k].z, c[k].w, sc[k].m0, sc[k].m1, sc[k].m2, sc[k].t0 - 8, sc[k].t1 - 8);
      } else {  // several boundaries (groups of fewer than 16 rows)
        emit16_runs<KIND, FMT, OUT>(p, blk, e, c[k]);
      }
    }
  }

  // ragged tail: the last n % 16 codes, one per thread
  const int64_t i = nvec * 16 + (int64_t)blockIdx.x * kDqThreads + threadIdx.x;
  if (i < p.n) emit1<KIND, FMT, OUT>(p, blk, i, __ldg(p.q + i));
  pdl_launch_dependents();
}

template <int KIND, int FMT, int OUT>
static cudaError_t launch_dq_t(const DqParams& p, cudaStream_t s) {
  size_t smem = 0;
  if (KIND == kDqMxCol) {
    smem = sizeof(int) * (size_t)((p.G + 4) & ~3);
    if (p.use_tab) smem += sizeof(ColTab) * (size_t)(p.rows / 16);
  }
  static int per_sm = [] {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, dequant_kernel<KIND, FMT, OUT>, kDqThreads, 0) !=
            cudaSuccess || v < 1)
      v = 1;
    return v;
  }();
  if (smem > 48 * 1024) {
    static bool opted = false;
    if (!opted) {
      const cudaError_t e = cudaFuncSetAttribute(dequant_kernel<KIND, FMT, OUT>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)(sizeof(int) * (FP8Q_MAX_GROUPS + 4) + kDqMaxTabBytes));
      if (e != cudaSuccess) return e;
      opted = true;
    }
  }
  int fit = 0;  // CTAs per SM at this launch's shared memory
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, dequant_kernel<KIND, FMT, OUT>, kDqThreads, smem) !=
          cudaSuccess || fit < 1)
    fit = 1;
  const int64_t nvec = p.n / 16;
  int64_t grid = (nvec + (int64_t)kDqThreads * kDqUnroll - 1) / ((int64_t)kDqThreads * kDqUnroll);
  const int64_t cap = (int64_t)min(per_sm, fit) * sm_count();
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
  p.use_tab = kind == kDqMxCol && off != nullptr && G > 1 && rows % 16 == 0 &&
              (rows / 16) * (int64_t)sizeof(ColTab) <= kDqMaxTabBytes;
  cudaError_t e;
  if (kind == kDqTensor) e = launch_dq_kind<kDqTensor>(p, fmt, out_dt, stream);
  else if (kind == kDqMxRow) e = launch_dq_kind<kDqMxRow>(p, fmt, out_dt, stream);
  else e = launch_dq_kind<kDqMxCol>(p, fmt, out_dt, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize kernel launch");
  return check_launch("dequantize kernel");
}

}  // namespace fp8q
