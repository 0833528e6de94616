// mxlow.cu -- MXFP4 (E2M1 elements) and MXFP6 (E2M3 or E3M2 elements):
// blocks of 32 elements sharing one E8M0 scale, rowwise and columnwise, both
// copies from a single pass over x.
//
// "混合精度与 FP8 训练" 13.1: an MX block is 32 elements and a power-of-two
// scale; the shared exponent is floor(log2 amax) - e_max (e_max = 2 for
// E2M1), elements are scaled and saturated.  13.2: E2M1 holds 0, 0.5, 1,
// 1.5, 2, 3, 4, 6 and negatives.  "Blackwell GPU MXFP8 预训练最佳实践" 3.2
// lists MXFP6 among Blackwell's block-scaled types; its elements are taken
// to be the OCP pair E2M3 (largest 7.5) and E3M2 (largest 28).  4.1: the
// round-up rule X = ceil(log2(amax / destmax)), destmax the element format's
// largest value.  Both rules are offered, as for MXFP8.
//
// Layout.  E2M1 codes are packed two per byte along the copy's rows (element
// 2i in the low nibble); FP6 codes take one byte each (bits 0-5), the
// unpacked form Blackwell's tensor cores read for mixed FP8/FP6/FP4 operands.
//   rowwise:    q_row [rows][cols / 2 or cols],  s_row [rows][cols / 32]
//   columnwise: q_col [cols][rows / 2 or rows],  s_col [cols][ceil(rows / 32)]
// A block whose amax is 0 gets scale byte 0 and +0 codes; one holding Inf or
// NaN gets 0xFF and +0 codes (the formats have no NaN; the scale marks it).
//
// Work split.  A CTA streams tiles of 32 rows x 1 KB of x (512 BF16 or 256
// FP32 columns) into shared memory with cp.async, kLowStages deep, so the
// next tiles are in flight while the current one is converted.  Rowwise: a
// thread takes a whole 32-element block of one row (its amax in registers,
// 16 paired conversions, one 16- or 32-byte store).  Columnwise: a thread
// takes a column pair over the tile's 32 rows.  The tile's 16-byte granules
// are XOR-swizzled within each 128-byte line so that both read patterns are
// free of bank conflicts.  Conversions are the hardware
// cvt.rn.satfinite.{e2m1,e2m3,e3m2}x2 (nearest even, saturating).
#include "fp8q_device.cuh"
#include "internal.h"

namespace fp8q {

enum : int { kE2M1 = FP8Q_E2M1, kE2M3 = FP8Q_E2M3, kE3M2 = FP8Q_E3M2 };

template <int EF> struct LowFmt;
template <> struct LowFmt<kE2M1> {  // 6 = 1.5 * 2^2
  static constexpr int kEmax = 2;
  static constexpr uint32_t kMaxMant = 0x400000u;
  static constexpr float kMax = 6.0f;
};
template <> struct LowFmt<kE2M3> {  // 7.5 = 1.875 * 2^2
  static constexpr int kEmax = 2;
  static constexpr uint32_t kMaxMant = 0x700000u;
  static constexpr float kMax = 7.5f;
};
template <> struct LowFmt<kE3M2> {  // 28 = 1.75 * 2^4
  static constexpr int kEmax = 4;
  static constexpr uint32_t kMaxMant = 0x600000u;
  static constexpr float kMax = 28.0f;
};

constexpr int kLowThreads = 256;
#ifndef FP8Q_LOW_MIN_CTAS  // CTAs per SM the register budget is sized for
#define FP8Q_LOW_MIN_CTAS 2
#endif
#ifndef FP8Q_LOW_STAGES  // tiles resident per CTA: one converted while the rest load
#define FP8Q_LOW_STAGES 2
#endif
constexpr int kLowStages = FP8Q_LOW_STAGES;
constexpr int kLowRowBytes = 1024;             // bytes of x per tile row
constexpr int kLowTileBytes = 32 * kLowRowBytes;

struct LowParams {
  const void* x;
  int64_t rows, cols;
  int dir;                  // MXFP8_ROW | MXFP8_COL
  int round_up;             // 1: round-up rule, 0: OCP rule
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  unsigned long long* sat;  // [2] or nullptr
};

// Scale byte of a block from its amax (FP32 magnitude bits): X + 127 with
// X = e - e_max (+1 under the round-up rule when the mantissa of amax is
// above the mantissa of destmax), clamped to [0, 254]; Inf/NaN -> 0xFF.
template <int EF>
__device__ __forceinline__ uint32_t low_scale_byte(uint32_t amax_bits, int round_up) {
  if (amax_bits >= 0x7F800000u) return 0xFFu;
  const int b = (int)(amax_bits >> 23) - LowFmt<EF>::kEmax +
                ((round_up && (amax_bits & 0x7FFFFFu) > LowFmt<EF>::kMaxMant) ? 1 : 0);
  return (uint32_t)min(max(b, 0), 254);
}

// 2^-X for scale byte X + 127 (byte 254: 2^-127, subnormal).
__device__ __forceinline__ float low_multiplier(uint32_t byte) {
  return byte <= 253u ? __uint_as_float((254u - byte) << 23) : __uint_as_float(0x00400000u);
}

// Two scaled values -> two codes: the low code from `lo`.  E2M1: one byte
// (lo in bits 0-3); FP6: two bytes (lo in bits 0-7).
template <int EF>
__device__ __forceinline__ uint32_t low_cvt2(float lo, float hi) {
  unsigned short r;
  if constexpr (EF == kE2M1)
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tmov.b16 %0, {t, 0};\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
  else if constexpr (EF == kE2M3)
    asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return EF == kE2M1 ? (uint32_t)(r & 0xFFu) : (uint32_t)r;
}

// Byte offset in a tile row of 16-byte granule g after the swizzle.
__device__ __forceinline__ int low_swz(int g) { return 16 * (g ^ ((g >> 3) & 7)); }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most kLowStages - 1 groups of this thread's copies are pending.
__device__ __forceinline__ void cp_async_wait_oldest() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kLowStages - 1) : "memory");
}

// Tile coordinates (row tile, column tile) of t = tr * ntc + tc, stepped by
// the grid size without a division per step.
struct LowTile {
  int64_t tr, tc;
  __device__ __forceinline__ void start(int64_t t, int64_t ntc) {
    tr = t / ntc;
    tc = t - tr * ntc;
  }
  __device__ __forceinline__ void step(int64_t dr, int64_t dc, int64_t ntc) {  // by dr * ntc + dc
    tr += dr;
    tc += dc;
    if (tc >= ntc) {
      tc -= ntc;
      tr++;
    }
  }
};

// Tile t into `stage`: 32 rows x 64 granules of 16 bytes, a thread taking
// one granule column (its tid % 64) of rows tid / 64 + 4k; granules past the
// last row or column are zero-filled (no bytes read).
__device__ __forceinline__ void low_issue(const LowParams& p, uint8_t* stage, const LowTile& at, int esz) {
  const int64_t tr = at.tr, tc = at.tc;
  const int64_t row_bytes = p.cols * esz;
  const int g = threadIdx.x & 63, row0 = threadIdx.x >> 6;
  const int64_t cb = tc * kLowRowBytes + 16 * g;  // byte of the granule in its row
  const int64_t r = tr * 32 + row0;
  const bool col_ok = cb < row_bytes;
  const char* src = (const char*)p.x + r * row_bytes + cb;
  uint8_t* dst = stage + row0 * kLowRowBytes + low_swz(g);
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const bool ok = col_ok && r + 4 * k < p.rows;
    cp_async16(dst + 4 * k * kLowRowBytes, ok ? src + 4 * k * row_bytes : p.x, ok ? 16 : 0);
  }
}

// Two FP32 lanes in one 64-bit register, for Blackwell's packed f32x2 multiply.
typedef unsigned long long low_f2;
__device__ __forceinline__ low_f2 low_f2_make(float lo, float hi) {
  low_f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ low_f2 low_f2_mul(low_f2 a, low_f2 b) {
  low_f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float low_f2_lo(low_f2 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float low_f2_hi(low_f2 v) { return __uint_as_float((uint32_t)(v >> 32)); }

// Codes of the pair x * m (x = two elements of one block): the low code
// from the low lane; counts saturated elements when asked (count: the
// block is finite and nonzero).
template <int EF, bool SAT>
__device__ __forceinline__ uint32_t low_pair(low_f2 x, low_f2 m, bool count, unsigned long long& sat) {
  const low_f2 sv = low_f2_mul(x, m);
  const float s0 = low_f2_lo(sv), s1 = low_f2_hi(sv);
  if constexpr (SAT)
    if (count) sat += (fabsf(s0) > LowFmt<EF>::kMax) + (fabsf(s1) > LowFmt<EF>::kMax);
  return low_cvt2<EF>(s0, s1);
}

// 16 code pairs of one block (pair k = elements 2k, 2k+1) packed in order:
// E2M1 one byte per pair (4 words), FP6 two bytes per pair (8 words).
template <int EF>
__device__ __forceinline__ void low_pack(const uint32_t (&pr)[16], uint32_t (&w)[8]) {
  if constexpr (EF == kE2M1) {
#pragma unroll
    for (int k = 0; k < 4; k++)
      w[k] = __byte_perm(__byte_perm(pr[4 * k], pr[4 * k + 1], 0x0040), __byte_perm(pr[4 * k + 2], pr[4 * k + 3], 0x0040),
                         0x5410);
  } else {
#pragma unroll
    for (int k = 0; k < 8; k++) w[k] = __byte_perm(pr[2 * k], pr[2 * k + 1], 0x5410);
  }
}

template <int DT, int EF, bool SAT>
__global__ void __launch_bounds__(kLowThreads, FP8Q_LOW_MIN_CTAS) mxlow_kernel(LowParams p) {
  constexpr bool kFp4 = EF == kE2M1;
  constexpr int kEsz = DT == kBF16 ? 2 : 4;
  constexpr int kTileCols = kLowRowBytes / kEsz;   // 512 or 256
  constexpr int kBlocks = kTileCols / 32;          // row blocks per tile row
  extern __shared__ __align__(128) uint8_t lsm[];  // kLowStages tiles
  pdl_wait();
  const int64_t ntr = (p.rows + 31) / 32, ntc = (p.cols + kTileCols - 1) / kTileCols;
  const int64_t ntiles = ntr * ntc;
  const int64_t col_len = kFp4 ? p.rows / 2 : p.rows;  // bytes per column of q_col
  const bool col_vec = (col_len % 16) == 0 && ((uintptr_t)p.q_col & 15) == 0;
  unsigned long long sat_r = 0, sat_c = 0;
  const int64_t G = gridDim.x, dr = G / ntc, dc = G - dr * ntc;
  int64_t t = blockIdx.x;
  LowTile cur, nxt;  // the tile converted now, the next one to load
  cur.start(t, ntc);
  nxt = cur;
#pragma unroll
  for (int k = 0; k < kLowStages - 1; k++) {  // the first tiles in flight
    if (t + k * G < ntiles) low_issue(p, lsm + k * kLowTileBytes, nxt, kEsz);
    cp_async_commit();
    nxt.step(dr, dc, ntc);
  }
  for (int st = 0; t < ntiles; t += G, st = st + 1 == kLowStages ? 0 : st + 1) {
    const int64_t tn = t + (kLowStages - 1) * G;
    const int sn = st == 0 ? kLowStages - 1 : st - 1;  // the stage converted last round
    if (tn < ntiles) low_issue(p, lsm + sn * kLowTileBytes, nxt, kEsz);
    cp_async_commit();
    nxt.step(dr, dc, ntc);
    cp_async_wait_oldest();  // this thread's copies of tile t have landed
    __syncthreads();         // and everyone else's
    const uint8_t* tile = lsm + st * kLowTileBytes;
    const int64_t tr = cur.tr, tc = cur.tc;
    cur.step(dr, dc, ntc);
    const int64_t r0 = tr * 32, c0 = tc * kTileCols;
    const int nr = (int)min(p.rows - r0, (int64_t)32);
    const int ncols = (int)min(p.cols - c0, (int64_t)kTileCols);  // a multiple of 32

    // columnwise: a column pair over the tile's rows
    if ((p.dir & MXFP8_COL) && 2 * (int)threadIdx.x < ncols) {
      const int b = kEsz * 2 * threadIdx.x;  // byte of the pair in a tile row
      const int off = low_swz(b >> 4) + (b & 15);
      // row i of the pair: BF16 one word kept in registers; FP32 read again
      uint32_t xw[DT == kBF16 ? 32 : 1] = {};
      auto row = [&](int i, float& a, float& c) {
        if constexpr (DT == kBF16) {
          a = bf16_lo(xw[i]);
          c = bf16_hi(xw[i]);
        } else {
          const float2 v = *(const float2*)(tile + i * kLowRowBytes + off);
          a = v.x;
          c = v.y;
        }
      };
      uint32_t ma = 0, mb = 0;  // magnitude bits of each column's amax (rows past nr are zeros)
      if constexpr (DT == kBF16) {
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 32; i++) {
          xw[i] = *(const uint32_t*)(tile + i * kLowRowBytes + off);
          m = absmax_nan_bf16x2(m, xw[i]);  // magnitude bits only; NaN stays above Inf
        }
        ma = (m & 0x7FFFu) << 16;
        mb = m & 0x7FFF0000u;
      } else {
#pragma unroll
        for (int i = 0; i < 32; i++) {
          float a, c;
          row(i, a, c);
          ma = max(ma, __float_as_uint(a) & 0x7FFFFFFFu);
          mb = max(mb, __float_as_uint(c) & 0x7FFFFFFFu);
        }
      }
      const uint32_t ba = low_scale_byte<EF>(ma, p.round_up), bb = low_scale_byte<EF>(mb, p.round_up);
      const bool za = ma == 0u || ba == 0xFFu, zb = mb == 0u || bb == 0xFFu;
      const low_f2 Ma = low_f2_make(low_multiplier(ba), low_multiplier(ba));
      const low_f2 Mb = low_f2_make(low_multiplier(bb), low_multiplier(bb));
      uint32_t pa[16], pb[16];
#pragma unroll
      for (int k = 0; k < 16; k++) {
        float a0, c0v, a1, c1v;
        row(2 * k, a0, c0v);
        row(2 * k + 1, a1, c1v);
        pa[k] = low_pair<EF, SAT>(low_f2_make(a0, a1), Ma, !za, sat_c);
        pb[k] = low_pair<EF, SAT>(low_f2_make(c0v, c1v), Mb, !zb, sat_c);
      }
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const uint32_t byte = h ? bb : ba;
        uint32_t w[8] = {};
        if (!(h ? zb : za)) low_pack<EF>(h ? pb : pa, w);
        const int64_t cc = c0 + 2 * threadIdx.x + h;
        uint8_t* dst = p.q_col + cc * col_len + (kFp4 ? r0 / 2 : r0);
        if (col_vec && nr == 32) {
          *(uint4*)dst = make_uint4(w[0], w[1], w[2], w[3]);
          if constexpr (!kFp4) *(uint4*)(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
          const int nbytes = kFp4 ? nr / 2 : nr;
#pragma unroll
          for (int k = 0; k < (kFp4 ? 16 : 32); k++)
            if (k < nbytes) dst[k] = (uint8_t)(w[k >> 2] >> (8 * (k & 3)));
        }
        p.s_col[cc * ntr + tr] = (uint8_t)byte;
      }
    }

    // rowwise: a whole block of one row per thread
    if (p.dir & MXFP8_ROW) {
#pragma unroll
      for (int uu = 0; uu < 32 * kBlocks / kLowThreads; uu++) {
        const int u = threadIdx.x + kLowThreads * uu;
        const int i = u / kBlocks, j = u % kBlocks;
        if (i >= nr || 32 * j >= ncols) continue;
        constexpr int kG = 32 * kEsz / 16;  // granules per block: 4 or 8
        uint32_t xw[4 * kG];
#pragma unroll
        for (int g = 0; g < kG; g++) {
          const uint4 v = *(const uint4*)(tile + i * kLowRowBytes + low_swz(kG * j + g));
          xw[4 * g] = v.x;
          xw[4 * g + 1] = v.y;
          xw[4 * g + 2] = v.z;
          xw[4 * g + 3] = v.w;
        }
        uint32_t amax = 0;
        if constexpr (DT == kBF16) {
          uint32_t m = 0;
#pragma unroll
          for (int q = 0; q < 16; q++) m = absmax_nan_bf16x2(m, xw[q]);
          amax = max((m & 0x7FFFu) << 16, m & 0x7FFF0000u);
        } else {
#pragma unroll
          for (int q = 0; q < 32; q++) amax = max(amax, xw[q] & 0x7FFFFFFFu);
        }
        const uint32_t byte = low_scale_byte<EF>(amax, p.round_up);
        const bool zero_codes = amax == 0u || byte == 0xFFu;
        const float mul = low_multiplier(byte);
        const low_f2 M = low_f2_make(mul, mul);
        uint32_t pr[16];
#pragma unroll
        for (int k = 0; k < 16; k++) {
          const low_f2 X = DT == kBF16 ? low_f2_make(bf16_lo(xw[k]), bf16_hi(xw[k]))
                                       : low_f2_make(__uint_as_float(xw[2 * k]), __uint_as_float(xw[2 * k + 1]));
          pr[k] = low_pair<EF, SAT>(X, M, !zero_codes, sat_r);
        }
        uint32_t w[8] = {};
        if (!zero_codes) low_pack<EF>(pr, w);
        const int64_t r = r0 + i, cb = c0 / 32 + j;  // the block's index in its row
        uint8_t* dst = p.q_row + r * (kFp4 ? p.cols / 2 : p.cols) + cb * (kFp4 ? 16 : 32);
        *(uint4*)dst = make_uint4(w[0], w[1], w[2], w[3]);
        if constexpr (!kFp4) *(uint4*)(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        p.s_row[r * (p.cols / 32) + cb] = (uint8_t)byte;
      }
    }
    __syncthreads();  // the stage is refilled next round
  }
  pdl_launch_dependents();
  if constexpr (SAT) {
    sat_r = warp_sum_u64(sat_r);
    sat_c = warp_sum_u64(sat_c);
    if ((threadIdx.x & 31) == 0) {
      if (sat_r) atomicAdd(p.sat, sat_r);
      if (sat_c) atomicAdd(p.sat + 1, sat_c);
    }
  }
}

template <int DT, int EF>
static cudaError_t low_launch_typed(const LowParams& p, cudaStream_t stream) {
  constexpr int kTileCols = kLowRowBytes / (DT == kBF16 ? 2 : 4);
  const int64_t tiles = ((p.rows + 31) / 32) * ((p.cols + kTileCols - 1) / kTileCols);
  auto kernel = p.sat ? mxlow_kernel<DT, EF, true> : mxlow_kernel<DT, EF, false>;
  constexpr size_t smem = (size_t)kLowStages * kLowTileBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kLowThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  int64_t grid = (int64_t)per_sm * sm_count();
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  return launch_kernel(kernel, dim3((unsigned)grid), dim3(kLowThreads), smem, stream, p);
}

fp8q_status launch_mxlow(const void* x, int dt, int64_t rows, int64_t cols, int elem, int dir, int round_up,
                         uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, unsigned long long* sat,
                         cudaStream_t stream) {
  LowParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.dir = dir;
  p.round_up = round_up;
  p.q_row = q_row;
  p.s_row = s_row;
  p.q_col = q_col;
  p.s_col = s_col;
  p.sat = sat;
  cudaError_t e;
  if (dt == kBF16)
    e = elem == kE2M1 ? low_launch_typed<kBF16, kE2M1>(p, stream)
        : elem == kE2M3 ? low_launch_typed<kBF16, kE2M3>(p, stream)
                        : low_launch_typed<kBF16, kE3M2>(p, stream);
  else
    e = elem == kE2M1 ? low_launch_typed<kFP32, kE2M1>(p, stream)
        : elem == kE2M3 ? low_launch_typed<kFP32, kE2M3>(p, stream)
                        : low_launch_typed<kFP32, kE3M2>(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "MXFP4/MXFP6 kernel launch");
  return check_launch("MXFP4/MXFP6 kernel");
}

}  // namespace fp8q
