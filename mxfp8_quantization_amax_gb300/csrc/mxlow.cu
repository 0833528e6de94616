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
//
// BF16 input takes a second kernel built like the MXFP8 one: a producer warp
// streams 32-row x 256-column blocks into a two-stage shared-memory ring with
// 2-D TMA loads (128-byte swizzle), four consumer warps convert them (a lane
// per rowwise block, a thread per column pair), four CTAs per SM, units of
// four blocks down one strip dealt out row band by row band.
#include <cudaTypedefs.h>

#include <mutex>

#include "fp8q_device.cuh"
#include "internal.h"
#include "tma.cuh"

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

// ---------------------------------------------------------------------------
// BF16: TMA-fed, warp-specialised kernel
// ---------------------------------------------------------------------------
constexpr int kLtCons = 128;                    // four consumer warps
constexpr int kLtThreads = kLtCons + 32;        // + one producer warp
constexpr int kLtCols = 256;                    // columns per block (a strip)
constexpr int kLtSubCols = 64;                  // columns per TMA box (128 bytes)
constexpr int kLtSubBytes = 32 * 128;           // one box in shared memory
constexpr int kLtStageBytes = 32 * kLtCols * 2; // one BF16 block: 16 KB
#ifndef FP8Q_LOW_TMA_STAGES  // TMA ring depth of the BF16 kernel (16 KB per stage)
#define FP8Q_LOW_TMA_STAGES 2
#endif
constexpr int kLtStages = FP8Q_LOW_TMA_STAGES;
constexpr int kLtUnit = 4;                      // blocks per unit
#ifndef FP8Q_LOW_GRID_ALL  // one CTA per unit instead of a persistent grid
#define FP8Q_LOW_GRID_ALL 1
#endif

// Failure word (bit 0: a bounded wait gave up) and wait budget of this
// kernel; read and cleared by fp8q_check_device().
__device__ unsigned int g_low_error;
__device__ unsigned long long g_low_budget_ns = 1000000000ull;

// Codes of scaled pairs written straight into their output word: E2M1, the
// four bytes of pairs a..d (each pair's first element in the low nibble);
// FP6, the two 16-bit halves of pairs a and b.  The conversions write parts
// of one register, with no masking or byte permutes to join them.
__device__ __forceinline__ uint32_t lt_fp4_word(low_f2 a, low_f2 b, low_f2 c, low_f2 d) {
  uint32_t r;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t.reg .f32 a0, a1, b0, b1, c0, c1, d0, d1;\n\t"
      "mov.b64 {a0, a1}, %1;\n\tmov.b64 {b0, b1}, %2;\n\tmov.b64 {c0, c1}, %3;\n\tmov.b64 {d0, d1}, %4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, a1, a0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, b1, b0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, c1, c0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, d1, d0;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(r)
      : "l"(a), "l"(b), "l"(c), "l"(d));
  return r;
}
template <int EF>
__device__ __forceinline__ uint32_t lt_fp6_word(low_f2 a, low_f2 b) {
  uint32_t r;
  if constexpr (EF == kE2M3)
    asm("{\n\t.reg .b16 t0, t1;\n\t.reg .f32 a0, a1, b0, b1;\n\t"
        "mov.b64 {a0, a1}, %1;\n\tmov.b64 {b0, b1}, %2;\n\t"
        "cvt.rn.satfinite.e2m3x2.f32 t0, a1, a0;\n\t"
        "cvt.rn.satfinite.e2m3x2.f32 t1, b1, b0;\n\t"
        "mov.b32 %0, {t0, t1};\n\t}"
        : "=r"(r)
        : "l"(a), "l"(b));
  else
    asm("{\n\t.reg .b16 t0, t1;\n\t.reg .f32 a0, a1, b0, b1;\n\t"
        "mov.b64 {a0, a1}, %1;\n\tmov.b64 {b0, b1}, %2;\n\t"
        "cvt.rn.satfinite.e3m2x2.f32 t0, a1, a0;\n\t"
        "cvt.rn.satfinite.e3m2x2.f32 t1, b1, b0;\n\t"
        "mov.b32 %0, {t0, t1};\n\t}"
        : "=r"(r)
        : "l"(a), "l"(b));
  return r;
}
// Saturated elements of a scaled pair (counted for finite, nonzero blocks).
template <int EF>
__device__ __forceinline__ uint32_t lt_sat2(low_f2 v) {
  return (uint32_t)(fabsf(low_f2_lo(v)) > LowFmt<EF>::kMax) + (uint32_t)(fabsf(low_f2_hi(v)) > LowFmt<EF>::kMax);
}
// The output words of 16 pairs x[k] scaled by m (FP4: words 0-3; FP6: 0-7),
// all zero when `zero`; saturated elements added to nsat when SAT.
template <int EF, bool SAT>
__device__ __forceinline__ void lt_codes16(const low_f2 (&x)[16], low_f2 m, bool zero, uint32_t (&o)[8],
                                           unsigned long long& nsat) {
  const uint32_t keep = zero ? 0u : 0xFFFFFFFFu;
  uint32_t ns = 0;
  if constexpr (EF == kE2M1) {
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const low_f2 a = low_f2_mul(x[4 * j], m), b = low_f2_mul(x[4 * j + 1], m);
      const low_f2 c = low_f2_mul(x[4 * j + 2], m), d = low_f2_mul(x[4 * j + 3], m);
      if constexpr (SAT) ns += lt_sat2<EF>(a) + lt_sat2<EF>(b) + lt_sat2<EF>(c) + lt_sat2<EF>(d);
      o[j] = lt_fp4_word(a, b, c, d) & keep;
    }
#pragma unroll
    for (int j = 4; j < 8; j++) o[j] = 0u;
  } else {
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const low_f2 a = low_f2_mul(x[2 * j], m), b = low_f2_mul(x[2 * j + 1], m);
      if constexpr (SAT) ns += lt_sat2<EF>(a) + lt_sat2<EF>(b);
      o[j] = lt_fp6_word<EF>(a, b) & keep;
    }
  }
  if constexpr (SAT)
    if (!zero) nsat += ns;
}

// Rowwise: one lane per 1x32 block (row r of the block's 32, column block b
// of the strip's 8).  Writes the codes, returns the scale byte (0 if the
// block is not ours).  Stage layout as in the MXFP8 kernel: 16-byte chunk c
// of row r of a 64-column box sits at chunk c ^ (r % 8).
template <int EF, bool SAT>
__device__ __forceinline__ uint32_t lt_row_block(const LowParams& p, const unsigned char* stage, int r, int b,
                                                 int64_t r0, int nr, int64_t c0, int nc, unsigned long long& nsat) {
  constexpr bool kFp4 = EF == kE2M1;
  if (r >= nr || 32 * b >= nc) return 0u;
  const unsigned char* line = stage + (b >> 1) * kLtSubBytes + r * 128;
  const int cb = (b & 1) * 4;
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const uint4 v = *(const uint4*)(line + (((cb + j) ^ (r & 7)) << 4));
    w[4 * j] = v.x;
    w[4 * j + 1] = v.y;
    w[4 * j + 2] = v.z;
    w[4 * j + 3] = v.w;
  }
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 16; q++) m = absmax_nan_bf16x2(m, w[q]);
  const uint32_t amax = max((m & 0x7FFFu) << 16, m & 0x7FFF0000u);
  const uint32_t byte = low_scale_byte<EF>(amax, p.round_up);
  const bool zero = amax == 0u || byte == 0xFFu;
  const float mul = low_multiplier(byte);
  low_f2 x[16];
#pragma unroll
  for (int k = 0; k < 16; k++) x[k] = low_f2_make(bf16_lo(w[k]), bf16_hi(w[k]));
  uint32_t o[8];
  lt_codes16<EF, SAT>(x, low_f2_make(mul, mul), zero, o, nsat);
  uint8_t* dst = p.q_row + (r0 + r) * (kFp4 ? p.cols / 2 : p.cols) + (c0 / 32 + b) * (kFp4 ? 16 : 32);
  *(uint4*)dst = make_uint4(o[0], o[1], o[2], o[3]);
  if constexpr (!kFp4) *(uint4*)(dst + 16) = make_uint4(o[4], o[5], o[6], o[7]);
  return byte;
}

// s_row bytes of one warp's 8 rows: lane l holds row 8w + l % 8, blocks
// l / 8 (y0) and 4 + l / 8 (y1).  All 32 lanes must call.
__device__ __forceinline__ void lt_row_scales(const LowParams& p, int warp, int lane, int64_t r0, int nr,
                                              int64_t c0, int nc, uint32_t y0, uint32_t y1) {
  const int r = 8 * warp + (lane & 7);
  const uint32_t v = y0 | (y1 << 8);
  const uint32_t v1 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 8);
  const uint32_t v2 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 16);
  const uint32_t v3 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 24);
  if (r >= nr) return;
  uint8_t* dst = p.s_row + (r0 + r) * (p.cols / 32) + c0 / 32;
  if (nc == kLtCols && ((uintptr_t)dst & 7u) == 0) {
    if (lane < 8) {
      const uint64_t lo = (v & 0xFFu) | ((v1 & 0xFFu) << 8) | ((v2 & 0xFFu) << 16) | ((v3 & 0xFFu) << 24);
      const uint64_t hi = (v >> 8) | ((v1 >> 8) << 8) | ((v2 >> 8) << 16) | ((v3 >> 8) << 24);
      *(uint64_t*)dst = lo | (hi << 32);
    }
    return;
  }
  const int b = lane >> 3;
  if (32 * b < nc) dst[b] = (uint8_t)y0;
  if (32 * (b + 4) < nc) dst[b + 4] = (uint8_t)y1;
}

// Columnwise: thread t owns columns 2t and 2t + 1 (one 32-bit word per row).
// Writes both columns' codes; returns their scale bytes (column 2t in bits
// 0-7).  Rows past the tensor's end are zeros (TMA fill).
template <int EF, bool SAT>
__device__ __forceinline__ uint32_t lt_col_pair(const LowParams& p, const unsigned char* stage, int tid, int64_t r0,
                                                int nr, int64_t c0, int64_t col_len, bool col_vec,
                                                unsigned long long& nsat) {
  constexpr bool kFp4 = EF == kE2M1;
  const unsigned char* seg = stage + (tid >> 5) * kLtSubBytes + 4 * (tid & 3);
  const int c = (tid & 31) >> 2;
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; i++) w[i] = *(const uint32_t*)(seg + i * 128 + ((c ^ (i & 7)) << 4));
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 32; i++) m = absmax_nan_bf16x2(m, w[i]);
  const uint32_t ma = (m & 0x7FFFu) << 16, mb = m & 0x7FFF0000u;
  const uint32_t ba = low_scale_byte<EF>(ma, p.round_up), bb = low_scale_byte<EF>(mb, p.round_up);
  const bool za = ma == 0u || ba == 0xFFu, zb = mb == 0u || bb == 0xFFu;
#pragma unroll
  for (int h = 0; h < 2; h++) {
    // rows 2k and 2k + 1 of column 2t (low halves, h = 0) or 2t + 1 (h = 1)
    low_f2 x[16];
#pragma unroll
    for (int k = 0; k < 16; k++)
      x[k] = h ? low_f2_make(bf16_hi(w[2 * k]), bf16_hi(w[2 * k + 1]))
               : low_f2_make(bf16_lo(w[2 * k]), bf16_lo(w[2 * k + 1]));
    const float mul = low_multiplier(h ? bb : ba);
    uint32_t o[8];
    lt_codes16<EF, SAT>(x, low_f2_make(mul, mul), h ? zb : za, o, nsat);
    uint8_t* dst = p.q_col + (c0 + 2 * tid + h) * col_len + (kFp4 ? r0 / 2 : r0);
    if (col_vec && nr == 32) {
      *(uint4*)dst = make_uint4(o[0], o[1], o[2], o[3]);
      if constexpr (!kFp4) *(uint4*)(dst + 16) = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      const int nbytes = kFp4 ? nr / 2 : nr;
#pragma unroll
      for (int k = 0; k < (kFp4 ? 16 : 32); k++)
        if (k < nbytes) dst[k] = (uint8_t)(o[k >> 2] >> (8 * (k & 3)));
    }
  }
  return ba | (bb << 8);
}

template <int EF, int DIR, bool SAT>
__global__ void __launch_bounds__(kLtThreads, 4) mxlow_tma_kernel(const __grid_constant__ CUtensorMap tmap, LowParams p) {
  constexpr bool kFp4 = EF == kE2M1;
  extern __shared__ unsigned char lt_smem[];
  __shared__ uint64_t full[kLtStages], empty[kLtStages];
  __shared__ volatile int abort_flag;
  unsigned char* stages = lt_smem + ((1024 - (smem_u32(lt_smem) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kLtStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kLtCons / 32);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (tid == kLtCons) prefetch_tensormap(&tmap);
  pdl_wait();
  __syncthreads();
  const int64_t nbr = (p.rows + 31) / 32, strips = (p.cols + kLtCols - 1) / kLtCols;
  const int64_t units = (nbr + kLtUnit - 1) / kLtUnit * strips;
  const uint64_t budget = g_low_budget_ns;

  if (warp == kLtCons / 32) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    int64_t k = 0;
    bool stop = false;
    for (int64_t u = blockIdx.x; u < units && !abort_flag && !stop; u += gridDim.x) {
      const int64_t ur = u / strips;
      const int c0 = (int)((u - ur * strips) * kLtCols);
      for (int j = 0; j < kLtUnit && ur * kLtUnit + j < nbr; j++, ++k) {
        const int s = (int)(k % kLtStages);
        const uint32_t round = (uint32_t)(k / kLtStages);
        if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1u, budget)) {
          atomicOr(&g_low_error, 1u);
          abort_flag = 1;
          stop = true;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kLtStageBytes);
        unsigned char* dst = stages + s * kLtStageBytes;
        const int row = (int)((ur * kLtUnit + j) * 32);
#pragma unroll
        for (int q = 0; q < kLtCols / kLtSubCols; q++)
          tma_load_2d(dst + q * kLtSubBytes, &tmap, c0 + q * kLtSubCols, row, &full[s]);
      }
    }
    pdl_launch_dependents();
    const int64_t first = k > kLtStages ? k - kLtStages : 0;  // every issued copy lands before exit
    for (int64_t j = first; j < k; j++)
      mbar_wait(&full[j % kLtStages], (uint32_t)((j / kLtStages) & 1), 2000000000ull);
    return;
  }

  // ---------------- consumers ----------------
  unsigned long long sat_r = 0, sat_c = 0;
  const int64_t col_len = kFp4 ? p.rows / 2 : p.rows;
  const bool col_vec = (col_len % 16) == 0 && ((uintptr_t)p.q_col & 15) == 0;
  int64_t k = 0;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t ur = u / strips;
    const int64_t c0 = (u - ur * strips) * kLtCols;
    const int nc = (int)min((int64_t)kLtCols, p.cols - c0);
    const int64_t rb0 = ur * kLtUnit;
    const int nblk = (int)min((int64_t)kLtUnit, nbr - rb0);
    uint32_t sc = 0, sd = 0;  // this thread's two columns' scale bytes over the unit
    bool gave_up = false;
    for (int j = 0; j < nblk; j++, ++k) {
      const int s = (int)(k % kLtStages);
      const uint32_t round = (uint32_t)(k / kLtStages);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], round & 1u, budget))) {
        atomicOr(&g_low_error, 1u);
        abort_flag = 1;
        gave_up = true;
        break;
      }
      const unsigned char* stage = stages + s * kLtStageBytes;
      const int64_t r0 = (rb0 + j) * 32;
      const int nr = (int)min((int64_t)32, p.rows - r0);
      if constexpr (DIR & MXFP8_ROW) {
        const int r = 8 * warp + (lane & 7);
        const uint32_t y0 = lt_row_block<EF, SAT>(p, stage, r, lane >> 3, r0, nr, c0, nc, sat_r);
        const uint32_t y1 = lt_row_block<EF, SAT>(p, stage, r, 4 + (lane >> 3), r0, nr, c0, nc, sat_r);
        lt_row_scales(p, warp, lane, r0, nr, c0, nc, y0, y1);
      }
      if constexpr (DIR & MXFP8_COL) {
        if (2 * tid < nc) {
          const uint32_t b = lt_col_pair<EF, SAT>(p, stage, tid, r0, nr, c0, col_len, col_vec, sat_c);
          sc |= (b & 0xFFu) << (8 * j);
          sd |= (b >> 8) << (8 * j);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (gave_up || abort_flag) return;
    if constexpr (DIR & MXFP8_COL) {
      if (2 * tid < nc) {  // s_col[c][rb0 .. rb0 + nblk): one word when aligned and whole
        uint8_t* d0 = p.s_col + (c0 + 2 * tid) * nbr + rb0;
        uint8_t* d1 = d0 + nbr;
        if (nblk == kLtUnit && ((uintptr_t)d0 & 3u) == 0 && ((uintptr_t)d1 & 3u) == 0) {
          *(uint32_t*)d0 = sc;
          *(uint32_t*)d1 = sd;
        } else {
          for (int j = 0; j < nblk; j++) {
            d0[j] = (uint8_t)(sc >> (8 * j));
            d1[j] = (uint8_t)(sd >> (8 * j));
          }
        }
      }
    }
  }
  if constexpr (SAT) {
    const unsigned long long a = warp_sum_u64(sat_r), c = warp_sum_u64(sat_c);
    if (lane == 0 && a) atomicAdd(p.sat, a);
    if (lane == 0 && c) atomicAdd(p.sat + 1, c);
  }
  pdl_launch_dependents();
}

static PFN_cuTensorMapEncodeTiled_v12000 lt_encode_fn() {
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

template <int EF, int DIR, bool SAT>
static cudaError_t lt_launch(const CUtensorMap& map, const LowParams& p, cudaStream_t stream) {
  auto kernel = mxlow_tma_kernel<EF, DIR, SAT>;
  constexpr size_t smem = 1024 + (size_t)kLtStages * kLtStageBytes;
  static bool attr = false;
  static int per_sm = 1;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kLtThreads, smem) != cudaSuccess ||
          per_sm < 1)
        per_sm = 1;
      attr = true;
    }
  }
  const int64_t units = ((p.rows + 31) / 32 + kLtUnit - 1) / kLtUnit * ((p.cols + kLtCols - 1) / kLtCols);
  // one CTA per unit (the hardware's block scheduler balances the tail), or
  // a persistent grid of every resident slot
  int64_t grid = FP8Q_LOW_GRID_ALL ? units : (int64_t)per_sm * sm_count();
  if (grid > units) grid = units;
  if (grid > 0x7FFFFFFF) grid = 0x7FFFFFFF;  // the kernel walks any remaining units
  if (grid < 1) grid = 1;
  return launch_kernel(kernel, dim3((unsigned)grid), dim3(kLtThreads), smem, stream, map, p);
}

template <int EF, bool SAT>
static cudaError_t lt_launch_dir(const CUtensorMap& map, const LowParams& p, cudaStream_t stream) {
  if (p.dir == MXFP8_ROW) return lt_launch<EF, MXFP8_ROW, SAT>(map, p, stream);
  if (p.dir == MXFP8_COL) return lt_launch<EF, MXFP8_COL, SAT>(map, p, stream);
  return lt_launch<EF, MXFP8_BOTH, SAT>(map, p, stream);
}

template <int EF>
static cudaError_t lt_launch_typed(const LowParams& p, cudaStream_t stream, bool* encoded) {
  auto enc = lt_encode_fn();
  *encoded = enc != nullptr;
  if (!enc) return cudaSuccess;
  CUtensorMap map;
  cuuint64_t dims[2] = {(cuuint64_t)p.cols, (cuuint64_t)p.rows};
  cuuint64_t strides[1] = {(cuuint64_t)p.cols * 2};
  cuuint32_t box[2] = {kLtSubCols, 32};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *encoded = false;
    return cudaSuccess;
  }
  return p.sat ? lt_launch_dir<EF, true>(map, p, stream) : lt_launch_dir<EF, false>(map, p, stream);
}

fp8q_status low_device_status(bool clear, unsigned* word) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_low_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (clear && v) {
    const unsigned z = 0;
    e = cudaMemcpyToSymbol(g_low_error, &z, sizeof(z));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
  }
  *word = v;
  return FP8Q_OK;
}

fp8q_status low_set_wait_budget(unsigned long long ns) {
  cudaError_t e = cudaMemcpyToSymbol(g_low_budget_ns, &ns, sizeof(ns));
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, "cudaMemcpyToSymbol(wait budget)");
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
#ifndef FP8Q_LOW_TMA  // BF16 input through the TMA-fed kernel
#define FP8Q_LOW_TMA 1
#endif
  if (dt == kBF16 && FP8Q_LOW_TMA) {
    // the TMA kernel needs a tensor map (16-byte aligned x, row pitch a
    // multiple of 16 bytes: cols % 32 == 0 gives it); it falls back to the
    // cp.async kernel when the driver cannot encode one
    bool encoded = false;
    e = elem == kE2M1 ? lt_launch_typed<kE2M1>(p, stream, &encoded)
        : elem == kE2M3 ? lt_launch_typed<kE2M3>(p, stream, &encoded)
                        : lt_launch_typed<kE3M2>(p, stream, &encoded);
    if (e != cudaSuccess) return cuda_fail(e, "MXFP4/MXFP6 TMA kernel launch");
    if (encoded) return check_launch("MXFP4/MXFP6 TMA kernel");
  }
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
