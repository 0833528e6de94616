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
// Work split.  Tiles of 32 rows x 512 columns, a thread per column pair: the
// thread's 32 x words (one 4-byte BF16 pair, or 8 bytes of FP32, per row)
// give the two columnwise blocks directly; a rowwise block is 32 columns =
// 16 lanes, whose amax is a max over those lanes by shuffles.  Conversions
// are the hardware cvt.rn.satfinite.{e2m1,e2m3,e3m2}x2 (nearest even,
// saturating).  Reads of x are whole rows of 1 or 2 KB; every store is
// contiguous across the warp.
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
constexpr int kLowTileCols = 2 * kLowThreads;

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

// A thread's x words for the 32 rows of its column pair (c, c + 1): BF16
// one word per row (column c in the low half), FP32 two words per row.
template <int DT> struct LowRows {
  uint32_t w[DT == kBF16 ? 32 : 64];
  __device__ __forceinline__ float a(int i) const {
    if constexpr (DT == kBF16) return bf16_lo(w[i]);
    else return __uint_as_float(w[2 * i]);
  }
  __device__ __forceinline__ float b(int i) const {
    if constexpr (DT == kBF16) return bf16_hi(w[i]);
    else return __uint_as_float(w[2 * i + 1]);
  }
};

template <int DT, int EF, bool SAT>
__global__ void __launch_bounds__(kLowThreads) mxlow_kernel(LowParams p) {
  constexpr bool kFp4 = EF == kE2M1;
  pdl_wait();
  const int64_t ntr = (p.rows + 31) / 32, ntc = (p.cols + kLowTileCols - 1) / kLowTileCols;
  const int64_t ntiles = ntr * ntc;
  const int lane16 = threadIdx.x & 15;
  const int64_t col_len = kFp4 ? p.rows / 2 : p.rows;  // bytes per column of q_col
  const bool col_vec = (col_len % 16) == 0 && ((uintptr_t)p.q_col & 15) == 0;
  unsigned long long sat_r = 0, sat_c = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t tr = t / ntc, tc = t - tr * ntc;
    const int64_t c = tc * kLowTileCols + 2 * threadIdx.x;
    const bool active = c < p.cols;  // cols % 32 == 0: whole 16-lane row blocks are active or not
    const int64_t r0 = tr * 32;
    const int nr = (int)min(p.rows - r0, (int64_t)32);
    LowRows<DT> x;
#pragma unroll
    for (int i = 0; i < 32; i++) {
      const bool ok = active && i < nr;
      if constexpr (DT == kBF16) {
        x.w[i] = ok ? __ldg((const unsigned*)((const uint16_t*)p.x + (r0 + i) * p.cols + c)) : 0u;
      } else {
        const float2 v = ok ? __ldg((const float2*)((const float*)p.x + (r0 + i) * p.cols + c)) : make_float2(0.f, 0.f);
        x.w[2 * i] = __float_as_uint(v.x);
        x.w[2 * i + 1] = __float_as_uint(v.y);
      }
    }

    if ((p.dir & MXFP8_COL) && active) {
      uint32_t ma = 0, mb = 0;
#pragma unroll
      for (int i = 0; i < 32; i++) {
        ma = max(ma, __float_as_uint(x.a(i)) & 0x7FFFFFFFu);
        mb = max(mb, __float_as_uint(x.b(i)) & 0x7FFFFFFFu);
      }
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const uint32_t amax = h ? mb : ma;
        const uint32_t byte = low_scale_byte<EF>(amax, p.round_up);
        const bool zero_codes = amax == 0u || byte == 0xFFu;
        const float mul = low_multiplier(byte);
        // FP6: 32 code bytes = 8 words; E2M1: 16 bytes = 4 words
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; k++) w[k] = 0u;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float s0 = __fmul_rn(h ? x.b(i) : x.a(i), mul), s1 = __fmul_rn(h ? x.b(i + 1) : x.a(i + 1), mul);
          if constexpr (SAT)
            if (!zero_codes) sat_c += (fabsf(s0) > LowFmt<EF>::kMax) + (fabsf(s1) > LowFmt<EF>::kMax);
          const uint32_t two = zero_codes ? 0u : low_cvt2<EF>(s0, s1);
          if constexpr (kFp4) w[i >> 3] |= two << (8 * ((i >> 1) & 3));
          else w[i >> 2] |= two << (16 * ((i >> 1) & 1));
        }
        const int64_t cc = c + h;
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

    if (p.dir & MXFP8_ROW) {
#pragma unroll
      for (int i = 0; i < 32; i++) {
        if (i >= nr) break;  // nr is the same for the whole CTA
        uint32_t m = max(__float_as_uint(x.a(i)) & 0x7FFFFFFFu, __float_as_uint(x.b(i)) & 0x7FFFFFFFu);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (!active) continue;
        const uint32_t byte = low_scale_byte<EF>(m, p.round_up);
        const bool zero_codes = m == 0u || byte == 0xFFu;
        const float mul = low_multiplier(byte);
        const float s0 = __fmul_rn(x.a(i), mul), s1 = __fmul_rn(x.b(i), mul);
        if constexpr (SAT)
          if (!zero_codes) sat_r += (fabsf(s0) > LowFmt<EF>::kMax) + (fabsf(s1) > LowFmt<EF>::kMax);
        const uint32_t two = zero_codes ? 0u : low_cvt2<EF>(s0, s1);
        const int64_t r = r0 + i;
        if constexpr (kFp4) p.q_row[r * (p.cols / 2) + c / 2] = (uint8_t)two;
        else *(uint16_t*)(p.q_row + r * p.cols + c) = (uint16_t)two;
        if (lane16 == 0) p.s_row[r * (p.cols / 32) + c / 32] = (uint8_t)byte;
      }
    }
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
  const int64_t tiles = ((p.rows + 31) / 32) * ((p.cols + kLowTileCols - 1) / kLowTileCols);
  auto kernel = p.sat ? mxlow_kernel<DT, EF, true> : mxlow_kernel<DT, EF, false>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kLowThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  int64_t grid = (int64_t)per_sm * sm_count();
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  return launch_kernel(kernel, dim3((unsigned)grid), dim3(kLowThreads), 0, stream, p);
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
