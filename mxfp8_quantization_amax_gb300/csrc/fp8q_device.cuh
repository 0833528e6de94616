// fp8q_device.cuh -- device-side building blocks shared by the kernels:
// element loads, magnitude-bit amax, the packed saturating RNE cast and the
// E8M0 scale unit.  sm_103a only; no fast-math, no flush-to-zero.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8q {

enum : int { kE4M3 = 0, kE5M2 = 1 };
enum : int { kBF16 = 0, kFP32 = 1 };

// Largest finite value and the exponent of the largest binade of each format
// ("混合精度与 FP8 训练" 2.2: E4M3 max 448 = 1.75 * 2^8; E5M2 shares FP16's
// exponent range, so its max is 1.75 * 2^15 = 57344).
template <int FMT> struct Fmt;
template <> struct Fmt<kE4M3> {
  static constexpr float kMax = 448.0f;
  static constexpr int kEmax = 8;
};
template <> struct Fmt<kE5M2> {
  static constexpr float kMax = 57344.0f;
  static constexpr int kEmax = 15;
};

__host__ __device__ inline float fmt_max(int fmt) { return fmt == kE4M3 ? 448.0f : 57344.0f; }

// ---------------------------------------------------------------------------
// Saturating round-to-nearest-even cast of two FP32 values; `a` lands in the
// low byte.  satfinite clamps overflow and +-Inf to +-max.
// ---------------------------------------------------------------------------
template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float a, float b) {
  uint16_t r;
  if constexpr (FMT == kE4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Four FP32 values -> four codes in one word (v0 in the low byte).  The two
// 16-bit results are the halves of one register (no byte permute and no
// zero-extension of each half: 12% fewer instructions in the MXFP8 rowwise
// pass).
#ifndef FP8Q_CVT4_MOV
#define FP8Q_CVT4_MOV 1
#endif
template <int FMT>
__device__ __forceinline__ uint32_t cvt4(float v0, float v1, float v2, float v3) {
#if FP8Q_CVT4_MOV
  uint32_t r;
  if constexpr (FMT == kE4M3)
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  else
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  return r;
#else
  return __byte_perm(cvt2<FMT>(v0, v1), cvt2<FMT>(v2, v3), 0x5410);
#endif
}

// Every NaN code becomes 0x7F (positive, all mantissa bits set) in both
// formats, whatever sign or payload the hardware conversion produced.  With
// satfinite a finite or infinite input never yields these codes, so only
// NaN inputs are touched.  Works on four codes at once.
template <int FMT>
__device__ __forceinline__ uint32_t canon_nan4(uint32_t w) {
  const uint32_t t = w & 0x7F7F7F7Fu;
  // E4M3 NaN: low 7 bits 0x7F.  E5M2 NaN: low 7 bits 0x7D..0x7F.
  const uint32_t m = (t + (FMT == kE4M3 ? 0x01010101u : 0x03030303u)) & 0x80808080u;
  const uint32_t fill = m - (m >> 7);  // 0x7F in every flagged byte
  return (w & ~(m | fill)) | fill;
}

// ---------------------------------------------------------------------------
// BF16 pairs: a 32-bit word holds element 2i in its low half.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed magnitude max of two BF16 pairs (16-bit unsigned max of |bits|).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(w & 0x7FFF7FFFu));
  return r;
}
// max(|a|, |b|) per BF16 half, NaN-propagating; only the magnitude bits of
// the result are meaningful (the sign is the xor of the operands' signs).
__device__ __forceinline__ uint32_t absmax_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two FP32 products in one packed instruction (IEEE round to nearest, no FTZ).
__device__ __forceinline__ void mul2(float& a, float& b, float sa, float sb) {
  unsigned long long x, s, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %2};" : "=l"(s) : "f"(sa), "f"(sb));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(s));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

// L2 eviction policies for stores: streamed outputs leave L2 first, the
// small scale arrays (written a few bytes at a time by many CTAs) stay until
// their sectors are complete.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
#ifndef FP8Q_PDL  // programmatic dependent launch between the library's kernels
#define FP8Q_PDL 1
#endif

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialization allowed, so it may start while the
// kernel before it on the stream is still finishing.  pdl_wait() blocks
// until the grids this one depends on have completed and their memory
// operations are visible; every kernel calls it before its first access to
// global memory (reads of its inputs and writes of its outputs alike).
// pdl_launch_dependents() lets the next kernel on the stream be scheduled
// early; that kernel waits in its own pdl_wait() for this grid to finish.
// Kernels call it once a CTA's main loop is done, not at their start: the
// next grid's CTAs then take the slots of CTAs that have finished instead
// of crowding onto whichever SMs had room first, which would unbalance a
// persistent grid whose work is dealt out by CTA index.
__device__ __forceinline__ void pdl_wait() {
#if FP8Q_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_launch_dependents() {
#if FP8Q_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Emits nothing; marks v as rewritten here.  A run of volatile loads
// followed by one of these per loaded vector keeps every load issued before
// the first use of any of them, so a thread has all its loads in flight.
__device__ __forceinline__ void reg_fence(uint4& v) {
  asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_u8_hint(void* p, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b8 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_u16_hint(void* p, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(p), "h"((unsigned short)v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_u32_hint(void* p, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_u64_hint(void* p, uint64_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(p), "l"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st32B_hint(void* p, const uint32_t (&d)[8], uint64_t pol) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(p),
               "r"(d[0]), "r"(d[1]), "r"(d[2]), "r"(d[3]), "r"(d[4]), "r"(d[5]), "r"(d[6]), "r"(d[7]), "l"(pol)
               : "memory");
}

// 32-byte store (one full sector) with no L1 allocation.
__device__ __forceinline__ void st32B(void* p, const uint32_t (&d)[8]) {
  asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(d[0]), "r"(d[1]),
               "r"(d[2]), "r"(d[3]), "r"(d[4]), "r"(d[5]), "r"(d[6]), "r"(d[7])
               : "memory");
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// ---------------------------------------------------------------------------
// E8M0 scale unit ("Blackwell GPU MXFP8 预训练最佳实践" 4.1).
// For amax = m * 2^e (m in [1,2)) and destmax = 1.75 * 2^emax:
//   ceil(log2(amax / destmax)) = e - emax + (m > 1.75)
// exactly, because m / 1.75 lies in [4/7, 8/7).  The byte is X + 127,
// clamped to [0, 254] (X in [-127, 127]); subnormal and zero amax land on
// X = -127.  Inf/NaN amax gives 0xFF.  amax_bits: FP32 bits, sign clear.
// ---------------------------------------------------------------------------
template <int FMT>
__device__ __forceinline__ uint32_t e8m0_from_amax(uint32_t amax_bits, int round_up = 1) {
  if (amax_bits >= 0x7F800000u) return 0xFFu;
  // round_up 0: the OCP rule, X = floor(log2 amax) - e_max (no mantissa term)
  const int b = (int)(amax_bits >> 23) - Fmt<FMT>::kEmax + ((round_up && (amax_bits & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  return (uint32_t)min(max(b, 0), 254);
}

// 2^-X for X = byte - 127 as an FP32 multiplier (exact; 2^-127 is subnormal).
__device__ __forceinline__ float e8m0_multiplier(uint32_t byte) {
  return byte <= 253u ? __uint_as_float((254u - byte) << 23) : __uint_as_float(0x00400000u);
}

// ---------------------------------------------------------------------------
// Per-tensor scale ("HiFloat8：高性能训练之路" 1.2 eqs. 1 and 3):
// fl32(fl32(F8max / amax) * 2^-margin); amax 0 -> 1; non-finite -> 1;
// an overflowing quotient -> FLT_MAX.  IEEE division, no approximation.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float scale_from_amax(uint32_t amax_bits, float f8max, int margin) {
  if (amax_bits >= 0x7F800000u || amax_bits == 0u) return 1.0f;
  float s = __fdiv_rn(f8max, __uint_as_float(amax_bits));
  if (s > 3.40282346638528859812e+38f) s = 3.40282346638528859812e+38f;
  return __fmul_rn(s, __uint_as_float((uint32_t)(127 - margin) << 23));
}

// ---------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) { return __reduce_max_sync(0xFFFFFFFFu, v); }

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Cache-hinted vector memory access.  Inputs are read once through the
// read-only path without L1 allocation; outputs are written once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_stream(void* p, uint2 v) {
  asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Group of flat element e for row offsets `off` (G+1 entries, NULL = one
// group): the last g with off[g] * cols <= e.  Offsets are clamped so a bad
// array cannot steer the caller out of range.
__device__ __forceinline__ int group_of_row(const int64_t* off, int G, int64_t row) {
  if (off == nullptr || G <= 1) return 0;
  int lo = 0, hi = G;  // answer in [0, G-1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(off + mid) <= row) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace fp8q
