// nvfp4.cu -- NVFP4: E2M1 elements, one E4M3 scale per 16 elements along a
// row, and one FP32 scale for the tensor.
//
// "混合精度与 FP8 训练" 13.2: NVFP4 blocks are 16 elements of E2M1 (0, 0.5,
// 1, 1.5, 2, 3, 4, 6 and negatives) sharing an E4M3 scale, which need not be
// a power of two and so puts the block's maximum close to 6; because E4M3
// alone lacks the range, an FP32 tensor-level scale is the second level.
// The arithmetic, step by step (each an IEEE single operation):
//   S = 448 * 6 / amax(tensor)          (amax 0 or non-finite -> 1;
//                                        a quotient above FLT_MAX -> FLT_MAX)
//   block code = RNE_sat_E4M3(amax_b * fl32(S / 6)),  d = its value
//   element    = RNE_sat_E2M1(x * fl32(S / d)),       all +0 when d is 0 or NaN
// with two element codes per byte, the even element in the low nibble.
//
// The tensor amax comes first (the amax kernel of percast.cu, into the
// caller's amax buffer); this kernel then streams the tensor once more: a
// thread takes one 16-element block per step (two or four 16-byte loads),
// writes its 8 code bytes and its scale byte.
#include "fp8q_device.cuh"
#include "internal.h"

namespace fp8q {

constexpr int kNvThreads = 256;

struct NvParams {
  const void* x;
  int64_t nblk;            // rows * cols / 16
  const unsigned* amax;    // FP32 bits of the tensor amax
  uint8_t* q;              // [nblk * 8]
  uint8_t* s;              // [nblk]
  float* scale_out;        // S, or nullptr
};

__device__ __forceinline__ float nv_tensor_scale(uint32_t amax_bits) {
  if (amax_bits == 0u || amax_bits >= 0x7F800000u) return 1.0f;
  const float s = __fdiv_rn(2688.0f, __uint_as_float(amax_bits));  // 448 * 6 is exact in FP32
  return s > 3.40282346638528859812e+38f ? 3.40282346638528859812e+38f : s;
}

// Two floats -> one byte of E2M1 codes, a in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
  unsigned short r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tmov.b16 %0, {t, 0};\n\t}"
      : "=h"(r)
      : "f"(b), "f"(a));
  return r & 0xFFu;
}

// E4M3 code -> its exact value (NaN for the NaN codes).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)code));
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((unsigned short)(h2 & 0xFFFFu)));
  return f;
}

template <int DT>
__global__ void __launch_bounds__(kNvThreads) nvfp4_kernel(NvParams p) {
  pdl_wait();
  const uint32_t amax_t = *p.amax;
  const float S = nv_tensor_scale(amax_t);
  const float t = __fdiv_rn(S, 6.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.scale_out) *p.scale_out = S;
  const int64_t stride = (int64_t)gridDim.x * kNvThreads;
  for (int64_t b = (int64_t)blockIdx.x * kNvThreads + threadIdx.x; b < p.nblk; b += stride) {
    float v[16];
    uint32_t am = 0;
    if constexpr (DT == kBF16) {
      const uint4 a = ld_stream((const uint16_t*)p.x + 16 * b);
      const uint4 c = ld_stream((const uint16_t*)p.x + 16 * b + 8);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < 8; k++) {
        m = absmax_bf16x2(m, w[k]);
        v[2 * k] = bf16_lo(w[k]);
        v[2 * k + 1] = bf16_hi(w[k]);
      }
      am = max(m << 16, m & 0xFFFF0000u);
    } else {
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint4 a = ld_stream((const float*)p.x + 16 * b + 4 * k);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          am = max(am, w[i] & 0x7FFFFFFFu);
          v[4 * k + i] = __uint_as_float(w[i]);
        }
      }
    }
    // block scale: E4M3 code of amax_b * (S / 6), NaN made canonical
    const float sval = __fmul_rn(__uint_as_float(am), t);
    const uint32_t code = canon_nan4<kE4M3>(cvt2<kE4M3>(sval, 0.0f)) & 0xFFu;
    const float d = e4m3_value(code);
    uint2 o = make_uint2(0u, 0u);
    if (d != 0.0f && d == d) {
      const float r = __fdiv_rn(S, d);
      uint32_t bytes[8];
#pragma unroll
      for (int i = 0; i < 8; i++) bytes[i] = e2m1x2(__fmul_rn(v[2 * i], r), __fmul_rn(v[2 * i + 1], r));
      o.x = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
      o.y = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
    }
    st_stream(p.q + 8 * b, o);
    p.s[b] = (uint8_t)code;
  }
  pdl_launch_dependents();
}

fp8q_status launch_nvfp4(const void* x, int dt, int64_t rows, int64_t cols, const unsigned* amax, uint8_t* q,
                         uint8_t* s, float* scale_out, cudaStream_t stream) {
  NvParams p{};
  p.x = x;
  p.nblk = rows * cols / 16;
  p.amax = amax;
  p.q = q;
  p.s = s;
  p.scale_out = scale_out;
  static int per_sm = [] {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, nvfp4_kernel<kBF16>, kNvThreads, 0) != cudaSuccess || v < 1)
      v = 1;
    return v;
  }();
  int64_t grid = (p.nblk + kNvThreads - 1) / kNvThreads;
  const int64_t cap = (int64_t)per_sm * sm_count();
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  cudaError_t e = dt == kBF16
                      ? launch_kernel(nvfp4_kernel<kBF16>, dim3((unsigned)grid), dim3(kNvThreads), 0, stream, p)
                      : launch_kernel(nvfp4_kernel<kFP32>, dim3((unsigned)grid), dim3(kNvThreads), 0, stream, p);
  if (e != cudaSuccess) return cuda_fail(e, "nvfp4 kernel launch");
  return check_launch("nvfp4 kernel");
}

}  // namespace fp8q
