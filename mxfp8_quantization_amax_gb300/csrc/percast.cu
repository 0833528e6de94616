// percast.cu -- per-tensor (per-group) amax and scaled cast.
//
// "HiFloat8：高性能训练之路" 1.2: Scale = F8max / Amax (eq. 1), X * Scale ->
// FP8 (eq. 2); delayed scaling replaces Amax by the history max and
// multiplies by 2^-N (eqs. 3-4).  "混合精度与 FP8 训练" 8.1-8.2: the cast
// saturates; computing amax costs a read of the whole tensor, which delayed
// scaling fuses into the cast itself.
//
// Work is split into chunks of kChunk elements; each CTA owns a contiguous
// run of chunks, so its group (rows [off[g], off[g+1]) of the flat tensor)
// changes rarely.  A chunk inside one group takes the vector path: every
// thread issues all of its 16-byte loads first, then converts.  Chunks that
// straddle a group boundary, and the ragged tail, take an element path.
// Per-group amax / saturation partials are reduced per CTA and merged with
// one atomic per CTA and group; the last CTA to finish (atomic ticket, no
// waiting) publishes the per-group results and re-zeroes the accumulators.
//
// Current scaling takes the amax kernel, then the cast kernel, except for an
// ungrouped tensor, which takes one launch: up to 2 MB, one thread-block
// cluster (current_cluster_kernel); beyond that, up to 8 times what fits on
// chip, a cooperative grid that keeps slices in registers and shared memory
// across a grid-wide wait for the scale and streams the rest
// (current_fused_kernel).
//
// The kernels wait for the grid before them (griddepcontrol.wait) but do not
// trigger the next launch early: a next grid launched into the slots this
// one frees first lands unevenly, which slowed back-to-back delayed steps on
// 8192^2 (resident grids with fixed shares): 33.8 -> 33.0 us per step
// without the trigger.  The exception is a single-launch grid of at most
// half the resident slots (1024^2 from a CUDA graph: 6.45 -> 6.30 us).
#include <stdio.h>

#include "fp8q_device.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fp8q {

constexpr int kPtThreads = 256;
#ifndef FP8Q_PT_VECS
#define FP8Q_PT_VECS 8
#endif
constexpr int kVecs = FP8Q_PT_VECS;  // 16-byte vectors per thread per chunk (bytes in flight per thread / 16)

template <int DT> struct InT;
template <> struct InT<kBF16> {
  static constexpr int kPerVec = 8;  // elements per 16-byte vector
  static constexpr int kChunk = kPtThreads * kVecs * kPerVec;  // elements per chunk
  static __device__ __forceinline__ uint32_t bits(const void* x, int64_t i) {
    return (uint32_t)__ldg((const unsigned short*)x + i) << 16;
  }
};
template <> struct InT<kFP32> {
  static constexpr int kPerVec = 4;
  static constexpr int kChunk = kPtThreads * kVecs * kPerVec;
  static __device__ __forceinline__ uint32_t bits(const void* x, int64_t i) {
    return __ldg((const unsigned*)x + i);
  }
};

// Failure word of this file's kernels: bit 0 is set when the single-launch
// current scaling gave up waiting for its scale.  Read and cleared by
// fp8q_check_device().
__device__ unsigned int g_pt_error;

struct KParams {
  const void* x;
  int64_t n, cols, rows;
  const int64_t* off;
  int G;
  int64_t n_chunks;
  float f8max;
  int margin;
  int src;
  const float* scale_in;
  const float* hist;
  int hist_count;
  unsigned* counter;
  unsigned* acc;
  float* ws_scale;
  unsigned long long* sat_acc;
  uint8_t* q;
  float* amax_out;
  float* scale_out;
  float* scale_inv_out;
  unsigned long long* sat_out;
  float* hist_slot;
  unsigned* flag;
  int l2_hint;  // 0: default, 1: keep the input in L2 (a second pass follows), 2: last use
  // elements [0, keep_n) of x are loaded with the hint l2_hint_pre instead:
  // the prefix of a tensor too large for L2 that the second pass re-reads
  int64_t keep_n;
  int l2_hint_pre;
  int early_trigger;  // single-launch path: trigger the next launch after the cast
};

// 16-byte read-only load with an L2 eviction policy (createpolicy value).
__device__ __forceinline__ uint4 ld_hint(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ uint64_t load_policy(int hint) {
  if (hint == 1) return policy_evict_last();
  if (hint == 2) return policy_evict_first();
  return policy_evict_normal();
}

__device__ __forceinline__ int group_of_elem(const KParams& p, int64_t e) {
  if (p.off == nullptr || p.G <= 1) return 0;
  return group_of_row(p.off, p.G, e / p.cols);
}

// Elements [e0, e1) of group g, from offsets clamped to [0, rows].
struct GroupSpan {
  int g;
  int64_t e0, e1;
};

__device__ __forceinline__ int64_t clamped_row(const KParams& p, int g) {
  if (p.off == nullptr) return g == 0 ? 0 : p.rows;
  const int64_t v = __ldg(p.off + g);
  return v < 0 ? 0 : (v > p.rows ? p.rows : v);
}

// The group of element e (the last g with offsets[g] <= its row, as
// group_of_elem) and that group's span.  e may lie outside the span when
// the offsets leave rows uncovered; such elements belong to group g all the
// same, as they always have.
__device__ __forceinline__ GroupSpan span_of(const KParams& p, int64_t e) {
  GroupSpan s;
  s.g = group_of_elem(p, e);
  s.e0 = clamped_row(p, s.g) * p.cols;
  s.e1 = clamped_row(p, s.g + 1) * p.cols;
  return s;
}

// A forward cursor over the groups: elements are visited in increasing
// order, so the span is looked up again (binary search) only when an
// element leaves it.  Returns the group of e.
__device__ __forceinline__ int cursor_group(const KParams& p, GroupSpan& s, int64_t e) {
  if (p.off == nullptr || p.G <= 1) return 0;
  if (!(s.e0 <= e && e < s.e1)) s = span_of(p, e);
  return s.g;
}

// Block-wide max / sum over NT threads (sh: NT / 32 entries); every thread
// must call (block-uniform control flow).
template <int NT = kPtThreads>
__device__ __forceinline__ uint32_t block_max(uint32_t v, uint32_t* sh) {
  v = warp_max_u32(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; i++) r = max(r, sh[i]);
  return r;
}
template <int NT = kPtThreads>
__device__ __forceinline__ unsigned long long block_sum(unsigned long long v, unsigned long long* sh) {
  v = warp_sum_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  unsigned long long r = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; i++) r += sh[i];
  return r;
}

// Last CTA to arrive returns true (all earlier CTAs' atomics are visible).
__device__ __forceinline__ bool arrive_last(unsigned* counter) {
  __shared__ bool last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (last) __threadfence();
  return last;
}

// ---------------------------------------------------------------------------
// Amax pass
// ---------------------------------------------------------------------------
// Amax of the CTA's chunks [c_begin, c_end), merged into p.acc[group] with
// one atomic per CTA and group.  Block-uniform: every thread calls it.
template <int DT>
__device__ __forceinline__ void amax_pass(const KParams& p, int64_t c_begin, int64_t c_end, uint64_t pol_rest,
                                          uint64_t pol_pre, uint32_t* sh_max) {
  int cur_g = -1;
  uint32_t cur = 0;
  auto flush = [&]() {  // block-uniform
    const uint32_t m = block_max(cur, sh_max);
    if (threadIdx.x == 0 && cur_g >= 0 && m != 0) atomicMax(p.acc + cur_g, m);
    cur = 0;
  };
  constexpr int PV = InT<DT>::kPerVec;
  constexpr int V = kVecs;
  GroupSpan span{0, 0, -1};  // the chunk's group (block-uniform)

  for (int64_t c = c_begin; c < c_end; ++c) {
    const int64_t e0 = c * InT<DT>::kChunk;
    const uint64_t pol = e0 < p.keep_n ? pol_pre : pol_rest;
    const int64_t e1 = min(e0 + (int64_t)InT<DT>::kChunk, p.n);
    const int g0 = cursor_group(p, span, e0);
    const bool one_group = p.off == nullptr || p.G <= 1 || (span.e0 <= e0 && e1 <= span.e1);
    if (one_group) {
      if (g0 != cur_g) {
        if (cur_g >= 0) flush();
        cur_g = g0;
      }
    } else if (cur_g >= 0) {
      flush();  // per-thread group runs below, merged with atomics
      cur_g = -1;
    }
    if (one_group && e1 - e0 == InT<DT>::kChunk) {
      // whole vectors: all loads first, then the maxima
      uint4 v[V];
#pragma unroll
      for (int k = 0; k < V; k++)
        v[k] = ld_hint((const char*)p.x + (e0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV) * (DT == kBF16 ? 2 : 4), pol);
#pragma unroll
      for (int k = 0; k < V; k++) reg_fence(v[k]);
      if constexpr (DT == kBF16) {
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < V; k++) {
          m = absmax_bf16x2(m, v[k].x);
          m = absmax_bf16x2(m, v[k].y);
          m = absmax_bf16x2(m, v[k].z);
          m = absmax_bf16x2(m, v[k].w);
        }
        cur = max(cur, max(m << 16, m & 0xFFFF0000u));
      } else {
#pragma unroll
        for (int k = 0; k < V; k++)
          cur = max(max(cur, max(v[k].x & 0x7FFFFFFFu, v[k].y & 0x7FFFFFFFu)),
                    max(v[k].z & 0x7FFFFFFFu, v[k].w & 0x7FFFFFFFu));
      }
    } else if (one_group) {
      for (int64_t e = e0 + threadIdx.x; e < e1; e += kPtThreads) cur = max(cur, InT<DT>::bits(p.x, e) & 0x7FFFFFFFu);
    } else {
      // a chunk that crosses groups (rare): per-thread group runs, merged
      // with atomics; whole vectors when no vector can straddle a group
      GroupSpan tspan{0, 0, -1};
      int tg = -1;
      uint32_t tm = 0;
      auto take = [&](int64_t e, uint32_t m) {
        const int g = cursor_group(p, tspan, e);
        if (g != tg) {
          if (tg >= 0 && tm) atomicMax(p.acc + tg, tm);
          tg = g;
          tm = 0;
        }
        tm = max(tm, m);
      };
      if (e1 - e0 == InT<DT>::kChunk && p.cols % PV == 0) {
        for (int k = 0; k < V; k++) {
          const int64_t e = e0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV;
          const uint4 v = ld_hint((const char*)p.x + e * (DT == kBF16 ? 2 : 4), pol);
          uint32_t m;
          if constexpr (DT == kBF16) {
            const uint32_t h = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(0u, v.x), v.y), v.z), v.w);
            m = max(h << 16, h & 0xFFFF0000u);
          } else {
            m = max(max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu));
          }
          take(e, m);
        }
      } else {
        for (int64_t e = e0 + threadIdx.x; e < e1; e += kPtThreads) take(e, InT<DT>::bits(p.x, e) & 0x7FFFFFFFu);
      }
      if (tg >= 0 && tm) atomicMax(p.acc + tg, tm);
    }
  }
  if (cur_g >= 0) flush();
}

// Turns the merged amaxes into the scales (current scaling) and publishes
// them; returns the accumulators to zero.  Run by the last CTA.
__device__ __forceinline__ void publish_scales(const KParams& p) {
  for (int g = threadIdx.x; g < p.G; g += kPtThreads) {
    const uint32_t a = *(volatile unsigned*)(p.acc + g);
    const float s = scale_from_amax(a, p.f8max, p.margin);
    p.ws_scale[g] = s;
    if (p.amax_out) p.amax_out[g] = __uint_as_float(a);
    if (p.scale_out) p.scale_out[g] = s;
    if (p.scale_inv_out) p.scale_inv_out[g] = __frcp_rn(s);
    if (g == 0) {
      if (p.hist_slot) *p.hist_slot = __uint_as_float(a);
      if (p.flag && a >= 0x7F800000u) atomicOr(p.flag, 1u);
    }
    p.acc[g] = 0;
  }
}

template <int DT, bool FINALIZE>
__global__ void __launch_bounds__(kPtThreads) amax_kernel(KParams p) {
  __shared__ uint32_t sh_max[kPtThreads / 32];
  pdl_wait();
  const int64_t c_begin = p.n_chunks * blockIdx.x / gridDim.x;
  const int64_t c_end = p.n_chunks * (blockIdx.x + 1) / gridDim.x;
  amax_pass<DT>(p, c_begin, c_end, load_policy(p.l2_hint), load_policy(p.l2_hint_pre), sh_max);

  if constexpr (FINALIZE) {
    if (arrive_last(p.counter)) {
      publish_scales(p);
      if (threadIdx.x == 0) *p.counter = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// Cast pass
// ---------------------------------------------------------------------------
__device__ __forceinline__ float group_scale(const KParams& p, int g, float hist_scale) {
  if (p.src == kSrcGiven) return __ldg(p.scale_in + g);
  if (p.src == kSrcWorkspace) return *(volatile float*)(p.ws_scale + g);
  return hist_scale;
}

// Cast of the CTA's chunks [c_begin, c_end) with the per-group scale of
// `p.src`; optional fused amax (p.acc) and saturation count (p.sat_acc).
// Block-uniform: every thread calls it.
// One 16-byte vector: codes of its PV elements scaled by s, stored at q[e];
// its amax and saturated elements are added to m / nsat.
template <int DT, int FMT>
__device__ __forceinline__ void cast_vec(const KParams& p, const uint4& v, int64_t e, float s, bool do_amax,
                                         bool do_sat, uint32_t& m, unsigned long long& nsat) {
  constexpr float kMax = Fmt<FMT>::kMax;
  if constexpr (DT == kBF16) {
    float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                  bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
    for (int i = 0; i < 8; i++) f[i] = __fmul_rn(f[i], s);
    if (do_sat) {
#pragma unroll
      for (int i = 0; i < 8; i++) nsat += fabsf(f[i]) > kMax;
    }
    if (do_amax) {
      const uint32_t h = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(0u, v.x), v.y), v.z), v.w);
      m = max(m, max(h << 16, h & 0xFFFF0000u));
    }
    uint2 o;
    o.x = canon_nan4<FMT>(cvt4<FMT>(f[0], f[1], f[2], f[3]));
    o.y = canon_nan4<FMT>(cvt4<FMT>(f[4], f[5], f[6], f[7]));
    st_stream(p.q + e, o);
  } else {
    float f[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w)};
    if (do_amax)
      m = max(max(m, max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu)), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu));
#pragma unroll
    for (int i = 0; i < 4; i++) f[i] = __fmul_rn(f[i], s);
    if (do_sat) {
#pragma unroll
      for (int i = 0; i < 4; i++) nsat += fabsf(f[i]) > kMax;
    }
    *(uint32_t*)(p.q + e) = canon_nan4<FMT>(cvt4<FMT>(f[0], f[1], f[2], f[3]));
  }
}

// Cast of the CTA's chunks [c_begin, c_end) with the per-group scale of
// `p.src`; optional fused amax (p.acc) and saturation count (p.sat_acc).
// Block-uniform: every thread calls it.
template <int DT, int FMT>
__device__ __forceinline__ void cast_pass(const KParams& p, int64_t c_begin, int64_t c_end, uint64_t pol_rest,
                                          uint64_t pol_pre, float hist_scale, uint32_t* sh_max,
                                          unsigned long long* sh_sum) {
  constexpr float kMax = Fmt<FMT>::kMax;
  constexpr int PV = InT<DT>::kPerVec;
  constexpr int V = kVecs;
  const bool do_amax = p.acc != nullptr;
  const bool do_sat = p.sat_acc != nullptr;
  int cur_g = -1;
  uint32_t cur = 0;
  unsigned long long nsat = 0;

  auto flush = [&]() {  // block-uniform
    if (do_amax) {
      const uint32_t m = block_max(cur, sh_max);
      if (threadIdx.x == 0 && m != 0) atomicMax(p.acc + cur_g, m);
    }
    if (do_sat) {
      const unsigned long long s = block_sum(nsat, sh_sum);
      if (threadIdx.x == 0 && s != 0) atomicAdd(p.sat_acc + cur_g, s);
    }
    cur = 0;
    nsat = 0;
  };
  GroupSpan span{0, 0, -1};

  for (int64_t c = c_begin; c < c_end; ++c) {
    const int64_t e0 = c * InT<DT>::kChunk;
    const uint64_t pol = e0 < p.keep_n ? pol_pre : pol_rest;
    const int64_t e1 = min(e0 + (int64_t)InT<DT>::kChunk, p.n);
    const int g0 = cursor_group(p, span, e0);
    const bool one_group = p.off == nullptr || p.G <= 1 || (span.e0 <= e0 && e1 <= span.e1);
    if (one_group) {
      if (g0 != cur_g) {
        if (cur_g >= 0) flush();
        cur_g = g0;
      }
    } else if (cur_g >= 0) {
      flush();
      cur_g = -1;
    }
    if (one_group) {
      const float s = group_scale(p, g0, hist_scale);
      if (e1 - e0 == InT<DT>::kChunk) {
        uint4 v[V];
#pragma unroll
        for (int k = 0; k < V; k++)
          v[k] = ld_hint((const char*)p.x + (e0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV) * (DT == kBF16 ? 2 : 4), pol);
#pragma unroll
        for (int k = 0; k < V; k++) reg_fence(v[k]);
#pragma unroll
        for (int k = 0; k < V; k++)
          cast_vec<DT, FMT>(p, v[k], e0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV, s, do_amax, do_sat, cur, nsat);
      } else {
        for (int64_t e = e0 + threadIdx.x; e < e1; e += kPtThreads) {
          const uint32_t b = InT<DT>::bits(p.x, e);
          const float f = __fmul_rn(__uint_as_float(b), s);
          if (do_sat) nsat += fabsf(f) > kMax;
          if (do_amax) cur = max(cur, b & 0x7FFFFFFFu);
          p.q[e] = (uint8_t)canon_nan4<FMT>(cvt2<FMT>(f, 0.0f));
        }
      }
    } else {
      // a chunk that crosses groups (rare): per-thread group runs, merged
      // with atomics; whole vectors when no vector can straddle a group
      GroupSpan tspan{0, 0, -1};
      int tg = -1;
      uint32_t tm = 0;
      unsigned long long ts = 0;
      float tscale = 1.0f;
      auto thread_group = [&](int g) {
        if (g == tg) return;
        if (tg >= 0) {
          if (do_amax && tm) atomicMax(p.acc + tg, tm);
          if (do_sat && ts) atomicAdd(p.sat_acc + tg, ts);
        }
        tg = g;
        tm = 0;
        ts = 0;
        if (g >= 0) tscale = group_scale(p, g, hist_scale);
      };
      if (e1 - e0 == InT<DT>::kChunk && p.cols % PV == 0) {
        for (int k = 0; k < V; k++) {
          const int64_t e = e0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV;
          const uint4 v = ld_hint((const char*)p.x + e * (DT == kBF16 ? 2 : 4), pol);
          thread_group(cursor_group(p, tspan, e));
          cast_vec<DT, FMT>(p, v, e, tscale, do_amax, do_sat, tm, ts);
        }
      } else {
        for (int64_t e = e0 + threadIdx.x; e < e1; e += kPtThreads) {
          thread_group(cursor_group(p, tspan, e));
          const uint32_t b = InT<DT>::bits(p.x, e);
          const float f = __fmul_rn(__uint_as_float(b), tscale);
          if (do_sat) ts += fabsf(f) > kMax;
          if (do_amax) tm = max(tm, b & 0x7FFFFFFFu);
          p.q[e] = (uint8_t)canon_nan4<FMT>(cvt2<FMT>(f, 0.0f));
        }
      }
      thread_group(-1);  // merge this thread's last run
    }
  }
  if (cur_g >= 0) flush();
}

// Publishes the fused amax / saturation results and returns the scratch
// (accumulators, the current-scaling scales) to zero.  Run by the last CTA.
__device__ __forceinline__ void publish_cast_results(const KParams& p) {
  const bool do_amax = p.acc != nullptr;
  const bool do_sat = p.sat_acc != nullptr;
  for (int g = threadIdx.x; g < p.G; g += kPtThreads) {
    if (p.src == kSrcWorkspace) p.ws_scale[g] = 0.0f;
    if (do_amax) {
      const uint32_t a = *(volatile unsigned*)(p.acc + g);
      if (p.amax_out) p.amax_out[g] = __uint_as_float(a);
      if (p.hist_slot && g == 0) {
        *p.hist_slot = __uint_as_float(a);
        if (a >= 0x7F800000u) atomicOr(p.flag, 1u);
      }
      p.acc[g] = 0;
    }
    if (do_sat) {
      const unsigned long long s = *(volatile unsigned long long*)(p.sat_acc + g);
      if (p.sat_out) p.sat_out[g] = s;
      p.sat_acc[g] = 0;
    }
  }
}

template <int DT, int FMT>
__global__ void __launch_bounds__(kPtThreads, 4) cast_kernel(KParams p) {
  __shared__ uint32_t sh_max[kPtThreads / 32];
  __shared__ unsigned long long sh_sum[kPtThreads / 32];
  constexpr float kMax = Fmt<FMT>::kMax;
  pdl_wait();

  float hist_scale = 1.0f;
  if (p.src == kSrcHistory) {  // max over the filled history entries
    uint32_t hm = 0;
    for (int i = threadIdx.x; i < p.hist_count; i += kPtThreads)
      hm = max(hm, __float_as_uint(p.hist[i]) & 0x7FFFFFFFu);
    hist_scale = scale_from_amax(block_max(hm, sh_max), kMax, p.margin);
  }
  if (blockIdx.x == 0 && p.src != kSrcWorkspace) {
    for (int g = threadIdx.x; g < p.G; g += kPtThreads) {
      const float s = group_scale(p, g, hist_scale);
      if (p.scale_out) p.scale_out[g] = s;
      if (p.scale_inv_out) p.scale_inv_out[g] = __frcp_rn(s);
    }
  }

  const int64_t c_begin = p.n_chunks * blockIdx.x / gridDim.x;
  const int64_t c_end = p.n_chunks * (blockIdx.x + 1) / gridDim.x;
  cast_pass<DT, FMT>(p, c_begin, c_end, load_policy(p.l2_hint), load_policy(p.l2_hint_pre), hist_scale, sh_max,
                     sh_sum);

  // The last CTA publishes per-group results and returns the scratch it used
  // (accumulators, counters, the current-scaling scales) to zero.
  if (p.acc != nullptr || p.sat_acc != nullptr || p.src == kSrcWorkspace) {
    if (arrive_last(p.counter)) {
      publish_cast_results(p);
      if (threadIdx.x == 0) *p.counter = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// Current scaling of a small ungrouped tensor in one launch
// ---------------------------------------------------------------------------
// One chunk per CTA, every CTA resident at once (a cooperative launch).  A
// CTA loads its chunk into registers and merges its amax; the last CTA to
// arrive turns the amax into the scale and publishes it (publish_scales);
// the others wait for it and cast from their registers.  x is read once and
// the two passes need no second launch.  The counter holds the arrivals and
// departures in its low bits and kPublished once the scale is out; the last
// CTA to depart publishes the saturation count and returns the workspace to
// zero.  The wait is bounded: a CTA that gives up records it in g_pt_error
// and writes no codes.
constexpr unsigned kPublished = 0x80000000u;
__device__ unsigned long long g_pt_wait_budget_ns = 1000000000ull;
// Test hook: while nonzero the last CTA to arrive does not publish, so
// every other CTA's wait runs out its budget.
__device__ unsigned g_pt_stall_publish;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Spins until `*word` has kPublished set; false once budget_ns has passed.
__device__ __forceinline__ bool wait_published(const unsigned* word, uint64_t budget_ns) {
  if (ld_acquire_u32(word) & kPublished) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1; !(ld_acquire_u32(word) & kPublished); ++n) {
    if ((n & 15u) == 0 && globaltimer_ns() - t0 > budget_ns) return false;
  }
  return true;
}

#ifndef FP8Q_PT_FUSED_VECS  // 16-byte vectors per thread of the single-launch path
#define FP8Q_PT_FUSED_VECS 8
#endif
template <int DT> struct FusedChunk {
  static constexpr int kVecs = FP8Q_PT_FUSED_VECS;
  static constexpr int kElems = kPtThreads * kVecs * InT<DT>::kPerVec;
};

// Magnitude bits of a 16-byte vector folded into h (BF16: two lanes of
// BF16 magnitudes, finished by absmax_bits; FP32: the bits themselves).
template <int DT>
__device__ __forceinline__ void absmax_fold(const uint4& v, uint32_t& h) {
  if constexpr (DT == kBF16) {
    h = absmax_bf16x2(h, v.x);
    h = absmax_bf16x2(h, v.y);
    h = absmax_bf16x2(h, v.z);
    h = absmax_bf16x2(h, v.w);
  } else {
    h = max(max(h, max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu)), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu));
  }
}
template <int DT>
__device__ __forceinline__ uint32_t absmax_bits(uint32_t h) {
  if constexpr (DT == kBF16) return max(h << 16, h & 0xFFFF0000u);
  return h;
}

// The streamed chunks [s0, s1) of this CTA when the tensor has more chunks
// than the grid's on-chip slices (two per CTA), and the end of the share
// kept in L2; false when there are none.
template <int DT>
__device__ __forceinline__ bool stream_range(const KParams& p, int64_t& s0, int64_t& s1, int64_t& keep) {
  static_assert(FusedChunk<DT>::kElems == InT<DT>::kChunk, "streamed chunks are slices");
  const int64_t on_chip = 2 * (int64_t)gridDim.x;
  if (p.n_chunks <= on_chip) return false;
  const int64_t rest = p.n_chunks - on_chip;
  s0 = on_chip + rest * blockIdx.x / gridDim.x;
  s1 = on_chip + rest * (blockIdx.x + 1) / gridDim.x;
  keep = s0 + kL2KeepBytes / ((int64_t)InT<DT>::kChunk * (DT == kBF16 ? 2 : 4)) / gridDim.x;
  return s1 > s0;
}

// SL slices per CTA: the first in registers, the second (SL == 2) staged in
// shared memory by one bulk copy, which doubles the tensors that fit.
template <int DT, int FMT, int SL>
__global__ void __launch_bounds__(kPtThreads, 4) current_fused_kernel(KParams p) {
  extern __shared__ uint4 fused_slice[];  // SL == 2: the CTA's second slice
  __shared__ uint64_t slice_bar;
  __shared__ uint32_t sh_max[kPtThreads / 32];
  __shared__ unsigned long long sh_sum[kPtThreads / 32];
  __shared__ float sh_scale;
  __shared__ int sh_state;  // 1: scale published, 0: wait gave up
  constexpr int PV = InT<DT>::kPerVec;
  constexpr int V = FusedChunk<DT>::kVecs;
  constexpr int kElems = FusedChunk<DT>::kElems;
  constexpr float kMax = Fmt<FMT>::kMax;
  constexpr int kEsz = DT == kBF16 ? 2 : 4;
  pdl_wait();

  // slice held in registers: [e0, e1); second slice: [f0, f1), staged when whole
  const int64_t e0 = (int64_t)blockIdx.x * SL * kElems;
  const int64_t e1 = min(e0 + (int64_t)kElems, p.n);
  const bool whole = e1 - e0 == kElems;
  const int64_t f0 = e1, f1 = SL == 2 ? min(f0 + (int64_t)kElems, p.n) : f0;
  const bool staged = SL == 2 && f1 - f0 == kElems;
  const uint64_t pol = policy_evict_first();
  const uint64_t budget = g_pt_wait_budget_ns;
  if constexpr (SL == 2) {
    if (staged) {  // block-uniform
      if (threadIdx.x == 0) {
        mbar_init(&slice_bar, 1);
        fence_barrier_init();
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&slice_bar, kElems * kEsz);
        bulk_load(fused_slice, (const char*)p.x + f0 * kEsz, kElems * kEsz, &slice_bar, pol);
      }
    }
  }

  // A tensor larger than the on-chip slices (two per CTA of a full grid):
  // every CTA also streams an equal range of the remaining chunks (slices),
  // reduced here and cast after the wait.  That range is read twice; its
  // first chunks (an equal share of kL2KeepBytes per CTA) are loaded
  // evict-last so that the second read finds them in L2.
  uint32_t h = 0, m = 0;
  if constexpr (SL == 2) {
    int64_t s0, s1, keep;
    if (stream_range<DT>(p, s0, s1, keep)) {  // block-uniform
      for (int64_t c = s0; c < s1; ++c) {
        const int64_t c0 = c * kElems, c1 = min(c0 + (int64_t)kElems, p.n);
        if (c1 - c0 == kElems) {
          const uint64_t pc = c < keep ? policy_evict_last() : pol;
          uint4 w[V];
#pragma unroll
          for (int k = 0; k < V; k++)
            w[k] = ld_hint((const char*)p.x + (c0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV) * kEsz, pc);
#pragma unroll
          for (int k = 0; k < V; k++) reg_fence(w[k]);
#pragma unroll
          for (int k = 0; k < V; k++) absmax_fold<DT>(w[k], h);
        } else {
          for (int64_t e = c0 + threadIdx.x; e < c1; e += kPtThreads) m = max(m, InT<DT>::bits(p.x, e) & 0x7FFFFFFFu);
        }
      }
    }
  }

  uint4 v[V];
  if (whole) {
#pragma unroll
    for (int k = 0; k < V; k++)
      v[k] = ld_hint((const char*)p.x + (e0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV) * kEsz, pol);
#pragma unroll
    for (int k = 0; k < V; k++) reg_fence(v[k]);
#pragma unroll
    for (int k = 0; k < V; k++) absmax_fold<DT>(v[k], h);
  } else {  // the ragged last slice: element by element (read again below)
    for (int64_t e = e0 + threadIdx.x; e < e1; e += kPtThreads) m = max(m, InT<DT>::bits(p.x, e) & 0x7FFFFFFFu);
  }
  bool landed = true;  // the staged slice arrived within the wait budget
  if constexpr (SL == 2) {
    if (staged) {
      landed = __syncthreads_and(mbar_wait(&slice_bar, 0, budget)) != 0;
      if (landed) {
#pragma unroll
        for (int k = 0; k < V; k++) absmax_fold<DT>(fused_slice[k * kPtThreads + threadIdx.x], h);
      } else if (threadIdx.x == 0) {
        atomicOr(&g_pt_error, 1u);
      }
    } else {
      for (int64_t e = f0 + threadIdx.x; e < f1; e += kPtThreads) m = max(m, InT<DT>::bits(p.x, e) & 0x7FFFFFFFu);
    }
  }
  m = max(m, absmax_bits<DT>(h));
  m = block_max(m, sh_max);

  // Arrival, by thread 0 for the CTA: its amax, then a ticket.  The tickets
  // form one chain of read-modify-writes with release semantics, so the last
  // CTA's acquiring ticket sees every other CTA's amax; it publishes the
  // scale with a releasing add, which the others' acquiring polls see.
  if (threadIdx.x == 0) {
    if (m != 0) atomicMax(p.acc, m);
    if (atom_add_acq_rel(p.counter, 1u) == gridDim.x - 1u) {
      if (!*(volatile unsigned*)&g_pt_stall_publish) {
        publish_scales(p);  // one group: thread 0 alone does all of it
        sh_scale = *(volatile float*)p.ws_scale;
        sh_state = 1;
        red_add_release(p.counter, kPublished);
      } else {
        sh_state = 0;
      }
    } else {
      const bool ok = wait_published(p.counter, g_pt_wait_budget_ns);
      sh_state = ok;
      if (ok) {
        sh_scale = *(volatile float*)p.ws_scale;
      } else {
        atomicOr(&g_pt_error, 1u);
      }
    }
  }
  __syncthreads();
  const bool ok = sh_state != 0;
  const float s = sh_scale;

  // cast from the registers (and the staged slice)
  unsigned long long nsat = 0;
  auto cast_elems = [&](int64_t a, int64_t b) {
    for (int64_t e = a + threadIdx.x; e < b; e += kPtThreads) {
      const float f = __fmul_rn(__uint_as_float(InT<DT>::bits(p.x, e)), s);
      nsat += fabsf(f) > kMax;
      p.q[e] = (uint8_t)canon_nan4<FMT>(cvt2<FMT>(f, 0.0f));
    }
  };
  if (ok) {
    uint32_t unused = 0;
    if (whole) {
#pragma unroll
      for (int k = 0; k < V; k++)
        cast_vec<DT, FMT>(p, v[k], e0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV, s, false,
                          p.sat_acc != nullptr, unused, nsat);
    } else {
      cast_elems(e0, e1);
    }
    if constexpr (SL == 2) {
      if (staged) {
        if (landed) {
#pragma unroll
          for (int k = 0; k < V; k++)
            cast_vec<DT, FMT>(p, fused_slice[k * kPtThreads + threadIdx.x],
                              f0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV, s, false, p.sat_acc != nullptr,
                              unused, nsat);
        }
      } else {
        cast_elems(f0, f1);
      }
      int64_t s0, s1, keep;
      if (stream_range<DT>(p, s0, s1, keep)) {  // the streamed range, read again (last use)
        for (int64_t c = s0; c < s1; ++c) {
          const int64_t c0 = c * kElems, c1 = min(c0 + (int64_t)kElems, p.n);
          if (c1 - c0 == kElems) {
            uint4 w[V];
#pragma unroll
            for (int k = 0; k < V; k++)
              w[k] = ld_hint((const char*)p.x + (c0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV) * kEsz, pol);
#pragma unroll
            for (int k = 0; k < V; k++) reg_fence(w[k]);
#pragma unroll
            for (int k = 0; k < V; k++)
              cast_vec<DT, FMT>(p, w[k], c0 + (int64_t)(k * kPtThreads + threadIdx.x) * PV, s, false,
                                p.sat_acc != nullptr, unused, nsat);
          } else {
            cast_elems(c0, c1);
          }
        }
      }
    }
  }
  // a grid of at most half the resident slots lets the next launch start
  // early (it then has room beside this one; larger grids do not: the note
  // at the top of the file)
  if (p.early_trigger) pdl_launch_dependents();
  unsigned long long t = 0;
  if (p.sat_acc != nullptr) t = block_sum(nsat, sh_sum);

  // Departure, by thread 0: its saturation count, then a ticket on the same
  // chain; the last CTA to depart publishes the count and clears the
  // workspace.  The codes need no ordering with it.
  if (threadIdx.x == 0) {
    if (t != 0) atomicAdd(p.sat_acc, t);
    const unsigned ticket = atom_add_acq_rel(p.counter, 1u) & ~kPublished;
    if (ticket == 2u * gridDim.x - 1u) {
      if (p.sat_acc != nullptr) {
        const unsigned long long total = *(volatile unsigned long long*)p.sat_acc;
        if (p.sat_out && ok) *p.sat_out = total;
        *p.sat_acc = 0;
      }
      *p.acc = 0;
      *p.ws_scale = 0.0f;
      *p.counter = 0;
    }
  }
  if constexpr (SL == 2) {
    // a copy that outlived the budget must land before the CTA exits
    if (staged && !landed && threadIdx.x == 0) mbar_wait(&slice_bar, 0, 2000000000ull);
  }
}

// ---------------------------------------------------------------------------
// Current scaling of a tiny ungrouped tensor: one thread-block cluster
// ---------------------------------------------------------------------------
// The 16 CTAs of one cluster (scheduled together by the hardware) each copy
// an equal share of x into shared memory with bulk copies, reduce its amax,
// and exchange the amaxes through distributed shared memory between
// hardware cluster barriers; every CTA then knows the scale and casts its
// share.  No workspace, no global ticket, no cooperative launch.
// Up to 2 MB of x: in a host loop of calls the one-cluster launch beats the
// cooperative single launch from 32 KB (3.4 against 8.2 us) to 2 MB (7.2
// against 8.4 us, where its device time is longer: 6.7 against 6.2 us from a
// CUDA graph); at 3 MB it is slower either way (8.3 against 6.5 us).
constexpr int kClusterCtas = 16;                          // non-portable cluster size
constexpr int kClusterCopy = 16384;                       // bytes per bulk copy
constexpr int kClusterMaxBytes = 8 * kClusterCopy;        // shared memory per CTA

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives, then waits for all.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The 32-bit word at this CTA's shared address `p`, read from CTA `rank`.
__device__ __forceinline__ uint32_t ld_cluster_u32(const void* p, uint32_t rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_cluster_u64(const void* p, uint32_t rank) {
  uint32_t remote;
  unsigned long long v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote) : "memory");
  return v;
}

// Threads per CTA of the one-cluster kernel.  2 MB, host loop / CUDA graph:
// 128 threads 8.45 / 7.97 us, 256 7.20 / 6.72, 512 6.84 / 6.36, 1024
// 7.36 / 6.89.
#ifndef FP8Q_PT_CLUSTER_THREADS
#define FP8Q_PT_CLUSTER_THREADS 512
#endif
constexpr int kClThreads = FP8Q_PT_CLUSTER_THREADS;

template <int DT, int FMT>
__global__ void __launch_bounds__(kClThreads, 1) current_cluster_kernel(KParams p) {
  extern __shared__ uint4 cl_data[];  // this CTA's share of x
  __shared__ uint64_t cl_bar;
  __shared__ uint32_t sh_max[kClThreads / 32];
  __shared__ unsigned long long sh_sum[kClThreads / 32];
  __shared__ uint32_t cl_amax;  // this CTA's amax bits; bit 31 set: its copy gave up
  __shared__ unsigned long long cl_sat;
  __shared__ float cl_scale;
  __shared__ int cl_ok;
  constexpr int PV = InT<DT>::kPerVec;
  constexpr float kMax = Fmt<FMT>::kMax;
  pdl_wait();

  // 16-byte vectors [v0, v1) of x; the last CTA also takes the n % PV tail
  const uint32_t rank = cluster_ctarank();
  const int64_t nvec = p.n / PV;
  const int64_t v0 = nvec * rank / kClusterCtas, v1 = nvec * (rank + 1) / kClusterCtas;
  const int nv = (int)(v1 - v0);
  const uint64_t pol = policy_evict_first();
  if (nv > 0) {  // block-uniform
    if (threadIdx.x == 0) {
      mbar_init(&cl_bar, 1);
      fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t bytes = (uint32_t)nv * 16u;
      mbar_arrive_expect_tx(&cl_bar, bytes);
      for (uint32_t o = 0; o < bytes; o += kClusterCopy)
        bulk_load((char*)cl_data + o, (const char*)p.x + v0 * 16 + o, min((uint32_t)kClusterCopy, bytes - o), &cl_bar,
                  pol);
    }
  }
  const bool landed = nv == 0 || __syncthreads_and(mbar_wait(&cl_bar, 0, g_pt_wait_budget_ns)) != 0;
  uint32_t h = 0, m = 0;
  if (landed) {
    for (int i = threadIdx.x; i < nv; i += kClThreads) absmax_fold<DT>(cl_data[i], h);
  }
  const int64_t t0 = nvec * PV;  // the tail elements, in the last CTA
  if (rank == kClusterCtas - 1)
    for (int64_t e = t0 + threadIdx.x; e < p.n; e += kClThreads) m = max(m, InT<DT>::bits(p.x, e) & 0x7FFFFFFFu);
  m = block_max<kClThreads>(max(m, absmax_bits<DT>(h)), sh_max);
  if (threadIdx.x == 0) {
    cl_amax = landed ? m : 0x80000000u;
    if (!landed) atomicOr(&g_pt_error, 1u);
  }
  cluster_sync();  // every CTA's amax is in its shared memory

  if (threadIdx.x < 32) {  // warp 0: the tensor's amax from all CTAs
    const uint32_t a = threadIdx.x < kClusterCtas ? ld_cluster_u32(&cl_amax, threadIdx.x) : 0u;
    const uint32_t all = __reduce_or_sync(0xFFFFFFFFu, a & 0x80000000u);
    const uint32_t amax = __reduce_max_sync(0xFFFFFFFFu, a & 0x7FFFFFFFu);
    if (threadIdx.x == 0) {
      const float s = scale_from_amax(amax, p.f8max, p.margin);
      cl_scale = s;
      cl_ok = all == 0u;
      if (rank == 0 && all == 0u) {
        if (p.amax_out) *p.amax_out = __uint_as_float(amax);
        if (p.scale_out) *p.scale_out = s;
        if (p.scale_inv_out) *p.scale_inv_out = __frcp_rn(s);
      }
    }
  }
  __syncthreads();
  const bool ok = cl_ok != 0;
  const float s = cl_scale;
  unsigned long long nsat = 0;
  if (ok) {
    uint32_t unused = 0;
    for (int i = threadIdx.x; i < nv; i += kClThreads)
      cast_vec<DT, FMT>(p, cl_data[i], (v0 + i) * PV, s, false, p.sat_acc != nullptr, unused, nsat);
    if (rank == kClusterCtas - 1) {
      for (int64_t e = t0 + threadIdx.x; e < p.n; e += kClThreads) {
        const float f = __fmul_rn(__uint_as_float(InT<DT>::bits(p.x, e)), s);
        nsat += fabsf(f) > kMax;
        p.q[e] = (uint8_t)canon_nan4<FMT>(cvt2<FMT>(f, 0.0f));
      }
    }
  }
  if (p.early_trigger) pdl_launch_dependents();
  if (p.sat_out != nullptr) {  // block-uniform
    const unsigned long long t = block_sum<kClThreads>(nsat, sh_sum);
    if (threadIdx.x == 0) cl_sat = t;
  }
  cluster_sync();  // every CTA's count is in its shared memory
  if (rank == 0 && p.sat_out != nullptr && ok && threadIdx.x < 32) {
    // a CTA holds at most 128 KB of x, so every count and the total fit 32 bits
    const unsigned c = threadIdx.x < kClusterCtas ? (unsigned)ld_cluster_u64(&cl_sat, threadIdx.x) : 0u;
    const unsigned total = __reduce_add_sync(0xFFFFFFFFu, c);
    if (threadIdx.x == 0) *p.sat_out = total;
  }
  cluster_sync();  // no CTA leaves while CTA 0 reads its shared memory
  // a copy that outlived the budget must land before the CTA exits
  if (nv > 0 && !landed && threadIdx.x == 0) mbar_wait(&cl_bar, 0, 2000000000ull);
}

// ---------------------------------------------------------------------------
// Scales from given amaxes (the cast pass of a tensor split across devices,
// after the per-device amaxes were combined)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPtThreads) scale_kernel(const float* amax, int G, float f8max, int margin,
                                                           float* scale_out, float* scale_inv_out) {
  pdl_wait();
  for (int g = blockIdx.x * kPtThreads + threadIdx.x; g < G; g += gridDim.x * kPtThreads) {
    const float s = scale_from_amax(__float_as_uint(amax[g]) & 0x7FFFFFFFu, f8max, margin);
    scale_out[g] = s;
    if (scale_inv_out) scale_inv_out[g] = __frcp_rn(s);
  }
}

// ---------------------------------------------------------------------------
// Zeroing of a few result words (counters, amax accumulators) in stream
// order, as a kernel: a memset between two kernels breaks the chain of
// programmatic launches, and the kernel after it could not start early (the
// MXFP8 quantizer with saturation counts at 4096^2: 20.0 against 14.4 us per
// call).  It lets the next kernel launch at once and only then waits for the
// kernel before it; the next kernel's own wait covers this one.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPtThreads) zero_words_kernel(uint32_t* p, int n) {
  pdl_launch_dependents();
  pdl_wait();
  for (int i = blockIdx.x * kPtThreads + threadIdx.x; i < n; i += gridDim.x * kPtThreads) p[i] = 0u;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static KParams make_params(const PtLaunch& L) {
  KParams p{};
  p.x = L.x;
  p.rows = L.rows;
  p.cols = L.cols;
  p.n = L.rows * L.cols;
  p.off = L.off;
  p.G = L.G;
  const int64_t chunk = L.dt == kBF16 ? InT<kBF16>::kChunk : InT<kFP32>::kChunk;
  p.n_chunks = (p.n + chunk - 1) / chunk;
  p.f8max = fmt_max(L.fmt);
  p.margin = L.margin;
  p.src = L.src;
  p.scale_in = L.scale_in;
  p.hist = L.hist;
  p.hist_count = L.hist_count;
  p.counter = L.counter;
  p.acc = L.acc;
  p.ws_scale = L.ws_scale;
  p.sat_acc = L.sat_acc;
  p.q = L.q;
  p.amax_out = L.amax_out;
  p.scale_out = L.scale_out;
  p.scale_inv_out = L.scale_inv_out;
  p.sat_out = L.sat_out;
  p.hist_slot = L.hist_slot;
  p.flag = L.flag;
  p.l2_hint = L.l2_hint;
  p.keep_n = L.keep_n;
  p.l2_hint_pre = L.l2_hint_pre;
  return p;
}

template <typename K>
static int ctas_per_sm(K kernel) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kPtThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return per_sm;
}

#ifndef FP8Q_PT_BALANCED_GRID  // 1: as few CTAs as give every CTA the same chunk count
#define FP8Q_PT_BALANCED_GRID 1
#endif
// Large tensors: CTAs of FP8Q_PT_CHUNKS_PER_CTA chunks, many waves of them,
// which the hardware's block scheduler hands out in order as slots free (the
// CTAs in flight then cover one moving window of the tensor, and the last
// wave is a small share of the launch).  Measured for amax + cast:
// 65536 x 7168 with 64 groups 386 -> 358 us, 16384 x 14336 192 -> 179 us.
// Smaller tensors (fewer than FP8Q_PT_MANY_WAVES waves of such CTAs) keep
// one wave of resident CTAs with equal contiguous ranges: at 8192 x 8192,
// 1.7 waves of small CTAs cost 55.8 -> 61.9 us.
#ifndef FP8Q_PT_CHUNKS_PER_CTA
#define FP8Q_PT_CHUNKS_PER_CTA 4
#endif
#ifndef FP8Q_PT_MANY_WAVES
#define FP8Q_PT_MANY_WAVES 2
#endif
static int grid_for(int64_t n_chunks, int per_sm) {
  const int64_t resident = (int64_t)per_sm * sm_count();
  if (FP8Q_PT_CHUNKS_PER_CTA > 0 && n_chunks >= (int64_t)FP8Q_PT_MANY_WAVES * FP8Q_PT_CHUNKS_PER_CTA * resident) {
    const int64_t g = (n_chunks + FP8Q_PT_CHUNKS_PER_CTA - 1) / FP8Q_PT_CHUNKS_PER_CTA;
    return (int)(g > 0x7FFFFFFF ? 0x7FFFFFFF : g);
  }
  int64_t g = n_chunks < resident ? n_chunks : resident;
  if (FP8Q_PT_BALANCED_GRID && n_chunks > resident) {
    const int64_t per_cta = (n_chunks + resident - 1) / resident;
    g = (n_chunks + per_cta - 1) / per_cta;
  }
  return (int)(g < 1 ? 1 : g);
}

fp8q_status launch_amax(const PtLaunch& L, bool finalize_scales) {
  KParams p = make_params(L);
  cudaError_t e;
  if (L.dt == kBF16) {
    if (finalize_scales) {
      static int r = ctas_per_sm(amax_kernel<kBF16, true>);
      e = launch_kernel(amax_kernel<kBF16, true>, dim3(grid_for(p.n_chunks, r)), dim3(kPtThreads), 0, L.stream, p);
    } else {
      static int r = ctas_per_sm(amax_kernel<kBF16, false>);
      e = launch_kernel(amax_kernel<kBF16, false>, dim3(grid_for(p.n_chunks, r)), dim3(kPtThreads), 0, L.stream, p);
    }
  } else {
    if (finalize_scales) {
      static int r = ctas_per_sm(amax_kernel<kFP32, true>);
      e = launch_kernel(amax_kernel<kFP32, true>, dim3(grid_for(p.n_chunks, r)), dim3(kPtThreads), 0, L.stream, p);
    } else {
      static int r = ctas_per_sm(amax_kernel<kFP32, false>);
      e = launch_kernel(amax_kernel<kFP32, false>, dim3(grid_for(p.n_chunks, r)), dim3(kPtThreads), 0, L.stream, p);
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "amax kernel launch");
  return check_launch("amax kernel");
}

template <int DT, int FMT>
static cudaError_t launch_cast_t(const KParams& p, cudaStream_t s) {
  static int r = ctas_per_sm(cast_kernel<DT, FMT>);
  return launch_kernel(cast_kernel<DT, FMT>, dim3(grid_for(p.n_chunks, r)), dim3(kPtThreads), 0, s, p);
}

fp8q_status launch_cast(const PtLaunch& L) {
  KParams p = make_params(L);
  cudaError_t e;
  if (L.dt == kBF16) {
    if (L.fmt == kE4M3) e = launch_cast_t<kBF16, kE4M3>(p, L.stream);
    else e = launch_cast_t<kBF16, kE5M2>(p, L.stream);
  } else {
    if (L.fmt == kE4M3) e = launch_cast_t<kFP32, kE4M3>(p, L.stream);
    else e = launch_cast_t<kFP32, kE5M2>(p, L.stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "cast kernel launch");
  return check_launch("cast kernel");
}

// Single-launch current scaling (current_fused_kernel): taken for an
// ungrouped, non-empty tensor whose chunks fit one per resident CTA.
#ifndef FP8Q_PT_FUSED  // 0: always the two-pass path
#define FP8Q_PT_FUSED 1
#endif
#ifndef FP8Q_PT_FUSED_PDL  // 1: the launch also allows programmatic overlap with the kernel before it
#define FP8Q_PT_FUSED_PDL 1
#endif
#ifndef FP8Q_PT_FUSED_COOP  // 1: a cooperative launch (all CTAs resident, or the launch fails)
#define FP8Q_PT_FUSED_COOP 1
#endif
#ifndef FP8Q_PT_FUSED_SLICES  // most slices per CTA of the single-launch path (1 or 2)
#define FP8Q_PT_FUSED_SLICES 2
#endif
// Beyond the on-chip slices the single launch streams the rest of the tensor
// (read twice, partly from L2), up to FP8Q_PT_STREAM_MAX times the on-chip
// slices; larger tensors take the two kernels, which a single launch no
// longer beats (16384 x 14336: 176.3 us two kernels, 178.4 us one launch).
#ifndef FP8Q_PT_STREAM_MAX
#define FP8Q_PT_STREAM_MAX 8
#endif
template <int DT, int FMT, int SL>
static cudaError_t launch_fused_sl(const KParams& p, int64_t grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kPtThreads);
  cfg.dynamicSmemBytes = SL == 2 ? (size_t)FusedChunk<DT>::kElems * (DT == kBF16 ? 2 : 4) : 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (FP8Q_PT_FUSED_COOP) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na++].val.cooperative = 1;
  }
  if (FP8Q_PT_FUSED_PDL && FP8Q_PDL) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na++].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, current_fused_kernel<DT, FMT, SL>, p);
}

// Resident CTAs per SM of current_fused_kernel<DT, FMT, SL> (SL == 2 with
// its shared-memory slice).
template <int DT, int FMT, int SL>
static int fused_per_sm() {
  int per_sm = 0;
  const size_t smem = SL == 2 ? (size_t)FusedChunk<DT>::kElems * (DT == kBF16 ? 2 : 4) : 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, current_fused_kernel<DT, FMT, SL>, kPtThreads, smem) !=
          cudaSuccess)
    per_sm = 0;
  return per_sm;
}

template <int DT, int FMT>
static cudaError_t launch_fused_t(const KParams& p, int64_t slices, cudaStream_t s, bool* taken) {
  static const int64_t cap1 = (int64_t)fused_per_sm<DT, FMT, 1>() * sm_count();
  static const int64_t cap2 = FP8Q_PT_FUSED_SLICES >= 2 ? (int64_t)fused_per_sm<DT, FMT, 2>() * sm_count() : 0;
  *taken = false;
  if (!FP8Q_PT_FUSED) return cudaSuccess;
  if (slices <= cap1) {
    *taken = true;
    KParams q = p;
    q.early_trigger = 2 * slices <= cap1;
    return launch_fused_sl<DT, FMT, 1>(q, slices, s);
  }
  if ((slices + 1) / 2 <= cap2) {
    *taken = true;
    return launch_fused_sl<DT, FMT, 2>(p, (slices + 1) / 2, s);
  }
  if (cap2 > 0 && slices <= (int64_t)FP8Q_PT_STREAM_MAX * 2 * cap2) {  // on-chip slices plus streamed chunks
    *taken = true;
    return launch_fused_sl<DT, FMT, 2>(p, cap2, s);
  }
  return cudaSuccess;
}

#ifndef FP8Q_PT_CLUSTER  // 1: tensors of up to 16 x 128 KB take the one-cluster kernel
#define FP8Q_PT_CLUSTER 1
#endif
// Whether current_cluster_kernel<DT, FMT> can be launched here (the cluster
// size is non-portable): attributes set once, then at least one cluster
// must fit.
template <int DT, int FMT>
static bool cluster_ready() {
  static const bool ok = [] {
    auto k = current_cluster_kernel<DT, FMT>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kClusterMaxBytes) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterCtas);
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = kClusterMaxBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    return n > 0;
  }();
  return ok;
}

template <int DT, int FMT>
static cudaError_t launch_cluster_t(const KParams& p, cudaStream_t s) {
  const int64_t share = (p.n / InT<DT>::kPerVec + kClusterCtas - 1) / kClusterCtas * 16;  // bytes per CTA, at most
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kClusterCtas);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = (size_t)share;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = FP8Q_PDL ? 2 : 1;
  KParams q = p;
  q.early_trigger = 1;
  return cudaLaunchKernelEx(&cfg, current_cluster_kernel<DT, FMT>, q);
}

fp8q_status launch_current_fused(const PtLaunch& L, bool* taken) {
  *taken = false;
  if (L.rows * L.cols == 0 || L.G != 1) return FP8Q_OK;
  KParams p = make_params(L);
  const int64_t n = p.n;
  cudaError_t e;
  const int64_t esz = L.dt == kBF16 ? 2 : 4;
  if (FP8Q_PT_CLUSTER && n * esz <= (int64_t)kClusterCtas * kClusterMaxBytes) {
    const bool ready = L.dt == kBF16 ? (L.fmt == kE4M3 ? cluster_ready<kBF16, kE4M3>() : cluster_ready<kBF16, kE5M2>())
                                     : (L.fmt == kE4M3 ? cluster_ready<kFP32, kE4M3>() : cluster_ready<kFP32, kE5M2>());
    if (ready) {
      *taken = true;
      if (L.dt == kBF16)
        e = L.fmt == kE4M3 ? launch_cluster_t<kBF16, kE4M3>(p, L.stream) : launch_cluster_t<kBF16, kE5M2>(p, L.stream);
      else
        e = L.fmt == kE4M3 ? launch_cluster_t<kFP32, kE4M3>(p, L.stream) : launch_cluster_t<kFP32, kE5M2>(p, L.stream);
      if (e != cudaSuccess) return cuda_fail(e, "current scaling cluster kernel launch");
      return check_launch("current scaling cluster kernel");
    }
  }
  if (L.dt == kBF16) {
    const int64_t c = (n + FusedChunk<kBF16>::kElems - 1) / FusedChunk<kBF16>::kElems;
    e = L.fmt == kE4M3 ? launch_fused_t<kBF16, kE4M3>(p, c, L.stream, taken)
                       : launch_fused_t<kBF16, kE5M2>(p, c, L.stream, taken);
  } else {
    const int64_t c = (n + FusedChunk<kFP32>::kElems - 1) / FusedChunk<kFP32>::kElems;
    e = L.fmt == kE4M3 ? launch_fused_t<kFP32, kE4M3>(p, c, L.stream, taken)
                       : launch_fused_t<kFP32, kE5M2>(p, c, L.stream, taken);
  }
  if (e != cudaSuccess) return cuda_fail(e, "current scaling kernel launch");
  return *taken ? check_launch("current scaling kernel") : FP8Q_OK;
}

fp8q_status launch_zero_words(void* p, size_t bytes, cudaStream_t s) {
  const int n = (int)(bytes / 4);
  if (n == 0) return FP8Q_OK;
  const int blocks = n < 64 * kPtThreads ? (n + kPtThreads - 1) / kPtThreads : 64;
  const cudaError_t e = launch_kernel(zero_words_kernel, dim3(blocks), dim3(kPtThreads), 0, s, (uint32_t*)p, n);
  if (e != cudaSuccess) return cuda_fail(e, "zeroing kernel launch");
  return check_launch("zeroing kernel");
}

fp8q_status launch_scale(const float* amax, int G, int fmt, int margin, float* scale_out, float* scale_inv_out,
                         cudaStream_t s) {
  const int blocks = (G + kPtThreads - 1) / kPtThreads;
  const cudaError_t e = launch_kernel(scale_kernel, dim3(blocks), dim3(kPtThreads), 0, s, amax, G, fmt_max(fmt),
                                      margin, scale_out, scale_inv_out);
  if (e != cudaSuccess) return cuda_fail(e, "scale kernel launch");
  return check_launch("scale kernel");
}

fp8q_status pt_device_status(bool clear, unsigned* word) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_pt_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (clear && v) {
    const unsigned z = 0;
    e = cudaMemcpyToSymbol(g_pt_error, &z, sizeof(z));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
  }
  *word = v;
  return FP8Q_OK;
}

fp8q_status pt_set_wait_budget(unsigned long long ns) {
  const cudaError_t e = cudaMemcpyToSymbol(g_pt_wait_budget_ns, &ns, sizeof(ns));
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, "cudaMemcpyToSymbol(wait budget)");
}

fp8q_status pt_set_stall_publish(bool on) {
  const unsigned v = on ? 1u : 0u;
  const cudaError_t e = cudaMemcpyToSymbol(g_pt_stall_publish, &v, sizeof(v));
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, "cudaMemcpyToSymbol(stall)");
}

}  // namespace fp8q
