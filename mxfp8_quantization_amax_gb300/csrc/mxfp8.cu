// mxfp8.cu -- MXFP8 quantization, rowwise and columnwise, in one HBM pass.
//
// "Blackwell GPU MXFP8 预训练最佳实践" 4.1: per block of 32 values,
// X = ceil(log2(amax / destmax)) saturated to the E8M0 range, elements
// RNE_sat(v / 2^X), amax = 0 -> X = -127 with all elements 0.  4.2 and
// "HiFloat8：高性能训练之路" 2: every tensor needs a copy quantized along
// rows and one along columns (transposed), both from the high-precision
// tensor ("混合精度与 FP8 训练" 13.1: MX does not commute with transposes).
//
// Geometry.  A block is 32 rows x 256 columns; its 32 rows are one
// columnwise MX block, so for ragged groups (MoE experts) blocks start at
// each group's first row and a group's last block may be shorter.  A unit
// is up to `super` consecutive blocks of one group in one 256-column strip.
// A shared-memory scan of the group sizes maps unit index -> (group, block).
//
// BF16 (the training path): a persistent, warp-specialised kernel.  One
// producer warp streams blocks into a ring of shared-memory stages with 2-D
// TMA loads (four 64-column boxes per block, 128-byte swizzle), each stage
// guarded by a "full" and an "empty" mbarrier; four consumer warps quantize:
//   * rowwise: one lane per 1x32 block (four 16-byte shared loads, one
//     E8M0 computation, one 32-byte store of the codes); the 8 lanes of a
//     quarter-warp read 8 rows of one block, distinct bank groups after the
//     swizzle;
//   * columnwise: thread t owns columns 2t and 2t+1 and reads one 32-bit
//     word (both columns) per row, so one packed abs-max gives both column
//     amaxes; each column's 32 codes leave as one 32-byte store into the
//     transposed output, and its scale bytes are gathered over the unit.
// FP32 inputs take a simpler kernel: loads into registers, rowwise pass from
// registers, the block staged in shared memory for the columnwise pass.
#include <cudaTypedefs.h>

#include <mutex>

#include "fp8q_device.cuh"
#include "internal.h"
#include "tma.cuh"

#ifndef FP8Q_MX_STAGES  // shared-memory ring depth (16 KB per stage)
#define FP8Q_MX_STAGES 2
#endif
#ifndef FP8Q_MX_SUPER  // 32-row blocks per unit of the BF16 kernel
#define FP8Q_MX_SUPER 4
#endif
#ifndef FP8Q_MX_SUPER_GROUPED  // the same for grouped calls (fewer unit boundaries inside a group)
#define FP8Q_MX_SUPER_GROUPED 16
#endif
#ifndef FP8Q_MX_MIN_CTAS  // CTAs per SM the register budget is sized for
#define FP8Q_MX_MIN_CTAS 4
#endif
#ifndef FP8Q_MX_SCOL_FLUSH  // scale bytes per s_col store (4 or 8)
#define FP8Q_MX_SCOL_FLUSH 4
#endif
#ifndef FP8Q_MX_HINTS  // L2 evict-first data stores, evict-last scale stores
#define FP8Q_MX_HINTS 1
#endif
#ifndef FP8Q_MX_SROW8  // one 8-byte s_row store per row and strip
#define FP8Q_MX_SROW8 1
#endif
#ifndef FP8Q_MX_LEAN_GRID_ALL  // lean kernel: one CTA per unit instead of a persistent grid
#define FP8Q_MX_LEAN_GRID_ALL 1
#endif
#ifndef FP8Q_MX_BAND_GRID_ALL  // band kernel: one CTA per unit instead of a persistent grid
#define FP8Q_MX_BAND_GRID_ALL 1
#endif
#ifndef FP8Q_MX_UNIT_BMUL  // packed BF16 scaling in the unit kernel too
#define FP8Q_MX_UNIT_BMUL 0
#endif

namespace fp8q {

constexpr int kTileRows = 32;
constexpr int kTileCols = 256;
constexpr int kConsumers = 128;  // 4 consumer warps
constexpr int kStageBytes = kTileRows * kTileCols * 2;  // one BF16 block: 16 KB
constexpr int kStages = FP8Q_MX_STAGES;
constexpr int kTmaThreads = kConsumers + 32;  // + one producer warp
constexpr int kSubCols = 64;                  // columns per TMA box (128 bytes)
constexpr int kSubBytes = kTileRows * 128;    // one box in shared memory

// Device-side failure word (bit 0: a bounded wait gave up) and the wait
// budget in ns.  Read and cleared by fp8q_check_device().
__device__ unsigned int g_mx_error;
// Failure-detection test hook: while nonzero, the BF16 kernel's producer
// issues no loads, so every consumer wait runs out its budget.
__device__ unsigned int g_mx_stall_producer;
__device__ unsigned long long g_wait_budget_ns = 1000000000ull;

struct MxParams {
  const void* x;
  int64_t rows, cols;
  const int64_t* off;  // device row offsets [G+1] or nullptr
  int G;
  int64_t strips;  // ceil(cols / 256)
  int super;       // blocks per unit
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t s_col_ld;
  int round_up;              // scale rule: 1 round-up (default), 0 OCP round-down
  unsigned long long* sat;   // saturated-element counts [row, col], or nullptr
  // scale layout: 0 row-major ([rows][cols/32], [cols][s_col_ld]); 1 the
  // 128 x 4 blocks of block-scaled MMA, with row_bcols / col_bcols blocks
  // per block row (ceil(cols/32 / 4), ceil(s_col_ld / 4))
  int mma;
  int64_t row_bcols, col_bcols;
};

// Byte of scale (r, c) in the 128 x 4 block layout: blocks of 128 scale
// rows x 4 scale columns (512 bytes) stored block row by block row, and in
// a block (r, c) at (r % 32) * 16 + (r / 32 % 4) * 4 + c % 4.
__device__ __forceinline__ int64_t mma_off(int64_t r, int64_t c, int64_t bcols) {
  return ((r >> 7) * bcols + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// Where column c's scale of block gb goes: the aligned window holding it
// (8 bytes of a row-major s_col row, or one 4-byte row of an MMA block), the
// byte's place `q` in that window and the block index of the window's first
// byte.  Consecutive blocks of a column fill a window from q = 0 to W - 1.
struct ScaleSlot {
  uint8_t* win;
  int q;
  int64_t gbw;
};
template <bool MMA>
__device__ __forceinline__ ScaleSlot col_scale_slot(const MxParams& p, int64_t c, int64_t gb) {
  ScaleSlot sl;
  if constexpr (MMA) {
    sl.q = (int)(gb & 3);
    sl.gbw = gb - sl.q;
    sl.win = p.s_col + mma_off(c, sl.gbw, p.col_bcols);
  } else {
    uint8_t* d = p.s_col + c * p.s_col_ld + gb;
    sl.q = (int)((uintptr_t)d & 7u);
    sl.gbw = gb - sl.q;
    sl.win = d - sl.q;
  }
  return sl;
}
template <bool MMA>
__device__ __forceinline__ constexpr int col_scale_window() { return MMA ? 4 : 8; }
// The row-major slot of the scale at d (block gb of its column).
__device__ __forceinline__ ScaleSlot scale_slot_at(uint8_t* d, int64_t gb) {
  ScaleSlot sl;
  sl.q = (int)((uintptr_t)d & 7u);
  sl.gbw = gb - sl.q;
  sl.win = d - sl.q;
  return sl;
}

// Clamped group boundary: offsets outside [0, rows] are pulled back in, so
// blocks never leave the tensor whatever the caller passes.
__device__ __forceinline__ int64_t grp_row(const MxParams& p, int g) {
  if (p.off == nullptr) return g == 0 ? 0 : p.rows;
  int64_t v = __ldg(p.off + g);
  return v < 0 ? 0 : (v > p.rows ? p.rows : v);
}

// ---------------------------------------------------------------------------
// Units and blocks
// ---------------------------------------------------------------------------
// blk[g] = sum_{h<g} ceil(n_h / 32), sup[g] = sum_{h<g} ceil(ceil(n_h / 32) / super),
// for g = 0..G (block-wide scan; ends with __syncthreads).
template <int NT>
__device__ void build_prefix(const MxParams& p, int* blk, int* sup) {
  __shared__ int tot_b[NT / 32], tot_s[NT / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (p.G + NT - 1) / NT;
  const int g_lo = tid * per, g_hi = min(p.G, g_lo + per);
  auto nblocks = [&](int g) {
    const int64_t n = grp_row(p, g + 1) - grp_row(p, g);
    return n > 0 ? (int)((n + 31) / 32) : 0;
  };
  int sb = 0, ss = 0;
  for (int g = g_lo; g < g_hi; g++) {
    const int nb = nblocks(g);
    sb += nb;
    ss += (nb + p.super - 1) / p.super;
  }
  int ib = sb, is = ss;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int vb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
    const int vs = __shfl_up_sync(0xFFFFFFFFu, is, o);
    if (lane >= o) {
      ib += vb;
      is += vs;
    }
  }
  if (lane == 31) {
    tot_b[warp] = ib;
    tot_s[warp] = is;
  }
  __syncthreads();
  int bb = 0, bs = 0;
  for (int w = 0; w < warp; w++) {
    bb += tot_b[w];
    bs += tot_s[w];
  }
  int rb = bb + ib - sb, rs = bs + is - ss;
  for (int g = g_lo; g < g_hi; g++) {
    blk[g] = rb;
    sup[g] = rs;
    const int nb = nblocks(g);
    rb += nb;
    rs += (nb + p.super - 1) / p.super;
  }
  if (tid == NT - 1) {
    blk[p.G] = bb + ib;
    sup[p.G] = bs + is;
  }
  __syncthreads();
}

struct Unit {
  int g;
  int nblk;          // blocks in this unit (1..super)
  int64_t rg1;       // end row of the group
  int64_t r_first;   // first row of the unit
  int64_t gb0;       // s_col index of the unit's first block
  int64_t c0;        // first column
  int nc;            // columns in the strip (multiple of 32)
};

struct Tile {
  int64_t r0;  // first row of the window
  int lo;      // window rows [lo, nr) are this CTA's rows
  int nr;      // end of those rows (1..32)
  int64_t c0;
  int nc;
};

__device__ __forceinline__ Unit unit_of(const MxParams& p, const int* blk, const int* sup, int64_t u) {
  Unit t;
  const int ti = (int)(u / p.strips);
  t.c0 = (u - (int64_t)ti * p.strips) * kTileCols;
  t.nc = (int)min((int64_t)kTileCols, p.cols - t.c0);
  int lo = 0, hi = p.G;  // last g with sup[g] <= ti
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sup[mid] <= ti) lo = mid; else hi = mid;
  }
  t.g = lo;
  const int b0 = p.super * (ti - sup[lo]);
  t.nblk = min(p.super, blk[lo + 1] - blk[lo] - b0);
  t.rg1 = grp_row(p, lo + 1);
  t.r_first = grp_row(p, lo) + 32LL * b0;
  t.gb0 = blk[lo] + b0;
  return t;
}

__device__ __forceinline__ Tile block_of(const Unit& U, int j) {
  Tile t;
  t.r0 = U.r_first + 32LL * j;
  t.lo = 0;
  t.nr = (int)min((int64_t)kTileRows, U.rg1 - t.r0);
  t.c0 = U.c0;
  t.nc = U.nc;
  return t;
}

// ---------------------------------------------------------------------------
// Stores
// ---------------------------------------------------------------------------
struct StorePolicy {
  uint64_t data, scale;
};

__device__ __forceinline__ StorePolicy make_policy() {
  StorePolicy sp{0, 0};
#if FP8Q_MX_HINTS
  sp.data = policy_evict_first();
  sp.scale = policy_evict_last();
#endif
  return sp;
}

__device__ __forceinline__ void st_data32(void* p, const uint32_t (&d)[8], const StorePolicy& sp) {
#if FP8Q_MX_HINTS
  st32B_hint(p, d, sp.data);
#else
  (void)sp;
  st32B(p, d);
#endif
}
__device__ __forceinline__ void st_scale8(uint8_t* p, uint32_t v, const StorePolicy& sp) {
#if FP8Q_MX_HINTS
  st_u8_hint(p, v, sp.scale);
#else
  (void)sp;
  *p = (uint8_t)v;
#endif
}
__device__ __forceinline__ void st_scale32(uint8_t* p, uint32_t v, const StorePolicy& sp) {
#if FP8Q_MX_HINTS
  st_u32_hint(p, v, sp.scale);
#else
  (void)sp;
  *(uint32_t*)p = v;
#endif
}
__device__ __forceinline__ void st_scale64(uint8_t* p, uint64_t v, const StorePolicy& sp) {
#if FP8Q_MX_HINTS
  st_u64_hint(p, v, sp.scale);
#else
  (void)sp;
  *(uint64_t*)p = v;
#endif
}

// First n (<= 32) bytes of d[0..7] to dst, at any alignment.
__device__ __forceinline__ void store_col32(uint8_t* dst, const uint32_t (&d)[8], int n, const StorePolicy& sp) {
  const uintptr_t a = (uintptr_t)dst;
  if (n == 32 && (a & 31u) == 0) {
    st_data32(dst, d, sp);
    return;
  }
  if (n == 32 && (a & 15u) == 0) {
    st_stream(dst, make_uint4(d[0], d[1], d[2], d[3]));
    st_stream(dst + 16, make_uint4(d[4], d[5], d[6], d[7]));
    return;
  }
  const int mis = (int)(a & 3u);
  uint8_t* base = dst - mis;
#pragma unroll
  for (int k = 0; k <= 8; k++) {
    const uint32_t lo = k > 0 ? d[k - 1] : 0u;
    const uint32_t hi = k < 8 ? d[k] : 0u;
    const uint32_t w = mis ? __funnelshift_r(lo, hi, 8 * (4 - mis)) : hi;
    const int s = 4 * k - mis;  // index of this word's first byte in the column run
    // partial sectors are completed by another unit: keep them in L2 until then
    if (s >= 0 && s + 4 <= n) {
      st_scale32(base + 4 * k, w, sp);
    } else {
#pragma unroll
      for (int i = 0; i < 4; i++)
        if (s + i >= 0 && s + i < n) st_scale8(base + 4 * k + i, w >> (8 * i), sp);
    }
  }
}

// ---------------------------------------------------------------------------
// Byte ranges of an aligned window as naturally aligned chunks.  The range
// bounds are compile-time, so every chunk reads registers at static
// indices; run-time bounds dispatch through a switch (they are the same for
// every column of a unit, so the branch is uniform).
// ---------------------------------------------------------------------------
template <int POS, int SZ>
__device__ __forceinline__ void store_chunk(uint8_t* base, const uint32_t (&o)[8], uint64_t pol) {
  uint8_t* p = base + POS;
  if constexpr (SZ == 16) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(o[POS / 4]),
                 "r"(o[POS / 4 + 1]), "r"(o[POS / 4 + 2]), "r"(o[POS / 4 + 3]), "l"(pol)
                 : "memory");
  } else if constexpr (SZ == 8) {
    asm volatile("st.global.L2::cache_hint.v2.b32 [%0], {%1,%2}, %3;" ::"l"(p), "r"(o[POS / 4]), "r"(o[POS / 4 + 1]),
                 "l"(pol)
                 : "memory");
  } else if constexpr (SZ == 4) {
    st_u32_hint(p, o[POS / 4], pol);
  } else if constexpr (SZ == 2) {
    st_u16_hint(p, o[POS / 4] >> (8 * (POS % 4)), pol);
  } else {
    st_u8_hint(p, o[POS / 4] >> (8 * (POS % 4)), pol);
  }
}

__host__ __device__ constexpr int chunk_for(int from, int to) {
  int sz = 16;
  while (sz > 1 && (from % sz != 0 || from + sz > to)) sz >>= 1;
  return sz;
}

template <int FROM, int TO>
__device__ __forceinline__ void store_range(uint8_t* base, const uint32_t (&o)[8], uint64_t pol) {
  if constexpr (FROM < TO) {
    constexpr int SZ = chunk_for(FROM, TO);
    store_chunk<FROM, SZ>(base, o, pol);
    store_range<FROM + SZ, TO>(base, o, pol);
  }
}

// bytes [from, 32) of the 32-byte aligned window at base (from in 1..31)
template <int F = 1>
__device__ __forceinline__ void store_suffix32(uint8_t* base, const uint32_t (&o)[8], int from, uint64_t pol) {
  if constexpr (F < 32) {
    if (from == F) store_range<F, 32>(base, o, pol);
    else store_suffix32<F + 1>(base, o, from, pol);
  }
}
// bytes [0, to) of the 32-byte aligned window at base (to in 1..31)
template <int T = 1>
__device__ __forceinline__ void store_prefix32(uint8_t* base, const uint32_t (&o)[8], int to, uint64_t pol) {
  if constexpr (T < 32) {
    if (to == T) store_range<0, T>(base, o, pol);
    else store_prefix32<T + 1>(base, o, to, pol);
  }
}
// bytes [from, 8) of the 8-byte aligned window at base (from in 0..7)
template <int F = 0>
__device__ __forceinline__ void store_suffix8(uint8_t* base, const uint32_t (&o)[8], int from, uint64_t pol) {
  if constexpr (F < 8) {
    if (from == F) store_range<F, 8>(base, o, pol);
    else store_suffix8<F + 1>(base, o, from, pol);
  }
}
// bytes [from, to) of the 8-byte aligned window at base (0 <= from < to <= 8)
template <int F, int T = F + 1>
__device__ __forceinline__ void store_range8_to(uint8_t* base, const uint32_t (&o)[8], int to, uint64_t pol) {
  if constexpr (T <= 8) {
    if (to == T) store_range<F, T>(base, o, pol);
    else store_range8_to<F, T + 1>(base, o, to, pol);
  }
}
template <int F = 0>
__device__ __forceinline__ void store_range8(uint8_t* base, const uint32_t (&o)[8], int from, int to, uint64_t pol) {
  if constexpr (F < 8) {
    if (from == F) store_range8_to<F>(base, o, to, pol);
    else store_range8<F + 1>(base, o, from, to, pol);
  }
}

// Scale bytes of column c for blocks gb0 .. gb0+n-1 (byte j of v).
__device__ __forceinline__ void store_scales(const MxParams& p, int64_t c, int64_t gb0, int n, uint64_t v,
                                             const StorePolicy& sp) {
  uint8_t* dst = p.s_col + c * p.s_col_ld + gb0;
  if (n == 8 && gb0 + 8 <= p.s_col_ld && ((uintptr_t)dst & 7u) == 0) {
    st_scale64(dst, v, sp);
    return;
  }
  if (n == 4 && gb0 + 4 <= p.s_col_ld && ((uintptr_t)dst & 3u) == 0) {
    st_scale32(dst, (uint32_t)v, sp);
    return;
  }
  for (int j = 0; j < n; j++)
    if (gb0 + j < p.s_col_ld) st_scale8(dst + j, (uint32_t)(v >> (8 * j)), sp);
}

// Scale bytes [from, to) of the 8-byte aligned window at `win`, whose first
// byte is s_col block index `gbw` of its column (blocks past s_col_ld are
// not written).
__device__ __forceinline__ void flush_scales8(const MxParams& p, uint8_t* win, int from, int to, int64_t gbw,
                                              uint64_t v, const StorePolicy& sp) {
  if (gbw + to > p.s_col_ld) to = (int)(p.s_col_ld - gbw);
  if (gbw + from < 0) from = (int)-gbw;  // window bytes before the column's first scale
  if (from >= to) return;
  const uint32_t o[8] = {(uint32_t)v, (uint32_t)(v >> 32), 0, 0, 0, 0, 0, 0};
  store_range8(win, o, from, to, sp.scale);
}

// ---------------------------------------------------------------------------
// Element conversion
// ---------------------------------------------------------------------------
// The two BF16 values of word w scaled by (m_lo, m_hi) with one packed
// multiply, as two floats ready for the packed conversion.
#ifndef FP8Q_MX_MUL2  // packed f32x2 multiply (1) or two scalar multiplies (0)
#define FP8Q_MX_MUL2 1
#endif
__device__ __forceinline__ void scale_pair(uint32_t w, float m_lo, float m_hi, float& lo, float& hi) {
#if FP8Q_MX_MUL2
  lo = bf16_lo(w);
  hi = bf16_hi(w);
  mul2(lo, hi, m_lo, m_hi);
#else
  lo = __fmul_rn(bf16_lo(w), m_lo);
  hi = __fmul_rn(bf16_hi(w), m_hi);
#endif
}

// BF16 packed multiply by a power of two.  x * 2^-X is exact in BF16
// whenever the result is a normal number, and every result that is not
// (below 2^-126) is far under half the smallest FP8 subnormal, so it
// converts to the same (signed) zero code as the exact FP32 product.  It
// replaces the unpack, pack and FP32 packed multiply of two elements by one
// packed BF16 multiply and the unpack, a cut in ALU work that pays in the
// grouped kernel (whose phase shifts load the ALU), not in the ungrouped
// one (measured: 395 -> 359 us and 339 -> 344 us on 65536 x 7168).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t w, uint32_t m) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(m));
  return r;
}
// The BF16 bits of an E8M0 multiplier (2^-127 is the BF16 subnormal 0x0040).
__device__ __forceinline__ uint32_t bf16_of_multiplier(float mult) { return __float_as_uint(mult) >> 16; }

template <int FMT, bool BMUL>
__device__ __forceinline__ uint32_t row_codes4(uint32_t w0, uint32_t w1, float mult) {
  if constexpr (BMUL) {
    const uint32_t m = bf16_of_multiplier(mult) * 0x10001u;
    const uint32_t p0 = mul_bf16x2(w0, m), p1 = mul_bf16x2(w1, m);
    return cvt4<FMT>(bf16_lo(p0), bf16_hi(p0), bf16_lo(p1), bf16_hi(p1));
  } else {
    float a, b, c, d;
    scale_pair(w0, mult, mult, a, b);
    scale_pair(w1, mult, mult, c, d);
    return cvt4<FMT>(a, b, c, d);
  }
}

template <int FMT>
__device__ __forceinline__ uint32_t mx_codes4(float a, float b, float c, float d, float mult) {
  return cvt4<FMT>(__fmul_rn(a, mult), __fmul_rn(b, mult), __fmul_rn(c, mult), __fmul_rn(d, mult));
}

// Elements of a BF16 pair whose scaled magnitude exceeds the format maximum
// (they clamp; only possible when the scale rule rounds X down).
template <int FMT>
__device__ __forceinline__ uint32_t sat_pair(uint32_t w, float m_lo, float m_hi) {
  constexpr float kMax = Fmt<FMT>::kMax;
  return (uint32_t)(fabsf(bf16_lo(w)) * m_lo > kMax) + (uint32_t)(fabsf(bf16_hi(w)) * m_hi > kMax);
}

// True when a finite, nonzero block's amax scaled by mult exceeds the
// format maximum (then its elements are counted one by one).
template <int FMT>
__device__ __forceinline__ bool block_saturates(uint32_t amax_bits, uint32_t byte, float mult) {
  return byte != 0xFFu && amax_bits != 0u && __uint_as_float(amax_bits) * mult > Fmt<FMT>::kMax;
}

// Final code word of a block: Inf/NaN block -> 0x7F codes, zero block -> 0.
__device__ __forceinline__ uint32_t mx_fix(uint32_t w, uint32_t byte, uint32_t amax_bits) {
  w = byte == 0xFFu ? 0x7F7F7F7Fu : w;
  return amax_bits == 0u ? 0u : w;
}

// ---------------------------------------------------------------------------
// BF16: TMA-fed, warp-specialised persistent kernel
// ---------------------------------------------------------------------------
// Stage layout: four 64-column boxes of 32 rows x 128 B, each written by one
// TMA load with the 128-byte swizzle: 16-byte chunk c of row r sits at chunk
// c ^ (r % 8).  Logical byte b of row r is therefore at
//   (b / 128) * 4096 + r * 128 + (((b % 128) / 16) ^ (r % 8)) * 16 + b % 16.

// Rowwise, one lane per 1x32 block: row r, block b (of the 8 in the strip).
// Writes the 32 codes; returns the scale byte (0 if the block is not ours).
template <int FMT, bool EXT, bool BMUL>
__device__ __forceinline__ uint32_t row_block_bf16(const MxParams& p, const Tile& t, const unsigned char* stage,
                                                   int r, int b, const StorePolicy& sp, uint32_t& nsat) {
  if (r < t.lo || r >= t.nr || 32 * b >= t.nc) return 0u;
  const unsigned char* line = stage + (b >> 1) * kSubBytes + r * 128;
  const int c0 = (b & 1) * 4;
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const uint4 v = *(const uint4*)(line + (((c0 + j) ^ (r & 7)) << 4));
    w[4 * j] = v.x;
    w[4 * j + 1] = v.y;
    w[4 * j + 2] = v.z;
    w[4 * j + 3] = v.w;
  }
  uint32_t m4[4];
#pragma unroll
  for (int j = 0; j < 4; j++)
    m4[j] = absmax_nan_bf16x2(absmax_nan_bf16x2(w[4 * j], w[4 * j + 1]), absmax_nan_bf16x2(w[4 * j + 2], w[4 * j + 3]));
  const uint32_t m = absmax_nan_bf16x2(absmax_nan_bf16x2(m4[0], m4[1]), absmax_nan_bf16x2(m4[2], m4[3]));
  const uint32_t am = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu) << 16;
  const uint32_t byte = e8m0_from_amax<FMT>(am, EXT ? p.round_up : 1);
  uint32_t d[8];
  if (byte == 0xFFu || am == 0u) {  // Inf/NaN block: 0x7F codes; zero block: +0 codes
    const uint32_t fill = am == 0u ? 0u : 0x7F7F7F7Fu;
#pragma unroll
    for (int k = 0; k < 8; k++) d[k] = fill;
  } else {
    const float mult = e8m0_multiplier(byte);
#pragma unroll
    for (int k = 0; k < 8; k++) d[k] = row_codes4<FMT, BMUL>(w[2 * k], w[2 * k + 1], mult);
    if constexpr (EXT) {
      if (p.sat != nullptr && block_saturates<FMT>(am, byte, mult)) {
#pragma unroll
        for (int k = 0; k < 16; k++) nsat += sat_pair<FMT>(w[k], mult, mult);
      }
    }
  }
  st_data32(p.q_row + (t.r0 + r) * p.cols + t.c0 + 32 * b, d, sp);
  return byte;
}

// s_row bytes of one warp's 8 rows: lane l holds row 8w + l % 8, blocks
// l / 8 (byte0) and 4 + l / 8 (byte1).  All 32 lanes must call.
template <bool MMA>
__device__ __forceinline__ void store_row_scales(const MxParams& p, const Tile& t, int warp, int lane,
                                                 uint32_t byte0, uint32_t byte1, const StorePolicy& sp) {
  const int r = 8 * warp + (lane & 7);
  const int64_t sld = p.cols / 32;
  uint8_t* dst = p.s_row + (t.r0 + r) * sld + t.c0 / 32;
#if FP8Q_MX_SROW8
  // gather the row's 8 bytes into lane r % 8 and store them at once
  const uint32_t v = byte0 | (byte1 << 8);
  const uint32_t v1 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 8);
  const uint32_t v2 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 16);
  const uint32_t v3 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 24);
  if (r < t.lo || r >= t.nr) return;
  if constexpr (MMA) {  // two 4-byte rows of MMA blocks: scale columns sc .. sc + 3 and sc + 4 .. sc + 7
    if (lane < 8) {
      const uint32_t lo = (v & 0xFFu) | ((v1 & 0xFFu) << 8) | ((v2 & 0xFFu) << 16) | ((v3 & 0xFFu) << 24);
      const uint32_t hi = (v >> 8) | ((v1 >> 8) << 8) | ((v2 >> 8) << 16) | ((v3 >> 8) << 24);
      const int64_t row = t.r0 + r, sc = t.c0 / 32;
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int64_t c = sc + 4 * h;
        const int64_t nvalid = min((int64_t)4, sld - c);
        if (nvalid <= 0) break;
        uint8_t* d = p.s_row + mma_off(row, c, p.row_bcols);
        const uint32_t w = h ? hi : lo;
        if (nvalid == 4) {
          st_scale32(d, w, sp);
        } else {
          for (int i = 0; i < nvalid; i++) st_scale8(d + i, w >> (8 * i), sp);
        }
      }
    }
    return;
  }
  if (t.nc == kTileCols && ((uintptr_t)dst & 7u) == 0) {
    if (lane < 8) {
      const uint64_t lo = (v & 0xFFu) | ((v1 & 0xFFu) << 8) | ((v2 & 0xFFu) << 16) | ((v3 & 0xFFu) << 24);
      const uint64_t hi = (v >> 8) | ((v1 >> 8) << 8) | ((v2 >> 8) << 16) | ((v3 >> 8) << 24);
      st_scale64(dst, lo | (hi << 32), sp);
    }
    return;
  }
#endif
  if (r >= t.lo && r < t.nr) {  // one byte per block
    const int b = lane >> 3;
    if (32 * b < t.nc) st_scale8(dst + b, byte0, sp);
    if (32 * (b + 4) < t.nc) st_scale8(dst + b + 4, byte1, sp);
  }
}

// The 32 bytes starting `off` bytes into the 64-byte concatenation a ++ b
// (0 < off < 32), for an offset known only at run time.
__device__ __forceinline__ void window32(const uint32_t (&a)[8], const uint32_t (&b)[8], int off, uint32_t (&o)[8]) {
  const int sh = 8 * (off & 3);
  uint32_t c[16];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    c[i] = a[i];
    c[8 + i] = b[i];
  }
  switch (off >> 2) {  // whole words; each case indexes registers statically
#define FP8Q_WINDOW_CASE(Q)                                                              \
  case Q:                                                                                \
    _Pragma("unroll") for (int i = 0; i < 8; i++) o[i] =                                 \
        __funnelshift_r(c[Q + i], (Q + i + 1 < 16 ? c[Q + i + 1] : 0u), sh); /* sh 0: c[Q+i] */ \
    break;
    FP8Q_WINDOW_CASE(0)
    FP8Q_WINDOW_CASE(1)
    FP8Q_WINDOW_CASE(2)
    FP8Q_WINDOW_CASE(3)
    FP8Q_WINDOW_CASE(4)
    FP8Q_WINDOW_CASE(5)
    FP8Q_WINDOW_CASE(6)
    default:
    FP8Q_WINDOW_CASE(7)
#undef FP8Q_WINDOW_CASE
  }
}

// Columnwise output of one column, block j of a unit whose codes form one
// run of `len` bytes starting at `run` (any alignment).  Every block of the
// run has the same offset `mis` inside its 32-byte sector, so after block j
// the sector holding the tail of block j-1 and the head of block j is
// complete and leaves with one 32-byte store; only the two ends of the run
// are partial.  `prev` carries block j-1's codes.
__device__ __forceinline__ void emit_col_block(uint8_t* run, int len, int j, int nblk, const uint32_t (&d)[8],
                                               uint32_t (&prev)[8], const StorePolicy& sp) {
  const int mis = (int)((uintptr_t)run & 31u);
  const int lo = 32 * j;  // run bytes of this block: [lo, lo + 32)
  if (mis == 0) {
    store_col32(run + lo, d, min(32, len - lo), sp);
    return;
  }
  const uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (j == 0) {
    // head: run bytes [0, 32 - mis) fill window bytes [mis, 32) of the first sector
    uint32_t o[8];
    window32(z, d, 32 - mis, o);
    if (len >= 32 - mis) store_suffix32(run - mis, o, mis, sp.scale);
    else store_col32(run, d, len, sp);  // the whole run ends inside the first sector
  } else {
    uint32_t o[8];
    window32(prev, d, 32 - mis, o);  // run bytes [lo - mis, lo + 32 - mis)
    store_col32(run + lo - mis, o, min(32, len - (lo - mis)), sp);
  }
  if (j == nblk - 1 && len > lo + 32 - mis) {  // tail after the last sector boundary
    uint32_t o[8];
    window32(d, z, 32 - mis, o);
    const int n = len - (lo + 32 - mis);  // 1 .. mis bytes
    store_prefix32(run + lo + 32 - mis, o, n, sp.scale);
  }
#pragma unroll
  for (int i = 0; i < 8; i++) prev[i] = d[i];
}

// Columnwise: thread t owns columns 2t, 2t+1 (one 32-bit word per row) of
// the block in window rows [0, t.nr).  Writes the two columns' 32 codes to
// d0 / d1 and returns the two scale bytes (column 2t in bits 0-7).
// Saturated elements are counted over window rows [sat_lo, sat_hi).
template <int FMT, bool EXT, bool BMUL>
__device__ __forceinline__ uint32_t col_codes_bf16(const MxParams& p, const Tile& t, const unsigned char* stage,
                                                   int tid, uint32_t (&d0)[8], uint32_t (&d1)[8], uint32_t& nsat,
                                                   int sat_lo, int sat_hi) {
  const unsigned char* seg = stage + (tid >> 5) * kSubBytes + 4 * (tid & 3);
  const int c = (tid & 31) >> 2;  // 16-byte chunk of the word within the 128-byte line
  uint32_t off[8];
#pragma unroll
  for (int k = 0; k < 8; k++) off[k] = (uint32_t)((c ^ k) << 4);
  uint32_t w[kTileRows];
  if (t.nr == kTileRows) {
#pragma unroll
    for (int r = 0; r < kTileRows; r++) w[r] = *(const uint32_t*)(seg + r * 128 + off[r & 7]);
  } else {
#pragma unroll
    for (int r = 0; r < kTileRows; r++) w[r] = r < t.nr ? *(const uint32_t*)(seg + r * 128 + off[r & 7]) : 0u;
  }
  uint32_t m8[8];
#pragma unroll
  for (int k = 0; k < 8; k++)
    m8[k] = absmax_nan_bf16x2(absmax_nan_bf16x2(w[4 * k], w[4 * k + 1]), absmax_nan_bf16x2(w[4 * k + 2], w[4 * k + 3]));
  const uint32_t m = absmax_nan_bf16x2(absmax_nan_bf16x2(absmax_nan_bf16x2(m8[0], m8[1]), absmax_nan_bf16x2(m8[2], m8[3])),
                                       absmax_nan_bf16x2(absmax_nan_bf16x2(m8[4], m8[5]), absmax_nan_bf16x2(m8[6], m8[7])));
  const uint32_t a0 = (m & 0x7FFFu) << 16, a1 = m & 0x7FFF0000u;
  const int up = EXT ? p.round_up : 1;
  const uint32_t b0 = e8m0_from_amax<FMT>(a0, up), b1 = e8m0_from_amax<FMT>(a1, up);
  const float m0 = e8m0_multiplier(b0), m1 = e8m0_multiplier(b1);
  if constexpr (EXT) {
    if (p.sat != nullptr) {
      const bool s0 = block_saturates<FMT>(a0, b0, m0), s1 = block_saturates<FMT>(a1, b1, m1);
      if (s0 || s1) {
#pragma unroll
        for (int r = 0; r < kTileRows; r++)
          if (r >= sat_lo && r < sat_hi) nsat += sat_pair<FMT>(w[r], s0 ? m0 : 0.0f, s1 ? m1 : 0.0f);
      }
    }
  }
  const uint32_t mw = bf16_of_multiplier(m0) | (bf16_of_multiplier(m1) << 16);
#define FP8Q_COL_PAIR(i)                                   \
  if constexpr (BMUL) {                                    \
    const uint32_t pw = mul_bf16x2(w[4 * k + i], mw);      \
    l[i] = bf16_lo(pw);                                    \
    h[i] = bf16_hi(pw);                                    \
  } else {                                                 \
    scale_pair(w[4 * k + i], m0, m1, l[i], h[i]);          \
  }
  if (b0 == 0xFFu || a0 == 0u || b1 == 0xFFu || a1 == 0u) {
#pragma unroll
    for (int k = 0; k < 8; k++) {
      float l[4], h[4];
      FP8Q_COL_PAIR(0) FP8Q_COL_PAIR(1) FP8Q_COL_PAIR(2) FP8Q_COL_PAIR(3)
      d0[k] = mx_fix(cvt4<FMT>(l[0], l[1], l[2], l[3]), b0, a0);
      d1[k] = mx_fix(cvt4<FMT>(h[0], h[1], h[2], h[3]), b1, a1);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; k++) {
      float l[4], h[4];
      FP8Q_COL_PAIR(0) FP8Q_COL_PAIR(1) FP8Q_COL_PAIR(2) FP8Q_COL_PAIR(3)
      d0[k] = cvt4<FMT>(l[0], l[1], l[2], l[3]);
      d1[k] = cvt4<FMT>(h[0], h[1], h[2], h[3]);
    }
  }
#undef FP8Q_COL_PAIR
  return b0 | (b1 << 8);
}

// The unit-based kernel's column pass: codes of block j of unit U, written
// into the unit's run of the transposed output.
template <int FMT, bool EXT>
__device__ __forceinline__ uint32_t col_pair_bf16(const MxParams& p, const Unit& U, const Tile& t,
                                                  const unsigned char* stage, int tid, const StorePolicy& sp, int j,
                                                  uint32_t (&prev0)[8], uint32_t (&prev1)[8], uint32_t& nsat) {
  uint32_t d0[8], d1[8];
  const uint32_t b = col_codes_bf16<FMT, EXT, FP8Q_MX_UNIT_BMUL>(p, t, stage, tid, d0, d1, nsat, 0, kTileRows);
  const int64_t col = t.c0 + 2 * tid;
  const int len = (int)min((int64_t)(32 * U.nblk), U.rg1 - U.r_first);
  emit_col_block(p.q_col + col * p.rows + U.r_first, len, j, U.nblk, d0, prev0, sp);
  emit_col_block(p.q_col + (col + 1) * p.rows + U.r_first, len, j, U.nblk, d1, prev1, sp);
  return b;
}

// EXT: the scale rule and saturation counting of mxfp8_quantize_rule; the
// plain instantiation (round-up rule, no counting) carries none of that code.
// MMA: scales in the 128 x 4 block layout of block-scaled MMA (a template
// parameter, so the row-major instantiations carry none of its code).
template <int FMT, int DIR, bool EXT, bool MMA>
__global__ void __launch_bounds__(kTmaThreads, FP8Q_MX_MIN_CTAS) mx_tma_kernel(const __grid_constant__ CUtensorMap tmap, MxParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ volatile int abort_flag;
  // stages start on a 1 KB boundary (required by the 128-byte swizzle)
  unsigned char* stages = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  int* blk = (int*)(stages + kStages * kStageBytes);
  int* sup = blk + (p.G + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (tid == kConsumers) prefetch_tensormap(&tmap);
  pdl_wait();
  build_prefix<kTmaThreads>(p, blk, sup);
  const int64_t units = (int64_t)sup[p.G] * p.strips;
  const uint64_t budget = g_wait_budget_ns;

  if (warp == kConsumers / 32) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    int64_t k = 0;
    const bool stall = *(volatile unsigned*)&g_mx_stall_producer != 0;
    for (int64_t u = blockIdx.x; u < units && !abort_flag && !stall; u += gridDim.x) {
      const Unit U = unit_of(p, blk, sup, u);
      for (int j = 0; j < U.nblk; j++, ++k) {
        const int s = (int)(k % kStages);
        const uint32_t round = (uint32_t)(k / kStages);
        if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1u, budget)) {
          atomicOr(&g_mx_error, 1u);
          abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        unsigned char* dst = stages + s * kStageBytes;
        const int row = (int)(U.r_first + 32 * j);
#pragma unroll
        for (int q = 0; q < kTileCols / kSubCols; q++)
          tma_load_2d(dst + q * kSubBytes, &tmap, (int)U.c0 + q * kSubCols, row, &full[s]);
      }
    }
    pdl_launch_dependents();  // all loads issued: the next kernel may launch
    // every issued copy lands before the CTA can exit (fixed 2 s bound)
    const int64_t first = k > kStages ? k - kStages : 0;
    for (int64_t j = first; j < k; j++)
      mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1), 2000000000ull);
    return;
  }

  // ---------------- consumers ----------------
  const StorePolicy sp = make_policy();
  uint32_t nsat_r = 0, nsat_c = 0;  // saturated elements (counted when p.sat is set)
  int64_t k = 0;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const Unit U = unit_of(p, blk, sup, u);
    uint64_t sc0 = 0, sc1 = 0;  // scale bytes of this thread's two columns
    uint32_t prev0[8], prev1[8];  // previous block's column codes (sector carry)
    bool gave_up = false;
    for (int j = 0; j < U.nblk; j++, ++k) {
      const int s = (int)(k % kStages);
      const uint32_t round = (uint32_t)(k / kStages);
      // every lane waits; the warp acts on one voted answer so it never splits
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], round & 1u, budget))) {
        atomicOr(&g_mx_error, 1u);
        abort_flag = 1;
        gave_up = true;
        break;
      }
      const Tile t = block_of(U, j);
      const unsigned char* stage = stages + s * kStageBytes;
      if constexpr (DIR & MXFP8_ROW) {
        const int r = 8 * warp + (lane & 7);
        const uint32_t y0 = row_block_bf16<FMT, EXT, FP8Q_MX_UNIT_BMUL>(p, t, stage, r, lane >> 3, sp, nsat_r);
        const uint32_t y1 = row_block_bf16<FMT, EXT, FP8Q_MX_UNIT_BMUL>(p, t, stage, r, 4 + (lane >> 3), sp, nsat_r);
        store_row_scales<MMA>(p, t, warp, lane, y0, y1, sp);
      }
      if constexpr (DIR & MXFP8_COL) {
        if (2 * tid < t.nc) {
          const uint32_t b = col_pair_bf16<FMT, EXT>(p, U, t, stage, tid, sp, j, prev0, prev1, nsat_c);
          // scale bytes go to s_col[c][gb0 + j]; they are gathered in the
          // 8-byte aligned window of the destination and leave when the
          // window is complete or the unit ends
          const ScaleSlot e0 = col_scale_slot<MMA>(p, U.c0 + 2 * tid, U.gb0 + j);
          const ScaleSlot e1 = col_scale_slot<MMA>(p, U.c0 + 2 * tid + 1, U.gb0 + j);
          constexpr int W = col_scale_window<MMA>();
          sc0 |= (uint64_t)(b & 0xFFu) << (8 * e0.q);
          sc1 |= (uint64_t)(b >> 8) << (8 * e1.q);
          const bool last = j == U.nblk - 1;
          if (e0.q == W - 1 || last) {
            const int from = j < e0.q ? e0.q - j : 0;  // window bytes before the unit's first block
            flush_scales8(p, e0.win, from, e0.q + 1, e0.gbw, sc0, sp);
            sc0 = 0;
          }
          if (e1.q == W - 1 || last) {
            const int from = j < e1.q ? e1.q - j : 0;
            flush_scales8(p, e1.win, from, e1.q + 1, e1.gbw, sc1, sp);
            sc1 = 0;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (gave_up || abort_flag) return;
  }
  if constexpr (EXT) {
    if (p.sat != nullptr) {  // one atomic per warp and direction
      const uint32_t a = __reduce_add_sync(0xFFFFFFFFu, nsat_r), c = __reduce_add_sync(0xFFFFFFFFu, nsat_c);
      if (lane == 0 && a) atomicAdd(p.sat, (unsigned long long)a);
      if (lane == 0 && c) atomicAdd(p.sat + 1, (unsigned long long)c);
    }
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// BF16, ungrouped, row-major scales: the lean unit kernel
// ---------------------------------------------------------------------------
// Same pipeline and units as mx_tma_kernel, for the common case the general
// kernel carries state for but never uses here: no groups, so every unit is
// `super` whole blocks from a row multiple of 32 * super, and (when the
// columnwise copy is written) rows % 32 == 0 with a 32-byte aligned q_col, so
// every column's 32 codes of a block are one aligned sector.  Output
// pointers are set up once per unit and advanced per block; a column's scale
// bytes of the unit leave in one store at its end.  Rowwise only, rows may
// be ragged (the last block's rows past the end are skipped).

// Unit u = ti * strips + strip of a CTA's walk u = blockIdx.x, + gridDim.x,
// ...: (ti, strip) advanced without a 64-bit division per unit.
struct UnitWalk {
  int64_t strips, ti, strip, dq, dr;
  __device__ __forceinline__ explicit UnitWalk(int64_t n) : strips(n) {
    ti = blockIdx.x / n;
    strip = blockIdx.x - ti * n;
    dq = gridDim.x / n;
    dr = gridDim.x - dq * n;
  }
  __device__ __forceinline__ void next() {
    ti += dq;
    strip += dr;
    if (strip >= strips) {
      strip -= strips;
      ++ti;
    }
  }
};

// Rowwise, one lane per 1x32 block: codes of block b of row r of the stage
// to dst; returns the scale byte.
template <int FMT, bool EXT>
__device__ __forceinline__ uint32_t lean_row_block(const MxParams& p, const unsigned char* stage, int r, int b,
                                                   uint8_t* dst, const StorePolicy& sp, uint32_t& nsat) {
  const unsigned char* line = stage + (b >> 1) * kSubBytes + r * 128;
  const int c0 = (b & 1) * 4;
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const uint4 v = *(const uint4*)(line + (((c0 + j) ^ (r & 7)) << 4));
    w[4 * j] = v.x;
    w[4 * j + 1] = v.y;
    w[4 * j + 2] = v.z;
    w[4 * j + 3] = v.w;
  }
  uint32_t m4[4];
#pragma unroll
  for (int j = 0; j < 4; j++)
    m4[j] = absmax_nan_bf16x2(absmax_nan_bf16x2(w[4 * j], w[4 * j + 1]), absmax_nan_bf16x2(w[4 * j + 2], w[4 * j + 3]));
  const uint32_t m = absmax_nan_bf16x2(absmax_nan_bf16x2(m4[0], m4[1]), absmax_nan_bf16x2(m4[2], m4[3]));
  const uint32_t am = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu) << 16;
  const uint32_t byte = e8m0_from_amax<FMT>(am, EXT ? p.round_up : 1);
  const float mult = e8m0_multiplier(byte);
  uint32_t d[8];
#pragma unroll
  for (int k = 0; k < 8; k++) d[k] = row_codes4<FMT, false>(w[2 * k], w[2 * k + 1], mult);
  if (byte == 0xFFu || am == 0u) {  // Inf/NaN block: 0x7F codes; zero block: +0 codes
    const uint32_t fill = am == 0u ? 0u : 0x7F7F7F7Fu;
#pragma unroll
    for (int k = 0; k < 8; k++) d[k] = fill;
  } else if constexpr (EXT) {
    if (p.sat != nullptr && block_saturates<FMT>(am, byte, mult)) {
#pragma unroll
      for (int k = 0; k < 16; k++) nsat += sat_pair<FMT>(w[k], mult, mult);
    }
  }
  st_data32(dst, d, sp);
  return byte;
}

// Row-major s_row bytes of one warp's 8 rows: lane l holds row 8w + l % 8,
// blocks l / 8 (y0) and 4 + l / 8 (y1); sr is the lane's row's first scale of
// the strip.  With a whole, 8-byte aligned strip the row's 8 bytes leave from
// lane l % 8 in one store.  All 32 lanes must call.
__device__ __forceinline__ void lean_row_scales(uint8_t* sr, int lane, bool row_ok, bool srow8, bool ok0, bool ok1,
                                                uint32_t y0, uint32_t y1, const StorePolicy& sp) {
  const uint32_t v = y0 | (y1 << 8);
  const uint32_t v1 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 8);
  const uint32_t v2 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 16);
  const uint32_t v3 = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 24);
  if (!row_ok) return;
  if (srow8) {
    if (lane < 8) {
      const uint32_t lo = (v & 0xFFu) | ((v1 & 0xFFu) << 8) | ((v2 & 0xFFu) << 16) | ((v3 & 0xFFu) << 24);
      const uint32_t hi = (v >> 8) | ((v1 >> 8) << 8) | ((v2 >> 8) << 16) | ((v3 >> 8) << 24);
      st_scale64(sr, (uint64_t)lo | ((uint64_t)hi << 32), sp);
    }
  } else {
    const int b = lane >> 3;
    if (ok0) st_scale8(sr + b, y0, sp);
    if (ok1) st_scale8(sr + b + 4, y1, sp);
  }
}

template <int FMT, int DIR, bool EXT>
__global__ void __launch_bounds__(kTmaThreads, FP8Q_MX_MIN_CTAS) mx_lean_kernel(const __grid_constant__ CUtensorMap tmap, MxParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ volatile int abort_flag;
  unsigned char* stages = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (tid == kConsumers) prefetch_tensormap(&tmap);
  pdl_wait();
  __syncthreads();
  const int64_t nbr = (p.rows + 31) / 32;
  const int S = p.super;
  const int64_t units = (nbr + S - 1) / S * p.strips;
  const uint64_t budget = g_wait_budget_ns;

  if (warp == kConsumers / 32) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    int64_t k = 0;
    const bool stall = *(volatile unsigned*)&g_mx_stall_producer != 0;
    bool stop = false;
    UnitWalk w(p.strips);
    for (int64_t u = blockIdx.x; u < units && !abort_flag && !stall && !stop; u += gridDim.x, w.next()) {
      const int c0 = (int)(w.strip * kTileCols);
      const int64_t rb0 = w.ti * S;
      const int nblk = (int)min((int64_t)S, nbr - rb0);
      for (int j = 0; j < nblk; j++, ++k) {
        const int s = (int)(k % kStages);
        const uint32_t round = (uint32_t)(k / kStages);
        if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1u, budget)) {
          atomicOr(&g_mx_error, 1u);
          abort_flag = 1;
          stop = true;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        unsigned char* dst = stages + s * kStageBytes;
        const int row = (int)((rb0 + j) * kTileRows);
#pragma unroll
        for (int q = 0; q < kTileCols / kSubCols; q++)
          tma_load_2d(dst + q * kSubBytes, &tmap, c0 + q * kSubCols, row, &full[s]);
      }
    }
    pdl_launch_dependents();
    const int64_t first = k > kStages ? k - kStages : 0;  // every issued copy lands before exit
    for (int64_t j = first; j < k; j++)
      mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1), 2000000000ull);
    return;
  }

  // ---------------- consumers ----------------
  const StorePolicy sp = make_policy();
  uint32_t nsat_r = 0, nsat_c = 0;
  const int64_t sld = p.cols / 32;
  const int r = 8 * warp + (lane & 7);  // rowwise: this lane's row of a block and its two blocks
  const int b0 = lane >> 3, b1 = 4 + (lane >> 3);
  int64_t k = 0;
  UnitWalk w(p.strips);
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x, w.next()) {
    const int64_t c0 = w.strip * kTileCols;
    const int nc = (int)min((int64_t)kTileCols, p.cols - c0);
    const int64_t rb0 = w.ti * S;
    const int nblk = (int)min((int64_t)S, nbr - rb0);
    const int64_t row0 = rb0 * kTileRows;
    // rowwise destinations of block 0; + 32 rows per block
    uint8_t* qr = p.q_row + (row0 + r) * p.cols + c0;
    uint8_t* sr = p.s_row + (row0 + r) * sld + c0 / 32;
    const bool rb0_ok = 32 * b0 < nc, rb1_ok = 32 * b1 < nc;
    const bool srow8 = nc == kTileCols && (((uintptr_t)sr | (uintptr_t)(32 * sld)) & 7u) == 0;
    // columnwise: columns c0 + 2 tid and + 1, block 0 at row0
    const bool col_ok = 2 * tid < nc;
    uint8_t* qc = p.q_col + (c0 + 2 * tid) * p.rows + row0;
    uint32_t sc0 = 0, sc1 = 0;
    bool gave_up = false;
    for (int j = 0; j < nblk; j++, ++k) {
      const int s = (int)(k % kStages);
      const uint32_t round = (uint32_t)(k / kStages);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], round & 1u, budget))) {
        atomicOr(&g_mx_error, 1u);
        abort_flag = 1;
        gave_up = true;
        break;
      }
      const unsigned char* stage = stages + s * kStageBytes;
      if constexpr (DIR & MXFP8_ROW) {
        const bool row_ok = row0 + 32 * j + r < p.rows;
        uint32_t y0 = 0, y1 = 0;
        if (row_ok && rb0_ok) y0 = lean_row_block<FMT, EXT>(p, stage, r, b0, qr + 32 * b0, sp, nsat_r);
        if (row_ok && rb1_ok) y1 = lean_row_block<FMT, EXT>(p, stage, r, b1, qr + 32 * b1, sp, nsat_r);
        lean_row_scales(sr, lane, row_ok, srow8, rb0_ok, rb1_ok, y0, y1, sp);
        qr += 32 * p.cols;
        sr += 32 * sld;
      }
      if constexpr (DIR & MXFP8_COL) {
        if (col_ok) {
          Tile t;
          t.r0 = row0 + 32 * j;
          t.lo = 0;
          t.nr = kTileRows;
          t.c0 = c0;
          t.nc = nc;
          uint32_t d0[8], d1[8];
          const uint32_t b = col_codes_bf16<FMT, EXT, false>(p, t, stage, tid, d0, d1, nsat_c, 0, kTileRows);
          st_data32(qc + 32 * j, d0, sp);
          st_data32(qc + p.rows + 32 * j, d1, sp);
          sc0 |= (b & 0xFFu) << (8 * j);
          sc1 |= (b >> 8) << (8 * j);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (gave_up || abort_flag) return;
    if constexpr (DIR & MXFP8_COL) {
      if (col_ok) {  // s_col[c][rb0 .. rb0 + nblk): one word when whole and aligned
        uint8_t* e0 = p.s_col + (c0 + 2 * tid) * p.s_col_ld + rb0;
        uint8_t* e1 = e0 + p.s_col_ld;
        if (nblk == 4 && (((uintptr_t)e0 | (uintptr_t)e1) & 3u) == 0) {
          st_scale32(e0, sc0, sp);
          st_scale32(e1, sc1, sp);
        } else {
          for (int j = 0; j < nblk; j++) {
            st_scale8(e0 + j, sc0 >> (8 * j), sp);
            st_scale8(e1 + j, sc1 >> (8 * j), sp);
          }
        }
      }
    }
  }
  if constexpr (EXT) {
    if (p.sat != nullptr) {  // one atomic per warp and direction
      const uint32_t a = __reduce_add_sync(0xFFFFFFFFu, nsat_r), c = __reduce_add_sync(0xFFFFFFFFu, nsat_c);
      if (lane == 0 && a) atomicAdd(p.sat, (unsigned long long)a);
      if (lane == 0 && c) atomicAdd(p.sat + 1, (unsigned long long)c);
    }
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// BF16, grouped, rows % 32 == 0: bands of aligned rows
// ---------------------------------------------------------------------------
// Units are bands of kBandRows aligned rows in one 256-column strip, dealt
// out band-major.  A unit walks, in row order, the column blocks that
// overlap its rows; each block is loaded as one 32-row window from its own
// first row (the window of a group's short last block also holds rows of
// the next group, which it leaves alone).  A block that straddles the
// band's first row is loaded by both bands: the earlier band owns its scale
// and its rows above the boundary, the later one takes only its rows below.
//
// The transposed codes of one column form a byte stream over the band's
// rows.  With rows % 32 == 0 and a 32-byte aligned q_col, each column's
// stream starts on a 32-byte boundary and every column is at the same phase
// `pos` (the structure of the blocks does not depend on the column), so
// every q_col store is one whole aligned sector and no sector is written by
// two CTAs.  Blocks are 32 rows except at a group's end, so inside a group
// the phase stays put and a sector is the previous block's last pos codes
// followed by this block's first 32 - pos.

#ifndef FP8Q_MX_BAND_SECTORS  // 32-row sectors per band
#define FP8Q_MX_BAND_SECTORS 32
#endif
constexpr int64_t kBandRows = 32 * FP8Q_MX_BAND_SECTORS;

struct BandBlk {
  int64_t s;   // first row of the block, and of its window
  int64_t e;   // end of the block's rows (e - s in 1..32)
  int64_t gb;  // s_col index of the block; -1: rows in no group
};

// The group whose rows a unit's walk is in: index and clamped bounds.  The
// walk moves forward, so the bounds are looked up again (binary search)
// only when it leaves them.
struct GroupCursor {
  int g = 0;
  int64_t o = 0, o1 = -1;  // empty until the first lookup
};

// The column block holding row `cur`.  Rows outside every group (offsets
// that do not cover [0, rows)) form gap blocks that end at the next 32-row
// boundary: their rowwise copy is produced, their transposed codes are 0 and
// they have no scale.  The walk advances by at least one row per block and
// stays in [0, rows) for any offsets.
__device__ __forceinline__ BandBlk band_block(const MxParams& p, const int* blk, GroupCursor& gc, int64_t cur) {
  if (!(gc.o <= cur && cur < gc.o1)) {
    gc.g = group_of_row(p.off, p.G, cur);
    gc.o = grp_row(p, gc.g);
    gc.o1 = grp_row(p, gc.g + 1);
  }
  BandBlk b;
  if (gc.o <= cur && cur < gc.o1) {
    const int64_t k = (cur - gc.o) >> 5;
    b.s = gc.o + 32 * k;
    b.e = min(b.s + 32, gc.o1);
    b.gb = (int64_t)blk[gc.g] + k;
  } else {
    b.s = cur;
    b.e = min((cur & ~(int64_t)31) + 32, p.rows);
    b.gb = -1;
  }
  return b;
}

// Appends `len` codes, bytes [skip, skip + len) of d, to a column's stream
// whose pending codes are the last `pos` bytes of prev; a completed sector
// is stored at dst.  pos, skip and len are the same for every thread of the
// CTA, so each branch is uniform.
__device__ __forceinline__ void stream_append(uint8_t* dst, uint32_t (&prev)[8], const uint32_t (&din)[8], int pos,
                                              int skip, int len, const StorePolicy& sp) {
  const uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  uint32_t d[8];
  if (skip) {
    window32(din, z, skip, d);
  } else {
#pragma unroll
    for (int i = 0; i < 8; i++) d[i] = din[i];
  }
  if (pos + len >= 32) {
    if (pos) {
      uint32_t o[8];
      window32(prev, d, 32 - pos, o);
      st_data32(dst, o, sp);
    } else {
      st_data32(dst, d, sp);
    }
  }
  if (len == 32) {
#pragma unroll
    for (int i = 0; i < 8; i++) prev[i] = d[i];
  } else {
    uint32_t o[8];
    window32(prev, d, len, o);  // ends with the pending codes
#pragma unroll
    for (int i = 0; i < 8; i++) prev[i] = o[i];
  }
}

template <int FMT, int DIR, bool EXT, bool MMA>
__global__ void __launch_bounds__(kTmaThreads, FP8Q_MX_MIN_CTAS) mx_band_kernel(const __grid_constant__ CUtensorMap tmap, MxParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ volatile int abort_flag;
  unsigned char* stages = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  int* blk = (int*)(stages + kStages * kStageBytes);
  int* sup = blk + (p.G + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (tid == kConsumers) prefetch_tensormap(&tmap);
  pdl_wait();
  build_prefix<kTmaThreads>(p, blk, sup);
  const int64_t bands = (p.rows + kBandRows - 1) / kBandRows;
  const int64_t units = bands * p.strips;
  const uint64_t budget = g_wait_budget_ns;

  if (warp == kConsumers / 32) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    int64_t k = 0;
    const bool stall = *(volatile unsigned*)&g_mx_stall_producer != 0;
    bool stop = false;
    for (int64_t u = blockIdx.x; u < units && !abort_flag && !stall && !stop; u += gridDim.x) {
      const int64_t band = u / p.strips;
      const int c0 = (int)((u - band * p.strips) * kTileCols);
      const int64_t A = band * kBandRows, B = min(A + kBandRows, p.rows);
      GroupCursor gc;
      for (int64_t cur = A; cur < B; ++k) {
        const BandBlk bb = band_block(p, blk, gc, cur);
        const int s = (int)(k % kStages);
        const uint32_t round = (uint32_t)(k / kStages);
        if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1u, budget)) {
          atomicOr(&g_mx_error, 1u);
          abort_flag = 1;
          stop = true;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        unsigned char* dst = stages + s * kStageBytes;
#pragma unroll
        for (int q = 0; q < kTileCols / kSubCols; q++)
          tma_load_2d(dst + q * kSubBytes, &tmap, c0 + q * kSubCols, (int)bb.s, &full[s]);
        cur = bb.e;
      }
    }
    pdl_launch_dependents();  // all loads issued: the next kernel may launch
    // every issued copy lands before the CTA can exit (fixed 2 s bound)
    const int64_t first = k > kStages ? k - kStages : 0;
    for (int64_t j = first; j < k; j++)
      mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1), 2000000000ull);
    return;
  }

  // ---------------- consumers ----------------
  const StorePolicy sp = make_policy();
  uint32_t nsat_r = 0, nsat_c = 0;  // saturated elements (counted when p.sat is set)
  int64_t k = 0;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t band = u / p.strips;
    const int64_t c0 = (u - band * p.strips) * kTileCols;
    const int nc = (int)min((int64_t)kTileCols, p.cols - c0);
    const int64_t A = band * kBandRows, B = min(A + kBandRows, p.rows);
    const int64_t col = c0 + 2 * tid;
    uint8_t* qc0 = p.q_col + col * p.rows;
    uint8_t* qc1 = qc0 + p.rows;
    uint8_t* sb0 = p.s_col + col * p.s_col_ld;  // row-major: the columns' scale rows
    uint8_t* sb1 = sb0 + p.s_col_ld;
    const int r = 8 * warp + (lane & 7);  // rowwise: this lane's window row and its two blocks
    const int rb0 = lane >> 3, rb1 = 4 + (lane >> 3);
    const bool rb0_ok = 32 * rb0 < nc, rb1_ok = 32 * rb1 < nc;
    uint64_t sc0 = 0, sc1 = 0;   // scale bytes of this thread's two columns, gathered per 8-byte window
    uint32_t prev0[8], prev1[8];  // the columns' pending codes (the last `pos` bytes)
    int pos = 0;                  // stream phase: pending codes
    int64_t sec = A;              // first row of the next sector to store
    int nown = 0;                 // blocks whose scale this unit has produced
    bool gave_up = false;
    GroupCursor gc;
    for (int64_t cur = A; cur < B; ++k) {
      const BandBlk bb = band_block(p, blk, gc, cur);
      const int s = (int)(k % kStages);
      const uint32_t round = (uint32_t)(k / kStages);
      // every lane waits; the warp acts on one voted answer so it never splits
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], round & 1u, budget))) {
        atomicOr(&g_mx_error, 1u);
        abort_flag = 1;
        gave_up = true;
        break;
      }
      const int64_t end = min(bb.e, B);
      Tile t;  // this unit's rows of the window
      t.r0 = bb.s;
      t.lo = (int)(cur - bb.s);
      t.nr = (int)(end - bb.s);
      t.c0 = c0;
      t.nc = nc;
      const unsigned char* stage = stages + s * kStageBytes;
      if constexpr (DIR & MXFP8_ROW) {
        if constexpr (MMA) {
          const uint32_t y0 = row_block_bf16<FMT, EXT, true>(p, t, stage, r, rb0, sp, nsat_r);
          const uint32_t y1 = row_block_bf16<FMT, EXT, true>(p, t, stage, r, rb1, sp, nsat_r);
          store_row_scales<MMA>(p, t, warp, lane, y0, y1, sp);
        } else {
          const bool row_ok = r >= t.lo && r < t.nr;
          uint8_t* qr = p.q_row + (bb.s + r) * p.cols + c0;
          uint8_t* sr = p.s_row + (bb.s + r) * (p.cols / 32) + c0 / 32;
          uint32_t y0 = 0, y1 = 0;
          if (row_ok && rb0_ok) y0 = lean_row_block<FMT, EXT>(p, stage, r, rb0, qr + 32 * rb0, sp, nsat_r);
          if (row_ok && rb1_ok) y1 = lean_row_block<FMT, EXT>(p, stage, r, rb1, qr + 32 * rb1, sp, nsat_r);
          lean_row_scales(sr, lane, row_ok, nc == kTileCols && ((uintptr_t)sr & 7u) == 0, rb0_ok, rb1_ok, y0, y1, sp);
        }
      }
      if constexpr (DIR & MXFP8_COL) {
        if (2 * tid < nc) {
          Tile tb = t;  // the whole block: its amax takes every one of its rows
          tb.lo = 0;
          tb.nr = (int)(bb.e - bb.s);
          uint32_t d0[8], d1[8];
          const uint32_t b =
              col_codes_bf16<FMT, EXT, true>(p, tb, stage, tid, d0, d1, nsat_c, t.lo, bb.gb < 0 ? t.lo : t.nr);
          if (bb.gb < 0) {
#pragma unroll
            for (int i = 0; i < 8; i++) d0[i] = d1[i] = 0u;
          }
          const int len = t.nr - t.lo;
          stream_append(qc0 + sec, prev0, d0, pos, t.lo, len, sp);
          stream_append(qc1 + sec, prev1, d1, pos, t.lo, len, sp);
          if (pos + len >= 32) sec += 32;
          pos = (pos + len) & 31;
          const bool last = bb.e >= B;
          if (bb.gb >= 0 && bb.s >= A) {
            // scale bytes go to s_col[c][gb]; gathered in the 8-byte aligned
            // window of the destination, stored when the window is complete
            // or the unit ends
            const ScaleSlot e0 = MMA ? col_scale_slot<MMA>(p, col, bb.gb) : scale_slot_at(sb0 + bb.gb, bb.gb);
            const ScaleSlot e1 = MMA ? col_scale_slot<MMA>(p, col + 1, bb.gb) : scale_slot_at(sb1 + bb.gb, bb.gb);
            constexpr int W = col_scale_window<MMA>();
            sc0 |= (uint64_t)(b & 0xFFu) << (8 * e0.q);
            sc1 |= (uint64_t)(b >> 8) << (8 * e1.q);
            if (e0.q == W - 1 || last) {
              const int from = nown < e0.q ? e0.q - nown : 0;  // window bytes before the unit's first scale
              flush_scales8(p, e0.win, from, e0.q + 1, e0.gbw, sc0, sp);
              sc0 = 0;
            }
            if (e1.q == W - 1 || last) {
              const int from = nown < e1.q ? e1.q - nown : 0;
              flush_scales8(p, e1.win, from, e1.q + 1, e1.gbw, sc1, sp);
              sc1 = 0;
            }
            ++nown;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      cur = bb.e;
    }
    if (gave_up || abort_flag) return;
  }
  if constexpr (EXT) {
    if (p.sat != nullptr) {  // one atomic per warp and direction
      const uint32_t a = __reduce_add_sync(0xFFFFFFFFu, nsat_r), c = __reduce_add_sync(0xFFFFFFFFu, nsat_c);
      if (lane == 0 && a) atomicAdd(p.sat, (unsigned long long)a);
      if (lane == 0 && c) atomicAdd(p.sat + 1, (unsigned long long)c);
    }
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// FP32: loads into registers, rowwise from registers, columnwise via smem
// ---------------------------------------------------------------------------
template <int FMT, int DIR>
__global__ void __launch_bounds__(kConsumers) mx_f32_kernel(MxParams p) {
  constexpr int kRowBytes = kTileCols * 4;
  constexpr int kRowSlots = kTileRows / (kConsumers / 32);
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* tile = smem;                           // [32][1024 B]
  int* blk = (int*)(smem + kTileRows * kRowBytes);     // [G + 1]
  int* sup = blk + (p.G + 1);                           // [G + 1] (super = 1)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const StorePolicy sp = make_policy();
  uint32_t nsat_r = 0, nsat_c = 0;
  pdl_wait();
  build_prefix<kConsumers>(p, blk, sup);
  const int64_t units = (int64_t)sup[p.G] * p.strips;

  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const Unit U = unit_of(p, blk, sup, u);
    const Tile t = block_of(U, 0);
    const bool col_ok = lane * 8 < t.nc;
    uint4 v[kRowSlots][2];
#pragma unroll
    for (int i = 0; i < kRowSlots; i++) {
      const int r = warp + 4 * i;
      const bool ok = col_ok && r < t.nr;
      const char* src = (const char*)p.x + ((t.r0 + r) * p.cols + t.c0 + lane * 8) * 4;
      v[i][0] = ok ? ld_stream(src) : make_uint4(0, 0, 0, 0);
      v[i][1] = ok ? ld_stream(src + 16) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kRowSlots; i++) {
      const int r = warp + 4 * i;
      if constexpr (DIR & MXFP8_ROW) {
        uint32_t am = max(max(max(v[i][0].x & 0x7FFFFFFFu, v[i][0].y & 0x7FFFFFFFu),
                              max(v[i][0].z & 0x7FFFFFFFu, v[i][0].w & 0x7FFFFFFFu)),
                          max(max(v[i][1].x & 0x7FFFFFFFu, v[i][1].y & 0x7FFFFFFFu),
                              max(v[i][1].z & 0x7FFFFFFFu, v[i][1].w & 0x7FFFFFFFu)));
        am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
        am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
        if (col_ok && r < t.nr) {
          const uint32_t byte = e8m0_from_amax<FMT>(am, p.round_up);
          const float mult = e8m0_multiplier(byte);
          if (p.sat != nullptr && block_saturates<FMT>(am, byte, mult)) {
            const uint32_t e[8] = {v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w,
                                   v[i][1].x, v[i][1].y, v[i][1].z, v[i][1].w};
#pragma unroll
            for (int q = 0; q < 8; q++) nsat_r += fabsf(__uint_as_float(e[q])) * mult > Fmt<FMT>::kMax;
          }
          uint2 o;
          o.x = mx_fix(mx_codes4<FMT>(__uint_as_float(v[i][0].x), __uint_as_float(v[i][0].y),
                                      __uint_as_float(v[i][0].z), __uint_as_float(v[i][0].w), mult), byte, am);
          o.y = mx_fix(mx_codes4<FMT>(__uint_as_float(v[i][1].x), __uint_as_float(v[i][1].y),
                                      __uint_as_float(v[i][1].z), __uint_as_float(v[i][1].w), mult), byte, am);
          const int64_t row = t.r0 + r;
          st_stream(p.q_row + row * p.cols + t.c0 + lane * 8, o);
          if ((lane & 3) == 0) {
            const int64_t sc = (t.c0 + lane * 8) / 32;
            p.s_row[p.mma ? mma_off(row, sc, p.row_bcols) : row * (p.cols / 32) + sc] = (uint8_t)byte;
          }
        }
      }
      if constexpr (DIR & MXFP8_COL) {
        *(uint4*)(tile + r * kRowBytes + lane * 32) = v[i][0];
        *(uint4*)(tile + r * kRowBytes + lane * 32 + 16) = v[i][1];
      }
    }
    if constexpr (DIR & MXFP8_COL) {
      __syncthreads();
      const int cl = 2 * tid;
      if (cl < t.nc) {
        uint32_t a0 = 0, a1 = 0;
#pragma unroll
        for (int r = 0; r < kTileRows; r++) {
          const uint2 w = *(const uint2*)(tile + r * kRowBytes + cl * 4);
          a0 = max(a0, w.x & 0x7FFFFFFFu);
          a1 = max(a1, w.y & 0x7FFFFFFFu);
        }
        const uint32_t b0 = e8m0_from_amax<FMT>(a0, p.round_up), b1 = e8m0_from_amax<FMT>(a1, p.round_up);
        const float m0 = e8m0_multiplier(b0), m1 = e8m0_multiplier(b1);
        if (p.sat != nullptr) {
          const bool s0 = block_saturates<FMT>(a0, b0, m0), s1 = block_saturates<FMT>(a1, b1, m1);
          if (s0 || s1) {
            for (int r = 0; r < t.nr; r++) {
              const uint2 w = *(const uint2*)(tile + r * kRowBytes + cl * 4);
              if (s0) nsat_c += fabsf(__uint_as_float(w.x)) * m0 > Fmt<FMT>::kMax;
              if (s1) nsat_c += fabsf(__uint_as_float(w.y)) * m1 > Fmt<FMT>::kMax;
            }
          }
        }
        uint32_t d0[8], d1[8];
#pragma unroll
        for (int k = 0; k < 8; k++) {
          const uint2 w0 = *(const uint2*)(tile + (4 * k) * kRowBytes + cl * 4);
          const uint2 w1 = *(const uint2*)(tile + (4 * k + 1) * kRowBytes + cl * 4);
          const uint2 w2 = *(const uint2*)(tile + (4 * k + 2) * kRowBytes + cl * 4);
          const uint2 w3 = *(const uint2*)(tile + (4 * k + 3) * kRowBytes + cl * 4);
          d0[k] = mx_fix(mx_codes4<FMT>(__uint_as_float(w0.x), __uint_as_float(w1.x), __uint_as_float(w2.x),
                                        __uint_as_float(w3.x), m0), b0, a0);
          d1[k] = mx_fix(mx_codes4<FMT>(__uint_as_float(w0.y), __uint_as_float(w1.y), __uint_as_float(w2.y),
                                        __uint_as_float(w3.y), m1), b1, a1);
        }
        const int64_t c = t.c0 + cl;
        store_col32(p.q_col + c * p.rows + t.r0, d0, t.nr, sp);
        store_col32(p.q_col + (c + 1) * p.rows + t.r0, d1, t.nr, sp);
        if (U.gb0 < p.s_col_ld) {
          p.s_col[p.mma ? mma_off(c, U.gb0, p.col_bcols) : c * p.s_col_ld + U.gb0] = (uint8_t)b0;
          p.s_col[p.mma ? mma_off(c + 1, U.gb0, p.col_bcols) : (c + 1) * p.s_col_ld + U.gb0] = (uint8_t)b1;
        }
      }
      __syncthreads();  // the tile is rewritten by the next unit
    }
  }
  if (p.sat != nullptr) {
    const uint32_t a = __reduce_add_sync(0xFFFFFFFFu, nsat_r), c = __reduce_add_sync(0xFFFFFFFFu, nsat_c);
    if (lane == 0 && a) atomicAdd(p.sat, (unsigned long long)a);
    if (lane == 0 && c) atomicAdd(p.sat + 1, (unsigned long long)c);
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Resident CTAs per SM for `kernel` with `smem` dynamic bytes (cached per
// instantiation; recomputed when a call needs more shared memory).
template <typename K>
static fp8q_status ctas_per_sm(K kernel, int threads, size_t smem, size_t* attr, int* per_sm, std::mutex* mu,
                               int* out) {
  std::lock_guard<std::mutex> lock(*mu);
  if (smem > *attr) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(mxfp8)");
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
    *per_sm = n;
    *attr = smem;
  }
  *out = *per_sm;
  return FP8Q_OK;
}

// Kernel kinds of the BF16 path.
enum : int { kUnitKernel = 0, kBandKernel = 1, kLeanKernel = 2 };

template <int FMT, int DIR, bool EXT, int KIND, bool MMA>
static fp8q_status launch_tma(const MxParams& p, cudaStream_t s) {
  constexpr bool BAND = KIND == kBandKernel, LEAN = KIND == kLeanKernel;
  static_assert(!(LEAN && MMA), "the lean kernel writes row-major scales");
  static_assert(FP8Q_MX_SUPER >= 1 && FP8Q_MX_SUPER <= 4, "a unit's scale bytes of a column fill one word");
  auto enc = encode_fn();
  if (!enc) return fail(FP8Q_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap map;
  cuuint64_t dims[2] = {(cuuint64_t)p.cols, (cuuint64_t)p.rows};
  cuuint64_t strides[1] = {(cuuint64_t)p.cols * 2};
  cuuint32_t box[2] = {kSubCols, kTileRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FP8Q_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  MxParams q = p;
  q.super = BAND ? 1 : (p.off != nullptr ? FP8Q_MX_SUPER_GROUPED : FP8Q_MX_SUPER);
  const size_t smem = 1024 + (size_t)kStages * kStageBytes + (LEAN ? 0 : 2 * sizeof(int) * (p.G + 1));
  auto kernel = LEAN ? mx_lean_kernel<FMT, DIR, EXT> : BAND ? mx_band_kernel<FMT, DIR, EXT, MMA> : mx_tma_kernel<FMT, DIR, EXT, MMA>;
  static size_t attr = 0;
  static int per_sm_cache = 0;
  static std::mutex mu;
  int per_sm = 0;
  fp8q_status st = ctas_per_sm(kernel, kTmaThreads, smem, &attr, &per_sm_cache, &mu, &per_sm);
  if (st != FP8Q_OK) return st;
  // units: bands x strips, or (over any valid offsets) blocks per group
  // rounded up to `super`, x strips
  const int64_t max_units = BAND   ? (p.rows + kBandRows - 1) / kBandRows * p.strips
                           : LEAN ? ((p.rows + 31) / 32 + q.super - 1) / q.super * p.strips
                                  : ((p.rows + 31) / 32 / q.super + 1 + p.G) * p.strips;
  int64_t grid = (int64_t)per_sm * sm_count();
  // One CTA per unit (the lean kernel; measured: 16384 x 14336 161 -> 144 us,
  // the hardware's block scheduler balancing what a strided persistent walk
  // left uneven), else a persistent grid of every resident slot.
  if (max_units < grid || (LEAN && FP8Q_MX_LEAN_GRID_ALL) || (BAND && FP8Q_MX_BAND_GRID_ALL)) grid = max_units;
  if (grid > 0x7FFFFFFF) grid = 0x7FFFFFFF;  // the kernels walk any remaining units
  if (grid < 1) grid = 1;
  const cudaError_t e = launch_kernel(kernel, dim3((unsigned)grid), dim3(kTmaThreads), smem, s, map, q);
  if (e != cudaSuccess) return cuda_fail(e, "mxfp8 tma kernel launch");
  return check_launch("mxfp8 tma kernel");
}

template <int FMT, int DIR>
static fp8q_status launch_f32(const MxParams& p, cudaStream_t s) {
  MxParams q = p;
  q.super = 1;
  const size_t smem = (size_t)kTileRows * kTileCols * 4 + 2 * sizeof(int) * (p.G + 1);
  static size_t attr = 0;
  static int per_sm_cache = 0;
  static std::mutex mu;
  int per_sm = 0;
  fp8q_status st = ctas_per_sm(mx_f32_kernel<FMT, DIR>, kConsumers, smem, &attr, &per_sm_cache, &mu, &per_sm);
  if (st != FP8Q_OK) return st;
  const int64_t max_units = ((p.rows + 31) / 32 + p.G) * p.strips;
  int64_t grid = (int64_t)per_sm * sm_count();
  if (max_units < grid) grid = max_units;
  if (grid < 1) grid = 1;
  const cudaError_t e = launch_kernel(mx_f32_kernel<FMT, DIR>, dim3((unsigned)grid), dim3(kConsumers), smem, s, q);
  if (e != cudaSuccess) return cuda_fail(e, "mxfp8 fp32 kernel launch");
  return check_launch("mxfp8 fp32 kernel");
}

#ifndef FP8Q_MX_BAND_UNGROUPED  // route ungrouped BF16 calls to the band kernel as well
#define FP8Q_MX_BAND_UNGROUPED 0
#endif

#ifndef FP8Q_MX_LEAN  // ungrouped BF16 calls with row-major scales take the lean kernel
#define FP8Q_MX_LEAN 1
#endif

template <int FMT, bool EXT, int KIND, bool MMA>
static fp8q_status launch_tma_dir(const MxParams& p, int dir, cudaStream_t s) {
  if (dir == MXFP8_ROW) return launch_tma<FMT, MXFP8_ROW, EXT, KIND, MMA>(p, s);
  if (dir == MXFP8_COL) return launch_tma<FMT, MXFP8_COL, EXT, KIND, MMA>(p, s);
  return launch_tma<FMT, MXFP8_BOTH, EXT, KIND, MMA>(p, s);
}

template <int FMT, int KIND, bool MMA>
static fp8q_status launch_tma_ext(const MxParams& p, int dir, bool ext, cudaStream_t s) {
  return ext ? launch_tma_dir<FMT, true, KIND, MMA>(p, dir, s) : launch_tma_dir<FMT, false, KIND, MMA>(p, dir, s);
}

template <int FMT, int KIND>
static fp8q_status launch_tma_layout(const MxParams& p, int dir, bool ext, cudaStream_t s) {
  if constexpr (KIND == kLeanKernel) return launch_tma_ext<FMT, KIND, false>(p, dir, ext, s);
  else
    return p.mma ? launch_tma_ext<FMT, KIND, true>(p, dir, ext, s) : launch_tma_ext<FMT, KIND, false>(p, dir, ext, s);
}

template <int FMT>
static fp8q_status launch_fmt(const MxParams& p, int dt, int dir, cudaStream_t s) {
  if (dt == kBF16) {
    const bool ext = p.round_up == 0 || p.sat != nullptr;
    MxParams q = p;
    if (dir == MXFP8_ROW && p.off != nullptr) {  // the rowwise copy does not depend on the groups
      q.off = nullptr;
      q.G = 1;
    }
    const bool col_aligned = p.rows % 32 == 0 && ((uintptr_t)p.q_col & 31u) == 0;
    // no groups and row-major scales: the lean kernel (the columnwise copy
    // needs every column's blocks on whole aligned sectors)
    if (FP8Q_MX_LEAN && q.off == nullptr && !q.mma && (!(dir & MXFP8_COL) || col_aligned))
      return launch_tma_layout<FMT, kLeanKernel>(q, dir, ext, s);
    // bands of aligned rows: every transposed store is a whole aligned sector
    const bool band = (dir & MXFP8_COL) && col_aligned && (q.off != nullptr || FP8Q_MX_BAND_UNGROUPED);
    return band ? launch_tma_layout<FMT, kBandKernel>(q, dir, ext, s)
                : launch_tma_layout<FMT, kUnitKernel>(q, dir, ext, s);
  }
  if (dir == MXFP8_ROW) return launch_f32<FMT, MXFP8_ROW>(p, s);
  if (dir == MXFP8_COL) return launch_f32<FMT, MXFP8_COL>(p, s);
  return launch_f32<FMT, MXFP8_BOTH>(p, s);
}

fp8q_status launch_mx(const void* x, int dt, int64_t rows, int64_t cols, const int64_t* off, int G, int fmt,
                      int dir, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, int64_t s_col_ld,
                      int round_up, unsigned long long* sat, int mma_layout, cudaStream_t stream) {
  MxParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.off = off;
  p.G = off ? G : 1;
  p.strips = (cols + kTileCols - 1) / kTileCols;
  p.super = 1;
  p.q_row = q_row;
  p.s_row = s_row;
  p.q_col = q_col;
  p.s_col = s_col;
  p.s_col_ld = s_col_ld;
  p.round_up = round_up;
  p.sat = sat;
  p.mma = mma_layout;
  p.row_bcols = (cols / 32 + 3) / 4;
  p.col_bcols = (s_col_ld + 3) / 4;
  return fmt == kE4M3 ? launch_fmt<kE4M3>(p, dt, dir, stream) : launch_fmt<kE5M2>(p, dt, dir, stream);
}

fp8q_status mx_device_status(cudaStream_t stream, bool clear, unsigned* word) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_mx_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (clear && v) {
    const unsigned z = 0;
    e = cudaMemcpyToSymbol(g_mx_error, &z, sizeof(z));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
  }
  *word = v;
  return FP8Q_OK;
}

fp8q_status mx_set_stall_producer(bool on) {
  const unsigned v = on ? 1u : 0u;
  cudaError_t e = cudaMemcpyToSymbol(g_mx_stall_producer, &v, sizeof(v));
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, "cudaMemcpyToSymbol(stall hook)");
}

fp8q_status mx_set_wait_budget(unsigned long long ns) {
  cudaError_t e = cudaMemcpyToSymbol(g_wait_budget_ns, &ns, sizeof(ns));
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, "cudaMemcpyToSymbol(wait budget)");
}

}  // namespace fp8q
