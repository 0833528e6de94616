// mxfp8.cu -- MXFP8 quantization, rowwise and columnwise, in one HBM pass.
//
// "Blackwell GPU MXFP8 预训练最佳实践" 4.1: per block of 32 values,
// X = ceil(log2(amax / destmax)) saturated to the E8M0 range, elements
// RNE_sat(v / 2^X), amax = 0 -> X = -127 with all elements 0.  4.2 and
// "HiFloat8：高性能训练之路" 2: every tensor needs a copy quantized along
// rows and one along columns (transposed), both from the high-precision
// tensor ("混合精度与 FP8 训练" 13.1: MX does not commute with transposes).
//
// Work unit: a tile of 32 rows x 256 columns.  The 32 rows are one
// columnwise block: for ragged groups (MoE experts) tiles start at each
// group's first row, the group's last tile may be shorter.  Each CTA
// (128 threads, persistent over units) does, per tile:
//   1. one 16-byte load per (row, 8 columns) from HBM into registers;
//   2. rowwise pass in registers: 4 lanes own one 1x32 block, the block
//      amax is a two-step shuffle, the E8M0 unit runs once per block, and
//      8 codes go out as one 8-byte store;
//   3. the raw tile goes to shared memory (row-major, 512 B per row, so row
//      stores and the column reads below are bank-conflict free);
//   4. columnwise pass: thread t owns columns 2t and 2t+1 and reads one
//      32-bit word (both columns) per row, so a single packed u16x2 max
//      gives both column amaxes; the 32 codes of each column are written
//      as two 16-byte stores into the transposed output.
// A shared-memory scan of the group sizes maps tile index -> (group, block).
#include "fp8q_device.cuh"
#include "internal.h"

namespace fp8q {

constexpr int kMxThreads = 128;
constexpr int kTileRows = 32;
constexpr int kTileCols = 256;
constexpr int kRowSlots = kTileRows / (kMxThreads / 32);  // rows per warp in the rowwise pass

struct MxParams {
  const void* x;
  int64_t rows, cols;
  const int64_t* off;  // device row offsets [G+1] or nullptr
  int G;
  int64_t strips;       // ceil(cols / 256)
  int64_t units;        // upper bound of tiles x strips
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t s_col_ld;
};

// Clamped group boundary: offsets outside [0, rows] are pulled back in, so
// tiles never leave the tensor whatever the caller passes.
__device__ __forceinline__ int64_t grp_row(const MxParams& p, int g) {
  if (p.off == nullptr) return g == 0 ? 0 : p.rows;
  int64_t v = __ldg(p.off + g);
  return v < 0 ? 0 : (v > p.rows ? p.rows : v);
}

// Write the first n (<= 32) bytes of d[0..7] to dst (any alignment).
__device__ __forceinline__ void store_col32(uint8_t* dst, const uint32_t (&d)[8], int n) {
  const uintptr_t a = (uintptr_t)dst;
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
    if (s >= 0 && s + 4 <= n) {
      *(uint32_t*)(base + 4 * k) = w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; i++)
        if (s + i >= 0 && s + i < n) base[4 * k + i] = (uint8_t)(w >> (8 * i));
    }
  }
}

template <int FMT>
__device__ __forceinline__ uint32_t mx_codes4(float a, float b, float c, float d, float mult) {
  return cvt4<FMT>(__fmul_rn(a, mult), __fmul_rn(b, mult), __fmul_rn(c, mult), __fmul_rn(d, mult));
}

// Final code word for a block: NaN block -> 0x7F..., zero block -> 0.
__device__ __forceinline__ uint32_t mx_fix(uint32_t w, uint32_t byte, uint32_t amax_bits) {
  w = byte == 0xFFu ? 0x7F7F7F7Fu : w;
  return amax_bits == 0u ? 0u : w;
}

template <int DT, int FMT, int DIR>
__global__ void __launch_bounds__(kMxThreads) mx_kernel(MxParams p) {
  constexpr int kElt = DT == kBF16 ? 2 : 4;
  constexpr int kRowBytes = kTileCols * kElt;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* tile = smem;                                      // [32][kRowBytes]
  int* prefix = (int*)(smem + kTileRows * kRowBytes);              // [G + 1]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- tile index -> (group, block): exclusive scan of ceil(n_g / 32) ----
  {
    __shared__ int warp_tot[kMxThreads / 32];
    const int per = (p.G + kMxThreads - 1) / kMxThreads;
    const int g_lo = tid * per, g_hi = min(p.G, g_lo + per);
    int sum = 0;
    for (int g = g_lo; g < g_hi; g++) {
      const int64_t n = grp_row(p, g + 1) - grp_row(p, g);
      sum += n > 0 ? (int)((n + 31) / 32) : 0;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; w++) base += warp_tot[w];
    int run = base + incl - sum;
    for (int g = g_lo; g < g_hi; g++) {
      prefix[g] = run;
      const int64_t n = grp_row(p, g + 1) - grp_row(p, g);
      run += n > 0 ? (int)((n + 31) / 32) : 0;
    }
    if (tid == kMxThreads - 1) prefix[p.G] = base + incl;
    __syncthreads();
  }
  const int total_tiles = prefix[p.G];
  const int64_t units = (int64_t)total_tiles * p.strips;
  const int64_t sblocks = p.cols / 32;

  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int t = (int)(u / p.strips);
    const int64_t c0 = (u - (int64_t)t * p.strips) * kTileCols;
    const int nc = (int)min((int64_t)kTileCols, p.cols - c0);
    // group of tile t: last g with prefix[g] <= t
    int lo = 0, hi = p.G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int b = t - prefix[g];
    const int64_t r0 = grp_row(p, g) + 32LL * b;
    const int nr = (int)min((int64_t)kTileRows, grp_row(p, g + 1) - r0);

    // ---- 1. loads: warp w covers rows w, w+4, ..; lane l covers 8 columns ----
    const bool col_ok = lane * 8 < nc;
    uint4 v[kRowSlots][kElt / 2];
#pragma unroll
    for (int i = 0; i < kRowSlots; i++) {
      const int r = warp + 4 * i;
      const bool ok = col_ok && r < nr;
      const char* src = (const char*)p.x + ((r0 + r) * p.cols + c0 + lane * 8) * kElt;
#pragma unroll
      for (int h = 0; h < kElt / 2; h++) v[i][h] = ok ? ld_stream(src + 16 * h) : make_uint4(0, 0, 0, 0);
    }

    // ---- 2. rowwise pass + 3. stage the tile ----
#pragma unroll
    for (int i = 0; i < kRowSlots; i++) {
      const int r = warp + 4 * i;
      if constexpr (DIR & MXFP8_ROW) {
        uint32_t am;
        if constexpr (DT == kBF16) {
          uint32_t m = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(0u, v[i][0].x), v[i][0].y),
                                                   v[i][0].z), v[i][0].w);
          am = max(m << 16, m & 0xFFFF0000u);
        } else {
          am = max(max(max(v[i][0].x & 0x7FFFFFFFu, v[i][0].y & 0x7FFFFFFFu),
                       max(v[i][0].z & 0x7FFFFFFFu, v[i][0].w & 0x7FFFFFFFu)),
                   max(max(v[i][1].x & 0x7FFFFFFFu, v[i][1].y & 0x7FFFFFFFu),
                       max(v[i][1].z & 0x7FFFFFFFu, v[i][1].w & 0x7FFFFFFFu)));
        }
        am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
        am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
        if (col_ok && r < nr) {
          const uint32_t byte = e8m0_from_amax<FMT>(am);
          const float mult = e8m0_multiplier(byte);
          uint2 o;
          if constexpr (DT == kBF16) {
            o.x = mx_codes4<FMT>(bf16_lo(v[i][0].x), bf16_hi(v[i][0].x), bf16_lo(v[i][0].y), bf16_hi(v[i][0].y), mult);
            o.y = mx_codes4<FMT>(bf16_lo(v[i][0].z), bf16_hi(v[i][0].z), bf16_lo(v[i][0].w), bf16_hi(v[i][0].w), mult);
          } else {
            o.x = mx_codes4<FMT>(__uint_as_float(v[i][0].x), __uint_as_float(v[i][0].y),
                                 __uint_as_float(v[i][0].z), __uint_as_float(v[i][0].w), mult);
            o.y = mx_codes4<FMT>(__uint_as_float(v[i][1].x), __uint_as_float(v[i][1].y),
                                 __uint_as_float(v[i][1].z), __uint_as_float(v[i][1].w), mult);
          }
          o.x = mx_fix(o.x, byte, am);
          o.y = mx_fix(o.y, byte, am);
          const int64_t row = r0 + r;
          st_stream(p.q_row + row * p.cols + c0 + lane * 8, o);
          if ((lane & 3) == 0) p.s_row[row * sblocks + (c0 + lane * 8) / 32] = (uint8_t)byte;
        }
      }
      if constexpr (DIR & MXFP8_COL) {
#pragma unroll
        for (int h = 0; h < kElt / 2; h++)
          *(uint4*)(tile + r * kRowBytes + lane * 8 * kElt + 16 * h) = v[i][h];
      }
    }

    // ---- 4. columnwise pass ----
    if constexpr (DIR & MXFP8_COL) {
      __syncthreads();
      const int cl = 2 * tid;  // this thread's first column within the tile
      if (cl < nc) {
        const int64_t gb = prefix[g] + b;  // block index within s_col rows
        const int64_t c = c0 + cl;
        uint32_t d0[8], d1[8];
        uint32_t a0, a1;
        if constexpr (DT == kBF16) {
          uint32_t w[kTileRows];
          uint32_t m = 0;
#pragma unroll
          for (int r = 0; r < kTileRows; r++) {
            w[r] = *(const uint32_t*)(tile + r * kRowBytes + cl * 2);
            m = absmax_bf16x2(m, w[r]);
          }
          a0 = m << 16;
          a1 = m & 0xFFFF0000u;
          const uint32_t b0 = e8m0_from_amax<FMT>(a0), b1 = e8m0_from_amax<FMT>(a1);
          const float m0 = e8m0_multiplier(b0), m1 = e8m0_multiplier(b1);
#pragma unroll
          for (int k = 0; k < 8; k++) {
            d0[k] = mx_fix(mx_codes4<FMT>(bf16_lo(w[4 * k]), bf16_lo(w[4 * k + 1]), bf16_lo(w[4 * k + 2]),
                                          bf16_lo(w[4 * k + 3]), m0), b0, a0);
            d1[k] = mx_fix(mx_codes4<FMT>(bf16_hi(w[4 * k]), bf16_hi(w[4 * k + 1]), bf16_hi(w[4 * k + 2]),
                                          bf16_hi(w[4 * k + 3]), m1), b1, a1);
          }
          store_col32(p.q_col + c * p.rows + r0, d0, nr);
          if (cl + 1 < nc) store_col32(p.q_col + (c + 1) * p.rows + r0, d1, nr);
          if (gb < p.s_col_ld) {
            p.s_col[c * p.s_col_ld + gb] = (uint8_t)b0;
            p.s_col[(c + 1) * p.s_col_ld + gb] = (uint8_t)b1;
          }
        } else {
          a0 = 0;
          a1 = 0;
#pragma unroll
          for (int r = 0; r < kTileRows; r++) {
            const uint2 w = *(const uint2*)(tile + r * kRowBytes + cl * 4);
            a0 = max(a0, w.x & 0x7FFFFFFFu);
            a1 = max(a1, w.y & 0x7FFFFFFFu);
          }
          const uint32_t b0 = e8m0_from_amax<FMT>(a0), b1 = e8m0_from_amax<FMT>(a1);
          const float m0 = e8m0_multiplier(b0), m1 = e8m0_multiplier(b1);
#pragma unroll
          for (int k = 0; k < 8; k++) {
            uint2 w0 = *(const uint2*)(tile + (4 * k) * kRowBytes + cl * 4);
            uint2 w1 = *(const uint2*)(tile + (4 * k + 1) * kRowBytes + cl * 4);
            uint2 w2 = *(const uint2*)(tile + (4 * k + 2) * kRowBytes + cl * 4);
            uint2 w3 = *(const uint2*)(tile + (4 * k + 3) * kRowBytes + cl * 4);
            d0[k] = mx_fix(mx_codes4<FMT>(__uint_as_float(w0.x), __uint_as_float(w1.x), __uint_as_float(w2.x),
                                          __uint_as_float(w3.x), m0), b0, a0);
            d1[k] = mx_fix(mx_codes4<FMT>(__uint_as_float(w0.y), __uint_as_float(w1.y), __uint_as_float(w2.y),
                                          __uint_as_float(w3.y), m1), b1, a1);
          }
          store_col32(p.q_col + c * p.rows + r0, d0, nr);
          if (cl + 1 < nc) store_col32(p.q_col + (c + 1) * p.rows + r0, d1, nr);
          if (gb < p.s_col_ld) {
            p.s_col[c * p.s_col_ld + gb] = (uint8_t)b0;
            p.s_col[(c + 1) * p.s_col_ld + gb] = (uint8_t)b1;
          }
        }
      }
      __syncthreads();  // the tile is rewritten by the next unit
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int DT, int FMT, int DIR>
static fp8q_status launch_mx_t(const MxParams& p, cudaStream_t s) {
  constexpr int kElt = DT == kBF16 ? 2 : 4;
  const size_t smem = (size_t)kTileRows * kTileCols * kElt + sizeof(int) * (p.G + 1);
  static int per_sm = -1;
  static size_t attr_smem = 0;
  if (smem > attr_smem) {
    cudaError_t e = cudaFuncSetAttribute(mx_kernel<DT, FMT, DIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(mx_kernel)");
    attr_smem = smem;
    per_sm = -1;
  }
  if (per_sm < 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mx_kernel<DT, FMT, DIR>, kMxThreads, smem) != cudaSuccess || n < 1)
      n = 1;
    per_sm = n;
  }
  int64_t grid = (int64_t)per_sm * sm_count();
  if (p.units < grid) grid = p.units;
  if (grid < 1) grid = 1;
  mx_kernel<DT, FMT, DIR><<<(unsigned)grid, kMxThreads, smem, s>>>(p);
  return check_launch("mxfp8 kernel");
}

template <int DT, int FMT>
static fp8q_status launch_mx_dir(const MxParams& p, int dir, cudaStream_t s) {
  if (dir == MXFP8_ROW) return launch_mx_t<DT, FMT, MXFP8_ROW>(p, s);
  if (dir == MXFP8_COL) return launch_mx_t<DT, FMT, MXFP8_COL>(p, s);
  return launch_mx_t<DT, FMT, MXFP8_BOTH>(p, s);
}

fp8q_status launch_mx(const void* x, int dt, int64_t rows, int64_t cols, const int64_t* off, int G,
                      int fmt, int dir, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                      int64_t s_col_ld, cudaStream_t stream) {
  MxParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.off = off;
  p.G = off ? G : 1;
  p.strips = (cols + kTileCols - 1) / kTileCols;
  p.units = ((rows + 31) / 32 + p.G) * p.strips;
  p.q_row = q_row;
  p.s_row = s_row;
  p.q_col = q_col;
  p.s_col = s_col;
  p.s_col_ld = s_col_ld;
  if (dt == kBF16) {
    return fmt == kE4M3 ? launch_mx_dir<kBF16, kE4M3>(p, dir, stream) : launch_mx_dir<kBF16, kE5M2>(p, dir, stream);
  }
  return fmt == kE4M3 ? launch_mx_dir<kFP32, kE4M3>(p, dir, stream) : launch_mx_dir<kFP32, kE5M2>(p, dir, stream);
}

}  // namespace fp8q
