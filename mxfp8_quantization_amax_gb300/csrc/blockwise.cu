// blockwise.cu -- blockwise FP8 with one FP32 scale per group: 1x128 groups
// (activations: 128 channels of one token), their 128x1 transposed copy, and
// 128x128 blocks (weights), BF16 input.
//
// "混合精度与 FP8 训练" 10.2: activations are grouped 1x128 and weights
// 128x128 along the GEMM reduction dimension; 10.3: every tensor in E4M3,
// the scale computed online from each group's amax; 10.4: scales may be
// integer powers of two; 10.5: a 1x128 result cannot be transposed into a
// 128x1 one, so the transposed copy is quantized from the high-precision
// tensor, while a 128x128 block transposes as it is.  Per group: amax, the
// current-scaling scale F8max / amax ("HiFloat8：高性能训练之路" 1.2, eq. 1,
// with the per-tensor special cases), optionally rounded down to a power of
// two, q = RNE_sat(fl32(x * scale)), and scale_inv = fl32(1 / scale) stored.
//
// Kernel.  Persistent and warp-specialised.  A tile is 128 rows x 128
// columns (one 128x128 block, 128 row groups, 128 column groups), loaded by
// one producer lane as two 2-D TMA boxes of 64 columns x 128 rows (128-byte
// swizzle) into a two-stage ring.  Eight consumer warps quantize:
//   * row groups: a half-warp owns one row (8 columns per lane, one 16-byte
//     shared load), reduces the amax over its 16 lanes and stores the row's
//     128 codes as 16 lanes x 8 bytes;
//   * column groups: a thread owns a column pair over 32 rows (one 4-byte
//     word per row, both columns), the four row quarters combine their
//     amaxes in shared memory, and each column's 32 codes leave as two
//     16-byte stores into the transposed output;
//   * 128x128 blocks: the tile's amax is reduced over all consumers first.
// Consumer barriers are named barriers among the consumer warps only; every
// bounded wait's outcome is combined over all of them first (bar.red.or), so
// they give up together and no barrier is left waiting.
#include <cudaTypedefs.h>

#include <mutex>

#include "fp8q_device.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fp8q {

constexpr int kBwTile = 128;
constexpr int kBwBoxCols = 64;
constexpr int kBwBoxBytes = kBwTile * 128;      // 128 rows x 128 bytes
constexpr int kBwStageBytes = 2 * kBwBoxBytes;  // 32 KB
constexpr int kBwStages = 2;
constexpr int kBwConsumers = 256;
constexpr int kBwThreads = kBwConsumers + 32;
constexpr int kBwBarCons = 1;  // named barrier ids among the consumers
constexpr int kBwBarOr = 2;

__device__ unsigned int g_bw_error;
__device__ unsigned long long g_bw_wait_budget_ns = 1000000000ull;

struct BwParams {
  int64_t rows, cols;
  int64_t tiles_r, tiles_c;  // ceil(rows / 128), ceil(cols / 128)
  int pow2;
  uint8_t* q;     // [rows][cols]
  float* s;       // 1x128: [rows][tiles_c]; 128x128: [tiles_r][tiles_c]
  uint8_t* q_t;   // [cols][rows]
  float* s_t;     // 128x1: [cols][tiles_r]; 128x128: [tiles_c][tiles_r]
};

// Byte offset in a stage of the 16-byte chunk part holding row r, column c
// (c even): box c / 64, then the 128-byte row line with its chunks swizzled.
__device__ __forceinline__ uint32_t bw_off(int r, int c) {
  const int b = (c & 63) * 2;
  return (uint32_t)((c >> 6) * kBwBoxBytes + r * 128 + ((((b >> 4) ^ (r & 7)) << 4) | (b & 15)));
}

template <int FMT>
__device__ __forceinline__ float bw_scale(uint32_t amax_bits, int pow2) {
  float s = scale_from_amax(amax_bits, Fmt<FMT>::kMax, 0);
  if (pow2) s = __uint_as_float(__float_as_uint(s) & 0xFF800000u);  // s is a positive normal float
  return s;
}

// Magnitude bits (as FP32 bits) of the largest of 8 BF16 values.
__device__ __forceinline__ uint32_t amax8(const uint4& v) {
  const uint32_t m = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(0u, v.x), v.y), v.z), v.w);
  return max(m << 16, m & 0xFFFF0000u);
}

template <int FMT>
__device__ __forceinline__ uint32_t codes4(float a, float b, float c, float d, float s) {
  return canon_nan4<FMT>(cvt4<FMT>(__fmul_rn(a, s), __fmul_rn(b, s), __fmul_rn(c, s), __fmul_rn(d, s)));
}

// Row pass: rows of the tile in 8 sweeps of 16 (a warp takes 2 rows, one
// per half-warp).  BLOCK 1: each row is a group; 128: every row uses s_tile.
template <int FMT, int BLOCK>
__device__ __forceinline__ void bw_rows(const BwParams& p, const unsigned char* st, int64_t r0, int64_t c0,
                                        float s_tile, int ctid) {
  const int w = ctid >> 5, l = ctid & 31, half = l >> 4, hl = l & 15;
  const int c = hl * 8;
  const bool col_ok = c0 + c < p.cols;
#pragma unroll 2
  for (int pass = 0; pass < kBwTile / 16; pass++) {
    const int r = pass * 16 + w * 2 + half;
    const uint4 v = *(const uint4*)(st + bw_off(r, c));
    float s = s_tile;
    if constexpr (BLOCK == 1) {
      uint32_t a = amax8(v);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
      s = bw_scale<FMT>(a, p.pow2);
      if (hl == 0 && r0 + r < p.rows) p.s[(r0 + r) * p.tiles_c + c0 / kBwTile] = __frcp_rn(s);
    }
    if (r0 + r < p.rows && col_ok) {
      uint2 o;
      o.x = codes4<FMT>(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), s);
      o.y = codes4<FMT>(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w), s);
      st_stream(p.q + (r0 + r) * p.cols + c0 + c, o);
    }
  }
}

// Column pass: thread = (column pair, row quarter).  BLOCK 1: each column is
// a group of 128 rows; 128: both columns use s_tile (the transposed block).
template <int FMT, int BLOCK>
__device__ __forceinline__ void bw_cols(const BwParams& p, const unsigned char* st, int64_t r0, int64_t c0,
                                        float s_tile, int ctid, uint32_t* sh_amax) {
  const int pp = ctid & 63, h = ctid >> 6;
  const int c = 2 * pp;
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; i++) {
    const int r = 32 * h + i;
    w[i] = *(const uint32_t*)(st + bw_off(r, c));
  }
  float s0 = s_tile, s1 = s_tile;
  if constexpr (BLOCK == 1) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; i++) m = absmax_bf16x2(m, w[i]);
    sh_amax[h * kBwTile + c] = (m & 0xFFFFu) << 16;
    sh_amax[h * kBwTile + c + 1] = m & 0xFFFF0000u;
    named_barrier_sync(kBwBarCons, kBwConsumers);
    uint32_t a0 = 0, a1 = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) {
      a0 = max(a0, sh_amax[k * kBwTile + c]);
      a1 = max(a1, sh_amax[k * kBwTile + c + 1]);
    }
    named_barrier_sync(kBwBarCons, kBwConsumers);  // sh_amax is rewritten by the next tile
    s0 = bw_scale<FMT>(a0, p.pow2);
    s1 = bw_scale<FMT>(a1, p.pow2);
    if (h == 0 && c0 + c < p.cols) {
      p.s_t[(c0 + c) * p.tiles_r + r0 / kBwTile] = __frcp_rn(s0);
      p.s_t[(c0 + c + 1) * p.tiles_r + r0 / kBwTile] = __frcp_rn(s1);
    }
  }
  if (c0 + c >= p.cols) return;
  uint32_t d0[8], d1[8];
#pragma unroll
  for (int k = 0; k < 8; k++) {
    d0[k] = codes4<FMT>(bf16_lo(w[4 * k]), bf16_lo(w[4 * k + 1]), bf16_lo(w[4 * k + 2]), bf16_lo(w[4 * k + 3]), s0);
    d1[k] = codes4<FMT>(bf16_hi(w[4 * k]), bf16_hi(w[4 * k + 1]), bf16_hi(w[4 * k + 2]), bf16_hi(w[4 * k + 3]), s1);
  }
  const int64_t rr = r0 + 32 * h;
  uint8_t* t0 = p.q_t + (c0 + c) * p.rows + rr;
  uint8_t* t1 = t0 + p.rows;
  if (rr < p.rows) {
    st_stream(t0, make_uint4(d0[0], d0[1], d0[2], d0[3]));
    st_stream(t1, make_uint4(d1[0], d1[1], d1[2], d1[3]));
  }
  if (rr + 16 < p.rows) {
    st_stream(t0 + 16, make_uint4(d0[4], d0[5], d0[6], d0[7]));
    st_stream(t1 + 16, make_uint4(d1[4], d1[5], d1[6], d1[7]));
  }
}

template <int FMT, int BLOCK, int DIR>
__global__ void __launch_bounds__(kBwThreads, 3) blockwise_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                  BwParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[kBwStages], empty[kBwStages];
  __shared__ uint32_t sh_amax[4 * kBwTile];
  __shared__ uint32_t sh_red[kBwConsumers / 32];
  __shared__ volatile int abort_flag;
  unsigned char* stages = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kBwStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kBwConsumers / 32);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (tid == kBwConsumers) prefetch_tensormap(&tmap);
  pdl_wait();
  __syncthreads();
  const int64_t tiles = p.tiles_r * p.tiles_c;
  const uint64_t budget = g_bw_wait_budget_ns;

  if (warp == kBwConsumers / 32) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    int64_t k = 0;
    for (int64_t t = blockIdx.x; t < tiles && !abort_flag; t += gridDim.x, ++k) {
      const int s = (int)(k % kBwStages);
      const uint32_t round = (uint32_t)(k / kBwStages);
      if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1u, budget)) {
        atomicOr(&g_bw_error, 1u);
        abort_flag = 1;
        break;
      }
      const int64_t tr = t / p.tiles_c, tc = t - tr * p.tiles_c;
      mbar_arrive_expect_tx(&full[s], kBwStageBytes);
      unsigned char* dst = stages + s * kBwStageBytes;
      tma_load_2d(dst, &tmap, (int)(tc * kBwTile), (int)(tr * kBwTile), &full[s]);
      tma_load_2d(dst + kBwBoxBytes, &tmap, (int)(tc * kBwTile + kBwBoxCols), (int)(tr * kBwTile), &full[s]);
    }
    pdl_launch_dependents();
    // every issued copy lands before the CTA can exit (fixed 2 s bound)
    const int64_t first = k > kBwStages ? k - kBwStages : 0;
    for (int64_t j = first; j < k; j++)
      mbar_wait(&full[j % kBwStages], (uint32_t)((j / kBwStages) & 1), 2000000000ull);
    return;
  }

  // ---------------- consumers ----------------
  int64_t k = 0;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++k) {
    const int s = (int)(k % kBwStages);
    const uint32_t round = (uint32_t)(k / kBwStages);
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[s], round & 1u, budget));
    // one decision for all consumer warps, so none is left at a barrier
    if (named_barrier_or(kBwBarOr, kBwConsumers, !ok || abort_flag)) {
      if (tid == 0) atomicOr(&g_bw_error, 1u);
      abort_flag = 1;
      return;
    }
    const int64_t tr = t / p.tiles_c, tc = t - tr * p.tiles_c;
    const int64_t r0 = tr * kBwTile, c0 = tc * kBwTile;
    const unsigned char* st = stages + s * kBwStageBytes;
    float s_tile = 1.0f;
    if constexpr (BLOCK == kBwTile) {  // the tile's amax over all consumers
      uint32_t a = 0;
      const int hl = lane & 15, half = lane >> 4;
#pragma unroll 4
      for (int pass = 0; pass < kBwTile / 16; pass++)
        a = max(a, amax8(*(const uint4*)(st + bw_off(pass * 16 + warp * 2 + half, hl * 8))));
      a = warp_max_u32(a);
      if (lane == 0) sh_red[warp] = a;
      named_barrier_sync(kBwBarCons, kBwConsumers);
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < kBwConsumers / 32; i++) m = max(m, sh_red[i]);
      named_barrier_sync(kBwBarCons, kBwConsumers);  // sh_red is rewritten by the next tile
      s_tile = bw_scale<FMT>(m, p.pow2);
      if (tid == 0) {
        if (DIR & MXFP8_ROW) p.s[tr * p.tiles_c + tc] = __frcp_rn(s_tile);
        if (DIR & MXFP8_COL) p.s_t[tc * p.tiles_r + tr] = __frcp_rn(s_tile);
      }
    }
    if constexpr (DIR & MXFP8_ROW) bw_rows<FMT, BLOCK>(p, st, r0, c0, s_tile, tid);
    if constexpr (DIR & MXFP8_COL) bw_cols<FMT, BLOCK>(p, st, r0, c0, s_tile, tid, sh_amax);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 bw_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}

template <int FMT, int BLOCK, int DIR>
static fp8q_status launch_bw_t(const CUtensorMap& map, const BwParams& p, cudaStream_t s) {
  const size_t smem = 1024 + (size_t)kBwStages * kBwStageBytes;
  static int per_sm = [smem] {
    int v = 0;
    if (cudaFuncSetAttribute(blockwise_kernel<FMT, BLOCK, DIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, blockwise_kernel<FMT, BLOCK, DIR>, kBwThreads, smem) !=
            cudaSuccess ||
        v < 1)
      v = 1;
    return v;
  }();
  int64_t grid = (int64_t)per_sm * sm_count();
  const int64_t tiles = p.tiles_r * p.tiles_c;
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  const cudaError_t e = launch_kernel(blockwise_kernel<FMT, BLOCK, DIR>, dim3((unsigned)grid), dim3(kBwThreads),
                                      smem, s, map, p);
  if (e != cudaSuccess) return cuda_fail(e, "blockwise kernel launch");
  return check_launch("blockwise kernel");
}

template <int FMT, int BLOCK>
static fp8q_status launch_bw_dir(const CUtensorMap& map, const BwParams& p, int dir, cudaStream_t s) {
  if (dir == MXFP8_ROW) return launch_bw_t<FMT, BLOCK, MXFP8_ROW>(map, p, s);
  if (dir == MXFP8_COL) return launch_bw_t<FMT, BLOCK, MXFP8_COL>(map, p, s);
  return launch_bw_t<FMT, BLOCK, MXFP8_BOTH>(map, p, s);
}

fp8q_status launch_blockwise(const void* x, int64_t rows, int64_t cols, int fmt, int block, int pow2, int dir,
                             uint8_t* q, float* s, uint8_t* q_t, float* s_t, cudaStream_t stream) {
  auto enc = bw_encode_fn();
  if (!enc) return fail(FP8Q_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap map;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {kBwBoxCols, kBwTile};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FP8Q_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  BwParams p{};
  p.rows = rows;
  p.cols = cols;
  p.tiles_r = (rows + kBwTile - 1) / kBwTile;
  p.tiles_c = (cols + kBwTile - 1) / kBwTile;
  p.pow2 = pow2;
  p.q = q;
  p.s = s;
  p.q_t = q_t;
  p.s_t = s_t;
  if (fmt == kE4M3)
    return block == 1 ? launch_bw_dir<kE4M3, 1>(map, p, dir, stream) : launch_bw_dir<kE4M3, kBwTile>(map, p, dir, stream);
  return block == 1 ? launch_bw_dir<kE5M2, 1>(map, p, dir, stream) : launch_bw_dir<kE5M2, kBwTile>(map, p, dir, stream);
}

fp8q_status bw_device_status(bool clear, unsigned* word) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_bw_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (clear && v) {
    const unsigned z = 0;
    e = cudaMemcpyToSymbol(g_bw_error, &z, sizeof(z));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
  }
  *word = v;
  return FP8Q_OK;
}

fp8q_status bw_set_wait_budget(unsigned long long ns) {
  cudaError_t e = cudaMemcpyToSymbol(g_bw_wait_budget_ns, &ns, sizeof(ns));
  return e == cudaSuccess ? FP8Q_OK : cuda_fail(e, "cudaMemcpyToSymbol(wait budget)");
}

}  // namespace fp8q
