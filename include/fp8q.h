/*
 * fp8q.h -- C ABI of libfp8q, FP8 / MXFP8 quantization for sm_103a (GB300).
 *
 * The library quantizes BF16 or FP32 tensors to 8-bit floats, the step that
 * runs before each Fprop / Dgrad / Wgrad matmul of FP8 training:
 *   - per-tensor amax, current scaling and delayed scaling, each followed by
 *     a saturating round-to-nearest-even cast to E4M3 or E5M2;
 *   - MXFP8: 1x32 blocks with one E8M0 scale each (exponent rounded up),
 *     rowwise and columnwise (transposed), optionally per ragged group;
 * and the steps around it: dequantization, blockwise FP8, NVFP4, and the
 * SQNR / zero-rate statistics of a quantized copy.
 *
 * Conventions for every entry point:
 *   - Pointers documented as "device" are CUDA device pointers owned by the
 *     caller; the library never frees them and never allocates on these
 *     calls (only fp8q_delayed_create allocates, for its own state).
 *   - All work is asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = the legacy default stream).  Return codes report argument
 *     validation and launch errors only; fp8q_last_error_string() gives the
 *     message of the most recent failure on the calling thread.
 *   - Inputs are contiguous row-major tensors; x must be 16-byte aligned.
 *     dt selects the element type: FP8Q_IN_BF16 (raw BF16 bits) or
 *     FP8Q_IN_FP32.  Outputs are raw 8-bit codes (uint8).
 *   - Groups: group_offsets is a device int64 array of num_groups + 1 row
 *     offsets, non-decreasing, from 0 to rows; group g is rows
 *     [offsets[g], offsets[g+1]).  NULL means one group of all rows
 *     (num_groups must then be 1).  Offsets that break these rules give
 *     unspecified values but never an out-of-bounds access.
 *   - num_groups is at most FP8Q_MAX_GROUPS.
 *
 * Readings of the source pages that fix bit-level results (the same as the
 * CPU oracle's): a NaN input encodes to 0x7F in both formats; +-Inf and any
 * overflow saturate to +-max; the sign of zero is kept except in an all-zero
 * MX block; amax compares magnitude bits, so NaN inputs make amax NaN.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8Q_MAX_GROUPS 4096

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_INVALID_ARG = 1, /* a pointer, size, enum or alignment is invalid */
    FP8Q_ERR_UNSUPPORTED = 2, /* valid request the library does not handle (e.g. cols % 32 for MX) */
    FP8Q_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed */
    FP8Q_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up */
} fp8q_status;

typedef enum { FP8Q_IN_BF16 = 0, FP8Q_IN_FP32 = 1 } fp8q_in_dtype;

/* E4M3: bias 7, no Inf, max 448.  E5M2: IEEE style, bias 15, max 57344.
 * ("混合精度与 FP8 训练", 2.2; "Blackwell GPU MXFP8 预训练最佳实践", 3.1)
 * MX element formats below 8 bits, for mx_quantize_fp4_fp6 only: E2M1
 * (MXFP4: 0, 0.5, 1, 1.5, 2, 3, 4, 6; "混合精度与 FP8 训练" 13.2) and the
 * MXFP6 pair E2M3 (bias 1, max 7.5) and E3M2 (bias 3, max 28), read as the
 * OCP microscaling formats that "Blackwell GPU MXFP8 预训练最佳实践" 3.2
 * names without defining.  None has Inf or NaN. */
typedef enum { FP8Q_E4M3 = 0, FP8Q_E5M2 = 1, FP8Q_E2M1 = 2, FP8Q_E2M3 = 3, FP8Q_E3M2 = 4 } fp8q_format;

typedef enum { MXFP8_ROW = 1, MXFP8_COL = 2, MXFP8_BOTH = 3 } mxfp8_dir;

/* MX scale rule.  FP8Q_MX_RULE_UP: X = ceil(log2(amax / destmax)), the
 * round-up rule ("Blackwell GPU MXFP8 预训练最佳实践" 4.1, Algorithm 1);
 * FP8Q_MX_RULE_OCP: X = floor(log2(amax)) - e_max, the OCP rule ("混合精度与
 * FP8 训练" 13.1; e_max = 8 for E4M3, 15 for E5M2), which can put elements
 * above the format maximum (they saturate).  Both saturate X to [-127, 127]. */
typedef enum { FP8Q_MX_RULE_UP = 0, FP8Q_MX_RULE_OCP = 1 } fp8q_mx_rule;

/* Blockwise group shapes.  FP8Q_BLOCK_1X128: 1x128 groups (one token's 128
 * channels) for the rowwise copy, 128x1 groups for the transposed copy;
 * FP8Q_BLOCK_128X128: 128x128 blocks, whose transposed copy is the same
 * blocks transposed. */
typedef enum { FP8Q_BLOCK_1X128 = 1, FP8Q_BLOCK_128X128 = 128 } fp8q_block;

/* Output type of the dequantizers. */
typedef enum { FP8Q_OUT_BF16 = 0, FP8Q_OUT_FP32 = 1 } fp8q_out_dtype;

/* Library version (major * 10000 + minor * 100 + patch). */
FP8Q_API int32_t fp8q_version(void);

/* Message of the last failed call on this thread ("" if none). */
FP8Q_API const char* fp8q_last_error_string(void);

/*
 * Synchronizes `stream`, then reports and clears device-side failures that
 * earlier calls on this device recorded: FP8Q_ERR_TIMEOUT when a bounded
 * wait inside a kernel (the shared-memory barriers of the MXFP8 and the
 * blockwise pipelines, the grid-wide wait for the scale in the single-launch
 * current scaling) gave up, in which case that call's outputs are
 * incomplete.  FP8Q_OK otherwise.
 */
FP8Q_API fp8q_status fp8q_check_device(void* stream);

/*
 * Time budget of every bounded device-side wait, in nanoseconds (default
 * 1e9), for kernels launched afterwards on the current device.  Waits never
 * spin longer than this; a stalled pipeline ends its kernel and is reported
 * by fp8q_check_device.
 */
FP8Q_API fp8q_status fp8q_set_wait_budget_ns(uint64_t ns);

/*
 * Test hook for the failure path above (the pages have no counterpart).
 * While `on` is nonzero, the BF16 MXFP8 kernel's producer warp issues no
 * loads, so its consumers' waits for data can never complete: each gives up
 * after the wait budget, the call's outputs are left unwritten and
 * fp8q_check_device reports FP8Q_ERR_TIMEOUT.  No copy is in flight when
 * the kernel ends.  Applies to kernels launched afterwards on the current
 * device; leave it off (the default) outside such tests.
 */
FP8Q_API fp8q_status fp8q_debug_stall_mx_producer(int32_t on);

/*
 * Test hook for the same failure path in the single-launch current scaling
 * of fp8q_cast_per_tensor (taken for an ungrouped tensor of more than 2 MB
 * and up to about 160M BF16 elements; smaller ones take a one-cluster
 * kernel that has no grid-wide wait).  While `on` is nonzero, the CTA
 * that should publish the scale does not, so every other CTA's wait for it
 * gives up after the wait budget: no codes are written, fp8q_check_device
 * reports FP8Q_ERR_TIMEOUT, and the workspace is zero-filled again by the
 * last CTA to leave.  Applies to kernels launched afterwards on the current
 * device; leave it off (the default) outside such tests.
 */
FP8Q_API fp8q_status fp8q_debug_stall_scale_publish(int32_t on);

/*
 * amax_out[g] = max |x| over group g, bit-exact: the FP32 value whose bits
 * are the largest magnitude bits in the group (BF16 widened exactly), so a
 * NaN makes the result NaN and an empty group gives 0.
 * ("HiFloat8：高性能训练之路" 1.2, ComputeAmax; "混合精度与 FP8 训练" 8.1.)
 *   x           device, rows*cols elements of type dt
 *   amax_out    device float[num_groups]
 * One reduction pass over x (2 or 4 bytes per element read).
 */
FP8Q_API fp8q_status fp8q_amax(const void* x, int32_t dt, int64_t rows, int64_t cols,
                      const int64_t* group_offsets, int32_t num_groups, float* amax_out,
                      void* stream);

/*
 * scale_out[g] = fl32(fl32(F8max / amax[g]) * 2^-margin) and
 * scale_inv_out[g] = fl32(1 / scale_out[g]), with the same special cases as
 * current scaling (amax 0 or non-finite -> scale 1; a quotient above FLT_MAX
 * -> FLT_MAX).  ("HiFloat8：高性能训练之路" 1.2, eqs. 1 and 3; "混合精度与 FP8
 * 训练" 8.2, the margin.)  It is the scale step of current scaling on its
 * own, for a tensor split across devices: each device takes fp8q_amax of
 * its part, the amaxes are combined with a MAX all-reduce (on the FP32 bit
 * patterns as int32, which keeps NaN), and each device casts its part with
 * fp8q_cast_per_tensor(scale_in = scale_out).
 *   amax           device float[num_groups] (taken by magnitude)
 *   scale_out      device float[num_groups]
 *   scale_inv_out  device float[num_groups] or NULL
 */
FP8Q_API fp8q_status fp8q_scale_from_amax(const float* amax, int32_t num_groups, int32_t fmt,
                                          int32_t margin, float* scale_out, float* scale_inv_out,
                                          void* stream);

/*
 * Bytes of workspace fp8q_cast_per_tensor needs for num_groups groups.
 */
FP8Q_API size_t fp8q_cast_workspace_bytes(int32_t num_groups);

/*
 * Per-tensor (per-group) scaled cast:  q = RNE_sat(fl32(x * scale[g])).
 *
 * scale_in == NULL: current scaling ("HiFloat8：高性能训练之路" 1.2, eqs.
 *   1-2; "混合精度与 FP8 训练" 8.2): amax[g] is reduced first, then
 *   scale[g] = fl32(fl32(F8max / amax[g]) * 2^-margin), with amax = 0 giving
 *   scale 1, a non-finite amax giving scale 1, and an overflowing quotient
 *   giving FLT_MAX.  Two passes over x (read, read + write) in two
 *   launches, except for an ungrouped tensor of up to about 160M BF16
 *   elements on a GB300, which takes one launch: up to 2 MB of x, one
 *   thread-block cluster of 16 CTAs holds it in shared memory and
 *   exchanges the amax between them; beyond that, the 32 KB slices that
 *   fit one or two per resident CTA (about 20M elements) stay on chip
 *   (registers, shared memory) while the scale is published and are read
 *   once, and the rest of the tensor is streamed by the same CTAs and read
 *   twice, partly from L2.
 * scale_in != NULL: device float[num_groups] scales are used as given; if
 *   amax_out is non-NULL the amax of x is reduced in the same single pass.
 *
 *   x              device, rows*cols elements of type dt
 *   fmt            FP8Q_E4M3 or FP8Q_E5M2
 *   margin         0..63
 *   q              device uint8[rows*cols], same layout as x
 *   amax_out       device float[G] or NULL
 *   scale_out      device float[G] or NULL: the scale used
 *   scale_inv_out  device float[G] or NULL: fl32(1 / scale)
 *   sat_count_out  device uint64[G] or NULL: elements with |fl32(x*scale)|
 *                  > F8max (NaN not counted), i.e. clamped by the cast
 *   workspace      device, >= fp8q_cast_workspace_bytes(num_groups) bytes,
 *                  8-byte aligned, zero-filled before its first use; every
 *                  successful call leaves it zero-filled again (after a
 *                  call that fp8q_check_device reports as timed out, fill
 *                  it with zeros again).  Calls that may overlap on the GPU
 *                  need separate workspaces.
 */
FP8Q_API fp8q_status fp8q_cast_per_tensor(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                 const int64_t* group_offsets, int32_t num_groups,
                                 int32_t fmt, int32_t margin, const float* scale_in,
                                 uint8_t* q, float* amax_out, float* scale_out,
                                 float* scale_inv_out, unsigned long long* sat_count_out,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * fp8q_cast_per_tensor without a caller workspace.  The source pages have
 * no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory where they quantize (a plugin inside a host
 * application whose allocator owns all device memory, or a step where a
 * cudaMalloc / cudaFree would synchronize the device).  It allocates
 * nothing: the workspace is a fixed 8 KB array in the library's device
 * memory, present on every GPU that loads the library until the process
 * exits.
 *   - Arguments and results are those of fp8q_cast_per_tensor, minus the
 *     workspace; num_groups must be at most 256 (FP8Q_ERR_INVALID_ARG
 *     otherwise).
 *   - The first call on each device looks up the array's device address
 *     and keeps it; make that first call before any stream capture.  A
 *     context reset (cudaDeviceReset) is not supported afterwards: the
 *     array may be reloaded at another address.
 *   - All calls on a device share the array.  A call checks its arguments
 *     first (a rejected call touches nothing), then clears the part it
 *     uses (one small zeroing kernel on `stream`).  Calls whose work may
 *     overlap on the GPU race on it: order them on one stream.
 */
FP8Q_API fp8q_status fp8q_cast_per_tensor_static_ws(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                                    const int64_t* group_offsets, int32_t num_groups,
                                                    int32_t fmt, int32_t margin, const float* scale_in,
                                                    uint8_t* q, float* amax_out, float* scale_out,
                                                    float* scale_inv_out, unsigned long long* sat_count_out,
                                                    void* stream);

/*
 * Delayed scaling ("HiFloat8：高性能训练之路" 1.2 eqs. 3-4 and section 3;
 * "混合精度与 FP8 训练" 8.2): a library-owned state holds an amax history
 * ring of history_len entries.  Step t:
 *   - if the history is empty (after create or reset): current scaling with
 *     no margin on x_t;
 *   - else scale = fl32(fl32(F8max / max(filled history)) * 2^-margin);
 *   - q_t = RNE_sat(fl32(x_t * scale));
 *   - if t % interval == 0 (t counted from create/reset), amax(x_t) is
 *     computed in the same pass and appended, dropping the oldest entry when
 *     the ring is full; a non-finite amax raises the state's flag.
 * The host keeps step, head and count, so the call never synchronizes.
 */
typedef struct fp8q_delayed_state fp8q_delayed_state;

/* Allocates the state on the current device (history_len 1..1024,
 * interval >= 1, margin 0..63).  That device owns the state: reset and step
 * must be called with it current (FP8Q_ERR_INVALID_ARG otherwise); get, set
 * and destroy switch to it themselves and restore the caller's device. */
FP8Q_API fp8q_status fp8q_delayed_create(int32_t history_len, int32_t interval, int32_t margin,
                                int32_t fmt, fp8q_delayed_state** out);
FP8Q_API fp8q_status fp8q_delayed_destroy(fp8q_delayed_state* st);
/* Empties the history and clears the flag (async on stream); step = 0. */
FP8Q_API fp8q_status fp8q_delayed_reset(fp8q_delayed_state* st, void* stream);
/*
 *   x, n            device, n elements of type dt
 *   q               device uint8[n]
 *   scale_used_out  device float[1] or NULL; scale_inv_out likewise
 *   amax_out        device float[1] or NULL: written on recording steps only
 *   sat_count_out   device uint64[1] or NULL
 * Consecutive steps on one state must be issued on one stream (or ordered).
 */
FP8Q_API fp8q_status fp8q_delayed_step(fp8q_delayed_state* st, const void* x, int32_t dt, int64_t n,
                              uint8_t* q, float* scale_used_out, float* scale_inv_out,
                              float* amax_out, unsigned long long* sat_count_out,
                              void* stream);
/* Copies the state to the host (synchronizes the state's device): history_host
 * float[history_len] (ring order), head (next slot), count (filled entries),
 * step, nonfinite flag.  Any output pointer may be NULL. */
FP8Q_API fp8q_status fp8q_delayed_get(const fp8q_delayed_state* st, float* history_host, int32_t* head,
                             int32_t* count, int64_t* step, int32_t* nonfinite);
/* Restores a state saved by fp8q_delayed_get (checkpoint resume); clears
 * the flag.  Synchronous. */
FP8Q_API fp8q_status fp8q_delayed_set(fp8q_delayed_state* st, const float* history_host, int32_t head,
                             int32_t count, int64_t step);

/*
 * Number of columnwise MX blocks per column: sum over groups of
 * ceil(n_g / 32), from HOST offsets (NULL: ceil(rows / 32)).  Returns -1 for
 * invalid offsets.
 */
FP8Q_API int64_t mxfp8_col_blocks(const int64_t* group_offsets_host, int32_t num_groups, int64_t rows);

/*
 * MXFP8 quantization ("Blackwell GPU MXFP8 预训练最佳实践" 4.1-4.2;
 * "混合精度与 FP8 训练" 13.1; "HiFloat8：高性能训练之路" 2), one pass over x.
 * Each block of k <= 32 values gets X = ceil(log2(amax / destmax)) computed
 * exactly and saturated to [-127, 127] (destmax 448 for E4M3, 57344 for
 * E5M2); the scale byte is X + 127 (E8M0), elements are RNE_sat(v / 2^X).
 * amax = 0 gives byte 0x00 and all-zero elements; a block holding Inf or
 * NaN gives byte 0xFF and elements 0x7F.
 *   rowwise (dir & MXFP8_ROW): blocks x[r, 32j .. 32j+31]
 *     q_row  device uint8[rows * cols]          (row-major, like x)
 *     s_row  device uint8[rows * (cols / 32)]   (row-major)
 *   columnwise (dir & MXFP8_COL): per group, blocks of 32 consecutive rows
 *     from the group's first row, the last one possibly shorter; taken from
 *     x itself, not from the rowwise copy; output transposed:
 *     q_col  device uint8[cols * rows]          q_col[c * rows + r]
 *     s_col  device uint8[cols * s_col_ld]      s_col[c * s_col_ld + b], b
 *            numbering the column blocks of all groups in order; s_col_ld
 *            must be >= mxfp8_col_blocks(...) for the offsets used (blocks
 *            past s_col_ld are not written); an s_col_ld that is a
 *            multiple of 16 keeps every scale row 16-byte aligned, which
 *            the grouped path stores faster
 * cols % 32 == 0 is required (FP8Q_ERR_UNSUPPORTED otherwise); rows is any.
 * x is 16-byte aligned and q_row 32-byte aligned (a block's 32 codes leave
 * in one 32-byte store; FP8Q_ERR_INVALID_ARG otherwise).  Pointers of the
 * unused direction may be NULL.  A rejected call writes nothing.
 */
FP8Q_API fp8q_status mxfp8_quantize(const void* x, int32_t dt, int64_t rows, int64_t cols,
                           const int64_t* group_offsets, int32_t num_groups, int32_t fmt,
                           int32_t dir, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                           uint8_t* s_col, int64_t s_col_ld, void* stream);

/*
 * mxfp8_quantize with a choice of scale rule (fp8q_mx_rule) and an optional
 * count of saturated elements: those whose scaled magnitude |v / 2^X|
 * exceeds the format maximum and are clamped to it ("Blackwell GPU MXFP8
 * 预训练最佳实践" 4.1 compares the two rules by exactly this saturation).
 *   sat_count  device uint64[2] or NULL: [0] rowwise copy, [1] columnwise
 *              copy; zeroed by the call, then accumulated on the stream.
 * Never saturates under FP8Q_MX_RULE_UP.  Other arguments as mxfp8_quantize.
 */
FP8Q_API fp8q_status mxfp8_quantize_rule(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                         const int64_t* group_offsets, int32_t num_groups, int32_t fmt,
                                         int32_t dir, int32_t scale_rule, uint8_t* q_row, uint8_t* s_row,
                                         uint8_t* q_col, uint8_t* s_col, int64_t s_col_ld,
                                         unsigned long long* sat_count, void* stream);

/*
 * Scale layouts of mxfp8_quantize_ex.  FP8Q_SCALES_ROW_MAJOR is the layout of
 * mxfp8_quantize.  FP8Q_SCALES_MMA_128X4 writes the same scales straight into
 * the 128 x 4 block layout that block-scaled tensor-core MMA reads, the
 * layout mx_scales_to_mma_layout produces from row-major scales (the pages
 * give none; "Blackwell GPU MXFP8 预训练最佳实践" 3.2 only says the tensor
 * cores take the MX types natively): the scale matrix is padded to 128-row
 * and 4-column multiples and cut into 512-byte blocks, stored block row by
 * block row; scale (r, c) sits at byte (r % 32) * 16 + (r / 32 % 4) * 4 +
 * c % 4 of its block.  Padding bytes are 0.
 */
typedef enum { FP8Q_SCALES_ROW_MAJOR = 0, FP8Q_SCALES_MMA_128X4 = 1 } fp8q_scale_layout;

/* Bytes of a scale matrix of rows x scale_cols in the 128 x 4 block layout:
 * ceil(rows / 128) * 128 * ceil(scale_cols / 4) * 4 (-1 for negative sizes). */
FP8Q_API int64_t mxfp8_mma_scale_bytes(int64_t rows, int64_t scale_cols);

/*
 * mxfp8_quantize_rule with a choice of scale layout (fp8q_scale_layout).
 * Under FP8Q_SCALES_MMA_128X4:
 *   s_row  device uint8[mxfp8_mma_scale_bytes(rows, cols / 32)]
 *   s_col  device uint8[mxfp8_mma_scale_bytes(cols, s_col_ld)], the columnwise
 *          scales as a cols x s_col_ld matrix; s_col_ld must be the column
 *          block count itself (mxfp8_col_blocks; checked without groups, a
 *          precondition with groups), so that no block index is padding
 * Both are written in full: the kernels store every scale and, for shapes
 * with padding (rows or cols not a multiple of 128, cols / 32 or s_col_ld
 * not a multiple of 4) and for FP32 input, the call clears the buffer with
 * one cudaMemsetAsync first.  Other arguments as mxfp8_quantize_rule.
 */
FP8Q_API fp8q_status mxfp8_quantize_ex(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                       const int64_t* group_offsets, int32_t num_groups, int32_t fmt,
                                       int32_t dir, int32_t scale_rule, int32_t scale_layout, uint8_t* q_row,
                                       uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, int64_t s_col_ld,
                                       unsigned long long* sat_count, void* stream);

/*
 * MXFP4 / MXFP6 quantization ("混合精度与 FP8 训练" 13.1-13.2; "Blackwell
 * GPU MXFP8 预训练最佳实践" 3.2 and 4.1): blocks of 32 elements with one E8M0
 * scale, as mxfp8_quantize_rule but with element format elem (FP8Q_E2M1,
 * FP8Q_E2M3 or FP8Q_E3M2): destmax 6, 7.5 or 28 under FP8Q_MX_RULE_UP, e_max
 * 2, 2 or 4 under FP8Q_MX_RULE_OCP.  Elements are the nearest codes of
 * v / 2^X, saturating.  A block whose amax is 0 gets scale byte 0 and +0
 * codes; one holding Inf or NaN gets 0xFF and +0 codes.  One pass over x
 * writes both copies.  No groups.
 *   rowwise (dir & MXFP8_ROW):
 *     q_row  E2M1: device uint8 [rows][cols / 2], two codes per byte, the
 *                  even element in the low nibble; FP6: [rows][cols], one
 *                  code per byte in bits 0-5
 *     s_row  device uint8 [rows][cols / 32]
 *   columnwise (dir & MXFP8_COL): blocks of 32 rows (the last one shorter),
 *   stored transposed:
 *     q_col  E2M1: [cols][rows / 2] (rows must be even); FP6: [cols][rows]
 *     s_col  device uint8 [cols][ceil(rows / 32)]
 *   sat_count  device uint64[2] or NULL: elements whose |v / 2^X| exceeds
 *              destmax (clamped), [0] rowwise, [1] columnwise; zeroed by
 *              the call.  Never nonzero under FP8Q_MX_RULE_UP.
 * cols % 32 == 0 (FP8Q_ERR_UNSUPPORTED otherwise); q_row and q_col 16-byte
 * aligned; pointers of an unused copy may be NULL.
 */
FP8Q_API fp8q_status mx_quantize_fp4_fp6(const void* x, int32_t dt, int64_t rows, int64_t cols, int32_t elem,
                                         int32_t dir, int32_t scale_rule, uint8_t* q_row, uint8_t* s_row,
                                         uint8_t* q_col, uint8_t* s_col, unsigned long long* sat_count,
                                         void* stream);

/*
 * Blockwise FP8 with one FP32 scale per group ("混合精度与 FP8 训练" 10.2:
 * activations in 1x128 groups, weights in 128x128 blocks, along the GEMM
 * reduction dimension; 10.3: scales taken online from each group's amax;
 * 10.4: optionally integer powers of two; 10.5: the transposed copy of a
 * 1x128-grouped tensor is quantized from x in 128x1 groups, never from the
 * rowwise codes).  Per group: scale = fl32(F8max / amax) with the
 * per-tensor special cases (amax 0 or non-finite -> 1, overflow -> FLT_MAX),
 * rounded down to a power of two when pow2_scales is set; q =
 * RNE_sat(fl32(x * scale)); scale_inv = fl32(1 / scale) is stored.
 *   x            device BF16 [rows][cols]; rows % 16 == 0, cols % 16 == 0
 *                (FP8Q_ERR_UNSUPPORTED otherwise, and for FP32 input)
 *   block        fp8q_block
 *   dir          MXFP8_ROW, MXFP8_COL or MXFP8_BOTH
 *   q            device uint8 [rows][cols] (rowwise copy)
 *   scale_inv    device float: 1x128 -> [rows][ceil(cols/128)];
 *                128x128 -> [ceil(rows/128)][ceil(cols/128)]
 *   q_t          device uint8 [cols][rows] (transposed copy)
 *   scale_inv_t  device float: 128x1 -> [cols][ceil(rows/128)];
 *                128x128 -> [ceil(cols/128)][ceil(rows/128)]
 * Pointers of the unused copy may be NULL; x, q and q_t 16-byte aligned.
 */
FP8Q_API fp8q_status fp8q_quantize_blockwise(const void* x, int32_t dt, int64_t rows, int64_t cols, int32_t fmt,
                                             int32_t block, int32_t pow2_scales, int32_t dir, uint8_t* q,
                                             float* scale_inv, uint8_t* q_t, float* scale_inv_t, void* stream);

/*
 * NVFP4 ("混合精度与 FP8 训练" 13.2): E2M1 elements (0, 0.5, 1, 1.5, 2, 3,
 * 4, 6 and negatives), one E4M3 scale per 16 elements along a row, and one
 * FP32 scale for the tensor.  Each step is one IEEE single operation:
 *   S = 448 * 6 / amax(tensor)   (amax 0 or non-finite -> 1; overflow -> FLT_MAX)
 *   block code = RNE_sat_E4M3(amax_b * fl32(S / 6)), d = its value
 *   element = RNE_sat_E2M1(x * fl32(S / d)), all +0 when d is 0 or NaN
 * The value a code stands for is e2m1(q) * d / S.
 *   x          device BF16 or FP32 [rows][cols], cols % 16 == 0
 *   q          device uint8 [rows][cols / 2], two codes per byte, the even
 *              element in the low nibble (8-byte aligned)
 *   s          device uint8 [rows][cols / 16], E4M3 codes
 *   amax_out   device float[1], required: receives the tensor amax (it is
 *              the reduction's accumulator, zeroed by the call)
 *   scale_out  device float[1] or NULL: receives S
 * Two passes over x: the amax, then the quantization.
 */
FP8Q_API fp8q_status fp8q_quantize_nvfp4(const void* x, int32_t dt, int64_t rows, int64_t cols, uint8_t* q,
                                         uint8_t* s, float* amax_out, float* scale_out, void* stream);

/*
 * Block scales rearranged for block-scaled tensor-core MMA.  The pages give
 * no layout ("Blackwell GPU MXFP8 预训练最佳实践" 3.2 says only that the
 * tensor cores take the MX types natively); this is NVIDIA's public one.
 * The rows x scale_cols scale array is padded to multiples of 128 rows and
 * 4 columns and cut into 128 x 4 blocks of 512 bytes, stored block row by
 * block row; inside a block, scale (r, c) is byte (r % 32) * 16 + (r / 32)
 * * 4 + c.  Padding bytes are 0.
 *   s     device uint8 [rows][s_ld], the first scale_cols bytes of each row
 *         used (e.g. s_row [rows][cols / 32], s_col [cols][s_col_ld] with
 *         scale_cols = its block count, NVFP4 s [rows][cols / 16])
 *   out   device uint8 [ceil(rows / 128) * 128 * ceil(scale_cols / 4) * 4],
 *         4-byte aligned, fully written
 */
FP8Q_API fp8q_status mx_scales_to_mma_layout(const uint8_t* s, int64_t rows, int64_t scale_cols, int64_t s_ld,
                                             uint8_t* out, void* stream);

/*
 * Dequantization.  ("HiFloat8：高性能训练之路" 1.1-1.2: a quantized tensor is
 * de-scaled by scale_inv = 1 / Scale; "Blackwell GPU MXFP8 预训练最佳实践"
 * 4.1 and 4.3: an MX element stands for value * 2^X, X = byte - 127, and
 * without MX hardware the blocks are dequantized to BF16 for a BF16
 * matmul.)  Codes are decoded exactly.  BF16 output rounds to nearest, ties
 * to even; every NaN result is the canonical quiet NaN (BF16 0x7FC0, FP32
 * 0x7FC00000).  q and y must be 16-byte aligned; out_dt is FP8Q_OUT_BF16
 * (2 bytes per element) or FP8Q_OUT_FP32 (4 bytes).
 */

/*
 * y[i] = fl_out(fl32(value(q[i]) * scale_inv[g])) for the rows of group g.
 *   q          device uint8[rows*cols], the codes of fp8q_cast_per_tensor
 *   scale_inv  device float[num_groups]
 *   y          device BF16 or FP32 [rows*cols]
 */
FP8Q_API fp8q_status fp8q_dequantize_per_tensor(const uint8_t* q, int64_t rows, int64_t cols,
                                                const int64_t* group_offsets, int32_t num_groups,
                                                int32_t fmt, const float* scale_inv, int32_t out_dt,
                                                void* y, void* stream);

/*
 * One MX copy back to high precision: y = fl_out(value(q) * 2^(s - 127)),
 * scale byte 0xFF -> NaN.  rows x cols is the original tensor (cols % 32 ==
 * 0).
 *   dir MXFP8_ROW: q = q_row [rows][cols], s = s_row [rows][cols/32]
 *                  (s_ld ignored), y [rows][cols].
 *   dir MXFP8_COL: q = q_col [cols][rows], s = s_col [cols][s_ld] with the
 *                  column blocks of all groups in order, as mxfp8_quantize
 *                  wrote them; y [cols][rows], the copy's own (transposed)
 *                  layout.  Blocks past s_ld dequantize to NaN.
 */
FP8Q_API fp8q_status mxfp8_dequantize(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols,
                                      const int64_t* group_offsets, int32_t num_groups, int32_t fmt,
                                      int32_t dir, int64_t s_ld, int32_t out_dt, void* y, void* stream);

/*
 * Quantization-error statistics of a quantized copy against the tensor it
 * was made from ("昇腾 Ascend 950 低精度格式", appendix 3.4: formats are
 * compared by the per-layer SQNR and zero-rate of weights, activations and
 * KV cache).  xh is the FP32 value a code stands for: per-tensor
 * fl32(value(q) * scale_inv[g]); MX value(q) * 2^X rounded to FP32 (exact
 * unless it reaches 2^128, which gives Inf; scale byte 0xFF gives NaN).
 * Over the elements where x and xh are both finite:
 *   SQNR = 10 log10(signal / noise) dB,  zero-rate = n_flushed / n,
 * both computed on the device from the sums and counts (SQNR +inf for an
 * exact copy of a nonzero signal, NaN when signal and noise are both 0;
 * zero-rate 0 for an empty tensor).  Sums are exact to about 2e-6 relative
 * (FP32 sums of 32 elements added in FP64) and repeat exactly from run to
 * run on one GPU.
 */
typedef struct fp8q_qstats {
    double signal;                   /* sum of x^2 over the finite pairs */
    double noise;                    /* sum of (x - xh)^2 over the finite pairs */
    unsigned long long n;            /* elements compared */
    unsigned long long n_zero;       /* elements with xh == 0 */
    unsigned long long n_flushed;    /* xh == 0 while x != 0 (a NaN x is not 0) */
    unsigned long long n_nonfinite;  /* x or xh Inf or NaN: left out of the sums */
    double sqnr_db;                  /* 10 log10(signal / noise) */
    double zero_rate;                /* n_flushed / n */
} fp8q_qstats;

/* Bytes of workspace the statistics calls need (a constant, under 100 KB). */
FP8Q_API size_t fp8q_qstats_workspace_bytes(void);

/*
 * Statistics of a per-tensor (per-group) copy, one pass over x and q.
 *   x          device BF16 or FP32 [rows][cols] (16-byte aligned)
 *   q          device uint8 [rows][cols], 16-byte aligned (the codes of
 *              fp8q_cast_per_tensor)
 *   scale_inv  device float[num_groups]
 *   out        device fp8q_qstats, 8-byte aligned: written by the call
 *   workspace  device, >= fp8q_qstats_workspace_bytes() bytes, 16-byte
 *              aligned, zero-filled before its first use; every call leaves
 *              it ready for the next.  Calls that may overlap on the GPU
 *              need separate workspaces.
 * Rows outside every group are not compared.
 */
FP8Q_API fp8q_status fp8q_qstats_per_tensor(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                            const int64_t* group_offsets, int32_t num_groups, int32_t fmt,
                                            const uint8_t* q, const float* scale_inv, fp8q_qstats* out,
                                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Statistics of one MX copy of x (cols % 32 == 0), one pass over x and the
 * copy.  Layouts as mxfp8_quantize wrote them:
 *   dir MXFP8_ROW: q = q_row [rows][cols] (16-byte aligned), s = s_row
 *                  [rows][cols/32]; group_offsets and s_ld are not used.
 *   dir MXFP8_COL: q = q_col [cols][rows], s = s_col [cols][s_ld] with the
 *                  column blocks of all groups in order; element (c, r) of
 *                  the copy is compared with x[r][c].  Blocks past s_ld
 *                  count as NaN scales.
 * Other arguments as fp8q_qstats_per_tensor.
 */
FP8Q_API fp8q_status mxfp8_qstats(const void* x, int32_t dt, int64_t rows, int64_t cols,
                                  const int64_t* group_offsets, int32_t num_groups, int32_t fmt, int32_t dir,
                                  const uint8_t* q, const uint8_t* s, int64_t s_ld, fp8q_qstats* out,
                                  void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
