/*
 * mq.h - C ABI of the GB300 (sm_103a) W4A4 + block-sparse 4-bit residual linear.
 *
 * The method: MosaicQuant, "Inlier-Outlier Disaggregation for Unified 4-Bit
 * LLM Quantization" (technical summary page).  The weight matrix W^ is
 * split into a dense 4-bit base Q(W^) and a sparse 4-bit residual R
 * (Metodologia 1); the residual budget is spent on 64x128 blocks chosen by a
 * Hessian-guided Delta-score, top-K (Metodologia 2); the ZipperEngine computes
 * the residual inside the dense 4-bit GEMM and reduce-adds the two partial
 * products (Metodologia 3).  The linear computed is
 *
 *     Y = Q(X) (Q(W^) + R^)^T,   R^ = 4-bit residual on the selected blocks.
 *
 * Formats (the pages fix none of them; these are this library's):
 *   - INT4 codes are symmetric, in [-7, 7]; two per byte, element 2j in the low
 *     nibble and 2j+1 in the high nibble, as 4-bit two's complement.
 *   - one fp16 scale per 128 inputs ("group"): per token for activations, per
 *     output row for base weights, per block row for residual blocks;
 *     scale = fp16_RNE(amax / 7) saturated to 65504, code = clamp(RNE(v/scale), -7, 7).
 *   - residual blocks are 64 output rows x 128 inputs (one group);
 *     Delta_b = sum_{k in block} h_k * sum_{n in block} R[n,k]^2 with
 *     h_k = mean over calibration rows of x_k^2; the top floor(budget * #blocks)
 *     blocks by Delta (ties: lower block index b = (n/64) * (K/128) + k/128) get
 *     a residual.
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated.  The caller owns every
 *     buffer; the library never allocates, frees or synchronizes (except
 *     mq_check_device_error, which synchronizes the given stream).
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).
 *   - Sizes: K % 128 == 0 and N % 128 == 0 (so N % 64 == 0 for residual
 *     blocks); M >= 1; K <= 2^20, N <= 2^20, M <= 2^20.
 *   - Errors are returned, never raised: MQ_ERR_INVALID_ARG for bad sizes or
 *     NULL pointers, MQ_ERR_ALIGNMENT for misaligned buffers,
 *     MQ_ERR_UNSUPPORTED_DEVICE when the current device is not compute
 *     capability 10.3, MQ_ERR_CUDA when a launch fails (detail in
 *     mq_last_error()).  Nothing is launched when an error is returned.
 *   - Device-side waits are bounded; a wait that runs out sets a device error
 *     word and the kernel returns early.  mq_check_device_error() reports it
 *     as MQ_ERR_TIMEOUT.
 */
#ifndef MQ_H_
#define MQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mq_stream_t; /* same as cudaStream_t */

typedef enum {
  MQ_OK = 0,
  MQ_ERR_INVALID_ARG = 1,
  MQ_ERR_ALIGNMENT = 2,
  MQ_ERR_UNSUPPORTED_DEVICE = 3,
  MQ_ERR_CUDA = 4,
  MQ_ERR_TIMEOUT = 5,
  MQ_ERR_WORKSPACE = 6
} mq_status;

typedef enum { MQ_F16 = 0, MQ_BF16 = 1, MQ_F32 = 2 } mq_dtype;

/* ------------------------------------------------------------------------ */
/* Online: activation quantizer (ZipperEngine's "quantization" stage,       */
/* Metodologia 3).                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Quantize X per token and per 128-input group.
 *   x    [M, ldx] MQ_F16 or MQ_BF16 (xt), row-major, row stride ldx >= K
 *        elements; x and ldx*2 bytes 8-byte aligned.  Values must be finite.
 *   Mp   = round_up(M, 8) (padding tokens m in [M, Mp) get zero codes and scales).
 *   xq   [K/128][Mp][64] bytes, group-major: byte (g*Mp + m)*64 + j holds the
 *        codes of token m, inputs 128g + 2j (low nibble) and 128g + 2j + 1
 *        (high nibble).  K*Mp/2 bytes, 16-byte aligned.
 *   xs   [K/128][Mp] fp16 scale bits: entry g*Mp + m is the scale of token m in
 *        group g.  16-byte aligned.
 *   (Group-major so the GEMM fetches a group's activation tile, codes and
 *   scales, with one bulk copy each.)
 * Bit-exact against the definition above: amax, amax/7 and v/scale are formed
 * in IEEE fp32 and each rounds to the same value the exact rational would.
 */
mq_status mq_quantize_act(const void* x, mq_dtype xt, int64_t M, int64_t K, int64_t ldx,
                          uint8_t* xq, uint16_t* xs, mq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Offline: Delta-score block selection (Metodologia 2) and packing          */
/* (Metodologia 1).                                                          */
/* ------------------------------------------------------------------------ */

/* floor(budget * (N/64) * (K/128) + 1e-9) clamped to [0, #blocks]; 0 for
 * budget <= 0 or invalid sizes.  Host-only, no device work. */
int64_t mq_num_selected(int64_t N, int64_t K, double budget);

/* Bytes of device workspace mq_select_blocks needs for (N, K). */
size_t mq_select_workspace_bytes(int64_t N, int64_t K);

/*
 * Select the residual blocks of W^ by Delta-score and write them as CSR over
 * 64-row block rows.
 *   w        [N, K] fp16 bits, row-major (the weight matrix W^).
 *   xcal     [C, K] calibration activations, MQ_F16 or MQ_BF16 (xct), C >= 1.
 *   budget   fraction of blocks in [0, 1].
 *   row_ptr  [N/64 + 1] int32: entries of block row br are
 *            col_idx[row_ptr[br] .. row_ptr[br+1]).
 *   col_idx  [mq_num_selected(N, K, budget)] int32 group index g, ascending
 *            within a row (may be NULL when that count is 0).
 *   h_out    optional [K] float64: the diagonal Hessian h_k.
 *   delta_out optional [(N/64)*(K/128)] float64: Delta_b, b = br*(K/128) + g.
 *   ws       workspace of at least mq_select_workspace_bytes(N, K) bytes,
 *            256-byte aligned (else MQ_ERR_WORKSPACE).
 * h and Delta are formed in float64 in a fixed order (ascending c, then
 * ascending rows, then ascending k) without fused multiply-add, so both are
 * reproducible bit for bit.
 */
mq_status mq_select_blocks(const uint16_t* w, int64_t N, int64_t K, const void* xcal,
                           mq_dtype xct, int64_t C, double budget, int32_t* row_ptr,
                           int32_t* col_idx, double* h_out, double* delta_out, void* ws,
                           size_t ws_bytes, mq_stream_t stream);

/* Bytes of one packed base-weight record (128 output rows x 128 inputs:
 * 8192 bytes of codes, then 128 fp16 scales) and of one packed residual-block
 * record (64 rows x 128 inputs: 4096 bytes of codes, then 64 fp16 scales). */
#define MQ_WREC_BYTES 8448
#define MQ_RREC_BYTES 4224

/*
 * Pack W^ into the dense 4-bit base and the 4-bit residual of the blocks
 * listed by (row_ptr, col_idx).
 *   w     [N, K] fp16 bits, row-major.
 *   nnzb  number of listed blocks (== row_ptr[N/64]); the host cannot read
 *         device row_ptr, so the caller passes it.
 *   wpk   base weights, (N/128)*(K/128) records of MQ_WREC_BYTES, record
 *           (t, g) at byte (t*(K/128) + g) * MQ_WREC_BYTES, for output rows
 *           128t..128t+127 and inputs of group g (16-byte aligned).  Inside a
 *           record:
 *             byte j*2048 + r*16 + b (j in [0,4), r in [0,128), b in [0,16))
 *               holds the codes of row 128t + r, inputs 128g + 32j + 2b (low
 *               nibble) and +1 (high nibble);
 *             bytes 8192 + 2r, +1: the fp16 scale of row 128t + r, group g.
 *           Consecutive groups of one row tile are consecutive records, so a
 *           run of groups, codes and scales, is one contiguous range.
 *   rpk   residual blocks, nnzb records of MQ_RREC_BYTES in CSR order
 *           (16-byte aligned).  Inside record i (block row br, group g):
 *             byte j*1024 + r*16 + b (r in [0,64)): row 64*br + r, inputs
 *               128g + 32j + 2b (low nibble) and +1 (high nibble);
 *             bytes 4096 + 2r, +1: the fp16 scale of block row r.
 * rpk may be NULL when nnzb == 0.
 */
mq_status mq_pack_weights(const uint16_t* w, int64_t N, int64_t K, const int32_t* row_ptr,
                          const int32_t* col_idx, int64_t nnzb, uint8_t* wpk, uint8_t* rpk,
                          mq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Online: the fused dense + sparse-residual GEMM (ZipperEngine,             */
/* Metodologia 3).                                                           */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace mq_w4a4_residual_gemm needs for (M, N, K).
 * From 128 tokens this includes the general kernel's image form: its
 * operand images (N*K bytes of E4M3 weights, residual images sized for the
 * densest block list, N*K bytes, and 128 bytes per padded token and
 * 128-input group), so the size does not depend on the block list.  A
 * caller that gives the GEMM less (mq_w4a4_residual_gemm_noalloc, whose
 * scratch is fixed) gets the converter form where the images do not fit. */
size_t mq_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Zero a GEMM workspace before its first use (and after an MQ_ERR_TIMEOUT);
 * the GEMM leaves it zeroed again on every normal exit. */
mq_status mq_gemm_workspace_init(void* ws, size_t ws_bytes, mq_stream_t stream);

/*
 *   Y[m, n] = sum_g sx[m,g] * ( sw[n,g] * Dw[m,n,g] + sr[n,g] * Dr[m,n,g] )
 * with the activation scales sx (xs), the base and residual scales sw, sr
 * (from wpk, rpk), the integer group dots Dw = sum_{k in g} qx[m,k] * qw[n,k]
 * and, for the listed blocks, Dr = sum_{k in g} qx[m,k] * qr[n,k]; the dots
 * are exact.  One
 * kernel streams each weight unit once, reads each activation tile once per
 * output tile, adds the residual product of a block in the same pass, and
 * reduce-adds both partial products in fp32 in ascending-g order (split-K
 * partials are summed in a fixed order, so the result is deterministic).
 *   xq, xs   from mq_quantize_act (M tokens).
 *   wpk, row_ptr, col_idx, nnzb, rpk   from mq_select_blocks /
 *            mq_pack_weights (nnzb == 0: row_ptr, col_idx and rpk may be NULL).
 *   y        [M, N] row-major, MQ_BF16 (round to nearest even) or MQ_F32.
 *   ws       at least mq_gemm_workspace_bytes(M, N, K) bytes on the current
 *            device, 256-byte aligned, zeroed once by mq_gemm_workspace_init
 *            (and again after an MQ_ERR_TIMEOUT).  Every call that finishes
 *            normally leaves it ready for the next, so one workspace can serve
 *            GEMMs of any shape run one after another on a stream; it must not
 *            be used by two GEMMs in flight at the same time.
 */
mq_status mq_w4a4_residual_gemm(const uint8_t* xq, const uint16_t* xs, int64_t M,
                                const uint8_t* wpk, int64_t N, int64_t K, const int32_t* row_ptr,
                                const int32_t* col_idx, int64_t nnzb, const uint8_t* rpk, void* y,
                                mq_dtype yt, void* ws, size_t ws_bytes, mq_stream_t stream);

/*
 * The fused GEMM without a caller-provided workspace, for callers that cannot
 * allocate device memory (their allocator belongs to another runtime, or they
 * may not call cudaMalloc while a captured graph or a latency-critical loop is
 * live) and can only hand over their own inputs and outputs.  This entry point
 * has no counterpart in the paper; it is a deployment convenience.
 *   Arguments and results as mq_w4a4_residual_gemm, without ws / ws_bytes.
 *   Scratch: one fixed 8 MiB array in the library's device memory (held on
 *     every GPU that loads the library until the process exits).  Any shape
 *     whose kernel needs at most that much (mq_gemm_workspace_bytes on the
 *     current device, for the kernel the shape runs on) is served: every
 *     decode batch of up to 32 tokens at K up to about 600k on a 152-SM GPU,
 *     and small larger-M problems; others return MQ_ERR_WORKSPACE.
 *   The first call on a device resolves the array's device address (with that
 *     device current); make that first call before any stream capture.
 *   The array is shared by every call and keeps the last call's contents.
 *     The kernels leave its counter prefix zeroed; after a device-side wait
 *     has run out (mq_check_device_error returned MQ_ERR_TIMEOUT), the next
 *     call clears that prefix on `stream` first.  Calls that overlap on the
 *     GPU (two streams, or several host threads on one device) race on the
 *     array: serialize them.
 *   Allocates nothing (no cudaMalloc / cudaFree, no allocating library call).
 */
mq_status mq_w4a4_residual_gemm_noalloc(const uint8_t* xq, const uint16_t* xs, int64_t M,
                                        const uint8_t* wpk, int64_t N, int64_t K,
                                        const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                                        const uint8_t* rpk, void* y, mq_dtype yt, mq_stream_t stream);

/*
 * One weight matrix of a grouped call (mq_w4a4_residual_linear): its packed
 * form from mq_select_blocks / mq_pack_weights and its output.
 *   wpk, N, row_ptr, col_idx, nnzb, rpk  as for mq_w4a4_residual_gemm (all
 *         matrices of one call share K); nnzb == 0: row_ptr, col_idx, rpk may be NULL.
 *   y     [M, ldy] row-major, columns 0..N-1 written (MQ_BF16 or MQ_F32, the
 *         call's yt); ldy >= N, so several matrices may write slices of one
 *         wider output.
 */
typedef struct {
  const uint8_t* wpk;
  int64_t N;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  int64_t nnzb;
  const uint8_t* rpk;
  void* y;
  int64_t ldy;
} mq_matrix;

/* Bytes of workspace mq_w4a4_residual_linear needs for M tokens, K inputs and
 * the nmat matrices of N[i] outputs each (0 for invalid sizes). */
size_t mq_linear_workspace_bytes(int64_t M, int64_t K, int nmat, const int64_t* N);

/*
 * The whole linear layer from unquantized activations, for up to 4 matrices
 * that read the same X (for example the q, k and v projections, or gate and
 * up):  Y_i = Q(X) (Q(W_i) + R_i)^T.
 * The activation quantizer is the ZipperEngine pipeline's first stage
 * (Metodologia 3); with at most 32 tokens it runs inside the GEMM launch: each
 * 128-input group of X is quantized once (by one CTA, with the same rule and
 * bits as mq_quantize_act), published to the workspace, and every weight tile
 * of every matrix reduce-adds its dense and residual products against it.
 * One kernel launch, no xq round trip through the caller.  Above 32 tokens it
 * runs mq_quantize_act's kernel, then the GEMM of each matrix.
 *   x     [M, ldx] MQ_F16 or MQ_BF16 (xt), ldx >= K, 8-byte aligned rows.
 *   mats  host array of nmat (1..4) mq_matrix; the matrices' tiles are
 *         processed as one sequence, so small matrices share the launch.
 *   xq, xs  optional (NULL: not written): the quantized activations in
 *         mq_quantize_act's layout, bit-identical to what it writes.
 *   ws    at least mq_linear_workspace_bytes(M, K, nmat, N) bytes, 256-byte
 *         aligned, zeroed once by mq_gemm_workspace_init (as for the GEMM).
 * Errors as mq_w4a4_residual_gemm.
 */
mq_status mq_w4a4_residual_linear(const void* x, mq_dtype xt, int64_t M, int64_t K, int64_t ldx, int nmat,
                                  const mq_matrix* mats, mq_dtype yt, uint8_t* xq, uint16_t* xs, void* ws,
                                  size_t ws_bytes, mq_stream_t stream);

/*
 * Test hook: the same kernel, but instead of the fp32 reduce-add it writes the
 * raw integer group dots it computed on the tensor cores:
 *   dw [M, N, K/128] int32 : Dw[m, n, g]
 *   dr [M, nnzb, 64] int32 : Dr of CSR entry i, block row r  (NULL if nnzb == 0)
 * Same argument rules as mq_w4a4_residual_gemm otherwise.
 */
mq_status mq_debug_group_dots(const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk,
                              int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx,
                              int64_t nnzb, const uint8_t* rpk, int32_t* dw, int32_t* dr, void* ws,
                              size_t ws_bytes, mq_stream_t stream);

/*
 * Which kernel mq_w4a4_residual_gemm (and the no-alloc and debug forms) runs
 * for a problem of M tokens, N outputs and K inputs on the current device.
 *   info  host array of 5 int32, written:
 *         [0] the decode kernel (stream-K over every SM, up to 32 tokens):
 *             4 = its warp-MMA form (the default; the fused call quantizes
 *             in a short kernel of its own first), 5 = its column form (warp
 *             MMA with the activation quantizer inside the GEMM) and 3 = its
 *             tensor-memory form (taken when the environment variable
 *             MQ_DECODE_VARIANT is "col" or "tc"); 0 = the general kernel
 *             in its converter form (33 to 127 tokens, or any M > 32 when
 *             the environment variable MQ_GENERAL_FORM is "conv"); 6 = the
 *             general kernel in its image form (a pre-pass writes the E4M3
 *             operand images, the GEMM runs both MMA operands from shared
 *             memory: from 128 tokens, or any M > 32 when MQ_GENERAL_FORM
 *             is "image"; it needs the workspace mq_gemm_workspace_bytes
 *             gives);
 *         for the decode kernel, [1] tokens per tile (8, 16 or 32), [2] CTAs
 *         per thread-block cluster (1 without clusters; the warp-MMA form
 *         gives each weight tile a cluster of this many CTAs when that uses
 *         about as many SMs as stream-K, unless MQ_DECODE_CLUSTER is "0"),
 *         [3] CTAs launched, [4] weight stages in shared memory; for the
 *         image form [1] tokens per tile (128) and [3] CTAs launched, the
 *         rest zero; zeros for the converter form.
 * MQ_ERR_INVALID_ARG for bad sizes (the same rules as the GEMM) or NULL info;
 * MQ_ERR_UNSUPPORTED_DEVICE if the current device is not compute capability 10.3.
 * Launches nothing.
 */
mq_status mq_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t* info);

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */

/* Synchronize `stream`, read and clear the device error word of the current
 * device: MQ_ERR_TIMEOUT if a bounded device-side wait ran out since the last
 * check, MQ_ERR_CUDA if the stream reports an error, else MQ_OK. */
mq_status mq_check_device_error(mq_stream_t stream);

/* Limit, in nanoseconds, of every device-side wait launched afterwards
 * (default 1e9; values outside [1e3, 6e10] are clamped). */
void mq_set_wait_timeout_ns(uint64_t ns);

/* Test hook for failure detection: launch one CTA whose bounded wait is on an
 * mbarrier that nothing ever arrives on; it gives up after the configured
 * limit, sets the device error word and exits.  Follow with
 * mq_check_device_error, which then returns MQ_ERR_TIMEOUT. */
mq_status mq_debug_wait_timeout(mq_stream_t stream);

const char* mq_status_string(mq_status s);
/* Thread-local detail of the last error returned on this host thread. */
const char* mq_last_error(void);
/* Library version string. */
const char* mq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MQ_H_ */
