/*
 * qgemv.h -- C ABI of the weight-only quantized decode GEMV for GB300 (sm_103a)
 *
 *     y[M x N] = x[M x K] . dequant(W)^T ,   1 <= M <= 16
 *
 * W is an N x K weight matrix (N outputs, K inputs) held in a packed low-bit
 * format; x holds M fp16 activation rows; y receives M fp32 output rows.  The
 * packed weights stream from HBM, are decoded in registers and multiplied and
 * accumulated in fp32 by the library's CUDA kernels.  The problem statement
 * (M rows, N outputs, K inputs per output) is the one of "Making a ternary
 * reasoning model fast in vLLM", section "Reading the prompt and writing the
 * answer"; the formats are listed with their sources below.
 *
 * Conventions for every call:
 *   - Sizes are int64_t element counts; all multi-byte values little-endian.
 *   - Device pointers are CUDA device (or managed) addresses on the current
 *     device.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).
 *   - A call returns QGEMV_OK (0) or one of the QGEMV_ERR_* codes; the handle
 *     constructor returns NULL on error.  qgemv_last_error() then gives a
 *     thread-local message.  No call aborts the process or throws.
 *   - Argument errors are found on the host before anything is launched or
 *     allocated.
 *   - Calls that launch kernels are asynchronous on `stream` unless stated
 *     otherwise.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats.  "Canonical" is the byte layout the caller passes in. */
typedef enum {
  /* ggml-style Q4_0 ("Model quantization, read carefully", sections "The
   * ladder" and "Anatomy of a block"): blocks of 32 weights along K, each
   * {fp16 d; uint8 qs[16]} = 18 bytes, 4.5 bits per weight.  Byte i of qs
   * holds element i in its low nibble and element i+16 in its high nibble;
   * the weight is (q - 8) * d.  packed = N*K/32 blocks, row-major over rows
   * n; K % 32 == 0; scales = codebooks = NULL.                              */
  QGEMV_Q4_0 = 1,
  /* Scalar 4-bit codebook ("Trapetum benchmarks", "Kernel microbenchmarks":
   * 4-bit index into K = 16 centroids): packed = uint8 [N][K/2], byte j of a
   * row holds k = 2j (low nibble) and k = 2j+1 (high nibble); codebooks =
   * 16 fp16 centroids shared by the whole matrix; K % 2 == 0; scales = NULL. */
  QGEMV_CBK4 = 2,
  /* Scalar 8-bit codebook (same page: uint8 index into 256 centroids, the
   * 8-bit LM head): packed = uint8 [N][K]; codebooks = 256 fp16; any K.    */
  QGEMV_CBK8 = 3,
  /* PQ2_0 ternary ("Making a ternary reasoning model fast in vLLM", "Anatomy
   * of a PQ2_0 block"): blocks of 128 weights along K, {fp16 d; uint8
   * qs[32]} = 34 bytes; byte j holds elements 4j..4j+3 as two-bit codes from
   * the low end; codes 0,1,2,3 decode to -1,0,+1,+2 times d.  packed = N*K/128
   * blocks, one row of blocks per output; K % 128 == 0.                      */
  QGEMV_PQ2_0 = 4,
  /* AQLM 2x8 additive codebooks ("Trapetum benchmarks", "Additive
   * vector-quantization GEMV" and "Llama-2-70B in 2 bits"): per group of 8
   * weights along K two uint8 codes; w[n][8g+j] = s[n] * (C0[c0][j] +
   * C1[c1][j]).  packed = codes uint8 [N][K/8][2] (codebook 0 first);
   * scales = fp16 [N]; codebooks = fp16 [2][256][8]; K % 8 == 0.          */
  QGEMV_AQLM_2X8 = 5,
  /* AQLM 1x16 ("Trapetum benchmarks", the PV-tuned Llama-2-70B in 1x16): one
   * codebook of 65,536 entries of 8 fp16 values per matrix and one 16-bit
   * code per group of 8 weights along K (2 bits per weight); w[n][8g+j] =
   * s[n] * C[code][j].  packed = codes uint16 little-endian [N][K/8];
   * scales = fp16 [N]; codebooks = fp16 [65536][8] (1 MiB); K % 8 == 0.
   * (Value 6 is reserved inside the library.)                              */
  QGEMV_AQLM_1X16 = 7,
  /* CBK4 with one codebook per output row, the pages' own 4-bit file layout
   * ("Trapetum benchmarks", "Model-level results": a 16-centroid k-means
   * codebook per output channel, stored in fp32): packed = uint8 [N][K/2]
   * as QGEMV_CBK4; codebooks = fp32 [N][16], row n's centroids together
   * (64 bytes per row); K % 2 == 0; scales = NULL.  Every M runs the
   * CUDA-core kernel (fp32 centroids), eight activation rows per launch
   * while eight remain, then two, then one; a row's bits do not depend on M
   * in batch-invariant mode (which keeps to the two- and one-row launches),
   * and otherwise differ at most in the last places between calls below and
   * above eight rows.                                                      */
  QGEMV_CBK4_ROW = 8,
  /* CBK8 with one codebook per output row, the 8-bit LM head of the same
   * files (256 fp32 centroids per row): packed = uint8 [N][K]; codebooks =
   * fp32 [N][256] (1 KB per row); 1 <= K <= 65536; scales = NULL.  One warp
   * per output row, the row's codebook in shared memory; a row's bits do not
   * depend on M.                                                            */
  QGEMV_CBK8_ROW = 9
} qgemv_format;

/* Status codes. */
enum {
  QGEMV_OK = 0,
  QGEMV_ERR_ARG = 1,     /* bad format, size, M, null pointer or handle     */
  QGEMV_ERR_ALIGN = 2,   /* x or y not aligned as required                  */
  QGEMV_ERR_CUDA = 3,    /* a CUDA call failed (message has its error text) */
  QGEMV_ERR_TIMEOUT = 4, /* a kernel's bounded wait gave up (qgemv_status)  */
  QGEMV_ERR_NOMEM = 5    /* device or host allocation failed                */
};

typedef struct qgemv_ctx* qgemv_handle; /* opaque */

/* Bytes of the canonical packed weights for (format, N, K); 0 if invalid. */
int64_t qgemv_packed_bytes(int format, int64_t N, int64_t K);

/* Create a handle for one weight matrix.
 *   packed, scales, codebooks: canonical inputs as described per format
 *     (unused ones must be NULL).  Each may be a host or a device pointer
 *     (told apart with cudaPointerGetAttributes); the data is copied into
 *     library-owned device memory and re-laid out there ("prepared" tiles),
 *     so the caller may free its buffers once this call returns.
 *   The call allocates the handle's device buffers (prepared weights and a
 *   small per-handle workspace), runs the re-layout kernel on the legacy
 *   default stream and synchronizes before returning.
 * Returns NULL on error (see qgemv_last_error).                              */
qgemv_handle qgemv_create(int format, int64_t N, int64_t K, const void* packed,
                          const void* scales, const void* codebooks);

/* Create one handle for several projections that share K and therefore the
 * activations (the attention's q, k and v, or an MLP's gate and up): their
 * weight rows stacked in order, so that one qgemv_run computes all of them,
 * y = [y_0 | y_1 | ...] along N, with one launch instead of one per
 * projection.  The pages fuse such projections in their runtimes; this call
 * has no further counterpart there.
 *   nseg >= 1 segments; segment s has seg_rows[s] > 0 output rows, and every
 *     segment but the last must have a multiple of the prepared tile height
 *     (128 rows; AQLM 2x8: 2048, its row block), so that no tile mixes two
 *     codebooks.
 *   packed: the segments' canonical bytes one after the other, which is the
 *     canonical layout of the stacked matrix (rows of all formats are
 *     independent).
 *   codebooks (CBK4, CBK8, AQLM 2x8): nseg codebooks one after the other
 *     (16 or 256 fp16 each; AQLM 2x8: a [2][256][8] fp16 pair each); segment
 *     s decodes with codebook s.  NULL for Q4_0 and PQ2_0, whose stacked
 *     handle is the plain concatenation.
 *   scales (AQLM 2x8): the N row scales of all segments in order.
 *   A stacked AQLM 2x8 handle runs its per-group-table kernel at every M (a
 *     pass per two activation rows), without the tensor-core form that a
 *     single-matrix handle uses from M = 3.
 *   AQLM 1x16, CBK4_ROW and CBK8_ROW are not accepted (QGEMV_ERR_ARG; 1x16
 *   keeps one 1 MiB codebook per handle, and the rows of a per-row-codebook
 *   matrix carry their own codebooks, so one handle over the concatenated
 *   rows does the same).
 * Host or device pointers, copying, errors: as for qgemv_create.             */
qgemv_handle qgemv_create_stacked(int format, int nseg, const int64_t* seg_rows, int64_t K,
                                  const void* packed, const void* scales, const void* codebooks);

/* Create one handle for the gate and up projections of a decoder MLP whose
 * runs store the fused activation y[m][n] = SiLU(x . G^T)[m][n] * (x . U^T)
 * [m][n], SiLU(v) = v / (1 + e^-v): the gate/up GEMV with "SiLU(gate) * up
 * in the reduce" of "Trapetum benchmarks" ("Short-context decode, step by
 * step"), with no separate activation kernel.  Q4_0, PQ2_0, CBK4 and CBK8
 * run every M in one launch (M >= 2 on the tensor-core kernel, the weights
 * read once per call); CBK4_ROW launches once per activation row.
 *   format: QGEMV_Q4_0, QGEMV_PQ2_0, QGEMV_CBK4, QGEMV_CBK8 or QGEMV_CBK4_ROW
 *     (CBK4 / CBK8: the gate and up tables share the kernels' table region,
 *     each lookup still one shared-memory read; per-row codebooks travel
 *     with their rows).
 *   N: rows of each projection (the output width), a positive multiple of
 *     64; K as for qgemv_create.
 *   packed_gate, packed_up: each projection's canonical bytes (host or
 *     device), copied.  The handle holds them interleaved in 64-row blocks.
 *   codebooks_gate, codebooks_up: each projection's codebook -- CBK4 fp16
 *     [16], CBK8 fp16 [256], CBK4_ROW fp32 [N][16]; NULL for Q4_0 and PQ2_0.
 * Runs: qgemv_run with y fp32 [M][N]; the residual form is refused, and so
 * are qgemv_set_x_int8 and qgemv_run_xq.  qgemv_dequant of such a handle
 * writes the 2N interleaved rows (64 gate rows, then the 64 up rows of the
 * same block, and so on).  The result is SiLU and the product in fp32
 * (expf, an IEEE division, one product) of the two GEMV sums.
 * Returns NULL on error (QGEMV_ERR_ARG for another format or a bad N).     */
qgemv_handle qgemv_create_glu(int format, int64_t N, int64_t K, const void* packed_gate,
                              const void* packed_up, const void* codebooks_gate, const void* codebooks_up);

/* y = x . dequant(W)^T for M rows.
 *   x: device fp16 [M][K] row-major, 4-byte aligned.
 *   y: device fp32 [M][N] row-major, 4-byte aligned; fully overwritten.
 *   1 <= M <= 16.
 * Asynchronous on `stream`; no allocation, no synchronization, so it can be
 * captured in a CUDA graph.  The handle's workspace is shared by its runs:
 * one handle must not run on two streams at the same time.  Results are
 * bitwise reproducible run to run for a given (handle, M).                  */
int qgemv_run(qgemv_handle h, const void* x, int M, float* y, void* stream);

/* y = residual + x . dequant(W)^T for M rows: the residual add of a decoder
 * layer's attention-output and MLP-down projections done in the GEMV's own
 * store instead of a separate kernel ("Trapetum benchmarks", "Short-context
 * decode, step by step": the residual add inside the o and down reduces).
 *   residual: device fp32 [M][N] row-major, 4-byte aligned, not NULL.  It may
 *     be y itself (y += x . W^T): each element is read and then written by
 *     the same thread.
 *   x, y, M, stream and the handle: as for qgemv_run.
 * Each output is the value qgemv_run would store, plus the residual in one
 * fp32 add (round to nearest), so the two calls agree bit for bit.         */
int qgemv_run_residual(qgemv_handle h, const void* x, int M, float* y, const float* residual,
                       void* stream);

/* Batch-invariant mode (off by default): when on, row m of y from any call
 * is bitwise the same whatever M the call has and wherever the row sits in
 * the batch (the same x row gives the same y row alone or batched, as a
 * verifier comparing batched and single-row decodes needs).  Off, M = 1 and
 * M = 2..8 run faster kernel geometries (and AQLM 2x8 with M <= 2 its
 * per-group table path), whose bits may differ in the last places (all
 * within the accuracy bound).  On, every M runs the tensor-core kernel's
 * default geometry (AQLM 2x8: its tensor-core layout; a stacked AQLM 2x8
 * handle: a one-row pass of its table kernel per row; CBK4_ROW: launches of
 * at most two rows; AQLM 1x16 and CBK8_ROW are batch invariant in either
 * mode).  Takes effect for runs issued after the call; returns
 * QGEMV_ERR_ARG for an invalid handle. */
int qgemv_set_batch_invariant(qgemv_handle h, int on);

/* INT8 activations for a PQ2_0 handle (off by default): the integer path of
 * "Making a ternary reasoning model fast in vLLM" (the section on quantising
 * the activation too).  When on, runs quantize each group of 128 activations
 * of a row to signed INT8 exactly as qgemv_quantize_x_int8 does, take every
 * block's inner sum over its codes in integer arithmetic (four-way INT8 dot
 * products) and apply d * a once per block in fp32.  The result is that of
 * the quantized activations: lossy against qgemv_run with the mode off (the
 * quantization error is a property of the method, at most half a step of
 * each group's scale per nonzero weight), and accurate to the usual fp32
 * bound against the exact integer-path value.  Up to three activation rows
 * run the CUDA-core kernel (DP4A inner sums, up to four rows per launch);
 * four or more run, in one call, the quantizer of qgemv_prepare_x_int8 into
 * a handle-owned workspace and one launch of the tensor-core kernel (the
 * INT8 codes as exact fp16 operands, exact integer block sums), so the
 * weights are read once per call.  A row's bits are the same in every call
 * of up to three rows and in every call of four or more; the two kernels
 * may differ in the last places (same bound) unless batch-invariant mode is
 * on, which puts every M on the tensor-core kernel.  Works with qgemv_run and qgemv_run_residual; takes
 * effect for runs issued after the call.  The first call that turns the mode
 * on allocates the workspace (qgemv_xq_bytes(16, K) bytes, freed with the
 * handle): QGEMV_ERR_NOMEM if that fails.  Returns QGEMV_ERR_ARG for an
 * invalid handle or a handle that is not PQ2_0 (stacked PQ2_0 handles are
 * accepted).                                                                */
int qgemv_set_x_int8(qgemv_handle h, int on);

/* The INT8 activation quantizer of the PQ2_0 integer path, on the device:
 *   x: device fp16 [M][K] row-major, K a positive multiple of 128, M >= 1;
 *   q_out: device int8 [M][K];  a_out: device fp32 [M][K/128].
 * Per group g of 128 consecutive inputs of a row: a = fl32(max|x| / 127),
 * q = clamp(rint(fl32(x / a)), -127, 127) with IEEE fp32 divisions and
 * ties to even; an all-zero group gives a = 0 and q = 0.  The same device
 * arithmetic as the GEMV's staging (for tests and for callers that keep
 * the quantized activations).  Asynchronous on `stream`.                   */
int qgemv_quantize_x_int8(const void* x, int M, int64_t K, int8_t* q_out, float* a_out, void* stream);

/* Prepared INT8 activations for PQ2_0 handles: the activation prologue of
 * the integer path, run once per activation vector and shared by every
 * projection that reads it (q, k and v; gate and up), with the Hadamard
 * mixing of "Making a ternary reasoning model fast in vLLM" (the section on
 * mixing the inputs) fused in when asked.
 *
 * Bytes of the prepared buffer of M rows of K inputs (K % 128 == 0), or 0
 * for invalid sizes: M*K codes, then M*K/128 fp32 scales, then M*K/128
 * int32 code sums.                                                          */
int64_t qgemv_xq_bytes(int M, int64_t K);

/* Fill xq (device, qgemv_xq_bytes(M, K) bytes, 4-byte aligned) from x
 * (device fp16 [M][K], 4-byte aligned).
 *   hadamard_block = 0: the codes of x itself, exactly as
 *     qgemv_quantize_x_int8 computes them.
 *   hadamard_block = 1024 (K % 1024 == 0): each block of 1024 inputs is
 *     first mixed, v = 2^-5 H (s . x) with H the 1024 x 1024 Sylvester
 *     Hadamard matrix, computed in fp32 as the page does (signs, then
 *     butterfly stages h = 1, 2, ..., 512 replacing (u, w) by (u + w,
 *     u - w), then the scaling), and the fp32 values v are quantized.
 *     signs: device int8 [K] of +1 / -1 over the row width (the same for
 *     every row), or NULL for none.
 * Layout of xq: row m's codes at byte m*K; within each group of 128 inputs
 * the code of input 16i + 4b + s (i = 0..7, b = 0..3, s = 0..3) is at byte
 * 16i + 4s + b of the group (the order the GEMV stages them); the scale of
 * group g of row m is float m*K/128 + g after the codes, and its code sum
 * the int32 of the same index after the scales.  Asynchronous on `stream`; returns
 * QGEMV_ERR_ARG for bad sizes, a block other than 0 or 1024, or signs
 * without the mixing; QGEMV_ERR_ALIGN for misaligned pointers.             */
int qgemv_prepare_x_int8(const void* x, int M, int64_t K, const int8_t* signs, int hadamard_block, void* xq,
                         void* stream);

/* y = residual + (prepared INT8 activations) . dequant(W)^T for a PQ2_0
 * handle: the integer path of qgemv_set_x_int8 on codes from
 * qgemv_prepare_x_int8 (with the same M and the handle's K): up to three
 * rows on the CUDA-core kernel, four or more in one launch of the
 * tensor-core kernel (as for qgemv_set_x_int8).  With hadamard_block = 0 the result equals qgemv_run in INT8 mode
 * bit for bit.
 * residual may be NULL (plain store) or y itself.  The handle's INT8 mode
 * setting does not matter here.  Asynchronous; as qgemv_run otherwise.     */
int qgemv_run_xq(qgemv_handle h, const void* xq, int M, float* y, const float* residual, void* stream);

/* Write the decoded weights, fp32 [N][K] row-major, to device memory w_out
 * (the exact value of every weight; read back from the prepared tiles, so it
 * also checks the re-layout).  Asynchronous on `stream`.                     */
int qgemv_dequant(qgemv_handle h, float* w_out, void* stream);

/* Q4_0 quantizer on the device: fp32 weights [N][K] (device) -> canonical
 * Q4_0 blocks (device, N*K/32*18 bytes).  Per block: d = (signed value of
 * largest magnitude, first on ties) / -8 in fp32; q = clamp(round(w/d) + 8,
 * 0, 15) with an IEEE fp32 division and round half away from zero; d stored
 * as fp16 (nearest even).  An all-zero block stores q = 8.  Asynchronous.  */
int qgemv_quantize_q4_0(const float* w, int64_t N, int64_t K, void* packed_out,
                        void* stream);

/* Synchronize with the handle's last run and return QGEMV_ERR_TIMEOUT if a
 * kernel of it gave up a bounded wait (then clear that flag), else QGEMV_OK. */
int qgemv_status(qgemv_handle h);

/* Release the handle's device memory (synchronizes the device first).
 * NULL is accepted and ignored.                                             */
void qgemv_destroy(qgemv_handle h);

/* Allocation-free Q4_0 GEMV.  No counterpart in the source pages: a service
 * for callers that cannot allocate device memory when they need the product,
 * for instance code running inside a framework whose caching allocator owns
 * all device memory, or a latency-critical loop that must not pay for (or
 * synchronize on) cudaMalloc.  It needs no handle: it reads the caller's
 * canonical Q4_0 blocks directly (same layout as QGEMV_Q4_0 above).
 *   packed: device, N*K/32 blocks of 18 bytes, 2-byte aligned; K % 32 == 0.
 *   x: device fp16 [M][K]; y: device fp32 [M][N] (4-byte aligned); 1<=M<=16.
 * The call allocates nothing: its scratch (split-K partial sums and arrival
 * counters) lives in one static device array of 8 MiB that every GPU which
 * loads this library holds until the process exits.  A shape needs
 * ceil(K/2048) * M * N * 4 bytes of partial sums (none when K <= 2048) plus
 * 4 bytes per 64 rows of counters; a shape that needs more than 8 MiB is
 * rejected with QGEMV_ERR_ARG and a message giving both sizes.
 * All calls share that array and leave in it whatever the last one wrote; the
 * counters, which must start at zero, are cleared by every call.  Calls whose
 * executions overlap on the GPU (different streams, or several processes'
 * worth of work on one context) race on the array: serialize them.
 * The first call on a device finds the array's device address
 * (cudaGetSymbolAddress) with that device current and sets the kernel's
 * shared-memory limit; make that first call before any stream capture.  If
 * that set-up fails, the call returns QGEMV_ERR_CUDA, nothing is remembered
 * and the next call on the device tries the set-up again.
 * Asynchronous on `stream`; results are bitwise reproducible call to call.  */
int qgemv_run_q4_0_noalloc(const void* packed, int64_t N, int64_t K, const void* x, int M,
                           float* y, void* stream);

/* The stream-K work split (host only, no GPU needed), as the handles use it:
 * `units` work units (prepared tiles; for AQLM_2X8 blocks of 2048 rows x 128
 * inputs) in row-major order, `units_per_row_tile` of them per row tile of
 * `rows` output rows, split over `grid` CTAs: split_unit 0, CTA c runs
 * units [c*units/grid, (c+1)*units/grid); split_unit 1 or 2, in chunks of
 * that many consecutive units, n = ceil(units / split_unit) chunks, q = n /
 * grid, r = n % grid, CTA c runs chunks [c*q + min(c, r), (c+1)*q + min(c+1,
 * r)) (the last chunk may be short).  A handle uses its format's mode.
 * Writes 12
 * int64 per CTA into `out` (caller-owned, grid*12 entries): for its two
 * shared-row-tile segments s = 0 (first row tile of its run), 1 (last):
 * out[c*12 + 0 + s] row tile (-1: none), [2 + s] first contributing CTA,
 * [4 + s] number of contributors, [6 + s] first row of this CTA's slice of
 * the rows to finish, [8 + s] rows in that slice, [10 + s] flags: bit 0 set
 * if the first contributor's run began before the row tile, bit 1 set if
 * this CTA finishes the whole row tile when it has at most 256 items (rows x
 * activation rows; then the others finish nothing).  Returns QGEMV_ERR_ARG if a
 * size is not positive, units % units_per_row_tile != 0, grid > units or
 * split_unit is not 0, 1 or 2.                                               */
int qgemv_stream_k_plan(int64_t units, int grid, int64_t units_per_row_tile, int rows, int split_unit,
                        int64_t* out);

/* Message and code of the last error on the calling thread ("" / 0 if none). */
const char* qgemv_last_error(void);
int qgemv_last_error_code(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
