/*
 * qlora.h -- C ABI of libqlora: the frozen-NF4 linear layer with a LoRA adapter
 * (QLoRA), hand-written CUDA for B300 (sm_103a).
 *
 * The method (arXiv 2305.14314, "QLoRA: Efficient Finetuning of Quantized
 * LLMs", abstract; the Chinese QLoRA news write-up, list of innovations):
 * weights are stored as 4-bit NormalFloat (NF4) codes with one constant per
 * block, the block constants are themselves quantized ("double
 * quantization"), and gradients flow through the frozen dequantized weights
 * into low-rank adapters (LoRA tutorial, Lit-LLaMA translation: h = Wx + dWx,
 * dW = W_A W_B, scale alpha).
 *
 * Conventions for every call:
 *  - Row-major matrices.  bf16 values are passed as their 16-bit patterns
 *    (uint16_t).  X is M x K (tokens x in), the weight W is N x K (out x in),
 *    Y is M x N, A is K x r, B is r x N, s = alpha / r.
 *  - All pointers are DEVICE pointers of the current CUDA device unless
 *    stated otherwise, 16-byte aligned, and owned by the caller.  The library
 *    allocates nothing and never synchronises (except ql_get_device_status).
 *  - Calls are asynchronous and ordered on `stream` (NULL = legacy default).
 *  - Return codes: QL_OK, or an error code with a message available from
 *    ql_last_error() (thread-local).  Argument errors are detected on the host
 *    before any launch.  Inputs must be finite; NaN/Inf behaviour is
 *    unspecified.
 *  - Workspace `ws` is caller-owned device scratch of at least
 *    ql_workspace_size(op, ...) bytes, 256-byte aligned; it may be reused
 *    between calls that are ordered on the same stream.
 */
#ifndef QLORA_H
#define QLORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QL_API __attribute__((visibility("default")))
#else
#define QL_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *ql_stream_t;

enum ql_status {
  QL_OK = 0,
  QL_ERR_INVALID = 1,     /* null pointer, non-positive or inconsistent size */
  QL_ERR_UNSUPPORTED = 2, /* blocksize != 64, dq_blocksize not 0/256, K % 64,
                             r not in {8,16,32,64,128}, too small workspace */
  QL_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned (ws: 256) */
  QL_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  QL_ERR_TIMEOUT = 5      /* a kernel gave up waiting (see ql_get_device_status) */
};

enum ql_op {
  QL_OP_QUANTIZE = 0,
  QL_OP_DEQUANTIZE = 1,
  QL_OP_LINEAR_FWD = 2,
  QL_OP_LINEAR_BWD = 3,
  QL_OP_QUANTIZE_HOST = 4,
  QL_OP_LINEAR_FWD_FP8 = 5,
  QL_OP_LINEAR_BWD_FP8 = 6
};

/*
 * A quantized weight (the NF4 storage of QLoRA; BitsAndBytes-style knobs of the
 * QLoRA project page's configuration example: 4-bit NF4, double quant on/off).
 *   rows x cols    : N x K of the bf16 weight it came from; cols % 64 == 0.
 *   blocksize      : 64 elements per first-level block (consecutive in a row).
 *   dq_blocksize   : 256 first-level blocks per second-level group, or 0 for
 *                    no double quantization.
 *   packed         : rows*cols/2 bytes; element 2j of the row-major matrix is
 *                    the HIGH nibble of byte j, element 2j+1 the low nibble.
 *   absmax         : n_b = rows*cols/64 floats, the block absmax values.
 *                    Required when dq_blocksize == 0; ignored otherwise.
 *   absmax_code    : n_b 8-bit second-level codes  (dq_blocksize != 0):
 *                    int8 or E4M3 bytes, as dq_type says
 *   dq_step        : n_2 = ceil(n_b/256) floats     (dq_blocksize != 0)
 *   dq_mean        : 1 float                         (dq_blocksize != 0)
 *   quant_type     : QL_NF4 (0, the default) or QL_FP4 (1): which 16-level
 *                    code table the 4-bit codes index (see ql_codebook).
 *   dq_type        : QL_DQ_INT8 (0, the default) or QL_DQ_E4M3 (1): the
 *                    8-bit code of the second level (see below).
 * Block b = row*(cols/64) + j covers row `row`, columns [64j, 64j+64).
 * Decoded block constant: dq off: absmax[b];
 *   dq on: fl32(fl32(v(absmax_code[b]) * dq_step[b/256]) + dq_mean[0]), where
 *   v is the code's value: the int8 itself (QL_DQ_INT8), or the E4M3 number
 *   the byte encodes (QL_DQ_E4M3: sign, 4-bit exponent with bias 7, 3-bit
 *   mantissa, subnormals at exponent 0, largest finite 448, byte 0x7F/0xFF
 *   never written).
 * Second-level quantization (QLoRA abstract, innovation (b): the
 *   quantization constants are themselves quantized; group of 256): c_b =
 *   fl32(absmax_b - mu), a2 = max |c_b| over the group, dq_step =
 *   fl32(a2 / L) with L = 127 (int8) or 448 (E4M3), code = the nearest code
 *   value to fl32(c_b / dq_step) (int8: round half to even, clamped to
 *   +-127; E4M3: round to nearest, ties to the even code, saturating at
 *   +-448); a group with a2 = 0 gets step 0 and codes 0.
 * Dequantized weight: bf16_rne(fl32(q[code] * constant)), q = the code table.
 */
typedef struct {
  int64_t rows;
  int64_t cols;
  int32_t blocksize;
  int32_t dq_blocksize;
  uint8_t *packed;
  float *absmax;
  int8_t *absmax_code;
  float *dq_step;
  float *dq_mean;
  int32_t quant_type;
  int32_t dq_type;
} ql_nf4_tensor;

/* Second-level codes (ql_nf4_tensor.dq_type). */
enum ql_dq_type {
  QL_DQ_INT8 = 0, /* linear int8, step = a2 / 127 */
  QL_DQ_E4M3 = 1  /* 8-bit float E4M3, step = a2 / 448 */
};

/* Code tables (ql_nf4_tensor.quant_type). */
enum ql_quant_type {
  QL_NF4 = 0, /* 4-bit NormalFloat: normal quantiles, the QLoRA data type */
  QL_FP4 = 1  /* 4-bit float E2M1 values, the baseline NF4 is compared with */
};

/*
 * Bytes of workspace the op needs for the given sizes (M tokens, N out, K in,
 * r rank; unused sizes may be 0).  Returns 0 when the op needs none, and
 * (size_t)-1 for an unknown op.
 */
QL_API size_t ql_workspace_size(int op, int64_t M, int64_t N, int64_t K, int32_t r);

/*
 * The 16 NF4 levels (ascending, fp32) the kernels use, written to host
 * memory `out16`.  Built at library load from the definition: standard-normal
 * quantiles normalised to [-1, 1] with an exact zero (8 positive levels,
 * 7 negative).  Returns QL_OK.
 */
QL_API int ql_nf4_codebook(float *out16);

/*
 * The 16 levels of a code table (ascending fp32, host memory `out16`):
 *   QL_NF4 as ql_nf4_codebook;
 *   QL_FP4: the values of the 4-bit float format E2M1 (sign, 2 exponent bits,
 *   1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives) divided
 *   by the largest, 6, so the endpoints are -1 and +1; the 15 distinct
 *   values ascending (one zero, at index 7 as in NF4) and index 15 repeating
 *   +1 (never produced by the quantizer: ties go to the lower index).  The
 *   QLoRA pages compare NF4 against 4-bit floats; this is the plainest 4-bit
 *   float.  Returns QL_OK, or QL_ERR_UNSUPPORTED for an unknown type.
 */
QL_API int ql_codebook(int32_t quant_type, float *out16);

/*
 * NF4 quantization with optional double quantization (QLoRA abstract,
 * innovations (a) and (b); news write-up: "Double Quantization" saves about
 * 0.37 bit per parameter).
 *   W  : rows x cols bf16 (device), finite.
 *   q  : host struct describing the device outputs (all written).
 *   ws : ql_workspace_size(QL_OP_QUANTIZE, 0, rows, cols, 0) bytes.
 * Block absmax m = max|w| over 64 elements; code = index of the nearest
 * level of the tensor's code table (q->quant_type) to fl32(w / m) (ties to
 * the lower index; all-zero block -> code 7).
 * Double quant: mu = fl32(S / n_b) with S the fp64 sum of all m (exact when
 * the exponents of the block absmax values span fewer than
 * 45 - log2(n_b) binades, which holds for real weights); per 256 blocks
 * step = fl32(max|fl32(m - mu)| / 127), code = clamp(rne(fl32((m-mu)/step)),
 * -127, 127) (0 when step == 0).  Results are deterministic.
 */
QL_API int nf4_quantize(const uint16_t *W, const ql_nf4_tensor *q, void *ws,
                 size_t ws_bytes, ql_stream_t stream);

/*
 * nf4_quantize for callers that cannot pass a workspace (no counterpart in the
 * paper: an interface convenience of this library).  Callers whose device
 * memory is all planned up front, callers embedded in a host runtime that owns
 * every allocation and hands them no allocator, and callers that must not
 * trigger cudaMalloc's implicit device synchronisation cannot allocate
 * scratch per call; this entry point uses a
 * fixed scratch array built into the library instead (about 16 MB per GPU that
 * loads the library, held until the process exits).  It allocates nothing.
 *   W, q, stream : as for nf4_quantize.
 * Limit: rows * cols / 64 <= 4,194,304 blocks (256 Mi parameters); larger
 * weights return QL_ERR_UNSUPPORTED with a message.
 * The first call on a device looks the array's device address up once, with
 * that device current; make that first call before any stream capture.  All
 * calls share the one array (its contents are those of the last call; the
 * part that must start at zero is cleared by every call), so calls that
 * overlap on the GPU -- on different streams, or from different host threads
 * -- race and must be ordered by the caller.
 */
QL_API int nf4_quantize_noalloc(const uint16_t *W, const ql_nf4_tensor *q, ql_stream_t stream);

/*
 * Quantize-on-load: nf4_quantize of a weight that is still in HOST memory, so
 * that loading a model in 4 bit (the QLoRA project page's load_in_4bit)
 * never needs the bf16 copy in device memory.  The weight streams through
 * two device staging chunks: chunk c is copied host -> device on
 * `copy_stream` while chunk c - 1 is coded on `stream`; the double-quant
 * constants follow once every chunk is coded.  The result equals
 * nf4_quantize of the same weight bit for bit.
 *   W_host      : rows x cols bf16 in HOST memory (page-locked memory lets the
 *                 copies overlap the kernels; pageable memory works too).
 *   q           : as for nf4_quantize (device outputs).
 *   ws          : ql_workspace_size(QL_OP_QUANTIZE_HOST, 0, rows, cols, 0)
 *                 bytes (the quantize scratch plus two staging chunks of about
 *                 16 MB), 256-byte aligned.
 *   copy_stream : the stream for the copies (may equal `stream`, then nothing
 *                 overlaps); it first waits for the work already queued on
 *                 `stream`, and `stream` waits for each chunk's copy.
 * When the call returns the work is queued; the caller keeps W_host unchanged
 * until `stream` has passed it.  The call creates and releases a few CUDA
 * events (no device memory).
 */
QL_API int nf4_quantize_host(const uint16_t *W_host, const ql_nf4_tensor *q, void *ws, size_t ws_bytes,
                             ql_stream_t copy_stream, ql_stream_t stream);

/*
 * Row-sharded quantization for data-parallel training (the QLoRA project
 * page runs multi-GPU finetuning through Accelerate; every rank then holds
 * the same frozen weight, and may quantize its share of the rows).  Rows are
 * independent except for the double-quant mean mu = fl32(S / n_b), which
 * needs the sum S of ALL block absmax values and the total block count n_b.
 *   nf4_quantize_shard_begin(W_shard, q_shard, ws, ws_bytes, stream):
 *     q_shard describes this rank's rows (rows_shard x cols); writes the
 *     packed codes (and, with double quant off, the absmax) and leaves this
 *     shard's fp64 absmax sum as one double at the head of `ws` (device).
 *   The caller then replaces that double with the sum over all shards (an
 *   fp64 all-reduce; each partial sum is exact for real weights, so the
 *   total is the same in any order and equals the unsharded sum).
 *   nf4_quantize_shard_end(q_shard, ws, ws_bytes, total_blocks, stream):
 *     mu = fl32(S / total_blocks); writes this shard's second-level codes,
 *     steps and mu (nothing to do with double quant off).
 * The shard's blocks must start on a 256-block group boundary of the whole
 * tensor (rows_before * cols / 64 a multiple of 256) for its codes and steps
 * to equal the unsharded ones; the same workspace must be passed to both
 * calls, with nothing else using it in between.  ws_bytes as for
 * nf4_quantize on the shard.  nf4_quantize(W, q, ...) is exactly begin + end
 * with total_blocks = the tensor's own block count.
 */
QL_API int nf4_quantize_shard_begin(const uint16_t *W_shard, const ql_nf4_tensor *q_shard, void *ws,
                                    size_t ws_bytes, ql_stream_t stream);
QL_API int nf4_quantize_shard_end(const ql_nf4_tensor *q_shard, void *ws, size_t ws_bytes,
                                  int64_t total_blocks, ql_stream_t stream);

/*
 * Dequantize to bf16 (the weight the linear layer computes with).
 *   q     : host struct of device inputs; W_out : rows x cols bf16 (device).
 */
QL_API int nf4_dequantize(const ql_nf4_tensor *q, uint16_t *W_out, ql_stream_t stream);

/*
 * Forward of the frozen-NF4 linear with LoRA (LoRA tutorial: h = Wx + dWx;
 * QLoRA abstract: frozen 4-bit weights):
 *   Y = X W_hat^T + s (X A) B        (fp32 accumulation, bf16 output)
 *   X  : M x K bf16, A : K x r bf16, B : r x N bf16,  W : N x K NF4 (q).
 *   Y  : M x N bf16 (output).
 *   XA_out : M x r bf16 (output, may be NULL): X A rounded to bf16, for the
 *            backward pass.
 *   scale  : s = alpha / r.
 *   ws     : ql_workspace_size(QL_OP_LINEAR_FWD, M, N, K, r) bytes.
 * M >= 1.  M <= 32 takes the decode (weight-streaming) path, larger M the
 * tensor-core path (the few-token kernel up to 128 tokens, the CTA-pair
 * kernel above).  Every path multiplies by the dequantized weight W_hat bit
 * for bit; results differ only in the order of the fp32 sums.
 * The decode path keeps partial results in `ws` (any initial contents work);
 * successive decode calls on a stream alternate between its two halves, so a
 * call may start while the previous one finishes.
 */
QL_API int qlora_linear_fwd(const uint16_t *X, int64_t M, const ql_nf4_tensor *W,
                     const uint16_t *A, const uint16_t *B, int32_t r,
                     float scale, uint16_t *Y, uint16_t *XA_out, void *ws,
                     size_t ws_bytes, ql_stream_t stream);

/*
 * The same forward with the main product on 8-bit floats (E4M3: 1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits, largest finite 448) -- the FP8
 * variant of the compute dtype the QLoRA project page's configuration example
 * sets (bnb_4bit_compute_dtype); the LoRA term stays bf16:
 *   maxm = max |m_hat| over the weight's blocks; E the largest integer with
 *          maxm 2^E <= 448 (0 if maxm = 0), clamped to [-60, 60]
 *   Wq   = e4m3(fl32(q[code] * m_hat) * 2^E)      (the weight before its
 *          bf16 rounding, scaled exactly)
 *   per row m of X: E_m the largest integer with amax_m 2^E_m <= 448 (0 for
 *          an all-zero row), same clamp; Xq = e4m3(x 2^E_m)  (exact scaling)
 *   Y[m] = bf16(2^(-E_m - E) (Xq Wq^T + XAs' B)),
 *          XAs' = bf16(fl32(s XA) 2^(E_m + E))
 * e4m3(x): nearest value, ties to the even code, saturating at +-448; the
 * products accumulate in fp32.  Arguments, layouts and XA_out as for
 * qlora_linear_fwd; K % 8 == 0 (always, as K % 64 == 0).
 *   ws : ql_workspace_size(QL_OP_LINEAR_FWD_FP8, M, N, K, r) bytes.
 * Every M takes the tensor-core path (tiles of 256 tokens).  Successive calls
 * on a stream alternate between the two halves of `ws` (any initial
 * contents work), so a call's first kernels may run while the previous
 * call's GEMM finishes when they read nothing it writes.
 */
QL_API int qlora_linear_fwd_fp8(const uint16_t *X, int64_t M, const ql_nf4_tensor *W,
                         const uint16_t *A, const uint16_t *B, int32_t r,
                         float scale, uint16_t *Y, uint16_t *XA_out, void *ws,
                         size_t ws_bytes, ql_stream_t stream);

/*
 * Backward of the same layer (QLoRA abstract: gradients back-propagate through
 * the frozen 4-bit weights into the adapters; the weights get none):
 *   G  = dY B^T                       (M x r, internal)
 *   dX = dY W_hat + s G A^T           (M x K bf16 output)
 *   dA = s X^T G                      (K x r fp32 output, overwritten)
 *   dB = s (X A)^T dY                 (r x N fp32 output, overwritten)
 *   XA : M x r bf16 from the forward, or NULL to recompute it from X and A.
 *   ws : ql_workspace_size(QL_OP_LINEAR_BWD, M, N, K, r) bytes.
 */
QL_API int qlora_linear_bwd(const uint16_t *dY, const uint16_t *X, const uint16_t *XA,
                     int64_t M, const ql_nf4_tensor *W, const uint16_t *A,
                     const uint16_t *B, int32_t r, float scale, uint16_t *dX,
                     float *dA, float *dB, void *ws, size_t ws_bytes,
                     ql_stream_t stream);

/*
 * The same backward with the dX main product on 8-bit floats (E4M3, as in
 * qlora_linear_fwd_fp8, with dY in the role of X):
 *   Wq   = the E4M3 weight of qlora_linear_fwd_fp8 (same E)
 *   per row m of dY: E_m and dYq = e4m3(dy 2^E_m) by the rule of the X rows
 *   G    = dY B^T (from the bf16 dY, fp32 accumulation)
 *   dX[m] = bf16(2^(-E_m - E) (dYq Wq + Gs' A^T)),
 *          Gs' = bf16(fl32(s G) 2^(E_m + E))
 *   dA = s X^T bf16(G), dB = s (X A)^T dY     (fp32, overwritten; bf16
 *          operands as in qlora_linear_bwd)
 * Arguments and layouts as for qlora_linear_bwd; N % 16 == 0 (the rows of
 * the dY codes are TMA rows), else QL_ERR_UNSUPPORTED.
 *   ws : ql_workspace_size(QL_OP_LINEAR_BWD_FP8, M, N, K, r) bytes.
 * Every M takes the tensor-core path (tiles of 256 tokens).  Successive calls
 * on a stream alternate between the two halves of `ws` (any initial
 * contents work), so a call's first kernels may run while the previous
 * call's GEMM finishes when they read nothing it writes.
 */
QL_API int qlora_linear_bwd_fp8(const uint16_t *dY, const uint16_t *X, const uint16_t *XA,
                         int64_t M, const ql_nf4_tensor *W, const uint16_t *A,
                         const uint16_t *B, int32_t r, float scale, uint16_t *dX,
                         float *dA, float *dB, void *ws, size_t ws_bytes,
                         ql_stream_t stream);

/*
 * LoRA merge for inference (LoRA tutorial, Lit-LLaMA translation: the
 * low-rank update can be added into the weight after training, W' = W + dW,
 * so that inference costs nothing extra):
 *   W_out = bf16(w_hat + s (A B)^T)   N x K bf16 (device), row n, column k:
 *           bf16_rne(fl32(w_hat[n][k] + s * acc)), acc = sum_j A[k][j] B[j][n]
 *           accumulated in fp32, w_hat the dequantized weight.
 *   W : N x K NF4 (input), A : K x r bf16, B : r x N bf16, scale : s.
 * With B = 0 the output is w_hat exactly.  To store the merged weight in NF4
 * again, pass W_out to nf4_quantize.  Reads the weight once and writes W_out
 * once; no workspace.
 */
QL_API int qlora_merge(const ql_nf4_tensor *W, const uint16_t *A, const uint16_t *B, int32_t r, float scale,
                       uint16_t *W_out, ql_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word, which kernels set when a bounded wait gives up.  Returns QL_OK,
 * QL_ERR_TIMEOUT, or QL_ERR_CUDA if the synchronisation itself failed.
 */
QL_API int ql_get_device_status(ql_stream_t stream);

/*
 * Optional timing of the tensor-core GEMM launches, off by default.
 * ql_timing_start(capacity): from now on every tensor-core GEMM that this host
 *   thread launches is bracketed by a CUDA event pair recorded on its stream
 *   (up to `capacity` launches; later ones are not timed).  Creates the events.
 * ql_timing_stop(total_ms, launches, flops): waits for the recorded events,
 *   writes the summed launch durations (ms), the number of timed launches and
 *   their summed algorithmic flops (2 M N_out (K_red + r) each) to host
 *   memory, destroys the events and turns timing off.
 * Device work is unchanged; only event records are added to the stream.
 */
QL_API int ql_timing_start(int capacity);
QL_API int ql_timing_stop(float *total_ms, int *launches, double *flops);

/*
 * Optional span record of the tensor-core GEMM launches, off by default (no
 * counterpart in the pages: it measures the library's own kernels inside a
 * running sequence of calls, where event records between launches would
 * stop the programmatic overlap of consecutive kernels).
 * ql_spans_start(buf, capacity): from now on, tensor-core GEMM launch i that
 *   this host thread makes (i < capacity) records into the caller's DEVICE
 *   buffer `buf` (2 * capacity uint64, 8-byte aligned): buf[2i] = the
 *   earliest %globaltimer (ns) at which one of its CTAs passed its dependency
 *   wait (atomic min), buf[2i + 1] = the latest at which one finished (atomic
 *   max).  The caller sets buf[2i] = UINT64_MAX and buf[2i + 1] = 0 first.
 * ql_spans_stop(launches, flops): turns recording off and writes the number
 *   of recorded launches and their summed algorithmic flops
 *   (2 M N_out (K_red + r) each) to host memory.  The caller reads `buf`
 *   once the launches have completed.
 * Each recording CTA adds two global atomics; nothing else changes.
 */
QL_API int ql_spans_start(uint64_t *device_buffer, int capacity);
QL_API int ql_spans_stop(int *launches, double *flops);

/*
 * Self-test of the failure path (no counterpart in the pages: it checks the
 * library's own bounded waits).  Launches one kernel on `stream` whose wait on
 * a barrier can never be satisfied; after `limit_ns` nanoseconds of wall time
 * (0 < limit_ns <= 2e9) the kernel gives up, records the timeout in the device
 * status word and returns, exactly as any library kernel does when a wait
 * runs out.  A following ql_get_device_status(stream) then returns
 * QL_ERR_TIMEOUT (and clears the word); the CUDA context stays usable.
 * Returns QL_OK once the kernel is launched, QL_ERR_INVALID for a limit
 * outside the range, QL_ERR_CUDA if the launch fails.
 */
QL_API int ql_selftest_wait(int64_t limit_ns, ql_stream_t stream);

/* Number of CUDA kernels the library has launched in this process. */
QL_API uint64_t ql_launch_count(void);

/* Message for the last error returned on this host thread ("" if none). */
QL_API const char *ql_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_H */
