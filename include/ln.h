/*
 * ln.h -- C ABI of the GB300 (sm_103a) fused residual-add + LayerNorm library (libln.so),
 * with the bias + dropout + residual prologue (ln_fwd_bias_dropout_*, ln_dropout_bwd_*), the
 * fused residual-add + RMSNorm (ln_rms_*), the fused row softmax (ln_softmax_*) and the fused
 * cross-entropy (ln_xent_*) alongside.
 *
 * The library computes, for a row-major [rows, cols] problem:
 *
 *   forward   s = x + res                      (stored as res_out, rounded to the I/O type)
 *             mu = mean(s), var = mean((s - mu)^2), rstd = 1 / sqrt(var + eps)
 *             out = gamma * (s - mu) * rstd + beta
 *   backward  xhat = (s - mu) * rstd, g = gamma * dy
 *             dx = rstd * (g - (sum_j g_j + xhat * sum_j g_j xhat_j) / cols)
 *             dgamma = sum over rows of dy * xhat,  dbeta = sum over rows of dy
 *
 * Definitions: "Accelerating Transformer on GPU (II): Training with LightSeq2", section 2.1
 * (forward; the HW4 form of the backward; dgamma and dbeta) and section 2.4 (column sums);
 * the residual sum is written out and then normalised as in "llm.c: the llmc/ CUDA kernel
 * layer", section 3.2 (fused_residual_forward5).  The variance is the biased one (divide by
 * cols) and eps sits inside the square root ("AI infra learning log (2): LayerNorm operator
 * optimisation", section 2.1).  The normalised tensor is the STORED res_out (rounded to the
 * I/O type), so the backward, which sees only res_out, mu and rstd, differentiates exactly
 * the function the forward evaluated.
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers owned by the caller, on the current CUDA
 *    device; row-major and contiguous ([rows, cols] with row stride cols, [cols], [rows]).
 *  - Element types: ``float`` is fp32; ``ln_bf16`` is the raw 16-bit pattern of a bfloat16
 *    (the same bits as CUDA's __nv_bfloat16).  Arithmetic is always fp32; results stored in
 *    bf16 are rounded to nearest even.  mean and rstd are always fp32.
 *  - Calls are asynchronous on ``stream`` (NULL = the legacy default stream) and return as
 *    soon as the work is enqueued.  Argument errors are detected on the host before anything
 *    is launched; nothing is launched when a call returns an error.
 *  - Pointers need no particular alignment.  When every pointer is 16-byte aligned and a row
 *    is a multiple of 16 bytes (cols % 4 == 0 for fp32, cols % 8 == 0 for bf16) the 128-bit
 *    vector kernels run; otherwise a scalar kernel computes the same result.
 *  - Limits: 1 <= cols <= LN_MAX_COLS; 0 <= rows <= LN_MAX_ROWS.  rows == 0 is a no-op for the
 *    forward; for the backward it writes dgamma = dbeta = 0.  With rows == 0 the pointers
 *    to [rows, cols] and [rows] arrays may be NULL (empty tensors often have no storage).
 *    eps must be finite and >= 0.
 *  - Kernels are launched with programmatic dependent launch allowed (backward kernels that
 *    finish their column sums in-kernel, and the dropout backward, cooperatively).  Each
 *    kernel still waits for the work before it in the stream to finish before it touches
 *    memory, so stream order is the usual one, in CUDA graphs too.
 *  - Thread safety: entry points may be called from several host threads.  Two backward
 *    calls that share a workspace (the same stream, or the same caller-owned workspace) must
 *    not overlap on the GPU; stream order takes care of that for one stream.
 */
#ifndef LN_H_
#define LN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LN_MAX_COLS 16384
/* Largest row count (2^31 - 2^16): row indices, including a block's look-ahead of a tile
   step past its last, stay within int range. */
#define LN_MAX_ROWS 2147418112LL

/* The raw bits of one bfloat16 value. */
typedef uint16_t ln_bf16;

/* The same type as cudaStream_t; NULL selects the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* ln_stream_t;

typedef enum ln_status {
    LN_OK = 0,
    LN_EINVAL = 1,        /* a NULL required pointer, rows < 0, cols <= 0, eps < 0 or not finite */
    LN_EALIGN = 2,        /* a workspace pointer that is not 256-byte aligned */
    LN_EUNSUPPORTED = 3,  /* cols > LN_MAX_COLS, rows > LN_MAX_ROWS, or not an sm_103 device */
    LN_ECUDA = 4,         /* a CUDA runtime call failed; see ln_last_cuda_error() */
    LN_ETIMEOUT = 5,      /* a bounded device-side wait ran out (reported by ln_device_check) */
    LN_ENOSPACE = 6       /* a caller-owned workspace smaller than ln_bwd_workspace_bytes() */
} ln_status;

/*
 * Forward of the fused residual-add + LayerNorm.
 *
 *   x        [rows, cols]  input
 *   res      [rows, cols]  residual added to x; may be NULL (plain LayerNorm of x)
 *   gamma    [cols]        scale
 *   beta     [cols]        shift
 *   eps                    added to the variance inside the square root
 *   out      [rows, cols]  gamma * xhat + beta                      (written)
 *   res_out  [rows, cols]  the residual sum x + res, rounded to the I/O type (written);
 *                          may be NULL.  When res is NULL it receives a copy of x.
 *   mean     [rows] fp32   per-row mean of res_out                  (written)
 *   rstd     [rows] fp32   per-row 1 / sqrt(var + eps)              (written)
 *
 * out, res_out, mean and rstd must not overlap any input.  Nothing is allocated.
 * Errors: LN_EINVAL, LN_EUNSUPPORTED, LN_ECUDA (launch failure).
 */
ln_status ln_fwd_f32(const float* x, const float* res, const float* gamma, const float* beta,
                     float eps, int64_t rows, int64_t cols, float* out, float* res_out,
                     float* mean, float* rstd, ln_stream_t stream);

ln_status ln_fwd_bf16(const ln_bf16* x, const ln_bf16* res, const ln_bf16* gamma,
                      const ln_bf16* beta, float eps, int64_t rows, int64_t cols, ln_bf16* out,
                      ln_bf16* res_out, float* mean, float* rstd, ln_stream_t stream);

/*
 * Backward of the fused residual-add + LayerNorm.
 *
 *   dy            [rows, cols]  gradient of the loss with respect to out
 *   x_or_res_out  [rows, cols]  the tensor the forward normalised: its res_out when it had a
 *                               residual, else its x
 *   gamma         [cols]
 *   mean, rstd    [rows] fp32   as written by the forward
 *   dx            [rows, cols]  gradient with respect to s = x + res, and therefore with
 *                               respect to both x and res (OVERWRITTEN, not accumulated)
 *   dgamma        [cols]        sum over rows of dy * xhat                (overwritten)
 *   dbeta         [cols]        sum over rows of dy                       (overwritten)
 *
 * The two row sums are taken in one reduction (HW4 form, "Training with LightSeq2",
 * section 2.2).  dgamma and dbeta are reduced in two deterministic stages without float
 * atomics (section 2.4; the last-block-finishes scheme of "llm.c: the llmc/ CUDA kernel
 * layer", section 3.3): each thread block writes fp32 partial column sums over a fixed set
 * of rows to a workspace (compensated, as (hi, lo) pairs, for fp32 I/O); the blocks that own
 * a slice of the columns read every block's partials of that slice as they land (a stored
 * partial is never the all-zero word, and the workspace is all zero between calls, so a zero
 * word is one not yet written), add them in a fixed order, and zero the words they read.
 * The result is bitwise identical from run to run on the same device and build.
 *
 * This variant uses a workspace owned by the library, one per (device, stream), allocated
 * with cudaMalloc on first use and grown when a larger problem arrives; ln_release() frees
 * them.  The first call on a stream (and a call that grows its workspace) must therefore
 * not happen during CUDA graph capture; use the _ws variant there.
 * Errors: LN_EINVAL, LN_EUNSUPPORTED, LN_ECUDA.
 */
ln_status ln_bwd_f32(const float* dy, const float* x_or_res_out, const float* gamma,
                     const float* mean, const float* rstd, float* dx, float* dgamma,
                     float* dbeta, int64_t rows, int64_t cols, ln_stream_t stream);

ln_status ln_bwd_bf16(const ln_bf16* dy, const ln_bf16* x_or_res_out, const ln_bf16* gamma,
                      const float* mean, const float* rstd, ln_bf16* dx, ln_bf16* dgamma,
                      ln_bf16* dbeta, int64_t rows, int64_t cols, ln_stream_t stream);

/*
 * Size in bytes of the caller-owned workspace the _ws backward variants need for a
 * [rows, cols] problem on the current device (an upper bound over element types and
 * alignments).  Returns 0 for invalid sizes or when no device is available.
 */
size_t ln_bwd_workspace_bytes(int64_t rows, int64_t cols);

/*
 * Backward with a caller-owned device workspace (256-byte aligned, at least
 * ln_bwd_workspace_bytes(rows, cols) bytes).  The caller must zero the whole workspace once
 * before its first use; every completed call leaves it all zero again, so it can be reused
 * by later calls in stream order (of any shape that fits) without clearing.  After
 * LN_ETIMEOUT it must be zeroed again: a call that gave up may leave partial sums in it.
 * Nothing is allocated.
 * Errors: as ln_bwd_*, plus LN_EALIGN and LN_ENOSPACE.
 */
ln_status ln_bwd_f32_ws(const float* dy, const float* x_or_res_out, const float* gamma,
                        const float* mean, const float* rstd, float* dx, float* dgamma,
                        float* dbeta, int64_t rows, int64_t cols, void* workspace,
                        size_t workspace_bytes, ln_stream_t stream);

ln_status ln_bwd_bf16_ws(const ln_bf16* dy, const ln_bf16* x_or_res_out, const ln_bf16* gamma,
                         const float* mean, const float* rstd, ln_bf16* dx, ln_bf16* dgamma,
                         ln_bf16* dbeta, int64_t rows, int64_t cols, void* workspace,
                         size_t workspace_bytes, ln_stream_t stream);

/*
 * Forward of the fused residual-add + RMSNorm ("GPU Performance from First Principles",
 * section 6.1, the fused add + RMSNorm, and its exercise 4: one kernel reads x and the
 * residual and writes the new residual stream and the normalised result).  The page names
 * the operation without printing its formula; this library takes the usual RMSNorm: no mean
 * is subtracted, no shift added, eps is added to the mean square inside the square root:
 *
 *   s = x + res (stored as res_out, rounded to the I/O type),  r = 1 / sqrt(mean(s^2) + eps),
 *   out = gamma * s * r.
 *
 *   x, res, gamma, eps, out, res_out   as for ln_fwd_* (res and res_out may be NULL)
 *   rrms     [rows] fp32   per-row r                                 (written)
 *
 * Conventions, limits and errors are those of ln_fwd_*.  Nothing is allocated.
 */
ln_status ln_rms_fwd_f32(const float* x, const float* res, const float* gamma, float eps,
                         int64_t rows, int64_t cols, float* out, float* res_out, float* rrms,
                         ln_stream_t stream);

ln_status ln_rms_fwd_bf16(const ln_bf16* x, const ln_bf16* res, const ln_bf16* gamma, float eps,
                          int64_t rows, int64_t cols, ln_bf16* out, ln_bf16* res_out, float* rrms,
                          ln_stream_t stream);

/*
 * Backward of the fused residual-add + RMSNorm, from the forward by the chain rule: with
 * shat = s * r and g = gamma * dy,
 *
 *   dx = r * (g - shat * sum_j g_j shat_j / cols)   (one row sum; gradient of s, hence of
 *                                                     x and res; OVERWRITTEN)
 *   dgamma = sum over rows of dy * shat             (overwritten)
 *
 *   dy, x_or_res_out, gamma, dx, dgamma   as for ln_bwd_* (x_or_res_out: the tensor the
 *                                         forward normalised)
 *   rrms     [rows] fp32   as written by ln_rms_fwd_*
 *
 * dgamma is reduced in the same two deterministic stages as ln_bwd_*'s (no float atomics,
 * bitwise identical run to run).  The plain variants use the library-owned workspace of the
 * stream, the _ws variants a caller-owned one of at least ln_bwd_workspace_bytes(rows, cols)
 * bytes, exactly as for ln_bwd_* and ln_bwd_*_ws (which may share it in stream order).
 */
ln_status ln_rms_bwd_f32(const float* dy, const float* x_or_res_out, const float* gamma,
                         const float* rrms, float* dx, float* dgamma, int64_t rows, int64_t cols,
                         ln_stream_t stream);

ln_status ln_rms_bwd_bf16(const ln_bf16* dy, const ln_bf16* x_or_res_out, const ln_bf16* gamma,
                          const float* rrms, ln_bf16* dx, ln_bf16* dgamma, int64_t rows,
                          int64_t cols, ln_stream_t stream);

ln_status ln_rms_bwd_f32_ws(const float* dy, const float* x_or_res_out, const float* gamma,
                            const float* rrms, float* dx, float* dgamma, int64_t rows,
                            int64_t cols, void* workspace, size_t workspace_bytes,
                            ln_stream_t stream);

ln_status ln_rms_bwd_bf16_ws(const ln_bf16* dy, const ln_bf16* x_or_res_out,
                             const ln_bf16* gamma, const float* rrms, ln_bf16* dx,
                             ln_bf16* dgamma, int64_t rows, int64_t cols, void* workspace,
                             size_t workspace_bytes, ln_stream_t stream);

/*
 * Fused row softmax, forward ("Accelerating Transformer on GPU (I)", section 4.1: scale,
 * add the mask, row maximum, exponentiate, row sum and divide in one kernel).  For each row
 * r of a row-major [rows, cols] problem:
 *
 *   z = scale * x + mask[r % mask_rows],   y = exp(z - max z) / sum exp(z - max z).
 *
 *   x      [rows, cols]       input (attention scores, say: rows = batch * heads * queries)
 *   mask   [mask_rows, cols]  additive mask (0 keeps an entry, -inf removes it), its rows
 *                             repeating every mask_rows rows; may be NULL (no mask; then
 *                             mask_rows is ignored)
 *   scale                     factor on x (finite)
 *   y      [rows, cols]       written; must not overlap x or mask
 *
 * A row whose entries are all -inf has no softmax; y is NaN there (0 / 0), as the
 * definition gives.  Conventions, limits and errors as for ln_fwd_*; nothing is allocated.
 */
ln_status ln_softmax_fwd_f32(const float* x, const float* mask, int64_t mask_rows, float scale,
                             int64_t rows, int64_t cols, float* y, ln_stream_t stream);

ln_status ln_softmax_fwd_bf16(const ln_bf16* x, const ln_bf16* mask, int64_t mask_rows,
                              float scale, int64_t rows, int64_t cols, ln_bf16* y,
                              ln_stream_t stream);

/*
 * Fused row softmax, backward ("Accelerating Transformer on GPU (II): Training with
 * LightSeq2", section 3.1: only the forward's output y is needed, and one row reduction):
 *
 *   dx = scale * y * (dy - sum_j dy_j y_j)      (the mask has no gradient)
 *
 *   dy, y  [rows, cols]   upstream gradient and the forward's output
 *   scale                 the forward's factor on x
 *   dx     [rows, cols]   written (may alias dy); must not overlap y
 *
 * Conventions, limits and errors as for ln_fwd_*; nothing is allocated.
 */
ln_status ln_softmax_bwd_f32(const float* dy, const float* y, float scale, int64_t rows,
                             int64_t cols, float* dx, ln_stream_t stream);

ln_status ln_softmax_bwd_bf16(const ln_bf16* dy, const ln_bf16* y, float scale, int64_t rows,
                              int64_t cols, ln_bf16* dx, ln_stream_t stream);

/*
 * Fused cross-entropy with label smoothing, forward and backward in one kernel
 * ("Accelerating Transformer on GPU (I): Kernel Fusion and LightSeq Inference", section 5.2;
 * the fused classifier of "llm.c: the llmc/ CUDA kernel layer", section 6).  For each row r
 * of V logits x with target t = targets[r]:
 *
 *   p = (1 - alpha) onehot(t) + alpha / V,   q = softmax(x)
 *   losses[r] = -sum_j p_j log q_j = log Z + m - [(1 - alpha) x_t + (alpha / V) sum_j x_j]
 *   dlogits   = dloss * (q - p)
 *
 * with m = max x and Z = sum exp(x - m).
 *
 *   logits   [rows, V]  input
 *   targets  [rows]     int32, each in [0, V) (a row with another target gets a NaN loss)
 *   alpha               label smoothing, 0 <= alpha <= 1
 *   dloss               factor of the gradient (1 / rows for a mean over rows)
 *   losses   [rows]     fp32, written; may be NULL
 *   dlogits  [rows, V]  written; may be NULL; may be the logits themselves (the gradient
 *                       then overwrites them in place)
 *
 * At least one of losses and dlogits must be given.  Limits: 1 <= V <= LN_XENT_MAX_V,
 * 0 <= rows <= LN_MAX_ROWS.  Other conventions and errors as for ln_fwd_*.
 */
#define LN_XENT_MAX_V (1 << 24)

ln_status ln_xent_f32(const float* logits, const int32_t* targets, int64_t rows, int64_t V,
                      float alpha, float dloss, float* losses, float* dlogits,
                      ln_stream_t stream);

ln_status ln_xent_bf16(const ln_bf16* logits, const int32_t* targets, int64_t rows, int64_t V,
                       float alpha, float dloss, float* losses, ln_bf16* dlogits,
                       ln_stream_t stream);

/*
 * LayerNorm forward with the bias + dropout + residual prologue fused in ("Accelerating
 * Transformer on GPU (I): Kernel Fusion and LightSeq Inference", section 2.3: after a linear
 * layer, add its bias, apply dropout, add the residual -- one kernel instead of three):
 *
 *   s = res + keep * (h + bias) / (1 - p)        (stored as res_out, rounded to the I/O type)
 *   out, mean, rstd = the LayerNorm of s exactly as ln_fwd_*
 *
 * keep is 0 with probability p: element i = row * cols + col is kept when word i % 4 of the
 * counter-based generator Philox-4x32-10 (Salmon, Moraes, Dror and Shaw, SC 2011) at counter
 * (i / 4 as two 32-bit words, offset as two 32-bit words) under key (seed as two 32-bit
 * words) is at least floor(p * 2^32).  The mask is a pure function of (seed, offset, i), so
 * the backward regenerates it and nothing need be stored (the _keep variants below also
 * store it, as bits, for a backward that reads them).  Use a new offset (or seed) per call.
 *
 *   h        [rows, cols]  the linear layer's output
 *   bias     [cols]        its bias
 *   res      [rows, cols]  the residual (required)
 *   p                      drop probability, 0 <= p < 1
 *   the rest               as for ln_fwd_*
 *
 * Errors as for ln_fwd_*; LN_EINVAL also for a NULL bias or res or p outside [0, 1).
 */
ln_status ln_fwd_bias_dropout_f32(const float* h, const float* bias, const float* res,
                                  const float* gamma, const float* beta, float eps, float p,
                                  uint64_t seed, uint64_t offset, int64_t rows, int64_t cols,
                                  float* out, float* res_out, float* mean, float* rstd,
                                  ln_stream_t stream);

ln_status ln_fwd_bias_dropout_bf16(const ln_bf16* h, const ln_bf16* bias, const ln_bf16* res,
                                   const ln_bf16* gamma, const ln_bf16* beta, float eps, float p,
                                   uint64_t seed, uint64_t offset, int64_t rows, int64_t cols,
                                   ln_bf16* out, ln_bf16* res_out, float* mean, float* rstd,
                                   ln_stream_t stream);

/*
 * Backward of the prologue.  ds is the gradient with respect to s -- the dx that ln_bwd_*
 * returns for the forward's res_out, mean and rstd, which is also the residual's gradient:
 *
 *   dh    = ds * keep / (1 - p)          [rows, cols]  (written)
 *   dbias = sum over rows of dh          [cols]        (written; bitwise reproducible, no
 *                                                       float atomics)
 *
 * p, seed and offset must be the forward's.  The plain variants use the library-owned
 * workspace of the stream, the _ws variants a caller-owned one of at least
 * ln_bwd_workspace_bytes(rows, cols) bytes (shared with ln_bwd_* in stream order); every
 * completed call leaves it all zero.  Errors as for ln_bwd_*.
 */
ln_status ln_dropout_bwd_f32(const float* ds, float p, uint64_t seed, uint64_t offset,
                             int64_t rows, int64_t cols, float* dh, float* dbias,
                             ln_stream_t stream);

ln_status ln_dropout_bwd_bf16(const ln_bf16* ds, float p, uint64_t seed, uint64_t offset,
                              int64_t rows, int64_t cols, ln_bf16* dh, ln_bf16* dbias,
                              ln_stream_t stream);

ln_status ln_dropout_bwd_f32_ws(const float* ds, float p, uint64_t seed, uint64_t offset,
                                int64_t rows, int64_t cols, float* dh, float* dbias,
                                void* workspace, size_t workspace_bytes, ln_stream_t stream);

ln_status ln_dropout_bwd_bf16_ws(const ln_bf16* ds, float p, uint64_t seed, uint64_t offset,
                                 int64_t rows, int64_t cols, ln_bf16* dh, ln_bf16* dbias,
                                 void* workspace, size_t workspace_bytes, ln_stream_t stream);

/*
 * The prologue with its keep decisions stored for the backward ("Accelerating Transformer on
 * GPU (II): Training with LightSeq2", section 3.2: the dropout backward needs the forward's
 * mask; LightSeq keeps one byte per element, this keeps one bit).  The forward decides each
 * element anyway; the _keep forward also writes the decisions as bits:
 *
 *   bit (col % 8) of keep[row * ceil(cols / 8) + col / 8] = 1  when (row, col) is kept
 *
 * (rows padded to whole bytes; the pad bits of a row's last byte are 0), and the _keep
 * backward reads them instead of running the generator again -- its result is bit for bit
 * that of ln_dropout_bwd_* with the forward's (p, seed, offset).  keep: caller-owned device
 * memory of ln_dropout_keep_bytes(rows, cols) bytes.  Arguments, workspace rules and errors as
 * for ln_fwd_bias_dropout_* / ln_dropout_bwd_*, plus LN_EINVAL for a NULL keep with
 * rows > 0.  ln_dropout_keep_bytes returns 0 for invalid sizes.
 */
size_t ln_dropout_keep_bytes(int64_t rows, int64_t cols);

ln_status ln_fwd_bias_dropout_keep_f32(const float* h, const float* bias, const float* res,
                                       const float* gamma, const float* beta, float eps, float p,
                                       uint64_t seed, uint64_t offset, int64_t rows, int64_t cols,
                                       float* out, float* res_out, float* mean, float* rstd,
                                       uint8_t* keep, ln_stream_t stream);

ln_status ln_fwd_bias_dropout_keep_bf16(const ln_bf16* h, const ln_bf16* bias,
                                        const ln_bf16* res, const ln_bf16* gamma,
                                        const ln_bf16* beta, float eps, float p, uint64_t seed,
                                        uint64_t offset, int64_t rows, int64_t cols,
                                        ln_bf16* out, ln_bf16* res_out, float* mean, float* rstd,
                                        uint8_t* keep, ln_stream_t stream);

ln_status ln_dropout_bwd_keep_f32(const float* ds, float p, const uint8_t* keep, int64_t rows,
                                  int64_t cols, float* dh, float* dbias, ln_stream_t stream);

ln_status ln_dropout_bwd_keep_bf16(const ln_bf16* ds, float p, const uint8_t* keep,
                                   int64_t rows, int64_t cols, ln_bf16* dh, ln_bf16* dbias,
                                   ln_stream_t stream);

ln_status ln_dropout_bwd_keep_f32_ws(const float* ds, float p, const uint8_t* keep,
                                     int64_t rows, int64_t cols, float* dh, float* dbias,
                                     void* workspace, size_t workspace_bytes, ln_stream_t stream);

ln_status ln_dropout_bwd_keep_bf16_ws(const ln_bf16* ds, float p, const uint8_t* keep,
                                      int64_t rows, int64_t cols, ln_bf16* dh, ln_bf16* dbias,
                                      void* workspace, size_t workspace_bytes,
                                      ln_stream_t stream);

/*
 * Backward (bf16) that allocates nothing.  The pages have no counterpart to this entry
 * point: it exists for callers that cannot call cudaMalloc when they run the backward --
 * a serving process that reserved its whole device-memory budget at start-up, or a plugin
 * whose host framework owns every device allocation -- and cannot hand in a workspace
 * either.  Arguments, results and errors are those of ln_bwd_bf16, and so are the kernels,
 * the LN_CHECK handling, ln_last_launch_count and the test hooks; the scratch (the
 * per-block partial sums) lives in a fixed array of LN_NOALLOC_SCRATCH_BYTES (16 MiB)
 * compiled into the library, which every GPU that loads the library holds until exit.
 *  - Size limit: every problem with ln_bwd_workspace_bytes(rows, cols) <=
 *    LN_NOALLOC_SCRATCH_BYTES is accepted (that bound covers every kernel choice, so a
 *    caller can check it in advance); some larger ones fit too, and those that do not are
 *    rejected with LN_EUNSUPPORTED before anything is launched.  8192 x 768 fits by
 *    that rule, 8192 x 1280 fits as well, 4096 x 8192 does not.
 *  - The first call on each device looks up the array's device address (once, with that
 *    device current); make that first call before any stream capture begins.
 *  - All calls share the one array, which every completed call leaves all zero (after
 *    LN_ETIMEOUT, ln_device_check zeroes it on the stream it is given): calls whose work
 *    overlaps on the GPU (different streams, or different host threads without ordering)
 *    race and corrupt each other's results; order them.
 *  - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 */
#define LN_NOALLOC_SCRATCH_BYTES (16u << 20)

ln_status ln_bwd_bf16_noalloc(const ln_bf16* dy, const ln_bf16* x_or_res_out,
                              const ln_bf16* gamma, const float* mean, const float* rstd,
                              ln_bf16* dx, ln_bf16* dgamma, ln_bf16* dbeta, int64_t rows,
                              int64_t cols, ln_stream_t stream);

/*
 * Device-side status.  Every wait inside a kernel (the bulk-copy barriers, the backward's
 * polls for other blocks' partial sums) is bounded; when one runs out the
 * kernel records LN_ETIMEOUT in a per-device status word and returns early without
 * faulting.  ln_device_check synchronizes ``stream``, reads and clears that word on the
 * current device and, if it was set, re-zeroes the library-owned workspace of ``stream`` and
 * the allocation-free entry point's array with copies enqueued on ``stream`` (so they are
 * ordered before later work on it) and waits for them; it returns LN_OK or LN_ETIMEOUT
 * (LN_ECUDA if a CUDA call fails).  Setting the environment
 * variable LN_CHECK=1 makes every entry point do this before returning
 * (except for calls made while their stream is being captured into a CUDA graph, which cannot
 * synchronise).
 */
ln_status ln_device_check(ln_stream_t stream);

/* Frees every library-owned workspace on every device (synchronizes those devices). */
ln_status ln_release(void);

/* A static, human-readable name for a status code. */
const char* ln_status_str(ln_status status);

/* The cudaError_t value behind the most recent LN_ECUDA returned on this host thread. */
int ln_last_cuda_error(void);

/* The library's version as major * 10000 + minor * 100 + patch. */
int ln_version(void);

/*
 * Tuning and test hooks.  They change no result beyond what the tests check: every path
 * computes the same function.
 *
 * ln_debug_force_path selects the kernel family for later calls on all threads:
 * 0 = automatic (default), 1 = tile kernels, one warp per row or, for rows wider than one
 * warp's registers, 2 or 4 warps per row (128-bit vectors; falls back to automatic when the
 * row does not fit), 2 = block per row with bulk-copy (TMA) staging, 3 = scalar kernels.
 * Returns the previous setting.
 *
 * ln_debug_wait_test makes the finishing blocks of the next backward launches also wait for
 * a workspace word that nothing writes, with a wait limit of ``limit_us`` microseconds, so
 * that the bounded wait runs out and LN_ETIMEOUT is reported by ln_device_check; 0 turns it
 * off.  Used by the test of the
 * timeout path; it never faults the device.
 */
int ln_debug_force_path(int path);
void ln_debug_wait_test(unsigned limit_us);

/* Number of kernels the most recent call of this library on this host thread launched (1 for
 * most calls; 2 for a backward on the block-per-row path, whose column sums are finished by
 * a second, dependent launch). */
int ln_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LN_H_ */
