/*
 * rms_norm.h -- C ABI of the GB300 fused RMSNorm forward/backward library
 * (librms_norm_gb300.so).
 *
 * The operation.  For each row r of a row-major [rows, hidden] activation x:
 *
 *   rstd[r] = 1 / sqrt( (1/hidden) * sum_j x[r,j]^2 + eps )
 *   x_hat   = x[r,j] * rstd[r]
 *   y[r,j]  = x_hat * gain_j,   gain_j = gamma_j (offset 0) or 1 + gamma_j
 *             (offset 1, the Gemma convention)
 *
 * as written in "Den dolda avrundningen i RMSNorm" (precisit.com), section
 * "En välbekant operation" (the two displayed equations), with the Gemma
 * gain of section "Vilken konvention hör till modellen?".  Statistics are
 * accumulated in fp32 for every input type and the per-row rstd is stored in
 * fp32 (Liger-Kernel PR #92 "feat: correct casts in RMSNorm to match
 * references", the author's comment after the benchmark tables).
 *
 * The backward is the exact derivative of the forward (candle PR #4059 "Add
 * backward passes to the fused rms_norm, layer_norm and softmax_last_dim
 * ops" adds it with f32 statistics for half types but prints no formula):
 *
 *   g       = dy[r,j] * gain_j
 *   c[r]    = (1/hidden) * sum_j g * x_hat
 *   dx[r,j] = rstd[r] * (g - x_hat * c[r])
 *   dw[j]   = sum_r dy[r,j] * x_hat      (fp32)
 *
 * Conventions common to every entry point:
 *  - All data pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no device memory, keeps no per-call state and never
 *    synchronises the stream.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) of the current device; results are ready when the stream is.
 *  - Layout: x, y, dy, dx are contiguous row-major [rows, hidden]; gamma and
 *    dw are [hidden]; rstd is [rows].  x, gamma, y, dy, dx share `dtype`;
 *    rstd, dw and the workspace are fp32.
 *  - 128-bit vector kernels run when every [rows, hidden] and [hidden] pointer
 *    is 16-byte aligned and hidden * element size is a multiple of 16; any
 *    other alignment runs a scalar kernel with the same results.
 *  - Every argument is checked on the host before anything is enqueued; on
 *    an error nothing is enqueued and the status says why.  No C++ exception
 *    crosses this interface.
 */
#ifndef RMS_NORM_GB300_H
#define RMS_NORM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage type of x, gamma, y, dy and dx. */
enum rmsn_dtype { RMSN_F32 = 0, RMSN_BF16 = 1, RMSN_F16 = 2 };

/* Where the forward output is rounded ("Den dolda avrundningen i RMSNorm",
 * section "Två ställen att avrunda"):
 *   RMSN_ROUND_ONCE  -- y = round(x_hat * gain), the product taken in fp32;
 *   RMSN_ROUND_TWICE -- y = round(round(x_hat) * gain), x_hat rounded to the
 *                       storage type before the gain multiply (the Llama /
 *                       MLX convention).
 * Both round to nearest, ties to even.  For RMSN_F32 the two coincide. */
enum rmsn_cast_mode { RMSN_ROUND_ONCE = 0, RMSN_ROUND_TWICE = 1 };

enum rmsn_status {
  RMSN_OK = 0,
  RMSN_ERR_NULL = 1,       /* a required pointer is NULL */
  RMSN_ERR_SHAPE = 2,      /* rows < 0, hidden < 1, hidden > RMSN_MAX_HIDDEN,
                              or rows > RMSN_MAX_ROWS */
  RMSN_ERR_EPS = 3,        /* eps negative, NaN or infinite */
  RMSN_ERR_DTYPE = 4,      /* dtype not one of rmsn_dtype */
  RMSN_ERR_ALIGN = 5,      /* workspace not 16-byte aligned */
  RMSN_ERR_WORKSPACE = 6,  /* workspace smaller than rms_norm_bwd_workspace_size */
  RMSN_ERR_CUDA = 7,       /* a CUDA call failed (see rms_norm_last_cuda_error) */
  RMSN_ERR_ARG = 8         /* offset not 0/1 or cast_mode not a rmsn_cast_mode */
};

#define RMSN_MAX_HIDDEN 65536
#define RMSN_MAX_ROWS 2147483647LL
/* Upper bound on the number of fp32 weight-gradient partial rows the
 * backward keeps in its workspace. */
#define RMSN_MAX_PARTIALS 1024

/*
 * Forward.  Reads x [rows, hidden] and gamma [hidden]; writes y [rows,
 * hidden] in `dtype` and rstd [rows] in fp32.  `eps` is added to the mean of
 * squares under the root; it must be finite and >= 0.  `offset` 1 uses the
 * gain 1 + gamma (formed in fp32).  `cast_mode` is a rmsn_cast_mode.
 * rows == 0 enqueues nothing and returns RMSN_OK (x, y, rstd may then be
 * NULL).  x and y must not overlap.
 */
int rms_norm_fwd(const void* x, const void* gamma, void* y, float* rstd,
                 int64_t rows, int64_t hidden, float eps, int offset,
                 int dtype, int cast_mode, void* stream);

/*
 * Bytes of fp32 workspace rms_norm_bwd needs for these sizes: room for
 * min(rows, RMSN_MAX_PARTIALS) partial weight-gradient rows of `hidden`
 * floats.  Depends only on its arguments (no device query).  Returns 0 for
 * invalid arguments and for rows == 0.
 */
size_t rms_norm_bwd_workspace_size(int64_t rows, int64_t hidden, int dtype);

/*
 * Backward.  Reads dy, x [rows, hidden], gamma [hidden] and the fp32 rstd
 * [rows] cached by the forward; writes dx [rows, hidden] in `dtype` and
 * OVERWRITES dw [hidden] (fp32) with the weight gradient summed over all rows.
 * The cast mode of the forward does not enter: the gradient is that of the
 * unrounded forward.  `workspace` is caller-owned device scratch of at least
 * rms_norm_bwd_workspace_size(rows, hidden, dtype) bytes, 16-byte aligned;
 * its contents need no initialisation and are clobbered.  dw is reduced in a
 * fixed order from fp32 partials over blocks of rows, one block per CTA of
 * the launch, or per cluster of CTAs for rows split over a cluster (the rows
 * split evenly over them, whose count the row width, the GPU's SM count and
 * the SM budget set; within a block the rows are added in row order):
 * partial b goes to lane b mod 16, each lane adds its partials in
 * increasing b, and the 16 lane sums are added in order.  Repeated calls
 * with the same sizes and SM budget therefore give bit-identical results.
 * rms_norm_bwd_blocked takes the block size from the caller instead, for
 * results that do not depend on the GPU or on how the rows are split.  rows == 0 zero-fills dw and returns
 * RMSN_OK (dy, x, rstd, dx, workspace may then be NULL).  Outputs must not
 * overlap inputs.
 */
int rms_norm_bwd(const void* dy, const void* x, const void* gamma,
                 const float* rstd, void* dx, float* dw,
                 int64_t rows, int64_t hidden, int offset, int dtype,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * The weight gradient over caller-chosen row blocks, for results that do not
 * depend on the GPU, on the SM budget, or on how the rows are split between
 * calls or ranks.  The pages fix the precision of dw (fp32, Liger-Kernel PR
 * #92, the author's comment after the benchmark tables) but not its
 * summation order; this fixes one that every split can reproduce:
 *
 *   the rows are cut into blocks of `block_rows` consecutive rows (the last
 *   may be shorter); block b's partial is sum over its rows, in row order, of
 *   dy * x_hat in fp32;
 *   the block partials form chunks of RMSN_DW_CHUNK_BLOCKS (32) consecutive
 *   blocks (the last may be shorter); with p_k the chunk's k-th partial (a
 *   missing one counting as +0) and s_t = p_t + p_(t+16), the chunk's sum is
 *   ((s_0 + s_1) + s_2) + ... + s_15;
 *   dw = ((chunk 0's sum + chunk 1's sum) + chunk 2's sum) + ... in chunk
 *   order.
 *
 * rms_norm_bwd_blocked computes dx (as rms_norm_bwd) and the chunk sums of
 * its rows into chunk_sums [rms_norm_dw_chunk_count(rows, block_rows),
 * hidden] fp32 (device, caller-owned, overwritten); rms_norm_dw_sum adds
 * nchunks chunk sums [nchunks, hidden] in order into dw [hidden] (nchunks
 * == 0 zero-fills dw).  One call over all rows followed by rms_norm_dw_sum
 * gives the same bits as any split of the rows into runs of whole chunks --
 * one call per run, the runs' chunk sums laid end to end in row order --
 * followed by rms_norm_dw_sum: a data-parallel job gathers the ranks' chunk
 * sums (e.g. an all-gather) instead of summing their dw.
 * rms_norm_rank_rows gives rank `rank` of `world` its slab of `rows` rows:
 * [*row_lo, *row_hi), whole chunks, the chunks split as evenly as possible
 * (a slab may be empty when there are fewer chunks than ranks).
 *
 * `workspace` holds the block partials:
 * rms_norm_bwd_blocked_workspace_size(rows, hidden, block_rows) bytes,
 * 16-byte aligned, contents clobbered.  block_rows >= 1 (RMSN_ERR_ARG
 * otherwise).  The kernels deal whole blocks to CTAs: a block of more rows
 * than an even split of the rows over the SMs would give one SM leaves SMs
 * idle, and small blocks cost partial traffic (4 * hidden bytes per block,
 * written and read once).  rows == 0 enqueues nothing (0 chunks).
 * rms_norm_dw_chunk_count returns -RMSN_ERR_SHAPE for invalid arguments, the
 * workspace size 0.  Errors otherwise as rms_norm_bwd.
 */
#define RMSN_DW_CHUNK_BLOCKS 32
size_t rms_norm_bwd_blocked_workspace_size(int64_t rows, int64_t hidden, int64_t block_rows);
int64_t rms_norm_dw_chunk_count(int64_t rows, int64_t block_rows);
int rms_norm_bwd_blocked(const void* dy, const void* x, const void* gamma,
                         const float* rstd, void* dx, float* chunk_sums,
                         int64_t rows, int64_t hidden, int64_t block_rows,
                         int offset, int dtype, void* workspace,
                         size_t workspace_bytes, void* stream);
int rms_norm_dw_sum(const float* chunk_sums, int64_t nchunks, int64_t hidden,
                    float* dw, void* stream);
int rms_norm_rank_rows(int64_t rows, int64_t block_rows, int world, int rank,
                       int64_t* row_lo, int64_t* row_hi);

/*
 * SM budget: the persistent kernels of every entry point launch at most as
 * many CTAs as `sms` SMs hold resident at once (one per SM for the staged
 * kernels), which leaves the other SMs to work running beside them on other
 * streams (a collective, a GEMM).  0 (the default) uses every SM.  A
 * process-wide setting read at each launch; change it between calls, not
 * during them.  The pages describe no such knob.  Returns RMSN_ERR_ARG for
 * sms < 0; rms_norm_sm_budget returns the current setting.
 */
int rms_norm_set_sm_budget(int sms);
int rms_norm_sm_budget(void);

/*
 * RMSNorm forward with an FP8 output and a per-tensor scale ("Den dolda
 * avrundningen i RMSNorm", section "Var implementationerna skiljer sig", the
 * Transformer Engine paragraph and footnote 3): the normalisation, the gain
 * and the output scale are applied in fp32 and only the final conversion to
 * FP8 rounds:
 *
 *   rstd[r] = 1 / sqrt( (1/hidden) sum_j x[r,j]^2 + eps )        (fp32)
 *   y[r,j]  = e4m3( ((x[r,j] * rstd[r]) * gain_j) * scale )
 *
 * gain_j = gamma_j (offset 0) or 1 + gamma_j (offset 1).  e4m3 is FP8 E4M3
 * (the "fn" variant: 1 sign, 4 exponent, 3 mantissa bits, no infinities,
 * largest finite value 448), rounding to nearest even and SATURATING: a
 * value beyond +-448 is stored as +-448; NaN stays NaN.
 *
 *   x, gamma  device, dtype (fp32/bf16/fp16), as rms_norm_fwd
 *   scale     device pointer to ONE fp32 value, read by the kernel (so a
 *             captured CUDA graph sees updates to it)
 *   y         device, rows x hidden bytes (E4M3 codes), row-major
 *   rstd      device, rows fp32 -- the same rstd as rms_norm_fwd, so
 *             rms_norm_bwd runs unchanged on (dy, x, gamma, rstd)
 *
 * There is no round-twice mode here.  Vector kernels run when x, gamma and
 * y are 16-byte aligned and hidden * sizeof(dtype) is a multiple of 16;
 * otherwise a scalar kernel.  Validation and error codes as rms_norm_fwd
 * (scale NULL with rows > 0: RMSN_ERR_NULL).
 */
int rms_norm_fwd_fp8(const void* x, const void* gamma, const float* scale,
                     void* y, float* rstd, int64_t rows, int64_t hidden,
                     float eps, int offset, int dtype, void* stream);

/*
 * LayerNorm, the sibling op: for each row r,
 *
 *   mean[r] = (1/hidden) sum_j x[r,j]
 *   rstd[r] = 1 / sqrt( (1/hidden) sum_j (x[r,j] - mean[r])^2 + eps )
 *   y[r,j]  = round( (x[r,j] - mean[r]) * rstd[r] * gamma_j + beta_j )
 *
 * with fp32 statistics, mean and rstd stored in fp32 (Liger-Kernel PR #1608
 * "fix(group_norm): keep the backward statistics and reductions in fp32"
 * notes layer_norm keeps them in fp32) and one rounding at the store.  The
 * backward (candle PR #4059 adds it with f32 statistics, no formula printed)
 * is the exact derivative:
 *
 *   g = dy * gamma,  c1 = mean_j g,  c2 = mean_j g * x_hat
 *   dx = rstd * (g - c1 - x_hat * c2);  dgamma = sum_r dy * x_hat;
 *   dbeta = sum_r dy   (fp32)
 *
 * Same conventions, validation and error codes as the RMSNorm entry points.
 * beta may be NULL (no bias); dbeta may be NULL (not computed).  The
 * workspace holds min(rows, RMSN_MAX_PARTIALS) partial rows of 2 * hidden
 * floats.
 */
int layer_norm_fwd(const void* x, const void* gamma, const void* beta, void* y,
                   float* mean, float* rstd, int64_t rows, int64_t hidden,
                   float eps, int dtype, void* stream);
size_t layer_norm_bwd_workspace_size(int64_t rows, int64_t hidden, int dtype);
int layer_norm_bwd(const void* dy, const void* x, const void* gamma,
                   const float* mean, const float* rstd, void* dx,
                   float* dgamma, float* dbeta, int64_t rows, int64_t hidden,
                   int dtype, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * Softmax over the last dimension (candle PR #4059 "Add backward passes to
 * the fused rms_norm, layer_norm and softmax_last_dim ops", description):
 *
 *   forward   y[r,j]  = round( exp(x[r,j] - m_r) / sum_k exp(x[r,k] - m_r) ),
 *             m_r = max_k x[r,k]; exp, the sum and the division in fp32
 *             (computed as exp(.) * (1 / sum)), one rounding at the store;
 *   backward  dx[r,j] = round( y[r,j] * (dy[r,j] - sum_k dy[r,k] * y[r,k]) ),
 *             from the forward's stored y, the sum in fp32.
 *
 * x, y, dy, dx: device, row-major [rows, cols], dtype (fp32/bf16/fp16),
 * owned by the caller; 1 <= cols <= RMSN_MAX_HIDDEN.  rows == 0 is a no-op.
 * A row of -inf (or one holding +inf) gives NaN, as the formula does.
 * Vector kernels run when the pointers are 16-byte aligned and
 * cols * sizeof(dtype) is a multiple of 16; otherwise scalar kernels.  One
 * kernel launch each, no workspace.  Errors as the RMSNorm entry points
 * (NULL pointers with rows > 0: RMSN_ERR_NULL; cols out of range:
 * RMSN_ERR_SHAPE).
 */
int softmax_fwd(const void* x, void* y, int64_t rows, int64_t cols, int dtype,
                void* stream);
int softmax_bwd(const void* dy, const void* y, void* dx, int64_t rows,
                int64_t cols, int dtype, void* stream);

/*
 * GroupNorm (Liger-Kernel PR #1608 "fix(group_norm): keep the backward
 * statistics and reductions in fp32": Mean and RSTD stored in fp32, the
 * backward's reductions in fp32).  x is [n, channels, spatial] row-major
 * (spatial = the flattened positions, e.g. H * W); the channels form
 * `groups` groups of channels / groups consecutive channels.  For each
 * sample i and group g, over the group's channels and positions:
 *
 *   mean[i,g] = average of x;  var = average of (x - mean)^2 (biased);
 *   rstd[i,g] = 1 / sqrt(var + eps)                      (fp32, stored fp32)
 *   y[i,c,s]  = round( (x[i,c,s] - mean) * rstd * gamma[c] + beta[c] )
 *
 * backward, with g = dy * gamma[c] and x_hat = (x - mean) * rstd:
 *
 *   dx = round( rstd * (g - avg_group(g) - x_hat * avg_group(g * x_hat)) )
 *   dgamma[c] = sum over samples and positions of dy * x_hat      (fp32)
 *   dbeta[c]  = sum over samples and positions of dy              (fp32)
 *
 * x, y, dy, dx: device, dtype (fp32/bf16/fp16); gamma, beta: device,
 * [channels] of the same dtype (beta may be NULL: no bias); mean, rstd:
 * device, [n, groups] fp32; dgamma, dbeta: device [channels] fp32,
 * overwritten (dbeta may be NULL: not computed).  Shapes: n >= 0,
 * channels % groups == 0, channels <= 2^24, (channels / groups) * spatial
 * <= 2^30, else RMSN_ERR_SHAPE.  n == 0: nothing to compute (the backward
 * zero-fills dgamma and dbeta).  The workspace holds fp32 partial rows of
 * the weight gradients (group_norm_bwd_workspace_size bytes, 16-byte
 * aligned); the result is reduced from them in a fixed order, so repeated
 * calls give bit-identical dgamma and dbeta.  Vector kernels (a thread-block
 * cluster of up to 16 CTAs per group) run when spatial * sizeof(dtype) is a
 * multiple of 16 and x, y (dy, dx) are 16-byte aligned; otherwise scalar
 * kernels.  Errors as the RMSNorm entry points.
 */
int group_norm_fwd(const void* x, const void* gamma, const void* beta, void* y,
                   float* mean, float* rstd, int64_t n, int64_t channels,
                   int64_t spatial, int64_t groups, float eps, int dtype,
                   void* stream);
size_t group_norm_bwd_workspace_size(int64_t n, int64_t channels, int64_t spatial,
                                     int64_t groups, int dtype);
int group_norm_bwd(const void* dy, const void* x, const void* gamma,
                   const float* mean, const float* rstd, void* dx,
                   float* dgamma, float* dbeta, int64_t n, int64_t channels,
                   int64_t spatial, int64_t groups, int dtype, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Introspection: the device kernels that the last call of any entry point
 * of this library on the calling thread launched, in launch order (at most
 * four are recorded).  names[i] receives a static, NUL-terminated string
 * (the kernel's symbol name as the CUDA runtime reports it) for
 * i < min(count, max_names); the return value is that count, or
 * -RMSN_ERR_NULL when names is NULL.  A call that launched nothing (rows ==
 * 0, a validation error) reports 0.  Needs no device work.
 */
int rms_norm_last_kernels(const char** names, int max_names);

/* Static, NUL-terminated description of a status code. */
const char* rms_norm_status_string(int status);

/* The cudaError_t of the last call that returned RMSN_ERR_CUDA on this
 * thread (0 if none). */
int rms_norm_last_cuda_error(void);

/* Number of kernels the last successful rms_norm_fwd / rms_norm_bwd call on
 * this thread enqueued (0 when nothing was launched). */
int rms_norm_last_launch_count(void);

/* The staged kernels bound every wait on a shared-memory barrier (about one
 * second); a wait that runs out abandons the rest of its CTA's rows, leaving
 * their outputs unwritten, and is counted on the device.  Writes to *count
 * how many such waits ran out on the current device since the library was
 * loaded (0 in correct operation).  Synchronises with the device. */
int rms_norm_wait_timeouts(unsigned int* count);

/* Self-test of those bounded waits (both arguments are host pointers):
 * launches one thread that waits on a shared-memory barrier nothing
 * completes, through the same bounded wait the staged kernels use.  The
 * wait runs out after its limit, counts in a device counter of its own (not
 * the one rms_norm_wait_timeouts reads) and the kernel returns, leaving the
 * context usable.  Writes that count to *timeouts (1 expected) and the
 * seconds the call took, measured on the host, to *seconds (about one).
 * Synchronises with the device; RMSN_ERR_NULL for a NULL argument,
 * RMSN_ERR_CUDA if the launch or a copy fails. */
int rms_norm_selftest_wait_limit(unsigned int* timeouts, double* seconds);

/*
 * Backward without caller-provided scratch.  The method's pages describe no
 * such call; it exists for callers that cannot allocate device memory at the
 * point where they run the backward -- for example a plugin whose enqueue
 * hook must not call cudaMalloc, or a service that works inside a fixed,
 * pre-reserved memory budget -- and so cannot supply the `workspace` that
 * rms_norm_bwd asks for.
 *
 * Same arguments, results and errors as rms_norm_bwd minus the workspace.
 * The per-block weight-gradient partials go to one fixed array of
 * RMSN_NOALLOC_SCRATCH_BYTES (16 MiB) that the library declares in device
 * memory; every GPU that loads the library holds it until the process exits.
 * Sizes whose rms_norm_bwd_workspace_size exceeds RMSN_NOALLOC_SCRATCH_BYTES
 * are rejected with RMSN_ERR_SHAPE before anything is enqueued.  This entry
 * point calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * The first call on each device looks up that device's address of the array
 * (with the device current); make that first call before any stream capture.
 * Every call on a device uses the same array and leaves its partials there;
 * no part of it needs clearing, because every partial the reduction reads is
 * written earlier in the same call.  Calls that may run at the same time on
 * the GPU (different streams without ordering) race on the array and give
 * wrong results: order them on one stream or with events.
 */
#define RMSN_NOALLOC_SCRATCH_BYTES (16u << 20)
int rms_norm_bwd_noalloc(const void* dy, const void* x, const void* gamma,
                         const float* rstd, void* dx, float* dw,
                         int64_t rows, int64_t hidden, int offset, int dtype,
                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RMS_NORM_GB300_H */
