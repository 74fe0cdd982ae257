// Host-side launchers of the forward and backward kernels, called by the
// C ABI in capi.cu after every argument has been validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rmsn {

// Inputs of one forward call, already validated (rows >= 1).
struct FwdArgs {
  const void* x;
  const void* gamma;
  void* y;
  float* rstd;
  int64_t rows;
  int hidden;
  float eps;
  int offset;      // 0: gain gamma, 1: gain 1 + gamma
  int twice;       // 1: round x_hat to the storage type before the gain
  bool vec_ok;     // 16-byte aligned rows: the vector kernels may run
  bool fp8;        // y is FP8 E4M3 of x_hat * gain * (*scale)
  const float* scale;  // device pointer (fp8 only)
};

// Inputs of one backward call, already validated (rows >= 1).
struct BwdArgs {
  const void* dy;
  const void* x;
  const void* gamma;
  const float* rstd;
  void* dx;
  float* dw;
  int64_t rows;
  int hidden;
  int offset;
  bool vec_ok;
  float* partial;          // fp32 workspace, >= max_partials * hidden floats
  int64_t max_partials;    // partial rows the workspace holds
  int64_t block_rows;      // rows per weight-gradient partial; 0: one block per
                           // CTA (or cluster) of the launch
  float* chunks;           // non-NULL: write the chunk sums [ceil(P / 32), hidden]
                           // here instead of reducing them into dw
};

// Rows per block, number of blocks (partial rows) and persistent units of
// a backward launch.  block_rows 0: one block per unit, the rows split
// evenly over min(rows, max_units) units (the kernels' brows 0).
struct BlockPlan {
  int brows;
  int64_t nblocks;
  int units;
};

inline BlockPlan plan_blocks(int64_t rows, int64_t block_rows, int64_t max_units) {
  if (max_units < 1) max_units = 1;
  BlockPlan p;
  if (block_rows <= 0) {
    p.brows = 0;
    p.units = (int)(rows < max_units ? rows : max_units);
    p.nblocks = p.units;
    return p;
  }
  p.brows = (int)block_rows;
  p.nblocks = (rows + block_rows - 1) / block_rows;
  p.units = (int)(p.nblocks < max_units ? p.nblocks : max_units);
  return p;
}

// Units a backward launch may use when up to `resident` fit on the GPU at
// once: with default blocks also limited by the partial rows the workspace
// holds (one per unit).
inline int64_t unit_cap(const BwdArgs& a, int64_t resident) {
  if (a.block_rows == 0 && resident > a.max_partials) return a.max_partials;
  return resident;
}

// dtype: 0 fp32, 1 bf16, 2 fp16.  Each returns the CUDA status of its
// launches and adds the number of kernels it enqueued to *launches.
cudaError_t launch_fwd(int dtype, const FwdArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_bwd(int dtype, const BwdArgs& a, cudaStream_t s, int* launches);

// TMA-staged persistent kernels (tma.cu).  Each returns false, having
// enqueued nothing, when the sizes or alignment do not suit it; otherwise
// true with the launch status in *err (and the partial count in *nparts).
bool try_launch_fwd_tma(int dtype, const FwdArgs& a, cudaStream_t s, cudaError_t* err);
bool try_launch_bwd_tma(int dtype, const BwdArgs& a, cudaStream_t s, cudaError_t* err,
                        int64_t* nparts);

// Cluster kernels for wide rows (cluster.cu), same contract.
bool try_launch_fwd_cluster(int dtype, const FwdArgs& a, cudaStream_t s, cudaError_t* err);
bool try_launch_bwd_cluster(int dtype, const BwdArgs& a, cudaStream_t s, cudaError_t* err,
                            int64_t* nparts);

// The kernels the current C-ABI call on this thread has launched, in order
// (the first four), for rms_norm_last_kernels().  capi.cu.
struct LaunchLog {
  const void* kern[4];
  int n;
};
LaunchLog& launch_log();
// Start of a C-ABI call on this thread: clears the launch count and log.
void begin_call();
// Record a failed CUDA call for rms_norm_last_cuda_error(); returns
// RMSN_ERR_CUDA.
int cuda_fail(cudaError_t e);
// Record how many kernels the current call enqueued, for
// rms_norm_last_launch_count().
void set_last_launches(int n);

// Launch `kern` with programmatic dependent launch allowed (see pdl_wait in
// common.cuh) and, when `cluster` > 1, thread-block clusters of `cluster`
// CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  LaunchLog& log = launch_log();
  if (e == cudaSuccess && log.n < 4) log.kern[log.n++] = reinterpret_cast<const void*>(kern);
  return e;
}

// out[j] = sum over the nparts rows of the fp32 matrix `partial`
// [nparts, ncols] in a fixed order -- chunks of 32 consecutive rows as a
// pairwise tree, the chunk sums added in chunk order; column j goes to
// out0[j] for j < split, to out1[j - split] otherwise (skipped when out1 is
// NULL).  bwd.cu.
cudaError_t launch_column_sums(const float* partial, int64_t nparts, int ncols, float* out0,
                               float* out1, int split, cudaStream_t s);
// The first half of that order alone: chunk c's tree sum to chunks[c][j].
cudaError_t launch_chunk_sums(const float* partial, int64_t nparts, int ncols, float* chunks,
                              cudaStream_t s);
// The second half alone: out[j] = chunks[0][j] + chunks[1][j] + ... in
// chunk order.
cudaError_t launch_chunk_totals(const float* chunks, int64_t nchunks, int ncols, float* out,
                                cudaStream_t s);
constexpr int kChunkParts = 32;  // partial rows per chunk of the fixed order

// Inputs of one LayerNorm call, already validated (rows >= 1).
struct LnFwdArgs {
  const void* x;
  const void* gamma;
  const void* beta;   // may be NULL (no bias)
  void* y;
  float* mean;
  float* rstd;
  int64_t rows;
  int hidden;
  float eps;
  bool vec_ok;
};

struct LnBwdArgs {
  const void* dy;
  const void* x;
  const void* gamma;
  const float* mean;
  const float* rstd;
  void* dx;
  float* dgamma;
  float* dbeta;       // may be NULL (not computed)
  int64_t rows;
  int hidden;
  bool vec_ok;
  float* partial;     // fp32 workspace, >= max_partials * 2 * hidden floats
  int64_t max_partials;
};

cudaError_t launch_ln_fwd(int dtype, const LnFwdArgs& a, cudaStream_t s, int* launches);
// TMA-staged LayerNorm kernels (tma.cu): false when the row does not fit the
// pipeline (nothing launched); true with *err set otherwise.  *nparts = the
// backward's partial rows.
bool try_launch_ln_fwd_tma(int dtype, const LnFwdArgs& a, cudaStream_t s, cudaError_t* err);
bool try_launch_ln_bwd_tma(int dtype, const LnBwdArgs& a, cudaStream_t s, cudaError_t* err,
                           int* nparts);
cudaError_t launch_ln_bwd(int dtype, const LnBwdArgs& a, cudaStream_t s, int* launches);

// Inputs of one softmax call (forward: x -> y; backward: dy, y -> dx),
// already validated (rows >= 1).
struct SoftmaxArgs {
  const void* x;
  const void* y;   // forward: the output (written); backward: the input
  const void* dy;
  void* dx;
  int64_t rows;
  int cols;
  bool vec_ok;
};

cudaError_t launch_softmax_fwd(int dtype, const SoftmaxArgs& a, cudaStream_t s);
cudaError_t launch_softmax_bwd(int dtype, const SoftmaxArgs& a, cudaStream_t s);

// Inputs of one GroupNorm call over x [n, channels, spatial] with `groups`
// groups of consecutive channels, already validated (n >= 1).
struct GnArgs {
  const void* x;
  const void* gamma;
  const void* beta;   // forward, may be NULL
  void* y;
  float* mean;        // [n, groups] fp32 (forward: written; backward: read)
  float* rstd;
  const void* dy;
  void* dx;
  float* dgamma;
  float* dbeta;       // may be NULL (not computed)
  float* partial;     // backward workspace, [n * 16, 2 * channels] fp32 at most
  int64_t n;
  int channels, spatial, groups;
  float eps;
  bool vec_ok;        // 16-byte aligned tensors and spatial * sizeof(T) % 16 == 0
};

cudaError_t launch_gn_fwd(int dtype, const GnArgs& a, cudaStream_t s);
// Bounded-wait timeouts counted by the GroupNorm kernels (group_norm.cu).
cudaError_t read_gn_wait_timeouts(unsigned int* out);
cudaError_t launch_gn_bwd(int dtype, const GnArgs& a, cudaStream_t s, int* launches);

// Device properties, cached per device.  sm_count honours the SM budget
// set with rms_norm_set_sm_budget (capi.cu).
int sm_count(int device);
int max_blocks_per_sm(const void* func, int block, size_t smem);

}  // namespace rmsn
