// C ABI of the fused RMSNorm library: argument validation and dispatch.
// Every check runs on the host before anything is enqueued.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "launch.h"
#include "rms_norm.h"

namespace rmsn {

namespace {
thread_local int t_last_cuda_error = 0;
thread_local int t_last_launches = 0;
thread_local LaunchLog t_launch_log = {{nullptr, nullptr, nullptr, nullptr}, 0};

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_sm_budget{0};  // 0: every SM

struct OccEntry {
  const void* func;
  int block;
  size_t smem;
  int device;
  int value;
};
std::mutex g_occ_mutex;
OccEntry g_occ[256];
int g_occ_n = 0;

int elem_bytes(int dtype) { return dtype == RMSN_F32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return RMSN_ERR_CUDA;
}

void set_last_launches(int n) { t_last_launches = n; }

LaunchLog& launch_log() { return t_launch_log; }

// Start of a C-ABI call: nothing launched yet.
void begin_call() {
  t_last_launches = 0;
  t_launch_log.n = 0;
}

int sm_count(int device) {
  const int budget = g_sm_budget.load(std::memory_order_relaxed);
  int n = 0;
  if (device >= 0 && device < kMaxDevices) n = g_sm_count[device].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        n <= 0)
      n = 1;
    if (device >= 0 && device < kMaxDevices)
      g_sm_count[device].store(n, std::memory_order_relaxed);
  }
  return budget > 0 && budget < n ? budget : n;
}

int max_blocks_per_sm(const void* func, int block, size_t smem) {
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    for (int i = 0; i < g_occ_n; ++i)
      if (g_occ[i].func == func && g_occ[i].block == block && g_occ[i].smem == smem &&
          g_occ[i].device == dev)
        return g_occ[i].value;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, block, smem) != cudaSuccess) n = 1;
  if (n < 1) n = 1;
  std::lock_guard<std::mutex> lock(g_occ_mutex);
  if (g_occ_n < 256) g_occ[g_occ_n++] = OccEntry{func, block, smem, dev, n};
  return n;
}

}  // namespace rmsn

using namespace rmsn;

extern "C" {

int rms_norm_fwd(const void* x, const void* gamma, void* y, float* rstd, int64_t rows,
                 int64_t hidden, float eps, int offset, int dtype, int cast_mode,
                 void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if ((offset != 0 && offset != 1) || (cast_mode != RMSN_ROUND_ONCE && cast_mode != RMSN_ROUND_TWICE))
    return RMSN_ERR_ARG;
  if (rows < 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  if (!(eps >= 0.f) || isinf(eps)) return RMSN_ERR_EPS;
  begin_call();
  if (rows == 0) return RMSN_OK;
  if (!x || !gamma || !y || !rstd) return RMSN_ERR_NULL;

  const int s = elem_bytes(dtype);
  FwdArgs a;
  a.x = x;
  a.gamma = gamma;
  a.y = y;
  a.rstd = rstd;
  a.rows = rows;
  a.hidden = (int)hidden;
  a.eps = eps;
  a.offset = offset;
  a.twice = cast_mode == RMSN_ROUND_TWICE ? 1 : 0;
  a.vec_ok = ((hidden * s) % 16 == 0) && aligned16(x) && aligned16(gamma) && aligned16(y);
  a.fp8 = false;
  a.scale = nullptr;
  int launches = 0;
  cudaError_t e = launch_fwd(dtype, a, static_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = launches;
  return RMSN_OK;
}

int rms_norm_fwd_fp8(const void* x, const void* gamma, const float* scale, void* y, float* rstd,
                     int64_t rows, int64_t hidden, float eps, int offset, int dtype,
                     void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (offset != 0 && offset != 1) return RMSN_ERR_ARG;
  if (rows < 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  if (!(eps >= 0.f) || isinf(eps)) return RMSN_ERR_EPS;
  begin_call();
  if (rows == 0) return RMSN_OK;
  if (!x || !gamma || !scale || !y || !rstd) return RMSN_ERR_NULL;
  const int s = elem_bytes(dtype);
  FwdArgs a;
  a.x = x;
  a.gamma = gamma;
  a.y = y;
  a.rstd = rstd;
  a.rows = rows;
  a.hidden = (int)hidden;
  a.eps = eps;
  a.offset = offset;
  a.twice = 0;
  // a 16-byte input vector becomes 16/s output bytes: rows of y start on
  // that boundary when y does
  a.vec_ok = ((hidden * s) % 16 == 0) && aligned16(x) && aligned16(gamma) && aligned16(y);
  a.fp8 = true;
  a.scale = scale;
  int launches = 0;
  cudaError_t e = launch_fwd(dtype, a, static_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = launches;
  return RMSN_OK;
}

size_t rms_norm_bwd_workspace_size(int64_t rows, int64_t hidden, int dtype) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return 0;
  if (rows <= 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN) return 0;
  const int64_t parts = rows < RMSN_MAX_PARTIALS ? rows : RMSN_MAX_PARTIALS;
  return (size_t)parts * (size_t)hidden * sizeof(float);
}

int rms_norm_bwd(const void* dy, const void* x, const void* gamma, const float* rstd, void* dx,
                 float* dw, int64_t rows, int64_t hidden, int offset, int dtype, void* workspace,
                 size_t workspace_bytes, void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (offset != 0 && offset != 1) return RMSN_ERR_ARG;
  if (rows < 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  begin_call();
  if (!dw) return RMSN_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0) {
    cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)hidden * sizeof(float), st);
    return e == cudaSuccess ? RMSN_OK : cuda_fail(e);
  }
  if (!dy || !x || !gamma || !rstd || !dx || !workspace) return RMSN_ERR_NULL;
  if (!aligned16(workspace)) return RMSN_ERR_ALIGN;
  const size_t need = rms_norm_bwd_workspace_size(rows, hidden, dtype);
  if (workspace_bytes < need) return RMSN_ERR_WORKSPACE;

  const int s = elem_bytes(dtype);
  BwdArgs a;
  a.dy = dy;
  a.x = x;
  a.gamma = gamma;
  a.rstd = rstd;
  a.dx = dx;
  a.dw = dw;
  a.rows = rows;
  a.hidden = (int)hidden;
  a.offset = offset;
  a.vec_ok = ((hidden * s) % 16 == 0) && aligned16(dy) && aligned16(x) && aligned16(gamma) &&
             aligned16(dx);
  a.partial = static_cast<float*>(workspace);
  a.max_partials = (int64_t)(workspace_bytes / ((size_t)hidden * sizeof(float)));
  if (a.max_partials > RMSN_MAX_PARTIALS) a.max_partials = RMSN_MAX_PARTIALS;
  a.block_rows = 0;
  a.chunks = nullptr;
  int launches = 0;
  cudaError_t e = launch_bwd(dtype, a, st, &launches);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = launches;
  return RMSN_OK;
}

static int64_t blocks_of(int64_t rows, int64_t block_rows) {
  return (rows + block_rows - 1) / block_rows;
}

size_t rms_norm_bwd_blocked_workspace_size(int64_t rows, int64_t hidden, int64_t block_rows) {
  if (rows <= 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN ||
      block_rows < 1)
    return 0;
  return (size_t)blocks_of(rows, block_rows) * (size_t)hidden * sizeof(float);
}

int64_t rms_norm_dw_chunk_count(int64_t rows, int64_t block_rows) {
  if (rows < 0 || rows > RMSN_MAX_ROWS || block_rows < 1) return -RMSN_ERR_SHAPE;
  return (blocks_of(rows, block_rows) + RMSN_DW_CHUNK_BLOCKS - 1) / RMSN_DW_CHUNK_BLOCKS;
}

int rms_norm_bwd_blocked(const void* dy, const void* x, const void* gamma, const float* rstd,
                         void* dx, float* chunk_sums, int64_t rows, int64_t hidden,
                         int64_t block_rows, int offset, int dtype, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (offset != 0 && offset != 1) return RMSN_ERR_ARG;
  if (rows < 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  if (block_rows < 1 || block_rows > RMSN_MAX_ROWS) return RMSN_ERR_ARG;
  begin_call();
  if (rows == 0) return RMSN_OK;
  if (!dy || !x || !gamma || !rstd || !dx || !chunk_sums || !workspace) return RMSN_ERR_NULL;
  if (!aligned16(workspace)) return RMSN_ERR_ALIGN;
  if (workspace_bytes < rms_norm_bwd_blocked_workspace_size(rows, hidden, block_rows))
    return RMSN_ERR_WORKSPACE;
  const int s = elem_bytes(dtype);
  BwdArgs a;
  a.dy = dy;
  a.x = x;
  a.gamma = gamma;
  a.rstd = rstd;
  a.dx = dx;
  a.dw = nullptr;
  a.rows = rows;
  a.hidden = (int)hidden;
  a.offset = offset;
  a.vec_ok = ((hidden * s) % 16 == 0) && aligned16(dy) && aligned16(x) && aligned16(gamma) &&
             aligned16(dx);
  a.partial = static_cast<float*>(workspace);
  a.max_partials = blocks_of(rows, block_rows);
  a.block_rows = block_rows;
  a.chunks = chunk_sums;
  int launches = 0;
  cudaError_t e = launch_bwd(dtype, a, static_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = launches;
  return RMSN_OK;
}

int rms_norm_dw_sum(const float* chunk_sums, int64_t nchunks, int64_t hidden, float* dw,
                    void* stream) {
  if (nchunks < 0 || hidden < 1 || hidden > RMSN_MAX_HIDDEN) return RMSN_ERR_SHAPE;
  begin_call();
  if (!dw) return RMSN_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (nchunks == 0) {
    const cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)hidden * sizeof(float), st);
    return e == cudaSuccess ? RMSN_OK : cuda_fail(e);
  }
  if (!chunk_sums) return RMSN_ERR_NULL;
  const cudaError_t e = launch_chunk_totals(chunk_sums, nchunks, (int)hidden, dw, st);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 1;
  return RMSN_OK;
}

int rms_norm_rank_rows(int64_t rows, int64_t block_rows, int world, int rank, int64_t* row_lo,
                       int64_t* row_hi) {
  if (!row_lo || !row_hi) return RMSN_ERR_NULL;
  if (rows < 0 || rows > RMSN_MAX_ROWS) return RMSN_ERR_SHAPE;
  if (block_rows < 1 || world < 1 || rank < 0 || rank >= world) return RMSN_ERR_ARG;
  const int64_t chunk_rows = block_rows * RMSN_DW_CHUNK_BLOCKS;
  const int64_t chunks = (rows + chunk_rows - 1) / chunk_rows;
  const int64_t c0 = chunks * rank / world, c1 = chunks * (rank + 1) / world;
  const int64_t lo = c0 * chunk_rows, hi = c1 * chunk_rows;
  *row_lo = lo < rows ? lo : rows;
  *row_hi = hi < rows ? hi : rows;
  return RMSN_OK;
}

int rms_norm_set_sm_budget(int sms) {
  if (sms < 0) return RMSN_ERR_ARG;
  g_sm_budget.store(sms, std::memory_order_relaxed);
  return RMSN_OK;
}

int rms_norm_sm_budget(void) { return g_sm_budget.load(std::memory_order_relaxed); }

int layer_norm_fwd(const void* x, const void* gamma, const void* beta, void* y, float* mean,
                   float* rstd, int64_t rows, int64_t hidden, float eps, int dtype,
                   void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (rows < 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  if (!(eps >= 0.f) || isinf(eps)) return RMSN_ERR_EPS;
  begin_call();
  if (rows == 0) return RMSN_OK;
  if (!x || !gamma || !y || !mean || !rstd) return RMSN_ERR_NULL;
  const int s = elem_bytes(dtype);
  LnFwdArgs a;
  a.x = x;
  a.gamma = gamma;
  a.beta = beta;
  a.y = y;
  a.mean = mean;
  a.rstd = rstd;
  a.rows = rows;
  a.hidden = (int)hidden;
  a.eps = eps;
  a.vec_ok = ((hidden * s) % 16 == 0) && aligned16(x) && aligned16(gamma) && aligned16(y) &&
             (beta == nullptr || aligned16(beta));
  int launches = 0;
  cudaError_t e = launch_ln_fwd(dtype, a, static_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = launches;
  return RMSN_OK;
}

size_t layer_norm_bwd_workspace_size(int64_t rows, int64_t hidden, int dtype) {
  return 2 * rms_norm_bwd_workspace_size(rows, hidden, dtype);
}

int layer_norm_bwd(const void* dy, const void* x, const void* gamma, const float* mean,
                   const float* rstd, void* dx, float* dgamma, float* dbeta, int64_t rows,
                   int64_t hidden, int dtype, void* workspace, size_t workspace_bytes,
                   void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (rows < 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  begin_call();
  if (!dgamma) return RMSN_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0) {
    cudaError_t e = cudaMemsetAsync(dgamma, 0, (size_t)hidden * sizeof(float), st);
    if (e == cudaSuccess && dbeta) e = cudaMemsetAsync(dbeta, 0, (size_t)hidden * sizeof(float), st);
    return e == cudaSuccess ? RMSN_OK : cuda_fail(e);
  }
  if (!dy || !x || !gamma || !mean || !rstd || !dx || !workspace) return RMSN_ERR_NULL;
  if (!aligned16(workspace)) return RMSN_ERR_ALIGN;
  if (workspace_bytes < layer_norm_bwd_workspace_size(rows, hidden, dtype))
    return RMSN_ERR_WORKSPACE;
  const int s = elem_bytes(dtype);
  LnBwdArgs a;
  a.dy = dy;
  a.x = x;
  a.gamma = gamma;
  a.mean = mean;
  a.rstd = rstd;
  a.dx = dx;
  a.dgamma = dgamma;
  a.dbeta = dbeta;
  a.rows = rows;
  a.hidden = (int)hidden;
  a.vec_ok = ((hidden * s) % 16 == 0) && aligned16(dy) && aligned16(x) && aligned16(gamma) &&
             aligned16(dx);
  a.partial = static_cast<float*>(workspace);
  a.max_partials = (int64_t)(workspace_bytes / ((size_t)hidden * 2 * sizeof(float)));
  if (a.max_partials > RMSN_MAX_PARTIALS) a.max_partials = RMSN_MAX_PARTIALS;
  int launches = 0;
  cudaError_t e = launch_ln_bwd(dtype, a, st, &launches);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = launches;
  return RMSN_OK;
}

int softmax_fwd(const void* x, void* y, int64_t rows, int64_t cols, int dtype, void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (rows < 0 || rows > RMSN_MAX_ROWS || cols < 1 || cols > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  begin_call();
  if (rows == 0) return RMSN_OK;
  if (!x || !y) return RMSN_ERR_NULL;
  SoftmaxArgs a{};
  a.x = x;
  a.y = y;
  a.rows = rows;
  a.cols = (int)cols;
  a.vec_ok = ((cols * elem_bytes(dtype)) % 16 == 0) && aligned16(x) && aligned16(y);
  cudaError_t e = launch_softmax_fwd(dtype, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 1;
  return RMSN_OK;
}

int softmax_bwd(const void* dy, const void* y, void* dx, int64_t rows, int64_t cols, int dtype,
                void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (rows < 0 || rows > RMSN_MAX_ROWS || cols < 1 || cols > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  begin_call();
  if (rows == 0) return RMSN_OK;
  if (!dy || !y || !dx) return RMSN_ERR_NULL;
  SoftmaxArgs a{};
  a.dy = dy;
  a.y = y;
  a.dx = dx;
  a.rows = rows;
  a.cols = (int)cols;
  a.vec_ok = ((cols * elem_bytes(dtype)) % 16 == 0) && aligned16(dy) && aligned16(y) &&
             aligned16(dx);
  cudaError_t e = launch_softmax_bwd(dtype, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 1;
  return RMSN_OK;
}

namespace {
// Shape check shared by the GroupNorm entry points.
bool gn_shape_ok(int64_t n, int64_t channels, int64_t spatial, int64_t groups) {
  if (n < 0 || channels < 1 || spatial < 1 || groups < 1) return false;
  if (channels > (1 << 24) || spatial > (1 << 30) || channels % groups != 0) return false;
  if ((channels / groups) * spatial > (1 << 30)) return false;
  if (n * groups > RMSN_MAX_ROWS) return false;
  return n <= (INT64_MAX / channels) / spatial;
}
}  // namespace

int group_norm_fwd(const void* x, const void* gamma, const void* beta, void* y, float* mean,
                   float* rstd, int64_t n, int64_t channels, int64_t spatial, int64_t groups,
                   float eps, int dtype, void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (!gn_shape_ok(n, channels, spatial, groups)) return RMSN_ERR_SHAPE;
  if (!(eps >= 0.f) || isinf(eps)) return RMSN_ERR_EPS;
  begin_call();
  if (n == 0) return RMSN_OK;
  if (!x || !gamma || !y || !mean || !rstd) return RMSN_ERR_NULL;
  GnArgs a{};
  a.x = x;
  a.gamma = gamma;
  a.beta = beta;
  a.y = y;
  a.mean = mean;
  a.rstd = rstd;
  a.n = n;
  a.channels = (int)channels;
  a.spatial = (int)spatial;
  a.groups = (int)groups;
  a.eps = eps;
  a.vec_ok = ((spatial * elem_bytes(dtype)) % 16 == 0) && aligned16(x) && aligned16(y);
  cudaError_t e = launch_gn_fwd(dtype, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 1;
  return RMSN_OK;
}

size_t group_norm_bwd_workspace_size(int64_t n, int64_t channels, int64_t spatial,
                                     int64_t groups, int dtype) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return 0;
  if (!gn_shape_ok(n, channels, spatial, groups) || n == 0) return 0;
  // partial rows: up to 16 (the largest cluster) per sample, dW and dB
  return (size_t)n * 16u * 2u * (size_t)channels * sizeof(float);
}

int group_norm_bwd(const void* dy, const void* x, const void* gamma, const float* mean,
                   const float* rstd, void* dx, float* dgamma, float* dbeta, int64_t n,
                   int64_t channels, int64_t spatial, int64_t groups, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  if (!gn_shape_ok(n, channels, spatial, groups)) return RMSN_ERR_SHAPE;
  begin_call();
  if (!dgamma) return RMSN_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n == 0) {
    cudaError_t e = cudaMemsetAsync(dgamma, 0, (size_t)channels * sizeof(float), st);
    if (e == cudaSuccess && dbeta) e = cudaMemsetAsync(dbeta, 0, (size_t)channels * sizeof(float), st);
    return e == cudaSuccess ? RMSN_OK : cuda_fail(e);
  }
  if (!dy || !x || !gamma || !mean || !rstd || !dx || !workspace) return RMSN_ERR_NULL;
  if (!aligned16(workspace)) return RMSN_ERR_ALIGN;
  if (workspace_bytes < group_norm_bwd_workspace_size(n, channels, spatial, groups, dtype))
    return RMSN_ERR_WORKSPACE;
  GnArgs a{};
  a.dy = dy;
  a.x = x;
  a.gamma = gamma;
  a.mean = const_cast<float*>(mean);
  a.rstd = const_cast<float*>(rstd);
  a.dx = dx;
  a.dgamma = dgamma;
  a.dbeta = dbeta;
  a.partial = static_cast<float*>(workspace);
  a.n = n;
  a.channels = (int)channels;
  a.spatial = (int)spatial;
  a.groups = (int)groups;
  a.vec_ok = ((spatial * elem_bytes(dtype)) % 16 == 0) && aligned16(dy) && aligned16(x) &&
             aligned16(dx);
  int launches = 0;
  cudaError_t e = launch_gn_bwd(dtype, a, st, &launches);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = launches;
  return RMSN_OK;
}

const char* rms_norm_status_string(int status) {
  switch (status) {
    case RMSN_OK: return "ok";
    case RMSN_ERR_NULL: return "a required pointer is NULL";
    case RMSN_ERR_SHAPE: return "rows or hidden out of range";
    case RMSN_ERR_EPS: return "eps must be finite and >= 0";
    case RMSN_ERR_DTYPE: return "unknown dtype";
    case RMSN_ERR_ALIGN: return "workspace must be 16-byte aligned";
    case RMSN_ERR_WORKSPACE: return "workspace smaller than rms_norm_bwd_workspace_size";
    case RMSN_ERR_CUDA: return "a CUDA call failed";
    case RMSN_ERR_ARG: return "offset must be 0 or 1 and cast_mode a rmsn_cast_mode";
    default: return "unknown status";
  }
}

int rms_norm_last_cuda_error(void) { return t_last_cuda_error; }

int rms_norm_last_launch_count(void) { return t_last_launches; }

int rms_norm_last_kernels(const char** names, int max_names) {
  if (!names || max_names < 0) return -RMSN_ERR_NULL;
  const int n = t_launch_log.n < max_names ? t_launch_log.n : max_names;
  for (int i = 0; i < n; ++i) {
    if (cudaFuncGetName(&names[i], t_launch_log.kern[i]) != cudaSuccess) {
      cudaGetLastError();
      names[i] = "?";
    }
  }
  return n;
}

}  // extern "C"
