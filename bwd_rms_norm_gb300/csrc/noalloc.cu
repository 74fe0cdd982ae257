// rms_norm_bwd_noalloc: the backward for callers that cannot allocate device
// memory where they run it (an enqueue hook that must not call cudaMalloc, a
// fixed pre-reserved memory budget).  Instead of a caller workspace, the
// weight-gradient partials go to one file-scope device array of fixed size.
//
// The array's name, used in host code, is a host-side stand-in and not a
// device address; the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the
// kernels.  The kernels and their launch configuration are those of
// rms_norm_bwd, so for the sizes accepted here both calls compute the same
// result.
#include <atomic>
#include <mutex>

#include "launch.h"
#include "rms_norm.h"

namespace rmsn {
namespace {

static __device__ __align__(256) float g_noalloc_scratch[RMSN_NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of g_noalloc_scratch on `device` (the current device).
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[device].load(std::memory_order_acquire);
  if (p != nullptr) {
    *out = p;
    return cudaSuccess;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  p = g_scratch_addr[device].load(std::memory_order_relaxed);
  if (p == nullptr) {
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_addr[device].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace rmsn

extern "C" int rms_norm_bwd_noalloc(const void* dy, const void* x, const void* gamma,
                                    const float* rstd, void* dx, float* dw, int64_t rows,
                                    int64_t hidden, int offset, int dtype, void* stream) {
  using namespace rmsn;
  if (dtype != RMSN_F32 && dtype != RMSN_BF16 && dtype != RMSN_F16) return RMSN_ERR_DTYPE;
  rmsn::begin_call();
  if (offset != 0 && offset != 1) return RMSN_ERR_ARG;
  if (rows < 0 || rows > RMSN_MAX_ROWS || hidden < 1 || hidden > RMSN_MAX_HIDDEN)
    return RMSN_ERR_SHAPE;
  if (!dw) return RMSN_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0) {
    const cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)hidden * sizeof(float), st);
    return e == cudaSuccess ? RMSN_OK : cuda_fail(e);
  }
  if (!dy || !x || !gamma || !rstd || !dx) return RMSN_ERR_NULL;
  const size_t need = rms_norm_bwd_workspace_size(rows, hidden, dtype);
  if (need > (size_t)RMSN_NOALLOC_SCRATCH_BYTES) return RMSN_ERR_SHAPE;

  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e);
  void* scratch = nullptr;
  e = scratch_address(device, &scratch);
  if (e != cudaSuccess) return cuda_fail(e);

  const int s = dtype == RMSN_F32 ? 4 : 2;
  auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
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
  a.partial = static_cast<float*>(scratch);
  // the partial count rms_norm_bwd would use with a workspace of exactly
  // rms_norm_bwd_workspace_size bytes
  a.max_partials = (int64_t)(need / ((size_t)hidden * sizeof(float)));
  a.block_rows = 0;
  a.chunks = nullptr;
  int launches = 0;
  e = launch_bwd(dtype, a, st, &launches);
  if (e != cudaSuccess) return cuda_fail(e);
  set_last_launches(launches);
  return RMSN_OK;
}
