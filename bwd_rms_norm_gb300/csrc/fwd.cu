// RMSNorm forward kernels for sm_103a.
//
// Per row: fp32 sum of squares, rstd = 1/sqrt(sum/hidden + eps) stored in
// fp32, then y = round(x * rstd * gain) with a single rounding (round once)
// or y = round(round(x * rstd) * gain) (round twice) -- "Den dolda
// avrundningen i RMSNorm", sections "En välbekant operation" and "Två
// ställen att avrunda"; statistics in fp32 as in Liger-Kernel PR #92.  The
// FP8 variant (template flag F8) stores E4M3 of ((x * rstd) * gain) * scale,
// every step in fp32 and one conversion at the end (same page, section "Var
// implementationerna skiljer sig", the Transformer Engine paragraph).
//
// The path is bound by HBM bandwidth: each element is read once and written
// once, so the row stays in registers between the reduction and the store.
// Three kernels:
//   fwd_warp_rows  one warp per row (rows of at most 128 vectors),
//   fwd_cta_row    one CTA per row (up to 1024 threads x 8 vectors),
//   fwd_scalar     any alignment or width: scalar loads, the row is read a
//                  second time for the store (from L1/L2).
#include "common.cuh"
#include "launch.h"

namespace rmsn {
namespace {

// rstd of a warp's row whose fp32 sum of squares overflowed (kOverflowScale),
// out of line: the rare branch costs the ordinary path no registers.
template <typename T>
__device__ __noinline__ float rstd_overflow_warp(const T* __restrict__ xr, int lane, int hidden,
                                                 float eps) {
  return rstd_rescaled(warp_sum(scaled_sum_sq(xr, lane, 32, hidden)), hidden, eps);
}

// Output of one vector of x (already unpacked) for the chosen store.
template <typename T>
__device__ __forceinline__ uint4 scale_vec(const float (&xf)[Traits<T>::kVec],
                                           const uint4& gv, float rs, float off,
                                           int twice) {
  constexpr int E = Traits<T>::kVec;
  float gf[E], o[E];
  unpack<T>(gv, gf);
  if (twice) {
#pragma unroll
    for (int i = 0; i < E; ++i) o[i] = round_trip<T>(xf[i] * rs) * (gf[i] + off);
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) o[i] = (xf[i] * rs) * (gf[i] + off);
  }
  return pack<T>(o);
}

// Store one vector of outputs at element `elem` of y: the storage type T, or
// FP8 E4M3 of ((x * rstd) * gain) * scale, every step in fp32 and a single
// conversion at the end.
template <typename T, bool F8>
__device__ __forceinline__ void store_vec(void* y, int64_t elem,
                                          const float (&xf)[Traits<T>::kVec], const uint4& gv,
                                          float rs, float off, int twice, float sc) {
  constexpr int E = Traits<T>::kVec;
  if constexpr (F8) {
    float gf[E], o[E];
    unpack<T>(gv, gf);
#pragma unroll
    for (int i = 0; i < E; ++i) o[i] = ((xf[i] * rs) * (gf[i] + off)) * sc;
    st_e4m3<E>(static_cast<unsigned char*>(y) + elem, o);
  } else {
    st_vec_stream(static_cast<T*>(y) + elem, scale_vec<T>(xf, gv, rs, off, twice));
  }
}

template <typename T, int VPT, bool F8>
__global__ void __launch_bounds__(256, 5) fwd_warp_rows(
    const T* __restrict__ x, const T* __restrict__ gamma, void* __restrict__ y,
    float* __restrict__ rstd, int64_t rows, int hidden, float eps, float off,
    int twice, const float* __restrict__ scale) {
  constexpr int E = Traits<T>::kVec;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_trigger();
  if (row >= rows) return;  // whole warps leave together
  if (lane == 0) prefetch_l2(x + row * hidden, (uint32_t)(hidden * sizeof(T)));
  pdl_wait();
  const int nvec = hidden / E;
  const T* xr = x + row * hidden;
  const float sc = F8 ? __ldg(scale) : 1.f;

  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + 32 * k;
    xv[k] = v < nvec ? ld_stream(xr + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    float f[E];
    unpack<T>(xv[k], f);
#pragma unroll
    for (int i = 0; i < E; ++i) ss = fmaf(f[i], f[i], ss);
  }
  ss = warp_sum(ss);
  float rs = rstd_of(ss / (float)hidden, eps);
  if (isinf(ss))  // the fp32 sum of squares overflowed (see kOverflowScale)
    rs = rstd_overflow_warp(xr, lane, hidden, eps);
  if (lane == 0) rstd[row] = rs;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + 32 * k;
    if (v < nvec) {
      float f[E];
      unpack<T>(xv[k], f);
      const uint4 gv = ld_shared_ro(gamma + (int64_t)v * E);
      store_vec<T, F8>(y, row * hidden + (int64_t)v * E, f, gv, rs, off, twice, sc);
    }
  }
}

template <typename T, int VPT, bool F8>
__global__ void __launch_bounds__(VPT >= 8 ? 512 : VPT >= 4 ? 1024 : 128, VPT <= 2 ? 16 : 1) fwd_cta_row(
    const T* __restrict__ x, const T* __restrict__ gamma, void* __restrict__ y,
    float* __restrict__ rstd, int hidden, float eps, float off, int twice,
    const float* __restrict__ scale) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  const int64_t row = blockIdx.x;
  const int nvec = hidden / E;
  const T* xr = x + row * hidden;
  pdl_trigger();
  if (threadIdx.x == 0) prefetch_l2(xr, (uint32_t)(hidden * sizeof(T)));
  pdl_wait();
  const float sc = F8 ? __ldg(scale) : 1.f;

  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    xv[k] = v < nvec ? ld_stream(xr + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    float f[E];
    unpack<T>(xv[k], f);
#pragma unroll
    for (int i = 0; i < E; ++i) ss = fmaf(f[i], f[i], ss);
  }
  ss = block_sum(ss, red, 0);
  float rs = rstd_of(ss / (float)hidden, eps);
  if (isinf(ss))  // the fp32 sum of squares overflowed (see kOverflowScale)
    rs = rstd_rescaled(block_sum(scaled_sum_sq(xr, threadIdx.x, blockDim.x, hidden), red, 1),
                       hidden, eps);
  if (threadIdx.x == 0) rstd[row] = rs;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec) {
      float f[E];
      unpack<T>(xv[k], f);
      const uint4 gv = ld_shared_ro(gamma + (int64_t)v * E);
      store_vec<T, F8>(y, row * hidden + (int64_t)v * E, f, gv, rs, off, twice, sc);
    }
  }
}

template <typename T, bool F8>
__global__ void __launch_bounds__(256) fwd_scalar(
    const T* __restrict__ x, const T* __restrict__ gamma, void* __restrict__ y,
    float* __restrict__ rstd, int hidden, float eps, float off, int twice,
    const float* __restrict__ scale) {
  __shared__ float red[64];
  const int64_t row = blockIdx.x;
  const T* xr = x + row * hidden;
  pdl_trigger();
  pdl_wait();
  const float sc = F8 ? __ldg(scale) : 1.f;
  float ss = 0.f;
  for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
    const float f = Traits<T>::to_f(xr[j]);
    ss = fmaf(f, f, ss);
  }
  ss = block_sum(ss, red, 0);
  float rs = rstd_of(ss / (float)hidden, eps);
  if (isinf(ss))  // the fp32 sum of squares overflowed (see kOverflowScale)
    rs = rstd_rescaled(block_sum(scaled_sum_sq(xr, threadIdx.x, blockDim.x, hidden), red, 1),
                       hidden, eps);
  if (threadIdx.x == 0) rstd[row] = rs;
  for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
    const float xh = Traits<T>::to_f(xr[j]) * rs;
    const float g = Traits<T>::to_f(gamma[j]) + off;
    if constexpr (F8) {
      static_cast<unsigned char*>(y)[row * hidden + j] = e4m3((xh * g) * sc);
    } else {
      const float o = twice ? round_trip<T>(xh) * g : xh * g;
      static_cast<T*>(y)[row * hidden + j] = Traits<T>::from_f(o);
    }
  }
}

template <typename T> int dtype_code();
template <> int dtype_code<float>() { return 0; }
template <> int dtype_code<__nv_bfloat16>() { return 1; }
template <> int dtype_code<__half>() { return 2; }

int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Rows of up to this many 16-byte vectors run one warp per row.
constexpr int kWarpRowMaxVec = 128;

template <typename T, bool F8>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s, int* launches) {
  constexpr int E = Traits<T>::kVec;
  const T* x = static_cast<const T*>(a.x);
  const T* g = static_cast<const T*>(a.gamma);
  void* y = a.y;
  const float off = a.offset ? 1.f : 0.f;
  const int nvec = a.hidden / E;
  const float* sc = a.scale;
  cudaError_t e = cudaSuccess;

  if (a.vec_ok && nvec <= kWarpRowMaxVec) {
    // one warp per row, 8 rows per CTA
    const int vpt = pow2_at_least((nvec + 31) / 32);
    const dim3 grid((unsigned)((a.rows + 7) / 8));
    switch (vpt) {
      case 1: e = launch_kernel(fwd_warp_rows<T, 1, F8>, grid, dim3(256), 0, s, 1, x, g, y, a.rstd, a.rows, a.hidden, a.eps, off, a.twice, sc); break;
      case 2: e = launch_kernel(fwd_warp_rows<T, 2, F8>, grid, dim3(256), 0, s, 1, x, g, y, a.rstd, a.rows, a.hidden, a.eps, off, a.twice, sc); break;
      case 4: e = launch_kernel(fwd_warp_rows<T, 4, F8>, grid, dim3(256), 0, s, 1, x, g, y, a.rstd, a.rows, a.hidden, a.eps, off, a.twice, sc); break;
      case 8: e = launch_kernel(fwd_warp_rows<T, 8, F8>, grid, dim3(256), 0, s, 1, x, g, y, a.rstd, a.rows, a.hidden, a.eps, off, a.twice, sc); break;
      default: e = launch_kernel(fwd_warp_rows<T, 16, F8>, grid, dim3(256), 0, s, 1, x, g, y, a.rstd, a.rows, a.hidden, a.eps, off, a.twice, sc); break;
    }
    if (e == cudaSuccess) *launches += 1;
    return e;
  }
  if (a.vec_ok) {
    // one CTA per row of about 128 threads with up to 4 vectors each (a
    // 4-warp reduction per row, 4 loads in flight per thread); wider rows
    // use more threads, and rows too wide for 1024 threads x 4 vectors use
    // 8 or 16 vectors per thread at 512 threads
    int vpt = pow2_at_least((nvec + 127) / 128);
    if (vpt > 4) vpt = 4;
    if ((nvec + vpt - 1) / vpt > 1024) vpt = pow2_at_least((nvec + 511) / 512);
    if (vpt > 16) vpt = 16;
    const int tpr = ((nvec + vpt - 1) / vpt + 31) / 32 * 32;
    if (tpr <= (vpt >= 8 ? 512 : 1024)) {
      const dim3 grid((unsigned)a.rows);
      switch (vpt) {
        case 1: e = launch_kernel(fwd_cta_row<T, 1, F8>, grid, dim3(tpr), 0, s, 1, x, g, y, a.rstd, a.hidden, a.eps, off, a.twice, sc); break;
        case 2: e = launch_kernel(fwd_cta_row<T, 2, F8>, grid, dim3(tpr), 0, s, 1, x, g, y, a.rstd, a.hidden, a.eps, off, a.twice, sc); break;
        case 4: e = launch_kernel(fwd_cta_row<T, 4, F8>, grid, dim3(tpr), 0, s, 1, x, g, y, a.rstd, a.hidden, a.eps, off, a.twice, sc); break;
        case 8: e = launch_kernel(fwd_cta_row<T, 8, F8>, grid, dim3(tpr), 0, s, 1, x, g, y, a.rstd, a.hidden, a.eps, off, a.twice, sc); break;
        default: e = launch_kernel(fwd_cta_row<T, 16, F8>, grid, dim3(tpr), 0, s, 1, x, g, y, a.rstd, a.hidden, a.eps, off, a.twice, sc); break;
      }
      if (e == cudaSuccess) *launches += 1;
      return e;
    }
  }
  // the cluster kernels store the storage type only; an FP8 row this wide
  // takes the scalar kernel
  if (!F8 && try_launch_fwd_cluster(dtype_code<T>(), a, s, &e)) {
    if (e == cudaSuccess) *launches += 1;
    return e;
  }
  e = launch_kernel(fwd_scalar<T, F8>, dim3((unsigned)a.rows), dim3(256), 0, s, 1, x, g, y,
                    a.rstd, a.hidden, a.eps, off, a.twice, sc);
  if (e == cudaSuccess) *launches += 1;
  return e;
}

}  // namespace

// Kernel choice by row width (measured on GB300 with the workloads of the
// tests, as forward+backward steps): rows over 4 KB run the staged TMA
// pipeline -- one persistent CTA per SM (fwd_tma), or a cluster of 2 or 4
// CTAs per row range for rows its ring and registers cannot hold
// (fwd_tma_split) -- which hands the SMs to the next kernel with less
// turnover than one CTA per row; rows up to 4 KB run the register kernels.
// Rows too wide for all of these (fp32 65536) are held in the registers of
// a thread-block cluster (fwd_cluster).
cudaError_t launch_fwd(int dtype, const FwdArgs& a, cudaStream_t s, int* launches) {
  cudaError_t e = cudaSuccess;
  const int row_bytes = a.hidden * (dtype == 0 ? 4 : 2);
  if (row_bytes > 4 * 1024 && try_launch_fwd_tma(dtype, a, s, &e)) {
    if (e == cudaSuccess) *launches += 1;
    return e;
  }
  if (a.fp8) {
    switch (dtype) {
      case 0: return launch_fwd_t<float, true>(a, s, launches);
      case 1: return launch_fwd_t<__nv_bfloat16, true>(a, s, launches);
      default: return launch_fwd_t<__half, true>(a, s, launches);
    }
  }
  switch (dtype) {
    case 0: return launch_fwd_t<float, false>(a, s, launches);
    case 1: return launch_fwd_t<__nv_bfloat16, false>(a, s, launches);
    default: return launch_fwd_t<__half, false>(a, s, launches);
  }
}

}  // namespace rmsn
