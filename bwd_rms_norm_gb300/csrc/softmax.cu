// Softmax over the last dimension, forward and backward, for sm_103a
// (candle PR #4059, "Add backward passes to the fused rms_norm, layer_norm
// and softmax_last_dim ops", description).
//
// Forward, per row: m = max_j x_j; e_j = exp(x_j - m) in fp32 (expf); s =
// sum_j e_j in fp32; y_j = round(e_j * (1 / s)) -- the arithmetic in fp32
// for every storage type and a single rounding at the store.
// Backward, per row, from the stored y: d = sum_j dy_j * y_j in fp32;
// dx_j = round(y_j * (dy_j - d)).
//
// Both are bound by HBM bandwidth (2 and 3 streams of the storage type,
// no parameters).  Kernels: one warp per row for rows of at most 128
// 16-byte vectors, one CTA per row with the row in registers, and scalar
// kernels for rows that are not 16-byte aligned or too wide for registers.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace rmsn {
namespace {

// Maximum of packed pairs of a 16-bit type (exact: no rounding involved;
// a NaN loses to a number, as with fmaxf).
__device__ __forceinline__ uint32_t max_pair(uint32_t a, uint32_t b, __nv_bfloat16) {
  __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a),
                             *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t max_pair(uint32_t a, uint32_t b, __half) {
  __half2 r = __hmax2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// The thread's max over the in-range elements of its VPT packed vectors.
// 16-bit types compare packed pairs and widen only the final pair.
template <typename T, int VPT>
__device__ __forceinline__ float local_max(const uint4 (&xv)[VPT], int first, int stride,
                                           int nvec) {
  constexpr int E = Traits<T>::kVec;
  if constexpr (sizeof(T) == 2) {
    uint32_t m2 = 0;
    bool any = false;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (first + k * stride < nvec) {
        const uint32_t w = max_pair(max_pair(xv[k].x, xv[k].y, T()),
                                    max_pair(xv[k].z, xv[k].w, T()), T());
        m2 = any ? max_pair(m2, w, T()) : w;
        any = true;
      }
    }
    if (!any) return -INFINITY;
    const T* h = reinterpret_cast<const T*>(&m2);
    return fmaxf(Traits<T>::to_f(h[0]), Traits<T>::to_f(h[1]));
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (first + k * stride < nvec) {
        float f[E];
        unpack<T>(xv[k], f);
#pragma unroll
        for (int e = 0; e < E; ++e) m = fmaxf(m, f[e]);
      }
    }
    return m;
  }
}

// One warp per row (8 rows per 256-thread CTA); exp(x - m) kept in fp32
// registers between the sum and the store.
template <typename T, int VPT>
__global__ void __launch_bounds__(256) sm_fwd_warp_rows(const T* __restrict__ x,
                                                        T* __restrict__ y, int64_t rows,
                                                        int cols) {
  constexpr int E = Traits<T>::kVec;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_trigger();
  if (row >= rows) return;  // whole warps leave together
  if (lane == 0) prefetch_l2(x + row * cols, (uint32_t)(cols * sizeof(T)));
  pdl_wait();
  const int nvec = cols / E;
  const T* xr = x + row * cols;
  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + 32 * k;
    xv[k] = v < nvec ? ld_stream(xr + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  const float m = warp_max(local_max<T, VPT>(xv, lane, 32, nvec));
  float ev[VPT][E];
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const bool in = lane + 32 * k < nvec;
    float f[E];
    unpack<T>(xv[k], f);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      ev[k][e] = in ? expf(f[e] - m) : 0.f;
      s += ev[k][e];
    }
  }
  const float r = 1.f / warp_sum(s);
  T* yr = y + row * cols;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + 32 * k;
    if (v < nvec) {
      float o[E];
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = ev[k][e] * r;
      st_vec(yr + (int64_t)v * E, pack<T>(o));
    }
  }
}

// One CTA per row, the row in registers.  Up to 32 fp32 values a thread the
// exponentials are kept between the sum and the store; beyond that they are
// computed a second time at the store.
template <typename T, int VPT>
__global__ void __launch_bounds__(VPT >= 8 ? 512 : 1024) sm_fwd_cta_row(
    const T* __restrict__ x, T* __restrict__ y, int cols) {
  constexpr int E = Traits<T>::kVec;
  constexpr bool kKeep = VPT * E <= 32;
  __shared__ float red[64];
  const int64_t row = blockIdx.x;
  const int nvec = cols / E;
  const T* xr = x + row * cols;
  pdl_trigger();
  if (threadIdx.x == 0) prefetch_l2(xr, (uint32_t)(cols * sizeof(T)));
  pdl_wait();
  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    xv[k] = v < nvec ? ld_stream(xr + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  const float m = block_max(local_max<T, VPT>(xv, threadIdx.x, blockDim.x, nvec), red, 0);
  float ev[kKeep ? VPT : 1][E];
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const bool in = threadIdx.x + k * blockDim.x < nvec;
    float f[E];
    unpack<T>(xv[k], f);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float t = in ? expf(f[e] - m) : 0.f;
      if (kKeep) ev[kKeep ? k : 0][e] = t;
      s += t;
    }
  }
  const float r = 1.f / block_sum(s, red, 1);
  if (!kKeep) {
    // unpack again at the store rather than hold the unpacked row
#pragma unroll
    for (int k = 0; k < VPT; ++k) opaque(xv[k]);
  }
  T* yr = y + row * cols;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec) {
      float o[E];
      if (kKeep) {
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = ev[kKeep ? k : 0][e] * r;
      } else {
        float f[E];
        unpack<T>(xv[k], f);
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = expf(f[e] - m) * r;
      }
      st_vec(yr + (int64_t)v * E, pack<T>(o));
    }
  }
}

// Any alignment or width: scalar loads, three passes over the row (the
// second and third from L1/L2).
template <typename T>
__global__ void __launch_bounds__(256) sm_fwd_scalar(const T* __restrict__ x, T* __restrict__ y,
                                                     int cols) {
  __shared__ float red[64];
  const int64_t row = blockIdx.x;
  const T* xr = x + row * cols;
  pdl_trigger();
  pdl_wait();
  float m = -INFINITY;
  for (int j = threadIdx.x; j < cols; j += blockDim.x) m = fmaxf(m, Traits<T>::to_f(xr[j]));
  m = block_max(m, red, 0);
  float s = 0.f;
  for (int j = threadIdx.x; j < cols; j += blockDim.x) s += expf(Traits<T>::to_f(xr[j]) - m);
  const float r = 1.f / block_sum(s, red, 1);
  T* yr = y + row * cols;
  for (int j = threadIdx.x; j < cols; j += blockDim.x)
    yr[j] = Traits<T>::from_f(expf(Traits<T>::to_f(xr[j]) - m) * r);
}

// The thread's part of sum(dy * y) over VPT vector pairs.
template <typename T, int VPT>
__device__ __forceinline__ float local_dot(const uint4 (&yv)[VPT], const uint4 (&dv)[VPT]) {
  constexpr int E = Traits<T>::kVec;
  float d = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    float a[E], b[E];
    unpack<T>(yv[k], a);
    unpack<T>(dv[k], b);
#pragma unroll
    for (int e = 0; e < E; ++e) d = fmaf(b[e], a[e], d);
  }
  return d;
}

// Unpack y and dy again for the store instead of holding both unpacked
// across the reduction (which does not fit the registers of wide rows).
template <int VPT>
__device__ __forceinline__ void forget(uint4 (&a)[VPT], uint4 (&b)[VPT]) {
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    opaque(a[k]);
    opaque(b[k]);
  }
}

template <typename T>
__device__ __forceinline__ uint4 sm_dx_vec(const uint4& yv, const uint4& dv, float d) {
  constexpr int E = Traits<T>::kVec;
  float a[E], b[E], o[E];
  unpack<T>(yv, a);
  unpack<T>(dv, b);
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = a[e] * (b[e] - d);
  return pack<T>(o);
}

template <typename T, int VPT>
__global__ void __launch_bounds__(256) sm_bwd_warp_rows(const T* __restrict__ dy,
                                                        const T* __restrict__ y,
                                                        T* __restrict__ dx, int64_t rows,
                                                        int cols) {
  constexpr int E = Traits<T>::kVec;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_trigger();
  if (row >= rows) return;
  if (lane == 0) {
    prefetch_l2(y + row * cols, (uint32_t)(cols * sizeof(T)));
    prefetch_l2(dy + row * cols, (uint32_t)(cols * sizeof(T)));
  }
  pdl_wait();
  const int nvec = cols / E;
  uint4 yv[VPT], dv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + 32 * k;
    const bool in = v < nvec;
    yv[k] = in ? ld_stream(y + row * cols + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    dv[k] = in ? ld_stream(dy + row * cols + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  const float d = warp_sum(local_dot<T, VPT>(yv, dv));
  forget(yv, dv);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + 32 * k;
    if (v < nvec) st_vec(dx + row * cols + (int64_t)v * E, sm_dx_vec<T>(yv[k], dv[k], d));
  }
}

template <typename T, int VPT>
__global__ void __launch_bounds__(VPT >= 8 ? 512 : 1024) sm_bwd_cta_row(
    const T* __restrict__ dy, const T* __restrict__ y, T* __restrict__ dx, int cols) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  const int64_t row = blockIdx.x;
  const int nvec = cols / E;
  pdl_trigger();
  if (threadIdx.x == 0) {
    prefetch_l2(y + row * cols, (uint32_t)(cols * sizeof(T)));
    prefetch_l2(dy + row * cols, (uint32_t)(cols * sizeof(T)));
  }
  pdl_wait();
  uint4 yv[VPT], dv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    const bool in = v < nvec;
    yv[k] = in ? ld_stream(y + row * cols + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    dv[k] = in ? ld_stream(dy + row * cols + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  const float d = block_sum(local_dot<T, VPT>(yv, dv), red, 0);
  forget(yv, dv);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec) st_vec(dx + row * cols + (int64_t)v * E, sm_dx_vec<T>(yv[k], dv[k], d));
  }
}

// Persistent backward for rows of one vector a thread: the CTA
// walks a contiguous range of rows and loads the next row's y and dy while
// the current row's dot is reduced, so loads stay in flight across the
// CTA reduction.
template <typename T>
__global__ void __launch_bounds__(1024) sm_bwd_rows(const T* __restrict__ dy,
                                                   const T* __restrict__ y,
                                                   T* __restrict__ dx, int64_t rows, int cols) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  const int nvec = cols / E;
  const int v = threadIdx.x;
  const bool in = v < nvec;
  const int64_t r0 = (int64_t)blockIdx.x * rows / gridDim.x;
  const int64_t r1 = (int64_t)(blockIdx.x + 1) * rows / gridDim.x;
  pdl_trigger();
  if (threadIdx.x == 0 && r1 > r0) {  // the first rows into L2 (prefetch_l2)
    const uint32_t b = (uint32_t)((r1 - r0 < 4 ? r1 - r0 : 4) * cols * (int64_t)sizeof(T));
    prefetch_l2(y + r0 * cols, b);
    prefetch_l2(dy + r0 * cols, b);
  }
  pdl_wait();
  auto load = [&](int64_t r, uint4& yb, uint4& db) {
    yb = in ? ld_stream(y + r * cols + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    db = in ? ld_stream(dy + r * cols + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  };
  uint4 yc[1], dc[1], yn, dn;
  if (r0 < r1) load(r0, yc[0], dc[0]);
  int parity = 0;
  for (int64_t r = r0; r < r1; ++r) {
    if (r + 1 < r1) load(r + 1, yn, dn);
    const float d = block_sum(local_dot<T, 1>(yc, dc), red, parity);
    parity ^= 1;
    if (in) st_vec(dx + r * cols + (int64_t)v * E, sm_dx_vec<T>(yc[0], dc[0], d));
    yc[0] = yn;
    dc[0] = dn;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) sm_bwd_scalar(const T* __restrict__ dy,
                                                     const T* __restrict__ y, T* __restrict__ dx,
                                                     int cols) {
  __shared__ float red[64];
  const int64_t row = blockIdx.x;
  const T* yr = y + row * cols;
  const T* dr = dy + row * cols;
  pdl_trigger();
  pdl_wait();
  float d = 0.f;
  for (int j = threadIdx.x; j < cols; j += blockDim.x)
    d = fmaf(Traits<T>::to_f(dr[j]), Traits<T>::to_f(yr[j]), d);
  d = block_sum(d, red, 0);
  T* xr = dx + row * cols;
  for (int j = threadIdx.x; j < cols; j += blockDim.x)
    xr[j] = Traits<T>::from_f(Traits<T>::to_f(yr[j]) * (Traits<T>::to_f(dr[j]) - d));
}

int pow2_up(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Forward register-kernel shape of a row of nvec vectors (as the RMSNorm
// forward): vectors per thread and threads per CTA, or vpt 0 when none fits.
void fwd_shape(int nvec, int* vpt, int* tpr) {
  int v = pow2_up((nvec + 127) / 128);
  if (v > 4) v = 4;
  if ((nvec + v - 1) / v > 1024) v = pow2_up((nvec + 511) / 512);
  const int t = ((nvec + v - 1) / v + 31) / 32 * 32;
  if (v > 16 || t > (v >= 8 ? 512 : 1024)) {
    *vpt = 0;
    return;
  }
  *vpt = v;
  *tpr = t;
}

// Backward shape: y and dy both held packed (8 registers a vector pair), so
// 1 or 2 vector pairs a thread up to 1024 threads, 8 at 512 threads (64 of
// the 128 registers), else the scalar kernel.
void bwd_shape(int nvec, int* vpt, int* tpr) {
  int v = 0;
  if (nvec <= 1024) v = 1;
  else if (nvec <= 2048) v = 2;
  else if (nvec <= 4096) v = 8;
  *vpt = v;
  if (v) *tpr = ((nvec + v - 1) / v + 31) / 32 * 32;
}

template <typename T>
cudaError_t sm_fwd_t(const SoftmaxArgs& a, cudaStream_t s) {
  constexpr int E = Traits<T>::kVec;
  const T* x = static_cast<const T*>(a.x);
  T* y = static_cast<T*>(const_cast<void*>(a.y));
  const int nvec = a.cols / E;
  if (a.vec_ok && nvec <= 128) {
    const dim3 grid((unsigned)((a.rows + 7) / 8));
    const int vpt = pow2_up((nvec + 31) / 32);
    if (vpt == 1) return launch_kernel(sm_fwd_warp_rows<T, 1>, grid, dim3(256), 0, s, 1, x, y, a.rows, a.cols);
    if (vpt == 2) return launch_kernel(sm_fwd_warp_rows<T, 2>, grid, dim3(256), 0, s, 1, x, y, a.rows, a.cols);
    return launch_kernel(sm_fwd_warp_rows<T, 4>, grid, dim3(256), 0, s, 1, x, y, a.rows, a.cols);
  }
  int vpt = 0, tpr = 0;
  if (a.vec_ok) fwd_shape(nvec, &vpt, &tpr);
  const dim3 grid((unsigned)a.rows);
  switch (vpt) {
    case 1: return launch_kernel(sm_fwd_cta_row<T, 1>, grid, dim3(tpr), 0, s, 1, x, y, a.cols);
    case 2: return launch_kernel(sm_fwd_cta_row<T, 2>, grid, dim3(tpr), 0, s, 1, x, y, a.cols);
    case 4: return launch_kernel(sm_fwd_cta_row<T, 4>, grid, dim3(tpr), 0, s, 1, x, y, a.cols);
    case 8: return launch_kernel(sm_fwd_cta_row<T, 8>, grid, dim3(tpr), 0, s, 1, x, y, a.cols);
    case 16: return launch_kernel(sm_fwd_cta_row<T, 16>, grid, dim3(tpr), 0, s, 1, x, y, a.cols);
    default: return launch_kernel(sm_fwd_scalar<T>, grid, dim3(256), 0, s, 1, x, y, a.cols);
  }
}

template <typename T>
cudaError_t sm_bwd_t(const SoftmaxArgs& a, cudaStream_t s) {
  constexpr int E = Traits<T>::kVec;
  const T* dy = static_cast<const T*>(a.dy);
  const T* y = static_cast<const T*>(a.y);
  T* dx = static_cast<T*>(a.dx);
  const int nvec = a.cols / E;
  if (a.vec_ok && nvec <= 128) {
    const dim3 grid((unsigned)((a.rows + 7) / 8));
    const int vpt = pow2_up((nvec + 31) / 32);
    if (vpt == 1) return launch_kernel(sm_bwd_warp_rows<T, 1>, grid, dim3(256), 0, s, 1, dy, y, dx, a.rows, a.cols);
    if (vpt == 2) return launch_kernel(sm_bwd_warp_rows<T, 2>, grid, dim3(256), 0, s, 1, dy, y, dx, a.rows, a.cols);
    return launch_kernel(sm_bwd_warp_rows<T, 4>, grid, dim3(256), 0, s, 1, dy, y, dx, a.rows, a.cols);
  }
  int vpt = 0, tpr = 0;
  if (a.vec_ok) bwd_shape(nvec, &vpt, &tpr);
  if (vpt == 1 && tpr > 512) {
    // rows that fill a CTA of more than 512 threads (at most two resident
    // per SM): persistent CTAs that keep the next row loading, as many as
    // are resident at once.  Measured on GB300: 6% faster at 8192 bf16
    // columns, 5% slower at 4096 (four row CTAs per SM overlap already).
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kern = sm_bwd_rows<T>;
    int64_t g = (int64_t)sm_count(dev) * max_blocks_per_sm((const void*)kern, tpr, 0);
    if (g > a.rows) g = a.rows;
    return launch_kernel(kern, dim3((unsigned)g), dim3(tpr), 0, s, 1, dy, y, dx, a.rows, a.cols);
  }
  const dim3 grid((unsigned)a.rows);
  switch (vpt) {
    case 1: return launch_kernel(sm_bwd_cta_row<T, 1>, grid, dim3(tpr), 0, s, 1, dy, y, dx, a.cols);
    case 2: return launch_kernel(sm_bwd_cta_row<T, 2>, grid, dim3(tpr), 0, s, 1, dy, y, dx, a.cols);
    case 8: return launch_kernel(sm_bwd_cta_row<T, 8>, grid, dim3(tpr), 0, s, 1, dy, y, dx, a.cols);
    default: return launch_kernel(sm_bwd_scalar<T>, grid, dim3(256), 0, s, 1, dy, y, dx, a.cols);
  }
}

}  // namespace

cudaError_t launch_softmax_fwd(int dtype, const SoftmaxArgs& a, cudaStream_t s) {
  switch (dtype) {
    case 0: return sm_fwd_t<float>(a, s);
    case 1: return sm_fwd_t<__nv_bfloat16>(a, s);
    default: return sm_fwd_t<__half>(a, s);
  }
}

cudaError_t launch_softmax_bwd(int dtype, const SoftmaxArgs& a, cudaStream_t s) {
  switch (dtype) {
    case 0: return sm_bwd_t<float>(a, s);
    case 1: return sm_bwd_t<__nv_bfloat16>(a, s);
    default: return sm_bwd_t<__half>(a, s);
  }
}

}  // namespace rmsn
