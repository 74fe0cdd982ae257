// RMSNorm backward kernels for sm_103a.
//
// Given dy, x, gamma and the fp32 rstd cached by the forward, per row:
//   x_hat = x * rstd,  g = dy * gain,  c = mean(g * x_hat),
//   dx = rstd * (g - x_hat * c)                     (one rounding at the store)
// and the weight gradient dw = sum over rows of dy * x_hat in fp32.  The
// pages fix the precision (fp32 statistics and reductions for half inputs,
// fp32 weight gradients: Liger-Kernel PR #92; candle PR #4059) but print no
// backward formula; the one above is the exact derivative of the forward.
//
// Structure (two launches on one stream, no host synchronisation):
//   1. a persistent row kernel.  CTA b of G owns the contiguous rows
//      [b*R/G, (b+1)*R/G).  Each thread owns a fixed set of columns, keeps
//      their gains and their fp32 dw accumulators in registers for all of
//      the CTA's rows, and at the end writes them as partial row b of the
//      workspace.  The next row's x, dy and rstd are loaded while the
//      current row is reduced.
//   2. dw_finalize: dw[j] = sum over b of partial[b][j] in a fixed order,
//      launched as a programmatic dependent launch so that its launch
//      overlaps the tail of kernel 1.
// Because G depends only on the sizes and the GPU's SM count and every sum
// has a fixed order, repeated calls give bit-identical dw.
#include "common.cuh"
#include "launch.h"

namespace rmsn {
namespace {

template <typename T, int VPT>
struct RowBuf {
  uint4 x[VPT];
  uint4 dy[VPT];
  float rstd;
};

template <typename T, int VPT>
__device__ __forceinline__ void load_row(RowBuf<T, VPT>& b, const T* __restrict__ dy,
                                         const T* __restrict__ x,
                                         const float* __restrict__ rstd, int64_t r,
                                         int hidden, int nvec) {
  constexpr int E = Traits<T>::kVec;
  const T* xr = x + r * hidden;
  const T* dr = dy + r * hidden;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec) {
      b.x[k] = ld_stream(xr + (int64_t)v * E);
      b.dy[k] = ld_stream(dr + (int64_t)v * E);
    } else {
      b.x[k] = make_uint4(0, 0, 0, 0);
      b.dy[k] = make_uint4(0, 0, 0, 0);
    }
  }
  b.rstd = __ldg(rstd + r);
}

template <typename T, int VPT, bool PREFETCH>
__global__ void __launch_bounds__(1024) bwd_cta_rows(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ rstd, T* __restrict__ dx, float* __restrict__ partial,
    int64_t rows, int hidden, float off) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  // Let the finalize kernel be scheduled now; it waits for this grid to
  // complete before reading the partials.
  pdl_trigger();
  pdl_wait();
  const int nvec = hidden / E;
  const int64_t r0 = (int64_t)blockIdx.x * rows / gridDim.x;
  const int64_t r1 = (int64_t)(blockIdx.x + 1) * rows / gridDim.x;
  const float inv_n_div = (float)hidden;

  float ge[VPT][E];
  float acc[VPT][E];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    uint4 gv = v < nvec ? ld_shared_ro(gamma + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    unpack<T>(gv, ge[k]);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      ge[k][i] += off;
      acc[k][i] = 0.f;
    }
  }

  // With PREFETCH the next row is in flight while this one is reduced
  // (short rows); long rows carry enough bytes in flight on their own.
  RowBuf<T, VPT> cur, nxt;
  if (PREFETCH && r0 < r1) load_row<T, VPT>(cur, dy, x, rstd, r0, hidden, nvec);
  int parity = 0;
  for (int64_t r = r0; r < r1; ++r) {
    if (PREFETCH) {
      if (r + 1 < r1) load_row<T, VPT>(nxt, dy, x, rstd, r + 1, hidden, nvec);
    } else {
      load_row<T, VPT>(cur, dy, x, rstd, r, hidden, nvec);
    }
    const float rs = cur.rstd;
    // pass 1 over the registers: row dot and dw accumulation
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      float xf[E], df[E];
      unpack<T>(cur.x[k], xf);
      unpack<T>(cur.dy[k], df);
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float xh = xf[i] * rs;
        dot = fmaf(df[i] * ge[k][i], xh, dot);
        acc[k][i] = fmaf(df[i], xh, acc[k][i]);
      }
    }
    dot = block_sum(dot, red, parity);
    parity ^= 1;
    const float c = dot / inv_n_div;
    // pass 2: dx
    T* dxr = dx + r * hidden;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nvec) {
        float xf[E], df[E], o[E];
        unpack<T>(cur.x[k], xf);
        unpack<T>(cur.dy[k], df);
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const float xh = xf[i] * rs;
          const float g = df[i] * ge[k][i];
          o[i] = fmaf(-xh, c, g) * rs;
        }
        st_vec(dxr + (int64_t)v * E, pack<T>(o));
      }
    }
    if (PREFETCH) cur = nxt;
  }

  float* pr = partial + (int64_t)blockIdx.x * hidden;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec) {
#pragma unroll
      for (int i = 0; i < E; i += 4) {
        const float4 q = make_float4(acc[k][i], acc[k][i + 1], acc[k][i + 2], acc[k][i + 3]);
        *reinterpret_cast<float4*>(pr + (int64_t)v * E + i) = q;
      }
    }
  }
}

// Any alignment and width: scalar loads; the partial row lives in the
// workspace and each thread updates only its own columns.
template <typename T>
__global__ void __launch_bounds__(256) bwd_scalar(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ rstd, T* __restrict__ dx, float* __restrict__ partial,
    int64_t rows, int hidden, float off) {
  __shared__ float red[64];
  pdl_trigger();
  pdl_wait();
  const int64_t r0 = (int64_t)blockIdx.x * rows / gridDim.x;
  const int64_t r1 = (int64_t)(blockIdx.x + 1) * rows / gridDim.x;
  float* pr = partial + (int64_t)blockIdx.x * hidden;
  int parity = 0;
  for (int64_t r = r0; r < r1; ++r) {
    const T* xr = x + r * hidden;
    const T* dr = dy + r * hidden;
    const float rs = rstd[r];
    float dot = 0.f;
    for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
      const float xh = Traits<T>::to_f(xr[j]) * rs;
      const float g = Traits<T>::to_f(dr[j]) * (Traits<T>::to_f(gamma[j]) + off);
      dot = fmaf(g, xh, dot);
    }
    dot = block_sum(dot, red, parity);
    parity ^= 1;
    const float c = dot / (float)hidden;
    T* dxr = dx + r * hidden;
    for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
      const float df = Traits<T>::to_f(dr[j]);
      const float xh = Traits<T>::to_f(xr[j]) * rs;
      const float g = df * (Traits<T>::to_f(gamma[j]) + off);
      dxr[j] = Traits<T>::from_f(fmaf(-xh, c, g) * rs);
      pr[j] = fmaf(df, xh, r == r0 ? 0.f : pr[j]);
    }
  }
}

// out[j] = sum_b partial[b][j] over the `ncols` columns of a [nparts, ncols]
// fp32 matrix, written to out0[j] for j < split and to out1[j - split]
// otherwise.  Block (32 columns) x (kFinLanes lanes over b): lane t sums
// b = t, t + kFinLanes, ... in increasing order, then lane 0 adds the lane
// sums in order.  The order depends only on nparts.  Blocks of 512 threads
// fit beside a resident CTA of the row kernel, so they are already waiting
// when it finishes (programmatic dependent launch); measured on GB300, 8
// lanes are slower (longer serial sums) and 32 no faster.
constexpr int kFinLanes = 16;

__global__ void __launch_bounds__(32 * kFinLanes) dw_finalize(const float* __restrict__ partial,
                                                             int nparts, int ncols,
                                                             float* __restrict__ out0,
                                                             float* __restrict__ out1, int split) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s[kFinLanes][33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int j = blockIdx.x * 32 + tx;
  float a = 0.f;
  if (j < ncols) {
#pragma unroll 8
    for (int b = ty; b < nparts; b += kFinLanes) a += partial[(int64_t)b * ncols + j];
  }
  s[ty][tx] = a;
  __syncthreads();
  if (ty == 0 && j < ncols) {
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < kFinLanes; ++q) t += s[q][tx];
    if (j < split)
      out0[j] = t;
    else if (out1 != nullptr)
      out1[j - split] = t;
  }
}

}  // namespace

cudaError_t launch_column_sums(const float* partial, int nparts, int ncols, float* out0,
                               float* out1, int split, cudaStream_t s) {
  return launch_kernel(dw_finalize, dim3((unsigned)((ncols + 31) / 32)), dim3(32, kFinLanes), 0, s, 1,
                       partial, nparts, ncols, out0, out1, split);
}

namespace {

cudaError_t launch_finalize(const float* partial, float* dw, int nparts, int hidden,
                            cudaStream_t s) {
  return launch_column_sums(partial, nparts, hidden, dw, nullptr, hidden, s);
}

template <typename T, int VPT>
cudaError_t launch_rows(const BwdArgs& a, int tpr, cudaStream_t s, int* nparts) {
  auto kern = bwd_cta_rows<T, VPT, VPT == 1>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int occ = max_blocks_per_sm((const void*)kern, tpr, 0);
  int64_t g = (int64_t)sm_count(dev) * (occ > 0 ? occ : 1);
  if (g > a.rows) g = a.rows;
  if (g > a.max_partials) g = a.max_partials;
  *nparts = (int)g;
  return launch_kernel(kern, dim3((unsigned)g), dim3(tpr), 0, s, 1,
                       static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                       static_cast<const T*>(a.gamma), a.rstd, static_cast<T*>(a.dx), a.partial,
                       a.rows, a.hidden, a.offset ? 1.f : 0.f);
}

template <typename T> int dtype_code();
template <> int dtype_code<float>() { return 0; }
template <> int dtype_code<__nv_bfloat16>() { return 1; }
template <> int dtype_code<__half>() { return 2; }

template <typename T>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t s, int* launches) {
  constexpr int E = Traits<T>::kVec;
  const int nvec = a.hidden / E;
  const int max_vpt = E == 4 ? 4 : 2;  // at most 16 columns per thread
  int nparts = 0;
  cudaError_t e = cudaErrorInvalidValue;
  // the staged pipeline where x and dy rows fit its ring, else the register
  // kernel, else (rows too wide for one CTA) a thread-block cluster, else the
  // scalar kernel
  bool done = try_launch_bwd_tma(dtype_code<T>(), a, s, &e, &nparts);
  if (!done && a.vec_ok) {
    int vpt = 1;
    while (vpt < max_vpt && (nvec + vpt - 1) / vpt > 1024) vpt <<= 1;
    const int tpr = ((nvec + vpt - 1) / vpt + 31) / 32 * 32;
    if (tpr <= 1024) {
      if (vpt == 1) e = launch_rows<T, 1>(a, tpr, s, &nparts);
      else if (vpt == 2 || E != 4) e = launch_rows<T, 2>(a, tpr, s, &nparts);
      else e = launch_rows<T, (E == 4 ? 4 : 2)>(a, tpr, s, &nparts);
      done = true;
    }
  }
  if (!done) done = try_launch_bwd_cluster(dtype_code<T>(), a, s, &e, &nparts);
  if (!done) {
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kern = bwd_scalar<T>;
    const int occ = max_blocks_per_sm((const void*)kern, 256, 0);
    int64_t g = (int64_t)sm_count(dev) * (occ > 0 ? occ : 1);
    if (g > a.rows) g = a.rows;
    if (g > a.max_partials) g = a.max_partials;
    nparts = (int)g;
    e = launch_kernel(kern, dim3((unsigned)g), dim3(256), 0, s, 1,
                      static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                      static_cast<const T*>(a.gamma), a.rstd, static_cast<T*>(a.dx), a.partial,
                      a.rows, a.hidden, a.offset ? 1.f : 0.f);
  }
  if (e != cudaSuccess) return e;
  *launches += 1;
  e = launch_finalize(a.partial, a.dw, nparts, a.hidden, s);
  if (e == cudaSuccess) *launches += 1;
  return e;
}

}  // namespace

cudaError_t launch_bwd(int dtype, const BwdArgs& a, cudaStream_t s, int* launches) {
  switch (dtype) {
    case 0: return launch_bwd_t<float>(a, s, launches);
    case 1: return launch_bwd_t<__nv_bfloat16>(a, s, launches);
    default: return launch_bwd_t<__half>(a, s, launches);
  }
}

}  // namespace rmsn
