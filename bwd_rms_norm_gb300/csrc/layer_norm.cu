// LayerNorm forward and backward kernels for sm_103a (the sibling of the
// RMSNorm path: same row-reduction skeleton plus a mean).
//
// Forward, per row: mean = sum(x)/N and var = sum((x - mean)^2)/N in fp32
// (two passes over the row held in registers), rstd = 1/sqrt(var + eps)
// correctly rounded, y = round(fma(x_hat, gamma, beta)) -- one rounding at
// the store; mean and rstd are stored in fp32 (Liger-Kernel PR #1608 notes
// that layer_norm keeps them in fp32).
//
// Backward, given the cached mean and rstd: x_hat = (x - mean) * rstd,
// g = dy * gamma, c1 = sum(g)/N, c2 = sum(g * x_hat)/N (one two-value CTA
// reduction), dx = rstd * (g - c1 - x_hat * c2); dgamma = sum_r dy * x_hat
// and dbeta = sum_r dy as fp32 per-CTA partials over contiguous row ranges,
// reduced in a fixed order by the column-sum kernel of bwd.cu.
//
// Kernels here: one warp per row (short rows), one CTA per row (the row in
// registers), and scalar kernels for rows that are not 16-byte aligned.  The
// TMA-staged warp-specialised LayerNorm kernels live in tma.cu and are tried
// first: the backward for every aligned row that fits the ring, the forward
// for rows over 4 KB.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace rmsn {
namespace {

template <typename T>
__device__ __forceinline__ uint4 ln_scale_vec(const float (&xf)[Traits<T>::kVec], float mu,
                                              float rs, const uint4& gv, const uint4& bv,
                                              bool has_beta) {
  constexpr int E = Traits<T>::kVec;
  float g[E], b[E], o[E];
  unpack<T>(gv, g);
  if (has_beta) {
    unpack<T>(bv, b);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) b[e] = 0.f;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = fmaf((xf[e] - mu) * rs, g[e], b[e]);
  return pack<T>(o);
}

// Row statistics from a thread's VPT vectors, reduced by `sum` (a warp or
// CTA sum): returns (mean, rstd).
template <typename T, int VPT, typename Sum>
__device__ __forceinline__ float2 ln_stats(const uint4 (&xv)[VPT], int first, int stride,
                                           int nvec, int hidden, float eps, Sum sum) {
  constexpr int E = Traits<T>::kVec;
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    float f[E];
    unpack<T>(xv[k], f);
#pragma unroll
    for (int e = 0; e < E; ++e) s += f[e];
  }
  const float mu = sum(s, 0) / (float)hidden;
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    if (first + k * stride < nvec) {
      float f[E];
      unpack<T>(xv[k], f);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float d = f[e] - mu;
        q = fmaf(d, d, q);
      }
    }
  }
  const float var = sum(q, 1) / (float)hidden;
  return make_float2(mu, rstd_of(var, eps));
}

template <typename T, int VPT>
__global__ void __launch_bounds__(256) ln_fwd_warp_rows(
    const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
    T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, int64_t rows,
    int hidden, float eps) {
  constexpr int E = Traits<T>::kVec;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_trigger();
  if (row >= rows) return;
  pdl_wait();
  const int nvec = hidden / E;
  const T* xr = x + row * hidden;
  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + 32 * k;
    xv[k] = v < nvec ? ld_stream(xr + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  const float2 st = ln_stats<T, VPT>(xv, lane, 32, nvec, hidden, eps,
                                     [](float v, int) { return warp_sum(v); });
  if (lane == 0) {
    mean[row] = st.x;
    rstd[row] = st.y;
  }
  T* yr = y + row * hidden;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + 32 * k;
    if (v < nvec) {
      float f[E];
      unpack<T>(xv[k], f);
      const uint4 gv = ld_shared_ro(gamma + (int64_t)v * E);
      const uint4 bv = beta ? ld_shared_ro(beta + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
      st_vec(yr + (int64_t)v * E, ln_scale_vec<T>(f, st.x, st.y, gv, bv, beta != nullptr));
    }
  }
}

template <typename T, int VPT>
__global__ void __launch_bounds__(VPT >= 8 ? 512 : 1024) ln_fwd_cta_row(
    const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
    T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, int hidden,
    float eps) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  const int64_t row = blockIdx.x;
  const int nvec = hidden / E;
  const T* xr = x + row * hidden;
  pdl_trigger();
  pdl_wait();
  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    xv[k] = v < nvec ? ld_stream(xr + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  const float2 st = ln_stats<T, VPT>(xv, threadIdx.x, blockDim.x, nvec, hidden, eps,
                                     [&](float v, int p) { return block_sum(v, red, p); });
  if (threadIdx.x == 0) {
    mean[row] = st.x;
    rstd[row] = st.y;
  }
  T* yr = y + row * hidden;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec) {
      float f[E];
      unpack<T>(xv[k], f);
      const uint4 gv = ld_shared_ro(gamma + (int64_t)v * E);
      const uint4 bv = beta ? ld_shared_ro(beta + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
      st_vec(yr + (int64_t)v * E, ln_scale_vec<T>(f, st.x, st.y, gv, bv, beta != nullptr));
    }
  }
}

// Any alignment: scalar loads, the row read from L1/L2 in each pass.
template <typename T>
__global__ void __launch_bounds__(256) ln_fwd_scalar(
    const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
    T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, int hidden,
    float eps) {
  __shared__ float red[64];
  const int64_t row = blockIdx.x;
  const T* xr = x + row * hidden;
  pdl_trigger();
  pdl_wait();
  float s = 0.f;
  for (int j = threadIdx.x; j < hidden; j += blockDim.x) s += Traits<T>::to_f(xr[j]);
  const float mu = block_sum(s, red, 0) / (float)hidden;
  float q = 0.f;
  for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
    const float d = Traits<T>::to_f(xr[j]) - mu;
    q = fmaf(d, d, q);
  }
  const float rs = rstd_of(block_sum(q, red, 1) / (float)hidden, eps);
  if (threadIdx.x == 0) {
    mean[row] = mu;
    rstd[row] = rs;
  }
  T* yr = y + row * hidden;
  for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
    const float b = beta ? Traits<T>::to_f(beta[j]) : 0.f;
    yr[j] = Traits<T>::from_f(fmaf((Traits<T>::to_f(xr[j]) - mu) * rs,
                                   Traits<T>::to_f(gamma[j]), b));
  }
}

// One vector per thread: gains in registers and the next row prefetched.
// Two vectors per thread: gains read from L1 at each use and no prefetch,
// so that the two fp32 accumulator sets fit the 64 registers of a
// 1024-thread CTA.
template <typename T, int VPT>
__global__ void __launch_bounds__(1024) ln_bwd_cta_rows(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd, T* __restrict__ dx,
    float* __restrict__ partial, int64_t rows, int hidden) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float2 red[64];
  pdl_trigger();
  pdl_wait();
  const int nvec = hidden / E;
  const int64_t r0 = (int64_t)blockIdx.x * rows / gridDim.x;
  const int64_t r1 = (int64_t)(blockIdx.x + 1) * rows / gridDim.x;
  constexpr bool kOne = VPT == 1;
  float ge[kOne ? 1 : 1][E], ag[VPT][E], ab[VPT][E];
  auto gains = [&](int k, float (&g)[E]) {
    if (kOne) {
#pragma unroll
      for (int e = 0; e < E; ++e) g[e] = ge[0][e];
    } else {
      const int v = threadIdx.x + k * blockDim.x;
      unpack<T>(v < nvec ? ld_shared_ro(gamma + (int64_t)v * E) : make_uint4(0, 0, 0, 0), g);
    }
  };
  if (kOne) {
    const int v = threadIdx.x;
    unpack<T>(v < nvec ? ld_shared_ro(gamma + (int64_t)v * E) : make_uint4(0, 0, 0, 0), ge[0]);
  }
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < E; ++e) ag[k][e] = ab[k][e] = 0.f;
  uint4 xc[VPT], dc[VPT], xn[kOne ? VPT : 1], dn[kOne ? VPT : 1];
  float mc = 0.f, rc = 0.f, mn = 0.f, rn = 0.f;
  auto load = [&](int64_t r, auto& xb, auto& db, float& mb, float& rb) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      const bool in = v < nvec;
      xb[k] = in ? ld_stream(x + r * hidden + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
      db[k] = in ? ld_stream(dy + r * hidden + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    }
    mb = __ldg(mean + r);
    rb = __ldg(rstd + r);
  };
  if (kOne && r0 < r1) load(r0, xc, dc, mc, rc);
  int parity = 0;
  for (int64_t r = r0; r < r1; ++r) {
    if (kOne) {
      if (r + 1 < r1) load(r + 1, xn, dn, mn, rn);
    } else {
      load(r, xc, dc, mc, rc);
    }
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      float xf[E], df[E], gf[E];
      unpack<T>(xc[k], xf);
      unpack<T>(dc[k], df);
      gains(k, gf);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float xh = (xf[e] - mc) * rc;
        const float g = df[e] * gf[e];
        s1 += g;
        s2 = fmaf(g, xh, s2);
        ag[k][e] = fmaf(df[e], xh, ag[k][e]);
        ab[k][e] += df[e];
      }
    }
    const float2 t = block_sum2(s1, s2, red, parity);
    parity ^= 1;
    const float c1 = t.x / (float)hidden, c2 = t.y / (float)hidden;
    if (!kOne) {
      // unpack again below rather than hold the unpacked row across the
      // reduction
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        opaque(xc[k]);
        opaque(dc[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nvec) {
        float xf[E], df[E], gf[E], o[E];
        unpack<T>(xc[k], xf);
        unpack<T>(dc[k], df);
        gains(k, gf);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float xh = (xf[e] - mc) * rc;
          o[e] = fmaf(-xh, c2, df[e] * gf[e] - c1) * rc;
        }
        st_vec(dx + r * hidden + (int64_t)v * E, pack<T>(o));
      }
    }
    if (kOne) {
      xc[0] = xn[0];
      dc[0] = dn[0];
      mc = mn;
      rc = rn;
    }
  }
  // partial row b: dgamma in columns [0, N), dbeta in [N, 2N)
  float* pr = partial + (int64_t)blockIdx.x * 2 * hidden;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nvec) {
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        *reinterpret_cast<float4*>(pr + (int64_t)v * E + e) =
            make_float4(ag[k][e], ag[k][e + 1], ag[k][e + 2], ag[k][e + 3]);
        *reinterpret_cast<float4*>(pr + hidden + (int64_t)v * E + e) =
            make_float4(ab[k][e], ab[k][e + 1], ab[k][e + 2], ab[k][e + 3]);
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) ln_bwd_scalar(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd, T* __restrict__ dx,
    float* __restrict__ partial, int64_t rows, int hidden) {
  __shared__ float2 red[64];
  pdl_trigger();
  pdl_wait();
  const int64_t r0 = (int64_t)blockIdx.x * rows / gridDim.x;
  const int64_t r1 = (int64_t)(blockIdx.x + 1) * rows / gridDim.x;
  float* pr = partial + (int64_t)blockIdx.x * 2 * hidden;
  int parity = 0;
  for (int64_t r = r0; r < r1; ++r) {
    const T* xr = x + r * hidden;
    const T* dr = dy + r * hidden;
    const float mu = mean[r], rs = rstd[r];
    float s1 = 0.f, s2 = 0.f;
    for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
      const float xh = (Traits<T>::to_f(xr[j]) - mu) * rs;
      const float g = Traits<T>::to_f(dr[j]) * Traits<T>::to_f(gamma[j]);
      s1 += g;
      s2 = fmaf(g, xh, s2);
    }
    const float2 t = block_sum2(s1, s2, red, parity);
    parity ^= 1;
    const float c1 = t.x / (float)hidden, c2 = t.y / (float)hidden;

    T* dxr = dx + r * hidden;
    for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
      const float df = Traits<T>::to_f(dr[j]);
      const float xh = (Traits<T>::to_f(xr[j]) - mu) * rs;
      const float g = df * Traits<T>::to_f(gamma[j]);
      dxr[j] = Traits<T>::from_f(fmaf(-xh, c2, g - c1) * rs);
      pr[j] = fmaf(df, xh, r == r0 ? 0.f : pr[j]);
      pr[hidden + j] = (r == r0 ? 0.f : pr[hidden + j]) + df;
    }
  }
}

template <typename T>
constexpr int dtype_of() {
  return std::is_same<T, float>::value ? 0 : std::is_same<T, __nv_bfloat16>::value ? 1 : 2;
}

int pow2_ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

template <typename T>
cudaError_t ln_fwd_t(const LnFwdArgs& a, cudaStream_t s, int* launches) {
  constexpr int E = Traits<T>::kVec;
  const T* x = static_cast<const T*>(a.x);
  const T* g = static_cast<const T*>(a.gamma);
  const T* b = static_cast<const T*>(a.beta);
  T* y = static_cast<T*>(a.y);
  const int nvec = a.hidden / E;
  cudaError_t e = cudaErrorInvalidValue;
  bool done = false;
  // rows over 4 KB: the TMA-staged pipeline (as the RMSNorm forward;
  // measured on GB300, whole LayerNorm steps 3.5-9% faster than with the
  // register kernels at those widths)
  if ((int64_t)a.hidden * (int64_t)sizeof(T) > 4 * 1024 &&
      try_launch_ln_fwd_tma(dtype_of<T>(), a, s, &e)) {
    if (e == cudaSuccess) *launches += 1;
    return e;
  }
  if (a.vec_ok && nvec <= 128) {
    const int vpt = pow2_ceil((nvec + 31) / 32);
    const dim3 grid((unsigned)((a.rows + 7) / 8));
    switch (vpt) {
      case 1: e = launch_kernel(ln_fwd_warp_rows<T, 1>, grid, dim3(256), 0, s, 1, x, g, b, y, a.mean, a.rstd, a.rows, a.hidden, a.eps); break;
      case 2: e = launch_kernel(ln_fwd_warp_rows<T, 2>, grid, dim3(256), 0, s, 1, x, g, b, y, a.mean, a.rstd, a.rows, a.hidden, a.eps); break;
      default: e = launch_kernel(ln_fwd_warp_rows<T, 4>, grid, dim3(256), 0, s, 1, x, g, b, y, a.mean, a.rstd, a.rows, a.hidden, a.eps); break;
    }
    done = true;
  } else if (a.vec_ok) {
    // about 128 threads with up to 4 vectors each per row (as the RMSNorm
    // forward); 8 or 16 vectors at 512 threads for the widest rows
    int vpt = pow2_ceil((nvec + 127) / 128);
    if (vpt > 4) vpt = 4;
    if ((nvec + vpt - 1) / vpt > 1024) vpt = pow2_ceil((nvec + 511) / 512);
    const int tpr = ((nvec + vpt - 1) / vpt + 31) / 32 * 32;
    if (vpt <= 16 && tpr <= (vpt >= 8 ? 512 : 1024)) {
      const dim3 grid((unsigned)a.rows);
      switch (vpt) {
        case 1: e = launch_kernel(ln_fwd_cta_row<T, 1>, grid, dim3(tpr), 0, s, 1, x, g, b, y, a.mean, a.rstd, a.hidden, a.eps); break;
        case 2: e = launch_kernel(ln_fwd_cta_row<T, 2>, grid, dim3(tpr), 0, s, 1, x, g, b, y, a.mean, a.rstd, a.hidden, a.eps); break;
        case 4: e = launch_kernel(ln_fwd_cta_row<T, 4>, grid, dim3(tpr), 0, s, 1, x, g, b, y, a.mean, a.rstd, a.hidden, a.eps); break;
        case 8: e = launch_kernel(ln_fwd_cta_row<T, 8>, grid, dim3(tpr), 0, s, 1, x, g, b, y, a.mean, a.rstd, a.hidden, a.eps); break;
        default: e = launch_kernel(ln_fwd_cta_row<T, 16>, grid, dim3(tpr), 0, s, 1, x, g, b, y, a.mean, a.rstd, a.hidden, a.eps); break;
      }
      done = true;
    }
  }
  if (!done)
    e = launch_kernel(ln_fwd_scalar<T>, dim3((unsigned)a.rows), dim3(256), 0, s, 1, x, g, b, y,
                      a.mean, a.rstd, a.hidden, a.eps);
  if (e == cudaSuccess) *launches += 1;
  return e;
}

template <typename T, int VPT>
cudaError_t ln_bwd_rows(const LnBwdArgs& a, int tpr, cudaStream_t s, int* nparts) {
  auto kern = ln_bwd_cta_rows<T, VPT>;
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
                       static_cast<const T*>(a.gamma), a.mean, a.rstd, static_cast<T*>(a.dx),
                       a.partial, a.rows, a.hidden);
}

template <typename T>
cudaError_t ln_bwd_t(const LnBwdArgs& a, cudaStream_t s, int* launches) {
  constexpr int E = Traits<T>::kVec;
  const int nvec = a.hidden / E;
  int nparts = 0;
  cudaError_t e = cudaErrorInvalidValue;
  bool done = false;
  if (try_launch_ln_bwd_tma(dtype_of<T>(), a, s, &e, &nparts)) {
    if (e != cudaSuccess) return e;
    done = true;
  }
  if (!done && a.vec_ok) {
    // one or two vectors per thread (gains and both accumulators in fp32
    // registers), up to 1024 threads
    const int vpt = nvec <= 1024 ? 1 : 2;
    const int tpr = ((nvec + vpt - 1) / vpt + 31) / 32 * 32;
    if (tpr <= 1024) {
      e = vpt == 1 ? ln_bwd_rows<T, 1>(a, tpr, s, &nparts) : ln_bwd_rows<T, 2>(a, tpr, s, &nparts);
      done = true;
    }
  }
  if (!done) {
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    auto kern = ln_bwd_scalar<T>;
    const int occ = max_blocks_per_sm((const void*)kern, 256, 0);
    int64_t g = (int64_t)sm_count(dev) * (occ > 0 ? occ : 1);
    if (g > a.rows) g = a.rows;
    if (g > a.max_partials) g = a.max_partials;
    nparts = (int)g;
    e = launch_kernel(kern, dim3((unsigned)g), dim3(256), 0, s, 1, static_cast<const T*>(a.dy),
                      static_cast<const T*>(a.x), static_cast<const T*>(a.gamma), a.mean, a.rstd,
                      static_cast<T*>(a.dx), a.partial, a.rows, a.hidden);
  }
  if (e != cudaSuccess) return e;
  *launches += 1;
  e = launch_column_sums(a.partial, nparts, 2 * a.hidden, a.dgamma, a.dbeta, a.hidden, s);
  if (e == cudaSuccess) *launches += 1;
  return e;
}

}  // namespace

cudaError_t launch_ln_fwd(int dtype, const LnFwdArgs& a, cudaStream_t s, int* launches) {
  switch (dtype) {
    case 0: return ln_fwd_t<float>(a, s, launches);
    case 1: return ln_fwd_t<__nv_bfloat16>(a, s, launches);
    default: return ln_fwd_t<__half>(a, s, launches);
  }
}

cudaError_t launch_ln_bwd(int dtype, const LnBwdArgs& a, cudaStream_t s, int* launches) {
  switch (dtype) {
    case 0: return ln_bwd_t<float>(a, s, launches);
    case 1: return ln_bwd_t<__nv_bfloat16>(a, s, launches);
    default: return ln_bwd_t<__half>(a, s, launches);
  }
}

}  // namespace rmsn
