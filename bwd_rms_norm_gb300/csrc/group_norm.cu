// GroupNorm forward and backward for sm_103a (Liger-Kernel PR #1608, "fix
// (group_norm): keep the backward statistics and reductions in fp32":
// Mean and RSTD stored in fp32, every backward reduction in fp32).
//
// x is [n, C, S] (S spatial positions, contiguous); the C channels form G
// groups of Cg = C / G consecutive channels, so group (n, g) is one
// contiguous run of M = Cg * S elements.  Per group: mean and the biased
// variance in fp32 (two passes over the group held in registers), rstd =
// 1/sqrt(var + eps) correctly rounded, y = round(fma(x_hat, W[c], B[c])).
// Backward, with g = dy * W[c]: c1 = mean(g), c2 = rstd * mean(g * (x -
// mean)) over the group, dx = rstd * (g - c1 - x_hat * c2); per channel
// dW = sum dy * x_hat and dB = sum dy over samples and positions.
//
// A group is long (65536 to 262144 elements in the shapes the PR times), so
// it is split over a thread-block cluster of up to 16 CTAs, each holding its
// slice in registers; the group sums go through distributed shared memory
// (cluster.cuh), and every element is read once.  The backward's per-channel
// sums are reduced inside the CTA in a fixed order (per-vector sums in
// shared memory, one warp per channel) and written as fp32 partial rows
// [n * csize, 2C] (dW columns, then dB), which the column-sum kernel of
// bwd.cu reduces in a fixed order: the result is deterministic.  Groups
// that are not 16-byte aligned, or too long for 16 CTAs, run scalar kernels
// (one CTA per group).
#include <mutex>

#include "cluster.cuh"

namespace rmsn {
namespace {

// Most 16-byte vectors one CTA holds: 8 a thread at 512 threads (x, and in
// the backward dy as well: 64 of the 128 registers a thread).  Cluster CTAs
// stay at 512 threads so that 16 of them fit one GPC.
constexpr int kGnMaxVec = 4096;
constexpr int kGnThreads = 512;

int gn_vpt(int nv) { return nv <= 512 ? 1 : nv <= 1024 ? 2 : nv <= 2048 ? 4 : 8; }

template <typename T, int VPT>
__global__ void __launch_bounds__(kGnThreads) gn_fwd_cluster(
    const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
    T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, int M, int spv,
    int Cg, int G, float eps, int csize) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  __shared__ float slots[2 * kMaxCluster];
  const uint32_t rank = csize > 1 ? cta_rank() : 0u;
  const int64_t grp = blockIdx.x / csize;
  const int cbase = (int)(grp % G) * Cg;
  const int nv = M / E / csize;
  const int base = (int)rank * nv;
  const T* xg = x + grp * M;
  if (csize > 1) cluster_sync();  // every CTA of the cluster is running
  pdl_trigger();
  pdl_wait();
  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    xv[k] = v < nv ? ld_stream(xg + (int64_t)(base + v) * E) : make_uint4(0, 0, 0, 0);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    float f[E];
    unpack<T>(xv[k], f);
#pragma unroll
    for (int e = 0; e < E; ++e) s += f[e];
  }
  s = csize > 1 ? cluster_sum(s, red, slots, 0, rank, csize) : block_sum(s, red, 0);
  const float mu = s / (float)M;
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    if (threadIdx.x + k * blockDim.x < nv) {
      float f[E];
      unpack<T>(xv[k], f);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float d = f[e] - mu;
        q = fmaf(d, d, q);
      }
    }
  }
  q = csize > 1 ? cluster_sum(q, red, slots, 1, rank, csize) : block_sum(q, red, 1);
  const float rs = rstd_of(q / (float)M, eps);
  if (rank == 0 && threadIdx.x == 0) {
    mean[grp] = mu;
    rstd[grp] = rs;
  }
  T* yg = y + grp * M;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      const int c = cbase + (base + v) / spv;  // a vector lies in one channel
      const float w = Traits<T>::to_f(gamma[c]);
      const float b = beta ? Traits<T>::to_f(beta[c]) : 0.f;
      float f[E], o[E];
      unpack<T>(xv[k], f);
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = fmaf((f[e] - mu) * rs, w, b);
      st_vec(yg + (int64_t)(base + v) * E, pack<T>(o));
    }
  }
}

template <typename T, int VPT>
__global__ void __launch_bounds__(kGnThreads) gn_bwd_cluster(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd, T* __restrict__ dx,
    float* __restrict__ partial, int M, int spv, int Cg, int G, int C, int csize) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float2 vsum[kGnMaxVec];
  __shared__ float2 red[64];
  __shared__ float2 slots[2 * kMaxCluster];
  const uint32_t rank = csize > 1 ? cta_rank() : 0u;
  const int64_t grp = blockIdx.x / csize;
  const int64_t n = grp / G;
  const int cbase = (int)(grp % G) * Cg;
  const int nv = M / E / csize;
  const int base = (int)rank * nv;
  const T* xg = x + grp * M;
  const T* dg = dy + grp * M;
  if (csize > 1) cluster_sync();
  pdl_trigger();
  pdl_wait();
  const float mu = __ldg(mean + grp), rs = __ldg(rstd + grp);
  uint4 xv[VPT], dv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    const bool in = v < nv;
    xv[k] = in ? ld_stream(xg + (int64_t)(base + v) * E) : make_uint4(0, 0, 0, 0);
    dv[k] = in ? ld_stream(dg + (int64_t)(base + v) * E) : make_uint4(0, 0, 0, 0);
  }
  float s1 = 0.f, s2 = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      const float w = Traits<T>::to_f(gamma[cbase + (base + v) / spv]);
      float xf[E], df[E];
      unpack<T>(xv[k], xf);
      unpack<T>(dv[k], df);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float gd = df[e] * w;
        s1 += gd;
        s2 = fmaf(gd, xf[e] - mu, s2);
      }
    }
  }
  const float2 t = csize > 1 ? cluster_sum2(s1, s2, red, slots, 0, rank, csize)
                             : block_sum2(s1, s2, red, 0);
  const float c1 = t.x / (float)M, c2 = t.y * rs / (float)M;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    // unpack again below rather than hold both rows unpacked across the sum
    opaque(xv[k]);
    opaque(dv[k]);
  }
  T* xo = dx + grp * M;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      const float w = Traits<T>::to_f(gamma[cbase + (base + v) / spv]);
      float xf[E], df[E], o[E];
      unpack<T>(xv[k], xf);
      unpack<T>(dv[k], df);
      float pg = 0.f, pb = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float xh = (xf[e] - mu) * rs;
        o[e] = fmaf(-xh, c2, df[e] * w - c1) * rs;
        pg = fmaf(df[e], xh, pg);
        pb += df[e];
      }
      st_vec(xo + (int64_t)(base + v) * E, pack<T>(o));
      vsum[v] = make_float2(pg, pb);
    }
  }
  __syncthreads();
  // Per-channel sums over this slice, one warp per channel, lanes striding
  // over the channel's vectors in order; channels of the group this slice
  // does not touch get 0 so that every column of the partial row is written.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  float* prow = partial + (n * csize + rank) * (int64_t)(2 * C);
  for (int cl = warp; cl < Cg; cl += nwarps) {
    int v0 = cl * spv - base, v1 = (cl + 1) * spv - base;
    if (v0 < 0) v0 = 0;
    if (v1 > nv) v1 = nv;
    float a = 0.f, b = 0.f;
    for (int v = v0 + lane; v < v1; v += 32) {
      a += vsum[v].x;
      b += vsum[v].y;
    }
    a = warp_sum(a);
    b = warp_sum(b);
    if (lane == 0) {
      prow[cbase + cl] = a;
      prow[C + cbase + cl] = b;
    }
  }
}

// One CTA per group, any alignment: scalar loads, the group read from L2 in
// every pass.
template <typename T>
__global__ void __launch_bounds__(256) gn_fwd_scalar(
    const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
    T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, int M, int S, int Cg,
    int G, float eps) {
  __shared__ float red[64];
  const int64_t grp = blockIdx.x;
  const int cbase = (int)(grp % G) * Cg;
  const T* xg = x + grp * M;
  pdl_trigger();
  pdl_wait();
  float s = 0.f;
  for (int j = threadIdx.x; j < M; j += blockDim.x) s += Traits<T>::to_f(xg[j]);
  const float mu = block_sum(s, red, 0) / (float)M;
  float q = 0.f;
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    const float d = Traits<T>::to_f(xg[j]) - mu;
    q = fmaf(d, d, q);
  }
  const float rs = rstd_of(block_sum(q, red, 1) / (float)M, eps);
  if (threadIdx.x == 0) {
    mean[grp] = mu;
    rstd[grp] = rs;
  }
  T* yg = y + grp * M;
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    const int c = cbase + j / S;
    const float b = beta ? Traits<T>::to_f(beta[c]) : 0.f;
    yg[j] = Traits<T>::from_f(fmaf((Traits<T>::to_f(xg[j]) - mu) * rs,
                                   Traits<T>::to_f(gamma[c]), b));
  }
}

template <typename T>
__global__ void __launch_bounds__(256) gn_bwd_scalar(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd, T* __restrict__ dx,
    float* __restrict__ partial, int M, int S, int Cg, int G, int C) {
  __shared__ float2 red[64];
  const int64_t grp = blockIdx.x;
  const int64_t n = grp / G;
  const int cbase = (int)(grp % G) * Cg;
  const T* xg = x + grp * M;
  const T* dg = dy + grp * M;
  pdl_trigger();
  pdl_wait();
  const float mu = mean[grp], rs = rstd[grp];
  float s1 = 0.f, s2 = 0.f;
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    const float gd = Traits<T>::to_f(dg[j]) * Traits<T>::to_f(gamma[cbase + j / S]);
    s1 += gd;
    s2 = fmaf(gd, Traits<T>::to_f(xg[j]) - mu, s2);
  }
  const float2 t = block_sum2(s1, s2, red, 0);
  const float c1 = t.x / (float)M, c2 = t.y * rs / (float)M;
  T* xo = dx + grp * M;
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    const float df = Traits<T>::to_f(dg[j]);
    const float xh = (Traits<T>::to_f(xg[j]) - mu) * rs;
    xo[j] = Traits<T>::from_f(
        fmaf(-xh, c2, df * Traits<T>::to_f(gamma[cbase + j / S]) - c1) * rs);
  }
  // per channel: one two-value CTA reduction each
  float* prow = partial + n * (int64_t)(2 * C);
  int parity = 1;
  for (int cl = 0; cl < Cg; ++cl) {
    float a = 0.f, b = 0.f;
    for (int j = threadIdx.x; j < S; j += blockDim.x) {
      const int64_t i = (int64_t)cl * S + j;
      const float df = Traits<T>::to_f(dg[i]);
      a = fmaf(df, (Traits<T>::to_f(xg[i]) - mu) * rs, a);
      b += df;
    }
    const float2 u = block_sum2(a, b, red, parity);
    parity ^= 1;
    if (threadIdx.x == 0) {
      prow[cbase + cl] = u.x;
      prow[C + cbase + cl] = u.y;
    }
  }
}

// Whether clusters of `csize` CTAs of `block` threads of `kern` can be
// resident on the current device (some sizes above 8 cannot), cached.
struct GnFit {
  const void* kern;
  int block, csize, device;
  bool ok;
};
std::mutex g_fit_mutex;
GnFit g_fit[128];
int g_fit_n = 0;

bool cluster_fits(const void* kern, int block, int csize) {
  if (csize <= 1) return true;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  {
    std::lock_guard<std::mutex> lock(g_fit_mutex);
    for (int i = 0; i < g_fit_n; ++i)
      if (g_fit[i].kern == kern && g_fit[i].block == block && g_fit[i].csize == csize &&
          g_fit[i].device == dev)
        return g_fit[i].ok;
  }
  bool ok = allow_cluster(kern, csize) == cudaSuccess;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)csize);
    cfg.blockDim = dim3((unsigned)block);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    ok = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0;
  }
  if (!ok) cudaGetLastError();  // a refused query leaves no error behind
  std::lock_guard<std::mutex> lock(g_fit_mutex);
  if (g_fit_n < 128) g_fit[g_fit_n++] = GnFit{kern, block, csize, dev, ok};
  return ok;
}

// Cluster size for a group of nvec vectors: the smallest power of two (at
// most 16) that divides nvec and leaves at most max_nv vectors a CTA, then
// doubled while the grid has fewer CTAs than SMs (small batches).  0 when
// none fits.
int pick_gn_cluster(int nvec, int max_nv, int64_t groups, int sms) {
  int c = 0;
  for (int k = 1; k <= kMaxCluster; k *= 2)
    if (nvec % k == 0 && nvec / k <= max_nv) {
      c = k;
      break;
    }
  if (c == 0) return 0;
  while (c < kMaxCluster && groups * c < sms && nvec % (2 * c) == 0 && nvec / (2 * c) >= 256)
    c *= 2;
  return c;
}

template <typename T>
cudaError_t gn_fwd_t(const GnArgs& a, cudaStream_t s) {
  constexpr int E = Traits<T>::kVec;
  const T* x = static_cast<const T*>(a.x);
  const T* g = static_cast<const T*>(a.gamma);
  const T* b = static_cast<const T*>(a.beta);
  T* y = static_cast<T*>(a.y);
  const int64_t groups = a.n * a.groups;
  const int Cg = a.channels / a.groups;
  const int M = Cg * a.spatial;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (a.vec_ok) {
    const int nvec = M / E;
    // halve the cluster while it cannot be resident, as long as a CTA
    // still holds its slice
    for (int csize = pick_gn_cluster(nvec, kGnMaxVec, groups, sm_count(dev));
         csize >= 1 && nvec / csize <= kGnMaxVec && groups * csize <= 0x7fffffff; csize /= 2) {
      const int nv = nvec / csize;
      const int vpt = gn_vpt(nv);
      const unsigned threads = (unsigned)(((nv + vpt - 1) / vpt + 31) / 32 * 32);
      auto kern = vpt == 1 ? gn_fwd_cluster<T, 1> : vpt == 2 ? gn_fwd_cluster<T, 2>
                : vpt == 4 ? gn_fwd_cluster<T, 4> : gn_fwd_cluster<T, 8>;
      if (!cluster_fits((const void*)kern, (int)threads, csize)) continue;
      return launch_clustered(kern, (unsigned)(groups * csize), threads, csize, s, x, g, b, y,
                              a.mean, a.rstd, M, a.spatial / E, Cg, a.groups, a.eps, csize);
    }
  }
  return launch_kernel(gn_fwd_scalar<T>, dim3((unsigned)groups), dim3(256), 0, s, 1, x, g, b, y,
                       a.mean, a.rstd, M, a.spatial, Cg, a.groups, a.eps);
}

template <typename T>
cudaError_t gn_bwd_t(const GnArgs& a, cudaStream_t s, int* launches) {
  constexpr int E = Traits<T>::kVec;
  const T* dy = static_cast<const T*>(a.dy);
  const T* x = static_cast<const T*>(a.x);
  const T* g = static_cast<const T*>(a.gamma);
  T* dx = static_cast<T*>(a.dx);
  const int64_t groups = a.n * a.groups;
  const int Cg = a.channels / a.groups;
  const int M = Cg * a.spatial;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int csize = 0;
  if (a.vec_ok) {
    const int nvec = M / E;
    for (int cs = pick_gn_cluster(nvec, kGnMaxVec, groups, sm_count(dev));
         cs >= 1 && nvec / cs <= kGnMaxVec && groups * cs <= 0x7fffffff; cs /= 2) {
      const int nv = nvec / cs;
      const int vpt = gn_vpt(nv);
      const unsigned threads = (unsigned)(((nv + vpt - 1) / vpt + 31) / 32 * 32);
      auto kern = vpt == 1 ? gn_bwd_cluster<T, 1> : vpt == 2 ? gn_bwd_cluster<T, 2>
                : vpt == 4 ? gn_bwd_cluster<T, 4> : gn_bwd_cluster<T, 8>;
      if (!cluster_fits((const void*)kern, (int)threads, cs)) continue;
      csize = cs;
      e = launch_clustered(kern, (unsigned)(groups * cs), threads, cs, s, dy, x, g, a.mean,
                           a.rstd, dx, a.partial, M, a.spatial / E, Cg, a.groups, a.channels,
                           cs);
      break;
    }
  }
  if (csize == 0) {
    csize = 1;
    e = launch_kernel(gn_bwd_scalar<T>, dim3((unsigned)groups), dim3(256), 0, s, 1, dy, x, g,
                      a.mean, a.rstd, dx, a.partial, M, a.spatial, Cg, a.groups, a.channels);
  }
  if (e != cudaSuccess) return e;
  *launches += 1;
  e = launch_column_sums(a.partial, (int)(a.n * csize), 2 * a.channels, a.dgamma, a.dbeta,
                         a.channels, s);
  if (e == cudaSuccess) *launches += 1;
  return e;
}

}  // namespace

cudaError_t launch_gn_fwd(int dtype, const GnArgs& a, cudaStream_t s) {
  switch (dtype) {
    case 0: return gn_fwd_t<float>(a, s);
    case 1: return gn_fwd_t<__nv_bfloat16>(a, s);
    default: return gn_fwd_t<__half>(a, s);
  }
}

cudaError_t launch_gn_bwd(int dtype, const GnArgs& a, cudaStream_t s, int* launches) {
  switch (dtype) {
    case 0: return gn_bwd_t<float>(a, s, launches);
    case 1: return gn_bwd_t<__nv_bfloat16>(a, s, launches);
    default: return gn_bwd_t<__half>(a, s, launches);
  }
}

}  // namespace rmsn
