// Wide-row forward and backward kernels for sm_103a: thread-block clusters.
//
// The widest rows (65536 fp32: 256 KB of x, twice that with dy) are too
// wide for one CTA to hold in registers and for the staged kernels' rings,
// even split over a cluster of 4 (the narrower wide rows take those).  Here
// a row is split
// over the C CTAs of a cluster (C = 2, 4, 8 or 16): CTA rank q owns columns
// [q*N/C, (q+1)*N/C), holds its slice in registers, reduces it (warp
// shuffles, then the CTA's warps in order), and pushes the CTA's partial sum
// into a slot of every CTA of the cluster through distributed shared memory
// (st.shared::cluster).  One cluster barrier later every CTA adds the C
// slots in rank order, so all of them hold the same row statistic, computed
// in the same order, and write their slice of the output.
//
//   fwd_cluster  one cluster per row (grid = rows x C CTAs).
//   bwd_cluster  persistent: cluster k owns a contiguous range of rows; each
//                thread keeps the fp32 gains and dw accumulators of its
//                columns in registers, prefetches the next row while the
//                current one is reduced, and the cluster writes one partial
//                dw row (each CTA its slice) at the end.
//
// Cluster barriers are hardware barriers that every thread of every CTA of
// the cluster reaches the same number of times (the control flow does not
// depend on the data), so they need no time limit.
#include <mutex>

#include "cluster.cuh"

namespace rmsn {
namespace {

template <typename T, int VPT>
__global__ void __launch_bounds__(512) fwd_cluster(
    const T* __restrict__ x, const T* __restrict__ gamma, T* __restrict__ y,
    float* __restrict__ rstd, int hidden, float eps, float off, int twice, int csize) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  __shared__ float slots[2 * kMaxCluster];
  const uint32_t rank = cta_rank();
  const int64_t row = blockIdx.x / csize;
  const int nv = hidden / E / csize;           // vectors of this CTA's slice
  const int64_t base = (int64_t)rank * nv;     // first vector of the slice
  const T* xr = x + row * hidden;
  T* yr = y + row * hidden;
  // every CTA of the cluster must be running before any writes into its
  // shared memory
  cluster_sync();
  pdl_trigger();
  pdl_wait();
  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    xv[k] = v < nv ? ld_stream(xr + (base + v) * E) : make_uint4(0, 0, 0, 0);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    float f[E];
    unpack<T>(xv[k], f);
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(f[e], f[e], ss);
  }
  ss = cluster_sum(ss, red, slots, 0, rank, csize);
  float rs = rstd_of(ss / (float)hidden, eps);
  if (isinf(ss))  // the fp32 sum of squares overflowed (see kOverflowScale)
    rs = rstd_rescaled(cluster_sum(scaled_sum_sq(xr + base * E, threadIdx.x, blockDim.x, nv * E),
                                   red, slots, 1, rank, csize),
                       hidden, eps);
  if (rank == 0 && threadIdx.x == 0) rstd[row] = rs;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      float f[E], g[E], o[E];
      unpack<T>(xv[k], f);
      unpack<T>(ld_shared_ro(gamma + (base + v) * E), g);
      if (twice) {
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = round_trip<T>(f[e] * rs) * (g[e] + off);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = (f[e] * rs) * (g[e] + off);
      }
      st_vec(yr + (base + v) * E, pack<T>(o));
    }
  }
}

template <typename T, int VPT>
__global__ void __launch_bounds__(512, 1) bwd_cluster(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ rstd, T* __restrict__ dx, float* __restrict__ partial,
    int64_t rows, int hidden, float off, int csize, int brows) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  __shared__ float slots[2 * kMaxCluster];
  pdl_trigger();
  pdl_wait();
  const uint32_t rank = cta_rank();
  const int64_t cid = blockIdx.x / csize;
  const int64_t nclusters = gridDim.x / csize;
  const RowBlocks blk = row_blocks(rows, brows, cid, nclusters);
  const int64_t r0 = blk.r0, r1 = blk.r0 + blk.n;
  const int nv = hidden / E / csize;
  const int64_t base = (int64_t)rank * nv;

  float ge[VPT][E], acc[VPT][E];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    const uint4 g4 = v < nv ? ld_shared_ro(gamma + (base + v) * E) : make_uint4(0, 0, 0, 0);
    unpack<T>(g4, ge[k]);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      ge[k][e] += off;
      acc[k][e] = 0.f;
    }
  }
  uint4 xc[VPT], dc[VPT], xn[VPT], dn[VPT];
  float rc = 0.f, rn = 0.f;
  auto load = [&](int64_t r, uint4 (&xb)[VPT], uint4 (&db)[VPT], float& rb) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      const bool in = v < nv;
      xb[k] = in ? ld_stream(x + r * hidden + (base + v) * E) : make_uint4(0, 0, 0, 0);
      db[k] = in ? ld_stream(dy + r * hidden + (base + v) * E) : make_uint4(0, 0, 0, 0);
    }
    rb = __ldg(rstd + r);
  };
  cluster_sync();  // every CTA of the cluster is running
  if (r0 < r1) load(r0, xc, dc, rc);
  int parity = 0;
  int64_t part = blk.b0;
  for (int64_t r = r0; r < r1; ++part) {
   for (const int64_t end = r0 + blk.block_end((int)(r - r0)); r < end; ++r) {
    if (r + 1 < r1) load(r + 1, xn, dn, rn);
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      float xf[E], df[E];
      unpack<T>(xc[k], xf);
      unpack<T>(dc[k], df);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float xh = xf[e] * rc;
        dot = fmaf(df[e] * ge[k][e], xh, dot);
        acc[k][e] = fmaf(df[e], xh, acc[k][e]);
      }
    }
    const float c = cluster_sum(dot, red, slots, parity, rank, csize) / (float)hidden;
    parity ^= 1;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        float xf[E], df[E], o[E];
        unpack<T>(xc[k], xf);
        unpack<T>(dc[k], df);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float xh = xf[e] * rc;
          o[e] = fmaf(-xh, c, df[e] * ge[k][e]) * rc;
        }
        st_vec(dx + r * hidden + (base + v) * E, pack<T>(o));
      }
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      xc[k] = xn[k];
      dc[k] = dn[k];
    }
    rc = rn;
   }
    flush_partial<VPT, E>(acc, partial, part, hidden, base * E, threadIdx.x, blockDim.x, nv);
  }
}

// Smallest cluster size (2, 4, 8, 16) that leaves each CTA at most `max_nv`
// vectors and divides the row's vectors evenly; 0 if none does.
int pick_cluster(int nvec, int max_nv) {
  for (int c = 2; c <= kMaxCluster; c *= 2)
    if (nvec % c == 0 && nvec / c <= max_nv) return c;
  return 0;
}

int pow2_ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

cudaLaunchConfig_t cluster_config(unsigned grid, unsigned block, int csize, cudaStream_t s,
                                  cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

struct ClusterOcc {
  const void* func;
  int block, csize, device, value;
};
std::mutex g_cocc_mutex;
ClusterOcc g_cocc[64];
int g_cocc_n = 0;

// Clusters of `csize` CTAs of `block` threads that can be resident at once
// on `device`, cached.
template <typename K>
cudaError_t max_active_clusters(K kern, int block, int csize, int device, int* out) {
  {
    std::lock_guard<std::mutex> lock(g_cocc_mutex);
    for (int i = 0; i < g_cocc_n; ++i)
      if (g_cocc[i].func == (const void*)kern && g_cocc[i].block == block &&
          g_cocc[i].csize == csize && g_cocc[i].device == device) {
        *out = g_cocc[i].value;
        return cudaSuccess;
      }
  }
  cudaError_t e = allow_cluster((const void*)kern, csize);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config((unsigned)csize, block, csize, 0, attr);
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) n = 1;
  std::lock_guard<std::mutex> lock(g_cocc_mutex);
  if (g_cocc_n < 64) g_cocc[g_cocc_n++] = ClusterOcc{(const void*)kern, block, csize, device, n};
  *out = n;
  return cudaSuccess;
}

template <typename T>
bool try_fwd_cluster_t(const FwdArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int E = Traits<T>::kVec;
  const int nvec = a.hidden / E;
  // up to 512 threads x 4 vectors per CTA
  const int csize = pick_cluster(nvec, 2048);
  if (csize == 0) return false;
  const int nv = nvec / csize;
  int vpt = pow2_ceil((nv + 511) / 512);
  if (vpt > 4) return false;
  const int threads = ((nv + vpt - 1) / vpt + 31) / 32 * 32;
  const int64_t grid = a.rows * csize;
  if (grid > 0x7fffffff) return false;
  const float off = a.offset ? 1.f : 0.f;
  const T* x = static_cast<const T*>(a.x);
  const T* g = static_cast<const T*>(a.gamma);
  T* y = static_cast<T*>(a.y);
  switch (vpt) {
    case 1: *err = launch_clustered(fwd_cluster<T, 1>, (unsigned)grid, threads, csize, s, x, g, y, a.rstd, a.hidden, a.eps, off, a.twice, csize); break;
    case 2: *err = launch_clustered(fwd_cluster<T, 2>, (unsigned)grid, threads, csize, s, x, g, y, a.rstd, a.hidden, a.eps, off, a.twice, csize); break;
    default: *err = launch_clustered(fwd_cluster<T, 4>, (unsigned)grid, threads, csize, s, x, g, y, a.rstd, a.hidden, a.eps, off, a.twice, csize); break;
  }
  return true;
}

template <typename T>
bool try_bwd_cluster_t(const BwdArgs& a, cudaStream_t s, cudaError_t* err, int64_t* nparts) {
  constexpr int E = Traits<T>::kVec;
  const int nvec = a.hidden / E;
  // up to 512 threads x 2 vectors per CTA
  const int csize = pick_cluster(nvec, 1024);
  if (csize == 0) return false;
  const int nv = nvec / csize;
  const int vpt = nv > 512 ? 2 : 1;
  const int threads = ((nv + vpt - 1) / vpt + 31) / 32 * 32;
  int dev = 0;
  if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return true;
  auto kern = vpt == 1 ? bwd_cluster<T, 1> : bwd_cluster<T, 2>;
  // a persistent grid: as many clusters as can be resident at once
  int active = 0;
  if ((*err = max_active_clusters(kern, threads, csize, dev, &active)) != cudaSuccess) return true;
  // the SM budget, in clusters
  const int budget = sm_count(dev) / csize;
  if (active > budget) active = budget > 0 ? budget : 1;
  const BlockPlan bp = plan_blocks(a.rows, a.block_rows, unit_cap(a, active));
  *nparts = bp.nblocks;
  *err = launch_clustered(kern, (unsigned)(bp.units * csize), threads, csize, s,
                          static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                          static_cast<const T*>(a.gamma), a.rstd, static_cast<T*>(a.dx),
                          a.partial, a.rows, a.hidden, a.offset ? 1.f : 0.f, csize, bp.brows);
  return true;
}

}  // namespace

bool try_launch_fwd_cluster(int dtype, const FwdArgs& a, cudaStream_t s, cudaError_t* err) {
  if (!a.vec_ok) return false;
  switch (dtype) {
    case 0: return try_fwd_cluster_t<float>(a, s, err);
    case 1: return try_fwd_cluster_t<__nv_bfloat16>(a, s, err);
    default: return try_fwd_cluster_t<__half>(a, s, err);
  }
}

bool try_launch_bwd_cluster(int dtype, const BwdArgs& a, cudaStream_t s, cudaError_t* err,
                            int64_t* nparts) {
  if (!a.vec_ok) return false;
  switch (dtype) {
    case 0: return try_bwd_cluster_t<float>(a, s, err, nparts);
    case 1: return try_bwd_cluster_t<__nv_bfloat16>(a, s, err, nparts);
    default: return try_bwd_cluster_t<__half>(a, s, err, nparts);
  }
}

}  // namespace rmsn
