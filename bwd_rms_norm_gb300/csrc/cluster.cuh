// Thread-block cluster helpers shared by the cluster kernels: the CTA's
// rank, the cluster barrier, stores into a peer CTA's shared memory
// (distributed shared memory) and fixed-order sums over a cluster.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace rmsn {

constexpr int kMaxCluster = 16;

__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Store `v` into the shared-memory word `local` of CTA `peer` of the cluster.
__device__ __forceinline__ void st_peer(float* local, uint32_t peer, float v) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(peer));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__device__ __forceinline__ void st_peer2(float2* local, uint32_t peer, float2 v) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(peer));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(v.x), "f"(v.y)
               : "memory");
}

// Sum of `v` over the cluster, the same value (and order) in every thread:
// CTA sum (block_sum), pushed to slot[rank] of every CTA, cluster barrier,
// slots added in rank order.  `slots` holds 2 x kMaxCluster floats; the
// parity alternates between calls (a slot is rewritten two calls later,
// after an intervening cluster barrier that every reader has passed).
__device__ __forceinline__ float cluster_sum(float v, float* red, float* slots, int parity,
                                             uint32_t rank, int csize) {
  const float cta = block_sum(v, red, parity);
  float* slot = slots + kMaxCluster * parity;
  if (threadIdx.x < (unsigned)csize) st_peer(slot + rank, threadIdx.x, cta);
  cluster_sync();
  float tot = 0.f;
  for (int q = 0; q < csize; ++q) tot += slot[q];
  return tot;
}

// The pair (a, b) summed over the cluster, same scheme; `slots` holds
// 2 x kMaxCluster float2.
__device__ __forceinline__ float2 cluster_sum2(float a, float b, float2* red, float2* slots,
                                               int parity, uint32_t rank, int csize) {
  const float2 cta = block_sum2(a, b, red, parity);
  float2* slot = slots + kMaxCluster * parity;
  if (threadIdx.x < (unsigned)csize) st_peer2(slot + rank, threadIdx.x, cta);
  cluster_sync();
  float2 tot = make_float2(0.f, 0.f);
  for (int q = 0; q < csize; ++q) {
    tot.x += slot[q].x;
    tot.y += slot[q].y;
  }
  return tot;
}

// Cluster sizes above 8 are not portable; allow them on the kernel first.
inline cudaError_t allow_cluster(const void* kern, int csize) {
  if (csize <= 8) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <typename K, typename... Args>
cudaError_t launch_clustered(K kern, unsigned grid, unsigned block, int csize, cudaStream_t s,
                             Args... args) {
  cudaError_t e = allow_cluster((const void*)kern, csize);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(block), 0, s, csize, args...);
}

}  // namespace rmsn
