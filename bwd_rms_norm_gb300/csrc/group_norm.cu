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
#include "mbar.cuh"

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
  // Per-channel sums over this slice, in a fixed order.  The slice touches
  // channels c_lo..c_hi of the group.  With at least as many channels as
  // warps, warp w sums channels c_lo + w, c_lo + w + nwarps, ... (lanes
  // striding over the channel's vectors, then a butterfly).  With fewer,
  // each channel's vectors are split into wpc equal runs, one warp each,
  // whose two sums meet in shared memory and are added in run order.
  // Channels of the group this slice does not touch get 0, so that every
  // column of the partial row is written.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  float* prow = partial + (n * csize + rank) * (int64_t)(2 * C);
  const int c_lo = base / spv, c_hi = (base + nv - 1) / spv;
  const int nch = c_hi - c_lo + 1;
  for (int cl = threadIdx.x; cl < Cg; cl += blockDim.x) {
    if (cl < c_lo || cl > c_hi) {
      prow[cbase + cl] = 0.f;
      prow[C + cbase + cl] = 0.f;
    }
  }
  auto run_sum = [&](int v0, int v1) {
    float a = 0.f, b = 0.f;
    for (int v = v0 + lane; v < v1; v += 32) {
      a += vsum[v].x;
      b += vsum[v].y;
    }
    return make_float2(warp_sum(a), warp_sum(b));
  };
  auto range_of = [&](int cl, int* v0, int* v1) {
    *v0 = cl * spv - base;
    *v1 = (cl + 1) * spv - base;
    if (*v0 < 0) *v0 = 0;
    if (*v1 > nv) *v1 = nv;
  };
  if (nch >= nwarps) {
    for (int cl = c_lo + warp; cl <= c_hi; cl += nwarps) {
      int v0, v1;
      range_of(cl, &v0, &v1);
      const float2 t2 = run_sum(v0, v1);
      if (lane == 0) {
        prow[cbase + cl] = t2.x;
        prow[C + cbase + cl] = t2.y;
      }
    }
  } else {
    const int wpc = nwarps / nch;  // warps per channel
    __shared__ float2 wsum[32];
    if (warp < nch * wpc) {
      const int cl = c_lo + warp / wpc, part = warp % wpc;
      int v0, v1;
      range_of(cl, &v0, &v1);
      const int len = v1 - v0;
      const int a0 = v0 + (int)((int64_t)len * part / wpc);
      const int a1 = v0 + (int)((int64_t)len * (part + 1) / wpc);
      const float2 t2 = run_sum(a0, a1);
      if (lane == 0) wsum[warp] = t2;
    }
    __syncthreads();
    if (threadIdx.x < nch) {
      float a = 0.f, b = 0.f;
      for (int q = 0; q < wpc; ++q) {
        a += wsum[threadIdx.x * wpc + q].x;
        b += wsum[threadIdx.x * wpc + q].y;
      }
      prow[cbase + c_lo + threadIdx.x] = a;
      prow[C + cbase + c_lo + threadIdx.x] = b;
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

// ---------------------------------------------------------------------------
// Persistent, TMA-fed, warp-specialised pipeline.  One cluster of csize
// CTAs (one CTA per SM) walks a contiguous range of groups; CTA rank q owns
// slice q of every group (nv 16-byte vectors).  Three roles meet at
// per-stage mbarriers, as in the RMSNorm staged kernels:
//
//   producer (warp 0, one thread)  streams the slices of the coming groups
//       into a ring of shared-memory stages with 1D bulk copies;   -> full[s]
//   reducers (three teams of kGnTeamWarps warps)  team d takes the CTA's
//       groups d, d + 3, ...: its warps split the slice sums (combined at a
//       team named barrier), then the team's first warp exchanges one pair
//       per group with the cluster
//       through distributed shared memory (the reducer stores its pair into
//       every peer's slot for that reducer and arrives on the peer's
//       exchange mbarrier), then the group's statistics;        -> red[s]
//   appliers (the other warps)  walk every group in order and write the
//       outputs of their vectors of the slice.
//
// The forward exchanges (slice mean, slice centred sum of squares) and
// combines them in rank order (Chan's formula for slices of equal length);
// the backward exchanges (sum g, sum g * (x - mean)).  A reducer waits for
// its peers while the appliers work on earlier groups and the producer's
// copies of later groups are in flight.  The stage count is a multiple of
// the reducer count, so that every mbarrier waiter sees every phase of the
// barriers it waits on; each reducer's exchange slots are double-buffered
// (a peer cannot start the group after next before this CTA has read the
// current one, since that needs this CTA's pair for the next group).
// Measured on GB300 against a variant in which all compute warps share
// every group with one group of lookahead: this split is 25-35% faster.
//
// Every wait is bounded (about one second); a wait that runs out counts in
// g_gn_wait_timeouts and aborts the CTA; decisions are taken per warp (and,
// among the appliers of the backward, which share a named barrier, with a
// predicate-reducing barrier), and every CTA ends with a cluster barrier,
// so that no CTA exits while a peer may still store into its shared memory.
// ---------------------------------------------------------------------------
__device__ unsigned int g_gn_wait_timeouts;

constexpr int kGnStages = 15;
constexpr int kGnReducers = 3;      // reducer teams (each takes every third group)
constexpr int kGnTeamMax = 4;       // warps a team
constexpr int kGnThreadsMax = 544;  // 17 warps: producer, 3 teams, appliers
constexpr int kGnSmem = 220 * 1024;  // dynamic shared memory a CTA
constexpr unsigned kFull = 0xffffffffu;

struct GnPipe {
  uint64_t full[kGnStages];    // the stage's bulk copies landed
  uint64_t red[kGnStages];     // the stage's group statistics are in stat[]
  uint64_t empty[kGnStages];   // its reducer and every applier warp are done
  float2 stat[kGnStages];      // forward (mean, rstd); backward (c1, c2)
  uint64_t xbar[kGnReducers][2];            // a reducer's pairs arrived
  float2 xch[kGnReducers][2][kMaxCluster];  // ... by sender rank
  float2 tred[kGnReducers][2][kGnTeamMax];  // team-warp partial sums
  float2 wsum[32];             // applier-warp channel sums (backward)
  int abort;
};

// Team barrier (named barrier 2 + team over its 32 * tw threads) that also
// tells whether `ok` held in every warp of the team.
__device__ __forceinline__ bool team_all(bool ok, int team, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(2 + team), "r"(nthreads)
      : "memory");
  return r != 0;
}

// The pair (a, b) summed over the warps of a team (each warp passes its own
// warp total), the same value and order in every lane; `par` alternates.
__device__ __forceinline__ float2 team_sum2(GnPipe& pp, float2 mine, int team, int tw, int ntw,
                                            int& par, int lane) {
  float2* slot = pp.tred[team][par];
  par ^= 1;
  if (lane == 0) slot[tw] = mine;
  asm volatile("bar.sync %0, %1;" ::"r"(2 + team), "r"(32 * ntw) : "memory");
  float2 t = make_float2(0.f, 0.f);
  for (int w = 0; w < ntw; ++w) {
    t.x += slot[w].x;
    t.y += slot[w].y;
  }
  return t;
}

__device__ bool gn_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return wait_phase_counted(bar, parity, abort, &g_gn_wait_timeouts);
}

__device__ void gn_drain(uint64_t* bar, uint32_t parity) {
  drain_phase_counted(bar, parity, &g_gn_wait_timeouts);
}

// Cluster-scope waits, counted in this file's timeout counter.
__device__ bool gn_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return wait_cluster_counted(bar, parity, abort, &g_gn_wait_timeouts);
}

// Named barrier 1 over the nthreads appliers; true when `ok` holds in every
// one of them.
__device__ __forceinline__ bool appliers_all(bool ok, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void appliers_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

__device__ __forceinline__ void gn_pipe_init(GnPipe& pp, int stages, int applier_warps,
                                             int csize) {
  const int t = threadIdx.x;
  if (t == 0) pp.abort = 0;
  if (t < stages) {
    mbar_init(&pp.full[t], 1);
    mbar_init(&pp.red[t], 1);
    mbar_init(&pp.empty[t], applier_warps + 1);
  }
  if (t < 2 * kGnReducers) mbar_init(&pp.xbar[t / 2][t % 2], csize);
  fence_mbar_init();
}

// The producer: NSRC slices of each of the CTA's `count` groups into the ring.
template <int NSRC>
__device__ void gn_produce(GnPipe& pp, unsigned char* ring, int stages, uint32_t sb,
                           const unsigned char* const (&src)[NSRC], int64_t g0, int count,
                           int64_t group_bytes, int64_t slice_off, volatile int* abort) {
  int stage = 0;
  uint32_t ph = 0;
  int i = 0;
  for (; i < count; ++i) {
    if (i >= stages && !gn_wait(&pp.empty[stage], ph ^ 1u, abort)) break;
    unsigned char* dst = ring + (size_t)stage * NSRC * sb;
    mbar_arrive_expect_tx(&pp.full[stage], NSRC * sb);
    const int64_t off = (g0 + i) * group_bytes + slice_off;
#pragma unroll
    for (int t = 0; t < NSRC; ++t) bulk_load(dst + t * sb, src[t] + off, sb, &pp.full[stage]);
    if (++stage == stages) {
      stage = 0;
      ph ^= 1u;
    }
  }
  // every copy issued must land before the CTA may exit: the latest
  // min(i, stages) issues are the last use of each stage
  const int outstanding = i < stages ? i : stages;
  for (int q = 0; q < outstanding; ++q) {
    if (stage == 0) {
      stage = stages - 1;
      ph ^= 1u;
    } else {
      --stage;
    }
    gn_drain(&pp.full[stage], ph);
  }
}

// A reducer's exchange of its pair with the cluster; false on abort.  On
// return every lane can read the pairs in pp.xch[d][par] by sender rank.
__device__ __forceinline__ bool exchange(GnPipe& pp, int d, int par, uint32_t xph,
                                         float2 mine, uint32_t rank, int csize, int lane,
                                         volatile int* abort) {
  if (lane < csize) {
    st_peer2(&pp.xch[d][par][rank], (uint32_t)lane, mine);
    mbar_arrive_peer(&pp.xbar[d][par], (uint32_t)lane);
  }
  return __all_sync(kFull, gn_wait_cluster(&pp.xbar[d][par], xph, abort));
}

// Channel of slice vectors v0, v0 + step, v0 + 2 step, ... without a
// division per vector: q = (vbase + v) / spv and its remainder, advanced by
// the quotient and remainder of the step.
struct ChanWalk {
  int q, r, dq, dr, spv;
  __device__ __forceinline__ ChanWalk(int first, int step, int spv_) : spv(spv_) {
    q = first / spv;
    r = first - q * spv;
    dq = step / spv;
    dr = step - dq * spv;
  }
  __device__ __forceinline__ void next() {
    q += dq;
    r += dr;
    if (r >= spv) {
      r -= spv;
      ++q;
    }
  }
};

template <int E>
__device__ __forceinline__ float lane_total(float (&p)[E]) {
#pragma unroll
  for (int w = E / 2; w >= 1; w /= 2)
#pragma unroll
    for (int e = 0; e < w; ++e) p[e] += p[e + w];
  return warp_sum(p[0]);
}

template <typename T>
__global__ void __launch_bounds__(kGnThreadsMax, 1) gn_fwd_pipe(
    const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
    T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, int64_t ngroups,
    int M, int spv, int Cg, int G, float eps, int csize, int stages, int nv, int ntw) {
  constexpr int E = Traits<T>::kVec;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ GnPipe pp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int napp = blockDim.x - 32 * (1 + kGnReducers * ntw);
  const uint32_t rank = csize > 1 ? cta_rank() : 0u;
  const int64_t cid = blockIdx.x / csize, ncl = gridDim.x / csize;
  const int64_t g0 = cid * ngroups / ncl;
  const int count = (int)((cid + 1) * ngroups / ncl - g0);
  const uint32_t sb = (uint32_t)nv * 16u;
  gn_pipe_init(pp, stages, napp / 32, csize);
  __syncthreads();
  if (csize > 1) cluster_sync();  // peers' barriers are initialised
  pdl_trigger();
  pdl_wait();
  volatile int* abort = &pp.abort;
  const int vbase = (int)rank * nv;  // first vector of this CTA's slice
  if (warp == 0) {
    if (lane == 0) {
      const unsigned char* const src[1] = {reinterpret_cast<const unsigned char*>(x)};
      gn_produce<1>(pp, ring, stages, sb, src, g0, count, (int64_t)M * sizeof(T),
                    (int64_t)vbase * 16, abort);
    }
  } else if (warp <= kGnReducers * ntw) {
    // reducer team d of ntw warps: warp tw takes vectors tw*32 + lane,
    // then every 32*ntw-th; warp 0 of the team exchanges and publishes
    const int d = (warp - 1) / ntw, tw = (warp - 1) % ntw;
    const int first = tw * 32 + lane, step = 32 * ntw;
    const float len = (float)(nv * E);
    int stage = d, par = 0, tpar = 0;
    uint32_t ph = 0, xph0 = 0, xph1 = 0;
    bool prev_ok = true;  // warp 0's last exchange
    for (int i = d; i < count; i += kGnReducers) {
      const int64_t grp = g0 + i;
      const bool ok = __all_sync(kFull, gn_wait(&pp.full[stage], ph, abort)) && prev_ok;
      if (!team_all(ok, d, 32 * ntw)) break;
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)stage * sb);
      float part[E];
#pragma unroll
      for (int e = 0; e < E; ++e) part[e] = 0.f;
#pragma unroll 4
      for (int v = first; v < nv; v += step) {
        float f[E];
        unpack<T>(st[v], f);
#pragma unroll
        for (int e = 0; e < E; ++e) part[e] += f[e];
      }
      const float ms =
          team_sum2(pp, make_float2(lane_total<E>(part), 0.f), d, tw, ntw, tpar, lane).x / len;
#pragma unroll
      for (int e = 0; e < E; ++e) part[e] = 0.f;
#pragma unroll 4
      for (int v = first; v < nv; v += step) {
        float f[E];
        unpack<T>(st[v], f);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float c = f[e] - ms;
          part[e] = fmaf(c, c, part[e]);
        }
      }
      const float Q =
          team_sum2(pp, make_float2(lane_total<E>(part), 0.f), d, tw, ntw, tpar, lane).x;
      if (tw == 0) {
        float mu = ms, m2 = Q;
        if (csize > 1) {
          prev_ok = exchange(pp, d, par, par ? xph1 : xph0, make_float2(ms, Q), rank, csize,
                             lane, abort);
          if (prev_ok) {
            if (par) xph1 ^= 1u; else xph0 ^= 1u;
            float sm = 0.f;
            for (int r = 0; r < csize; ++r) sm += pp.xch[d][par][r].x;
            mu = sm / (float)csize;
            m2 = 0.f;
            for (int r = 0; r < csize; ++r) {
              const float c = pp.xch[d][par][r].x - mu;
              m2 += fmaf(len * c, c, pp.xch[d][par][r].y);
            }
            par ^= 1;
          }
        }
        if (prev_ok && lane == 0) {
          const float rs = rstd_of(m2 / (float)M, eps);
          pp.stat[stage] = make_float2(mu, rs);
          if (rank == 0) {
            mean[grp] = mu;
            rstd[grp] = rs;
          }
          mbar_arrive(&pp.red[stage]);
          mbar_arrive(&pp.empty[stage]);
        }
      }
      stage += kGnReducers;
      if (stage >= stages) {
        stage -= stages;
        ph ^= 1u;
      }
    }
  } else {
    const int a = threadIdx.x - 32 * (1 + kGnReducers * ntw);
    int stage = 0;
    uint32_t ph = 0;
    for (int i = 0; i < count; ++i) {
      const int64_t grp = g0 + i;
      bool ok = gn_wait(&pp.red[stage], ph, abort);
      ok = ok && gn_wait(&pp.full[stage], ph, abort);
      if (!__all_sync(kFull, ok)) break;
      const float2 mr = pp.stat[stage];
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)stage * sb);
      const int cbase = (int)(grp % G) * Cg;
      T* yg = y + grp * M;
      ChanWalk cw(vbase + a, napp, spv);  // a vector lies in one channel
      for (int v = a; v < nv; v += napp, cw.next()) {
        const int c = cbase + cw.q;
        const float w = Traits<T>::to_f(gamma[c]);
        const float b = beta ? Traits<T>::to_f(beta[c]) : 0.f;
        float f[E], o[E];
        unpack<T>(st[v], f);
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = fmaf((f[e] - mr.x) * mr.y, w, b);
        st_vec(yg + (int64_t)(vbase + v) * E, pack<T>(o));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&pp.empty[stage]);
      if (++stage == stages) {
        stage = 0;
        ph ^= 1u;
      }
    }
  }
  __syncwarp();
  if (csize > 1) cluster_sync();  // no peer stores into this CTA after it exits
}

template <typename T>
__global__ void __launch_bounds__(kGnThreadsMax, 1) gn_bwd_pipe(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd, T* __restrict__ dx,
    float* __restrict__ partial, int64_t ngroups, int M, int spv, int Cg, int G, int C,
    int csize, int stages, int nv, int ntw) {
  constexpr int E = Traits<T>::kVec;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ GnPipe pp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int napp = blockDim.x - 32 * (1 + kGnReducers * ntw);
  const uint32_t rank = csize > 1 ? cta_rank() : 0u;
  const int64_t cid = blockIdx.x / csize, ncl = gridDim.x / csize;
  const int64_t g0 = cid * ngroups / ncl;
  const int count = (int)((cid + 1) * ngroups / ncl - g0);
  const uint32_t sb = (uint32_t)nv * 16u;
  float2* vsum = reinterpret_cast<float2*>(ring + (size_t)stages * 2 * sb);
  gn_pipe_init(pp, stages, napp / 32, csize);
  __syncthreads();
  if (csize > 1) cluster_sync();
  pdl_trigger();
  pdl_wait();
  volatile int* abort = &pp.abort;
  const int vbase = (int)rank * nv;
  if (warp == 0) {
    if (lane == 0) {
      const unsigned char* const src[2] = {reinterpret_cast<const unsigned char*>(x),
                                           reinterpret_cast<const unsigned char*>(dy)};
      gn_produce<2>(pp, ring, stages, sb, src, g0, count, (int64_t)M * sizeof(T),
                    (int64_t)vbase * 16, abort);
    }
  } else if (warp <= kGnReducers * ntw) {
    const int d = (warp - 1) / ntw, tw = (warp - 1) % ntw;
    const int first = tw * 32 + lane, step = 32 * ntw;
    int stage = d, par = 0, tpar = 0;
    uint32_t ph = 0, xph0 = 0, xph1 = 0;
    bool prev_ok = true;
    for (int i = d; i < count; i += kGnReducers) {
      const int64_t grp = g0 + i;
      const float mu = __ldg(mean + grp), rs = __ldg(rstd + grp);
      const int cbase = (int)(grp % G) * Cg;
      const bool ok = __all_sync(kFull, gn_wait(&pp.full[stage], ph, abort)) && prev_ok;
      if (!team_all(ok, d, 32 * ntw)) break;
      const uint4* sx = reinterpret_cast<const uint4*>(ring + (size_t)stage * 2 * sb);
      const uint4* sd = sx + nv;
      float p1[E], p2[E];
#pragma unroll
      for (int e = 0; e < E; ++e) p1[e] = p2[e] = 0.f;
      ChanWalk cw(vbase + first, step, spv);
#pragma unroll 2
      for (int v = first; v < nv; v += step, cw.next()) {
        const float w = Traits<T>::to_f(gamma[cbase + cw.q]);
        float xf[E], df[E];
        unpack<T>(sx[v], xf);
        unpack<T>(sd[v], df);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float gd = df[e] * w;
          p1[e] += gd;
          p2[e] = fmaf(gd, xf[e] - mu, p2[e]);
        }
      }
      float2 t = team_sum2(pp, make_float2(lane_total<E>(p1), lane_total<E>(p2)), d, tw, ntw,
                           tpar, lane);
      if (tw == 0) {
        if (csize > 1) {
          prev_ok = exchange(pp, d, par, par ? xph1 : xph0, t, rank, csize, lane, abort);
          if (prev_ok) {
            if (par) xph1 ^= 1u; else xph0 ^= 1u;
            t = make_float2(0.f, 0.f);
            for (int r = 0; r < csize; ++r) {
              t.x += pp.xch[d][par][r].x;
              t.y += pp.xch[d][par][r].y;
            }
            par ^= 1;
          }
        }
        if (prev_ok && lane == 0) {
          pp.stat[stage] = make_float2(t.x / (float)M, t.y * rs / (float)M);
          mbar_arrive(&pp.red[stage]);
          mbar_arrive(&pp.empty[stage]);
        }
      }
      stage += kGnReducers;
      if (stage >= stages) {
        stage -= stages;
        ph ^= 1u;
      }
    }
  } else {
    const int a = threadIdx.x - 32 * (1 + kGnReducers * ntw);
    const int cwi = a >> 5, ncw = napp >> 5;
    const int c_lo = vbase / spv, c_hi = (vbase + nv - 1) / spv;
    const int nch = c_hi - c_lo + 1;
    int stage = 0;
    uint32_t ph = 0;
    for (int i = 0; i < count; ++i) {
      const int64_t grp = g0 + i;
      const float mu = __ldg(mean + grp), rs = __ldg(rstd + grp);
      const int cbase = (int)(grp % G) * Cg;
      bool ok = gn_wait(&pp.red[stage], ph, abort);
      ok = ok && gn_wait(&pp.full[stage], ph, abort);
      if (!appliers_all(ok, napp)) break;
      const float2 cc = pp.stat[stage];
      const uint4* sx = reinterpret_cast<const uint4*>(ring + (size_t)stage * 2 * sb);
      const uint4* sd = sx + nv;
      T* xo = dx + grp * M;
      ChanWalk chw(vbase + a, napp, spv);
      for (int v = a; v < nv; v += napp, chw.next()) {
        const float w = Traits<T>::to_f(gamma[cbase + chw.q]);
        float xf[E], df[E], o[E];
        unpack<T>(sx[v], xf);
        unpack<T>(sd[v], df);
        float pg = 0.f, pb = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float xh = (xf[e] - mu) * rs;
          o[e] = fmaf(-xh, cc.y, df[e] * w - cc.x) * rs;
          pg = fmaf(df[e], xh, pg);
          pb += df[e];
        }
        st_vec(xo + (int64_t)(vbase + v) * E, pack<T>(o));
        vsum[v] = make_float2(pg, pb);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&pp.empty[stage]);  // the stage is no longer read
      if (++stage == stages) {
        stage = 0;
        ph ^= 1u;
      }
      appliers_sync(napp);  // vsum complete
      // Per-channel sums of this slice in a fixed order (as in
      // gn_bwd_cluster); channels of the group it does not touch get 0.
      float* prow = partial + ((grp / G) * csize + rank) * (int64_t)(2 * C);
      for (int cl = a; cl < Cg; cl += napp) {
        if (cl < c_lo || cl > c_hi) {
          prow[cbase + cl] = 0.f;
          prow[C + cbase + cl] = 0.f;
        }
      }
      if (nch >= ncw) {
        for (int cl = c_lo + cwi; cl <= c_hi; cl += ncw) {
          int v0 = cl * spv - vbase, v1 = (cl + 1) * spv - vbase;
          if (v0 < 0) v0 = 0;
          if (v1 > nv) v1 = nv;
          float s1 = 0.f, s2 = 0.f;
          for (int v = v0 + lane; v < v1; v += 32) {
            s1 += vsum[v].x;
            s2 += vsum[v].y;
          }
          s1 = warp_sum(s1);
          s2 = warp_sum(s2);
          if (lane == 0) {
            prow[cbase + cl] = s1;
            prow[C + cbase + cl] = s2;
          }
        }
      } else {
        const int wpc = ncw / nch;
        if (cwi < nch * wpc) {
          const int cl = c_lo + cwi / wpc, part = cwi % wpc;
          int v0 = cl * spv - vbase, v1 = (cl + 1) * spv - vbase;
          if (v0 < 0) v0 = 0;
          if (v1 > nv) v1 = nv;
          const int len = v1 - v0;
          const int a0 = v0 + (int)((int64_t)len * part / wpc);
          const int a1 = v0 + (int)((int64_t)len * (part + 1) / wpc);
          float s1 = 0.f, s2 = 0.f;
          for (int v = a0 + lane; v < a1; v += 32) {
            s1 += vsum[v].x;
            s2 += vsum[v].y;
          }
          s1 = warp_sum(s1);
          s2 = warp_sum(s2);
          if (lane == 0) pp.wsum[cwi] = make_float2(s1, s2);
        }
        appliers_sync(napp);
        if (a < nch) {
          float s1 = 0.f, s2 = 0.f;
          for (int q = 0; q < wpc; ++q) {
            s1 += pp.wsum[a * wpc + q].x;
            s2 += pp.wsum[a * wpc + q].y;
          }
          prow[cbase + c_lo + a] = s1;
          prow[C + cbase + c_lo + a] = s2;
        }
      }
      appliers_sync(napp);  // vsum and wsum are free for the next group
    }
  }
  __syncwarp();
  if (csize > 1) cluster_sync();
}

// Pipeline shape: the smallest cluster (1..16 CTAs) whose slices leave at
// least min_stages ring stages (a multiple of the reducer count) in kGnSmem
// (the backward also keeps a float2 per slice vector); false when none
// does.
struct PipeShape {
  int csize, stages, nv, threads;
  size_t smem;
  int ntw;  // warps a reducer team
};

// Warps a reducer team (measured on GB300: 2 beat 1, 3 and 4).
constexpr int kGnTeamWarps = 2;

bool pick_pipe_min(int nvec, bool bwd, int min_stages, PipeShape* ps) {
  for (int k = 1; k <= kMaxCluster; k *= 2) {
    if (nvec % k) continue;
    const int nv = nvec / k;
    const size_t sb = (size_t)nv * 16;
    const size_t per = bwd ? 2 * sb : sb;
    const size_t extra = bwd ? (size_t)nv * sizeof(float2) : 0;
    if (extra + (size_t)min_stages * per > (size_t)kGnSmem) continue;
    int st = (int)(((size_t)kGnSmem - extra) / per);
    if (st > kGnStages) st = kGnStages;
    st -= st % kGnReducers;
    const int ntw = kGnTeamWarps;
    int apps = (nv + 31) / 32;
    const int max_apps = kGnThreadsMax / 32 - 1 - kGnReducers * ntw;
    if (apps > max_apps) apps = max_apps;
    *ps = PipeShape{k, st, nv, 32 * (1 + kGnReducers * ntw + apps), (size_t)st * per + extra, ntw};
    return true;
  }
  return false;
}

// The smallest cluster with three stages: measured on GB300, larger
// clusters with deeper rings are slower (fewer resident clusters, costlier
// exchanges), e.g. the (16, 512, 64, 64) backward takes 101 us with six
// stages in clusters of 8 against 63 us with three in clusters of 4.
bool pick_pipe(int nvec, bool bwd, PipeShape* ps) { return pick_pipe_min(nvec, bwd, 3, ps); }

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

std::mutex g_gn_attr_mutex;
const void* g_gn_attr_done[64];
int g_gn_attr_device[64];
int g_gn_attr_n = 0;

// Clusters of the pipeline kernel that can be resident at once (0: none).
int pipe_clusters(const void* kern, const PipeShape& ps) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(g_gn_attr_mutex);
    bool done = false;
    for (int i = 0; i < g_gn_attr_n; ++i)
      done |= g_gn_attr_done[i] == kern && g_gn_attr_device[i] == dev;
    if (!done) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGnSmem) !=
          cudaSuccess) {
        cudaGetLastError();
        return 0;
      }
      if (g_gn_attr_n < 64) {
        g_gn_attr_done[g_gn_attr_n] = kern;
        g_gn_attr_device[g_gn_attr_n++] = dev;
      }
    }
  }
  if (ps.csize == 1) return sm_count(dev) * max_blocks_per_sm(kern, ps.threads, ps.smem);
  if (allow_cluster(kern, ps.csize) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ps.csize);
  cfg.blockDim = dim3((unsigned)ps.threads);
  cfg.dynamicSmemBytes = ps.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ps.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Slices of at most 2048 vectors where a cluster of 16 allows it (about 64
// registers a thread: two CTAs of 512 threads per SM, so that one CTA's
// loads overlap another's reductions and stores), else up to 4096.
int pick_gn_size(int nvec, int64_t groups, int sms) {
  const int c = pick_gn_cluster(nvec, 2048, groups, sms);
  return c ? c : pick_gn_cluster(nvec, kGnMaxVec, groups, sms);
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
    PipeShape ps;
    if (pick_pipe(nvec, false, &ps)) {
      auto kern = gn_fwd_pipe<T>;
      const int64_t active = pipe_clusters((const void*)kern, ps);
      if (active > 0) {
        const int64_t ncl = active < groups ? active : groups;
        return launch_kernel(kern, dim3((unsigned)(ncl * ps.csize)), dim3(ps.threads), ps.smem,
                             s, ps.csize, x, g, b, y, a.mean, a.rstd, groups, M,
                             a.spatial / E, Cg, a.groups, a.eps, ps.csize, ps.stages, ps.nv,
                             ps.ntw);
      }
    }
    // halve the cluster while it cannot be resident, as long as a CTA
    // still holds its slice
    for (int csize = pick_gn_size(nvec, groups, sm_count(dev));
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
  PipeShape ps;
  if (a.vec_ok && pick_pipe(M / E, true, &ps)) {
    auto kern = gn_bwd_pipe<T>;
    const int64_t active = pipe_clusters((const void*)kern, ps);
    if (active > 0) {
      const int64_t ncl = active < groups ? active : groups;
      csize = ps.csize;
      e = launch_kernel(kern, dim3((unsigned)(ncl * ps.csize)), dim3(ps.threads), ps.smem, s,
                        ps.csize, dy, x, g, a.mean, a.rstd, dx, a.partial, groups, M,
                        a.spatial / E, Cg, a.groups, a.channels, ps.csize, ps.stages, ps.nv,
                        ps.ntw);
    }
  }
  if (csize == 0 && a.vec_ok) {
    const int nvec = M / E;
    for (int cs = pick_gn_size(nvec, groups, sm_count(dev));
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

cudaError_t read_gn_wait_timeouts(unsigned int* out) {
  return cudaMemcpyFromSymbol(out, g_gn_wait_timeouts, sizeof(unsigned int));
}

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
