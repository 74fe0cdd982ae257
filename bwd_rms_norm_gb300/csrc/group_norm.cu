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
// it is split over a thread-block cluster of up to 16 CTAs whose group sums
// go through distributed shared memory (cluster.cuh).  The forward holds a
// CTA's slice in registers (gn_fwd_cluster) or streams it through a
// shared-memory ring (gn_fwd_pipe), reading every element once.  The
// backward (gn_bwd_l2) reads x and dy twice: from HBM through a ring for
// its sums, then from L2 for dx.  Its per-channel sums are reduced inside
// the CTA in a fixed order (per-vector sums in shared memory, warps per
// channel) and written as fp32 partial rows [n * csize, 2C] (dW columns,
// then dB), which the column-sum kernel of bwd.cu reduces in a fixed order:
// the result is deterministic.  Groups that are not 16-byte aligned, or too
// long for these kernels, run scalar kernels (one CTA per group).
#include <mutex>

#include "cluster.cuh"
#include "mbar.cuh"

namespace rmsn {
namespace {

// Most 16-byte vectors one CTA of the register forward holds: 8 a thread at
// 512 threads.  Cluster CTAs stay at 512 threads so that 16 of them fit one
// GPC.
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
// Persistent, TMA-fed, warp-specialised forward.  One cluster of csize
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
// A reducer exchanges (slice mean, slice centred sum of squares) and
// combines them in rank order (Chan's formula for slices of equal length).
// It waits for
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
// g_gn_wait_timeouts and aborts the CTA; decisions are taken per warp, and
// every CTA ends with a cluster barrier, so that no CTA exits while a peer
// may still store into its shared memory.
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
  float2 stat[kGnStages];      // the group's (mean, rstd)
  uint64_t xbar[kGnReducers][2];            // a reducer's pairs arrived
  float2 xch[kGnReducers][2][kMaxCluster];  // ... by sender rank
  float2 tred[kGnReducers][2][kGnTeamMax];  // team-warp partial sums
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
  if (threadIdx.x == 0)  // the first slices into L2 (prefetch_l2)
    for (int i = 0; i < count && i < 2; ++i)
      prefetch_l2(x + (g0 + i) * M + (int64_t)rank * nv * E, sb);
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


// ---------------------------------------------------------------------------
// Backward with the group held in L2 rather than in shared memory.  A
// cluster of csize CTAs (one CTA per SM) walks a contiguous range of groups;
// CTA rank q owns slice q of every group (nv 16-byte vectors).  Roles:
//
//   producer (warp 0, one thread)  streams the slices, in chunks of
//       kL2Chunk vectors of x and of dy, into a ring of shared-memory
//       stages with 1D bulk copies                              -> full[s]
//   reducers (warps 1 .. kL2Red)  take every chunk: per thread the sums of
//       W[c] * dy and W[c] * dy * (x - mean), per vector (dy * (x - mean),
//       dy) into shared memory; at the end of the slice they reduce the
//       per-vector sums per channel into the partial row, and thread 0
//       posts the CTA's pair (warps in a fixed order)          -> sum_ready
//   exchanger (the next warp)  trades the pair with the cluster through
//       distributed shared memory, adds the csize pairs in rank order and
//       posts (c1, c2)                                          -> red
//   appliers (the other warps)  read the slice again, from L2 where the
//       producer's copies left it, and write dx                 -> free
//
// The ring only has to cover the latency of HBM, not a whole slice, so the
// cluster size is free of shared memory: the host picks it so that two
// groups of slices of every resident CTA fit in a fraction of L2 (the
// reducers start group i + 2 only after the appliers have finished group
// i).  Per-group buffers and mbarriers alternate with b = i & 1; the phase
// of group i on them is (i >> 1) & 1.  Every wait is bounded, the reducers
// take their decisions at predicate-reducing barriers, and every CTA of a
// cluster ends at a cluster barrier.
// ---------------------------------------------------------------------------
constexpr int kL2Threads = 768;
constexpr int kL2Red = 8;                                  // reducer warps
constexpr int kL2App = kL2Threads / 32 - kL2Red - 2;       // applier warps
constexpr int kL2Chunk = 512;                              // vectors of x (and dy) a stage
constexpr int kL2Stages = 4;
constexpr int kL2Unroll = 4;                               // vectors an applier loads at once
constexpr int kL2MaxVec = 8192;                            // slice vectors
static_assert(kL2Chunk % (32 * kL2Red) == 0, "every reducer thread takes whole chunks");

struct GnL2 {
  uint64_t full[kL2Stages], empty[kL2Stages];
  uint64_t sum_ready[2], red[2], free[2], xbar[2];
  float2 csum[2];                 // the CTA's pair of group i
  float2 stat[2];                 // (c1, c2) of group i
  float2 wred[kL2Red];            // reducer-warp pairs
  float2 xch[2][kMaxCluster];     // peers' pairs by sender rank
  float2 wsum[kL2Red];            // channel part sums
  int abort;
};

// Reducer barrier (named barrier 2 over the reducer warps); the voting form
// tells whether `ok` held in every reducer thread.
__device__ __forceinline__ bool red_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 2, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(32 * kL2Red)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void red_sync() {
  asm volatile("bar.sync 2, %0;" ::"r"(32 * kL2Red) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kL2Threads, 1) gn_bwd_l2(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd, T* __restrict__ dx,
    float* __restrict__ partial, int64_t ngroups, int M, int spv, int Cg, int G, int C,
    int csize, int nv, int stages) {
  constexpr int E = Traits<T>::kVec;
  constexpr int CH = kL2Chunk;
  constexpr uint32_t stride = 2u * CH * 16u;
  extern __shared__ __align__(128) unsigned char ring[];   // stages x stride, then vsum
  float2* vsum = reinterpret_cast<float2*>(ring + (size_t)stages * stride);
  __shared__ GnL2 st;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = csize > 1 ? cta_rank() : 0u;
  const int64_t cid = blockIdx.x / csize, ncl = gridDim.x / csize;
  const int64_t g0 = cid * ngroups / ncl;
  const int count = (int)((cid + 1) * ngroups / ncl - g0);
  const int vbase = (int)rank * nv;
  if (threadIdx.x == 0) st.abort = 0;
  if (threadIdx.x < stages) {
    mbar_init(&st.full[threadIdx.x], 1);
    mbar_init(&st.empty[threadIdx.x], kL2Red);
  }
  if (threadIdx.x < 2) {
    mbar_init(&st.sum_ready[threadIdx.x], 1);
    mbar_init(&st.red[threadIdx.x], 1);
    mbar_init(&st.free[threadIdx.x], kL2App);
    mbar_init(&st.xbar[threadIdx.x], csize);
  }
  fence_mbar_init();
  __syncthreads();
  if (csize > 1) cluster_sync();
  pdl_trigger();
  if (threadIdx.x == 0 && count > 0) {  // the first chunks into L2 (prefetch_l2)
    const int64_t off = g0 * M + (int64_t)vbase * E;
    const uint32_t b = (uint32_t)(nv < stages * CH ? nv : stages * CH) * 16u;
    prefetch_l2(x + off, b);
    prefetch_l2(dy + off, b);
  }
  pdl_wait();
  volatile int* abort = &st.abort;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int i = 0; i < count && ok; ++i) {
        const int64_t off = ((g0 + i) * M + (int64_t)vbase * E) * (int64_t)sizeof(T);
        const unsigned char* xs = reinterpret_cast<const unsigned char*>(x) + off;
        const unsigned char* ds = reinterpret_cast<const unsigned char*>(dy) + off;
        for (int c0 = 0; c0 < nv; c0 += CH) {
          if (issued >= stages && !gn_wait(&st.empty[stage], ph ^ 1u, abort)) {
            ok = false;
            break;
          }
          const uint32_t bytes = (uint32_t)(nv - c0 < CH ? nv - c0 : CH) * 16u;
          unsigned char* dst = ring + (size_t)stage * stride;
          mbar_arrive_expect_tx(&st.full[stage], 2u * bytes);
          bulk_load(dst, xs + (size_t)c0 * 16, bytes, &st.full[stage]);
          bulk_load(dst + CH * 16, ds + (size_t)c0 * 16, bytes, &st.full[stage]);
          ++issued;
          if (++stage == stages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      // every copy issued must land before the CTA may exit: the latest
      // min(issued, stages) issues are the last use of each stage
      const int outstanding = issued < stages ? (int)issued : stages;
      for (int q = 0; q < outstanding; ++q) {
        if (stage == 0) {
          stage = stages - 1;
          ph ^= 1u;
        } else {
          --stage;
        }
        gn_drain(&st.full[stage], ph);
      }
    }
  } else if (warp <= kL2Red) {
    const int rw = warp - 1, rt = threadIdx.x - 32, step = 32 * kL2Red;
    const int c_lo = vbase / spv, c_hi = (vbase + nv - 1) / spv;
    const int nch = c_hi - c_lo + 1;
    int stage = 0;
    uint32_t ph = 0;
    for (int i = 0; i < count; ++i) {
      const int b = i & 1;
      const int64_t grp = g0 + i;
      bool ok = true;
      if (i >= 2) ok = gn_wait(&st.free[b], ((i - 2) >> 1) & 1, abort);
      if (!red_all(__all_sync(kFull, ok))) break;
      const float mu = __ldg(mean + grp);
      const int cbase = (int)(grp % G) * Cg;
      float p1 = 0.f, p2 = 0.f;
      ChanWalk cw(vbase + rt, step, spv);
      for (int c0 = 0; c0 < nv && ok; c0 += CH) {
        ok = __all_sync(kFull, gn_wait(&st.full[stage], ph, abort));
        if (!ok) break;
        const uint4* sx = reinterpret_cast<const uint4*>(ring + (size_t)stage * stride);
        const uint4* sd = sx + CH;
        const int len = nv - c0 < CH ? nv - c0 : CH;
#pragma unroll
        for (int k = 0; k < CH / (32 * kL2Red); ++k) {
          const int l = rt + k * step;
          if (l < len) {
            float xf[E], df[E];
            unpack<T>(sx[l], xf);
            unpack<T>(sd[l], df);
            float q2 = 0.f, sb = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
              q2 = fmaf(df[e], xf[e] - mu, q2);
              sb += df[e];
            }
            const float w = Traits<T>::to_f(gamma[cbase + cw.q]);
            p1 = fmaf(w, sb, p1);
            p2 = fmaf(w, q2, p2);
            vsum[c0 + l] = make_float2(q2, sb);
          }
          cw.next();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&st.empty[stage]);
        if (++stage == stages) {
          stage = 0;
          ph ^= 1u;
        }
      }
      p1 = warp_sum(p1);
      p2 = warp_sum(p2);
      if (lane == 0) st.wred[rw] = make_float2(p1, p2);
      if (!red_all(ok)) break;  // vsum and wred complete
      if (rt == 0) {
        float2 t = make_float2(0.f, 0.f);
        for (int w = 0; w < kL2Red; ++w) {
          t.x += st.wred[w].x;
          t.y += st.wred[w].y;
        }
        st.csum[b] = t;
        mbar_arrive(&st.sum_ready[b]);
      }
      // Per-channel sums of this slice in a fixed order: dW = rstd * sum
      // dy * (x - mean), dB = sum dy; channels of the group the slice does
      // not touch get 0.  (The next group's first barrier orders these
      // reads of vsum and wred before their next writes.)
      const float rs = __ldg(rstd + grp);
      float* prow = partial + ((grp / G) * csize + rank) * (int64_t)(2 * C);
      for (int cl = rt; cl < Cg; cl += step) {
        if (cl < c_lo || cl > c_hi) {
          prow[cbase + cl] = 0.f;
          prow[C + cbase + cl] = 0.f;
        }
      }
      if (nch >= kL2Red) {
        for (int cl = c_lo + rw; cl <= c_hi; cl += kL2Red) {
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
            prow[cbase + cl] = rs * s1;
            prow[C + cbase + cl] = s2;
          }
        }
      } else {
        const int wpc = kL2Red / nch;
        if (rw < nch * wpc) {
          const int cl = c_lo + rw / wpc, part = rw % wpc;
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
          if (lane == 0) st.wsum[rw] = make_float2(s1, s2);
        }
        red_sync();
        if (rt < nch) {
          float s1 = 0.f, s2 = 0.f;
          for (int q = 0; q < wpc; ++q) {
            s1 += st.wsum[rt * wpc + q].x;
            s2 += st.wsum[rt * wpc + q].y;
          }
          prow[cbase + c_lo + rt] = rs * s1;
          prow[C + cbase + c_lo + rt] = s2;
        }
      }
    }
  } else if (warp == kL2Red + 1) {
    for (int i = 0; i < count; ++i) {
      const int b = i & 1;
      const uint32_t ph = (uint32_t)(i >> 1) & 1u;
      const int64_t grp = g0 + i;
      if (!__all_sync(kFull, gn_wait(&st.sum_ready[b], ph, abort))) break;
      float2 t = st.csum[b];
      if (csize > 1) {
        if (lane < csize) {
          st_peer2(&st.xch[b][rank], (uint32_t)lane, t);
          mbar_arrive_peer(&st.xbar[b], (uint32_t)lane);
        }
        if (!__all_sync(kFull, gn_wait_cluster(&st.xbar[b], ph, abort))) break;
        t = make_float2(0.f, 0.f);
        for (int r = 0; r < csize; ++r) {
          t.x += st.xch[b][r].x;
          t.y += st.xch[b][r].y;
        }
      }
      if (lane == 0) {
        const float rs = __ldg(rstd + grp);
        st.stat[b] = make_float2(t.x / (float)M, t.y * rs / (float)M);
        mbar_arrive(&st.red[b]);
      }
    }
  } else {
    constexpr int U = kL2Unroll;
    const int at = threadIdx.x - 32 * (kL2Red + 2), step = 32 * kL2App;
    for (int i = 0; i < count; ++i) {
      const int b = i & 1;
      const int64_t grp = g0 + i;
      if (!__all_sync(kFull, gn_wait(&st.red[b], (uint32_t)(i >> 1) & 1u, abort))) break;
      const float2 cc = st.stat[b];
      const float mu = __ldg(mean + grp), rs = __ldg(rstd + grp);
      const int cbase = (int)(grp % G) * Cg;
      const T* xs = x + grp * M + (int64_t)vbase * E;
      const T* ds = dy + grp * M + (int64_t)vbase * E;
      T* xo = dx + grp * M + (int64_t)vbase * E;
      ChanWalk cw(vbase + at, step, spv);
      for (int v0 = at; v0 < nv; v0 += U * step) {
        uint4 xv[U], dv[U];
        int ch[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * step;
          ch[u] = cw.q;
          cw.next();
          if (v < nv) {
            xv[u] = ld_stream(xs + (int64_t)v * E);
            dv[u] = ld_stream(ds + (int64_t)v * E);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * step;
          if (v < nv) {
            const float w = Traits<T>::to_f(gamma[cbase + ch[u]]);
            float xf[E], df[E], o[E];
            unpack<T>(xv[u], xf);
            unpack<T>(dv[u], df);
#pragma unroll
            for (int e = 0; e < E; ++e) {
              const float xh = (xf[e] - mu) * rs;
              o[e] = fmaf(-xh, cc.y, df[e] * w - cc.x) * rs;
            }
            st_vec(xo + (int64_t)v * E, pack<T>(o));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&st.free[b]);
    }
  }
  __syncwarp();
  if (csize > 1) cluster_sync();
}

// Pipeline shape: the smallest cluster (1..16 CTAs) whose slices leave at
// least min_stages ring stages (a multiple of the reducer count) in kGnSmem;
// false when none does.
struct PipeShape {
  int csize, stages, nv, threads;
  size_t smem;
  int ntw;  // warps a reducer team
};

// Warps a reducer team (measured on GB300: 2 beat 1, 3 and 4).
constexpr int kGnTeamWarps = 2;

bool pick_pipe_min(int nvec, int min_stages, PipeShape* ps) {
  for (int k = 1; k <= kMaxCluster; k *= 2) {
    if (nvec % k) continue;
    const int nv = nvec / k;
    const size_t sb = (size_t)nv * 16;
    if ((size_t)min_stages * sb > (size_t)kGnSmem) continue;
    int st = (int)((size_t)kGnSmem / sb);
    if (st > kGnStages) st = kGnStages;
    st -= st % kGnReducers;
    const int ntw = kGnTeamWarps;
    int apps = (nv + 31) / 32;
    const int max_apps = kGnThreadsMax / 32 - 1 - kGnReducers * ntw;
    if (apps > max_apps) apps = max_apps;
    *ps = PipeShape{k, st, nv, 32 * (1 + kGnReducers * ntw + apps), (size_t)st * sb, ntw};
    return true;
  }
  return false;
}

// The smallest cluster with three stages: measured on GB300, larger
// clusters with deeper rings are slower (fewer resident clusters, costlier
// exchanges).
bool pick_pipe(int nvec, PipeShape* ps) { return pick_pipe_min(nvec, 3, ps); }

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

// Shape of the L2-staged backward: among the power-of-two clusters (1..16)
// that divide the group's vectors and leave at most kL2MaxVec a CTA, those
// whose in-flight slices (two groups of x and dy a CTA, over every resident
// CTA) fit in kL2Budget bytes of L2; of these the fewest rounds of groups
// times (slice + a fixed cost a group for its barriers and exchange), the
// smaller cluster on a tie.  The ring takes what shared memory the per-vector
// sums leave (at least three stages).  False when none fits.
constexpr size_t kL2Budget = (size_t)96 << 20;
constexpr int kL2GroupCost = 1024;  // in slice vectors

struct L2Shape {
  int csize, nv, stages;
  int64_t ncl;
  size_t smem;
};

template <typename T>
bool pick_l2(int nvec, int64_t groups, L2Shape* out) {
  const void* kern = (const void*)gn_bwd_l2<T>;
  const size_t stride = (size_t)2 * kL2Chunk * 16;
  int64_t best = -1;
  for (int k = 1; k <= kMaxCluster; k *= 2) {
    if (nvec % k || nvec / k > kL2MaxVec) continue;
    const int nv = nvec / k;
    const size_t vs = (size_t)nv * sizeof(float2);
    int stages = (int)(((size_t)kGnSmem - vs) / stride);
    if (stages > kL2Stages) stages = kL2Stages;
    if (stages < 3) continue;
    const size_t smem = (size_t)stages * stride + vs;
    const int64_t active = pipe_clusters(kern, PipeShape{k, stages, nv, kL2Threads, smem, 0});
    if (active <= 0) continue;
    if ((size_t)4 * nv * 16 * (size_t)(active * k) > kL2Budget) continue;
    const int64_t ncl = active < groups ? active : groups;
    const int64_t cost = (groups + ncl - 1) / ncl * (nv + kL2GroupCost);
    if (best < 0 || cost < best) {
      best = cost;
      *out = L2Shape{k, nv, stages, ncl, smem};
    }
  }
  return best >= 0;
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
    if (pick_pipe(nvec, &ps)) {
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
  L2Shape ls{};
  if (a.vec_ok && pick_l2<T>(M / E, groups, &ls)) {
    csize = ls.csize;
    e = launch_kernel(gn_bwd_l2<T>, dim3((unsigned)(ls.ncl * ls.csize)), dim3(kL2Threads),
                      ls.smem, s, ls.csize, dy, x, g, a.mean, a.rstd, dx, a.partial, groups, M,
                      a.spatial / E, Cg, a.groups, a.channels, ls.csize, ls.nv, ls.stages);
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
