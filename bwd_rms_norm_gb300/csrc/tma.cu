// Persistent, TMA-staged, warp-specialised forward and backward kernels for
// sm_103a (RMSNorm, and LayerNorm on the same pipeline).
//
// The path is bound by HBM bandwidth.  A row-wise normalisation cannot
// write any output of a row before the whole row has been reduced, so two
// things decide the speed: how many bytes each SM keeps in flight, and that
// the latency of each row's reduction never stalls the stream of outputs.
// One CTA per SM owns a contiguous range of rows (in the forwards of rows of
// 16 KB and more, every grid-th row; rows too wide for one CTA's ring are
// split over a cluster of 2 or 4 CTAs, each staging its part of every row)
// and splits its warps into three roles that meet at per-stage mbarriers:
//
//   producer (warp 0, one thread)  streams the CTA's rows into a ring of
//       shared-memory stages with 1D bulk copies (cp.async.bulk, the TMA
//       engine) -- up to 96 KB of rows in flight per SM in the forward of
//       rows up to 16 KB (but for the FP8 store of 16 KB rows), up to
//       200 KB otherwise, none of it held in registers;          -> full[s]
//   reducers (warps 1..R)  one warp per row (warp d takes the CTA's rows
//       d, d + R, ...): the row statistic -- rstd in the forward,
//       c = sum(g * x_hat) / hidden in the backward -- into the stage's slot;
//                                                                 -> red[s]
//   appliers (the remaining threads)  walk every row in order; each thread
//       owns the same 16-byte vectors of every row (8-byte slices in the
//       narrow-row backward), keeps their gains (and in the backward their
//       fp32 dw accumulators) in registers, and writes y or dx with 128-bit
//       stores.  No barrier among the appliers.
//
// Narrow rows (up to 4 KB) are staged several to a stage in the backward
// (bwd_tma_rows), so that a stage's handshakes serve several rows; rows too
// wide for one CTA's ring are split over a cluster (fwd_tma_split,
// bwd_tma_split), and the widest single-CTA backward (bwd_tma_wide) keeps a
// packed copy of the gains beside its ring.
//
// A stage is released (empty[s]) when its reducer and every applier warp
// have read it.  The stage count is a multiple of R, so reducer d only ever
// uses the stages s = d (mod R) and sees every phase of their barriers in
// order, like the producer and the appliers, which walk all stages in order:
// an mbarrier parity wait is only unambiguous for a waiter that has seen the
// phase before it.  Numerics are those of the register kernels: fp32 sums of
// squares and dots, rstd = 1/sqrt(mean + eps) correctly rounded, one rounding
// at the store (two for the round-twice forward).
//
// Every wait on an mbarrier is bounded (about one second of %globaltimer).
// A wait that runs out counts in a device error counter, raises an abort
// flag in shared memory so that every other wait of the CTA returns at once,
// and the CTA drains: the producer waits (again bounded) for each bulk copy
// it issued before it exits.  rms_norm_wait_timeouts() reports the count.
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "cluster.cuh"
#include "launch.h"
#include "mbar.cuh"
#include "rms_norm.h"

namespace rmsn {

namespace {

__device__ unsigned int g_wait_timeouts;

constexpr int kMaxStages = 32;
constexpr int kMaxThreads = 1024;
constexpr int kMaxReducers = 12;
// Dynamic shared memory for the ring (and the backward's fp32 gain row).
constexpr int kRingBudget = 200 * 1024;
// Rows (stages, for the narrow-row backward) a CTA prefetches into L2
// before its griddepcontrol.wait (see prefetch_l2): measured on GB300, four
// beat two and a whole ring -- a whole ring's prefetches delayed the first
// loads of a call made alone (4096 x 4096 backward alone 27.6 -> 28.7 us).
constexpr int kPrefetchRows = 4;

// Bounded waits counted in this file's timeout counter.
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return wait_phase_counted(bar, parity, abort, &g_wait_timeouts);
}

__device__ void drain_phase(uint64_t* bar, uint32_t parity) {
  drain_phase_counted(bar, parity, &g_wait_timeouts);
}

// Barriers and per-stage values of the pipeline (static shared memory).
struct Pipe {
  uint64_t full[kMaxStages];   // the stage's bulk copies landed
  uint64_t red[kMaxStages];    // a reducer wrote stat[s]
  uint64_t empty[kMaxStages];  // reducer and appliers are done with the stage
  float stat[kMaxStages];      // rstd (forward) or c (backward) of the stage's row
  float stat2[kMaxStages];     // LayerNorm: mean (forward) or c2 (backward)
  int abort;
};

// The rows a CTA owns: the contiguous range [r0, r0 + n) of an even split
// of all rows over the grid.
struct Rows {
  int64_t r0;
  int n;
  __device__ __forceinline__ int64_t row(int i) const { return r0 + i; }
};

__device__ __forceinline__ Rows cta_rows(int64_t rows) {
  Rows r;
  r.r0 = (int64_t)blockIdx.x * rows / gridDim.x;
  r.n = (int)((int64_t)(blockIdx.x + 1) * rows / gridDim.x - r.r0);
  return r;
}

// The rows of a forward CTA dealt round-robin (a forward keeps no row
// order: every row's outputs are its own): its i-th row is r0 + i * step,
// r0 the CTA's index and step the grid, so that the grid streams one window
// of consecutive rows at a time.  The forwards take it for rows of
// kRoundRobinBytes and more (a template switch; narrower rows keep the
// contiguous split).  Measured on GB300 (forward alone, and steps of forward
// + backward): 16384 x 8192 bf16 87.0 -> 85.6 us (step 201.3 -> 200.3 us),
// its LayerNorm 92.9 -> 88.6 us (step 221.1 -> 217.1 us), 4096 x 16384 fp16
// 44.4 -> 43.0 us (step 106.8 -> 105.6 us); slower for 6 KB rows (8192 x
// 3072 bf16 17.31 -> 17.56 us).  Under the FP8 store they pay only
// together with the full ring (see kFwdRingBytes).
struct StridedRows {
  int64_t r0, step;
  int n;
  __device__ __forceinline__ int64_t row(int i) const { return r0 + (int64_t)i * step; }
};

constexpr int kRoundRobinBytes = 16 * 1024;

template <bool RR>
__device__ __forceinline__ std::conditional_t<RR, StridedRows, Rows> fwd_rows(int64_t rows) {
  if constexpr (RR) {
    StridedRows r;
    r.r0 = blockIdx.x;
    r.step = gridDim.x;
    r.n = (int)((rows - blockIdx.x + gridDim.x - 1) / gridDim.x);
    return r;
  } else {
    return cta_rows(rows);
  }
}

// The CTA's first rows of x into L2 (prefetch_l2): one hint over a
// contiguous range, one a row when they are dealt round-robin.
template <typename T>
__device__ __forceinline__ void prefetch_first_rows(const T* x, const Rows& rw, int hidden) {
  if (rw.n > 0)
    prefetch_l2(x + rw.r0 * hidden,
                (uint32_t)((rw.n < kPrefetchRows ? rw.n : kPrefetchRows) * hidden * sizeof(T)));
}

template <typename T>
__device__ __forceinline__ void prefetch_first_rows(const T* x, const StridedRows& rw, int hidden) {
  for (int q = 0; q < rw.n && q < kPrefetchRows; ++q)
    prefetch_l2(x + rw.row(q) * hidden, (uint32_t)(hidden * sizeof(T)));
}

// Position in the ring: stage index and phase parity, advanced without
// division.
struct RingPos {
  int stage;
  uint32_t phase;
  __device__ __forceinline__ void advance(int by, int stages) {
    stage += by;
    while (stage >= stages) {
      stage -= stages;
      phase ^= 1u;
    }
  }
};

// Called by every thread; thread s initialises stage s's barriers.  The
// caller synchronises the CTA afterwards.
__device__ __forceinline__ void init_pipe(Pipe& p, int stages, int applier_warps) {
  const int s = threadIdx.x;
  if (s == 0) p.abort = 0;
  if (s < stages) {
    mbar_init(&p.full[s], 1);
    mbar_init(&p.red[s], 1);
    mbar_init(&p.empty[s], 1 + applier_warps);
    fence_mbar_init();
  }
}

// Producer: issue the copies of the CTA's rows (its i-th row is rw.row(i))
// into the ring.  NSRC source tensors go to consecutive parts of a stage.
// Rows are `pitch` bytes apart in global memory; `bytes` of each are copied
// (a whole row, or the slice a CTA of a cluster owns).
template <int NSRC, class RW = Rows>
__device__ void produce_pitched(Pipe& p, unsigned char* ring, int stride, int stages,
                                const void* const (&src)[NSRC], const RW& rw, size_t pitch,
                                uint32_t bytes, volatile int* abort) {
  RingPos pos{0, 0u};
  int i = 0;
  const int n = rw.n;
  for (; i < n; ++i) {
    // the stage's previous use (parity phase ^ 1) must be released first
    if (i >= stages && !wait_phase(&p.empty[pos.stage], pos.phase ^ 1u, abort)) break;
    unsigned char* dst = ring + (size_t)pos.stage * stride;
    mbar_arrive_expect_tx(&p.full[pos.stage], NSRC * bytes);
    const size_t off = (size_t)rw.row(i) * pitch;
#pragma unroll
    for (int t = 0; t < NSRC; ++t)
      bulk_load(dst + t * bytes, static_cast<const unsigned char*>(src[t]) + off, bytes,
                &p.full[pos.stage]);
    pos.advance(1, stages);
  }
  // Before the CTA may exit every copy issued must have landed: the last
  // min(i, stages) issues are the latest use of each stage; walk back.
  const int outstanding = i < stages ? i : stages;
  for (int q = 0; q < outstanding; ++q) {
    if (pos.stage == 0) {
      pos.stage = stages - 1;
      pos.phase ^= 1u;
    } else {
      --pos.stage;
    }
    drain_phase(&p.full[pos.stage], pos.phase);
  }
}

template <int NSRC, class RW = Rows>
__device__ __forceinline__ void produce(Pipe& p, unsigned char* ring, int stride, int stages,
                                        const void* const (&src)[NSRC], const RW& rw,
                                        uint32_t row_bytes, volatile int* abort) {
  produce_pitched<NSRC, RW>(p, ring, stride, stages, src, rw, row_bytes, row_bytes, abort);
}

// Producer of stages that hold K consecutive rows each (narrow rows): stage
// j takes the CTA's rows [jK, min(jK + K, n)).  A tensor's rows are
// contiguous in global memory, so one bulk copy a tensor fills the stage;
// tensor t's rows go to bytes [t * K * row_bytes, (t + 1) * K * row_bytes)
// of the stage.  Copies and drain as in produce_pitched.
template <int NSRC, int K>
__device__ void produce_rows(Pipe& p, unsigned char* ring, int stride, int stages,
                             const void* const (&src)[NSRC], const Rows& rw, uint32_t row_bytes,
                             volatile int* abort) {
  RingPos pos{0, 0u};
  const int nst = (rw.n + K - 1) / K;
  int j = 0;
  for (; j < nst; ++j) {
    if (j >= stages && !wait_phase(&p.empty[pos.stage], pos.phase ^ 1u, abort)) break;
    const int i = j * K;
    const uint32_t bytes = (uint32_t)(rw.n - i < K ? rw.n - i : K) * row_bytes;
    unsigned char* dst = ring + (size_t)pos.stage * stride;
    mbar_arrive_expect_tx(&p.full[pos.stage], NSRC * bytes);
    const size_t off = (size_t)rw.row(i) * row_bytes;
#pragma unroll
    for (int t = 0; t < NSRC; ++t)
      bulk_load(dst + (size_t)t * K * row_bytes, static_cast<const unsigned char*>(src[t]) + off,
                bytes, &p.full[pos.stage]);
    pos.advance(1, stages);
  }
  const int outstanding = j < stages ? j : stages;
  for (int q = 0; q < outstanding; ++q) {
    if (pos.stage == 0) {
      pos.stage = stages - 1;
      pos.phase ^= 1u;
    } else {
      --pos.stage;
    }
    drain_phase(&p.full[pos.stage], pos.phase);
  }
}

// Sum of per-element partial sums, pairwise.
template <int E>
__device__ __forceinline__ float pairwise(float (&p)[E]) {
#pragma unroll
  for (int w = E / 2; w >= 1; w /= 2)
#pragma unroll
    for (int e = 0; e < w; ++e) p[e] += p[e + w];
  return p[0];
}

// The fp32 gains (gamma + off) in shared memory for the reducers, one
// 16-byte vector of gamma per load.  Vector v's E gains are stored as E/4
// float4 in E/4 planes of nvec float4 each (plane q holds elements 4q..4q+3
// of every vector), so that a warp reading the planes of 32 consecutive
// vectors reads 512 contiguous bytes: no bank conflicts.
template <typename T>
__device__ __forceinline__ void stage_gains(float* gain, const T* __restrict__ gamma, int nvec,
                                            float off, int t, int nthreads) {
  constexpr int E = Traits<T>::kVec;
  float4* g4 = reinterpret_cast<float4*>(gain);
  for (int v = t; v < nvec; v += nthreads) {
    float f[E];
    unpack<T>(ld_shared_ro(gamma + (int64_t)v * E), f);
#pragma unroll
    for (int e = 0; e < E; e += 4)
      g4[(e / 4) * nvec + v] = make_float4(f[e] + off, f[e + 1] + off, f[e + 2] + off,
                                           f[e + 3] + off);
  }
}

// Forward.  Reducer: sum of squares of its row, rstd, written to global and
// to the stage's slot.  Appliers: y = round((x * rstd) * gain) (or the
// round-twice store) for their vectors of every row.  RR: rows dealt
// round-robin (StridedRows).
template <typename T, int VPT, bool F8, bool RR>
__global__ void __launch_bounds__(kMaxThreads, 1) fwd_tma(
    const T* __restrict__ x, const T* __restrict__ gamma, void* __restrict__ y,
    float* __restrict__ rstd, int64_t rows, int hidden, float eps, float off, int twice,
    const float* __restrict__ scale, int stages, int reducers) {
  constexpr int E = Traits<T>::kVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Pipe pipe;
  const int row_bytes = hidden * (int)sizeof(T);
  const int stride = (row_bytes + 127) / 128 * 128;
  const int appliers = blockDim.x - 32 * (1 + reducers);
  const auto rw = fwd_rows<RR>(rows);
  const int n = rw.n;
  init_pipe(pipe, stages, appliers / 32);
  __syncthreads();
  pdl_trigger();
  if (threadIdx.x == 0) prefetch_first_rows(x, rw, hidden);
  pdl_wait();
  volatile int* abort = &pipe.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = hidden / E;

  if (warp == 0) {
    if (lane == 0) {
      const void* const src[1] = {x};
      produce<1>(pipe, smem, stride, stages, src, rw, (uint32_t)row_bytes, abort);
    }
    return;
  }

  if (warp <= reducers) {
    const int d = warp - 1;
    RingPos pos{0, 0u};
    pos.advance(d, stages);
    for (int i = d; i < n; i += reducers) {
      // a warp leaves as a whole: a wait that failed on any lane ends it
      if (!__all_sync(0xffffffffu, wait_phase(&pipe.full[pos.stage], pos.phase, abort))) return;
      const uint4* st = reinterpret_cast<const uint4*>(smem + (size_t)pos.stage * stride);
      float part[E];
#pragma unroll
      for (int e = 0; e < E; ++e) part[e] = 0.f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float f[E];
        unpack<T>(st[v], f);
#pragma unroll
        for (int e = 0; e < E; ++e) part[e] = fmaf(f[e], f[e], part[e]);
      }
      const float ss = warp_sum(pairwise<E>(part));
      float rs = rstd_of(ss / (float)hidden, eps);
      if (isinf(ss)) {  // the fp32 sum of squares overflowed (see kOverflowScale)
        float s2 = 0.f;
        for (int v = lane; v < nvec; v += 32) {
          float f[E];
          unpack<T>(st[v], f);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float t = f[e] * kOverflowScale;
            s2 = fmaf(t, t, s2);
          }
        }
        rs = rstd_rescaled(warp_sum(s2), hidden, eps);
      }
      if (lane == 0) {
        rstd[rw.row(i)] = rs;
        pipe.stat[pos.stage] = rs;
        mbar_arrive(&pipe.red[pos.stage]);
        mbar_arrive(&pipe.empty[pos.stage]);
      }
      pos.advance(reducers, stages);
    }
    return;
  }

  const int a = threadIdx.x - 32 * (1 + reducers);
  const float sc = F8 ? __ldg(scale) : 1.f;
  float ge[VPT][E];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = a + j * appliers;
    const uint4 g4 = v < nvec ? ld_shared_ro(gamma + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    unpack<T>(g4, ge[j]);
#pragma unroll
    for (int e = 0; e < E; ++e) ge[j][e] += off;
  }
  RingPos pos{0, 0u};
  for (int i = 0; i < n; ++i) {
    bool ok = wait_phase(&pipe.red[pos.stage], pos.phase, abort);
    ok = ok && wait_phase(&pipe.full[pos.stage], pos.phase, abort);
    if (!__all_sync(0xffffffffu, ok)) return;
    const float rs = pipe.stat[pos.stage];
    const uint4* st = reinterpret_cast<const uint4*>(smem + (size_t)pos.stage * stride);
    T* yr = static_cast<T*>(y) + rw.row(i) * hidden;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = a + j * appliers;
      if (v < nvec) {
        float f[E], o[E];
        unpack<T>(st[v], f);
        if constexpr (F8) {
          // ((x * rstd) * gain) * scale in fp32, one conversion to E4M3
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = ((f[e] * rs) * ge[j][e]) * sc;
          st_e4m3<E>(static_cast<unsigned char*>(y) + rw.row(i) * hidden + (int64_t)v * E, o);
          continue;
        }
        if (twice) {
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = round_trip<T>(f[e] * rs) * ge[j][e];
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = (f[e] * rs) * ge[j][e];
        }
        st_vec(yr + (int64_t)v * E, pack<T>(o));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pipe.empty[pos.stage]);
    pos.advance(1, stages);
  }
}

// Backward.  Reducer: c = sum(dy * gain * x * rstd) / hidden of its row,
// reading the fp32 gains from a shared-memory copy.  Appliers: dx =
// rstd * (dy * gain - x_hat * c) for their vectors of every row, and the
// fp32 dw accumulators of those columns, written as the block's partial
// row at the end of every block of rows (RowBlocks).
template <typename T, int VPT>
__global__ void __launch_bounds__(kMaxThreads, 1) bwd_tma(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ rstd, T* __restrict__ dx, float* __restrict__ partial,
    int64_t rows, int hidden, float off, int stages, int reducers, int brows) {
  constexpr int E = Traits<T>::kVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Pipe pipe;
  const int row_bytes = hidden * (int)sizeof(T);
  const int stride = (2 * row_bytes + 127) / 128 * 128;
  const int gain_bytes = (hidden * 4 + 127) / 128 * 128;
  float* gain = reinterpret_cast<float*>(smem);
  unsigned char* ring = smem + gain_bytes;
  const int appliers = blockDim.x - 32 * (1 + reducers);
  const RowBlocks blk = row_blocks(rows, brows, blockIdx.x, gridDim.x);
  const Rows rw{blk.r0, blk.n};
  const int n = rw.n;
  init_pipe(pipe, stages, appliers / 32);
  __syncthreads();
  // the next kernel (the dw finalize) may be scheduled now; it waits for
  // this grid to complete before reading the partials
  pdl_trigger();
  if (threadIdx.x == 0 && n > 0) {  // the first rows into L2 (prefetch_l2)
    const uint32_t b = (uint32_t)((n < kPrefetchRows ? n : kPrefetchRows) * row_bytes);
    prefetch_l2(x + rw.r0 * hidden, b);
    prefetch_l2(dy + rw.r0 * hidden, b);
  }
  pdl_wait();
  volatile int* abort = &pipe.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = hidden / E;
  const int doff = row_bytes / 16;  // dy part of a stage, in 16-byte vectors

  if (warp == 0) {
    if (lane == 0) {
      const void* const src[2] = {x, dy};
      produce<2>(pipe, ring, stride, stages, src, rw, (uint32_t)row_bytes, abort);
    }
    return;
  }

  if (warp <= reducers) {
    // The reducers stage the fp32 gains (plane-split, see stage_gains).
    stage_gains<T>(gain, gamma, nvec, off, threadIdx.x - 32, 32 * reducers);
    asm volatile("bar.sync 1, %0;" ::"r"(32 * reducers) : "memory");
    const float4* g4 = reinterpret_cast<const float4*>(gain);
    const int d = warp - 1;
    RingPos pos{0, 0u};
    pos.advance(d, stages);
    for (int i = d; i < n; i += reducers) {
      const float rs = __ldg(rstd + rw.row(i));
      if (!__all_sync(0xffffffffu, wait_phase(&pipe.full[pos.stage], pos.phase, abort))) return;
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)pos.stage * stride);
      float part[E];
#pragma unroll
      for (int e = 0; e < E; ++e) part[e] = 0.f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float xf[E], df[E], gf[E];
        unpack<T>(st[v], xf);
        unpack<T>(st[doff + v], df);
#pragma unroll
        for (int e = 0; e < E; e += 4) {
          const float4 q = g4[(e / 4) * nvec + v];
          gf[e] = q.x;
          gf[e + 1] = q.y;
          gf[e + 2] = q.z;
          gf[e + 3] = q.w;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) part[e] = fmaf(df[e] * gf[e], xf[e], part[e]);
      }
      // sum(g * x) * rstd: the row's rstd is applied once, to the sum
      const float dot = warp_sum(pairwise<E>(part)) * rs;
      if (lane == 0) {
        pipe.stat[pos.stage] = dot / (float)hidden;
        mbar_arrive(&pipe.red[pos.stage]);
        mbar_arrive(&pipe.empty[pos.stage]);
      }
      pos.advance(reducers, stages);
    }
    return;
  }

  const int a = threadIdx.x - 32 * (1 + reducers);
  float ge[VPT][E], acc[VPT][E];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = a + j * appliers;
    const uint4 q = v < nvec ? ld_shared_ro(gamma + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    unpack<T>(q, ge[j]);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      ge[j][e] += off;
      acc[j][e] = 0.f;
    }
  }
  RingPos pos{0, 0u};
  float rs_next = n > 0 ? __ldg(rstd + rw.row(0)) : 0.f;
  int64_t part = blk.b0;
  for (int i = 0; i < n; ++part) {
   const int end = blk.block_end(i);
   for (; i < end; ++i) {
    const float rs = rs_next;
    if (i + 1 < n) rs_next = __ldg(rstd + rw.row(i + 1));
    bool ok = wait_phase(&pipe.red[pos.stage], pos.phase, abort);
    ok = ok && wait_phase(&pipe.full[pos.stage], pos.phase, abort);
    if (!__all_sync(0xffffffffu, ok)) return;
    const float c = pipe.stat[pos.stage];
    const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)pos.stage * stride);
    T* dxr = dx + rw.row(i) * hidden;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = a + j * appliers;
      if (v < nvec) {
        float xf[E], df[E], o[E];
        unpack<T>(st[v], xf);
        unpack<T>(st[doff + v], df);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float xh = xf[e] * rs;
          acc[j][e] = fmaf(df[e], xh, acc[j][e]);
          o[e] = fmaf(-xh, c, df[e] * ge[j][e]) * rs;
        }
        st_vec(dxr + (int64_t)v * E, pack<T>(o));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pipe.empty[pos.stage]);
    pos.advance(1, stages);
   }
    flush_partial<VPT, E>(acc, partial, part, hidden, 0, a, appliers, nvec);
  }
}


// A thread's slice of a row: 8 bytes (HALF) or a 16-byte vector.
template <typename T, bool HALF, typename V>
__device__ __forceinline__ void unpack_s(const V& v, float (&f)[HALF ? Traits<T>::kVec / 2
                                                                  : Traits<T>::kVec]) {
  if constexpr (HALF)
    unpack_h<T>(v, f);
  else
    unpack<T>(v, f);
}

template <typename T, bool HALF>
__device__ __forceinline__ void store_s(T* p, const float (&f)[HALF ? Traits<T>::kVec / 2
                                                                   : Traits<T>::kVec]) {
  if constexpr (HALF)
    *reinterpret_cast<uint2*>(p) = pack_h<T>(f);
  else
    st_vec(p, pack<T>(f));
}

// Backward for narrow rows, in stages of K consecutive rows (produce_rows).
// One row a stage leaves such rows paced by handshakes rather than by
// bandwidth: every row cost the producer an mbarrier arm and two bulk
// copies, and every applier warp two waits and an arrive, against about a
// hundred instructions of arithmetic.  The roles are those of bwd_tma, with
// the producer's and the appliers' handshakes shared by a stage's K rows.
// The reducers still take rows, not stages (reducer d: rows d, d + R, ...),
// so that a stage's rows are reduced side by side; each writes its row's c
// and rstd into the stage's slot for that row, and red[s] completes when
// all K have (a last stage with fewer rows gets an arrival for each missing
// row too, after its copy landed).  R divides the stage count, so reducer d
// meets a stage again only at its own row K * stages later.  The appliers
// walk the stage's rows in order, so every dw accumulator still adds its
// rows in row order and the results are bit for bit those of bwd_tma.  An
// applier owns an 8-byte slice of every row (HALF: twice the threads of
// 16-byte vectors, each with half the arithmetic a row; measured faster for
// rows up to 2 KB, slower for 4 KB rows) or a 16-byte vector.  Blocks of
// rows (RowBlocks) are whole stages: K divides brows.
template <typename T, int K, bool HALF>
__global__ void __launch_bounds__(kMaxThreads, 1) bwd_tma_rows(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ rstd, T* __restrict__ dx, float* __restrict__ partial,
    int64_t rows, int hidden, float off, int stages, int reducers, int brows) {
  constexpr int E = Traits<T>::kVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Pipe pipe;
  __shared__ float cst[kMaxStages * K], rst[kMaxStages * K];
  const int row_bytes = hidden * (int)sizeof(T);
  const int stride = (2 * K * row_bytes + 127) / 128 * 128;
  const int gain_bytes = (hidden * 4 + 127) / 128 * 128;
  float* gain = reinterpret_cast<float*>(smem);
  unsigned char* ring = smem + gain_bytes;
  const int appliers = blockDim.x - 32 * (1 + reducers);
  const RowBlocks blk = row_blocks(rows, brows, blockIdx.x, gridDim.x);
  const Rows rw{blk.r0, blk.n};
  const int n = rw.n;
  const int nst = (n + K - 1) / K;
  if (threadIdx.x == 0) pipe.abort = 0;
  if (threadIdx.x < stages) {
    mbar_init(&pipe.full[threadIdx.x], 1);
    mbar_init(&pipe.red[threadIdx.x], K);
    mbar_init(&pipe.empty[threadIdx.x], K + appliers / 32);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  if (threadIdx.x == 0 && n > 0) {  // the first stages into L2 (prefetch_l2)
    const int pr = n < kPrefetchRows * K ? n : kPrefetchRows * K;
    const uint32_t b = (uint32_t)(pr * row_bytes);
    prefetch_l2(x + rw.r0 * hidden, b);
    prefetch_l2(dy + rw.r0 * hidden, b);
  }
  pdl_wait();
  volatile int* abort = &pipe.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = hidden / E;

  if (warp == 0) {
    if (lane == 0) {
      const void* const src[2] = {x, dy};
      produce_rows<2, K>(pipe, ring, stride, stages, src, rw, (uint32_t)row_bytes, abort);
    }
    return;
  }

  if (warp <= reducers) {
    stage_gains<T>(gain, gamma, nvec, off, threadIdx.x - 32, 32 * reducers);
    asm volatile("bar.sync 1, %0;" ::"r"(32 * reducers) : "memory");
    const float4* g4 = reinterpret_cast<const float4*>(gain);
    const int d = warp - 1;
    // slot i: row i of the CTA, or a missing row of the last stage (i >= n)
    for (int i = d; i < nst * K; i += reducers) {
      const int j = i / K, r = i - j * K;
      const int stage = j % stages;
      const uint32_t phase = (uint32_t)(j / stages) & 1u;
      const float rs = i < n ? __ldg(rstd + rw.row(i)) : 0.f;
      if (!__all_sync(0xffffffffu, wait_phase(&pipe.full[stage], phase, abort))) return;
      if (i < n) {
        const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)stage * stride);
        float part[E];
#pragma unroll
        for (int e = 0; e < E; ++e) part[e] = 0.f;
#pragma unroll 2
        for (int v = lane; v < nvec; v += 32) {
          float xf[E], df[E], gf[E];
          unpack<T>(st[r * nvec + v], xf);
          unpack<T>(st[(K + r) * nvec + v], df);
#pragma unroll
          for (int e = 0; e < E; e += 4) {
            const float4 q = g4[(e / 4) * nvec + v];
            gf[e] = q.x;
            gf[e + 1] = q.y;
            gf[e + 2] = q.z;
            gf[e + 3] = q.w;
          }
#pragma unroll
          for (int e = 0; e < E; ++e) part[e] = fmaf(df[e] * gf[e], xf[e], part[e]);
        }
        // sum(g * x) * rstd: the row's rstd is applied once, to the sum
        const float dot = warp_sum(pairwise<E>(part)) * rs;
        if (lane == 0) {
          cst[stage * K + r] = dot / (float)hidden;
          rst[stage * K + r] = rs;
        }
      }
      if (lane == 0) {
        mbar_arrive(&pipe.red[stage]);
        mbar_arrive(&pipe.empty[stage]);
      }
    }
    return;
  }

  // an applier's slice of a row: H columns in one V
  constexpr int H = HALF ? E / 2 : E;
  using V = std::conditional_t<HALF, uint2, uint4>;
  const int npieces = hidden / H;
  const int a = threadIdx.x - 32 * (1 + reducers);
  float ge[H], acc[H];
  {
    const V q = a < npieces ? __ldg(reinterpret_cast<const V*>(gamma) + a) : V{};
    unpack_s<T, HALF>(q, ge);
#pragma unroll
    for (int e = 0; e < H; ++e) {
      ge[e] += off;
      acc[e] = 0.f;
    }
  }
  RingPos pos{0, 0u};
  int64_t part = blk.b0;
  int bend = blk.block_end(0);
  for (int j = 0, i = 0; j < nst; ++j) {
    const int k = n - i < K ? n - i : K;
    bool ok = wait_phase(&pipe.red[pos.stage], pos.phase, abort);
    ok = ok && wait_phase(&pipe.full[pos.stage], pos.phase, abort);
    if (!__all_sync(0xffffffffu, ok)) return;
    const V* st = reinterpret_cast<const V*>(ring + (size_t)pos.stage * stride);
#pragma unroll
    for (int r = 0; r < K; ++r) {
      if (r < k && a < npieces) {
        const float c = cst[pos.stage * K + r], rs = rst[pos.stage * K + r];
        float xf[H], df[H], o[H];
        unpack_s<T, HALF>(st[r * npieces + a], xf);
        unpack_s<T, HALF>(st[(K + r) * npieces + a], df);
#pragma unroll
        for (int e = 0; e < H; ++e) {
          const float xh = xf[e] * rs;
          acc[e] = fmaf(df[e], xh, acc[e]);
          o[e] = fmaf(-xh, c, df[e] * ge[e]) * rs;
        }
        store_s<T, HALF>(dx + rw.row(i + r) * hidden + (int64_t)a * H, o);
      }
    }
    i += k;
    __syncwarp();
    if (lane == 0) mbar_arrive(&pipe.empty[pos.stage]);
    pos.advance(1, stages);
    if (i == bend) {
      flush_piece<H>(acc, partial, part, hidden, a, npieces);
      ++part;
      bend = blk.block_end(i);
    }
  }
}

// LayerNorm forward.  Reducer: mean, then sum((x - mean)^2) over the row in
// the stage (two passes over shared memory), rstd; both to global and to
// the stage's slots.  Appliers: y = round(fma((x - mean) * rstd, gamma,
// beta)), gains and biases kept packed in registers and widened at use.
// RR: rows dealt round-robin, as in fwd_tma.
template <typename T, int VPT, bool RR>
__global__ void __launch_bounds__(kMaxThreads, 1) ln_fwd_tma(
    const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
    T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, int64_t rows,
    int hidden, float eps, int stages, int reducers) {
  constexpr int E = Traits<T>::kVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Pipe pipe;
  const int row_bytes = hidden * (int)sizeof(T);
  const int stride = (row_bytes + 127) / 128 * 128;
  const int appliers = blockDim.x - 32 * (1 + reducers);
  const auto rw = fwd_rows<RR>(rows);
  const int n = rw.n;
  init_pipe(pipe, stages, appliers / 32);
  __syncthreads();
  pdl_trigger();
  if (threadIdx.x == 0) prefetch_first_rows(x, rw, hidden);
  pdl_wait();
  volatile int* abort = &pipe.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = hidden / E;

  if (warp == 0) {
    if (lane == 0) {
      const void* const src[1] = {x};
      produce<1>(pipe, smem, stride, stages, src, rw, (uint32_t)row_bytes, abort);
    }
    return;
  }

  if (warp <= reducers) {
    const int d = warp - 1;
    RingPos pos{0, 0u};
    pos.advance(d, stages);
    for (int i = d; i < n; i += reducers) {
      if (!__all_sync(0xffffffffu, wait_phase(&pipe.full[pos.stage], pos.phase, abort))) return;
      const uint4* st = reinterpret_cast<const uint4*>(smem + (size_t)pos.stage * stride);
      float part[E];
#pragma unroll
      for (int e = 0; e < E; ++e) part[e] = 0.f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float f[E];
        unpack<T>(st[v], f);
#pragma unroll
        for (int e = 0; e < E; ++e) part[e] += f[e];
      }
      const float mu = warp_sum(pairwise<E>(part)) / (float)hidden;
#pragma unroll
      for (int e = 0; e < E; ++e) part[e] = 0.f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float f[E];
        unpack<T>(st[v], f);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float c = f[e] - mu;
          part[e] = fmaf(c, c, part[e]);
        }
      }
      const float rs = rstd_of(warp_sum(pairwise<E>(part)) / (float)hidden, eps);
      if (lane == 0) {
        mean[rw.row(i)] = mu;
        rstd[rw.row(i)] = rs;
        pipe.stat[pos.stage] = rs;
        pipe.stat2[pos.stage] = mu;
        mbar_arrive(&pipe.red[pos.stage]);
        mbar_arrive(&pipe.empty[pos.stage]);
      }
      pos.advance(reducers, stages);
    }
    return;
  }

  const int a = threadIdx.x - 32 * (1 + reducers);
  uint4 gp[VPT], bp[VPT];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = a + j * appliers;
    const bool in = v < nvec;
    gp[j] = in ? ld_shared_ro(gamma + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    bp[j] = in && beta ? ld_shared_ro(beta + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
  }
  RingPos pos{0, 0u};
  for (int i = 0; i < n; ++i) {
    bool ok = wait_phase(&pipe.red[pos.stage], pos.phase, abort);
    ok = ok && wait_phase(&pipe.full[pos.stage], pos.phase, abort);
    if (!__all_sync(0xffffffffu, ok)) return;
    const float rs = pipe.stat[pos.stage], mu = pipe.stat2[pos.stage];
    const uint4* st = reinterpret_cast<const uint4*>(smem + (size_t)pos.stage * stride);
    T* yr = y + rw.row(i) * hidden;
    // widen the packed gains and biases at each use instead of holding them
    // widened across rows
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      opaque(gp[j]);
      opaque(bp[j]);
    }
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = a + j * appliers;
      if (v < nvec) {
        float f[E], g[E], b[E], o[E];
        unpack<T>(st[v], f);
        unpack<T>(gp[j], g);
        unpack<T>(bp[j], b);
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = fmaf((f[e] - mu) * rs, g[e], b[e]);
        st_vec(yr + (int64_t)v * E, pack<T>(o));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pipe.empty[pos.stage]);
    pos.advance(1, stages);
  }
}

// LayerNorm backward.  Reducer: c1 = sum(g) / hidden and c2 = rstd *
// sum(g * (x - mean)) / hidden with g = dy * gamma (fp32 gains from the
// plane-split shared-memory copy).  Appliers: dx = rstd * (g - c1 - x_hat *
// c2), and fp32 accumulators of dy * x_hat (dgamma) and dy (dbeta) for
// their columns, written at the end as the CTA's partial row [dgamma | dbeta].
// Two vectors per applier hold two fp32 accumulator sets of 2E floats each:
// those blocks are limited to 768 threads, which leaves 80 registers a thread.
constexpr int kLnBwd2Threads = 768;

template <typename T, int VPT>
__global__ void __launch_bounds__(VPT == 2 ? kLnBwd2Threads : kMaxThreads, 1) ln_bwd_tma(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd, T* __restrict__ dx,
    float* __restrict__ partial, int64_t rows, int hidden, int stages, int reducers) {
  constexpr int E = Traits<T>::kVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Pipe pipe;
  const int row_bytes = hidden * (int)sizeof(T);
  const int stride = (2 * row_bytes + 127) / 128 * 128;
  const int gain_bytes = (hidden * 4 + 127) / 128 * 128;
  float* gain = reinterpret_cast<float*>(smem);
  unsigned char* ring = smem + gain_bytes;
  const int appliers = blockDim.x - 32 * (1 + reducers);
  const Rows rw = cta_rows(rows);
  const int n = rw.n;
  init_pipe(pipe, stages, appliers / 32);
  __syncthreads();
  pdl_trigger();
  if (threadIdx.x == 0 && n > 0) {  // the first rows into L2 (prefetch_l2)
    const uint32_t b = (uint32_t)((n < kPrefetchRows ? n : kPrefetchRows) * row_bytes);
    prefetch_l2(x + rw.r0 * hidden, b);
    prefetch_l2(dy + rw.r0 * hidden, b);
  }
  pdl_wait();
  volatile int* abort = &pipe.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = hidden / E;
  const int doff = row_bytes / 16;

  if (warp == 0) {
    if (lane == 0) {
      const void* const src[2] = {x, dy};
      produce<2>(pipe, ring, stride, stages, src, rw, (uint32_t)row_bytes, abort);
    }
    return;
  }

  if (warp <= reducers) {
    stage_gains<T>(gain, gamma, nvec, 0.f, threadIdx.x - 32, 32 * reducers);
    asm volatile("bar.sync 1, %0;" ::"r"(32 * reducers) : "memory");
    const float4* g4 = reinterpret_cast<const float4*>(gain);
    const int d = warp - 1;
    RingPos pos{0, 0u};
    pos.advance(d, stages);
    for (int i = d; i < n; i += reducers) {
      const float mu = __ldg(mean + rw.row(i)), rs = __ldg(rstd + rw.row(i));
      if (!__all_sync(0xffffffffu, wait_phase(&pipe.full[pos.stage], pos.phase, abort))) return;
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)pos.stage * stride);
      float p1[E], p2[E];
#pragma unroll
      for (int e = 0; e < E; ++e) p1[e] = p2[e] = 0.f;
#pragma unroll(VPT == 2 ? 4 : 2)
      for (int v = lane; v < nvec; v += 32) {
        float xf[E], df[E], gf[E];
        unpack<T>(st[v], xf);
        unpack<T>(st[doff + v], df);
#pragma unroll
        for (int e = 0; e < E; e += 4) {
          const float4 q = g4[(e / 4) * nvec + v];
          gf[e] = q.x;
          gf[e + 1] = q.y;
          gf[e + 2] = q.z;
          gf[e + 3] = q.w;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float g = df[e] * gf[e];
          p1[e] += g;
          p2[e] = fmaf(g, xf[e] - mu, p2[e]);
        }
      }
      const float s1 = warp_sum(pairwise<E>(p1));
      const float s2 = warp_sum(pairwise<E>(p2)) * rs;
      if (lane == 0) {
        pipe.stat[pos.stage] = s1 / (float)hidden;
        pipe.stat2[pos.stage] = s2 / (float)hidden;
        mbar_arrive(&pipe.red[pos.stage]);
        mbar_arrive(&pipe.empty[pos.stage]);
      }
      pos.advance(reducers, stages);
    }
    return;
  }

  const int a = threadIdx.x - 32 * (1 + reducers);
  uint4 gp[VPT];
  float ag[VPT][E], ab[VPT][E];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = a + j * appliers;
    gp[j] = v < nvec ? ld_shared_ro(gamma + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int e = 0; e < E; ++e) ag[j][e] = ab[j][e] = 0.f;
  }
  RingPos pos{0, 0u};
  float mu_next = 0.f, rs_next = 0.f;
  if (n > 0) {
    mu_next = __ldg(mean + rw.row(0));
    rs_next = __ldg(rstd + rw.row(0));
  }
  for (int i = 0; i < n; ++i) {
    const float mu = mu_next, rs = rs_next;
    if (i + 1 < n) {
      mu_next = __ldg(mean + rw.row(i + 1));
      rs_next = __ldg(rstd + rw.row(i + 1));
    }
    bool ok = wait_phase(&pipe.red[pos.stage], pos.phase, abort);
    ok = ok && wait_phase(&pipe.full[pos.stage], pos.phase, abort);
    if (!__all_sync(0xffffffffu, ok)) return;
    const float c1 = pipe.stat[pos.stage], c2 = pipe.stat2[pos.stage];
    const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)pos.stage * stride);
    T* dxr = dx + rw.row(i) * hidden;
#pragma unroll
    for (int j = 0; j < VPT; ++j) opaque(gp[j]);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = a + j * appliers;
      if (v < nvec) {
        float xf[E], df[E], gf[E], o[E];
        unpack<T>(st[v], xf);
        unpack<T>(st[doff + v], df);
        unpack<T>(gp[j], gf);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float xh = (xf[e] - mu) * rs;
          ag[j][e] = fmaf(df[e], xh, ag[j][e]);
          ab[j][e] += df[e];
          o[e] = fmaf(-xh, c2, df[e] * gf[e] - c1) * rs;
        }
        st_vec(dxr + (int64_t)v * E, pack<T>(o));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pipe.empty[pos.stage]);
    pos.advance(1, stages);
  }
  float* pr = partial + (int64_t)blockIdx.x * 2 * hidden;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = a + j * appliers;
    if (v < nvec) {
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        *reinterpret_cast<float4*>(pr + (int64_t)v * E + e) =
            make_float4(ag[j][e], ag[j][e + 1], ag[j][e + 2], ag[j][e + 3]);
        *reinterpret_cast<float4*>(pr + hidden + (int64_t)v * E + e) =
            make_float4(ab[j][e], ab[j][e + 1], ab[j][e + 2], ab[j][e + 3]);
      }
    }
  }
}

// Backward for wide rows (2048 vectors: 16384 16-bit or 8192 fp32 elements)
// that bwd_tma cannot hold: its fp32 gain copy and two ring stages would
// fill shared memory, and two vectors per applier do not cover the row.
// Here the gains are staged once in their own dtype (one bulk copy, behind
// the ring's three stages: up to kWideBudget of shared memory), and each
// applier owns four vectors with its gains kept packed in registers
// (widened at each use) next to its fp32 dw accumulators; the block is
// limited to 736 threads, which leaves 88 registers a thread.  A row's dot
// is split over a team of kWideTeam reducer warps (three teams, each taking
// every third row) that meet at their own named barrier.  The row dot is
// what paces these rows: measured on GB300, a backward whose reducers skip
// it runs 25 % faster, one whose appliers skip theirs 10 % -- hence the
// shared-memory gains (read through L1 every row they cost a load from L2
// a vector).
constexpr int kWideThreads = 736;
constexpr int kWideTeam = 2;  // warps a reducer team (three teams)
// Dynamic shared memory of the wide and split kernels: ring and gain copy
// (the opt-in limit is 227 KB a block, static shared memory included).
constexpr int kWideBudget = 225 * 1024;

template <typename T>
__global__ void __launch_bounds__(kWideThreads, 1) bwd_tma_wide(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ rstd, T* __restrict__ dx, float* __restrict__ partial,
    int64_t rows, int hidden, float off, int stages, int reducers, int brows) {
  constexpr int E = Traits<T>::kVec;
  constexpr int VPT = 4;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Pipe pipe;
  __shared__ uint64_t gbar;  // the gain copy landed
  const int row_bytes = hidden * (int)sizeof(T);
  const int stride = (2 * row_bytes + 127) / 128 * 128;
  unsigned char* ring = smem;
  const uint4* gsm = reinterpret_cast<const uint4*>(smem + (size_t)stages * stride);
  const int appliers = blockDim.x - 32 * (1 + reducers * kWideTeam);
  const RowBlocks blk = row_blocks(rows, brows, blockIdx.x, gridDim.x);
  const Rows rw{blk.r0, blk.n};
  const int n = rw.n;
  init_pipe(pipe, stages, appliers / 32);
  if (threadIdx.x == 0) {
    mbar_init(&gbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  // the first row into L2 (prefetch_l2; one row: a whole ring was slower)
  if (threadIdx.x == 0 && n > 0) {
    prefetch_l2(x + rw.r0 * hidden, (uint32_t)row_bytes);
    prefetch_l2(dy + rw.r0 * hidden, (uint32_t)row_bytes);
  }
  pdl_wait();
  volatile int* abort = &pipe.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = hidden / E;
  const int doff = row_bytes / 16;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&gbar, (uint32_t)row_bytes);
      bulk_load(smem + (size_t)stages * stride, gamma, (uint32_t)row_bytes, &gbar);
      const void* const src[2] = {x, dy};
      produce<2>(pipe, ring, stride, stages, src, rw, (uint32_t)row_bytes, abort);
      drain_phase(&gbar, 0);
    }
    return;
  }

  if (warp <= reducers * kWideTeam) {
    __shared__ float tred[3][2][kWideTeam];
    const int d = (warp - 1) / kWideTeam, tw = (warp - 1) % kWideTeam;
    const int nthr = 32 * kWideTeam;
    int tpar = 0;
    RingPos pos{0, 0u};
    pos.advance(d, stages);
    const bool gok = d < n ? __all_sync(0xffffffffu, wait_phase(&gbar, 0, abort)) : true;
    for (int i = d; i < n; i += reducers) {
      const float rs = __ldg(rstd + rw.row(i));
      // the team decides together: a named barrier that ANDs every warp's wait
      const bool ok =
          __all_sync(0xffffffffu, wait_phase(&pipe.full[pos.stage], pos.phase, abort)) && gok;
      uint32_t all_ok;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\t"
          "setp.ne.u32 p, %1, 0;\n\t"
          "bar.red.and.pred q, %2, %3, p;\n\t"
          "selp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(all_ok)
          : "r"((uint32_t)ok), "r"(2 + d), "r"(nthr)
          : "memory");
      if (!all_ok) return;
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)pos.stage * stride);
      float part[E];
#pragma unroll
      for (int e = 0; e < E; ++e) part[e] = 0.f;
      for (int v = tw * 32 + lane; v < nvec; v += nthr) {
        float xf[E], df[E], gf[E];
        unpack<T>(st[v], xf);
        unpack<T>(st[doff + v], df);
        unpack<T>(gsm[v], gf);
#pragma unroll
        for (int e = 0; e < E; ++e) part[e] = fmaf(df[e] * (gf[e] + off), xf[e], part[e]);
      }
      const float wdot = warp_sum(pairwise<E>(part));
      float* slot = tred[d][tpar];
      tpar ^= 1;
      if (lane == 0) slot[tw] = wdot;
      asm volatile("bar.sync %0, %1;" ::"r"(2 + d), "r"(nthr) : "memory");
      if (tw == 0 && lane == 0) {
        float dot = 0.f;
        for (int w = 0; w < kWideTeam; ++w) dot += slot[w];
        pipe.stat[pos.stage] = dot * rs / (float)hidden;
        mbar_arrive(&pipe.red[pos.stage]);
        mbar_arrive(&pipe.empty[pos.stage]);
      }
      pos.advance(reducers, stages);
    }
    return;
  }

  const int a = threadIdx.x - 32 * (1 + reducers * kWideTeam);
  uint4 gp[VPT];
  float acc[VPT][E];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = a + j * appliers;
    gp[j] = v < nvec ? ld_shared_ro(gamma + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[j][e] = 0.f;
  }
  RingPos pos{0, 0u};
  float rs_next = n > 0 ? __ldg(rstd + rw.row(0)) : 0.f;
  int64_t part = blk.b0;
  for (int i = 0; i < n; ++part) {
   for (const int end = blk.block_end(i); i < end; ++i) {
    const float rs = rs_next;
    if (i + 1 < n) rs_next = __ldg(rstd + rw.row(i + 1));
    bool ok = wait_phase(&pipe.red[pos.stage], pos.phase, abort);
    ok = ok && wait_phase(&pipe.full[pos.stage], pos.phase, abort);
    if (!__all_sync(0xffffffffu, ok)) return;
    const float c = pipe.stat[pos.stage];
    const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)pos.stage * stride);
    T* dxr = dx + rw.row(i) * hidden;
    // widen the packed gains at each use rather than holding them widened
#pragma unroll
    for (int j = 0; j < VPT; ++j) opaque(gp[j]);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = a + j * appliers;
      if (v < nvec) {
        float xf[E], df[E], gf[E], o[E];
        unpack<T>(st[v], xf);
        unpack<T>(st[doff + v], df);
        unpack<T>(gp[j], gf);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float xh = xf[e] * rs;
          acc[j][e] = fmaf(df[e], xh, acc[j][e]);
          o[e] = fmaf(-xh, c, df[e] * (gf[e] + off)) * rs;
        }
        st_vec(dxr + (int64_t)v * E, pack<T>(o));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pipe.empty[pos.stage]);
    pos.advance(1, stages);
   }
    flush_partial<VPT, E>(acc, partial, part, hidden, 0, a, appliers, nvec);
  }
}

std::mutex g_attr_mutex;
struct AttrEntry {
  const void* func;
  int device;
};
AttrEntry g_attr_done[128];
int g_attr_n = 0;

// Raise a kernel's dynamic shared memory limit, once per (kernel, device).
cudaError_t allow_smem(const void* kern, int bytes = kRingBudget) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  for (int i = 0; i < g_attr_n; ++i)
    if (g_attr_done[i].func == kern && g_attr_done[i].device == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && g_attr_n < 128) g_attr_done[g_attr_n++] = AttrEntry{kern, dev};
  return e;
}

// Applier threads: the fewest vectors per thread that keep them within
// `max_a` threads, at most `max_vpt`.  Returns 0 when no split fits.
int pick_vpt(int nvec, int max_a, int max_vpt, int* appliers) {
  int vpt = 1;
  while (vpt < max_vpt && (nvec + vpt - 1) / vpt > max_a) vpt <<= 1;
  const int a = ((nvec + vpt - 1) / vpt + 31) / 32 * 32;
  if (a > max_a) return 0;
  *appliers = a;
  return vpt;
}

// Stage and reducer counts from the number of stages that fit: every
// reducer owns the same number of stages (see the note at the top).
void split_stages(int fit, int* stages, int* reducers) {
  if (fit > kMaxStages) fit = kMaxStages;
  if (fit <= kMaxReducers) {
    *stages = fit;
    *reducers = fit;
    return;
  }
  // the most stages that some reducer count from 8 to 12 divides; among
  // equals, the most reducers (a row's reduction is on the critical path of
  // its outputs, so more reducers beat a few more stages)
  *stages = 0;
  for (int r = 8; r <= kMaxReducers; ++r) {
    const int st = fit / r * r;
    if (st >= *stages) {
      *stages = st;
      *reducers = r;
    }
  }
}

// Forward ring of rows up to 16 KB: at most kFwdRingBytes of them in
// flight a CTA.  Measured on GB300, deeper rings slow the forward (more
// reads in flight beside its stores): 4096 x 4096 bf16 0.785 of the copy
// bandwidth with 24 stages, 0.809 with 12; 16384 x 8192 bf16 0.877 with 12
// stages, 0.903 with 6; its FP8 forward 0.887 with 12, 0.92 with 6.  The
// FP8 forward of rows of 16 KB, whose rows go round-robin, takes the full
// ring: 16384 x 8192 bf16 63.3 -> 59.4 us (steps 183.1 -> 178.7 us),
// where the full ring alone gained 0.4 % and round-robin rows alone lost
// 1.4 %; narrower FP8 rows keep kFwdRingBytes (4096 x 4096 bf16 10.75
// against 11.12 us with the full ring).
constexpr int kFwdRingBytes = 96 * 1024;

int grid_for(int64_t rows, int64_t cap, cudaError_t* err) {
  int dev = 0;
  if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return 0;
  int64_t g = sm_count(dev);
  if (g > rows) g = rows;
  if (g > cap) g = cap;
  return (int)g;
}

template <typename T, int VPT, bool F8>
cudaError_t launch_fwd_tma_vf(const FwdArgs& a, int appliers, int stages, int reducers, int grid,
                              cudaStream_t s) {
  auto kern = fwd_tma<T, VPT, F8, false>;
  // rows of 16 KB and more need two vectors an applier at least
  if constexpr (VPT >= 2)
    if (a.hidden * (int)sizeof(T) >= kRoundRobinBytes) kern = fwd_tma<T, VPT, F8, true>;
  const int stride = (a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  cudaError_t e = allow_smem((const void*)kern);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(32 * (1 + reducers) + appliers),
                       (size_t)stages * stride, s, 1, static_cast<const T*>(a.x),
                       static_cast<const T*>(a.gamma), a.y, a.rstd, a.rows, a.hidden, a.eps,
                       a.offset ? 1.f : 0.f, a.twice, a.scale, stages, reducers);
}

template <typename T, int VPT>
cudaError_t launch_fwd_tma_v(const FwdArgs& a, int appliers, int stages, int reducers, int grid,
                             cudaStream_t s) {
  return a.fp8 ? launch_fwd_tma_vf<T, VPT, true>(a, appliers, stages, reducers, grid, s)
               : launch_fwd_tma_vf<T, VPT, false>(a, appliers, stages, reducers, grid, s);
}

template <typename T>
bool try_fwd_split_t(const FwdArgs& a, cudaStream_t s, cudaError_t* err);

template <typename T>
bool try_fwd_tma_t(const FwdArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int E = Traits<T>::kVec;
  const int stride = (a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  int stages = 0, reducers = 0;
  const bool full_ring = stride > 16 * 1024 ||
                         (a.fp8 && a.hidden * (int)sizeof(T) >= kRoundRobinBytes);
  split_stages((full_ring ? kRingBudget : kFwdRingBytes) / stride, &stages,
               &reducers);
  // rows too wide for this kernel go over a cluster (fwd_tma_split)
  if (stages < 3) return try_fwd_split_t<T>(a, s, err);
  int appliers = 0;
  // at most 4 vectors per applier (gains in fp32 registers)
  const int vpt = pick_vpt(a.hidden / E, kMaxThreads - 32 * (1 + reducers), 4, &appliers);
  if (vpt == 0) return try_fwd_split_t<T>(a, s, err);
  const int grid = grid_for(a.rows, a.rows, err);
  if (*err != cudaSuccess) return true;
  switch (vpt) {
    case 1: *err = launch_fwd_tma_v<T, 1>(a, appliers, stages, reducers, grid, s); break;
    case 2: *err = launch_fwd_tma_v<T, 2>(a, appliers, stages, reducers, grid, s); break;
    default: *err = launch_fwd_tma_v<T, 4>(a, appliers, stages, reducers, grid, s); break;
  }
  return true;
}

template <typename T, int VPT>
cudaError_t launch_bwd_tma_v(const BwdArgs& a, int appliers, int stages, int reducers,
                             const BlockPlan& bp, cudaStream_t s) {
  auto kern = bwd_tma<T, VPT>;
  const int stride = (2 * a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  const int gain_bytes = (a.hidden * 4 + 127) / 128 * 128;
  cudaError_t e = allow_smem((const void*)kern);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(bp.units), dim3(32 * (1 + reducers) + appliers),
                       (size_t)gain_bytes + (size_t)stages * stride, s, 1,
                       static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                       static_cast<const T*>(a.gamma), a.rstd, static_cast<T*>(a.dx), a.partial,
                       a.rows, a.hidden, a.offset ? 1.f : 0.f, stages, reducers, bp.brows);
}

// The block plan of a persistent backward with one CTA per SM.
BlockPlan bwd_plan(const BwdArgs& a, cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  return plan_blocks(a.rows, a.block_rows, unit_cap(a, sm_count(dev)));
}

// Backward for wide rows over a cluster of csize (2 or 4) CTAs: CTA q of
// the cluster stages, reduces and writes columns [q * N/csize, (q+1) *
// N/csize) of every row of the cluster's contiguous row range, so that a
// ring stage (its parts of x and dy) is small enough for six stages and
// more.  The roles are those of bwd_tma_wide (reducer teams of kWideTeam
// warps, appliers of four vectors with packed gains); a team's part of the
// row dot goes to every CTA of the cluster through distributed shared
// memory -- the team's first warp stores it into each CTA's slot and
// arrives on that CTA's exchange mbarrier -- and every CTA adds the parts
// in rank order.  Exchange slots are double-buffered per team (no CTA can
// start the team's row after next before every CTA has read the current
// one: that row needs every CTA's part of the next).  Every CTA ends with a
// cluster barrier so that no CTA exits while a peer may still store into it.
constexpr int kMaxSplit = 4;

template <typename T, int CS>
__global__ void __launch_bounds__(kWideThreads, 1) bwd_tma_split(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ rstd, T* __restrict__ dx, float* __restrict__ partial,
    int64_t rows, int hidden, float off, int stages, int reducers, int brows) {
  constexpr int csize = CS;
  constexpr int E = Traits<T>::kVec;
  constexpr int VPT = 4;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Pipe pipe;
  __shared__ uint64_t xbar[3][2];
  __shared__ float xch[3][2][CS];
  __shared__ float tred[3][2][kWideTeam];
  __shared__ uint64_t gbar;  // the gain copy landed
  const uint32_t rank = cta_rank();
  const int part = hidden / csize;           // columns a CTA owns
  const int part_bytes = part * (int)sizeof(T);
  const int stride = (2 * part_bytes + 127) / 128 * 128;
  unsigned char* ring = smem;
  const uint4* gsm = reinterpret_cast<const uint4*>(smem + (size_t)stages * stride);
  const int appliers = blockDim.x - 32 * (1 + reducers * kWideTeam);
  const int64_t cid = blockIdx.x / csize, ncl = gridDim.x / csize;
  const RowBlocks blk = row_blocks(rows, brows, cid, ncl);
  const Rows rw{blk.r0, blk.n};
  const int n = rw.n;
  init_pipe(pipe, stages, appliers / 32);
  if (threadIdx.x < 6) mbar_init(&xbar[threadIdx.x / 2][threadIdx.x % 2], csize);
  if (threadIdx.x == 6) mbar_init(&gbar, 1);
  fence_mbar_init();
  __syncthreads();
  cluster_sync();  // the peers' barriers are initialised
  pdl_trigger();
  // the first row's slices into L2 (prefetch_l2; one row: a whole ring was
  // slower)
  if (threadIdx.x == 0 && n > 0) {
    const int64_t c0 = (int64_t)rank * part;
    prefetch_l2(x + rw.row(0) * hidden + c0, (uint32_t)part_bytes);
    prefetch_l2(dy + rw.row(0) * hidden + c0, (uint32_t)part_bytes);
  }
  pdl_wait();
  volatile int* abort = &pipe.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = part / E;                 // vectors of this CTA's columns
  const int doff = part_bytes / 16;
  const int64_t col0 = (int64_t)rank * part; // first column of this CTA

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&gbar, (uint32_t)part_bytes);
      bulk_load(smem + (size_t)stages * stride, gamma + col0, (uint32_t)part_bytes, &gbar);
      const void* const src[2] = {x + col0, dy + col0};
      produce_pitched<2>(pipe, ring, stride, stages, src, rw, (size_t)hidden * sizeof(T),
                         (uint32_t)part_bytes, abort);
      drain_phase(&gbar, 0);
    }
  } else if (warp <= reducers * kWideTeam) {
    const int d = (warp - 1) / kWideTeam, tw = (warp - 1) % kWideTeam;
    const int nthr = 32 * kWideTeam;
    int tpar = 0, par = 0;
    uint32_t xph0 = 0, xph1 = 0;
    bool prev_ok = true;  // the team's last exchange (its first warp)
    RingPos pos{0, 0u};
    pos.advance(d, stages);
    const bool gok = d < n ? __all_sync(0xffffffffu, wait_phase(&gbar, 0, abort)) : true;
    for (int i = d; i < n; i += reducers) {
      const float rs = __ldg(rstd + rw.row(i));
      const bool ok = __all_sync(0xffffffffu, wait_phase(&pipe.full[pos.stage], pos.phase, abort)) &&
                      prev_ok && gok;
      uint32_t all_ok;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\t"
          "setp.ne.u32 p, %1, 0;\n\t"
          "bar.red.and.pred q, %2, %3, p;\n\t"
          "selp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(all_ok)
          : "r"((uint32_t)ok), "r"(2 + d), "r"(nthr)
          : "memory");
      if (!all_ok) break;
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)pos.stage * stride);
      float acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.f;
      for (int v = tw * 32 + lane; v < nvec; v += nthr) {
        float xf[E], df[E], gf[E];
        unpack<T>(st[v], xf);
        unpack<T>(st[doff + v], df);
        unpack<T>(gsm[v], gf);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(df[e] * (gf[e] + off), xf[e], acc[e]);
      }
      const float wdot = warp_sum(pairwise<E>(acc));
      float* slot = tred[d][tpar];
      tpar ^= 1;
      if (lane == 0) slot[tw] = wdot;
      asm volatile("bar.sync %0, %1;" ::"r"(2 + d), "r"(nthr) : "memory");
      if (tw == 0) {
        float mine = 0.f;
        for (int w = 0; w < kWideTeam; ++w) mine += slot[w];
        // send this CTA's part to every CTA of the cluster (itself included)
        if (lane < csize) {
          st_peer(&xch[d][par][rank], (uint32_t)lane, mine);
          mbar_arrive_peer(&xbar[d][par], (uint32_t)lane);
        }
        prev_ok = __all_sync(0xffffffffu,
                             wait_cluster_counted(&xbar[d][par], par ? xph1 : xph0, abort,
                                                  &g_wait_timeouts));
        if (prev_ok) {
          if (par) xph1 ^= 1u; else xph0 ^= 1u;
          float dot = 0.f;
#pragma unroll
          for (int r = 0; r < csize; ++r) dot += xch[d][par][r];
          dot *= rs;
          par ^= 1;
          if (lane == 0) {
            pipe.stat[pos.stage] = dot / (float)hidden;
            mbar_arrive(&pipe.red[pos.stage]);
            mbar_arrive(&pipe.empty[pos.stage]);
          }
        }
      }
      pos.advance(reducers, stages);
    }
  } else {
    const int a = threadIdx.x - 32 * (1 + reducers * kWideTeam);
    uint4 gp[VPT];
    float acc[VPT][E];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = a + j * appliers;
      gp[j] = v < nvec ? ld_shared_ro(gamma + col0 + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[j][e] = 0.f;
    }
    RingPos pos{0, 0u};
    float rs_next = n > 0 ? __ldg(rstd + rw.row(0)) : 0.f;
    bool ok = true;
    int64_t part = blk.b0;
    for (int i = 0; i < n && ok; ++part) {
     for (const int end = blk.block_end(i); i < end && ok; ++i) {
      const float rs = rs_next;
      if (i + 1 < n) rs_next = __ldg(rstd + rw.row(i + 1));
      ok = wait_phase(&pipe.red[pos.stage], pos.phase, abort);
      ok = __all_sync(0xffffffffu, ok && wait_phase(&pipe.full[pos.stage], pos.phase, abort));
      if (!ok) break;
      const float c = pipe.stat[pos.stage];
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)pos.stage * stride);
      T* dxr = dx + rw.row(i) * hidden + col0;
#pragma unroll
      for (int j = 0; j < VPT; ++j) opaque(gp[j]);
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int v = a + j * appliers;
        if (v < nvec) {
          float xf[E], df[E], gf[E], o[E];
          unpack<T>(st[v], xf);
          unpack<T>(st[doff + v], df);
          unpack<T>(gp[j], gf);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float xh = xf[e] * rs;
            acc[j][e] = fmaf(df[e], xh, acc[j][e]);
            o[e] = fmaf(-xh, c, df[e] * (gf[e] + off)) * rs;
          }
          st_vec(dxr + (int64_t)v * E, pack<T>(o));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&pipe.empty[pos.stage]);
      pos.advance(1, stages);
     }
      if (ok) flush_partial<VPT, E>(acc, partial, part, hidden, col0, a, appliers, nvec);
    }
  }
  __syncwarp();
  cluster_sync();  // no peer stores into this CTA after it exits
}

// The split backward: clusters of csize CTAs, the smallest csize (2 or 4)
// whose parts of a row leave at least min_stages ring stages (a multiple of
// the three reducer teams), else the largest that leaves three.  Measured
// on GB300: six stages beat three (16384 fp32: 0.78 of the copy bandwidth
// in clusters of 4 against 0.69 in pairs; 32768 fp16, gains in shared
// memory: 158.7 against 164.1 us).  False when none fits.

template <typename T>
bool try_bwd_split_t(const BwdArgs& a, cudaStream_t s, cudaError_t* err, int64_t* nparts) {
  constexpr int E = Traits<T>::kVec;
  const int reducers = 3;
  const int min_stages = 6;
  int csize = 0, stages = 0, appliers = 0;
  for (int k = 2; k <= kMaxSplit; k *= 2) {
    if (a.hidden % (k * E)) continue;
    const int stride = (2 * (a.hidden / k) * (int)sizeof(T) + 127) / 128 * 128;
    const int gain = ((a.hidden / k) * (int)sizeof(T) + 127) / 128 * 128;
    int st = (kWideBudget - gain) / stride;
    if (st > kMaxStages) st = kMaxStages;
    st -= st % reducers;
    // four vectors an applier (the kernel's packed gains)
    const int app = ((a.hidden / k / E + 3) / 4 + 31) / 32 * 32;
    if (st < 3 || app > kWideThreads - 32 * (1 + reducers * kWideTeam)) continue;
    csize = k;
    stages = st;
    appliers = app;
    if (st >= min_stages) break;
  }
  if (csize == 0) return false;
  const int stride = (2 * (a.hidden / csize) * (int)sizeof(T) + 127) / 128 * 128;
  const int gain = ((a.hidden / csize) * (int)sizeof(T) + 127) / 128 * 128;
  const int threads = 32 * (1 + reducers * kWideTeam) + appliers;
  auto kern = csize == 2 ? bwd_tma_split<T, 2> : bwd_tma_split<T, 4>;
  if ((*err = allow_smem((const void*)kern, kWideBudget)) != cudaSuccess) return true;
  // as many clusters as can be resident at once (one CTA per SM)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)csize);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)stages * stride + gain;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active < 1) {
    cudaGetLastError();
    return false;
  }
  // the SM budget, in clusters
  int dev = 0;
  if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return true;
  const int budget = sm_count(dev) / csize;
  if (active > budget) active = budget > 0 ? budget : 1;
  const BlockPlan bp = plan_blocks(a.rows, a.block_rows, unit_cap(a, active));
  *nparts = bp.nblocks;
  *err = launch_kernel(kern, dim3((unsigned)(csize * bp.units)), dim3(threads),
                       (size_t)stages * stride + gain, s, csize, static_cast<const T*>(a.dy),
                       static_cast<const T*>(a.x), static_cast<const T*>(a.gamma), a.rstd,
                       static_cast<T*>(a.dx), a.partial, a.rows, a.hidden,
                       a.offset ? 1.f : 0.f, stages, reducers, bp.brows);
  return true;
}

// Forward for rows too wide for fwd_tma (its appliers would need more than
// four vectors each, or its ring would hold fewer than three rows): a row is
// split over a cluster of CS (2 or 4) CTAs as in bwd_tma_split -- CTA q
// stages columns [q * N/CS, (q + 1) * N/CS) of every row of the cluster's
// contiguous rows -- so that a stage is small enough for six or more.
// Reducer warp d takes the cluster's rows d, d + R, ...: the sum of squares
// of its slice (as fwd_tma's reducers), sent to every CTA of the cluster
// through distributed shared memory (slot `rank` of the warp's buffer, two
// buffers used in turn, each with an mbarrier that counts the CS arrivals),
// then the CS parts added in rank order, so that every CTA holds the same
// rstd.  A row whose fp32 total overflows takes a second exchange, of the
// rescaled sums (every CTA sees the same total, so all of them take it).
// The double buffer is safe for the same reason as bwd_tma_split's: a CTA
// sends its part of exchange e + 1 only after reading exchange e, so no
// part of exchange e + 2 lands before every CTA has read exchange e.  The
// appliers are fwd_tma's on the CTA's columns, with the gains packed in
// registers.  No role leaves early: every CTA ends at a cluster barrier,
// so that none exits while a peer may still store into its shared memory.
template <int CS>
__device__ __forceinline__ bool exchange_sum(float mine, float (&slot)[CS], uint64_t* bar,
                                             uint32_t& phase, uint32_t rank, int lane,
                                             volatile int* abort, float* total) {
  if (lane < CS) {
    st_peer(&slot[rank], (uint32_t)lane, mine);
    mbar_arrive_peer(bar, (uint32_t)lane);
  }
  if (!__all_sync(0xffffffffu, wait_cluster_counted(bar, phase, abort, &g_wait_timeouts)))
    return false;
  phase ^= 1u;
  float t = 0.f;
#pragma unroll
  for (int r = 0; r < CS; ++r) t += slot[r];
  *total = t;
  return true;
}

template <typename T, int CS, bool F8>
__global__ void __launch_bounds__(kWideThreads, 1) fwd_tma_split(
    const T* __restrict__ x, const T* __restrict__ gamma, void* __restrict__ y,
    float* __restrict__ rstd, int64_t rows, int hidden, float eps, float off, int twice,
    const float* __restrict__ scale, int stages, int reducers) {
  constexpr int E = Traits<T>::kVec;
  constexpr int VPT = 4;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Pipe pipe;
  __shared__ uint64_t xbar[kMaxReducers][2];
  __shared__ float xch[kMaxReducers][2][CS];
  const uint32_t rank = cta_rank();
  const int part = hidden / CS;  // columns a CTA owns
  const int part_bytes = part * (int)sizeof(T);
  const int stride = (part_bytes + 127) / 128 * 128;
  const int appliers = blockDim.x - 32 * (1 + reducers);
  const int64_t cid = blockIdx.x / CS, ncl = gridDim.x / CS;
  const int64_t r0 = cid * rows / ncl;
  const Rows rw{r0, (int)((cid + 1) * rows / ncl - r0)};
  const int n = rw.n;
  init_pipe(pipe, stages, appliers / 32);
  if (threadIdx.x < 2 * kMaxReducers) mbar_init(&xbar[threadIdx.x / 2][threadIdx.x % 2], CS);
  fence_mbar_init();
  __syncthreads();
  cluster_sync();  // the peers' barriers are initialised
  pdl_trigger();
  if (threadIdx.x == 0) {  // the first rows' slices into L2 (prefetch_l2)
    const int64_t c0 = (int64_t)rank * part;
    for (int i = 0; i < n && i < kPrefetchRows; ++i)
      prefetch_l2(x + rw.row(i) * hidden + c0, (uint32_t)part_bytes);
  }
  pdl_wait();
  volatile int* abort = &pipe.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = part / E;                  // vectors of this CTA's columns
  const int64_t col0 = (int64_t)rank * part;  // first column of this CTA

  if (warp == 0) {
    if (lane == 0) {
      const void* const src[1] = {x + col0};
      produce_pitched<1>(pipe, smem, stride, stages, src, rw, (size_t)hidden * sizeof(T),
                         (uint32_t)part_bytes, abort);
    }
  } else if (warp <= reducers) {
    const int d = warp - 1;
    int par = 0;
    uint32_t ph[2] = {0u, 0u};
    RingPos pos{0, 0u};
    pos.advance(d, stages);
    for (int i = d; i < n; i += reducers) {
      if (!__all_sync(0xffffffffu, wait_phase(&pipe.full[pos.stage], pos.phase, abort))) break;
      const uint4* st = reinterpret_cast<const uint4*>(smem + (size_t)pos.stage * stride);
      float acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float f[E];
        unpack<T>(st[v], f);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(f[e], f[e], acc[e]);
      }
      float ss;
      if (!exchange_sum<CS>(warp_sum(pairwise<E>(acc)), xch[d][par], &xbar[d][par], ph[par], rank,
                            lane, abort, &ss))
        break;
      par ^= 1;
      float rs = rstd_of(ss / (float)hidden, eps);
      if (isinf(ss)) {  // the fp32 sum of squares overflowed (see kOverflowScale)
        float s2 = 0.f;
        for (int v = lane; v < nvec; v += 32) {
          float f[E];
          unpack<T>(st[v], f);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float t = f[e] * kOverflowScale;
            s2 = fmaf(t, t, s2);
          }
        }
        float tot;
        if (!exchange_sum<CS>(warp_sum(s2), xch[d][par], &xbar[d][par], ph[par], rank, lane,
                              abort, &tot))
          break;
        par ^= 1;
        rs = rstd_rescaled(tot, hidden, eps);
      }
      if (lane == 0) {
        if (rank == 0) rstd[rw.row(i)] = rs;
        pipe.stat[pos.stage] = rs;
        mbar_arrive(&pipe.red[pos.stage]);
        mbar_arrive(&pipe.empty[pos.stage]);
      }
      pos.advance(reducers, stages);
    }
  } else {
    const int a = threadIdx.x - 32 * (1 + reducers);
    const float sc = F8 ? __ldg(scale) : 1.f;
    uint4 gp[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = a + j * appliers;
      gp[j] = v < nvec ? ld_shared_ro(gamma + col0 + (int64_t)v * E) : make_uint4(0, 0, 0, 0);
    }
    RingPos pos{0, 0u};
    for (int i = 0; i < n; ++i) {
      bool ok = wait_phase(&pipe.red[pos.stage], pos.phase, abort);
      ok = ok && wait_phase(&pipe.full[pos.stage], pos.phase, abort);
      if (!__all_sync(0xffffffffu, ok)) break;
      const float rs = pipe.stat[pos.stage];
      const uint4* st = reinterpret_cast<const uint4*>(smem + (size_t)pos.stage * stride);
      const int64_t yoff = rw.row(i) * hidden + col0;
      // widen the packed gains at each use rather than holding them widened
#pragma unroll
      for (int j = 0; j < VPT; ++j) opaque(gp[j]);
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int v = a + j * appliers;
        if (v < nvec) {
          float f[E], g[E], o[E];
          unpack<T>(st[v], f);
          unpack<T>(gp[j], g);
          if constexpr (F8) {
            // ((x * rstd) * gain) * scale in fp32, one conversion to E4M3
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = ((f[e] * rs) * (g[e] + off)) * sc;
            st_e4m3<E>(static_cast<unsigned char*>(y) + yoff + (int64_t)v * E, o);
          } else {
            if (twice) {
#pragma unroll
              for (int e = 0; e < E; ++e) o[e] = round_trip<T>(f[e] * rs) * (g[e] + off);
            } else {
#pragma unroll
              for (int e = 0; e < E; ++e) o[e] = (f[e] * rs) * (g[e] + off);
            }
            st_vec(static_cast<T*>(y) + yoff + (int64_t)v * E, pack<T>(o));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&pipe.empty[pos.stage]);
      pos.advance(1, stages);
    }
  }
  __syncwarp();
  cluster_sync();  // no peer stores into this CTA after it exits
}

// The split forward: clusters of CS CTAs, the smallest CS (2 or 4) whose
// parts of a row leave at least six ring stages, else the largest that
// leaves three, with four vectors an applier; false when none fits.
template <typename T, bool F8>
bool try_fwd_split_tf(const FwdArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int E = Traits<T>::kVec;
  int csize = 0, stages = 0, reducers = 0, appliers = 0;
  for (int k = 2; k <= kMaxSplit; k *= 2) {
    if (a.hidden % (k * E)) continue;
    const int stride = ((int)(a.hidden / k) * (int)sizeof(T) + 127) / 128 * 128;
    int st = 0, r = 0;
    split_stages(kRingBudget / stride, &st, &r);
    const int app = ((int)(a.hidden / k / E + 3) / 4 + 31) / 32 * 32;
    if (st < 3 || app > kWideThreads - 32 * (1 + r)) continue;
    csize = k;
    stages = st;
    reducers = r;
    appliers = app;
    if (st >= 6) break;
  }
  if (csize == 0) return false;
  const int stride = ((int)(a.hidden / csize) * (int)sizeof(T) + 127) / 128 * 128;
  const int threads = 32 * (1 + reducers) + appliers;
  auto kern = csize == 2 ? fwd_tma_split<T, 2, F8> : fwd_tma_split<T, 4, F8>;
  if ((*err = allow_smem((const void*)kern)) != cudaSuccess) return true;
  // as many clusters as can be resident at once (one CTA per SM)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)csize);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)stages * stride;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active < 1) {
    cudaGetLastError();
    return false;
  }
  int dev = 0;
  if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return true;
  const int budget = sm_count(dev) / csize;  // the SM budget, in clusters
  if (active > budget) active = budget > 0 ? budget : 1;
  const int64_t clusters = a.rows < active ? a.rows : active;
  *err = launch_kernel(kern, dim3((unsigned)(csize * clusters)), dim3(threads),
                       (size_t)stages * stride, s, csize, static_cast<const T*>(a.x),
                       static_cast<const T*>(a.gamma), a.y, a.rstd, a.rows, a.hidden, a.eps,
                       a.offset ? 1.f : 0.f, a.twice, a.scale, stages, reducers);
  return true;
}

template <typename T>
bool try_fwd_split_t(const FwdArgs& a, cudaStream_t s, cudaError_t* err) {
  return a.fp8 ? try_fwd_split_tf<T, true>(a, s, err) : try_fwd_split_tf<T, false>(a, s, err);
}

// The wide-row backward: three stages with a packed gain copy and four
// vectors per applier within kWideThreads threads; false when that does not
// fit either.
template <typename T>
bool try_bwd_wide_t(const BwdArgs& a, cudaStream_t s, cudaError_t* err, int64_t* nparts) {
  constexpr int E = Traits<T>::kVec;
  const int stride = (2 * a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  const int gain = (a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  const int stages = 3 * stride + gain <= kWideBudget ? 3 : 0, reducers = 3;
  if (stages < 3) return false;
  int appliers = 0;
  if (pick_vpt(a.hidden / E, kWideThreads - 32 * (1 + reducers * kWideTeam), 4, &appliers) != 4)
    return false;
  const BlockPlan bp = bwd_plan(a, err);
  if (*err != cudaSuccess) return true;
  *nparts = bp.nblocks;
  auto kern = bwd_tma_wide<T>;
  if ((*err = allow_smem((const void*)kern, kWideBudget)) != cudaSuccess) return true;
  *err = launch_kernel(kern, dim3(bp.units), dim3(32 * (1 + reducers * kWideTeam) + appliers),
                       (size_t)stages * stride + gain, s, 1, static_cast<const T*>(a.dy),
                       static_cast<const T*>(a.x), static_cast<const T*>(a.gamma), a.rstd,
                       static_cast<T*>(a.dx), a.partial, a.rows, a.hidden,
                       a.offset ? 1.f : 0.f, stages, reducers, bp.brows);
  return true;
}

// Rows per stage of the narrow-row backward: four rows up to 2 KB, two up to
// 4 KB, else one (bwd_tma); with caller-sized blocks, a divisor of the block.
int rows_per_stage(int64_t row_bytes, int64_t block_rows) {
  int k = row_bytes <= 2048 ? 4 : row_bytes <= 4096 ? 2 : 1;
  if (block_rows > 0)
    while (k > 1 && block_rows % k != 0) k /= 2;
  return k;
}

template <typename T, int K, bool HALF>
bool try_bwd_rows_k(const BwdArgs& a, cudaStream_t s, cudaError_t* err, int64_t* nparts) {
  constexpr int E = Traits<T>::kVec;
  const int stride = (2 * K * a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  const int gain_bytes = (a.hidden * 4 + 127) / 128 * 128;
  int stages = 0, reducers = 0;
  split_stages((kRingBudget - gain_bytes) / stride, &stages, &reducers);
  // a slice of every row an applier (bwd_tma_rows)
  const int appliers = ((int)(a.hidden / (HALF ? E / 2 : E)) + 31) / 32 * 32;
  if (stages < 3 || appliers > kMaxThreads - 32 * (1 + reducers)) return false;
  const BlockPlan bp = bwd_plan(a, err);
  if (*err != cudaSuccess) return true;
  *nparts = bp.nblocks;
  auto kern = bwd_tma_rows<T, K, HALF>;
  if ((*err = allow_smem((const void*)kern)) != cudaSuccess) return true;
  *err = launch_kernel(kern, dim3(bp.units), dim3(32 * (1 + reducers) + appliers),
                       (size_t)gain_bytes + (size_t)stages * stride, s, 1,
                       static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                       static_cast<const T*>(a.gamma), a.rstd, static_cast<T*>(a.dx), a.partial,
                       a.rows, a.hidden, a.offset ? 1.f : 0.f, stages, reducers, bp.brows);
  return true;
}

template <typename T>
bool try_bwd_tma_t(const BwdArgs& a, cudaStream_t s, cudaError_t* err, int64_t* nparts) {
  constexpr int E = Traits<T>::kVec;
  // 8-byte applier slices for rows up to 2 KB, 16-byte ones above
  const bool half = a.hidden * (int64_t)sizeof(T) <= 2048;
  switch (rows_per_stage(a.hidden * (int64_t)sizeof(T), a.block_rows)) {
    case 4:
      if (try_bwd_rows_k<T, 4, true>(a, s, err, nparts)) return true;
      break;
    case 2:
      if (half ? try_bwd_rows_k<T, 2, true>(a, s, err, nparts)
               : try_bwd_rows_k<T, 2, false>(a, s, err, nparts))
        return true;
      break;
    default:
      break;
  }
  const int stride = (2 * a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  const int gain_bytes = (a.hidden * 4 + 127) / 128 * 128;
  int stages = 0, reducers = 0;
  split_stages((kRingBudget - gain_bytes) / stride, &stages, &reducers);
  int appliers = 0;
  // at most 2 vectors per applier: gains and dw accumulators in registers
  const int vpt = stages < 3 ? 0
                             : pick_vpt(a.hidden / E, kMaxThreads - 32 * (1 + reducers), 2,
                                        &appliers);
  if (vpt == 0) return try_bwd_wide_t<T>(a, s, err, nparts) || try_bwd_split_t<T>(a, s, err, nparts);
  const BlockPlan bp = bwd_plan(a, err);
  if (*err != cudaSuccess) return true;
  *nparts = bp.nblocks;
  if (vpt == 1)
    *err = launch_bwd_tma_v<T, 1>(a, appliers, stages, reducers, bp, s);
  else
    *err = launch_bwd_tma_v<T, 2>(a, appliers, stages, reducers, bp, s);
  return true;
}


template <typename T, int VPT>
cudaError_t launch_ln_fwd_tma_v(const LnFwdArgs& a, int appliers, int stages, int reducers,
                                int grid, cudaStream_t s) {
  auto kern = ln_fwd_tma<T, VPT, false>;
  if constexpr (VPT >= 2)
    if (a.hidden * (int)sizeof(T) >= kRoundRobinBytes) kern = ln_fwd_tma<T, VPT, true>;
  const int stride = (a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  cudaError_t e = allow_smem((const void*)kern);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(32 * (1 + reducers) + appliers),
                       (size_t)stages * stride, s, 1, static_cast<const T*>(a.x),
                       static_cast<const T*>(a.gamma), static_cast<const T*>(a.beta),
                       static_cast<T*>(a.y), a.mean, a.rstd, a.rows, a.hidden, a.eps, stages,
                       reducers);
}

template <typename T>
bool try_ln_fwd_tma_t(const LnFwdArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int E = Traits<T>::kVec;
  const int stride = (a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  int stages = 0, reducers = 0;
  split_stages(kRingBudget / stride, &stages, &reducers);
  if (stages < 3) return false;
  int appliers = 0;
  const int vpt = pick_vpt(a.hidden / E, kMaxThreads - 32 * (1 + reducers), 4, &appliers);
  if (vpt == 0) return false;
  const int grid = grid_for(a.rows, a.rows, err);
  if (*err != cudaSuccess) return true;
  switch (vpt) {
    case 1: *err = launch_ln_fwd_tma_v<T, 1>(a, appliers, stages, reducers, grid, s); break;
    case 2: *err = launch_ln_fwd_tma_v<T, 2>(a, appliers, stages, reducers, grid, s); break;
    default: *err = launch_ln_fwd_tma_v<T, 4>(a, appliers, stages, reducers, grid, s); break;
  }
  return true;
}

template <typename T, int VPT>
cudaError_t launch_ln_bwd_tma_v(const LnBwdArgs& a, int appliers, int stages, int reducers,
                                int grid, cudaStream_t s) {
  auto kern = ln_bwd_tma<T, VPT>;
  const int stride = (2 * a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  const int gain_bytes = (a.hidden * 4 + 127) / 128 * 128;
  cudaError_t e = allow_smem((const void*)kern);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(32 * (1 + reducers) + appliers),
                       (size_t)gain_bytes + (size_t)stages * stride, s, 1,
                       static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                       static_cast<const T*>(a.gamma), a.mean, a.rstd, static_cast<T*>(a.dx),
                       a.partial, a.rows, a.hidden, stages, reducers);
}

template <typename T>
bool try_ln_bwd_tma_t(const LnBwdArgs& a, cudaStream_t s, cudaError_t* err, int* nparts) {
  constexpr int E = Traits<T>::kVec;
  const int stride = (2 * a.hidden * (int)sizeof(T) + 127) / 128 * 128;
  const int gain_bytes = (a.hidden * 4 + 127) / 128 * 128;
  int stages = 0, reducers = 0;
  split_stages((kRingBudget - gain_bytes) / stride, &stages, &reducers);
  if (stages < 3) return false;
  int appliers = 0;
  // at most 2 vectors per applier: two fp32 accumulator sets in registers
  const int vpt = pick_vpt(a.hidden / E, kMaxThreads - 32 * (1 + reducers), 2, &appliers);
  if (vpt == 0) return false;
  if (vpt == 2 && 32 * (1 + reducers) + appliers > kLnBwd2Threads) return false;
  const int grid = grid_for(a.rows, a.max_partials, err);
  if (*err != cudaSuccess) return true;
  *nparts = grid;
  if (vpt == 1)
    *err = launch_ln_bwd_tma_v<T, 1>(a, appliers, stages, reducers, grid, s);
  else
    *err = launch_ln_bwd_tma_v<T, 2>(a, appliers, stages, reducers, grid, s);
  return true;
}

}  // namespace

bool try_launch_fwd_tma(int dtype, const FwdArgs& a, cudaStream_t s, cudaError_t* err) {
  if (!a.vec_ok) return false;
  switch (dtype) {
    case 0: return try_fwd_tma_t<float>(a, s, err);
    case 1: return try_fwd_tma_t<__nv_bfloat16>(a, s, err);
    default: return try_fwd_tma_t<__half>(a, s, err);
  }
}

bool try_launch_bwd_tma(int dtype, const BwdArgs& a, cudaStream_t s, cudaError_t* err,
                        int64_t* nparts) {
  if (!a.vec_ok) return false;
  switch (dtype) {
    case 0: return try_bwd_tma_t<float>(a, s, err, nparts);
    case 1: return try_bwd_tma_t<__nv_bfloat16>(a, s, err, nparts);
    default: return try_bwd_tma_t<__half>(a, s, err, nparts);
  }
}

bool try_launch_ln_fwd_tma(int dtype, const LnFwdArgs& a, cudaStream_t s, cudaError_t* err) {
  if (!a.vec_ok) return false;
  switch (dtype) {
    case 0: return try_ln_fwd_tma_t<float>(a, s, err);
    case 1: return try_ln_fwd_tma_t<__nv_bfloat16>(a, s, err);
    default: return try_ln_fwd_tma_t<__half>(a, s, err);
  }
}

bool try_launch_ln_bwd_tma(int dtype, const LnBwdArgs& a, cudaStream_t s, cudaError_t* err,
                           int* nparts) {
  if (!a.vec_ok) return false;
  switch (dtype) {
    case 0: return try_ln_bwd_tma_t<float>(a, s, err, nparts);
    case 1: return try_ln_bwd_tma_t<__nv_bfloat16>(a, s, err, nparts);
    default: return try_ln_bwd_tma_t<__half>(a, s, err, nparts);
  }
}

cudaError_t read_wait_timeouts(unsigned int* out) {
  unsigned int mine = 0, other = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&mine, g_wait_timeouts, sizeof(unsigned int));
  if (e == cudaSuccess) e = read_gn_wait_timeouts(&other);
  *out = mine + other;
  return e;
}

}  // namespace rmsn

extern "C" int rms_norm_wait_timeouts(unsigned int* count) {
  if (!count) return RMSN_ERR_NULL;
  return rmsn::read_wait_timeouts(count) == cudaSuccess ? RMSN_OK : RMSN_ERR_CUDA;
}
