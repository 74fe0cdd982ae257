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
//   1. a persistent row kernel.  The rows are cut into blocks (RowBlocks in
//      common.cuh): one per CTA, the rows split evenly, for rms_norm_bwd;
//      `brows` rows each, whole blocks dealt to the CTAs, for the
//      fixed-block backward.  Each thread owns a fixed set of columns, keeps
//      their gains and their fp32 dw accumulators in registers, and at the
//      end of every block writes them as that block's partial row of the
//      workspace.  The next row's x, dy and rstd are loaded while the
//      current row is reduced.
//   2. dw_finalize (or, for the fixed-block backward, dw_chunk_sums): the
//      partial rows added in a fixed order, launched as a programmatic
//      dependent launch so that its launch overlaps the tail of kernel 1.
// A block's partial depends only on its rows, and every sum has a fixed
// order: repeated calls are bit-identical, and the fixed-block backward's
// chunk sums do not change when the same rows are split over more or fewer
// CTAs, or over several calls along whole chunks.
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
    int64_t rows, int hidden, float off, int brows) {
  constexpr int E = Traits<T>::kVec;
  __shared__ float red[64];
  // Let the finalize kernel be scheduled now; it waits for this grid to
  // complete before reading the partials.
  pdl_trigger();
  pdl_wait();
  const int nvec = hidden / E;
  const RowBlocks rw = row_blocks(rows, brows, blockIdx.x, gridDim.x);
  const int64_t r0 = rw.r0, r1 = rw.r0 + rw.n;
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
  int64_t part = rw.b0;
  for (int64_t r = r0; r < r1; ++part) {
   for (const int64_t end = r0 + rw.block_end((int)(r - r0)); r < end; ++r) {
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
    flush_partial<VPT, E>(acc, partial, part, hidden, 0, threadIdx.x, blockDim.x, nvec);
  }
}

// Any alignment and width: scalar loads; the partial row lives in the
// workspace and each thread updates only its own columns.
template <typename T>
__global__ void __launch_bounds__(256) bwd_scalar(
    const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
    const float* __restrict__ rstd, T* __restrict__ dx, float* __restrict__ partial,
    int64_t rows, int hidden, float off, int brows) {
  __shared__ float red[64];
  pdl_trigger();
  pdl_wait();
  const RowBlocks rw = row_blocks(rows, brows, blockIdx.x, gridDim.x);
  const int64_t r0 = rw.r0, r1 = rw.r0 + rw.n;
  int parity = 0;
  for (int64_t r = r0; r < r1; ++r) {
    // the block's partial row; its first row starts the sums
    const int64_t in_block = (r - r0) % rw.brows;
    float* pr = partial + (rw.b0 + (r - r0) / rw.brows) * (int64_t)hidden;
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
      pr[j] = fmaf(df, xh, in_block == 0 ? 0.f : pr[j]);
    }
  }
}

// Two fixed summation orders of the partial rows [nparts, ncols].
//
// dw_finalize (every backward's own reduction): lane t of 16 adds rows t,
// t + 16, t + 32, ... in increasing order, then lane 0 adds the 16 lane
// sums in order.  The order depends only on nparts.  Blocks of 32 columns
// x 16 lanes (512 threads): measured on GB300 behind the row kernels, this
// shape -- loads in flight at once, one barrier, one short chain in shared
// memory -- beat every form of a pairwise tree (per-thread trees of 32 loads,
// trees across lanes through shared memory, warp-shuffle trees after a
// transpose) by 1 to 3 us a call.
//
// dw_chunk_sums (the fixed-block backward): the rows form chunks of
// kChunkParts = 32 consecutive rows (the last may be shorter); chunk c's sum
// is ((s_0 + s_1) + ...) + s_15 with s_t = row 32c + t + row 32c + t + 16 (a
// missing row counts as +0).  A chunk's sum depends on its 32 rows alone,
// so a split of the rows into runs of whole chunks can form them
// separately; dw_chunk_totals then adds chunk sums in chunk order.
constexpr int kFinLanes = 16;

__global__ void __launch_bounds__(32 * kFinLanes) dw_finalize(const float* __restrict__ partial,
                                                             int64_t nparts, int ncols,
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
    for (int64_t b = ty; b < nparts; b += kFinLanes) a += partial[b * ncols + j];
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

// Chunk sums in passes of kPassChunks chunks: lane t forms s_t of every
// chunk of the pass (its two loads per chunk all in flight at once), lanes
// 0 .. nc-1 each add one chunk's 16 values in order, and the sums go to
// chunks[c][j].
constexpr int kPassChunks = 8;

__global__ void __launch_bounds__(32 * kFinLanes) dw_chunk_sums(const float* __restrict__ partial,
                                                               int64_t nparts, int ncols,
                                                               float* __restrict__ chunks) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s[kPassChunks][kFinLanes][33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int j = blockIdx.x * 32 + tx;
  const bool in = j < ncols;
  const int64_t nchunks = (nparts + kChunkParts - 1) / kChunkParts;
  for (int64_t g0 = 0; g0 < nchunks; g0 += kPassChunks) {
    const int nc = (int)(nchunks - g0 < kPassChunks ? nchunks - g0 : kPassChunks);
#pragma unroll
    for (int c = 0; c < kPassChunks; ++c) {
      const int64_t r = (g0 + c) * kChunkParts + ty;
      const float lo = (c < nc && in && r < nparts) ? partial[r * ncols + j] : 0.f;
      const float hi = (c < nc && in && r + kFinLanes < nparts)
                           ? partial[(r + kFinLanes) * ncols + j] : 0.f;
      s[c][ty][tx] = lo + hi;
    }
    __syncthreads();
    if (ty < nc && in) {
      float t = s[ty][0][tx];
#pragma unroll
      for (int l = 1; l < kFinLanes; ++l) t += s[ty][l][tx];
      chunks[(g0 + ty) * ncols + j] = t;
    }
    __syncthreads();
  }
}

// out[j] = chunks[0][j] + chunks[1][j] + ... in chunk order.
__global__ void __launch_bounds__(256) dw_chunk_totals(const float* __restrict__ chunks,
                                                       int64_t nchunks, int ncols,
                                                       float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= ncols) return;
  float t = chunks[j];
#pragma unroll 8
  for (int64_t c = 1; c < nchunks; ++c) t += chunks[c * ncols + j];
  out[j] = t;
}

}  // namespace

cudaError_t launch_column_sums(const float* partial, int64_t nparts, int ncols, float* out0,
                               float* out1, int split, cudaStream_t s) {
  return launch_kernel(dw_finalize, dim3((unsigned)((ncols + 31) / 32)), dim3(32, kFinLanes), 0,
                       s, 1, partial, nparts, ncols, out0, out1, split);
}

cudaError_t launch_chunk_sums(const float* partial, int64_t nparts, int ncols, float* chunks,
                              cudaStream_t s) {
  return launch_kernel(dw_chunk_sums, dim3((unsigned)((ncols + 31) / 32)), dim3(32, kFinLanes),
                       0, s, 1, partial, nparts, ncols, chunks);
}

cudaError_t launch_chunk_totals(const float* chunks, int64_t nchunks, int ncols, float* out,
                                cudaStream_t s) {
  return launch_kernel(dw_chunk_totals, dim3((unsigned)((ncols + 255) / 256)), dim3(256), 0, s,
                       1, chunks, nchunks, ncols, out);
}

namespace {

template <typename T, int VPT>
cudaError_t launch_rows(const BwdArgs& a, int tpr, cudaStream_t s, int64_t* nparts) {
  auto kern = bwd_cta_rows<T, VPT, VPT == 1>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int occ = max_blocks_per_sm((const void*)kern, tpr, 0);
  const BlockPlan bp = plan_blocks(a.rows, a.block_rows,
                                   unit_cap(a, (int64_t)sm_count(dev) * (occ > 0 ? occ : 1)));
  *nparts = bp.nblocks;
  return launch_kernel(kern, dim3((unsigned)bp.units), dim3(tpr), 0, s, 1,
                       static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                       static_cast<const T*>(a.gamma), a.rstd, static_cast<T*>(a.dx), a.partial,
                       a.rows, a.hidden, a.offset ? 1.f : 0.f, bp.brows);
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
  int64_t nparts = 0;
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
    const BlockPlan bp = plan_blocks(a.rows, a.block_rows,
                                     unit_cap(a, (int64_t)sm_count(dev) * (occ > 0 ? occ : 1)));
    nparts = bp.nblocks;
    e = launch_kernel(kern, dim3((unsigned)bp.units), dim3(256), 0, s, 1,
                      static_cast<const T*>(a.dy), static_cast<const T*>(a.x),
                      static_cast<const T*>(a.gamma), a.rstd, static_cast<T*>(a.dx), a.partial,
                      a.rows, a.hidden, a.offset ? 1.f : 0.f, bp.brows);
  }
  if (e != cudaSuccess) return e;
  *launches += 1;
  e = a.chunks != nullptr ? launch_chunk_sums(a.partial, nparts, a.hidden, a.chunks, s)
                          : launch_column_sums(a.partial, nparts, a.hidden, a.dw, nullptr,
                                               a.hidden, s);
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
