// Device-side tile enumeration for the grouped GEMMs.
//
// Rows [off[e], off[e+1]) of the expert-major buffer belong to expert e.  The
// tiles of a grouped GEMM are (expert, m-tile, n-tile) with
// ceil(M_e / BM) m-tiles per expert; experts without rows have no tile.
// Offsets are read on the device, so no count ever crosses to the host.
// Each CTA stages them in shared memory once, sanitised (clamped to [0, N],
// then made non-decreasing by a running maximum; valid offsets come through
// unchanged), so that corrupt offsets can never address rows outside the
// buffers and no two experts' row ranges overlap.
#pragma once

#include "common.cuh"

namespace moe {

struct ExpertRows {
  int lo, hi;  // row range of the expert, clamped to [0, N]
};

__device__ __forceinline__ ExpertRows expert_rows(const int32_t* __restrict__ off, int e, int N) {
  int lo = off[e], hi = off[e + 1];
  lo = min(max(lo, 0), N);
  hi = min(max(hi, lo), N);
  return {lo, hi};
}

// Stage off[0..E] in shared memory as offs[0..E], sanitised: clamped to
// [0, N], then offs[i] = max(offs[0..i]).  off == nullptr means one expert
// owning all N rows (offs = {0, N}).  Called by every thread of the CTA
// (contains __syncthreads; blockDim.x a multiple of 32).  offs: smem, E+1
// ints; scratch: smem, 32 ints.
__device__ inline void stage_offsets(const int32_t* __restrict__ off, int E, int N, int32_t* offs,
                                     int32_t* scratch) {
  const int n = E + 1;
  const int nthr = blockDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = nthr >> 5;
  const int per = (n + nthr - 1) / nthr;
  const int lo = min(tid * per, n), hi = min(lo + per, n);
  int m = 0;  // clamped offsets are >= 0, so 0 is the identity of the max
  for (int i = lo; i < hi; ++i) {
    const int v = off != nullptr ? off[i] : (i == 0 ? 0 : N);
    m = max(m, min(max(v, 0), N));
    offs[i] = m;  // running maximum inside this thread's run
  }
  // inclusive max-scan of the runs' maxima: over the warp, then over warps
  int incl = m;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl = max(incl, v);
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? scratch[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w = max(w, v);
    }
    if (lane < nwarps) scratch[lane] = w;
  }
  __syncthreads();
  // maximum of every run before this thread's
  int before = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) before = 0;
  if (warp > 0) before = max(before, scratch[warp - 1]);
  for (int i = lo; i < hi; ++i) offs[i] = max(offs[i], before);
  __syncthreads();
}

// prefix[e] = number of m-tiles of experts < e, prefix[E] = total.  Called by
// every thread of the CTA (contains __syncthreads).  prefix: smem, E+1 ints;
// scratch: smem, 32 ints.
__device__ inline void build_tile_prefix(const int32_t* __restrict__ off, int E, int N, int BM,
                                  int32_t* prefix, int32_t* scratch) {
  const int nthr = blockDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = (nthr + 31) >> 5;
  const int per = (E + nthr - 1) / nthr;
  const int lo = min(tid * per, E), hi = min(lo + per, E);
  int s = 0;
  for (int e = lo; e < hi; ++e) {
    const ExpertRows r = expert_rows(off, e, N);
    const int m = (r.hi - r.lo + BM - 1) / BM;
    prefix[e] = m;
    s += m;
  }
  int incl = s;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31 || tid == nthr - 1) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? scratch[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    if (lane < nwarps) scratch[lane] = w;
  }
  __syncthreads();
  int run = incl - s + (warp > 0 ? scratch[warp - 1] : 0);
  for (int e = lo; e < hi; ++e) {
    const int m = prefix[e];
    prefix[e] = run;
    run += m;
  }
  if (tid == nthr - 1) prefix[E] = run;
  __syncthreads();
}

// Largest e with prefix[e] <= tile (the expert owning m-tile slot `tile`).
__device__ __forceinline__ int find_expert(const int32_t* prefix, int E, int tile) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

}  // namespace moe
