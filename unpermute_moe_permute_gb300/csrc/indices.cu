// Rank-major -> expert-major permute indices (hyper_parallel
// expert_parallel.py, _generate_permute_indices) and the deredundancy
// dispatch indices of the same page (_generate_deredundency_dispatch_indices),
// which are the same construction restricted to a window of expert columns.
//
// counts[r*E + e] rows arrived from rank r for local expert e, stored
// rank-major: [r0.e0 | r0.e1 | ... | r1.e0 | ...].  The expert-major buffer
// visits the same blocks as [e0.r0 | e0.r1 | ... | e1.r0 | ...].  Destination
// i inside block (e, r) at offset j reads source start_rm(r, e) + j.
//
// One launch, no host round trip (the page drains `total` to the host before
// building the indices; here it stays on the device).  Every CTA stages the
// R*E counts in shared memory and computes both exclusive scans (rank-major
// source starts, expert-major destination starts), then the CTAs split the
// blocks between them and each warp writes one block's run of indices.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kIdxThreads = 1024;
constexpr int kMaxBlocks = 2048;  // R * E (combine_v2 constraints: local experts x EP size <= 2048)

// Exclusive scan of n values in smem (in place) by one CTA of kIdxThreads.
// Each thread scans a contiguous run serially, then the run totals are
// scanned across the CTA.
__device__ void cta_exclusive_scan(int32_t* a, int n, int32_t* tmp /* >= 32 */,
                                   int32_t* total_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kIdxThreads - 1) / kIdxThreads;
  const int lo = min(tid * per, n), hi = min(lo + per, n);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += a[i];
  int incl = s;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = tmp[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    tmp[lane] = w;
  }
  __syncthreads();
  int run = incl - s + (warp > 0 ? tmp[warp - 1] : 0);
  for (int i = lo; i < hi; ++i) {
    const int c = a[i];
    a[i] = run;
    run += c;
  }
  if (total_out && tid == 0) *total_out = tmp[31];
  __syncthreads();
}

// counts: [R, E_all] row-major (source r, column e).  The source buffer holds
// the blocks in that row-major order; the output visits the blocks of the
// column window [c0, c0 + C) column-major: (c0, r=0..R-1), (c0+1, ...), ...
__global__ void __launch_bounds__(kIdxThreads)
permute_indices_kernel(const int32_t* __restrict__ counts, int R, int E_all, int c0, int C,
                       int32_t* __restrict__ indices, int capacity,
                       int32_t* __restrict__ tokens_per_column, int32_t* total, int32_t* status) {
  __shared__ int32_t src_rm[kMaxBlocks];  // source starts, (r, e) order over all columns
  __shared__ int32_t cnt_w[kMaxBlocks];   // window counts in (c, r) order
  __shared__ int32_t dst_w[kMaxBlocks];   // destination starts, (c, r) order
  __shared__ int32_t tmp[32];
  __shared__ int32_t s_total;
  __shared__ int32_t s_bad;
  __shared__ unsigned long long s_sum;  // sum of all counts, in 64 bits
  const int nb = R * E_all, nw = R * C;
  if (threadIdx.x == 0) {
    s_bad = 0;
    s_sum = 0ull;
  }
  __syncthreads();
  long long my_sum = 0;
  for (int b = threadIdx.x; b < nb; b += kIdxThreads) {
    int c = counts[b];
    if (c < 0) {
      s_bad = 1;
      c = 0;
    }
    my_sum += c;
    src_rm[b] = c;
    const int r = b / E_all, e = b - r * E_all;
    if (e >= c0 && e < c0 + C) {
      cnt_w[(e - c0) * R + r] = c;
      dst_w[(e - c0) * R + r] = c;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) my_sum += __shfl_down_sync(0xffffffffu, my_sum, o);
  if ((threadIdx.x & 31) == 0 && my_sum) atomicAdd(&s_sum, (unsigned long long)my_sum);
  __syncthreads();
  // The int32 scans below need every prefix sum to fit in int32: a larger
  // sum is reported as a capacity error and nothing else is written.
  if (s_sum > 0x7fffffffull) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      *total = -1;
      if (s_bad) set_status(status, MOE_ERR_INVALID_ARG);
      set_status(status, MOE_ERR_CAPACITY);
    }
    return;
  }
  cta_exclusive_scan(src_rm, nb, tmp, nullptr);
  cta_exclusive_scan(dst_w, nw, tmp, &s_total);
  const int tot = s_total;
  if (blockIdx.x == 0) {
    for (int c = threadIdx.x; c < C; c += kIdxThreads) {
      int s = 0;
      for (int r = 0; r < R; ++r) s += cnt_w[c * R + r];
      tokens_per_column[c] = s;
    }
    if (threadIdx.x == 0) {
      *total = tot;
      if (s_bad) set_status(status, MOE_ERR_INVALID_ARG);
      if (tot > capacity) set_status(status, MOE_ERR_CAPACITY);
    }
  }
  if (tot > capacity) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = kIdxThreads / 32;
  for (int b = blockIdx.x * nwarps + warp; b < nw; b += gridDim.x * nwarps) {
    const int c = b / R, r = b - c * R;
    const int cnt = cnt_w[b];
    const int src = src_rm[r * E_all + c0 + c];
    const int dst = dst_w[b];
    for (int j = lane; j < cnt; j += 32) indices[dst + j] = src + j;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_permute_indices_window(const int32_t* counts, int R, int E_all, int col_start,
                                          int col_count, int32_t* indices, int capacity,
                                          int32_t* tokens_per_column, int32_t* total,
                                          int32_t* dev_status, cudaStream_t stream) {
  if (R <= 0 || E_all <= 0 || col_start < 0 || col_count < 0 || capacity < 0)
    return MOE_ERR_INVALID_ARG;
  if ((long long)col_start + col_count > E_all) return MOE_ERR_SHAPE;
  if ((long long)R * E_all > kMaxBlocks) return MOE_ERR_SHAPE;
  if (!counts || !total || (col_count > 0 && !tokens_per_column) || (capacity > 0 && !indices))
    return MOE_ERR_INVALID_ARG;
  // Enough CTAs that each warp writes about one block; at most one wave.
  const int nw = R * col_count;
  int grid = (nw + 31) / 32;
  grid = max(1, min(grid, sm_count()));
  permute_indices_kernel<<<grid, kIdxThreads, 0, stream>>>(counts, R, E_all, col_start, col_count,
                                                           indices, capacity, tokens_per_column,
                                                           total, dev_status);
  count_launches(1);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_permute_indices(const int32_t* counts, int R, int E, int32_t* indices,
                                   int capacity, int32_t* tokens_per_expert, int32_t* total,
                                   int32_t* dev_status, cudaStream_t stream) {
  if (R <= 0 || E <= 0 || capacity < 0) return MOE_ERR_INVALID_ARG;
  return moe_permute_indices_window(counts, R, E, 0, E, indices, capacity, tokens_per_expert,
                                    total, dev_status, stream);
}
