// Token permute for the MoE expert layer: expert histogram, scan, stable
// expert-major rank, row copy.  Also the inverse of sorted_indices.
//
// Layout (hyper_parallel expert_parallel.py, _generate_permute_indices
// docstring): the permuted buffer holds all rows routed to expert 0, then all
// rows of expert 1, ...; inside one expert the rows keep increasing flat slot
// order f = t*K + k.  sorted_indices uses the gather convention of that
// page's permuted_indices: entry i is the slot whose row lands at row i.
//
// Design: three small kernels over int32 ids (about 4 bytes per slot each)
// and one bandwidth kernel that reads every token row once and writes it to
// its K destinations with 16-byte vectors.  The rank pass is deterministic:
// per-block counts -> per-(block, expert) bases -> per-warp bases -> in-warp
// rank from __match_any_sync peers, so no atomic ordering reaches the output.
#include <atomic>
#include <chrono>
#include <map>
#include <mutex>
#include <random>
#include <utility>

#include <unistd.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kSlotsPerWarp = 64;
constexpr int kChunk = kRouteWarps * kSlotsPerWarp;  // slots per block
constexpr int kRowUnroll = 16;  // 16-byte vectors in flight per lane in the row copy

// Optional activity mask (the x_active_mask of the torch_npu
// npu_moe_distribute_combine_v2 parameters): mask_dims 1 = one byte per token
// [T], 2 = one byte per slot [T, K]; zero = not participating.
struct SlotMask {
  const uint8_t* mask;
  int dims;
  __device__ __forceinline__ bool active(int f, int K) const {
    if (mask == nullptr) return true;
    return (dims == 1 ? mask[f / K] : mask[f]) != 0;
  }
};

// Expert a slot is dispatched to, or -1: ids outside [0, E_total) and ids
// repeated earlier in the same row are not dispatched (and are errors);
// special ids in [E, E_total) and masked-off slots are legal but not
// dispatched.
__device__ __forceinline__ int slot_expert(const int32_t* __restrict__ ids, int f, int K, int E,
                                           int E_total, SlotMask m, bool* bad) {
  const int id = ids[f];
  const int row0 = (f / K) * K;
  bool ok = (id >= 0) && (id < E_total);
  // no short-circuit: the loads of the earlier ids of the row are independent
  for (int j = row0; j < f; ++j) ok &= (ids[j] != id);
  *bad = !ok;
  return (ok && id < E && m.active(f, K)) ? id : -1;
}

__global__ void __launch_bounds__(kRouteThreads)
route_hist_kernel(const int32_t* __restrict__ ids, int TK, int K, int E, int E_total, SlotMask m,
                  int32_t* __restrict__ blk_counts, int32_t* status) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += kRouteThreads) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kChunk;
  const int end = min(base + kChunk, TK);
  bool any_bad = false;
  for (int f = base + threadIdx.x; f < end; f += kRouteThreads) {
    bool bad;
    const int e = slot_expert(ids, f, K, E, E_total, m, &bad);
    any_bad |= bad;
    if (e >= 0) atomicAdd(&hist[e], 1);
  }
  if (any_bad) set_status(status, MOE_ERR_BAD_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kRouteThreads)
    blk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// One block of 1024 threads.  Thread t owns expert e = t % E and the p-th of
// P = 1024 / E ranges of blocks (E <= 1024).  In place: blk_counts[b][e]
// becomes the first permuted row of block b's slots of expert e.
__global__ void __launch_bounds__(1024)
route_scan_kernel(int32_t* __restrict__ blk, int nblk, int E, int32_t* __restrict__ tokens_per_expert,
                  int32_t* __restrict__ expert_offsets) {
  __shared__ int32_t part[1024];  // [P][E] partial counts, then partial bases
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x;
  const int P = 1024 / E;
  const int e = tid % E, pi = tid / E;
  const bool active = pi < P;
  const int b_lo = active ? (int)((long long)nblk * pi / P) : 0;
  const int b_hi = active ? (int)((long long)nblk * (pi + 1) / P) : 0;
  int psum = 0;
  for (int b = b_lo; b < b_hi; ++b) psum += blk[(size_t)b * E + e];
  if (active) part[pi * E + e] = psum;
  __syncthreads();
  // totals per expert and their exclusive scan (thread e < E)
  const int lane = tid & 31, warp = tid >> 5;
  int cnt = 0;
  if (tid < E)
    for (int q = 0; q < P; ++q) cnt += part[q * E + tid];
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  if (tid < E) {
    const int excl = incl - cnt + (warp > 0 ? warp_tot[warp - 1] : 0);
    tokens_per_expert[tid] = cnt;
    expert_offsets[tid] = excl;
    if (tid == E - 1) expert_offsets[E] = excl + cnt;
    // partial bases: the expert's offset plus the ranges before each range
    int run = excl;
    for (int q = 0; q < P; ++q) {
      const int c = part[q * E + tid];
      part[q * E + tid] = run;
      run += c;
    }
  }
  __syncthreads();
  if (active) {
    int run = part[pi * E + e];
    for (int b = b_lo; b < b_hi; ++b) {
      const int c = blk[(size_t)b * E + e];
      blk[(size_t)b * E + e] = run;
      run += c;
    }
  }
}

__global__ void __launch_bounds__(kRouteThreads)
route_scatter_kernel(const int32_t* __restrict__ ids, int TK, int K, int E, int E_total, SlotMask m,
                     const int32_t* __restrict__ blk_base, int32_t* __restrict__ sorted_indices,
                     int32_t* __restrict__ row_map) {
  extern __shared__ int32_t cnt[];  // [kRouteWarps][E]
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = threadIdx.x; i < kRouteWarps * E; i += kRouteThreads) cnt[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wbase = blockIdx.x * kChunk + warp * kSlotsPerWarp;
  int32_t* my = cnt + warp * E;
  // 1. per-warp counts; each lane keeps the experts of its slots for step 3
  constexpr int kSteps = kSlotsPerWarp / 32;
  int ex[kSteps];
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int f = wbase + i * 32 + lane;
    ex[i] = -1;
    if (f < TK) {
      bool bad;
      ex[i] = slot_expert(ids, f, K, E, E_total, m, &bad);
      if (ex[i] >= 0) atomicAdd(&my[ex[i]], 1);
    }
  }
  __syncthreads();
  // 2. per-warp bases: block base of the expert + counts of earlier warps
  for (int e = threadIdx.x; e < E; e += kRouteThreads) {
    int run = blk_base[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // 3. stable rank inside each 32-slot step: peers with the same expert and a
  //    lower lane come first; the step's leader advances the warp's base.
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int f = wbase + i * 32 + lane;
    const int e = ex[i];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lanemask_lt());
    if (e >= 0) {
      const int pos = my[e] + rank;
      sorted_indices[pos] = f;
      row_map[f] = pos;
    } else if (f < TK) {
      row_map[f] = -1;
    }
    __syncwarp();
    if (e >= 0 && rank == 0) my[e] += __popc(peers);
    __syncwarp();
  }
}

// ---- the three passes above in one cooperative launch -----------------------
//
// For small and medium T*K the three routing kernels are bound by launch
// latency, not by their few bytes.  This kernel runs them as phases of one
// grid whose blocks are all resident (cooperative launch): each block counts
// its chunk per warp (phase 1), publishes its block counts and then a flag
// stamped with a value unique to the call, waits for every block's flag,
// reduces the counts of all blocks itself (the totals, and the counts of
// earlier blocks, per expert), scans the totals and places its slots exactly
// as route_scatter_kernel does.  The stamps make stale workspace contents
// harmless, so nothing has to be cleared before a call.  The wait is bounded:
// on timeout the block records MOE_ERR_TIMEOUT and leaves.

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr unsigned long long kFlagWaitNs = 2000000000ull;  // 2 s

template <int kSteps>
__global__ void __launch_bounds__(kRouteThreads)
route_fused_kernel(const int32_t* __restrict__ ids, int TK, int K, int E, int E_total, SlotMask m,
                   int32_t* __restrict__ blk_counts, unsigned long long* __restrict__ flags,
                   unsigned long long stamp, int32_t* __restrict__ sorted_indices,
                   int32_t* __restrict__ row_map, int32_t* __restrict__ tokens_per_expert,
                   int32_t* __restrict__ expert_offsets, int32_t* status) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                     // [kRouteWarps][E] counts, then warp bases
  int32_t* tot = cnt + kRouteWarps * E;  // [E] totals, then expert offsets
  int32_t* below = tot + E;              // [E] counts of earlier blocks
  __shared__ int32_t scan_part[kRouteThreads];
  __shared__ int timed_out;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, nblk = gridDim.x;
  // the row copy may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = tid; i < (kRouteWarps + 2) * E; i += kRouteThreads) sm[i] = 0;
  if (tid == 0) timed_out = 0;
  __syncthreads();
  // 1. experts of this warp's 32 * kSteps slots (kept for phase 7) and warp
  //    counts
  constexpr int kWarpSlots = 32 * kSteps, kBlockSlots = kRouteWarps * kWarpSlots;
  const int wbase = b * kBlockSlots + warp * kWarpSlots;
  int32_t* my = cnt + warp * E;
  int ex[kSteps];
  bool any_bad = false;
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int f = wbase + i * 32 + lane;
    ex[i] = -1;
    if (f < TK) {
      bool bad;
      ex[i] = slot_expert(ids, f, K, E, E_total, m, &bad);
      any_bad |= bad;
      if (ex[i] >= 0) atomicAdd(&my[ex[i]], 1);
    }
  }
  if (any_bad) set_status(status, MOE_ERR_BAD_ID);
  __syncthreads();
  // 2. publish the block counts, then the block's flag
  for (int e = tid; e < E; e += kRouteThreads) {
    int c = 0;
    for (int w = 0; w < kRouteWarps; ++w) c += cnt[w * E + e];
    blk_counts[(size_t)b * E + e] = c;
  }
  // The block barrier orders every thread's count stores before thread 0's
  // release of the flag, and a release is cumulative: a block that acquires
  // the flag sees the counts (a fence by every thread measured 0.9 us slower
  // at 64 blocks).
  __syncthreads();
  if (tid == 0) st_release_u64(&flags[b], stamp);
  // 3. wait for every block's flag
  for (int i = tid; i < nblk; i += kRouteThreads) {
    unsigned long long t0 = 0;
    for (uint32_t it = 0; ld_acquire_u64(&flags[i]) != stamp; ++it) {
      if ((it & 63u) == 63u) {
        const unsigned long long now = global_ns();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > kFlagWaitNs) {
          timed_out = 1;
          break;
        }
      }
    }
  }
  __syncthreads();
  if (timed_out) {
    // Leave no stale entry behind: this block's slots are not dispatched
    // (the row copy skips them), and block 0 publishes an empty routing.
    if (tid == 0) set_status(status, MOE_ERR_TIMEOUT);
    for (int f = b * kBlockSlots + tid; f < min((b + 1) * kBlockSlots, TK); f += kRouteThreads)
      row_map[f] = -1;
    if (b == 0) {
      for (int e = tid; e < E; e += kRouteThreads) tokens_per_expert[e] = 0;
      for (int e = tid; e <= E; e += kRouteThreads) expert_offsets[e] = 0;
    }
    return;
  }
  // 4. per expert: total over all blocks and the counts of blocks before b
  //    (read through L2).  With E a multiple of 4 (the workspace is
  //    16-byte aligned), a thread reads 4 experts' counts per 16-byte load
  //    and Q4 threads per 4 experts split the blocks: four times the bytes
  //    in flight per load (T=8192 K=8 E=256: routing 19.2 -> 16.3 us);
  //    otherwise Q threads per expert read one count per load.
  const bool vec4 = (E & 3) == 0;
  if (vec4) {
    const int EQ = E >> 2;
    const int Q4 = EQ < kRouteThreads ? kRouteThreads / EQ : 1;
    for (int i = tid; i < EQ * Q4; i += kRouteThreads) {
      const int eq = i % EQ, q = i / EQ;
      const int b_lo = (int)((long long)nblk * q / Q4), b_hi = (int)((long long)nblk * (q + 1) / Q4);
      int4 ts = make_int4(0, 0, 0, 0), bs = make_int4(0, 0, 0, 0);
#pragma unroll 8
      for (int bb = b_lo; bb < b_hi; ++bb) {
        const int4 c = __ldcg(reinterpret_cast<const int4*>(blk_counts + (size_t)bb * E) + eq);
        ts.x += c.x;
        ts.y += c.y;
        ts.z += c.z;
        ts.w += c.w;
        if (bb < b) {
          bs.x += c.x;
          bs.y += c.y;
          bs.z += c.z;
          bs.w += c.w;
        }
      }
      const int t4[4] = {ts.x, ts.y, ts.z, ts.w}, b4[4] = {bs.x, bs.y, bs.z, bs.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (t4[j]) atomicAdd(&tot[4 * eq + j], t4[j]);
        if (b4[j]) atomicAdd(&below[4 * eq + j], b4[j]);
      }
    }
  }
  const int Q = E < kRouteThreads ? kRouteThreads / E : 1;
  for (int i = tid; !vec4 && i < E * Q; i += kRouteThreads) {
    const int e = i % E, q = i / E;
    const int b_lo = (int)((long long)nblk * q / Q), b_hi = (int)((long long)nblk * (q + 1) / Q);
    int t_sum = 0, b_sum = 0;
#pragma unroll 8
    for (int bb = b_lo; bb < b_hi; ++bb) {
      const int c = __ldcg(&blk_counts[(size_t)bb * E + e]);
      t_sum += c;
      if (bb < b) b_sum += c;
    }
    if (t_sum) atomicAdd(&tot[e], t_sum);
    if (b_sum) atomicAdd(&below[e], b_sum);
  }
  __syncthreads();
  // 5. exclusive scan of the totals over experts: thread i owns the
  //    consecutive experts [i*per, (i+1)*per)
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += tot[e];
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) scan_part[warp] = incl;
  __syncthreads();
  int wprefix = 0;
  for (int w = 0; w < warp; ++w) wprefix += scan_part[w];
  int run = wprefix + incl - local;  // exclusive prefix of expert e0
  __syncthreads();
  for (int e = e0; e < e1; ++e) {
    const int c = tot[e];
    if (b == 0) {
      tokens_per_expert[e] = c;
      expert_offsets[e] = run;
    }
    tot[e] = run;
    run += c;
  }
  if (b == 0 && e1 == E && e0 < e1) expert_offsets[E] = run;
  __syncthreads();
  // 6. warp bases: expert offset + earlier blocks + earlier warps of this block
  for (int e = tid; e < E; e += kRouteThreads) {
    int r = tot[e] + below[e];
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = r;
      r += c;
    }
  }
  __syncthreads();
  // 7. stable rank inside each 32-slot step (as in route_scatter_kernel)
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int f = wbase + i * 32 + lane;
    const int e = ex[i];
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lanemask_lt());
    if (e >= 0) {
      const int pos = my[e] + rank;
      sorted_indices[pos] = f;
      row_map[f] = pos;
    } else if (f < TK) {
      row_map[f] = -1;
    }
    __syncwarp();
    if (e >= 0 && rank == 0) my[e] += __popc(peers);
    __syncwarp();
  }
}

// One warp per token: read the row once (16-byte vectors), write it to each
// of its K permuted rows.  A lane keeps up to kUnroll vectors in flight
// (kRowUnroll = 16: a 4 KB row in one round of loads) and writes with
// streaming stores, since the permuted rows are not re-read here: at
// T=4096 H=2048 K=8 this measured 35.9 us against 40.9 with 4 vectors and
// plain stores (routing included), 202.7 against 210.7 at T=16384 H=4096.
// Slots whose row lies outside [0, N) (N = rows of the permuted buffer) are
// skipped: -1 marks a slot that is not dispatched, and nothing else may
// address memory outside the buffer.
template <int kUnroll>
__global__ void __launch_bounds__(256)
permute_rows_kernel(const uint8_t* __restrict__ tokens, const int32_t* __restrict__ row_map, int T,
                    int K, int N, int row_bytes, uint8_t* __restrict__ permuted) {
  // Launched as a programmatic dependent of the routing: wait until that
  // grid has completed and its row_map is visible (a no-op otherwise).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const int my_rm = lane < K ? row_map[(size_t)t * K + lane] : -1;
  const int nvec = row_bytes >> 4;
  const uint8_t* src = tokens + (size_t)t * row_bytes;
  // The trip count is the same for every lane (the shuffles below need the
  // whole warp); lanes past the row end only skip their loads and stores.
  for (int base = 0; base < nvec; base += 32 * kUnroll) {
    const int v0 = base + lane;
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * 32;
      if (v < nvec) x[u] = ld_nc_v4(src + ((size_t)v << 4));
    }
    for (int k = 0; k < K; ++k) {
      const int r = __shfl_sync(0xffffffffu, my_rm, k);
      if (r < 0 || r >= N) continue;
      uint8_t* dst = permuted + (size_t)r * row_bytes;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * 32;
        if (v < nvec) st_cs_v4(dst + ((size_t)v << 4), x[u]);
      }
    }
  }
}

__global__ void fill_kernel(int32_t* __restrict__ p, int n, int32_t value) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    p[i] = value;
}

__global__ void invert_kernel(const int32_t* __restrict__ sorted_indices, int N, int TK,
                              int32_t* __restrict__ row_map) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x) {
    const int f = sorted_indices[i];
    if (f >= 0 && f < TK) row_map[f] = i;
  }
}

}  // namespace

// ---- host entry points -------------------------------------------------------

static inline int route_blocks(int TK) { return (TK + kChunk - 1) / kChunk; }

// Workspace: per-block expert counts [nblk][E] int32, then (8-byte aligned)
// the per-block flags of the fused routing [nblk] uint64.
static inline size_t flags_offset(long long nblk, int E) {
  return (size_t)((nblk * E * (long long)sizeof(int32_t) + 7) & ~7LL);
}

static inline size_t fused_smem_bytes(int E) { return (size_t)(kRouteWarps + 2) * E * sizeof(int32_t); }

// Whether nblk blocks of the fused routing kernel fit on the current device
// at once (cooperative launch); cached per (kernel, device, E).
template <int kSteps>
static bool fused_fits(int nblk, int E) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cap;  // (device, E) -> resident blocks
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cap.find({dev, E});
  if (it == cap.end()) {
    int coop = 0, per_sm = 0;
    int n = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_fused_kernel<kSteps>,
                                                      kRouteThreads, fused_smem_bytes(E)) ==
            cudaSuccess)
      n = per_sm * sm_count();
    (void)cudaGetLastError();
    it = cap.emplace(std::make_pair(dev, E), n).first;
  }
  return nblk <= it->second;
}

// splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014): spreads every input bit over the output.
static unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// A value no earlier call of this process used.  The counter starts from a
// hash of the clock, the process id and a random_device draw, so a stamp
// found in a workspace that another process left behind matches only by a
// 64-bit coincidence; within one process the stamps are unique.
static unsigned long long stamp_seed() {
  unsigned long long rd = 0;
  try {
    std::random_device dev;
    rd = ((unsigned long long)dev() << 32) ^ dev();
  } catch (...) {
  }
  const unsigned long long ns =
      (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
  return mix64(ns ^ mix64((unsigned long long)getpid() ^ mix64(rd)));
}

static unsigned long long next_stamp() {
  static std::atomic<unsigned long long> counter{stamp_seed()};
  unsigned long long v;
  do {
    v = counter.fetch_add(1ull);
  } while (v == 0ull);
  return v;
}

// One cooperative launch of the fused routing with kSteps 32-slot steps per
// warp; false if its blocks do not all fit at once or the launch fails.
template <int kSteps>
static bool launch_route_fused(const int32_t* expert_ids, int TK, int K, int E, int E_total,
                               SlotMask m, void* workspace, int32_t* sorted_indices,
                               int32_t* row_map, int32_t* tokens_per_expert,
                               int32_t* expert_offsets, int32_t* dev_status,
                               cudaStream_t stream) {
  constexpr int kBlockSlots = kRouteWarps * 32 * kSteps;
  const int nblk = (TK + kBlockSlots - 1) / kBlockSlots;
  if (!fused_fits<kSteps>(nblk, E)) return false;
  int32_t* blk = static_cast<int32_t*>(workspace);
  unsigned long long* flags =
      reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + flags_offset(nblk, E));
  unsigned long long stamp = next_stamp();
  void* args[] = {(void*)&expert_ids, (void*)&TK, (void*)&K, (void*)&E, (void*)&E_total,
                  (void*)&m, (void*)&blk, (void*)&flags, (void*)&stamp, (void*)&sorted_indices,
                  (void*)&row_map, (void*)&tokens_per_expert, (void*)&expert_offsets,
                  (void*)&dev_status};
  if (cudaLaunchCooperativeKernel((const void*)route_fused_kernel<kSteps>, dim3(nblk),
                                  dim3(kRouteThreads), args, fused_smem_bytes(E), stream) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  count_launches(1);
  return true;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_workspace_size(int T, int K, int E) {
  if (T < 0 || K <= 0 || E <= 0) return 0;
  const long long TK = (long long)T * K;
  const long long nblk = (TK + kChunk - 1) / kChunk > 0 ? (TK + kChunk - 1) / kChunk : 1;
  return flags_offset(nblk, E) + (size_t)nblk * sizeof(unsigned long long);
}

extern "C" int moe_permute_masked(const void* tokens, int dtype, const int32_t* expert_ids, int T,
                                  int H, int K, int E, int num_special, const uint8_t* active_mask,
                                  int mask_dims, void* permuted, int32_t* sorted_indices,
                                  int32_t* row_map, int32_t* tokens_per_expert,
                                  int32_t* expert_offsets, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, cudaStream_t stream) {
  if (active_mask != nullptr && mask_dims != 1 && mask_dims != 2) return MOE_ERR_INVALID_ARG;
  if (T < 0 || H <= 0 || K <= 0 || E <= 0 || num_special < 0) return MOE_ERR_INVALID_ARG;
  if (K > kMaxK || E > kMaxExperts || (long long)K > (long long)E + num_special)
    return MOE_ERR_SHAPE;
  if ((long long)T * K > 0x7fffffffLL || (long long)E + num_special > 0x7fffffffLL)
    return MOE_ERR_SHAPE;
  if (tokens != nullptr) {
    const int esz = dtype_size(dtype);
    if (esz == 0) return MOE_ERR_INVALID_ARG;
    if (permuted == nullptr) return MOE_ERR_INVALID_ARG;
    if (((size_t)H * esz) % 16 != 0) return MOE_ERR_SHAPE;
    if (!aligned16(tokens) || !aligned16(permuted)) return MOE_ERR_INVALID_ARG;
  }
  if (!tokens_per_expert || !expert_offsets) return MOE_ERR_INVALID_ARG;
  const int TK = T * K;
  if (TK > 0 && (!expert_ids || !sorted_indices || !row_map)) return MOE_ERR_INVALID_ARG;
  const int nblk = route_blocks(TK);
  if (TK > 0 && (workspace == nullptr || workspace_bytes < moe_permute_workspace_size(T, K, E)))
    return MOE_ERR_INVALID_ARG;
  // the flags are 8-byte words and the counts are read 16 bytes at a time
  if (TK > 0 && !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  if (TK == 0) {
    // Nothing routed: zero counts, zero offsets.
    fill_kernel<<<1, 256, 0, stream>>>(tokens_per_expert, E, 0);
    fill_kernel<<<1, 256, 0, stream>>>(expert_offsets, E + 1, 0);
    count_launches(2);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
  }
  int32_t* blk = static_cast<int32_t*>(workspace);
  const int E_total = E + num_special;
  const SlotMask m{active_mask, mask_dims};
  // All blocks resident: the three routing passes as one launch.  Each
  // block reads every block's counts, so past 64 blocks of 512 slots the
  // blocks take 1024 slots (T=8192 K=8 E=256: 16.7 -> 12.5 us; at 64 or
  // fewer blocks the 512-slot blocks measured faster).  The workspace is
  // sized for 512-slot blocks, which covers both layouts.
  const bool fused =
      TK > 64 * kChunk
          ? launch_route_fused<4>(expert_ids, TK, K, E, E_total, m, workspace, sorted_indices,
                                  row_map, tokens_per_expert, expert_offsets, dev_status, stream)
          : launch_route_fused<2>(expert_ids, TK, K, E, E_total, m, workspace, sorted_indices,
                                  row_map, tokens_per_expert, expert_offsets, dev_status, stream);
  if (!fused) {
    route_hist_kernel<<<nblk, kRouteThreads, E * sizeof(int32_t), stream>>>(
        expert_ids, TK, K, E, E_total, m, blk, dev_status);
    route_scan_kernel<<<1, 1024, 0, stream>>>(blk, nblk, E, tokens_per_expert, expert_offsets);
    const size_t scatter_smem = (size_t)kRouteWarps * E * sizeof(int32_t);
    if (scatter_smem > 48 * 1024)
      cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)scatter_smem);
    route_scatter_kernel<<<nblk, kRouteThreads, scatter_smem, stream>>>(
        expert_ids, TK, K, E, E_total, m, blk, sorted_indices, row_map);
    count_launches(3);
  }
  if (tokens != nullptr && T > 0) {
    const int row_bytes = H * dtype_size(dtype);
    // Programmatic dependent launch: the copy's launch overlaps the routing.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((T + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const uint8_t* tok = static_cast<const uint8_t*>(tokens);
    uint8_t* dst = static_cast<uint8_t*>(permuted);
    const int32_t* rm = row_map;
    if (cudaLaunchKernelEx(&cfg, permute_rows_kernel<kRowUnroll>, tok, rm, T, K, TK, row_bytes, dst) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    count_launches(1);
  }
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_permute(const void* tokens, int dtype, const int32_t* expert_ids, int T, int H,
                           int K, int E, int num_special, void* permuted, int32_t* sorted_indices,
                           int32_t* row_map, int32_t* tokens_per_expert, int32_t* expert_offsets,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           cudaStream_t stream) {
  return moe_permute_masked(tokens, dtype, expert_ids, T, H, K, E, num_special, nullptr, 0,
                            permuted, sorted_indices, row_map, tokens_per_expert, expert_offsets,
                            workspace, workspace_bytes, dev_status, stream);
}

extern "C" int moe_permute_rows(const void* tokens, int dtype, const int32_t* row_map, int T, int H,
                                int K, int N, void* permuted, cudaStream_t stream) {
  const int esz = dtype_size(dtype);
  if (esz == 0 || T < 0 || H <= 0 || K <= 0 || N < 0) return MOE_ERR_INVALID_ARG;
  if (K > kMaxK) return MOE_ERR_SHAPE;
  if (((size_t)H * esz) % 16 != 0) return MOE_ERR_SHAPE;
  if ((long long)T * K > 0x7fffffffLL) return MOE_ERR_SHAPE;
  if (T == 0 || N == 0) return MOE_OK;
  if (!tokens || !row_map || !permuted) return MOE_ERR_INVALID_ARG;
  if (!aligned16(tokens) || !aligned16(permuted)) return MOE_ERR_INVALID_ARG;
  permute_rows_kernel<kRowUnroll><<<(T + 7) / 8, 256, 0, stream>>>(
      static_cast<const uint8_t*>(tokens), row_map, T, K, N, H * esz,
      static_cast<uint8_t*>(permuted));
  count_launches(1);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_invert_sorted_indices(const int32_t* sorted_indices, int N, int TK,
                                         int32_t* row_map, cudaStream_t stream) {
  if (N < 0 || TK < 0 || N > TK) return MOE_ERR_INVALID_ARG;
  if (TK == 0) return MOE_OK;
  if (!row_map || (N > 0 && !sorted_indices)) return MOE_ERR_INVALID_ARG;
  const int grid = min((TK + 255) / 256, 4 * sm_count());
  fill_kernel<<<grid, 256, 0, stream>>>(row_map, TK, -1);
  if (N > 0)
    invert_kernel<<<min((N + 255) / 256, 4 * sm_count()), 256, 0, stream>>>(sorted_indices, N, TK,
                                                                             row_map);
  count_launches(N > 0 ? 2 : 1);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

// ---- allocation-free variant -------------------------------------------------
//
// Scratch for the per-block expert counts of moe_permute_static_scratch: one
// array per device, alive for the whole process.  Host code must not pass
// the symbol itself to a kernel (on the host it names a host-side shadow,
// not device memory); the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) int32_t g_permute_scratch[MOE_PERMUTE_STATIC_SCRATCH_INTS];

namespace {

constexpr int kMaxDevices = 64;

// Device address of g_permute_scratch on the current device, looked up once
// per device (with that device current).  nullptr on failure.
int32_t* permute_scratch_address() {
  static std::mutex mu;
  static int32_t* addr[kMaxDevices] = {nullptr};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    addr[dev] = static_cast<int32_t*>(p);
  }
  return addr[dev];
}

}  // namespace

extern "C" int moe_permute_static_scratch(const void* tokens, int dtype, const int32_t* expert_ids,
                                          int T, int H, int K, int E, int num_special,
                                          void* permuted, int32_t* sorted_indices,
                                          int32_t* row_map, int32_t* tokens_per_expert,
                                          int32_t* expert_offsets, int32_t* dev_status,
                                          cudaStream_t stream) {
  if (T < 0 || K <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_permute_workspace_size(T, K, E);
  const size_t have = sizeof(int32_t) * MOE_PERMUTE_STATIC_SCRATCH_INTS;
  if (need > have) return MOE_ERR_CAPACITY;
  int32_t* scratch = permute_scratch_address();
  if (scratch == nullptr) return MOE_ERR_CUDA;
  return moe_permute(tokens, dtype, expert_ids, T, H, K, E, num_special, permuted, sorted_indices,
                     row_map, tokens_per_expert, expert_offsets, scratch, have, dev_status, stream);
}
