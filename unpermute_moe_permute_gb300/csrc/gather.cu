// Token-order reductions of the MoE layer: unpermute forward and backward,
// permute backward, and the combine with shared and special experts.
//
// All four are HBM-bound row gathers: one warp owns one token, reads the K
// rows its slots map to through row_map (16-byte vectors, all K loads of a
// column chunk issued before the arithmetic), accumulates in fp32 in fixed k
// order and writes the token row once.  No atomics, so results do not depend
// on scheduling.
//
// Definitions:
//   unpermute      out[t] = sum_k probs[t,k] * expanded[row_map[t*K+k]]
//                  (the weighted inverse of the permute; torch_npu
//                  npu_moe_token_unpermute as sharded in the Ascend/pytorch
//                  PR "Update moe token unpermute DTensor support")
//   unpermute bwd  grad_permuted[row_map[f]] = probs[f] * grad_out[t],
//                  grad_probs[t,k] = <permuted[row_map[f]], grad_out[t]>
//                  (the probs grad is a sum over the hidden dim: 'Partial'
//                  under hidden-dim sharding in that PR)
//   permute bwd    grad_tokens[t] = sum_k grad_permuted[row_map[t*K+k]]
//                  (the gather x[idx] accumulates duplicate indices in its
//                  backward; twinkle PR "NPU EP experts forward uses NPU
//                  grouped matmul")
//   combine        x[t] = sum_k scales[t,k] * y(t,k) + shared_x[t] with the
//                  zero / copy / const expert closed forms of the torch_npu
//                  npu_moe_distribute_combine_v2 API reference.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

// Slot k of token t, broadcast to the warp: row in the expert-major buffer
// (-1 when not dispatched) and weight.
template <int KMAX>
struct Slots {
  int row[KMAX];
  float w[KMAX];
};

template <int KMAX>
__device__ __forceinline__ Slots<KMAX> load_slots(const int32_t* __restrict__ row_map,
                                                  const float* __restrict__ probs, int t, int K,
                                                  int N, int lane) {
  int my_row = -1;
  float my_w = 0.f;
  if (lane < K) {
    my_row = row_map[(size_t)t * K + lane];
    if (my_row >= N) my_row = -1;
    my_w = probs ? probs[(size_t)t * K + lane] : 1.f;
  }
  Slots<KMAX> s;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    s.row[k] = __shfl_sync(0xffffffffu, my_row, k);
    s.w[k] = __shfl_sync(0xffffffffu, my_w, k);
    if (k >= K) s.row[k] = -1;
  }
  return s;
}

// out[t] = round( sum_k w_k * Y[row_k] )   (also the permute backward, w = 1)
template <typename T, int KMAX>
__global__ void __launch_bounds__(256)
unpermute_kernel(const T* __restrict__ Y, const int32_t* __restrict__ row_map,
                 const float* __restrict__ probs, int Tn, int H, int K, int N, T* __restrict__ out) {
  using VT = VecTraits<T>;
  constexpr int EL = VT::kElems;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + warp;
  if (t >= Tn) return;
  const Slots<KMAX> s = load_slots<KMAX>(row_map, probs, t, K, N, lane);
  const int nvec = H / EL;
  // one column chunk per lane per iteration (two chunks measured slower
  // here, unlike in the backward below)
  constexpr int U = 1;
  for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
    uint4 x[U][KMAX];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (s.row[k] >= 0 && v < nvec) x[u][k] = ld_nc_v4(Y + (size_t)s.row[k] * H + (size_t)v * EL);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nvec) break;
      float acc[EL];
#pragma unroll
      for (int e = 0; e < EL; ++e) acc[e] = 0.f;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (s.row[k] < 0) continue;
        float f[EL];
        VT::unpack(x[u][k], f);
#pragma unroll
        for (int e = 0; e < EL; ++e) acc[e] = fmaf(s.w[k], f[e], acc[e]);
      }
      st_v4(out + (size_t)t * H + (size_t)v * EL, VT::pack(acc));
    }
  }
}

template <typename T, int KMAX>
__global__ void __launch_bounds__(256)
unpermute_grad_kernel(const T* __restrict__ grad_out, const T* __restrict__ X,
                      const int32_t* __restrict__ row_map, const float* __restrict__ probs, int Tn,
                      int H, int K, int N, T* __restrict__ grad_perm, float* __restrict__ grad_probs) {
  using VT = VecTraits<T>;
  constexpr int EL = VT::kElems;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + warp;
  if (t >= Tn) return;
  const Slots<KMAX> s = load_slots<KMAX>(row_map, probs, t, K, N, lane);
  float dot[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) dot[k] = 0.f;
  const int nvec = H / EL;
  // two column chunks per lane per iteration: 2*(K+1) loads in flight
  constexpr int U = KMAX <= 8 ? 2 : 1;
  for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
    uint4 gv[U], x[U][KMAX];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nvec) gv[u] = ld_nc_v4(grad_out + (size_t)t * H + (size_t)v * EL);
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (s.row[k] >= 0 && v < nvec) x[u][k] = ld_nc_v4(X + (size_t)s.row[k] * H + (size_t)v * EL);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nvec) break;
      const size_t col = (size_t)v * EL;
      float g[EL];
      VT::unpack(gv[u], g);
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (s.row[k] < 0) continue;
        float o[EL], f[EL];
        VT::unpack(x[u][k], f);
#pragma unroll
        for (int e = 0; e < EL; ++e) {
          o[e] = s.w[k] * g[e];
          dot[k] = fmaf(f[e], g[e], dot[k]);
        }
        st_v4(grad_perm + (size_t)s.row[k] * H + col, VT::pack(o));
      }
    }
  }
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    float d = dot[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0 && k < K) grad_probs[(size_t)t * K + k] = s.row[k] >= 0 ? d : 0.f;
  }
}

// Kinds of a combine slot.
enum : int { kRouted = 0, kZero = 1, kCopy = 2, kConst = 3, kBad = 4 };

// The combine splits each token's columns into `parts` runs of whole
// 32-vector steps, one warp each, in blocks of 4 warps: at H=7168 K=8 this
// measured 93.3 us against 106.7 for one warp per token in blocks of 8 (the
// shorter tasks leave less of a partial last wave, and the smaller blocks
// fit more resident warps at this kernel's register count).
constexpr int kCombineWarps = 4;

template <typename T, int KMAX>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const T* __restrict__ Y, const int32_t* __restrict__ row_map,
               const int32_t* __restrict__ ids, const float* __restrict__ scales,
               const T* __restrict__ shared_x, const T* __restrict__ ori_x,
               const uint8_t* __restrict__ active_mask, int mask_dims, int Tn, int H, int K,
               int N, int E, int zero_num, int copy_num, int const_num, const T* __restrict__ alpha1,
               const T* __restrict__ alpha2, const T* __restrict__ const_v, T* __restrict__ out,
               int32_t* status, int parts) {
  using VT = VecTraits<T>;
  constexpr int EL = VT::kElems;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long task = (long long)blockIdx.x * kCombineWarps + warp;
  const int t = (int)(task / parts), part = (int)(task - (long long)t * parts);
  if (t >= Tn) return;
  int my_kind = kBad, my_arg = -1;
  float my_s = 0.f;
  if (lane < K) {
    const int id = ids[(size_t)t * K + lane];
    my_s = scales[(size_t)t * K + lane];
    const long long zlo = E, clo = zlo + zero_num, klo = clo + copy_num, khi = klo + const_num;
    // A slot masked off takes no part: it adds nothing, like a zero expert,
    // and the permute gave it no row (row_map -1).  Its id must still lie in
    // [0, E + Z + C + Cn).
    const bool active =
        active_mask == nullptr ||
        (mask_dims == 1 ? active_mask[t] : active_mask[(size_t)t * K + lane]) != 0;
    if (id < 0 || (long long)id >= khi) {
      my_kind = kBad;
    } else if (!active || (id >= zlo && id < clo)) {
      my_kind = kZero;
    } else if (id < E) {
      // a routed slot must have a row inside the expert-major buffer
      const int r = row_map[(size_t)t * K + lane];
      if (r >= 0 && r < N) {
        my_kind = kRouted;
        my_arg = r;
      }
    } else if (id < klo) {
      my_kind = kCopy;
    } else {
      my_kind = kConst;
      my_arg = (int)(id - klo);
    }
    if (my_kind == kBad) set_status(status, MOE_ERR_BAD_ID);
  }
  int kind[KMAX], arg[KMAX];
  float sc[KMAX];
  bool need_ori = false;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    kind[k] = __shfl_sync(0xffffffffu, my_kind, k);
    arg[k] = __shfl_sync(0xffffffffu, my_arg, k);
    sc[k] = __shfl_sync(0xffffffffu, my_s, k);
    if (k >= K) kind[k] = kBad;
    need_ori |= (kind[k] == kCopy || kind[k] == kConst);
  }
  // this warp's columns: vectors [v_lo, v_hi) of the row
  const int nvec = H / EL;
  const int plen = ((nvec + parts - 1) / parts + 31) / 32 * 32;
  const int v_lo = part * plen, v_hi = min(nvec, v_lo + plen);
  for (int v = v_lo + lane; v < v_hi; v += 32) {
    const size_t col = (size_t)v * EL;
    // every load of this column chunk is issued before any arithmetic, so an
    // iteration waits for one memory round trip
    uint4 x[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (kind[k] == kRouted) x[k] = ld_nc_v4(Y + (size_t)arg[k] * H + col);
    uint4 ov = make_uint4(0u, 0u, 0u, 0u), sv = make_uint4(0u, 0u, 0u, 0u);
    if (need_ori) ov = ld_nc_v4(ori_x + (size_t)t * H + col);
    if (shared_x != nullptr) sv = ld_nc_v4(shared_x + (size_t)t * H + col);
    float ori[EL];
    if (need_ori) VT::unpack(ov, ori);
    float acc[EL];
#pragma unroll
    for (int e = 0; e < EL; ++e) acc[e] = 0.f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (kind[k] == kRouted) {
        float f[EL];
        VT::unpack(x[k], f);
#pragma unroll
        for (int e = 0; e < EL; ++e) acc[e] = fmaf(sc[k], f[e], acc[e]);
      } else if (kind[k] == kCopy) {
#pragma unroll
        for (int e = 0; e < EL; ++e) acc[e] = fmaf(sc[k], ori[e], acc[e]);
      } else if (kind[k] == kConst) {
        float a1[EL], a2[EL], cv[EL];
        const size_t off = (size_t)arg[k] * H + col;
        VT::unpack(ld_v4(alpha1 + off), a1);
        VT::unpack(ld_v4(alpha2 + off), a2);
        VT::unpack(ld_v4(const_v + off), cv);
#pragma unroll
        for (int e = 0; e < EL; ++e) acc[e] = fmaf(sc[k], fmaf(a1[e], ori[e], a2[e] * cv[e]), acc[e]);
      }
      // kZero and kBad add nothing
    }
    if (shared_x != nullptr) {
      float sh[EL];
      VT::unpack(sv, sh);
#pragma unroll
      for (int e = 0; e < EL; ++e) acc[e] += sh[e];
    }
    st_v4(out + (size_t)t * H + col, VT::pack(acc));
  }
}

template <typename T, int KMAX>
void launch_unpermute(const void* Y, const int32_t* rm, const float* p, int Tn, int H, int K, int N,
                      void* out, cudaStream_t s) {
  unpermute_kernel<T, KMAX><<<(Tn + kWarpsPerBlock - 1) / kWarpsPerBlock, 256, 0, s>>>(
      static_cast<const T*>(Y), rm, p, Tn, H, K, N, static_cast<T*>(out));
  count_launches(1);
}

template <typename T, int KMAX>
void launch_unpermute_grad(const void* g, const void* X, const int32_t* rm, const float* p, int Tn,
                           int H, int K, int N, void* gp, float* gprobs, cudaStream_t s) {
  unpermute_grad_kernel<T, KMAX><<<(Tn + kWarpsPerBlock - 1) / kWarpsPerBlock, 256, 0, s>>>(
      static_cast<const T*>(g), static_cast<const T*>(X), rm, p, Tn, H, K, N, static_cast<T*>(gp),
      gprobs);
  count_launches(1);
}

template <typename T, int KMAX>
void launch_combine(const void* Y, const int32_t* rm, const int32_t* ids, const float* sc,
                    const void* sh, const void* ori, const uint8_t* mask, int mask_dims, int Tn,
                    int H, int K, int N, int E, int Z, int C, int Cn, const void* a1,
                    const void* a2, const void* cv, void* out, int32_t* st, cudaStream_t s) {
  // column runs per token: up to 4, each at least 128 vectors
  const int parts = std::max(1, std::min(4, H / VecTraits<T>::kElems / 128));
  const long long tasks = (long long)Tn * parts;
  combine_kernel<T, KMAX><<<(unsigned)((tasks + kCombineWarps - 1) / kCombineWarps), kCombineWarps * 32, 0, s>>>(
      static_cast<const T*>(Y), rm, ids, sc, static_cast<const T*>(sh),
      static_cast<const T*>(ori), mask, mask_dims, Tn, H, K, N, E, Z, C, Cn,
      static_cast<const T*>(a1),
      static_cast<const T*>(a2), static_cast<const T*>(cv), static_cast<T*>(out), st, parts);
  count_launches(1);
}

// Pick the smallest compiled K bound that covers K (keeps the per-slot
// arrays in registers).
#define MOE_DISPATCH_K(K, FN, T, ...)          \
  do {                                         \
    if ((K) <= 2) FN<T, 2>(__VA_ARGS__);       \
    else if ((K) <= 4) FN<T, 4>(__VA_ARGS__);  \
    else if ((K) <= 8) FN<T, 8>(__VA_ARGS__);  \
    else FN<T, 16>(__VA_ARGS__);               \
  } while (0)

int check_rows(int dtype, int T, int H, int K, int N) {
  const int esz = dtype_size(dtype);
  if (esz == 0 || T < 0 || H <= 0 || K <= 0 || N < 0) return MOE_ERR_INVALID_ARG;
  if (K > kMaxK) return MOE_ERR_SHAPE;
  if (((size_t)H * esz) % 16 != 0) return MOE_ERR_SHAPE;
  if ((long long)T * K > 0x7fffffffLL) return MOE_ERR_SHAPE;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_unpermute(const void* expanded, int dtype, const int32_t* row_map,
                             const float* probs, int T, int H, int K, int N, void* out,
                             cudaStream_t stream) {
  int rc = check_rows(dtype, T, H, K, N);
  if (rc) return rc;
  if (T == 0) return MOE_OK;
  if (!row_map || !out || (N > 0 && !expanded)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(out) || (expanded && !aligned16(expanded))) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_BF16)
    MOE_DISPATCH_K(K, launch_unpermute, __nv_bfloat16, expanded, row_map, probs, T, H, K, N, out, stream);
  else
    MOE_DISPATCH_K(K, launch_unpermute, float, expanded, row_map, probs, T, H, K, N, out, stream);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_permute_grad(const void* grad_permuted, int dtype, const int32_t* row_map, int T,
                                int H, int K, int N, void* grad_tokens, cudaStream_t stream) {
  return moe_unpermute(grad_permuted, dtype, row_map, nullptr, T, H, K, N, grad_tokens, stream);
}

extern "C" int moe_unpermute_grad(const void* grad_out, const void* permuted_tokens, int dtype,
                                  const int32_t* row_map, const float* probs, int T, int H, int K,
                                  int N, void* grad_permuted, float* grad_probs,
                                  cudaStream_t stream) {
  int rc = check_rows(dtype, T, H, K, N);
  if (rc) return rc;
  if (T == 0) return MOE_OK;
  if (!grad_out || !row_map || !grad_probs || (N > 0 && (!permuted_tokens || !grad_permuted)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(grad_out) || (N > 0 && (!aligned16(permuted_tokens) || !aligned16(grad_permuted))))
    return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_BF16)
    MOE_DISPATCH_K(K, launch_unpermute_grad, __nv_bfloat16, grad_out, permuted_tokens, row_map,
                   probs, T, H, K, N, grad_permuted, grad_probs, stream);
  else
    MOE_DISPATCH_K(K, launch_unpermute_grad, float, grad_out, permuted_tokens, row_map, probs, T,
                   H, K, N, grad_permuted, grad_probs, stream);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_combine_masked(const void* expanded, int dtype, const int32_t* row_map,
                                  const int32_t* expert_ids, const float* scales,
                                  const void* shared_x, const void* ori_x,
                                  const uint8_t* active_mask, int mask_dims, int T, int H, int K,
                                  int N, int E, int zero_num, int copy_num, int const_num,
                                  const void* alpha1, const void* alpha2, const void* const_v,
                                  void* out, int32_t* dev_status, cudaStream_t stream) {
  if (active_mask != nullptr && mask_dims != 1 && mask_dims != 2) return MOE_ERR_INVALID_ARG;
  int rc = check_rows(dtype, T, H, K, N);
  if (rc) return rc;
  if (E <= 0 || zero_num < 0 || copy_num < 0 || const_num < 0) return MOE_ERR_INVALID_ARG;
  if ((long long)E + zero_num + copy_num + const_num > 0x7fffffffLL) return MOE_ERR_SHAPE;
  if ((long long)K > (long long)E + zero_num + copy_num + const_num) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!row_map || !expert_ids || !scales || !out) return MOE_ERR_INVALID_ARG;
  if (N > 0 && !expanded) return MOE_ERR_INVALID_ARG;
  if ((copy_num > 0 || const_num > 0) && !ori_x) return MOE_ERR_INVALID_ARG;
  if (const_num > 0 && (!alpha1 || !alpha2 || !const_v)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {expanded, shared_x, ori_x, alpha1, alpha2, const_v, out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_BF16)
    MOE_DISPATCH_K(K, launch_combine, __nv_bfloat16, expanded, row_map, expert_ids, scales,
                   shared_x, ori_x, active_mask, mask_dims, T, H, K, N, E, zero_num, copy_num,
                   const_num, alpha1, alpha2, const_v, out, dev_status, stream);
  else
    MOE_DISPATCH_K(K, launch_combine, float, expanded, row_map, expert_ids, scales, shared_x,
                   ori_x, active_mask, mask_dims, T, H, K, N, E, zero_num, copy_num, const_num,
                   alpha1, alpha2, const_v, out, dev_status, stream);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

extern "C" int moe_combine(const void* expanded, int dtype, const int32_t* row_map,
                           const int32_t* expert_ids, const float* scales, const void* shared_x,
                           const void* ori_x, int T, int H, int K, int N, int E, int zero_num,
                           int copy_num, int const_num, const void* alpha1, const void* alpha2,
                           const void* const_v, void* out, int32_t* dev_status,
                           cudaStream_t stream) {
  return moe_combine_masked(expanded, dtype, row_map, expert_ids, scales, shared_x, ori_x,
                            nullptr, 0, T, H, K, N, E, zero_num, copy_num, const_num, alpha1,
                            alpha2, const_v, out, dev_status, stream);
}
