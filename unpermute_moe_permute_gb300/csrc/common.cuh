// Shared device/host helpers of the MoE GB300 library (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (GB300) only"
#endif

namespace moe {

constexpr int kMaxK = 16;
constexpr int kMaxExperts = 1024;

// First device-side error wins; later ones are dropped.
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// 16-byte vector of activations: 8 bf16 or 4 fp32.
struct alignas(16) Vec16 {
  uint4 u;
};

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// Streaming store: the written rows are not re-read by this kernel.
__device__ __forceinline__ void st_cs_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Elements per 16-byte vector for each dtype.
template <typename T>
struct VecTraits;
template <>
struct VecTraits<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};
template <>
struct VecTraits<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void unpack2(uint32_t w, float* f) {
    // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32.
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xFFFF0000u);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    unpack2(v.x, f + 0);
    unpack2(v.y, f + 2);
    unpack2(v.z, f + 4);
    unpack2(v.w, f + 6);
  }
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                      pack2(f[6], f[7]));
  }
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace moe

// ---- host-side helpers ------------------------------------------------------

#define MOE_LAUNCH_CHECK()                                   \
  do {                                                       \
    if (cudaPeekAtLastError() != cudaSuccess) {              \
      (void)cudaGetLastError();                              \
      return MOE_ERR_CUDA;                                   \
    }                                                        \
  } while (0)

// Launch accounting: every host entry point adds the kernels it launched.
namespace moe {
void count_launches(int n);
}

namespace moe {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int dtype_size(int dtype) { return dtype == MOE_F32 ? 4 : (dtype == MOE_BF16 ? 2 : 0); }

// Number of SMs of the current device (cached per device).
int sm_count();

}  // namespace moe
