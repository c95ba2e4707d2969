// fp32 grouped GEMMs of the expert MLP on the FP32 FMA pipes.
//
// fp32 inputs need fp32 products: TF32 tensor cores round the operands to 10
// mantissa bits, far outside a 1e-5 relative tolerance, so this path stays on
// FFMA.  Tiles of 64 x 64 outputs, 256 threads, 4 x 4 outputs per thread, a
// 16-deep k slice staged in shared memory.  One CTA per (expert m-tile,
// n-tile); the expert of an m-tile comes from the device-side offsets.
//
// gate/up variant: two accumulators (gate and up) share the A tile, and the
// epilogue writes act = silu(g) * u (SwiGLU, fused), optionally saving g, u.
#include "common.cuh"
#include "sched.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, kThreads = 256;

template <bool kSwiglu>
__global__ void __launch_bounds__(kThreads)
gmm_f32_kernel(const float* __restrict__ A, const float* __restrict__ B0, const float* __restrict__ B1,
               const int32_t* __restrict__ off, int N, int Kd, int Nout, int E,
               float* __restrict__ out, float* __restrict__ save) {
  __shared__ int32_t prefix[kMaxExperts + 1];
  __shared__ int32_t offs[kMaxExperts + 1];
  __shared__ int32_t scratch[32];
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs0[BK][BN + 4];
  __shared__ float Bs1[kSwiglu ? BK : 1][BN + 4];
  stage_offsets(off, E, N, offs, scratch);
  build_tile_prefix(offs, E, N, BM, prefix, scratch);
  const int tile = blockIdx.x;
  if (tile >= prefix[E]) return;  // uniform across the CTA
  const int e = find_expert(prefix, E, tile);
  const ExpertRows rows = expert_rows(offs, e, N);
  const int row0 = rows.lo + (tile - prefix[e]) * BM;
  const int n0 = blockIdx.y * BN;
  const float* b0 = B0 + (size_t)e * Nout * Kd;
  const float* b1 = kSwiglu ? B1 + (size_t)e * Nout * Kd : nullptr;

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;  // 16 x 16 threads
  float acc0[4][4] = {}, acc1[4][4] = {};
  // loader mapping: 64 rows x 16 k = 256 float4
  const int lr = tid >> 2, lc = (tid & 3) * 4;
  for (int k0 = 0; k0 < Kd; k0 += BK) {
    {
      const int r = row0 + lr, c = k0 + lc;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < rows.hi && c < Kd) v = *reinterpret_cast<const float4*>(A + (size_t)r * Kd + c);
      As[lc + 0][lr] = v.x;
      As[lc + 1][lr] = v.y;
      As[lc + 2][lr] = v.z;
      As[lc + 3][lr] = v.w;
      const int n = n0 + lr;
      float4 w0 = make_float4(0.f, 0.f, 0.f, 0.f), w1 = w0;
      if (n < Nout && c < Kd) {
        w0 = *reinterpret_cast<const float4*>(b0 + (size_t)n * Kd + c);
        if (kSwiglu) w1 = *reinterpret_cast<const float4*>(b1 + (size_t)n * Kd + c);
      }
      Bs0[lc + 0][lr] = w0.x;
      Bs0[lc + 1][lr] = w0.y;
      Bs0[lc + 2][lr] = w0.z;
      Bs0[lc + 3][lr] = w0.w;
      if (kSwiglu) {
        Bs1[lc + 0][lr] = w1.x;
        Bs1[lc + 1][lr] = w1.y;
        Bs1[lc + 2][lr] = w1.z;
        Bs1[lc + 3][lr] = w1.w;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4], c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs0[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc0[i][j] = fmaf(a[i], b[j], acc0[i][j]);
      if (kSwiglu) {
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = Bs1[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc1[i][j] = fmaf(a[i], c[j], acc1[i][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= rows.hi) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= Nout) continue;
      if (kSwiglu) {
        const float g = acc0[i][j], u = acc1[i][j];
        out[(size_t)r * Nout + n] = g / (1.f + expf(-g)) * u;
        if (save) {
          save[(size_t)r * 2 * Nout + n] = g;
          save[(size_t)r * 2 * Nout + Nout + n] = u;
        }
      } else {
        out[(size_t)r * Nout + n] = acc0[i][j];
      }
    }
  }
}

}  // namespace

// Upper bound of sum_e ceil(M_e / BM) over experts: N / BM + E.
int launch_gmm_f32(bool swiglu, const float* A, const float* B0, const float* B1,
                   const int32_t* off, int N, int Kd, int Nout, int E, float* out, float* save,
                   cudaStream_t s) {
  if (N == 0) return MOE_OK;
  const dim3 grid((N + BM - 1) / BM + E, (Nout + BN - 1) / BN);
  if (grid.x > 0x7fffffffu) return MOE_ERR_SHAPE;
  if (swiglu)
    gmm_f32_kernel<true><<<grid, kThreads, 0, s>>>(A, B0, B1, off, N, Kd, Nout, E, out, save);
  else
    gmm_f32_kernel<false><<<grid, kThreads, 0, s>>>(A, B0, nullptr, off, N, Kd, Nout, E, out, nullptr);
  count_launches(1);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
