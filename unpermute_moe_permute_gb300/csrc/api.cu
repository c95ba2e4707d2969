// C-ABI glue: status strings, device status readback, argument checks and
// dtype dispatch of the expert-MLP GEMMs.
#include <atomic>
#include <initializer_list>

#include "common.cuh"

namespace moe {

int launch_gmm_f32(bool swiglu, const float* A, const float* B0, const float* B1,
                   const int32_t* off, int N, int Kd, int Nout, int E, float* out, float* save,
                   cudaStream_t s);
int launch_gmm_bf16_gate_up(const void* A, const void* Wg, const void* Wu, const int32_t* off,
                            int N, int H, int I, int E, void* act, void* save, int32_t* status,
                            cudaStream_t s);
int launch_gmm_bf16_down(const void* A, const void* Wd, const int32_t* off, int N, int H, int I,
                         int E, void* out, int32_t* status, cudaStream_t s);
int launch_down_dgrad_bf16(const void* dY, const void* gate_up, const int32_t* off, int N, int H,
                           int I, int E, const void* Wd, void* dgu, int32_t* status,
                           cudaStream_t s);
int launch_gate_up_dgrad_bf16(const void* dgu, const int32_t* off, int N, int H, int I, int E,
                              const void* Wg, const void* Wu, void* dX, int32_t* status,
                              cudaStream_t s);
int launch_down_wgrad_bf16(const void* dY, const void* act, const int32_t* off, int N, int H,
                           int I, int E, void* dWd, int32_t* status, cudaStream_t s);
int launch_gate_up_wgrad_bf16(const void* dgu, const void* X, const int32_t* off, int N, int H,
                              int I, int E, void* dWg, void* dWu, int32_t* status,
                              cudaStream_t s);
int launch_wait_selftest(int32_t* status, cudaStream_t s);
int launch_gmm_bf16_gate_up_gather(const void* tokens, int T, const int32_t* sorted_indices, int K,
                                   const void* Wg, const void* Wu, const int32_t* off, int N, int H,
                                   int I, int E, void* act, void* save, int32_t* status,
                                   cudaStream_t s);
int launch_gate_up_wgrad_bf16_gather(const void* dgu, const void* tokens, int T,
                                     const int32_t* sorted_indices, int K, const int32_t* off,
                                     int N, int H, int I, int E, void* dWg, void* dWu,
                                     int32_t* status, cudaStream_t s);

static std::atomic<unsigned long long> g_launches{0};

void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

int check_mlp(const void* A, int dtype, const int32_t* off, int N, int H, int I, int E) {
  if (N < 0 || H <= 0 || I <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts) return MOE_ERR_SHAPE;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (!off || (N > 0 && !A)) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_F32 && (H % 4 || I % 4)) return MOE_ERR_SHAPE;
  if (dtype == MOE_BF16 && (H % 64 || I % 64)) return MOE_ERR_SHAPE;
  if ((long long)N * (2LL * I > H ? 2LL * I : H) > (1LL << 40)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_UNSUPPORTED: return "unsupported dtype, shape or device";
    case MOE_ERR_CAPACITY: return "output capacity exceeded";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_BAD_ID: return "expert id out of range or repeated in a row";
    default: return "unknown status";
  }
}

extern "C" int moe_abi_version(void) { return 1; }

extern "C" unsigned long long moe_kernel_launches(void) {
  return g_launches.load(std::memory_order_relaxed);
}

extern "C" int moe_selftest_bounded_wait(int32_t* dev_status, cudaStream_t stream) {
  if (dev_status == nullptr) return MOE_ERR_INVALID_ARG;
  return launch_wait_selftest(dev_status, stream);
}

extern "C" int moe_check_status(const int32_t* dev_status, cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (dev_status == nullptr) return MOE_OK;
  int32_t v = 0;
  if (cudaMemcpy(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return v;
}

extern "C" int moe_gate_up_swiglu(const void* permuted, int dtype, const int32_t* expert_offsets,
                                  int N, int H, int I, int E, const void* W_gate,
                                  const void* W_up, void* act, void* gate_up_save,
                                  int32_t* dev_status, cudaStream_t stream) {
  int rc = check_mlp(permuted, dtype, expert_offsets, N, H, I, E);
  if (rc) return rc;
  if (N == 0) return MOE_OK;
  if (!W_gate || !W_up || !act) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {permuted, W_gate, W_up, act, gate_up_save};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_F32)
    return launch_gmm_f32(true, static_cast<const float*>(permuted),
                          static_cast<const float*>(W_gate), static_cast<const float*>(W_up),
                          expert_offsets, N, H, I, E, static_cast<float*>(act),
                          static_cast<float*>(gate_up_save), stream);
  return launch_gmm_bf16_gate_up(permuted, W_gate, W_up, expert_offsets, N, H, I, E, act,
                                 gate_up_save, dev_status, stream);
}

extern "C" int moe_down_proj(const void* act, int dtype, const int32_t* expert_offsets, int N,
                             int H, int I, int E, const void* W_down, void* expanded,
                             int32_t* dev_status, cudaStream_t stream) {
  int rc = check_mlp(act, dtype, expert_offsets, N, H, I, E);
  if (rc) return rc;
  if (N == 0) return MOE_OK;
  if (!W_down || !expanded) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {act, W_down, expanded};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_F32)
    return launch_gmm_f32(false, static_cast<const float*>(act),
                          static_cast<const float*>(W_down), nullptr, expert_offsets, N, I, H, E,
                          static_cast<float*>(expanded), nullptr, stream);
  return launch_gmm_bf16_down(act, W_down, expert_offsets, N, H, I, E, expanded, dev_status,
                              stream);
}

extern "C" int moe_expert_mlp(const void* permuted, int dtype, const int32_t* expert_offsets,
                              int N, int H, int I, int E, const void* W_gate, const void* W_up,
                              const void* W_down, void* act, void* expanded, void* gate_up_save,
                              int32_t* dev_status, cudaStream_t stream) {
  int rc = moe_gate_up_swiglu(permuted, dtype, expert_offsets, N, H, I, E, W_gate, W_up, act,
                              gate_up_save, dev_status, stream);
  if (rc) return rc;
  return moe_down_proj(act, dtype, expert_offsets, N, H, I, E, W_down, expanded, dev_status,
                       stream);
}

static int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

extern "C" int moe_down_dgrad_swiglu(const void* grad_expanded, const void* gate_up_save,
                                     int dtype, const int32_t* expert_offsets, int N, int H,
                                     int I, int E, const void* W_down, void* dgu,
                                     int32_t* dev_status, cudaStream_t stream) {
  if (int rc = check_mlp(grad_expanded, dtype, expert_offsets, N, H, I, E)) return rc;
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (int rc = check_ptrs({grad_expanded, gate_up_save, W_down, dgu})) return rc;
  return launch_down_dgrad_bf16(grad_expanded, gate_up_save, expert_offsets, N, H, I, E, W_down,
                                dgu, dev_status, stream);
}

extern "C" int moe_gate_up_dgrad(const void* dgu, int dtype, const int32_t* expert_offsets, int N,
                                 int H, int I, int E, const void* W_gate, const void* W_up,
                                 void* d_permuted, int32_t* dev_status, cudaStream_t stream) {
  if (int rc = check_mlp(dgu, dtype, expert_offsets, N, H, I, E)) return rc;
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (int rc = check_ptrs({dgu, W_gate, W_up, d_permuted})) return rc;
  return launch_gate_up_dgrad_bf16(dgu, expert_offsets, N, H, I, E, W_gate, W_up, d_permuted,
                                   dev_status, stream);
}

extern "C" int moe_down_wgrad(const void* grad_expanded, const void* act, int dtype,
                              const int32_t* expert_offsets, int N, int H, int I, int E,
                              void* dW_down, int32_t* dev_status, cudaStream_t stream) {
  if (int rc = check_mlp(grad_expanded, dtype, expert_offsets, N, H, I, E)) return rc;
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (int rc = check_ptrs({dW_down})) return rc;
  if (N > 0)
    if (int rc = check_ptrs({grad_expanded, act})) return rc;
  return launch_down_wgrad_bf16(grad_expanded, act, expert_offsets, N, H, I, E, dW_down,
                                dev_status, stream);
}

extern "C" int moe_gate_up_wgrad(const void* dgu, const void* permuted, int dtype,
                                 const int32_t* expert_offsets, int N, int H, int I, int E,
                                 void* dW_gate, void* dW_up, int32_t* dev_status,
                                 cudaStream_t stream) {
  if (int rc = check_mlp(dgu, dtype, expert_offsets, N, H, I, E)) return rc;
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (int rc = check_ptrs({dW_gate, dW_up})) return rc;
  if (N > 0)
    if (int rc = check_ptrs({dgu, permuted})) return rc;
  return launch_gate_up_wgrad_bf16(dgu, permuted, expert_offsets, N, H, I, E, dW_gate, dW_up,
                                   dev_status, stream);
}

extern "C" int moe_shared_expert_mlp(const void* x, int T, int H, int I, const void* W_gate,
                                     const void* W_up, const void* W_down, void* act, void* out,
                                     int32_t* dev_status, cudaStream_t stream) {
  if (T < 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 64 || I % 64) return MOE_ERR_SHAPE;
  if ((long long)T * (2LL * I > H ? 2LL * I : H) > (1LL << 40)) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (int rc = check_ptrs({x, W_gate, W_up, W_down, act, out})) return rc;
  // one expert owning all T rows (no offsets array: the kernels imply [0, T])
  if (int rc = launch_gmm_bf16_gate_up(x, W_gate, W_up, nullptr, T, H, I, 1, act, nullptr,
                                       dev_status, stream))
    return rc;
  return launch_gmm_bf16_down(act, W_down, nullptr, T, H, I, 1, out, dev_status, stream);
}

// Arguments of the gathering gate/up calls beyond those of check_mlp.
static int check_gather(const void* tokens, int T, const int32_t* sorted_indices, int K, int N) {
  if (K < 1 || K > kMaxK || T < 0) return MOE_ERR_INVALID_ARG;
  if (N > 0 && (T < 1 || !tokens || !sorted_indices || !aligned16(tokens)))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

extern "C" int moe_gate_up_swiglu_gather(const void* tokens, int T, const int32_t* sorted_indices,
                                         int K, const int32_t* expert_offsets, int N, int H, int I,
                                         int E, const void* W_gate, const void* W_up, void* act,
                                         void* gate_up_save, int32_t* dev_status,
                                         cudaStream_t stream) {
  if (int rc = check_mlp(tokens, MOE_BF16, expert_offsets, N, H, I, E)) return rc;
  if (int rc = check_gather(tokens, T, sorted_indices, K, N)) return rc;
  if (N == 0) return MOE_OK;
  if (int rc = check_ptrs({W_gate, W_up, act})) return rc;
  if (gate_up_save && !aligned16(gate_up_save)) return MOE_ERR_INVALID_ARG;
  return launch_gmm_bf16_gate_up_gather(tokens, T, sorted_indices, K, W_gate, W_up,
                                        expert_offsets, N, H, I, E, act, gate_up_save,
                                        dev_status, stream);
}

extern "C" int moe_gate_up_wgrad_gather(const void* dgu, const void* tokens, int T,
                                        const int32_t* sorted_indices, int K,
                                        const int32_t* expert_offsets, int N, int H, int I, int E,
                                        void* dW_gate, void* dW_up, int32_t* dev_status,
                                        cudaStream_t stream) {
  if (int rc = check_mlp(dgu, MOE_BF16, expert_offsets, N, H, I, E)) return rc;
  if (int rc = check_gather(tokens, T, sorted_indices, K, N)) return rc;
  if (int rc = check_ptrs({dW_gate, dW_up})) return rc;
  if (N > 0)
    if (int rc = check_ptrs({dgu})) return rc;
  return launch_gate_up_wgrad_bf16_gather(dgu, tokens, T, sorted_indices, K, expert_offsets, N, H,
                                          I, E, dW_gate, dW_up, dev_status, stream);
}

extern "C" int moe_expert_mlp_grad(const void* grad_expanded, const void* permuted,
                                   const void* act, const void* gate_up_save, int dtype,
                                   const int32_t* expert_offsets, int N, int H, int I, int E,
                                   const void* W_gate, const void* W_up, const void* W_down,
                                   void* dgu, void* d_permuted, void* dW_gate, void* dW_up,
                                   void* dW_down, int32_t* dev_status, cudaStream_t stream) {
  int rc = moe_down_dgrad_swiglu(grad_expanded, gate_up_save, dtype, expert_offsets, N, H, I, E,
                                 W_down, dgu, dev_status, stream);
  if (rc) return rc;
  rc = moe_gate_up_dgrad(dgu, dtype, expert_offsets, N, H, I, E, W_gate, W_up, d_permuted,
                         dev_status, stream);
  if (rc) return rc;
  rc = moe_down_wgrad(grad_expanded, act, dtype, expert_offsets, N, H, I, E, dW_down, dev_status,
                      stream);
  if (rc) return rc;
  return moe_gate_up_wgrad(dgu, permuted, dtype, expert_offsets, N, H, I, E, dW_gate, dW_up,
                           dev_status, stream);
}
