/*
 * moe_gb300.h - C ABI of the single-GPU Mixture-of-Experts expert layer for
 * GB300 (sm_103a).
 *
 * The layer, in the order it runs:
 *   permute      expert histogram, scan and a stable expert-major scatter of
 *                the T*K routed slots (moe_permute)
 *   expert MLP   grouped gate/up GEMM with SwiGLU fused, grouped down GEMM
 *                (moe_gate_up_swiglu, moe_down_proj, moe_expert_mlp)
 *   unpermute    probability-weighted gather-sum back to token order
 *                (moe_unpermute) or the combine with shared and special
 *                experts (moe_combine)
 *   backward     moe_unpermute_grad, moe_expert_mlp_grad, moe_permute_grad
 *   indices      rank-major -> expert-major permute indices from per-(rank,
 *                expert) counts (moe_permute_indices)
 *
 * Notation: T tokens, H hidden size, K experts per token (top-K), E routed
 * experts, I expert intermediate size, f = t*K + k the flat slot index.
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless stated otherwise.  The caller
 *     allocates and owns every input, output and workspace buffer; the library
 *     never allocates or frees memory and never synchronises, except
 *     moe_check_status.
 *   - Every call is asynchronous and ordered on the given CUDA stream
 *     (0 = legacy default stream).
 *   - Tensors are dense, row-major, contiguous, with 16-byte aligned base
 *     pointers.  dtype is MOE_F32 or MOE_BF16 for activations and weights;
 *     router probabilities / scales are always float32; indices are int32.
 *   - Return value: MOE_OK, or an MOE_ERR_* code for arguments rejected on the
 *     host before anything is launched, or MOE_ERR_CUDA if a launch failed.
 *   - Errors only visible on the device (an expert id out of range or
 *     repeated within a row, an index capacity overflow, a bounded wait that
 *     ran out) are written, first one wins, to the optional caller-provided
 *     device int32 *dev_status (initialise it to 0).  moe_check_status reads
 *     it.  A kernel that meets such an error skips the offending element and
 *     still terminates.
 *   - Shapes: 1 <= K <= 16 and K <= E + number of special experts; E <= 1024;
 *     H % 8 == 0 (16-byte rows for bf16; fp32 needs H % 4 == 0 too).  The
 *     bf16 tensor-core GEMMs need H % 64 == 0 and I % 64 == 0.
 *
 * Sources: the id/range rules and the combine formulas follow the torch_npu
 * npu_moe_distribute_combine_v2 API reference (function description,
 * parameters, constraints); the expert-major layout and the index generation
 * follow hyper_parallel expert_parallel.py (_generate_permute_indices,
 * _permute, _unpermute); the unpermute forward/backward pair follows the
 * Ascend/pytorch PR "Update moe token unpermute DTensor support"; the grouped
 * GEMM + SwiGLU expert MLP follows the twinkle PR "NPU EP experts forward uses
 * NPU grouped matmul".
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1 /* null pointer, bad dtype, negative size       */
#define MOE_ERR_SHAPE 2       /* size rule broken (K, E, H alignment, ...)    */
#define MOE_ERR_UNSUPPORTED 3 /* dtype/shape combination not implemented, or
                                 the device is not sm_103                     */
#define MOE_ERR_CAPACITY 4    /* output capacity too small (device side)      */
#define MOE_ERR_CUDA 5        /* a CUDA launch or runtime call failed         */
#define MOE_ERR_TIMEOUT 6     /* a bounded device-side wait ran out           */
#define MOE_ERR_BAD_ID 7      /* expert id out of range or repeated in a row  */

/* ---- dtypes ------------------------------------------------------------ */
#define MOE_F32 0
#define MOE_BF16 1

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(int status);

/* ABI version: bumped when a signature changes. */
int moe_abi_version(void);

/* Number of kernels this library has launched in the process so far (all
 * devices, all streams).  For tracing and launch accounting. */
unsigned long long moe_kernel_launches(void);

/* Self-test of the bounded waits that every tensor-core kernel here relies
 * on.  The paper has no counterpart; it lets a deployment exercise the
 * failure path without faulting or hanging a GPU.  One thread waits, with
 * the same bounded mbarrier wait the GEMMs use, on a barrier that nothing
 * arrives on; after the wait limit (2 s) it records MOE_ERR_TIMEOUT in
 * dev_status (required, device int32, initialise to 0) and returns, so the
 * context stays usable.  Returns MOE_ERR_INVALID_ARG for a NULL dev_status. */
int moe_selftest_bounded_wait(int32_t* dev_status, cudaStream_t stream);

/* Synchronise `stream`, then read the device status word written by earlier
 * calls.  Returns MOE_OK or the first device-side MOE_ERR_* code, or
 * MOE_ERR_CUDA if the stream reported an error.  Does not reset the word. */
int moe_check_status(const int32_t* dev_status, cudaStream_t stream);

/* ---- permute (steps: histogram, scan, stable rank, row copy) -----------
 *
 * Definition (expert-major layout of hyper_parallel expert_parallel.py,
 * _generate_permute_indices docstring; gather convention of its
 * permuted_indices; id rules of the combine_v2 expert_ids parameter):
 *   tokens_per_expert[e] = #{f : expert_ids[f] == e}          (e < E)
 *   expert_offsets       = exclusive prefix sum, length E+1,
 *                          expert_offsets[E] = N = number of routed slots
 *   row_map[f]           = expert_offsets[e_f] + #{f' < f : e_f' == e_f}
 *                          (stable), or -1 when e_f >= E (special expert)
 *   sorted_indices[row_map[f]] = f
 *   permuted[row_map[f]] = tokens[f / K]                      (exact copy)
 * Ids in [E, E + num_special) are legal but not dispatched (zero/copy/const
 * experts handled by moe_combine).  With num_special == 0, N = T*K.
 *
 * Arguments
 *   tokens          [T, H] dtype, or NULL to compute only the routing
 *   expert_ids      [T, K] int32
 *   permuted        [T*K, H] dtype capacity (rows >= N untouched), or NULL
 *                   when tokens is NULL
 *   sorted_indices  [T*K] int32 capacity; first N entries written
 *   row_map         [T*K] int32
 *   tokens_per_expert [E] int32, expert_offsets [E+1] int32
 *   workspace       device scratch of moe_permute_workspace_size(T, K, E)
 *                   bytes, 16-byte aligned (else MOE_ERR_INVALID_ARG):
 *                   ceil(T*K/512) blocks of E int32 expert counts
 *                   (padded to 8 bytes), then one 8-byte completion flag
 *                   per block (a routing with more than 64 such blocks
 *                   uses half as many blocks of 1024 slots, in the same
 *                   bytes).  Its contents need no clearing: each call
 *                   stamps the flags with a value no earlier call of the
 *                   process used (seeded from the clock, the process id and
 *                   a random draw, so a stamp left by another process
 *                   matches only by a 64-bit coincidence).
 *   dev_status      optional; receives MOE_ERR_BAD_ID for an id outside
 *                   [0, E + num_special) or repeated within a row (the slot
 *                   is then treated as not dispatched), and MOE_ERR_TIMEOUT
 *                   if the one-launch routing's bounded wait for its other
 *                   blocks ran out (then the waiting blocks' slots get
 *                   row_map -1 and are not copied; the result is incomplete
 *                   but no write leaves the output buffers)
 */
size_t moe_permute_workspace_size(int T, int K, int E);
int moe_permute(const void* tokens, int dtype, const int32_t* expert_ids, int T, int H, int K,
                int E, int num_special, void* permuted, int32_t* sorted_indices, int32_t* row_map,
                int32_t* tokens_per_expert, int32_t* expert_offsets, void* workspace,
                size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/* moe_permute without a caller-provided workspace.  The paper has no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory themselves: a plugin that its host framework hands
 * only input and output buffers, or a process whose device memory is all
 * reserved by another allocator (a cudaMalloc there would fail, or
 * synchronise the device at a bad moment).
 *
 * The workspace of moe_permute (per-block expert counts and completion
 * flags) lives in one file-scope device array of
 * MOE_PERMUTE_STATIC_SCRATCH_INTS int32 (256 KiB) that every GPU which loads
 * this library holds until the process exits.  It is enough when
 * moe_permute_workspace_size(T, K, E) <= 4 * MOE_PERMUTE_STATIC_SCRATCH_INTS,
 * about ceil(T*K / 512) * (E + 2) int32; larger problems return
 * MOE_ERR_CAPACITY before anything is launched.
 *   - The first call on a device looks up that device's address of the
 *     array (cudaGetSymbolAddress, with the device current); make that first
 *     call before any stream capture.
 *   - Every call uses the same array, so calls whose kernels can overlap on
 *     the GPU (different streams, no ordering between them) race with each
 *     other and must be serialised by the caller.  The array keeps the last
 *     call's contents; a call reads only counts it wrote itself and flags
 *     stamped with its own value, so nothing needs clearing between calls.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * Arguments and results are those of moe_permute. */
#define MOE_PERMUTE_STATIC_SCRATCH_INTS 65536
int moe_permute_static_scratch(const void* tokens, int dtype, const int32_t* expert_ids, int T,
                               int H, int K, int E, int num_special, void* permuted,
                               int32_t* sorted_indices, int32_t* row_map,
                               int32_t* tokens_per_expert, int32_t* expert_offsets,
                               int32_t* dev_status, cudaStream_t stream);

/* moe_permute with an activity mask (the x_active_mask parameter of the
 * torch_npu npu_moe_distribute_combine_v2 API reference): mask_dims 1 =
 * active_mask [T] (one byte per token), 2 = active_mask [T, K] (one byte per
 * slot); a zero byte means the token / slot takes no part, so it is not
 * dispatched (row_map = -1, not counted).  Ids of masked slots are still
 * validated.  active_mask NULL = every slot active (moe_permute). */
int moe_permute_masked(const void* tokens, int dtype, const int32_t* expert_ids, int T, int H,
                       int K, int E, int num_special, const uint8_t* active_mask, int mask_dims,
                       void* permuted, int32_t* sorted_indices, int32_t* row_map,
                       int32_t* tokens_per_expert, int32_t* expert_offsets, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/* The row copy of moe_permute on its own, for a routing the caller already
 * holds (a second tensor permuted the same way, or a routing rebuilt with
 * moe_invert_sorted_indices):
 *   permuted[row_map[t*K+k]] = tokens[t]          (exact copy)
 * tokens [T, H] dtype, row_map [T*K] int32, permuted [N, H] dtype (N = rows
 * of the buffer).  Slots whose row_map entry lies outside [0, N) (-1 marks a
 * slot that is not dispatched) are skipped, so no entry can address memory
 * outside permuted; rows no slot maps to are not written.  Row gather of
 * hyper_parallel expert_parallel.py, _permute (x[permuted_indices]). */
int moe_permute_rows(const void* tokens, int dtype, const int32_t* row_map, int T, int H, int K,
                     int N, void* permuted, cudaStream_t stream);

/* Rebuild row_map [TK] from sorted_indices [N] (row_map[sorted[i]] = i,
 * every other entry -1).  For callers that keep only sorted_indices. */
int moe_invert_sorted_indices(const int32_t* sorted_indices, int N, int TK, int32_t* row_map,
                              cudaStream_t stream);

/* ---- expert MLP (grouped GEMMs; twinkle PR: GMM + SwiGLU) --------------
 *
 * Rows [expert_offsets[e], expert_offsets[e+1]) of the expert-major buffer
 * belong to expert e; expert_offsets is read on the device (no host sync).
 * Weights are stacked per expert, nn.Linear layout (reduction dim last):
 *   W_gate, W_up [E, I, H]      W_down [E, H, I]
 * moe_gate_up_swiglu:  g = X W_gate[e]^T, u = X W_up[e]^T (fp32 accumulate),
 *                      act = silu(g) * u, silu(x) = x / (1 + e^-x)
 *                      act [N, I] dtype.  gate_up_save [N, 2I] dtype
 *                      (nullable) receives g in columns [0, I) and u in
 *                      [I, 2I) for the backward.
 * moe_down_proj:       expanded = act W_down[e]^T, expanded [N, H] dtype.
 * N is the row capacity of the buffers; rows >= expert_offsets[E] are not
 * touched.  bf16 runs on tcgen05 tensor cores (fp32 accumulators in tensor
 * memory); fp32 runs on FP32 FMA units.
 */
int moe_gate_up_swiglu(const void* permuted, int dtype, const int32_t* expert_offsets, int N,
                       int H, int I, int E, const void* W_gate, const void* W_up, void* act,
                       void* gate_up_save, int32_t* dev_status, cudaStream_t stream);
int moe_down_proj(const void* act, int dtype, const int32_t* expert_offsets, int N, int H, int I,
                  int E, const void* W_down, void* expanded, int32_t* dev_status,
                  cudaStream_t stream);
/* Both of the above, in order. */
int moe_expert_mlp(const void* permuted, int dtype, const int32_t* expert_offsets, int N, int H,
                   int I, int E, const void* W_gate, const void* W_up, const void* W_down,
                   void* act, void* expanded, void* gate_up_save, int32_t* dev_status,
                   cudaStream_t stream);

/* ---- shared expert (torch_npu npu_moe_distribute_combine_v2 API reference,
 * shared_expert_x: the value added after the combine; hyper_parallel
 * expert_parallel.py, combine_start: the combine split so that a shared
 * expert forward can run meanwhile) ---------------------------------------
 *
 * The shared expert's MLP over every token, on the caller's stream:
 *   act = silu(x W_gate^T) * (x W_up^T),   out = act W_down^T
 * x [T, H] bf16, W_gate and W_up [I, H], W_down [H, I] bf16, act [T, I] and
 * out [T, H] bf16 (caller-owned).  The same tcgen05 kernels as the routed
 * experts, as one expert that owns all T rows.  Run it on a second stream,
 * concurrently with the routed path, and pass out as moe_combine's
 * shared_x after the stream join (an event); moe_combine adds it.
 * H and I multiples of 64; returns MOE_ERR_SHAPE otherwise.
 */
int moe_shared_expert_mlp(const void* x, int T, int H, int I, const void* W_gate,
                          const void* W_up, const void* W_down, void* act, void* out,
                          int32_t* dev_status, cudaStream_t stream);

/* ---- the permute fused into the gate/up GEMMs (bf16) --------------------
 *
 * The twinkle PR "NPU EP experts forward uses NPU grouped matmul" feeds the
 * grouped matmul with x[permuted_indices], a gathered copy of the tokens.
 * These two calls give exactly what moe_gate_up_swiglu and
 * moe_gate_up_wgrad give on that copy,
 *   permuted[i] = tokens[sorted_indices[i] / K]      (i < expert_offsets[E]),
 * but read its rows straight from the token matrix (16-byte cp.async copies
 * by the GEMMs' producer warp), so neither the permute's row copy nor the [N, H]
 * permuted buffer is needed: run moe_permute with tokens = NULL for
 * sorted_indices and expert_offsets.
 *   tokens          [T, H] bf16 (T >= 1 when N > 0)
 *   sorted_indices  [N] int32 from moe_permute (its first expert_offsets[E]
 *                   entries are read; an entry outside [0, T*K) reads token
 *                   row 0 instead of faulting)
 *   K               slots per token of that routing (1 <= K <= 16)
 * Other arguments as moe_gate_up_swiglu / moe_gate_up_wgrad (bf16 only;
 * the gathering kernels are single-CTA).  Returns MOE_ERR_UNSUPPORTED for
 * fp32, MOE_ERR_INVALID_ARG for a NULL or misaligned pointer or bad T, K.
 */
int moe_gate_up_swiglu_gather(const void* tokens, int T, const int32_t* sorted_indices, int K,
                              const int32_t* expert_offsets, int N, int H, int I, int E,
                              const void* W_gate, const void* W_up, void* act,
                              void* gate_up_save, int32_t* dev_status, cudaStream_t stream);
int moe_gate_up_wgrad_gather(const void* dgu, const void* tokens, int T,
                             const int32_t* sorted_indices, int K, const int32_t* expert_offsets,
                             int N, int H, int I, int E, void* dW_gate, void* dW_up,
                             int32_t* dev_status, cudaStream_t stream);

/* ---- unpermute forward / backward (Ascend/pytorch PR "Update moe token
 * unpermute DTensor support": tokens shard on H, the probs grad is a sum
 * over H) -----------------------------------------------------------------
 *
 * moe_unpermute:       out[t] = sum_{k ascending} probs[t,k] * expanded[row_map[t*K+k]]
 *                      fp32 accumulation, one rounding to dtype; probs NULL
 *                      means weight 1; row_map -1 slots add nothing.
 *                      expanded [N, H], probs [T, K] f32, out [T, H].
 * moe_unpermute_grad:  grad_permuted[row_map[f]] = probs[f] * grad_out[t]
 *                      grad_probs[t, k] = sum_h permuted_tokens[row_map[f], h] * grad_out[t, h]
 *                      (fp32; 0 for row_map -1).  permuted_tokens is the
 *                      forward input of moe_unpermute.  grad_permuted rows
 *                      that no slot maps to are not written.
 * moe_permute_grad:    grad_tokens[t] = sum_k grad_permuted[row_map[t*K+k]]
 *                      (backward of the permute row gather: duplicate
 *                      slots of one token accumulate).
 */
int moe_unpermute(const void* expanded, int dtype, const int32_t* row_map, const float* probs,
                  int T, int H, int K, int N, void* out, cudaStream_t stream);
int moe_unpermute_grad(const void* grad_out, const void* permuted_tokens, int dtype,
                       const int32_t* row_map, const float* probs, int T, int H, int K, int N,
                       void* grad_permuted, float* grad_probs, cudaStream_t stream);
int moe_permute_grad(const void* grad_permuted, int dtype, const int32_t* row_map, int T, int H,
                     int K, int N, void* grad_tokens, cudaStream_t stream);

/* ---- combine with shared and special experts (npu_moe_distribute_combine_v2
 * API reference, function description: x = Sum(expert_scales * y) +
 * shared_expert_x, special-expert closed forms) ----------------------------
 *
 *   x[t] = sum_k scales[t,k] * y(t,k) + shared_x[t]      (fp32, k ascending)
 *   y(t,k) = expanded[row_map[t*K+k]]                    id <  E
 *          = 0                                           E <= id < E+Z        (zero)
 *          = ori_x[t]                                    E+Z <= id < E+Z+C    (copy)
 *          = alpha1[j] * ori_x[t] + alpha2[j] * const_v[j],  j = id-E-Z-C    (const)
 * shared_x [T,H] nullable; ori_x [T,H] required when copy_num + const_num > 0;
 * alpha1/alpha2/const_v [const_num, H] (dtype) required when const_num > 0.
 * Ids outside [0, E+Z+C+Cn) set MOE_ERR_BAD_ID and contribute 0; so does a
 * routed slot (id < E) whose row_map entry lies outside [0, N).
 */
int moe_combine(const void* expanded, int dtype, const int32_t* row_map, const int32_t* expert_ids,
                const float* scales, const void* shared_x, const void* ori_x, int T, int H, int K,
                int N, int E, int zero_num, int copy_num, int const_num, const void* alpha1,
                const void* alpha2, const void* const_v, void* out, int32_t* dev_status,
                cudaStream_t stream);

/* moe_combine with the activity mask of moe_permute_masked: a slot (or every
 * slot of a token) masked off contributes nothing to the weighted sum, and
 * its row_map entry is not read (moe_permute_masked gives it -1); its id must
 * still lie in [0, E+Z+C+Cn), else MOE_ERR_BAD_ID.  The shared-expert term is
 * still added.  active_mask NULL = moe_combine. */
int moe_combine_masked(const void* expanded, int dtype, const int32_t* row_map,
                       const int32_t* expert_ids, const float* scales, const void* shared_x,
                       const void* ori_x, const uint8_t* active_mask, int mask_dims, int T, int H,
                       int K, int N, int E, int zero_num, int copy_num, int const_num,
                       const void* alpha1, const void* alpha2, const void* const_v, void* out,
                       int32_t* dev_status, cudaStream_t stream);

/* ---- rank-major -> expert-major permute indices (hyper_parallel
 * expert_parallel.py, _generate_permute_indices) -----------------------------
 *
 * counts [R*E] int32, entry r*E+e = rows received from rank r for local
 * expert e, laid out rank-major.  Writes
 *   indices[i]  = rank-major source position of expert-major destination i
 *                 (blocks visited e-major then r), i < total
 *   tokens_per_expert[e] = sum_r counts[r*E+e]
 *   *total      = sum of counts (device int32)
 * If total > capacity nothing is written to indices and dev_status gets
 * MOE_ERR_CAPACITY.  R*E <= 2048 (the combine_v2 constraint on local experts
 * times EP size).  The counts are summed in 64 bits first: if the sum of all
 * counts does not fit in int32, nothing but *total = -1 is written and
 * dev_status gets MOE_ERR_CAPACITY.  Negative counts count as 0 and set
 * MOE_ERR_INVALID_ARG.
 */
int moe_permute_indices(const int32_t* counts, int R, int E, int32_t* indices, int capacity,
                        int32_t* tokens_per_expert, int32_t* total, int32_t* dev_status,
                        cudaStream_t stream);

/* Deredundancy dispatch indices (hyper_parallel expert_parallel.py,
 * _generate_deredundency_dispatch_indices): counts [R, E_all] row-major, entry
 * r*E_all+e = rows that source r holds for expert e; the source buffer is the
 * sources' expert-major buffers concatenated, i.e. blocks in (r, e) order.
 * For the window of experts [col_start, col_start + col_count) (an outer
 * expert range: iep_size * num_local_experts experts) the output visits
 * blocks column-major (e = col_start.., then r = 0..R-1), i.e. ordered
 * [destination, local expert, source]:
 *   indices[i] = source position of destination i,  i < *total
 *   tokens_per_column[c] = sum_r counts[r*E_all + col_start + c]
 * moe_permute_indices is the full window (col_start 0, col_count E).
 * Same limits and capacity behaviour as moe_permute_indices (R*E_all <= 2048). */
int moe_permute_indices_window(const int32_t* counts, int R, int E_all, int col_start,
                               int col_count, int32_t* indices, int capacity,
                               int32_t* tokens_per_column, int32_t* total, int32_t* dev_status,
                               cudaStream_t stream);

/* ---- expert MLP backward (bf16) -----------------------------------------
 *
 * For the rows of expert e: X = permuted, dY = grad_expanded, A = act,
 * (g, u) = gate_up_save (from moe_gate_up_swiglu), s = sigmoid(g):
 *   dA  = dY W_down[e]
 *   dg  = dA * u * s * (1 + g (1 - s)),  du = dA * silu(g)   -> dgu [N, 2I]
 *   d_permuted = dg W_gate[e] + du W_up[e]
 *   dW_down[e] = dY^T A,  dW_gate[e] = dg^T X,  dW_up[e] = du^T X
 * Experts without rows get zero weight gradients.  dgu is a caller-owned
 * [N, 2I] dtype buffer that holds (dg, du) between the kernels.
 */
int moe_expert_mlp_grad(const void* grad_expanded, const void* permuted, const void* act,
                        const void* gate_up_save, int dtype, const int32_t* expert_offsets, int N,
                        int H, int I, int E, const void* W_gate, const void* W_up,
                        const void* W_down, void* dgu, void* d_permuted, void* dW_gate,
                        void* dW_up, void* dW_down, int32_t* dev_status, cudaStream_t stream);

/* The four grouped GEMMs of moe_expert_mlp_grad, one kernel each, in the
 * order that call runs them (bf16 only).  A caller whose expert weights are
 * frozen (adapter training) runs the two dgrads and skips the wgrads.
 *   moe_down_dgrad_swiglu: dgu = SwiGLU-backward(grad_expanded W_down[e], g, u)
 *   moe_gate_up_dgrad:     d_permuted = dg W_gate[e] + du W_up[e]
 *   moe_down_wgrad:        dW_down[e] = grad_expanded_e^T act_e
 *   moe_gate_up_wgrad:     dW_gate[e] = dg_e^T X_e,  dW_up[e] = du_e^T X_e  */
int moe_down_dgrad_swiglu(const void* grad_expanded, const void* gate_up_save, int dtype,
                          const int32_t* expert_offsets, int N, int H, int I, int E,
                          const void* W_down, void* dgu, int32_t* dev_status, cudaStream_t stream);
int moe_gate_up_dgrad(const void* dgu, int dtype, const int32_t* expert_offsets, int N, int H,
                      int I, int E, const void* W_gate, const void* W_up, void* d_permuted,
                      int32_t* dev_status, cudaStream_t stream);
int moe_down_wgrad(const void* grad_expanded, const void* act, int dtype,
                   const int32_t* expert_offsets, int N, int H, int I, int E, void* dW_down,
                   int32_t* dev_status, cudaStream_t stream);
int moe_gate_up_wgrad(const void* dgu, const void* permuted, int dtype,
                      const int32_t* expert_offsets, int N, int H, int I, int E, void* dW_gate,
                      void* dW_up, int32_t* dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
