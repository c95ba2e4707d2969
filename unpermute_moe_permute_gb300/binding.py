"""Python binding of the C ABI in ``include/moe_gb300.h`` (ctypes).

Argument marshalling only: every step of the layer runs in the CUDA kernels
of ``libmoe_gb300.so``.  PyTorch supplies device memory (outputs are
allocated with ``torch.empty`` when the caller does not pass them) and the
current CUDA stream.  There is no CPU path: if the library is not built, or a
tensor is not on a CUDA device, the call raises.

Function names match the C entry points.  A non-zero status raises
:class:`MoeError`.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import NamedTuple, Optional

import torch

from .build import LIB_PATH, INCLUDE

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_SHAPE = 2
MOE_ERR_UNSUPPORTED = 3
MOE_ERR_CAPACITY = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_BAD_ID = 7

MOE_F32 = 0
MOE_BF16 = 1

_DTYPES = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16}


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: status {status} ({text})")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_abi_version": ([], _I),
    "moe_kernel_launches": ([], ctypes.c_ulonglong),
    "moe_check_status": ([_P, _P], _I),
    "moe_permute_workspace_size": ([_I, _I, _I], _SZ),
    "moe_permute": ([_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P], _I),
    "moe_permute_masked": ([_P, _I, _P, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P, _SZ,
                            _P, _P], _I),
    "moe_combine_masked": ([_P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                            _P, _P, _P, _P, _P, _P], _I),
    "moe_invert_sorted_indices": ([_P, _I, _I, _P, _P], _I),
    "moe_permute_rows": ([_P, _I, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_permute_static_scratch": ([_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P],
                                   _I),
    "moe_gate_up_swiglu": ([_P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_down_proj": ([_P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_expert_mlp": ([_P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_unpermute": ([_P, _I, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_unpermute_grad": ([_P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_permute_grad": ([_P, _I, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_combine": ([_P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P,
                     _P, _P, _P], _I),
    "moe_permute_indices": ([_P, _I, _I, _P, _I, _P, _P, _P, _P], _I),
    "moe_permute_indices_window": ([_P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P], _I),
    "moe_expert_mlp_grad": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                             _P, _P, _P, _P], _I),
    "moe_down_dgrad_swiglu": ([_P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_gate_up_dgrad": ([_P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_down_wgrad": ([_P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_gate_up_wgrad": ([_P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_selftest_bounded_wait": ([_P, _P], _I),
    "moe_shared_expert_mlp": ([_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_gate_up_swiglu_gather": ([_P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_gate_up_wgrad_gather": ([_P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
}


def header_symbols() -> list:
    """Function names declared in include/moe_gb300.h."""
    text = open(os.path.join(INCLUDE, "moe_gb300.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def load_library(path: Optional[str] = None):
    """Load libmoe_gb300.so (no CUDA call is made) and declare signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is not built; run `python -m unpermute_moe_permute_gb300.build` "
            "(there is no fallback path)")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def _call(name: str, *args):
    lib = load_library()
    rc = getattr(lib, name)(*args)
    if rc != MOE_OK:
        raise MoeError(name, rc, lib.moe_status_string(rc).decode())


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device (no CPU path)")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _check(t: Optional[torch.Tensor], dtype, name: str):
    if t is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


# ---------------------------------------------------------------- status

def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word for the dev_status arguments."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def status_name(status: int) -> str:
    """Name of a status code (moe_status_string)."""
    return load_library().moe_status_string(int(status)).decode()


def moe_selftest_bounded_wait(dev_status) -> None:
    """Run the bounded-wait self-test (about 2 s on the GPU): dev_status
    receives MOE_ERR_TIMEOUT."""
    _call("moe_selftest_bounded_wait", _ptr(dev_status), _stream())


def moe_kernel_launches() -> int:
    """Kernels launched by the library in this process so far."""
    return int(load_library().moe_kernel_launches())


def moe_check_status(dev_status: Optional[torch.Tensor]) -> int:
    """Synchronise the current stream and return the device status word."""
    lib = load_library()
    return int(lib.moe_check_status(_ptr(dev_status), _stream()))


# ---------------------------------------------------------------- permute

class PermuteResult(NamedTuple):
    permuted: Optional[torch.Tensor]      # [T*K, H] capacity, rows < expert_offsets[E] valid
    sorted_indices: torch.Tensor          # [T*K] int32 capacity
    row_map: torch.Tensor                 # [T*K] int32, -1 for special slots
    tokens_per_expert: torch.Tensor       # [E] int32
    expert_offsets: torch.Tensor          # [E+1] int32


def _mask(m: torch.Tensor, T: int, K: int) -> torch.Tensor:
    if m.dtype not in (torch.bool, torch.uint8):
        raise ValueError("active_mask must be bool or uint8")
    if tuple(m.shape) not in ((T,), (T, K)):
        raise ValueError("active_mask must be [T] or [T, K]")
    return m


def moe_permute_workspace_size(T: int, K: int, E: int) -> int:
    return int(load_library().moe_permute_workspace_size(T, K, E))


def moe_permute(tokens: Optional[torch.Tensor], expert_ids: torch.Tensor, num_experts: int,
                num_special: int = 0, *, permuted=None, sorted_indices=None, row_map=None,
                tokens_per_expert=None, expert_offsets=None, workspace=None,
                dev_status=None, active_mask=None) -> PermuteResult:
    """active_mask: optional bool/uint8 [T] (per token) or [T, K] (per slot);
    masked-off slots are not dispatched."""
    _check(expert_ids, torch.int32, "expert_ids")
    T, K = expert_ids.shape
    dev = expert_ids.device
    H = tokens.shape[1] if tokens is not None else 0
    dt = _dtype(tokens) if tokens is not None else MOE_BF16
    TK = T * K
    if tokens is not None and permuted is None:
        permuted = torch.empty((TK, H), dtype=tokens.dtype, device=dev)
    if sorted_indices is None:
        sorted_indices = torch.empty(TK, dtype=torch.int32, device=dev)
    if row_map is None:
        row_map = torch.empty(TK, dtype=torch.int32, device=dev)
    if tokens_per_expert is None:
        tokens_per_expert = torch.empty(num_experts, dtype=torch.int32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    ws = moe_permute_workspace_size(T, K, num_experts)
    if workspace is None:
        workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
    if active_mask is None:
        _call("moe_permute", _ptr(tokens), dt, _ptr(expert_ids), T, max(H, 1), K, num_experts,
              num_special, _ptr(permuted), _ptr(sorted_indices), _ptr(row_map),
              _ptr(tokens_per_expert), _ptr(expert_offsets), _ptr(workspace),
              workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream())
    else:
        _call("moe_permute_masked", _ptr(tokens), dt, _ptr(expert_ids), T, max(H, 1), K,
              num_experts, num_special, _ptr(_mask(active_mask, T, K)), active_mask.dim(),
              _ptr(permuted), _ptr(sorted_indices), _ptr(row_map), _ptr(tokens_per_expert),
              _ptr(expert_offsets), _ptr(workspace),
              workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream())
    return PermuteResult(permuted, sorted_indices, row_map, tokens_per_expert, expert_offsets)


MOE_PERMUTE_STATIC_SCRATCH_INTS = 65536


def moe_permute_static_scratch(tokens: Optional[torch.Tensor], expert_ids: torch.Tensor,
                               num_experts: int, num_special: int = 0, *, permuted=None,
                               sorted_indices=None, row_map=None, tokens_per_expert=None,
                               expert_offsets=None, dev_status=None) -> PermuteResult:
    """moe_permute for callers that cannot allocate device memory: the
    library keeps its routing workspace (per-block counts and flags) in its
    own fixed device array
    (MOE_PERMUTE_STATIC_SCRATCH_INTS int32), shared by every call, so calls
    must not overlap on the GPU.  Outputs the caller does not pass are
    allocated here by torch only for convenience of this binding."""
    _check(expert_ids, torch.int32, "expert_ids")
    T, K = expert_ids.shape
    dev = expert_ids.device
    H = tokens.shape[1] if tokens is not None else 0
    dt = _dtype(tokens) if tokens is not None else MOE_BF16
    TK = T * K
    if tokens is not None and permuted is None:
        permuted = torch.empty((TK, H), dtype=tokens.dtype, device=dev)
    if sorted_indices is None:
        sorted_indices = torch.empty(TK, dtype=torch.int32, device=dev)
    if row_map is None:
        row_map = torch.empty(TK, dtype=torch.int32, device=dev)
    if tokens_per_expert is None:
        tokens_per_expert = torch.empty(num_experts, dtype=torch.int32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    _call("moe_permute_static_scratch", _ptr(tokens), dt, _ptr(expert_ids), T, max(H, 1), K,
          num_experts, num_special, _ptr(permuted), _ptr(sorted_indices), _ptr(row_map),
          _ptr(tokens_per_expert), _ptr(expert_offsets), _ptr(dev_status), _stream())
    return PermuteResult(permuted, sorted_indices, row_map, tokens_per_expert, expert_offsets)


def moe_permute_rows(tokens, row_map, K: int, N: int, *, permuted=None):
    """permuted[row_map[t*K+k]] = tokens[t] for a routing the caller holds;
    slots whose row lies outside [0, N) are skipped."""
    _check(row_map, torch.int32, "row_map")
    T, H = tokens.shape
    if permuted is None:
        permuted = torch.empty((N, H), dtype=tokens.dtype, device=tokens.device)
    _call("moe_permute_rows", _ptr(tokens), _dtype(tokens), _ptr(row_map), T, H, K, N,
          _ptr(permuted), _stream())
    return permuted


def moe_invert_sorted_indices(sorted_indices: torch.Tensor, N: int, TK: int, *, row_map=None):
    if row_map is None:
        row_map = torch.empty(TK, dtype=torch.int32, device=sorted_indices.device)
    _call("moe_invert_sorted_indices", _ptr(sorted_indices), N, TK, _ptr(row_map), _stream())
    return row_map


# ---------------------------------------------------------------- expert MLP

def moe_gate_up_swiglu(permuted, expert_offsets, W_gate, W_up, *, act=None, gate_up_save=None,
                       save: bool = False, dev_status=None):
    N, H = permuted.shape
    E, I, _ = W_gate.shape
    if act is None:
        act = torch.empty((N, I), dtype=permuted.dtype, device=permuted.device)
    if save and gate_up_save is None:
        gate_up_save = torch.empty((N, 2 * I), dtype=permuted.dtype, device=permuted.device)
    _call("moe_gate_up_swiglu", _ptr(permuted), _dtype(permuted), _ptr(expert_offsets), N, H, I,
          E, _ptr(W_gate), _ptr(W_up), _ptr(act), _ptr(gate_up_save), _ptr(dev_status),
          _stream())
    return act, gate_up_save


def moe_down_proj(act, expert_offsets, W_down, *, expanded=None, dev_status=None):
    N, I = act.shape
    E, H, _ = W_down.shape
    if expanded is None:
        expanded = torch.empty((N, H), dtype=act.dtype, device=act.device)
    _call("moe_down_proj", _ptr(act), _dtype(act), _ptr(expert_offsets), N, H, I, E,
          _ptr(W_down), _ptr(expanded), _ptr(dev_status), _stream())
    return expanded


def moe_expert_mlp(permuted, expert_offsets, W_gate, W_up, W_down, *, act=None, expanded=None,
                   gate_up_save=None, save: bool = False, dev_status=None):
    N, H = permuted.shape
    E, I, _ = W_gate.shape
    if act is None:
        act = torch.empty((N, I), dtype=permuted.dtype, device=permuted.device)
    if expanded is None:
        expanded = torch.empty((N, H), dtype=permuted.dtype, device=permuted.device)
    if save and gate_up_save is None:
        gate_up_save = torch.empty((N, 2 * I), dtype=permuted.dtype, device=permuted.device)
    _call("moe_expert_mlp", _ptr(permuted), _dtype(permuted), _ptr(expert_offsets), N, H, I, E,
          _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(act), _ptr(expanded), _ptr(gate_up_save),
          _ptr(dev_status), _stream())
    return act, expanded, gate_up_save


def moe_expert_mlp_grad(grad_expanded, permuted, act, gate_up_save, expert_offsets, W_gate, W_up,
                        W_down, *, dgu=None, d_permuted=None, dW_gate=None, dW_up=None,
                        dW_down=None, dev_status=None):
    N, H = permuted.shape
    E, I, _ = W_gate.shape
    dev, dt = permuted.device, permuted.dtype
    if dgu is None:
        dgu = torch.empty((N, 2 * I), dtype=dt, device=dev)
    if d_permuted is None:
        d_permuted = torch.empty((N, H), dtype=dt, device=dev)
    if dW_gate is None:
        dW_gate = torch.empty_like(W_gate)
    if dW_up is None:
        dW_up = torch.empty_like(W_up)
    if dW_down is None:
        dW_down = torch.empty_like(W_down)
    _call("moe_expert_mlp_grad", _ptr(grad_expanded), _ptr(permuted), _ptr(act),
          _ptr(gate_up_save), _dtype(permuted), _ptr(expert_offsets), N, H, I, E, _ptr(W_gate),
          _ptr(W_up), _ptr(W_down), _ptr(dgu), _ptr(d_permuted), _ptr(dW_gate), _ptr(dW_up),
          _ptr(dW_down), _ptr(dev_status), _stream())
    return d_permuted, dW_gate, dW_up, dW_down


def moe_down_dgrad_swiglu(grad_expanded, gate_up_save, expert_offsets, W_down, *, dgu=None,
                          dev_status=None):
    N, H = grad_expanded.shape
    E, _, I = W_down.shape
    if dgu is None:
        dgu = torch.empty((N, 2 * I), dtype=grad_expanded.dtype, device=grad_expanded.device)
    _call("moe_down_dgrad_swiglu", _ptr(grad_expanded), _ptr(gate_up_save), _dtype(grad_expanded),
          _ptr(expert_offsets), N, H, I, E, _ptr(W_down), _ptr(dgu), _ptr(dev_status), _stream())
    return dgu


def moe_gate_up_dgrad(dgu, expert_offsets, W_gate, W_up, *, d_permuted=None, dev_status=None):
    N = dgu.shape[0]
    E, I, H = W_gate.shape
    if d_permuted is None:
        d_permuted = torch.empty((N, H), dtype=dgu.dtype, device=dgu.device)
    _call("moe_gate_up_dgrad", _ptr(dgu), _dtype(dgu), _ptr(expert_offsets), N, H, I, E,
          _ptr(W_gate), _ptr(W_up), _ptr(d_permuted), _ptr(dev_status), _stream())
    return d_permuted


def moe_down_wgrad(grad_expanded, act, expert_offsets, *, dW_down, dev_status=None):
    N, H = grad_expanded.shape
    E, _, I = dW_down.shape
    _call("moe_down_wgrad", _ptr(grad_expanded), _ptr(act), _dtype(grad_expanded),
          _ptr(expert_offsets), N, H, I, E, _ptr(dW_down), _ptr(dev_status), _stream())
    return dW_down


def moe_gate_up_wgrad(dgu, permuted, expert_offsets, *, dW_gate, dW_up, dev_status=None):
    N, H = permuted.shape
    E, I, _ = dW_gate.shape
    _call("moe_gate_up_wgrad", _ptr(dgu), _ptr(permuted), _dtype(permuted), _ptr(expert_offsets),
          N, H, I, E, _ptr(dW_gate), _ptr(dW_up), _ptr(dev_status), _stream())
    return dW_gate, dW_up


def moe_shared_expert_mlp(x, W_gate, W_up, W_down, *, act=None, out=None, dev_status=None):
    """Shared-expert MLP over all tokens (bf16): out = (silu(x Wg^T) * x Wu^T) Wd^T.
    Runs on the current stream; pass out as moe_combine's shared_x."""
    _check(x, torch.bfloat16, "x")
    T, H = x.shape
    I = W_gate.shape[0]
    if act is None:
        act = torch.empty((T, I), dtype=x.dtype, device=x.device)
    if out is None:
        out = torch.empty((T, H), dtype=x.dtype, device=x.device)
    _call("moe_shared_expert_mlp", _ptr(x), T, H, I, _ptr(W_gate), _ptr(W_up), _ptr(W_down),
          _ptr(act), _ptr(out), _ptr(dev_status), _stream())
    return out


def moe_gate_up_swiglu_gather(tokens, sorted_indices, K: int, expert_offsets, W_gate, W_up, *,
                              N: Optional[int] = None, act=None, gate_up_save=None,
                              save: bool = False, dev_status=None):
    """moe_gate_up_swiglu of tokens[sorted_indices[i] // K] without building
    that permuted copy: the GEMM gathers the token rows itself (bf16)."""
    _check(tokens, torch.bfloat16, "tokens")
    _check(sorted_indices, torch.int32, "sorted_indices")
    T, H = tokens.shape
    N = sorted_indices.shape[0] if N is None else N
    E, I, _ = W_gate.shape
    if act is None:
        act = torch.empty((N, I), dtype=tokens.dtype, device=tokens.device)
    if save and gate_up_save is None:
        gate_up_save = torch.empty((N, 2 * I), dtype=tokens.dtype, device=tokens.device)
    _call("moe_gate_up_swiglu_gather", _ptr(tokens), T, _ptr(sorted_indices), K,
          _ptr(expert_offsets), N, H, I, E, _ptr(W_gate), _ptr(W_up), _ptr(act),
          _ptr(gate_up_save), _ptr(dev_status), _stream())
    return act, gate_up_save


def moe_gate_up_wgrad_gather(dgu, tokens, sorted_indices, K: int, expert_offsets, *, dW_gate,
                             dW_up, dev_status=None):
    """moe_gate_up_wgrad with X = tokens[sorted_indices[i] // K], gathered in
    the GEMM (bf16)."""
    _check(tokens, torch.bfloat16, "tokens")
    _check(sorted_indices, torch.int32, "sorted_indices")
    T, H = tokens.shape
    N = dgu.shape[0]
    E, I, _ = dW_gate.shape
    _call("moe_gate_up_wgrad_gather", _ptr(dgu), _ptr(tokens), T, _ptr(sorted_indices), K,
          _ptr(expert_offsets), N, H, I, E, _ptr(dW_gate), _ptr(dW_up), _ptr(dev_status),
          _stream())
    return dW_gate, dW_up


# ---------------------------------------------------------------- unpermute / combine

def moe_unpermute(expanded, row_map, probs, T: int, K: int, *, out=None):
    N, H = expanded.shape
    if probs is not None:
        _check(probs, torch.float32, "probs")
    if out is None:
        out = torch.empty((T, H), dtype=expanded.dtype, device=expanded.device)
    _call("moe_unpermute", _ptr(expanded), _dtype(expanded), _ptr(row_map), _ptr(probs), T, H, K,
          N, _ptr(out), _stream())
    return out


def moe_unpermute_grad(grad_out, permuted_tokens, row_map, probs, K: int, *, grad_permuted=None,
                       grad_probs=None):
    T, H = grad_out.shape
    N = permuted_tokens.shape[0]
    if grad_permuted is None:
        grad_permuted = torch.empty_like(permuted_tokens)
    if grad_probs is None:
        grad_probs = torch.empty((T, K), dtype=torch.float32, device=grad_out.device)
    _call("moe_unpermute_grad", _ptr(grad_out), _ptr(permuted_tokens), _dtype(grad_out),
          _ptr(row_map), _ptr(probs), T, H, K, N, _ptr(grad_permuted), _ptr(grad_probs),
          _stream())
    return grad_permuted, grad_probs


def moe_permute_grad(grad_permuted, row_map, T: int, K: int, *, out=None):
    N, H = grad_permuted.shape
    if out is None:
        out = torch.empty((T, H), dtype=grad_permuted.dtype, device=grad_permuted.device)
    _call("moe_permute_grad", _ptr(grad_permuted), _dtype(grad_permuted), _ptr(row_map), T, H, K,
          N, _ptr(out), _stream())
    return out


def moe_combine(expanded, row_map, expert_ids, scales, num_experts: int, *, shared_x=None,
                ori_x=None, zero_num: int = 0, copy_num: int = 0, const_num: int = 0,
                alpha1=None, alpha2=None, const_v=None, out=None, dev_status=None,
                active_mask=None):
    T, K = expert_ids.shape
    N, H = expanded.shape
    if out is None:
        out = torch.empty((T, H), dtype=expanded.dtype, device=expanded.device)
    if active_mask is None:
        _call("moe_combine", _ptr(expanded), _dtype(expanded), _ptr(row_map), _ptr(expert_ids),
              _ptr(scales), _ptr(shared_x), _ptr(ori_x), T, H, K, N, num_experts, zero_num,
              copy_num, const_num, _ptr(alpha1), _ptr(alpha2), _ptr(const_v), _ptr(out),
              _ptr(dev_status), _stream())
    else:
        _call("moe_combine_masked", _ptr(expanded), _dtype(expanded), _ptr(row_map),
              _ptr(expert_ids), _ptr(scales), _ptr(shared_x), _ptr(ori_x),
              _ptr(_mask(active_mask, T, K)), active_mask.dim(), T, H, K, N, num_experts,
              zero_num, copy_num, const_num, _ptr(alpha1), _ptr(alpha2), _ptr(const_v), _ptr(out),
              _ptr(dev_status), _stream())
    return out


# ---------------------------------------------------------------- permute indices

def moe_permute_indices(counts, R: int, E: int, capacity: int, *, indices=None,
                        tokens_per_expert=None, total=None, dev_status=None):
    dev = counts.device
    if indices is None:
        indices = torch.empty(max(capacity, 1), dtype=torch.int32, device=dev)
    if tokens_per_expert is None:
        tokens_per_expert = torch.empty(E, dtype=torch.int32, device=dev)
    if total is None:
        total = torch.empty(1, dtype=torch.int32, device=dev)
    _call("moe_permute_indices", _ptr(counts), R, E, _ptr(indices), capacity,
          _ptr(tokens_per_expert), _ptr(total), _ptr(dev_status), _stream())
    return indices, tokens_per_expert, total


def moe_permute_indices_window(counts, R: int, E_all: int, col_start: int, col_count: int,
                               capacity: int, *, indices=None, tokens_per_column=None, total=None,
                               dev_status=None):
    """Deredundancy dispatch indices: blocks of the expert window
    [col_start, col_start + col_count) ordered (expert, source)."""
    dev = counts.device
    if indices is None:
        indices = torch.empty(max(capacity, 1), dtype=torch.int32, device=dev)
    if tokens_per_column is None:
        tokens_per_column = torch.empty(max(col_count, 1), dtype=torch.int32, device=dev)
    if total is None:
        total = torch.empty(1, dtype=torch.int32, device=dev)
    _call("moe_permute_indices_window", _ptr(counts), R, E_all, col_start, col_count,
          _ptr(indices), capacity, _ptr(tokens_per_column), _ptr(total), _ptr(dev_status),
          _stream())
    return indices, tokens_per_column, total
