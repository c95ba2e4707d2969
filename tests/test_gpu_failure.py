"""Failure handling on the GPU, exercised without faulting or hanging it.

- The bounded waits the tensor-core kernels rely on give up after their limit
  with MOE_ERR_TIMEOUT in the caller's status word, and the context stays
  usable (a library self-test waits on a barrier that nothing arrives on).
- Corrupt expert offsets made on the host are sanitised: clamped to the
  buffer, then made non-decreasing (each offset raised to the largest one
  before it), so expert ranges never overlap; the grouped GEMMs touch only
  rows inside those ranges, and their results there are those of the oracle
  on the same ranges.
"""

import time

import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from gpu_util import BF16_TOL, assert_normwise, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_bounded_wait_times_out_and_context_survives(lib):
    st = lib.new_status()
    t0 = time.perf_counter()
    lib.moe_selftest_bounded_wait(st)
    assert lib.moe_check_status(st) == lib.MOE_ERR_TIMEOUT
    assert 1.0 < time.perf_counter() - t0 < 30.0        # the 2 s limit, not a hang
    # the context still works: a routing call afterwards is exact
    rng = np.random.Generator(np.random.PCG64(9))
    ids = moe_inputs.uniform_distinct_ids(rng, 300, 4, 16)
    ok = lib.new_status()
    r = lib.moe_permute(None, ids.to(DEV), 16, 0, dev_status=ok)
    assert lib.moe_check_status(ok) == lib.MOE_OK
    si, rm, tpe, off = O.permute_routing(ids.numpy(), 16)
    assert np.array_equal(np64(r.row_map), rm)
    assert np.array_equal(np64(r.expert_offsets), off)


# (offsets as given, the sanitised offsets, first row no range covers)
CORRUPT = [
    ([-5, 40, 30, 30, 25], [0, 40, 40, 40, 40], 40),               # negative, decreasing
    ([-5, 40, 10 ** 9, 10 ** 9, -7], [0, 40, 300, 300, 300], 300),  # past the buffer, negative last
    ([0, 100, 50, 150, 200], [0, 100, 100, 150, 200], 200),         # would overlap expert 0
]


@pytest.mark.parametrize("given,clamped,untouched", CORRUPT)
def test_gemms_clamp_corrupt_offsets(lib, given, clamped, untouched):
    """Over a 300-row buffer, offset i becomes max(clamp(off[j], 0, N), j <= i)
    and expert e takes rows [off[e], off[e+1]): the ranges never overlap, so
    no two tiles write one row and the results are the oracle's on the
    sanitised offsets."""
    d = moe_inputs.layer_fwd_bwd(8, T=300, H=128, E=4, K=1, I=64)
    N, H, I = 300, 128, 64
    X = d["tokens"].to(DEV)                               # used as the expert-major rows
    Wg, Wu, Wd = d["W_gate"].to(DEV), d["W_up"].to(DEV), d["W_down"].to(DEV)
    off = torch.tensor(given, dtype=torch.int32, device=DEV)
    sentinel = 7.0
    act = torch.full((N, I), sentinel, dtype=torch.bfloat16, device=DEV)
    gu = torch.full((N, 2 * I), sentinel, dtype=torch.bfloat16, device=DEV)
    out = torch.full((N, H), sentinel, dtype=torch.bfloat16, device=DEV)
    st = lib.new_status()
    lib.moe_gate_up_swiglu(X, off, Wg, Wu, act=act, gate_up_save=gu, dev_status=st)
    lib.moe_down_proj(act, off, Wd, expanded=out, dev_status=st)
    dY = d["grad_out"].to(DEV)                             # [300, H] as the expert-major grads
    dWd = torch.full_like(Wd, sentinel)
    lib.moe_down_wgrad(dY, act, off, dW_down=dWd, dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_OK
    # rows outside every clamped range are untouched
    assert torch.all(act[untouched:] == sentinel) and torch.all(gu[untouched:] == sentinel)
    assert torch.all(out[untouched:] == sentinel)
    c = np.array(clamped)
    n = untouched
    w_act, w_exp, g, u = O.expert_mlp(np64(X)[:n], c, np64(d["W_gate"]), np64(d["W_up"]),
                                      np64(d["W_down"]), "bf16")
    assert_normwise(np64(act)[:n], w_act, BF16_TOL, "act")
    assert_normwise(np64(out)[:n], w_exp, BF16_TOL, "expanded")
    # weight gradient from the same clamped ranges (fed the kernel's own act)
    _, _, _, w_dWd = O.expert_mlp_grad(np64(dY)[:n], np64(X)[:n], np64(act)[:n], c,
                                       np64(d["W_gate"]), np64(d["W_up"]), np64(d["W_down"]),
                                       "bf16")
    assert_normwise(np64(dWd), w_dWd, BF16_TOL, "dW_down")
    for e in range(4):
        if c[e + 1] == c[e]:                               # empty experts: zero gradients
            assert not np64(dWd[e]).any()
