"""GPU parity of the expert MLP and of the whole layer against the oracle."""

import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from gpu_util import BF16_TOL, F32_TOL, assert_normwise, np64, tol_for

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _layer_forward_gpu(lib, d, save=True):
    E, K, T = d["E"], d["K"], d["T"]
    r = lib.moe_permute(d["tokens"].to(DEV), d["expert_ids"].to(DEV), E, 0)
    act, expanded, gu = lib.moe_expert_mlp(r.permuted, r.expert_offsets, d["W_gate"].to(DEV),
                                           d["W_up"].to(DEV), d["W_down"].to(DEV), save=save)
    out = lib.moe_unpermute(expanded, r.row_map, d["probs"].to(DEV), T, K)
    return r, act, expanded, gu, out


def _layer_forward_oracle(d):
    E, K, T, dt = d["E"], d["K"], d["T"], d["dtype"]
    si, rm, tpe, off = O.permute_routing(d["expert_ids"].numpy(), E)
    perm = O.permute_rows(np64(d["tokens"]), si, K)
    act, expd, g, u = O.expert_mlp(perm, off, np64(d["W_gate"]), np64(d["W_up"]),
                                   np64(d["W_down"]), dt)
    out = O.unpermute(expd, rm, d["probs"].numpy(), T, K, dt)
    return (si, rm, tpe, off), perm, act, expd, g, u, out


@pytest.mark.parametrize("kw", [
    dict(),                                            # T=64 H=128 E=8 K=2 I=256
    dict(T=300, H=96, E=5, K=2, I=80),                 # ragged 64-row tiles, N and I tails
    dict(T=5, H=64, E=16, K=2, I=64),                  # most experts without rows
])
def test_fp32_layer_forward(lib, kw):
    d = moe_inputs.tiny_fp32_layer(0, **kw)
    r, act, expanded, gu, out = _layer_forward_gpu(lib, d)
    (si, rm, tpe, off), perm, w_act, w_exp, g, u, w_out = _layer_forward_oracle(d)
    N = len(si)
    I = d["I"]
    assert np.array_equal(np64(r.row_map), rm)
    assert_normwise(np64(act)[:N], w_act, F32_TOL, "act")
    assert_normwise(np64(gu)[:N, :I], g, F32_TOL, "gate pre-activation")
    assert_normwise(np64(gu)[:N, I:], u, F32_TOL, "up pre-activation")
    assert_normwise(np64(expanded)[:N], w_exp, F32_TOL, "expanded")
    assert_normwise(np64(out), w_out, F32_TOL, "layer output")
