"""GPU parity of the gate/up GEMMs that gather their token rows themselves
(the permute's row copy fused into the GEMM loads).

Each gathering call is checked two ways: against the float64 oracle (the
permute's gather followed by the plain GEMM definition), within the bf16
tolerance of the other GEMM tests; and bit for bit against the same GEMM run
on the permuted buffer, since the gathered tiles land in shared memory
exactly as the plain box loads put them.
"""

import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from gpu_util import BF16_TOL, assert_normwise, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = [
    dict(T=200, H=256, E=8, K=4, I=192),     # partial 128-column gate/up tile
    dict(T=700, H=320, E=16, K=8, I=128),    # 3 m-tiles per expert, ragged tails
    dict(T=333, H=128, E=8, K=3, I=64),      # K not a power of two
    dict(T=64, H=128, E=64, K=2, I=64),      # many experts without rows
    dict(T=1, H=64, E=4, K=1, I=64),         # a single row
]


def _weights(d):
    return d["W_gate"].to(DEV), d["W_up"].to(DEV), d["W_down"].to(DEV)


def _oracle_forward(d):
    si, rm, tpe, off = O.permute_routing(d["expert_ids"].numpy(), d["E"])
    perm = O.permute_rows(np64(d["tokens"]), si, d["K"])
    act, expd, g, u = O.expert_mlp(perm, off, np64(d["W_gate"]), np64(d["W_up"]),
                                   np64(d["W_down"]), "bf16")
    return (si, rm, tpe, off), perm, act, expd, g, u


@pytest.mark.parametrize("kw", CASES)
def test_gate_up_gather_forward(lib, kw):
    d = moe_inputs.layer_fwd_bwd(4, **kw)
    K, E, I = d["K"], d["E"], d["I"]
    tok = d["tokens"].to(DEV)
    r = lib.moe_permute(tok, d["expert_ids"].to(DEV), E, 0)
    Wg, Wu, _ = _weights(d)
    st = lib.new_status()
    act_g, gu_g = lib.moe_gate_up_swiglu_gather(tok, r.sorted_indices, K, r.expert_offsets, Wg,
                                                Wu, save=True, dev_status=st)
    act_p, gu_p = lib.moe_gate_up_swiglu(r.permuted, r.expert_offsets, Wg, Wu, save=True)
    assert lib.moe_check_status(st) == lib.MOE_OK
    (si, rm, tpe, off), perm, w_act, w_exp, g, u = _oracle_forward(d)
    N = len(si)
    assert torch.equal(act_g[:N], act_p[:N]) and torch.equal(gu_g[:N], gu_p[:N])
    assert_normwise(np64(gu_g)[:N, :I], O.round_to_bf16(g), BF16_TOL, "gate")
    assert_normwise(np64(gu_g)[:N, I:], O.round_to_bf16(u), BF16_TOL, "up")
    assert_normwise(np64(act_g)[:N], w_act, BF16_TOL, "act")


def test_gate_up_gather_forward_zipf_skew(lib):
    """Skewed routing: empty experts and experts spanning many tiles."""
    d = moe_inputs.layer_forward_zipf(5, T=1024, H=512, E=64, K=8, I=256, num_empty=8)
    K, E = d["K"], d["E"]
    tok = d["tokens"].to(DEV)
    r = lib.moe_permute(None, d["expert_ids"].to(DEV), E, 0)     # routing only: no permuted copy
    Wg, Wu, Wd = _weights(d)
    act, _ = lib.moe_gate_up_swiglu_gather(tok, r.sorted_indices, K, r.expert_offsets, Wg, Wu)
    expanded = lib.moe_down_proj(act, r.expert_offsets, Wd)
    (si, rm, tpe, off), perm, w_act, w_exp, g, u = _oracle_forward(d)
    N = len(si)
    assert (tpe == 0).sum() >= 8 and tpe.max() > 512
    assert_normwise(np64(act)[:N], w_act, BF16_TOL, "act")
    assert_normwise(np64(expanded)[:N], w_exp, BF16_TOL, "expanded")


@pytest.mark.parametrize("kw", CASES + [dict(T=300, H=192, E=6, K=3, I=320)])
def test_gate_up_wgrad_gather(lib, kw):
    d = moe_inputs.layer_fwd_bwd(6, **kw)
    T, K, E = d["T"], d["K"], d["E"]
    tok = d["tokens"].to(DEV)
    r = lib.moe_permute(tok, d["expert_ids"].to(DEV), E, 0)
    Wg, Wu, Wd = _weights(d)
    act, expanded, gu = lib.moe_expert_mlp(r.permuted, r.expert_offsets, Wg, Wu, Wd, save=True)
    probs = d["probs"].to(DEV)
    gexp, _ = lib.moe_unpermute_grad(d["grad_out"].to(DEV), expanded, r.row_map, probs, K)
    dgu = lib.moe_down_dgrad_swiglu(gexp, gu, r.expert_offsets, Wd)
    st = lib.new_status()
    dWg_g, dWu_g = lib.moe_gate_up_wgrad_gather(dgu, tok, r.sorted_indices, K, r.expert_offsets,
                                                dW_gate=torch.empty_like(Wg),
                                                dW_up=torch.empty_like(Wu), dev_status=st)
    dWg_p, dWu_p = lib.moe_gate_up_wgrad(dgu, r.permuted, r.expert_offsets,
                                         dW_gate=torch.empty_like(Wg), dW_up=torch.empty_like(Wu))
    assert lib.moe_check_status(st) == lib.MOE_OK
    assert torch.equal(dWg_g, dWg_p) and torch.equal(dWu_g, dWu_p)
    (si, rm, tpe, off), perm, w_act, w_exp, g, u = _oracle_forward(d)
    w_gexp, _ = O.unpermute_grad(np64(d["grad_out"]), w_exp, rm, d["probs"].numpy(), T, K, "bf16")
    _, dWg, dWu, _ = O.expert_mlp_grad(w_gexp, perm, w_act, off, np64(d["W_gate"]),
                                       np64(d["W_up"]), np64(d["W_down"]), "bf16")
    assert_normwise(np64(dWg_g), dWg, BF16_TOL, "dW_gate")
    assert_normwise(np64(dWu_g), dWu, BF16_TOL, "dW_up")
    for e in np.nonzero(tpe == 0)[0]:                    # experts without rows: zero grads
        assert not np64(dWg_g[int(e)]).any() and not np64(dWu_g[int(e)]).any()


def test_gather_full_size_matches_permuted(lib):
    """T=4096 H=2048 E=128 K=8 I=768 (the layer benchmark): the gathering
    forward and wgrad equal the permuted-buffer GEMMs bit for bit."""
    d = moe_inputs.layer_fwd_bwd(0)
    K, E = d["K"], d["E"]
    tok = d["tokens"].to(DEV)
    r = lib.moe_permute(tok, d["expert_ids"].to(DEV), E, 0)
    Wg, Wu, Wd = _weights(d)
    act_p, gu_p = lib.moe_gate_up_swiglu(r.permuted, r.expert_offsets, Wg, Wu, save=True)
    act_g, gu_g = lib.moe_gate_up_swiglu_gather(tok, r.sorted_indices, K, r.expert_offsets, Wg,
                                                Wu, save=True)
    assert torch.equal(act_g, act_p) and torch.equal(gu_g, gu_p)
    dgu = (torch.randn(gu_p.shape, device=DEV, generator=torch.Generator(DEV).manual_seed(1))
           * 0.01).to(torch.bfloat16)
    dWg_p, dWu_p = lib.moe_gate_up_wgrad(dgu, r.permuted, r.expert_offsets,
                                         dW_gate=torch.empty_like(Wg), dW_up=torch.empty_like(Wu))
    dWg_g, dWu_g = lib.moe_gate_up_wgrad_gather(dgu, tok, r.sorted_indices, K, r.expert_offsets,
                                                dW_gate=torch.empty_like(Wg),
                                                dW_up=torch.empty_like(Wu))
    assert torch.equal(dWg_g, dWg_p) and torch.equal(dWu_g, dWu_p)


def test_gather_rejects_bad_arguments(lib):
    d = moe_inputs.layer_fwd_bwd(7, T=16, H=64, E=4, K=2, I=64)
    tok = d["tokens"].to(DEV)
    r = lib.moe_permute(tok, d["expert_ids"].to(DEV), 4, 0)
    Wg, Wu, _ = _weights(d)
    with pytest.raises(lib.MoeError) as e:
        lib.moe_gate_up_swiglu_gather(tok, r.sorted_indices, 0, r.expert_offsets, Wg, Wu)   # K = 0
    assert e.value.status == lib.MOE_ERR_INVALID_ARG
    with pytest.raises(lib.MoeError) as e:
        lib.moe_gate_up_swiglu_gather(tok, r.sorted_indices, 17, r.expert_offsets, Wg, Wu)  # K > 16
    assert e.value.status == lib.MOE_ERR_INVALID_ARG
    with pytest.raises(ValueError):                      # the gathering GEMMs are bf16 only
        lib.moe_gate_up_swiglu_gather(tok.float(), r.sorted_indices, 2, r.expert_offsets, Wg, Wu)
