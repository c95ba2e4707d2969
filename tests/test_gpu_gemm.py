"""GPU parity of the bf16 tcgen05 grouped GEMMs (forward and backward) and of
the whole bf16 layer against the float64 oracle.

Small cases span several 128-row tiles per expert, ragged row tails, partial
output-column tiles, experts without rows and Zipf-skewed routing; the
full-size workloads are checked on sampled rows and sampled experts.
"""

import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from gpu_util import BF16_TOL, assert_normwise, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _weights(d):
    return d["W_gate"].to(DEV), d["W_up"].to(DEV), d["W_down"].to(DEV)


def _oracle_forward(d):
    E, K = d["E"], d["K"]
    si, rm, tpe, off = O.permute_routing(d["expert_ids"].numpy(), E)
    perm = O.permute_rows(np64(d["tokens"]), si, K)
    act, expd, g, u = O.expert_mlp(perm, off, np64(d["W_gate"]), np64(d["W_up"]),
                                   np64(d["W_down"]), "bf16")
    return (si, rm, tpe, off), perm, act, expd, g, u


SMALL = [
    dict(T=200, H=256, E=8, K=4, I=192),      # partial 128-column gate/up tile
    dict(T=700, H=320, E=16, K=8, I=128),     # 3 m-tiles per expert, partial 256-column down tile
    dict(T=64, H=128, E=64, K=2, I=64),       # many experts without rows
    dict(T=1, H=64, E=4, K=1, I=64),          # a single row
    # about 1950 rows per expert: gate/up runs as CTA pairs (odd and even
    # per-expert tile counts), down single
    dict(T=2600, H=256, E=4, K=3, I=192),
    # about 2250 rows per expert: both forward GEMMs run as CTA pairs,
    # partial 256-column down tile
    dict(T=4500, H=320, E=4, K=2, I=128),
]


@pytest.mark.parametrize("kw", SMALL)
def test_bf16_expert_mlp_forward(lib, kw):
    d = moe_inputs.layer_fwd_bwd(1, **kw)
    r = lib.moe_permute(d["tokens"].to(DEV), d["expert_ids"].to(DEV), d["E"], 0)
    Wg, Wu, Wd = _weights(d)
    st = lib.new_status()
    act, expanded, gu = lib.moe_expert_mlp(r.permuted, r.expert_offsets, Wg, Wu, Wd, save=True,
                                           dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_OK
    (si, rm, tpe, off), perm, w_act, w_exp, g, u = _oracle_forward(d)
    N, I = len(si), d["I"]
    assert_normwise(np64(gu)[:N, :I], O.round_to_bf16(g), BF16_TOL, "gate")
    assert_normwise(np64(gu)[:N, I:], O.round_to_bf16(u), BF16_TOL, "up")
    assert_normwise(np64(act)[:N], w_act, BF16_TOL, "act")
    assert_normwise(np64(expanded)[:N], w_exp, BF16_TOL, "expanded")


def test_bf16_expert_mlp_zipf_skew(lib):
    d = moe_inputs.layer_forward_zipf(0, T=1024, H=512, E=64, K=8, I=256, num_empty=8)
    r = lib.moe_permute(d["tokens"].to(DEV), d["expert_ids"].to(DEV), d["E"], 0)
    Wg, Wu, Wd = _weights(d)
    act, expanded, _ = lib.moe_expert_mlp(r.permuted, r.expert_offsets, Wg, Wu, Wd)
    (si, rm, tpe, off), perm, w_act, w_exp, g, u = _oracle_forward(d)
    N = len(si)
    assert (tpe == 0).sum() >= 8 and tpe.max() > 512      # skewed: empty and multi-tile experts
    assert_normwise(np64(act)[:N], w_act, BF16_TOL, "act")
    assert_normwise(np64(expanded)[:N], w_exp, BF16_TOL, "expanded")


def test_bf16_expert_mlp_paired_with_tiny_and_empty_experts(lib):
    """About 2048 rows per expert on average, so both forward GEMMs run as
    CTA pairs, but one expert has 5 rows (a single 128-row tile: the peer
    CTA's rows are all past the expert's end) and one has none."""
    d = moe_inputs.layer_fwd_bwd(3, T=8192, H=256, E=8, K=2, I=128)
    rng = np.random.Generator(np.random.PCG64(3))
    ids = moe_inputs.uniform_distinct_ids(rng, 8192, 2, 6)      # experts 0..5 only
    ids[:5, 1] = 7                                                # expert 7: 5 rows, expert 6: none
    d["expert_ids"] = ids
    r = lib.moe_permute(d["tokens"].to(DEV), ids.to(DEV), d["E"], 0)
    Wg, Wu, Wd = _weights(d)
    act, expanded, gu = lib.moe_expert_mlp(r.permuted, r.expert_offsets, Wg, Wu, Wd, save=True)
    (si, rm, tpe, off), perm, w_act, w_exp, g, u = _oracle_forward(d)
    N, I = len(si), d["I"]
    assert tpe[6] == 0 and tpe[7] == 5 and N == 8192 * 2
    assert_normwise(np64(gu)[:N, :I], O.round_to_bf16(g), BF16_TOL, "gate")
    assert_normwise(np64(gu)[:N, I:], O.round_to_bf16(u), BF16_TOL, "up")
    assert_normwise(np64(act)[:N], w_act, BF16_TOL, "act")
    assert_normwise(np64(expanded)[:N], w_exp, BF16_TOL, "expanded")
    # the tiny expert's rows on their own
    lo = int(off[7])
    assert_normwise(np64(expanded)[lo:lo + 5], w_exp[lo:lo + 5], BF16_TOL, "tiny expert")


def _sub_forward(perm_rows, experts, d):
    """Oracle forward of selected permuted rows (rows are independent given
    their expert): a sub-problem whose offsets group the rows by expert."""
    E = d["E"]
    counts = np.bincount(experts, minlength=E)
    off = np.concatenate([[0], np.cumsum(counts)])
    return O.expert_mlp(perm_rows, off, np64(d["W_gate"]), np64(d["W_up"]), np64(d["W_down"]), "bf16")


def _token_outputs(d, rm, ts):
    """Oracle layer output of tokens ts: their K slots' rows through the
    expert MLP (as a sub-problem grouped by expert) and the unpermute."""
    K = d["K"]
    flat = d["expert_ids"].numpy().reshape(-1)
    slots = (ts[:, None] * K + np.arange(K)).reshape(-1)
    order = np.argsort(rm[slots], kind="stable")
    perm_rows = O.permute_rows(np64(d["tokens"]), slots[order], K)
    _, y, _, _ = _sub_forward(perm_rows, flat[slots[order]], d)
    sub_rm = np.empty(len(slots), dtype=np.int64)
    sub_rm[order] = np.arange(len(slots))
    return O.unpermute(y, sub_rm, d["probs"].numpy()[ts], len(ts), K, "bf16")


def _check_sampled_forward(d, si, rm, act, expanded, out, seed, n_rows=600, n_tokens=64):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(len(si), n_rows, replace=False))
    flat = d["expert_ids"].numpy().reshape(-1)
    perm_rows = O.permute_rows(np64(d["tokens"]), si[rows], d["K"])
    w_act, w_exp, _, _ = _sub_forward(perm_rows, flat[si[rows]], d)
    sel = torch.from_numpy(rows).to(DEV)
    assert_normwise(np64(act[sel]), w_act, BF16_TOL, "act rows")
    assert_normwise(np64(expanded[sel]), w_exp, BF16_TOL, "expanded rows")
    ts = np.sort(rng.choice(d["T"], n_tokens, replace=False))
    w_out = _token_outputs(d, rm, ts)
    assert_normwise(np64(out[torch.from_numpy(ts).to(DEV)]), w_out, BF16_TOL, "layer output rows")


def test_bf16_layer_forward_full_size_zipf(lib):
    """T=8192 H=2048 E=256 K=8 I=512, Zipf(1.2) routing with 8 empty experts:
    routing bit-exact, sampled rows of act / expanded / output."""
    d = moe_inputs.layer_forward_zipf(0)
    T, K, E = d["T"], d["K"], d["E"]
    r = lib.moe_permute(d["tokens"].to(DEV), d["expert_ids"].to(DEV), E, 0)
    Wg, Wu, Wd = _weights(d)
    act, expanded, _ = lib.moe_expert_mlp(r.permuted, r.expert_offsets, Wg, Wu, Wd)
    out = lib.moe_unpermute(expanded, r.row_map, d["probs"].to(DEV), T, K)
    si, rm, tpe, off = O.permute_routing(d["expert_ids"].numpy(), E)
    assert np.array_equal(np64(r.row_map), rm)
    assert (tpe == 0).sum() == 8
    _check_sampled_forward(d, si, rm, act, expanded, out, seed=0)


# ---------------------------------------------------------------- backward

def _gpu_layer_fwd_bwd(lib, d):
    T, K, E = d["T"], d["K"], d["E"]
    Wg, Wu, Wd = _weights(d)
    st = lib.new_status()
    r = lib.moe_permute(d["tokens"].to(DEV), d["expert_ids"].to(DEV), E, 0, dev_status=st)
    act, expanded, gu = lib.moe_expert_mlp(r.permuted, r.expert_offsets, Wg, Wu, Wd, save=True,
                                           dev_status=st)
    probs = d["probs"].to(DEV)
    out = lib.moe_unpermute(expanded, r.row_map, probs, T, K)
    gexp, gprobs = lib.moe_unpermute_grad(d["grad_out"].to(DEV), expanded, r.row_map, probs, K)
    dperm, dWg, dWu, dWd = lib.moe_expert_mlp_grad(gexp, r.permuted, act, gu, r.expert_offsets,
                                                   Wg, Wu, Wd, dev_status=st)
    gtok = lib.moe_permute_grad(dperm, r.row_map, T, K)
    assert lib.moe_check_status(st) == lib.MOE_OK
    return dict(r=r, act=act, expanded=expanded, out=out, gexp=gexp, gprobs=gprobs, dperm=dperm,
                dWg=dWg, dWu=dWu, dWd=dWd, gtok=gtok)


@pytest.mark.parametrize("kw", SMALL + [dict(T=300, H=192, E=6, K=3, I=320),
                                  dict(T=200, H=128, E=256, K=4, I=128),  # many small experts
                                  # the down dgrad's four-stage variant (control
                                  # block for at most 192 experts) and the
                                  # three-stage one on either side of that bound
                                  dict(T=500, H=128, E=192, K=6, I=256),
                                  dict(T=500, H=128, E=193, K=6, I=256)])
def test_bf16_layer_backward(lib, kw):
    d = moe_inputs.layer_fwd_bwd(2, **kw)
    T, K, E = d["T"], d["K"], d["E"]
    g = _gpu_layer_fwd_bwd(lib, d)
    (si, rm, tpe, off), perm, act, expd, _, _ = _oracle_forward(d)
    out = O.unpermute(expd, rm, d["probs"].numpy(), T, K, "bf16")
    gexp, gprobs = O.unpermute_grad(np64(d["grad_out"]), expd, rm, d["probs"].numpy(), T, K, "bf16")
    dperm, dWg, dWu, dWd = O.expert_mlp_grad(gexp, perm, act, off, np64(d["W_gate"]),
                                             np64(d["W_up"]), np64(d["W_down"]), "bf16")
    gtok = O.permute_grad(dperm, rm, T, K, "bf16")
    N = len(si)
    assert_normwise(np64(g["out"]), out, BF16_TOL, "out")
    assert_normwise(np64(g["gprobs"]), gprobs, BF16_TOL, "grad probs")
    assert_normwise(np64(g["dperm"])[:N], dperm, BF16_TOL, "d_permuted")
    assert_normwise(np64(g["dWd"]), dWd, BF16_TOL, "dW_down")
    assert_normwise(np64(g["dWg"]), dWg, BF16_TOL, "dW_gate")
    assert_normwise(np64(g["dWu"]), dWu, BF16_TOL, "dW_up")
    assert_normwise(np64(g["gtok"]), gtok, BF16_TOL, "grad tokens")
    for e in np.nonzero(tpe == 0)[0]:                    # experts without rows: zero grads
        assert not np64(g["dWd"][int(e)]).any() and not np64(g["dWg"][int(e)]).any()


def test_bf16_layer_backward_zipf_skew(lib):
    """Zipf(1.2) routing with 8 experts without rows and the largest expert
    at several hundred rows: the weight-gradient GEMMs' long k loops, their
    expert tails (partial last k blocks zero-filled by the TMA unit) and
    the dgrads' skewed tiles, on every row and every expert's weight grads."""
    d = moe_inputs.layer_forward_zipf(0, T=1024, H=256, E=64, K=8, I=256, num_empty=8)
    rng = np.random.default_rng(7)
    d["grad_out"] = torch.from_numpy(rng.standard_normal((d["T"], d["H"])).astype(np.float32)).bfloat16()
    T, K, E = d["T"], d["K"], d["E"]
    g = _gpu_layer_fwd_bwd(lib, d)
    (si, rm, tpe, off), perm, act, expd, _, _ = _oracle_forward(d)
    assert (tpe == 0).sum() == 8 and tpe.max() > 300 and (tpe % 16 != 0).any()
    gexp, gprobs = O.unpermute_grad(np64(d["grad_out"]), expd, rm, d["probs"].numpy(), T, K, "bf16")
    dperm, dWg, dWu, dWd = O.expert_mlp_grad(gexp, perm, act, off, np64(d["W_gate"]),
                                             np64(d["W_up"]), np64(d["W_down"]), "bf16")
    N = len(si)
    assert_normwise(np64(g["dperm"])[:N], dperm, BF16_TOL, "d_permuted")
    for e in range(E):
        assert_normwise(np64(g["dWg"][e]), dWg[e], BF16_TOL, f"dW_gate[{e}]")
        assert_normwise(np64(g["dWu"][e]), dWu[e], BF16_TOL, f"dW_up[{e}]")
        assert_normwise(np64(g["dWd"][e]), dWd[e], BF16_TOL, f"dW_down[{e}]")


def _down_dgrad_last_wave_split(tiles: int, grid: int) -> int:
    """How the single-CTA down projection and dgrads split their last wave
    along N: when the tiles leave a last wave that fills at most half of the
    persistent grid (one CTA per SM), each of its tiles becomes 4 (at most a
    quarter full) or 2 narrower tiles; 1 = no split."""
    left = tiles % grid
    if left == 0 or 2 * left > grid:
        return 1
    return 4 if 4 * left <= grid else 2


@pytest.mark.parametrize("T,split", [(850, 4), (1000, 2), (1200, 1)])
def test_bf16_layer_backward_down_dgrad_last_wave(lib, T, split):
    """K = E = 8 gives every expert exactly T rows, so the down dgrad has
    8 * ceil(T/128) * 3 tiles (I = 768): with 152 SMs, 168 tiles (a last wave
    of 16, split 4 ways), 192 (40, split 2 ways) and 240 (88, not split).  The
    backward is checked on every row of d_permuted and every expert's weight
    grads, which all depend on the down dgrad's output."""
    E, K, I, H = 8, 8, 768, 256
    tiles = E * -(-T // 128) * (I // 256)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if _down_dgrad_last_wave_split(tiles, sms) != split:
        pytest.skip(f"{sms} SMs: this shape does not give the intended last wave")
    d = moe_inputs.layer_fwd_bwd(3, T=T, H=H, E=E, K=K, I=I)
    g = _gpu_layer_fwd_bwd(lib, d)
    (si, rm, tpe, off), perm, act, expd, _, _ = _oracle_forward(d)
    assert (tpe == T).all()
    gexp, _ = O.unpermute_grad(np64(d["grad_out"]), expd, rm, d["probs"].numpy(), T, K, "bf16")
    dperm, dWg, dWu, dWd = O.expert_mlp_grad(gexp, perm, act, off, np64(d["W_gate"]),
                                             np64(d["W_up"]), np64(d["W_down"]), "bf16")
    assert_normwise(np64(g["dperm"]), dperm, BF16_TOL, "d_permuted")
    for e in range(E):
        assert_normwise(np64(g["dWg"][e]), dWg[e], BF16_TOL, f"dW_gate[{e}]")
        assert_normwise(np64(g["dWu"][e]), dWu[e], BF16_TOL, f"dW_up[{e}]")
        assert_normwise(np64(g["dWd"][e]), dWd[e], BF16_TOL, f"dW_down[{e}]")


def test_bf16_layer_split_last_waves_with_full_waves(lib):
    """T=800 H=2048 E=32 K=8 I=256: fewer than 256 rows per expert, so the
    down projection and the gate/up dgrad run single-CTA, each with 512
    tiles (64 m-tiles x 8 n-tiles): with 152 SMs, three full waves and a last
    wave of 56 tiles split 2 ways.  Forward and backward on every row and
    every expert against the oracle."""
    d = moe_inputs.layer_fwd_bwd(5, T=800, H=2048, E=32, K=8, I=256)
    T, K, E = d["T"], d["K"], d["E"]
    (si, rm, tpe, off), perm, act, expd, _, _ = _oracle_forward(d)
    tiles = int(np.sum(-(-tpe // 128))) * (2048 // 256)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if tiles < sms or _down_dgrad_last_wave_split(tiles, sms) == 1:
        pytest.skip(f"{sms} SMs: this shape does not give a split last wave after full waves")
    assert tpe.max() < 256                               # single-CTA gate/up dgrad
    g = _gpu_layer_fwd_bwd(lib, d)
    N = len(si)
    assert_normwise(np64(g["expanded"])[:N], O.round_to_bf16(expd), BF16_TOL, "expanded")
    gexp, _ = O.unpermute_grad(np64(d["grad_out"]), expd, rm, d["probs"].numpy(), T, K, "bf16")
    dperm, dWg, dWu, dWd = O.expert_mlp_grad(gexp, perm, act, off, np64(d["W_gate"]),
                                             np64(d["W_up"]), np64(d["W_down"]), "bf16")
    assert_normwise(np64(g["dperm"])[:N], dperm, BF16_TOL, "d_permuted")
    for e in range(E):
        assert_normwise(np64(g["dWg"][e]), dWg[e], BF16_TOL, f"dW_gate[{e}]")
        assert_normwise(np64(g["dWd"][e]), dWd[e], BF16_TOL, f"dW_down[{e}]")


def test_bf16_mlp_grad_without_rows_writes_zero_weight_grads(lib):
    E, H, I = 3, 128, 64
    Wg = torch.randn(E, I, H, device=DEV).bfloat16()
    Wu = torch.randn(E, I, H, device=DEV).bfloat16()
    Wd = torch.randn(E, H, I, device=DEV).bfloat16()
    off = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    x = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    a = torch.empty((0, I), dtype=torch.bfloat16, device=DEV)
    gu = torch.empty((0, 2 * I), dtype=torch.bfloat16, device=DEV)
    fill = dict(dW_gate=torch.full_like(Wg, 3.0), dW_up=torch.full_like(Wu, 3.0),
                dW_down=torch.full_like(Wd, 3.0))
    _, dWg, dWu, dWd = lib.moe_expert_mlp_grad(x, x, a, gu, off, Wg, Wu, Wd, **fill)
    torch.cuda.synchronize()
    assert not dWg.any() and not dWu.any() and not dWd.any()


def test_bf16_layer_backward_full_size(lib):
    """T=4096 H=2048 E=128 K=8 I=768 forward + backward: sampled rows of the
    forward's act, expanded and layer output, sampled experts' weight grads
    and rows of d_permuted against the oracle."""
    d = moe_inputs.layer_fwd_bwd(0)
    T, K, E = d["T"], d["K"], d["E"]
    g = _gpu_layer_fwd_bwd(lib, d)
    si, rm, tpe, off = O.permute_routing(d["expert_ids"].numpy(), E)
    assert np.array_equal(np64(g["r"].row_map), rm)
    _check_sampled_forward(d, si, rm, g["act"], g["expanded"], g["out"], seed=4)
    probs = d["probs"].numpy()
    gout = np64(d["grad_out"])
    tok = np64(d["tokens"])
    Wg, Wu, Wd = np64(d["W_gate"]), np64(d["W_up"]), np64(d["W_down"])
    for e in [0, 37, 127]:
        lo, hi = int(off[e]), int(off[e + 1])
        slots = si[lo:hi]
        X = O.permute_rows(tok, slots, K)
        sub_off = np.array([0, hi - lo])
        act, y, _, _ = O.expert_mlp(X, sub_off, Wg[e:e + 1], Wu[e:e + 1], Wd[e:e + 1], "bf16")
        # grad of the expert outputs: probs[f] * grad_out[t] for each slot f
        dY = O.round_to_bf16(probs.reshape(-1)[slots][:, None] * gout[slots // K])
        dX, dWg, dWu, dWd = O.expert_mlp_grad(dY, X, act, sub_off, Wg[e:e + 1], Wu[e:e + 1],
                                              Wd[e:e + 1], "bf16")
        assert_normwise(np64(g["dWd"][e]), dWd[0], BF16_TOL, f"dW_down[{e}]")
        assert_normwise(np64(g["dWg"][e]), dWg[0], BF16_TOL, f"dW_gate[{e}]")
        assert_normwise(np64(g["dWu"][e]), dWu[0], BF16_TOL, f"dW_up[{e}]")
        assert_normwise(np64(g["dperm"][lo:hi]), dX, BF16_TOL, f"d_permuted rows of expert {e}")
