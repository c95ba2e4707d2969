"""GPU parity of the shared expert and of its overlap with the routed path.

The shared expert is the dense MLP over every token (the oracle's expert MLP
with one expert that owns all rows); the combine adds its output as
shared_x.  The layer test runs it on a second stream concurrently with the
routed path and joins the streams with an event before the combine.
"""

import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from gpu_util import BF16_TOL, assert_normwise, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _shared_weights(seed, H, I):
    w = moe_inputs.layer_fwd_bwd(seed, T=1, H=H, E=1, K=1, I=I)
    return w["W_gate"][0], w["W_up"][0], w["W_down"][0]


def _oracle_shared(x, Wg, Wu, Wd):
    T = x.shape[0]
    act, out, _, _ = O.expert_mlp(np64(x), np.array([0, T]), np64(Wg)[None], np64(Wu)[None],
                                  np64(Wd)[None], "bf16")
    return act, out


@pytest.mark.parametrize("T,H,I", [
    (700, 256, 192), (1, 64, 64), (300, 320, 128),
    (1100, 256, 192),     # paired: four full pair tiles and a half tile
])
def test_shared_expert_mlp(lib, T, H, I):
    x = moe_inputs.layer_fwd_bwd(T + I, T=T, H=H, E=1, K=1, I=64)["tokens"]
    Wg, Wu, Wd = _shared_weights(T + H, H, I)
    st = lib.new_status()
    out = lib.moe_shared_expert_mlp(x.to(DEV), Wg.to(DEV), Wu.to(DEV), Wd.to(DEV), dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_OK
    _, w_out = _oracle_shared(x, Wg, Wu, Wd)
    assert_normwise(np64(out), w_out, BF16_TOL, "shared expert")


def test_shared_expert_mlp_full_size(lib):
    """T=4096 H=2048 I=768: 4096 rows in one expert, so both GEMMs run as CTA
    pairs; checked on all rows."""
    x = moe_inputs.layer_fwd_bwd(0)["tokens"]
    Wg, Wu, Wd = _shared_weights(11, 2048, 768)
    out = lib.moe_shared_expert_mlp(x.to(DEV), Wg.to(DEV), Wu.to(DEV), Wd.to(DEV))
    _, w_out = _oracle_shared(x, Wg, Wu, Wd)
    assert_normwise(np64(out), w_out, BF16_TOL, "shared expert")


def test_layer_forward_with_shared_expert_on_a_second_stream(lib):
    d = moe_inputs.layer_fwd_bwd(12, T=600, H=256, E=16, K=4, I=128)
    T, K, E = d["T"], d["K"], d["E"]
    x, ids, probs = d["tokens"].to(DEV), d["expert_ids"].to(DEV), d["probs"].to(DEV)
    Wg, Wu, Wd = d["W_gate"].to(DEV), d["W_up"].to(DEV), d["W_down"].to(DEV)
    Sg, Su, Sd = _shared_weights(13, 256, 192)
    Sg, Su, Sd = Sg.to(DEV), Su.to(DEV), Sd.to(DEV)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ready = torch.cuda.Event()
    ready.record(main)
    with torch.cuda.stream(side):                          # shared expert, concurrently
        side.wait_event(ready)
        shared = lib.moe_shared_expert_mlp(x, Sg, Su, Sd)
        done = torch.cuda.Event()
        done.record(side)
    r = lib.moe_permute(x, ids, E, 0)                      # routed path on the main stream
    _, expanded, _ = lib.moe_expert_mlp(r.permuted, r.expert_offsets, Wg, Wu, Wd)
    main.wait_event(done)
    out = lib.moe_combine(expanded, r.row_map, ids, probs, E, shared_x=shared)
    torch.cuda.synchronize()
    (si, rm, tpe, off) = O.permute_routing(d["expert_ids"].numpy(), E)
    perm = O.permute_rows(np64(d["tokens"]), si, K)
    _, w_exp, _, _ = O.expert_mlp(perm, off, np64(d["W_gate"]), np64(d["W_up"]),
                                  np64(d["W_down"]), "bf16")
    _, w_shared = _oracle_shared(d["tokens"], *_shared_weights(13, 256, 192))
    want = O.combine(O.round_to_bf16(w_exp), rm, d["expert_ids"].numpy(), d["probs"].numpy(),
                     O.round_to_bf16(w_shared), None, E, 0, 0, 0, None, None, None, "bf16")
    assert_normwise(np64(out), want, BF16_TOL, "combine with the shared expert")


def test_shared_expert_rejects_bad_shapes(lib):
    x = torch.zeros((8, 96), dtype=torch.bfloat16, device=DEV)            # H not a multiple of 64
    w = torch.zeros((64, 96), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(lib.MoeError) as e:
        lib.moe_shared_expert_mlp(x, w, w, w.t().contiguous())
    assert e.value.status == lib.MOE_ERR_SHAPE
