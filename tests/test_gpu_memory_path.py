"""GPU parity of the routing and bandwidth kernels against the CPU oracle.

Integer outputs (routing, indices) and copied rows are compared bit for bit;
floating outputs within the normwise tolerances of tests/gpu_util.py.  Sizes
span several kernel blocks with ragged tails; the full-size workloads are
checked on every integer output and on sampled token rows.
"""

import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from gpu_util import BF16_TOL, F32_TOL, assert_normwise, np64, tol_for, torch_dtype

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _ids(seed, T, K, n_ids):
    rng = np.random.Generator(np.random.PCG64(seed))
    return moe_inputs.uniform_distinct_ids(rng, T, K, n_ids)


def _routing_check(lib, ids_cpu, E, special):
    T, K = ids_cpu.shape
    r = lib.moe_permute(None, ids_cpu.to(DEV), E, special)
    si, rm, tpe, off = O.permute_routing(ids_cpu.numpy(), E, special)
    N = len(si)
    assert np.array_equal(np64(r.expert_offsets), off)
    assert np.array_equal(np64(r.tokens_per_expert), tpe)
    assert np.array_equal(np64(r.row_map), rm)
    assert np.array_equal(np64(r.sorted_indices)[:N], si)
    return r, (si, rm, tpe, off)


ROUTING_CASES = [
    (1, 1, 1, 0),
    (3, 2, 4, 0),
    (100, 8, 64, 0),
    (2049, 3, 17, 0),        # 6147 slots: twelve 512-slot blocks and a ragged tail
    (5000, 8, 256, 12),      # special ids are not dispatched
    (777, 16, 1024, 0),      # K and E at their limits
    (300, 4, 8, 8),
]


@pytest.mark.parametrize("T,K,E,special", ROUTING_CASES)
def test_routing_bit_exact(lib, T, K, E, special):
    _routing_check(lib, _ids(T + K + E, T, K, E + special), E, special)


def _routing_launches(lib, ids_cpu, E):
    before = lib.moe_kernel_launches()
    r = lib.moe_permute(None, ids_cpu.to(DEV), E, 0)
    torch.cuda.synchronize()
    return r, lib.moe_kernel_launches() - before


def _assert_routing(r, ids_cpu, E):
    si, rm, tpe, off = O.permute_routing(ids_cpu.numpy(), E)
    assert np.array_equal(np64(r.expert_offsets), off)
    assert np.array_equal(np64(r.tokens_per_expert), tpe)
    assert np.array_equal(np64(r.row_map), rm)
    assert np.array_equal(np64(r.sorted_indices)[: len(si)], si)


def test_routing_is_one_launch_when_its_blocks_fit(lib):
    """6147 slots, twelve 512-slot blocks: histogram, scan and stable
    placement run as one cooperative launch."""
    ids = _ids(11, 2049, 3, 17)
    r, launches = _routing_launches(lib, ids, 17)
    assert launches == 1
    _assert_routing(r, ids, 17)


def test_routing_three_passes_past_residency(lib):
    """2,097,152 slots need 4096 blocks, more than the GPU holds at once: the
    routing falls back to its three launches and stays bit exact."""
    ids = _ids(12, 262144, 8, 64)
    r, launches = _routing_launches(lib, ids, 64)
    assert launches == 3
    _assert_routing(r, ids, 64)


def test_routing_twice_on_one_workspace(lib):
    """The fused routing's completion flags are stamped per call, so a
    workspace that still holds an earlier call's counts and flags (here a
    different routing of the same size) gives the same result as a fresh
    one."""
    T, K, E = 3000, 8, 64
    ws = torch.zeros(lib.moe_permute_workspace_size(T, K, E), dtype=torch.uint8, device=DEV)
    for seed in (21, 22, 21):
        ids = _ids(seed, T, K, E)
        r = lib.moe_permute(None, ids.to(DEV), E, 0, workspace=ws)
        _assert_routing(r, ids, E)


def test_routing_empty_and_all_special(lib):
    ids = torch.zeros((0, 4), dtype=torch.int32)
    r = lib.moe_permute(None, ids.to(DEV), 8, 0)
    assert not np64(r.tokens_per_expert).any() and not np64(r.expert_offsets).any()
    ids = torch.tensor([[8, 9], [9, 8]], dtype=torch.int32)     # only special ids
    r, (si, rm, tpe, off) = _routing_check(lib, ids, 8, 2)
    assert off[-1] == 0 and np.all(np64(r.row_map) == -1)


def test_routing_reports_bad_ids(lib):
    ids = _ids(5, 64, 4, 16)
    bad_range = ids.clone()
    bad_range[3, 1] = 16                       # outside [0, E + special)
    st = lib.new_status()
    lib.moe_permute(None, bad_range.to(DEV), 16, 0, dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_ERR_BAD_ID
    repeated = ids.clone()
    repeated[7, 2] = repeated[7, 0]
    st = lib.new_status()
    r = lib.moe_permute(None, repeated.to(DEV), 16, 0, dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_ERR_BAD_ID
    # the repeated slot is not dispatched; every other slot is
    assert int(np64(r.row_map)[7 * 4 + 2]) == -1
    assert int(np64(r.expert_offsets)[-1]) == 64 * 4 - 1
    ok = lib.new_status()
    lib.moe_permute(None, ids.to(DEV), 16, 0, dev_status=ok)
    assert lib.moe_check_status(ok) == lib.MOE_OK


def test_host_rejects_bad_shapes(lib):
    ids = _ids(1, 8, 4, 8).to(DEV)
    with pytest.raises(lib.MoeError) as e:
        lib.moe_permute(None, ids, 2, 0)           # K = 4 > E = 2
    assert e.value.status == lib.MOE_ERR_SHAPE
    tok = torch.zeros((8, 12), dtype=torch.bfloat16, device=DEV)   # 24-byte rows
    with pytest.raises(lib.MoeError) as e:
        lib.moe_permute(tok, ids, 8, 0)
    assert e.value.status == lib.MOE_ERR_SHAPE


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,K,E,H", [(37, 2, 5, 64), (1000, 8, 64, 520), (2100, 3, 33, 8)])
def test_permute_rows_bit_exact(lib, dtype, T, K, E, H):
    if dtype == "f32" and H % 4:
        pytest.skip("fp32 rows need H % 4 == 0")
    ids = _ids(T * 7 + H, T, K, E)
    rng = np.random.default_rng(T)
    tokens = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch_dtype(dtype))
    r = lib.moe_permute(tokens.to(DEV), ids.to(DEV), E, 0)
    si, rm, tpe, off = O.permute_routing(ids.numpy(), E)
    want = O.permute_rows(np64(tokens), si, K)
    assert np.array_equal(np64(r.permuted)[: len(si)], want)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,K,E,H,special", [(37, 2, 5, 64, 0), (513, 8, 64, 256, 0),
                                             (300, 4, 8, 128, 3), (1, 16, 16, 8, 0)])
def test_unpermute_and_grads(lib, dtype, T, K, E, H, special):
    if dtype == "f32" and H % 4:
        pytest.skip("fp32 rows need H % 4 == 0")
    tol = tol_for(dtype)
    td = torch_dtype(dtype)
    ids = _ids(T + 3 * K + H, T, K, E + special)
    rng = np.random.default_rng(H + T)
    si, rm, tpe, off = O.permute_routing(ids.numpy(), E, special)
    N = len(si)
    expanded = torch.from_numpy(rng.standard_normal((max(N, 1), H)).astype(np.float32)).to(td)[:N]
    probs = moe_inputs.softmax_probs(rng, T, K)
    grad_out = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(td)
    r = lib.moe_permute(None, ids.to(DEV), E, special)
    assert np.array_equal(np64(r.row_map), rm)
    ex_d = expanded.to(DEV).contiguous()
    out = lib.moe_unpermute(ex_d, r.row_map, probs.to(DEV), T, K)
    assert_normwise(np64(out), O.unpermute(np64(expanded), rm, probs.numpy(), T, K, dtype), tol, "unpermute")
    out1 = lib.moe_unpermute(ex_d, r.row_map, None, T, K)
    assert_normwise(np64(out1), O.unpermute(np64(expanded), rm, None, T, K, dtype), tol, "unpermute p=1")
    gp, gprob = lib.moe_unpermute_grad(grad_out.to(DEV), ex_d, r.row_map, probs.to(DEV), K)
    w_gp, w_gprob = O.unpermute_grad(np64(grad_out), np64(expanded), rm, probs.numpy(), T, K, dtype)
    assert_normwise(np64(gp), w_gp, tol, "grad_permuted")
    assert_normwise(np64(gprob), w_gprob, F32_TOL, "grad_probs")
    gt = lib.moe_permute_grad(ex_d, r.row_map, T, K)
    assert_normwise(np64(gt), O.permute_grad(np64(expanded), rm, T, K, dtype), tol, "permute_grad")


def test_unpermute_k1_roundtrip_is_identity(lib):
    T, H, E = 3000, 136, 7
    ids = torch.from_numpy(np.random.default_rng(2).integers(0, E, (T, 1)).astype(np.int32))
    tok = torch.from_numpy(np.random.default_rng(3).standard_normal((T, H)).astype(np.float32))
    tok = tok.to(torch.bfloat16).to(DEV)
    r = lib.moe_permute(tok, ids.to(DEV), E, 0)
    back = lib.moe_unpermute(r.permuted, r.row_map, None, T, 1)
    assert torch.equal(back, tok)
    back2 = lib.moe_unpermute(r.permuted, r.row_map, torch.ones((T, 1), device=DEV), T, 1)
    assert torch.equal(back2, tok)


def test_invert_sorted_indices(lib):
    ids = _ids(11, 999, 4, 40)
    r = lib.moe_permute(None, ids.to(DEV), 37, 3)
    si, rm, _, _ = O.permute_routing(ids.numpy(), 37, 3)
    rm2 = lib.moe_invert_sorted_indices(r.sorted_indices, len(si), 999 * 4)
    assert np.array_equal(np64(rm2), rm)


# ---------------------------------------------------------------- combine

@pytest.mark.parametrize("T,K,E,H,Z,C,Cn,shared", [
    (37, 4, 16, 64, 1, 1, 1, True),
    (500, 8, 64, 264, 4, 4, 4, True),
    (200, 8, 32, 128, 0, 0, 0, False),
    (64, 2, 4, 64, 2, 0, 3, False),
    (300, 8, 32, 520, 2, 2, 2, True),     # 65 column vectors: a ragged last lane pass
    (5000, 4, 16, 520, 1, 1, 1, True),    # 625 blocks of 8 tokens
])
def test_combine(lib, T, K, E, H, Z, C, Cn, shared):
    d = moe_inputs.index_combine(T + H, R=1, E_local=E, T=T, H=H, K=K, zero_num=Z, copy_num=C,
                                 const_num=Cn)
    ids = d["expert_ids"]
    si, rm, _, _ = O.permute_routing(ids.numpy(), E, Z + C + Cn)
    r = lib.moe_permute(None, ids.to(DEV), E, Z + C + Cn)
    assert np.array_equal(np64(r.row_map), rm)
    sx = d["shared_x"] if shared else None
    st = lib.new_status()
    out = lib.moe_combine(d["expanded"].to(DEV), r.row_map, ids.to(DEV), d["scales"].to(DEV), E,
                          shared_x=sx.to(DEV) if shared else None, ori_x=d["ori_x"].to(DEV),
                          zero_num=Z, copy_num=C, const_num=Cn, alpha1=d["alpha1"].to(DEV),
                          alpha2=d["alpha2"].to(DEV), const_v=d["const_v"].to(DEV), dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_OK
    want = O.combine(np64(d["expanded"]), rm, ids.numpy(), d["scales"].numpy(),
                     np64(sx) if shared else None, np64(d["ori_x"]), E, Z, C, Cn,
                     np64(d["alpha1"]), np64(d["alpha2"]), np64(d["const_v"]), "bf16")
    assert_normwise(np64(out), want, BF16_TOL, "combine")


def test_combine_page_example_ids(lib):
    """The 8x8 expert ids of the combine_v2 call example (32 experts, one
    zero, one copy and one const expert)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "combine_v2_example_expert_ids.txt")
    rows = [[int(v) for v in ln.split()] for ln in open(path) if ln.strip() and not ln.startswith("#")]
    ids = torch.tensor(rows, dtype=torch.int32)
    T, K, E, H = 8, 8, 32, 7168
    rng = np.random.Generator(np.random.PCG64(0))
    si, rm, _, _ = O.permute_routing(ids.numpy(), E, 3)
    expanded = torch.from_numpy(rng.standard_normal((len(si), H)).astype(np.float32)).bfloat16()
    ori = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).bfloat16()
    a1 = torch.from_numpy(rng.uniform(-1, 1, (1, H)).astype(np.float32)).bfloat16()
    a2 = torch.from_numpy(rng.uniform(-1, 1, (1, H)).astype(np.float32)).bfloat16()
    v = torch.from_numpy(rng.uniform(-1, 1, (1, H)).astype(np.float32)).bfloat16()
    s = torch.from_numpy(rng.standard_normal((T, K)).astype(np.float32))
    r = lib.moe_permute(None, ids.to(DEV), E, 3)
    out = lib.moe_combine(expanded.to(DEV), r.row_map, ids.to(DEV), s.to(DEV), E, ori_x=ori.to(DEV),
                          zero_num=1, copy_num=1, const_num=1, alpha1=a1.to(DEV), alpha2=a2.to(DEV),
                          const_v=v.to(DEV))
    want = O.combine(np64(expanded), rm, ids.numpy(), s.numpy(), None, np64(ori), E, 1, 1, 1,
                     np64(a1), np64(a2), np64(v), "bf16")
    assert_normwise(np64(out), want, BF16_TOL, "combine page example")


def test_combine_reports_ids_past_special_ranges(lib):
    ids = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32)
    r = lib.moe_permute(None, ids.to(DEV), 4, 5)        # routing accepts id 9 < 4 + 5
    st = lib.new_status()
    lib.moe_combine(torch.zeros((3, 64), dtype=torch.bfloat16, device=DEV), r.row_map,
                    ids.to(DEV), torch.ones((2, 2), device=DEV), 4, ori_x=torch.zeros((2, 64), dtype=torch.bfloat16, device=DEV),
                    zero_num=1, copy_num=1, const_num=0, dev_status=st)   # 9 >= 4 + 2
    assert lib.moe_check_status(st) == lib.MOE_ERR_BAD_ID


# ---------------------------------------------------------------- permute indices

@pytest.mark.parametrize("R,E,lam", [(1, 1, 5.0), (1, 7, 3.0), (5, 1, 3.0), (16, 16, 64.0),
                                     (32, 64, 2.0), (3, 4, 0.0)])
def test_permute_indices_bit_exact(lib, R, E, lam):
    rng = np.random.Generator(np.random.PCG64(R * 100 + E))
    counts = torch.from_numpy(rng.poisson(lam, R * E).astype(np.int32))
    want_idx, want_tpe, want_total = O.permute_indices(counts.numpy(), R, E)
    cap = max(want_total, 1)
    st = lib.new_status()
    idx, tpe, total = lib.moe_permute_indices(counts.to(DEV), R, E, cap, dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_OK
    assert int(total.item()) == want_total
    assert np.array_equal(np64(tpe), want_tpe)
    assert np.array_equal(np64(idx)[:want_total], want_idx)


def test_permute_indices_capacity_overflow(lib):
    counts = torch.full((4,), 10, dtype=torch.int32)
    st = lib.new_status()
    idx = torch.full((16,), -7, dtype=torch.int32, device=DEV)
    lib.moe_permute_indices(counts.to(DEV), 2, 2, 16, indices=idx, dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_ERR_CAPACITY
    assert torch.all(idx == -7)                  # nothing written past the check


# ---------------------------------------------------------------- full-size workloads (sampled)

def _sample(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, size=min(k, n), replace=False))


def test_permute_unpermute_full_size_bf16(lib):
    """T=16384, H=4096, E=64, K=8: every integer output bit-exact, sampled
    rows of permuted, out, grad_permuted, grad_probs against the oracle."""
    d = moe_inputs.permute_unpermute(0)
    T, H, E, K = d["T"], d["H"], d["E"], d["K"]
    ids = d["expert_ids"]
    tok = d["tokens"]
    r, (si, rm, tpe, off) = None, O.permute_routing(ids.numpy(), E)
    r = lib.moe_permute(tok.to(DEV), ids.to(DEV), E, 0)
    assert np.array_equal(np64(r.row_map), rm)
    assert np.array_equal(np64(r.sorted_indices), si)
    assert np.array_equal(np64(r.expert_offsets), off)
    rows = _sample(T * K, 3000, 1)
    got_rows = np64(r.permuted[torch.from_numpy(rows).to(DEV)])
    assert np.array_equal(got_rows, O.permute_rows(np64(tok), si[rows], K))
    probs, gout = d["probs"], d["grad_out"]
    out = lib.moe_unpermute(r.permuted, r.row_map, probs.to(DEV), T, K)
    gp, gprob = lib.moe_unpermute_grad(gout.to(DEV), r.permuted, r.row_map, probs.to(DEV), K)
    ts = _sample(T, 400, 2)
    slots = (ts[:, None] * K + np.arange(K)[None, :]).reshape(-1)
    # sub-problem of the sampled tokens: their K oracle-permuted rows
    sub_rows = O.permute_rows(np64(tok), slots, K)
    sub_rm = np.arange(len(slots))
    w_out = O.unpermute(sub_rows, sub_rm, probs.numpy()[ts], len(ts), K, "bf16")
    assert_normwise(np64(out[torch.from_numpy(ts).to(DEV)]), w_out, BF16_TOL, "unpermute full")
    w_gp, w_gprob = O.unpermute_grad(np64(gout)[ts], sub_rows, sub_rm, probs.numpy()[ts], len(ts), K, "bf16")
    got_gp = np64(gp[torch.from_numpy(rm[slots]).to(DEV)])
    assert_normwise(got_gp, w_gp, BF16_TOL, "grad_permuted full")
    assert_normwise(np64(gprob)[ts], w_gprob, F32_TOL, "grad_probs full")
    gt = lib.moe_permute_grad(gp, r.row_map, T, K)
    w_gt = O.permute_grad(w_gp, sub_rm, len(ts), K, "bf16")
    assert_normwise(np64(gt[torch.from_numpy(ts).to(DEV)]), w_gt, BF16_TOL, "permute_grad full")


def test_index_and_combine_full_size(lib):
    """counts[16 x 16] ~ Poisson(64) and combine T=4096, H=7168, K=8 over 256
    real + 4 zero + 4 copy + 4 const experts, all outputs compared."""
    d = moe_inputs.index_combine(0)
    R, El = d["R"], d["E_local"]
    want_idx, want_tpe, want_total = O.permute_indices(d["counts"].numpy(), R, El)
    idx, tpe, total = lib.moe_permute_indices(d["counts"].to(DEV), R, El, want_total)
    assert int(total.item()) == want_total
    assert np.array_equal(np64(idx)[:want_total], want_idx)
    assert np.array_equal(np64(tpe), want_tpe)
    E, Z, C, Cn = d["E"], d["zero_num"], d["copy_num"], d["const_num"]
    ids = d["expert_ids"]
    si, rm, _, _ = O.permute_routing(ids.numpy(), E, Z + C + Cn)
    r = lib.moe_permute(None, ids.to(DEV), E, Z + C + Cn)
    assert np.array_equal(np64(r.row_map), rm)
    out = lib.moe_combine(d["expanded"].to(DEV), r.row_map, ids.to(DEV), d["scales"].to(DEV), E,
                          shared_x=d["shared_x"].to(DEV), ori_x=d["ori_x"].to(DEV), zero_num=Z,
                          copy_num=C, const_num=Cn, alpha1=d["alpha1"].to(DEV),
                          alpha2=d["alpha2"].to(DEV), const_v=d["const_v"].to(DEV))
    want = O.combine(np64(d["expanded"]), rm, ids.numpy(), d["scales"].numpy(), np64(d["shared_x"]),
                     np64(d["ori_x"]), E, Z, C, Cn, np64(d["alpha1"]), np64(d["alpha2"]),
                     np64(d["const_v"]), "bf16")
    assert_normwise(np64(out), want, BF16_TOL, "combine full")


# ---------------------------------------------------------------- deredundancy indices

@pytest.mark.parametrize("nsrc,NE,start,D,L,lam", [(2, 4, 2, 1, 2, 2.0), (8, 256, 64, 4, 16, 8.0),
                                                   (3, 40, 0, 5, 8, 1.0), (8, 256, 0, 1, 1, 0.0),
                                                   (16, 128, 120, 2, 4, 64.0)])
def test_deredundancy_indices_bit_exact(lib, nsrc, NE, start, D, L, lam):
    rng = np.random.Generator(np.random.PCG64(nsrc * 1000 + NE + start))
    counts = rng.poisson(lam, size=(nsrc, NE)).astype(np.int32)
    want_idx, want_n, want_total = O.deredundancy_dispatch_indices(counts, start, D, L)
    st = lib.new_status()
    idx, n, total = lib.moe_permute_indices_window(torch.from_numpy(counts.reshape(-1)).to(DEV), nsrc,
                                                   NE, start, D * L, max(want_total, 1),
                                                   dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_OK
    assert int(total.item()) == want_total
    assert np.array_equal(np64(idx)[:want_total], want_idx)
    assert np.array_equal(np64(n)[:D * L], want_n)


def test_full_window_equals_permute_indices(lib):
    rng = np.random.Generator(np.random.PCG64(9))
    counts = torch.from_numpy(rng.poisson(5.0, 12 * 20).astype(np.int32)).to(DEV)
    a, na, ta = lib.moe_permute_indices(counts, 12, 20, 12 * 20 * 20)
    b, nb, tb = lib.moe_permute_indices_window(counts, 12, 20, 0, 20, 12 * 20 * 20)
    n = int(ta.item())
    assert n == int(tb.item()) and torch.equal(a[:n], b[:n]) and torch.equal(na, nb[:20])


# ---------------------------------------------------------------- activity mask

@pytest.mark.parametrize("dims", [1, 2])
def test_masked_permute_and_combine(lib, dims):
    d = moe_inputs.index_combine(3, R=1, E_local=32, T=700, H=128, K=8, zero_num=2, copy_num=2,
                                 const_num=2)
    T, K, E = d["T"], d["K"], d["E"]
    ids = d["expert_ids"]
    rng = np.random.default_rng(dims)
    mask = rng.random(T) < 0.7 if dims == 1 else rng.random((T, K)) < 0.7
    mask_t = torch.from_numpy(mask).to(DEV)
    si, rm, tpe, off = O.permute_routing(ids.numpy(), E, 6, active_mask=mask)
    tok = torch.from_numpy(rng.standard_normal((T, 128)).astype(np.float32)).bfloat16()
    r = lib.moe_permute(tok.to(DEV), ids.to(DEV), E, 6, active_mask=mask_t)
    assert np.array_equal(np64(r.row_map), rm)
    assert np.array_equal(np64(r.expert_offsets), off)
    assert np.array_equal(np64(r.permuted)[: len(si)], O.permute_rows(np64(tok), si, K))
    expanded = torch.from_numpy(rng.standard_normal((max(len(si), 1), 128)).astype(np.float32)).bfloat16()[: len(si)]
    out = lib.moe_combine(expanded.to(DEV).contiguous(), r.row_map, ids.to(DEV), d["scales"].to(DEV), E,
                          shared_x=d["shared_x"].to(DEV), ori_x=d["ori_x"].to(DEV), zero_num=2,
                          copy_num=2, const_num=2, alpha1=d["alpha1"].to(DEV),
                          alpha2=d["alpha2"].to(DEV), const_v=d["const_v"].to(DEV),
                          active_mask=mask_t)
    want = O.combine(np64(expanded), rm, ids.numpy(), d["scales"].numpy(), np64(d["shared_x"]),
                     np64(d["ori_x"]), E, 2, 2, 2, np64(d["alpha1"]), np64(d["alpha2"]),
                     np64(d["const_v"]), "bf16", active_mask=mask)
    assert_normwise(np64(out), want, BF16_TOL, "masked combine")
