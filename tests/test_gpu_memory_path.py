"""GPU parity of the routing and bandwidth kernels against the CPU oracle.

Integer outputs (routing, indices) and copied rows are compared bit for bit.
Floating outputs are held to what each kernel's arithmetic guarantees: the
unpermute, the permute backward and the combine accumulate in fp32 and round
once, so every element must lie within one step of the storage format plus
the fp32 summation error bound of the oracle's value (assert_elementwise);
grad_permuted is one fp32 product rounded once, exactly as the oracle rounds
it, so it is compared bit for bit.  The normwise bars of tests/gpu_util.py
are kept beside them.  Sizes span several kernel blocks with ragged tails;
the full-size workloads are checked on every integer output and on sampled
token rows.
"""

import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from gpu_util import (BF16_TOL, F32_TOL, assert_bitwise, assert_elementwise, assert_normwise,
                      np64, tol_for, torch_dtype)

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


@pytest.mark.parametrize("E", [64, 17])
def test_routing_workspace_alignment(lib, E):
    """The routing's per-block counts are read 16 bytes at a time when E is
    a multiple of 4 (one count at a time otherwise) and its flags are
    8-byte words, so the workspace must be 16-byte aligned: a workspace 4
    bytes past a 16-byte boundary is refused on the host, before any launch,
    and an aligned one gives the oracle's routing bit for bit."""
    T, K = 2049, 8
    ids = _ids(5, T, K, E)
    size = lib.moe_permute_workspace_size(T, K, E)
    base = torch.zeros(size + 16, dtype=torch.uint8, device=DEV)
    assert base.data_ptr() % 16 == 0
    with pytest.raises(lib.MoeError) as err:
        lib.moe_permute(None, ids.to(DEV), E, 0, workspace=base[4: 4 + size])
    assert err.value.status == lib.MOE_ERR_INVALID_ARG
    r = lib.moe_permute(None, ids.to(DEV), E, 0, workspace=base[:size])
    _assert_routing(r, ids, E)


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


@pytest.mark.parametrize("T,K,E", [(32768, 8, 256), (29127, 9, 1000), (13, 5, 7)])
def test_routing_one_launch_sizes(lib, T, K, E):
    """The one-launch routing from 65 to 262143 slots (blocks of 512 slots up
    to 64 blocks, of 1024 slots past that: up to 256 blocks), with K that
    does and does not divide a warp's 32 slots and up to 1000 experts."""
    ids = _ids(T + K, T, K, E)
    r, launches = _routing_launches(lib, ids, E)
    assert launches == 1
    _assert_routing(r, ids, E)


def test_routing_one_launch_625_blocks(lib):
    """320000 slots, 313 blocks of 1024 slots, resident at once: one
    cooperative launch, bit exact."""
    ids = _ids(13, 40000, 8, 64)
    r, launches = _routing_launches(lib, ids, 64)
    assert launches == 1
    _assert_routing(r, ids, 64)


def test_routing_three_passes_past_residency(lib):
    """2,097,152 slots need 2048 blocks of 1024 slots, more than the GPU
    holds at once: the routing falls back to its three launches (blocks of
    512 slots) and stays bit exact."""
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


def test_empty_token_batches(lib):
    """T = 0 through every memory-bound entry point: each returns MOE_OK,
    writes nothing and reads nothing (empty buffers, counts all zero)."""
    H, K, E = 64, 4, 8
    bf = torch.bfloat16
    tok = torch.empty((0, H), dtype=bf, device=DEV)
    ids = torch.empty((0, K), dtype=torch.int32, device=DEV)
    r = lib.moe_permute(tok, ids, E, 0)
    assert r.permuted.shape[0] == 0 and not np64(r.tokens_per_expert).any()
    assert not np64(r.expert_offsets).any()
    rm = torch.empty(0, dtype=torch.int32, device=DEV)
    probs = torch.empty((0, K), dtype=torch.float32, device=DEV)
    rows = torch.empty((0, H), dtype=bf, device=DEV)
    assert lib.moe_unpermute(rows, rm, probs, 0, K).shape == (0, H)
    assert lib.moe_permute_grad(rows, rm, 0, K).shape == (0, H)
    gp, gprobs = lib.moe_unpermute_grad(tok, rows, rm, probs, K)
    assert gp.shape == (0, H) and gprobs.shape == (0, K)
    assert lib.moe_permute_rows(tok, rm, K, 0).shape == (0, H)
    out = lib.moe_combine(rows, rm, ids, probs, E)
    assert out.shape == (0, H)
    # counts all zero: no index, every expert empty, total 0
    counts = torch.zeros(4 * E, dtype=torch.int32, device=DEV)
    _, tpe, total = lib.moe_permute_indices(counts, 4, E, 16)
    assert int(total.item()) == 0 and not np64(tpe).any()


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
    # K = 6 does not divide a 32-slot step: rows straddle steps and warps
    ids6 = _ids(6, 300, 6, 16)
    rep6 = ids6.clone()
    rep6[171, 5] = rep6[171, 0]                # slot 1031 repeats slot 1026 (row 171 spans slots 1026-1031)
    st = lib.new_status()
    r = lib.moe_permute(None, rep6.to(DEV), 16, 0, dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_ERR_BAD_ID
    assert int(np64(r.row_map)[171 * 6 + 5]) == -1
    assert int(np64(r.expert_offsets)[-1]) == 300 * 6 - 1


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
    Y, G, p = np64(expanded), np64(grad_out), probs.numpy()
    out = lib.moe_unpermute(ex_d, r.row_map, probs.to(DEV), T, K)
    want = O.unpermute(Y, rm, p, T, K, dtype)
    assert_normwise(np64(out), want, tol, "unpermute")
    mag = O.unpermute(np.abs(Y), rm, np.abs(p), T, K, "f64")
    assert_elementwise(np64(out), want, mag, K, dtype, "unpermute")
    out1 = lib.moe_unpermute(ex_d, r.row_map, None, T, K)
    want = O.unpermute(Y, rm, None, T, K, dtype)
    assert_normwise(np64(out1), want, tol, "unpermute p=1")
    assert_elementwise(np64(out1), want, O.unpermute(np.abs(Y), rm, None, T, K, "f64"), K, dtype,
                       "unpermute p=1")
    gp, gprob = lib.moe_unpermute_grad(grad_out.to(DEV), ex_d, r.row_map, probs.to(DEV), K)
    w_gp, w_gprob = O.unpermute_grad(G, Y, rm, p, T, K, dtype)
    assert_normwise(np64(gp), w_gp, tol, "grad_permuted")
    assert_bitwise(np64(gp), w_gp, "grad_permuted")
    assert_normwise(np64(gprob), w_gprob, F32_TOL, "grad_probs")
    # each lane chains H/32 fp32 FMAs, then five shuffle additions
    _, mag_p = O.unpermute_grad(np.abs(G), np.abs(Y), rm, None, T, K, "f64")
    assert_elementwise(np64(gprob), w_gprob, mag_p, H // 32 + 5, "f32", "grad_probs")
    gt = lib.moe_permute_grad(ex_d, r.row_map, T, K)
    want = O.permute_grad(Y, rm, T, K, dtype)
    assert_normwise(np64(gt), want, tol, "permute_grad")
    assert_elementwise(np64(gt), want, O.permute_grad(np.abs(Y), rm, T, K, "f64"), K, dtype,
                       "permute_grad")


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

def _combine_mag(expanded, rm, ids, scales, shared_x, ori_x, E, Z, C, Cn, a1, a2, v,
                 active_mask=None):
    """Per element, the sum of the absolute values of the combine's terms:
    the oracle's combine of the inputs' absolute values, unrounded."""
    ab = lambda x: None if x is None else np.abs(x)  # noqa: E731
    return O.combine(ab(expanded), rm, ids, ab(scales), ab(shared_x), ab(ori_x), E, Z, C, Cn,
                     ab(a1), ab(a2), ab(v), "f64", active_mask=active_mask)


def _combine_roundings(K):
    # per slot: a const expert's two fp32 operations and the FMA into the sum;
    # then the shared-expert addition
    return 3 * K + 1


@pytest.mark.parametrize("T,K,E,H,Z,C,Cn,shared", [
    (37, 4, 16, 64, 1, 1, 1, True),
    (500, 8, 64, 264, 4, 4, 4, True),
    (200, 8, 32, 128, 0, 0, 0, False),
    (64, 2, 4, 64, 2, 0, 3, False),
    (300, 8, 32, 520, 2, 2, 2, True),     # 65 column vectors: a ragged last lane pass
    (5000, 4, 16, 520, 1, 1, 1, True),    # 625 blocks of 8 tokens
    # rows split into column runs of whole 32-vector steps, one warp each,
    # the last run ragged: 2 runs (257 vectors), 3 (385), 4 (513)
    (300, 8, 32, 2056, 2, 2, 2, True),
    (129, 6, 24, 3080, 1, 2, 1, True),
    (70, 8, 32, 4104, 2, 2, 2, False),
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
    args = (np64(d["expanded"]), rm, ids.numpy(), d["scales"].numpy(),
            np64(sx) if shared else None, np64(d["ori_x"]), E, Z, C, Cn,
            np64(d["alpha1"]), np64(d["alpha2"]), np64(d["const_v"]))
    want = O.combine(*args, "bf16")
    assert_normwise(np64(out), want, BF16_TOL, "combine")
    assert_elementwise(np64(out), want, _combine_mag(*args), _combine_roundings(K), "bf16",
                       "combine")


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
    args = (np64(expanded), rm, ids.numpy(), s.numpy(), None, np64(ori), E, 1, 1, 1,
            np64(a1), np64(a2), np64(v))
    want = O.combine(*args, "bf16")
    assert_normwise(np64(out), want, BF16_TOL, "combine page example")
    assert_elementwise(np64(out), want, _combine_mag(*args), _combine_roundings(K), "bf16",
                       "combine page example")


def test_combine_reports_ids_past_special_ranges(lib):
    ids = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32)
    r = lib.moe_permute(None, ids.to(DEV), 4, 6)        # routing accepts id 9 < 4 + 6
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


def test_permute_indices_sum_past_int32(lib):
    """Counts whose sum passes 2^31 - 1 (four of 2^30 - 1, and one more): the
    64-bit check reports a capacity error, sets total = -1 and writes no
    index or count."""
    counts = torch.tensor([2 ** 30 - 1] * 4 + [3], dtype=torch.int32)
    assert int(counts.sum(dtype=torch.int64)) > 2 ** 31 - 1
    idx = torch.full((64,), -7, dtype=torch.int32, device=DEV)
    tpe = torch.full((5,), -7, dtype=torch.int32, device=DEV)
    st = lib.new_status()
    _, _, total = lib.moe_permute_indices(counts.to(DEV), 1, 5, 64, indices=idx,
                                          tokens_per_expert=tpe, dev_status=st)
    assert lib.moe_check_status(st) == lib.MOE_ERR_CAPACITY
    assert int(total.item()) == -1
    assert torch.all(idx == -7) and torch.all(tpe == -7)


# ---------------------------------------------------------------- row copy with a given routing

def test_permute_rows_skips_rows_outside_the_buffer(lib):
    """moe_permute_rows copies token rows to the rows row_map names, and
    skips every entry outside [0, N): -1, N, large and negative values made
    on the host leave the buffer untouched; valid entries are exact copies."""
    T, K, H, N = 40, 3, 64, 100
    rng = np.random.default_rng(5)
    tok = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).bfloat16()
    rm = np.full(T * K, -1, dtype=np.int64)
    valid = rng.choice(T * K, 60, replace=False)
    rm[valid] = rng.choice(N - 10, 60, replace=False)      # rows [0, 90) only
    junk = np.setdiff1d(np.arange(T * K), valid)
    rm[junk[0::4]] = N
    rm[junk[1::4]] = N + 12345
    rm[junk[2::4]] = 2 ** 31 - 1
    rm[junk[3::4]] = -(2 ** 31)
    sentinel = 3.0
    out = torch.full((N + 16, H), sentinel, dtype=torch.bfloat16, device=DEV)  # 16 rows past N
    lib.moe_permute_rows(tok.to(DEV), torch.from_numpy(rm.astype(np.int32)).to(DEV), K, N,
                         permuted=out)
    torch.cuda.synchronize()
    got = np64(out)
    assert np.all(got[N:] == sentinel)
    written = np.zeros(N + 16, dtype=bool)
    written[rm[valid]] = True
    assert np.all(got[~written] == sentinel)
    assert np.array_equal(got[rm[valid]], np64(tok)[valid // K])


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
    p_s, g_s = probs.numpy()[ts], np64(gout)[ts]
    w_out = O.unpermute(sub_rows, sub_rm, p_s, len(ts), K, "bf16")
    got_out = np64(out[torch.from_numpy(ts).to(DEV)])
    assert_normwise(got_out, w_out, BF16_TOL, "unpermute full")
    assert_elementwise(got_out, w_out, O.unpermute(np.abs(sub_rows), sub_rm, np.abs(p_s), len(ts), K, "f64"),
                       K, "bf16", "unpermute full")
    w_gp, w_gprob = O.unpermute_grad(g_s, sub_rows, sub_rm, p_s, len(ts), K, "bf16")
    got_gp = np64(gp[torch.from_numpy(rm[slots]).to(DEV)])
    assert_normwise(got_gp, w_gp, BF16_TOL, "grad_permuted full")
    assert_bitwise(got_gp, w_gp, "grad_permuted full")
    assert_normwise(np64(gprob)[ts], w_gprob, F32_TOL, "grad_probs full")
    _, mag_p = O.unpermute_grad(np.abs(g_s), np.abs(sub_rows), sub_rm, None, len(ts), K, "f64")
    assert_elementwise(np64(gprob)[ts], w_gprob, mag_p, H // 32 + 5, "f32", "grad_probs full")
    gt = lib.moe_permute_grad(gp, r.row_map, T, K)
    w_gt = O.permute_grad(w_gp, sub_rm, len(ts), K, "bf16")
    got_gt = np64(gt[torch.from_numpy(ts).to(DEV)])
    assert_normwise(got_gt, w_gt, BF16_TOL, "permute_grad full")
    assert_elementwise(got_gt, w_gt, O.permute_grad(np.abs(w_gp), sub_rm, len(ts), K, "f64"), K,
                       "bf16", "permute_grad full")


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
    args = (np64(d["expanded"]), rm, ids.numpy(), d["scales"].numpy(), np64(d["shared_x"]),
            np64(d["ori_x"]), E, Z, C, Cn, np64(d["alpha1"]), np64(d["alpha2"]),
            np64(d["const_v"]))
    want = O.combine(*args, "bf16")
    assert_normwise(np64(out), want, BF16_TOL, "combine full")
    assert_elementwise(np64(out), want, _combine_mag(*args), _combine_roundings(d["K"]), "bf16",
                       "combine full")


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


@pytest.mark.parametrize("nsrc,NE,start,D,L,H", [(4, 32, 8, 2, 4, 64), (16, 128, 0, 4, 8, 2048),
                                                 (3, 10, 9, 1, 1, 8)])
def test_whiteboard_combine_of_the_deredundancy_dispatch(lib, nsrc, NE, start, D, L, H):
    """The deredundancy dispatcher's combine (scale each expert output row by
    its router coefficient, scatter-add it to its gathered row of a zero
    whiteboard) on one outer-EP rank, as this library runs it: the dispatch
    indices of moe_permute_indices_window, inverted into a row map by
    moe_invert_sorted_indices, and the unpermute with one slot per gathered
    row weighted by its coefficient.  Each whiteboard row is at most one
    product rounded once, so it matches the oracle bit for bit."""
    rng = np.random.Generator(np.random.PCG64(nsrc * 7 + NE + H))
    counts = rng.poisson(6.0, size=(nsrc, NE)).astype(np.int32)
    n_gathered = int(counts.sum())
    want_idx, _, n = O.deredundancy_dispatch_indices(counts, start, D, L)
    Y = torch.from_numpy(rng.standard_normal((max(n, 1), H)).astype(np.float32)).bfloat16()[:n]
    coeff = torch.from_numpy(rng.random(n_gathered).astype(np.float32))
    idx, _, total = lib.moe_permute_indices_window(torch.from_numpy(counts.reshape(-1)).to(DEV),
                                                   nsrc, NE, start, D * L, max(n, 1))
    assert int(total.item()) == n
    rm = lib.moe_invert_sorted_indices(idx, n, n_gathered)
    wb = lib.moe_unpermute(Y.to(DEV).contiguous(), rm, coeff.reshape(n_gathered, 1).to(DEV),
                           n_gathered, 1)
    want = O.whiteboard_combine(np64(Y), want_idx, coeff.numpy(), n_gathered, "bf16")
    assert_bitwise(np64(wb), want, "whiteboard")


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
    args = (np64(expanded), rm, ids.numpy(), d["scales"].numpy(), np64(d["shared_x"]),
            np64(d["ori_x"]), E, 2, 2, 2, np64(d["alpha1"]), np64(d["alpha2"]),
            np64(d["const_v"]))
    want = O.combine(*args, "bf16", active_mask=mask)
    assert_normwise(np64(out), want, BF16_TOL, "masked combine")
    assert_elementwise(np64(out), want, _combine_mag(*args, active_mask=mask),
                       _combine_roundings(K), "bf16", "masked combine")


@pytest.mark.parametrize("dims", [1, 2])
def test_masked_combine_still_validates_ids(lib, dims):
    """A masked-off slot is not read, but its id must still name an expert:
    an id past the special ranges on a masked slot is reported; routed ids
    on masked slots (row_map -1 after the masked permute) are not."""
    T, K, E, H = 64, 4, 16, 64
    rng = np.random.Generator(np.random.PCG64(40 + dims))
    ids = moe_inputs.uniform_distinct_ids(rng, T, K, E + 3)
    mask = np.ones(T, dtype=bool) if dims == 1 else np.ones((T, K), dtype=bool)
    mask[5] = False                                      # token 5 (all its slots) masked off
    mask_t = torch.from_numpy(mask).to(DEV)
    r = lib.moe_permute(None, ids.to(DEV), E, 3, active_mask=mask_t)
    n = int(r.expert_offsets[-1].item())
    expanded = torch.randn((max(n, 1), H), device=DEV).bfloat16()
    ori = torch.randn((T, H), device=DEV).bfloat16()
    a = torch.ones((1, H), dtype=torch.bfloat16, device=DEV)
    kw = dict(ori_x=ori, zero_num=1, copy_num=1, const_num=1, alpha1=a, alpha2=a, const_v=a,
              active_mask=mask_t)
    st = lib.new_status()
    lib.moe_combine(expanded, r.row_map, ids.to(DEV), torch.ones((T, K), device=DEV), E,
                    dev_status=st, **kw)
    assert lib.moe_check_status(st) == lib.MOE_OK
    bad = ids.clone()
    bad[5, 2] = E + 3                                    # past the special ranges, masked slot
    st = lib.new_status()
    lib.moe_combine(expanded, r.row_map, bad.to(DEV), torch.ones((T, K), device=DEV), E,
                    dev_status=st, **kw)
    assert lib.moe_check_status(st) == lib.MOE_ERR_BAD_ID
