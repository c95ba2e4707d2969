"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against something other than itself:
brute force on tiny inputs, closed forms from the combine_v2 API reference,
identities (permute then unpermute is the identity), adjoint identities,
central finite differences in float64, special cases that reduce to a library
routine, and the small worked cases under tests/golden/.  No GPU.
"""

import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
import moe_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return rows


def _rand_ids(rng, T, K, E):
    return np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int64)


# ---------------------------------------------------------------- rounding

def test_bf16_rounding_matches_torch_conversion():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
        # exact ties between two bf16 neighbours: mantissa low half = 0x8000
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -8 * 1.5]),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38]),
    ])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    got = O.round_to_bf16(x)
    assert np.array_equal(got, want)


def test_round_to_f32_is_ieee_single():
    x = np.array([1.0 + 2.0 ** -30, np.pi, -np.e, 1e-40])
    assert np.array_equal(O.round_to_f32(x), x.astype(np.float32).astype(np.float64))


def test_silu_special_values():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(40.0) - 40.0) < 1e-12           # silu(x) -> x for large x
    assert abs(O.silu(-40.0)) < 1e-15                 # silu(x) -> 0 for very negative x
    assert O.silu(-800.0) == 0.0                      # no overflow blow-up
    # silu(x) - silu(-x) = x (since sigmoid(x) + sigmoid(-x) = 1)
    x = np.linspace(-5, 5, 11)
    assert np.allclose(O.silu(x) - O.silu(-x), x, atol=1e-14)


# ---------------------------------------------------------------- routing

def _brute_routing(ids, E):
    """pos(f) = start of expert e_f + #{f' < f : e_f' = e_f}, by counting."""
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    counts = [0] * E
    for v in flat:
        if v < E:
            counts[v] += 1
    starts = []
    s = 0
    for e in range(E):
        starts.append(s)
        s += counts[e]
    row_map = []
    for f, v in enumerate(flat):
        if v >= E:
            row_map.append(-1)
            continue
        earlier = sum(1 for g in range(f) if flat[g] == v)
        row_map.append(starts[v] + earlier)
    sorted_idx = [None] * s
    for f, p in enumerate(row_map):
        if p >= 0:
            sorted_idx[p] = f
    return sorted_idx, row_map, counts, starts + [s]


@pytest.mark.parametrize("T,K,E,special", [(1, 1, 1, 0), (5, 2, 4, 0), (8, 3, 6, 2), (7, 4, 9, 3)])
def test_permute_routing_brute_force(T, K, E, special):
    rng = np.random.default_rng(T * 100 + K)
    ids = _rand_ids(rng, T, K, E + special)
    si, rm, tpe, off = O.permute_routing(ids, E, special)
    b_si, b_rm, b_tpe, b_off = _brute_routing(ids, E)
    assert si.tolist() == b_si
    assert rm.tolist() == b_rm
    assert tpe.tolist() == b_tpe
    assert off.tolist() == b_off


def test_permute_routing_invariants_medium():
    rng = np.random.default_rng(7)
    T, K, E = 300, 8, 64
    ids = _rand_ids(rng, T, K, E)
    si, rm, tpe, off = O.permute_routing(ids, E)
    flat = ids.reshape(-1)
    assert tpe.sum() == T * K
    assert np.array_equal(np.sort(si), np.arange(T * K))          # a permutation
    assert np.all(np.diff(flat[si]) >= 0)                            # expert-major
    same = np.diff(flat[si]) == 0
    assert np.all(np.diff(si)[same] > 0)                             # stable inside an expert
    assert np.array_equal(rm[si], np.arange(T * K))                  # inverse maps
    assert np.array_equal(tpe, np.bincount(flat, minlength=E))       # library histogram


def test_permute_routing_page_example_with_special_ids():
    ids = np.array(_read_rows("combine_v2_example_expert_ids.txt"), dtype=np.int64)
    assert ids.shape == (8, 8)
    E = 32
    si, rm, tpe, off = O.permute_routing(ids, E, num_special=3)
    b_si, b_rm, b_tpe, b_off = _brute_routing(ids, E)
    assert si.tolist() == b_si and rm.tolist() == b_rm and tpe.tolist() == b_tpe
    specials = int((ids >= E).sum())
    assert specials == 4                       # three 33s and one 32 on the page
    assert tpe.sum() == 64 - specials
    assert np.all(rm[ids.reshape(-1) >= E] == -1)


def test_validate_rejects_bad_ids():
    with pytest.raises(ValueError):
        O.permute_routing(np.array([[1, 1]]), 4)            # repeated id in a row
    with pytest.raises(ValueError):
        O.permute_routing(np.array([[0, 4]]), 4)            # out of range
    with pytest.raises(ValueError):
        O.permute_routing(np.zeros((2, 17), dtype=np.int64), 64)   # K > 16
    O.permute_routing(np.array([[0, 4]]), 4, num_special=1)       # special id is legal


# ---------------------------------------------------------------- permute rows / unpermute

def test_permute_then_unpermute_k1_is_identity():
    rng = np.random.default_rng(3)
    T, H, E = 37, 16, 5
    ids = rng.integers(0, E, size=(T, 1))
    x = O.round_to_bf16(rng.standard_normal((T, H)))
    si, rm, tpe, off = O.permute_routing(ids, E)
    perm = O.permute_rows(x, si, 1)
    back = O.unpermute(perm, rm, np.ones((T, 1)), T, 1, "bf16")
    assert np.array_equal(back, x)
    back2 = O.unpermute(perm, rm, None, T, 1, "bf16")
    assert np.array_equal(back2, x)


def test_permuted_rows_are_exact_copies_of_the_source_token():
    rng = np.random.default_rng(4)
    T, K, E, H = 20, 3, 7, 8
    ids = _rand_ids(rng, T, K, E)
    x = rng.standard_normal((T, H))
    si, rm, tpe, off = O.permute_routing(ids, E)
    perm = O.permute_rows(x, si, K)
    for t in range(T):
        for k in range(K):
            assert np.array_equal(perm[rm[t * K + k]], x[t])


def test_unpermute_identical_rows_and_probs_summing_to_one():
    rng = np.random.default_rng(5)
    T, K, E, H = 9, 4, 6, 8
    ids = _rand_ids(rng, T, K, E)
    x = O.round_to_bf16(rng.standard_normal((T, H)))
    si, rm, tpe, off = O.permute_routing(ids, E)
    perm = O.permute_rows(x, si, K)                      # every slot carries its token's row
    p = np.full((T, K), 1.0 / K)                          # 1/4 is exact in binary
    out = O.unpermute(perm, rm, p, T, K, "f64")
    assert np.allclose(out, x, rtol=0, atol=1e-15)


def test_unpermute_is_linear_in_probs():
    rng = np.random.default_rng(6)
    T, K, E, H = 6, 2, 3, 5
    ids = _rand_ids(rng, T, K, E)
    si, rm, _, _ = O.permute_routing(ids, E)
    y = rng.standard_normal((T * K, H))
    p1, p2 = rng.random((T, K)), rng.random((T, K))
    a = O.unpermute(y, rm, p1 + 2 * p2, T, K, "f64")
    b = O.unpermute(y, rm, p1, T, K, "f64") + 2 * O.unpermute(y, rm, p2, T, K, "f64")
    assert np.allclose(a, b, atol=1e-13)


def test_unpermute_grad_finite_differences():
    rng = np.random.default_rng(8)
    T, K, E, H = 4, 2, 3, 8
    ids = _rand_ids(rng, T, K, E)
    si, rm, _, _ = O.permute_routing(ids, E)
    y = rng.standard_normal((T * K, H))
    p = rng.random((T, K))
    G = rng.standard_normal((T, H))

    def loss(yy, pp):
        return float(np.sum(O.unpermute(yy, rm, pp, T, K, "f64") * G))

    gy, gp = O.unpermute_grad(G, y, rm, p, T, K, "f64")
    eps = 1e-6
    for i in range(T * K):
        for h in range(0, H, 3):
            d = np.zeros_like(y)
            d[i, h] = eps
            fd = (loss(y + d, p) - loss(y - d, p)) / (2 * eps)
            assert abs(fd - gy[i, h]) < 1e-7
    for t in range(T):
        for k in range(K):
            d = np.zeros_like(p)
            d[t, k] = eps
            fd = (loss(y, p + d) - loss(y, p - d)) / (2 * eps)
            assert abs(fd - gp[t, k]) < 1e-5 * max(1.0, abs(fd))


def test_unpermute_grad_probs_is_sum_of_hidden_shards():
    """The probs grad is 'Partial' under hidden-dim sharding: the sum of the
    per-shard results equals the unsharded result."""
    rng = np.random.default_rng(9)
    T, K, E, H = 5, 3, 4, 12
    ids = _rand_ids(rng, T, K, E)
    _, rm, _, _ = O.permute_routing(ids, E)
    y = rng.standard_normal((T * K, H))
    G = rng.standard_normal((T, H))
    p = rng.random((T, K))
    full = O.unpermute_grad(G, y, rm, p, T, K, "f64")[1]
    parts = sum(O.unpermute_grad(G[:, s], y[:, s], rm, p, T, K, "f64")[1]
                for s in (slice(0, 4), slice(4, 9), slice(9, 12)))
    assert np.allclose(full, parts, atol=1e-5)


def test_permute_grad_is_adjoint_of_permute():
    rng = np.random.default_rng(10)
    T, K, E, H = 11, 3, 5, 6
    ids = _rand_ids(rng, T, K, E)
    si, rm, _, _ = O.permute_routing(ids, E)
    x = rng.standard_normal((T, H))
    g = rng.standard_normal((T * K, H))
    lhs = np.sum(O.permute_rows(x, si, K) * g)
    rhs = np.sum(x * O.permute_grad(g, rm, T, K, "f64"))
    assert abs(lhs - rhs) < 1e-10


def test_unpermute_grad_is_adjoint_of_unpermute():
    rng = np.random.default_rng(11)
    T, K, E, H = 7, 2, 4, 5
    ids = _rand_ids(rng, T, K, E)
    _, rm, _, _ = O.permute_routing(ids, E)
    y = rng.standard_normal((T * K, H))
    p = rng.random((T, K))
    G = rng.standard_normal((T, H))
    lhs = np.sum(O.unpermute(y, rm, p, T, K, "f64") * G)
    rhs = np.sum(y * O.unpermute_grad(G, y, rm, p, T, K, "f64")[0])
    assert abs(lhs - rhs) < 1e-10


# ---------------------------------------------------------------- expert MLP

def test_expert_mlp_single_expert_is_dense_swiglu_via_torch():
    rng = np.random.default_rng(12)
    M, H, I = 10, 12, 6
    X = rng.standard_normal((M, H))
    Wg, Wu = rng.standard_normal((1, I, H)), rng.standard_normal((1, I, H))
    Wd = rng.standard_normal((1, H, I))
    act, out, g, u = O.expert_mlp(X, np.array([0, M]), Wg, Wu, Wd, "f64")
    tX = torch.from_numpy(X)
    tg = tX @ torch.from_numpy(Wg[0]).T
    tu = tX @ torch.from_numpy(Wu[0]).T
    tact = torch.nn.functional.silu(tg) * tu
    tout = tact @ torch.from_numpy(Wd[0]).T
    assert np.allclose(act, tact.numpy(), atol=1e-12)
    assert np.allclose(out, tout.numpy(), atol=1e-11)


def test_expert_mlp_naive_loops_and_empty_experts():
    rng = np.random.default_rng(13)
    H, I, E = 4, 3, 4
    off = np.array([0, 2, 2, 5, 5])        # experts 1 and 3 are empty
    N = 5
    X = rng.standard_normal((N, H))
    Wg, Wu = rng.standard_normal((E, I, H)), rng.standard_normal((E, I, H))
    Wd = rng.standard_normal((E, H, I))
    act, out, _, _ = O.expert_mlp(X, off, Wg, Wu, Wd, "f64")
    expert_of_row = [0, 0, 2, 2, 2]
    for i in range(N):
        e = expert_of_row[i]
        a = []
        for j in range(I):
            gj = sum(X[i, h] * Wg[e, j, h] for h in range(H))
            uj = sum(X[i, h] * Wu[e, j, h] for h in range(H))
            a.append(gj / (1.0 + np.exp(-gj)) * uj)
        for h in range(H):
            y = sum(a[j] * Wd[e, h, j] for j in range(I))
            assert abs(out[i, h] - y) < 1e-12
        assert np.allclose(act[i], a, atol=1e-13)


def test_expert_mlp_rows_past_last_offset_stay_zero():
    rng = np.random.default_rng(14)
    X = rng.standard_normal((6, 4))
    W = rng.standard_normal((2, 3, 4))
    act, out, _, _ = O.expert_mlp(X, np.array([0, 2, 4]), W, W, rng.standard_normal((2, 4, 3)), "f64")
    assert not act[4:].any() and not out[4:].any()


def test_expert_mlp_grad_finite_differences():
    rng = np.random.default_rng(15)
    H, I, E = 5, 4, 3
    off = np.array([0, 3, 3, 7])            # expert 1 empty
    N = 7
    X = rng.standard_normal((N, H))
    Wg, Wu = rng.standard_normal((E, I, H)) * 0.5, rng.standard_normal((E, I, H)) * 0.5
    Wd = rng.standard_normal((E, H, I)) * 0.5
    G = rng.standard_normal((N, H))

    def loss(X_, Wg_, Wu_, Wd_):
        return float(np.sum(O.expert_mlp(X_, off, Wg_, Wu_, Wd_, "f64")[1] * G))

    act = O.expert_mlp(X, off, Wg, Wu, Wd, "f64")[0]
    dX, dWg, dWu, dWd = O.expert_mlp_grad(G, X, act, off, Wg, Wu, Wd, "f64")
    eps = 1e-6

    def fd(which, idx):
        args = [X, Wg, Wu, Wd]
        plus = [a.copy() for a in args]
        minus = [a.copy() for a in args]
        plus[which][idx] += eps
        minus[which][idx] -= eps
        return (loss(*plus) - loss(*minus)) / (2 * eps)

    for idx in [(0, 0), (2, 4), (5, 1), (6, 3)]:
        assert abs(fd(0, idx) - dX[idx]) < 1e-6
    for idx in [(0, 1, 2), (2, 3, 4), (1, 0, 0)]:
        assert abs(fd(1, idx) - dWg[idx]) < 1e-6
        assert abs(fd(2, idx) - dWu[idx]) < 1e-6
    for idx in [(0, 4, 3), (2, 1, 0), (1, 2, 2)]:
        assert abs(fd(3, idx) - dWd[idx]) < 1e-6
    assert not dWg[1].any() and not dWu[1].any() and not dWd[1].any()


def test_full_layer_gradient_chain_finite_differences():
    """loss = <unpermute(mlp(permute(x))), G>; its x-grad through
    unpermute_grad -> expert_mlp_grad -> permute_grad matches FD."""
    rng = np.random.default_rng(16)
    T, K, E, H, I = 5, 2, 3, 4, 3
    ids = _rand_ids(rng, T, K, E)
    si, rm, tpe, off = O.permute_routing(ids, E)
    x = rng.standard_normal((T, H))
    p = rng.random((T, K))
    Wg, Wu = rng.standard_normal((E, I, H)), rng.standard_normal((E, I, H))
    Wd = rng.standard_normal((E, H, I))
    G = rng.standard_normal((T, H))

    def fwd(x_, p_):
        perm = O.permute_rows(x_, si, K)
        act, y, _, _ = O.expert_mlp(perm, off, Wg, Wu, Wd, "f64")
        return perm, act, y, O.unpermute(y, rm, p_, T, K, "f64")

    perm, act, y, out = fwd(x, p)
    gy, gp = O.unpermute_grad(G, y, rm, p, T, K, "f64")
    dperm = O.expert_mlp_grad(gy, perm, act, off, Wg, Wu, Wd, "f64")[0]
    gx = O.permute_grad(dperm, rm, T, K, "f64")
    eps = 1e-6
    for t in range(T):
        for h in range(H):
            d = np.zeros_like(x)
            d[t, h] = eps
            fdv = (np.sum(fwd(x + d, p)[3] * G) - np.sum(fwd(x - d, p)[3] * G)) / (2 * eps)
            assert abs(fdv - gx[t, h]) < 1e-6 * max(1, abs(fdv))


# ---------------------------------------------------------------- combine

def _combine_setup(rng, T, K, E, Z, C, Cn, H):
    ids = _rand_ids(rng, T, K, E + Z + C + Cn)
    si, rm, tpe, off = O.permute_routing(ids, E, Z + C + Cn)
    Y = rng.standard_normal((len(si), H))
    return ids, rm, Y


def test_combine_without_specials_equals_unpermute():
    rng = np.random.default_rng(17)
    T, K, E, H = 12, 3, 6, 8
    ids, rm, Y = _combine_setup(rng, T, K, E, 0, 0, 0, H)
    s = rng.random((T, K))
    a = O.combine(Y, rm, ids, s, None, None, E, 0, 0, 0, None, None, None, "f64")
    b = O.unpermute(Y, rm, s, T, K, "f64")
    assert np.allclose(a, b, atol=1e-14)


def test_combine_special_expert_closed_forms():
    """zero expert -> 0, copy expert -> ori_x, const expert -> a1*ori_x + a2*v,
    each checked through a case where the closed form is known."""
    H, E, Z, C, Cn = 6, 4, 1, 1, 2
    zero_id, copy_id, c0, c1 = E, E + 1, E + 2, E + 3
    rng = np.random.default_rng(18)
    ori = rng.standard_normal((3, H))
    shared = rng.standard_normal((3, H))
    v = rng.standard_normal((Cn, H))
    a1 = np.stack([np.ones(H), np.zeros(H)])      # const 0 acts like a copy expert
    a2 = np.stack([np.zeros(H), np.ones(H)])      # const 1 returns v[1]
    ids = np.array([[zero_id, copy_id], [copy_id, c0], [c1, zero_id]])
    s = np.array([[0.3, 0.7], [0.25, 0.75], [0.5, 0.5]])
    Y = np.zeros((0, H))
    rm = -np.ones(6, dtype=np.int64)
    out = O.combine(Y, rm, ids, s, shared, ori, E, Z, C, Cn, a1, a2, v, "f64")
    assert np.allclose(out[0], 0.7 * ori[0] + shared[0], atol=1e-14)
    assert np.allclose(out[1], ori[1] + shared[1], atol=1e-14)        # 0.25 + 0.75 of copies
    assert np.allclose(out[2], 0.5 * v[1] + shared[2], atol=1e-14)
    # without shared_x, a token routed only to zero experts combines to 0
    out0 = O.combine(Y, rm[:1], np.array([[zero_id]]), np.array([[0.9]]), None, ori[:1], E, Z, C, Cn,
                     a1, a2, v, "f64")
    assert not out0.any()


def test_combine_const_expert_with_v_equal_ori_x():
    """With v = ori_x and a1 + a2 = 1 the const expert returns ori_x."""
    rng = np.random.default_rng(19)
    H, E = 5, 3
    ori = rng.standard_normal((1, H))
    a1 = rng.random((1, H))
    a2 = 1.0 - a1
    out = O.combine(np.zeros((0, H)), -np.ones(1, dtype=np.int64), np.array([[E]]), np.array([[1.0]]),
                    None, ori, E, 0, 0, 1, a1, a2, ori.copy(), "f64")
    assert np.allclose(out, ori, atol=1e-15)


def test_combine_page_example_ids():
    """The 8x8 ids of the combine_v2 example (ids 32 zero, 33 copy) against
    a brute force written from the closed forms and the routed rows."""
    ids = np.array(_read_rows("combine_v2_example_expert_ids.txt"), dtype=np.int64)
    T, K = ids.shape
    E, H = 32, 16
    rng = np.random.default_rng(20)
    si, rm, tpe, off = O.permute_routing(ids, E, 3)
    Y = rng.standard_normal((len(si), H))
    s = rng.random((T, K))
    ori = rng.standard_normal((T, H))
    shared = rng.standard_normal((T, H))
    a1, a2, v = rng.random((1, H)), rng.random((1, H)), rng.standard_normal((1, H))
    out = O.combine(Y, rm, ids, s, shared, ori, E, 1, 1, 1, a1, a2, v, "f64")
    flat = ids.reshape(-1)
    for t in range(T):
        want = shared[t].copy()
        for k in range(K):
            e = flat[t * K + k]
            if e == 33:
                want += s[t, k] * ori[t]
            elif e < 32:
                # the routed row: the one whose sorted index is this slot
                want += s[t, k] * Y[list(si).index(t * K + k)]
        assert np.allclose(out[t], want, atol=1e-13)


def test_combine_rejects_ids_past_special_ranges():
    with pytest.raises(ValueError):
        O.combine(np.zeros((0, 2)), -np.ones(1, dtype=np.int64), np.array([[5]]), np.ones((1, 1)),
                  None, np.zeros((1, 2)), 3, 1, 1, 0, None, None, None, "f64")


# ---------------------------------------------------------------- permute indices

def test_permute_indices_docstring_case():
    rows = _read_rows("permute_indices_docstring_case.txt")
    (R, E), counts, want, want_tpe = rows
    idx, tpe, total = O.permute_indices(np.array(counts), R, E)
    assert idx.tolist() == want and tpe.tolist() == want_tpe and total == len(want)


def _brute_permute_indices(counts, R, E):
    """Label each rank-major source position with its (e, r) block and stable
    sort by (e, r): destination i holds the i-th source position in that
    order."""
    labels = []
    for r in range(R):
        for e in range(E):
            labels += [(e, r)] * int(counts[r * E + e])
    return sorted(range(len(labels)), key=lambda p: labels[p])


@pytest.mark.parametrize("R,E", [(1, 1), (1, 5), (4, 1), (3, 4), (16, 16)])
def test_permute_indices_brute_force(R, E):
    rng = np.random.default_rng(R * 31 + E)
    counts = rng.poisson(3.0, size=R * E)
    idx, tpe, total = O.permute_indices(counts, R, E)
    assert idx.tolist() == _brute_permute_indices(counts, R, E)
    assert tpe.tolist() == counts.reshape(R, E).sum(axis=0).tolist()
    assert total == counts.sum()
    assert np.array_equal(np.sort(idx), np.arange(total))
    if R == 1 or E == 1:
        assert np.array_equal(idx, np.arange(total))      # nothing to reorder


def test_permute_indices_empty():
    idx, tpe, total = O.permute_indices(np.zeros(6, dtype=np.int64), 2, 3)
    assert total == 0 and idx.shape == (0,) and not tpe.any()


# ---------------------------------------------------------------- input generators

def test_input_generators_shapes_and_routing_rules():
    d = moe_inputs.layer_forward_zipf(0, T=512, H=64, E=64, K=8, I=32, num_empty=8)
    ids = d["expert_ids"].numpy()
    O.validate_expert_ids(ids, 64)
    counts = np.bincount(ids.reshape(-1), minlength=64)
    assert (counts == 0).sum() >= 8
    p = d["probs"].numpy()
    assert np.allclose(p.sum(1), 1.0, atol=1e-6)
    d2 = moe_inputs.index_combine(0, R=2, E_local=2, T=16, H=32, K=4)
    assert d2["expanded"].shape[0] == int((d2["expert_ids"] < d2["E"]).sum())
    a = moe_inputs.permute_unpermute(3, T=8, H=16, E=8, K=2)
    b = moe_inputs.permute_unpermute(3, T=8, H=16, E=8, K=2)
    assert torch.equal(a["tokens"], b["tokens"]) and torch.equal(a["expert_ids"], b["expert_ids"])


# ---------------------------------------------------------------- deredundancy indices

def test_deredundancy_indices_docstring_case():
    (nsrc, NE, s, D, L), counts, want, want_n = _read_rows("deredundancy_indices_case.txt")
    idx, n, total = O.deredundancy_dispatch_indices(np.array(counts).reshape(nsrc, NE), s, D, L)
    assert idx.tolist() == want and n.tolist() == want_n and total == len(want)


def _brute_deredundancy(counts, start, D, L):
    """Label every source row with (d, l, o) if its expert is in the range,
    then stable-sort the labelled rows by that key."""
    nsrc, NE = counts.shape
    labels = []
    pos = 0
    for o in range(nsrc):
        for e in range(NE):
            for _ in range(int(counts[o, e])):
                if start <= e < start + D * L:
                    d, l = divmod(e - start, L)
                    labels.append(((d, l, o), pos))
                pos += 1
    return [p for _, p in sorted(labels, key=lambda kv: kv[0])]


@pytest.mark.parametrize("nsrc,NE,start,D,L", [(1, 1, 0, 1, 1), (3, 8, 2, 2, 3), (4, 16, 0, 4, 4),
                                               (8, 32, 16, 4, 4), (2, 5, 4, 1, 1)])
def test_deredundancy_indices_brute_force(nsrc, NE, start, D, L):
    rng = np.random.default_rng(nsrc * 7 + NE)
    counts = rng.poisson(2.0, size=(nsrc, NE))
    idx, n, total = O.deredundancy_dispatch_indices(counts, start, D, L)
    assert idx.tolist() == _brute_deredundancy(counts, start, D, L)
    assert n.tolist() == [int(counts[:, start + j].sum()) for j in range(D * L)]
    assert total == len(idx)


def test_deredundancy_full_range_is_the_rank_to_expert_permutation():
    """With the whole expert range the deredundancy order (expert, source)
    is the rank-major -> expert-major permutation of the same counts."""
    rng = np.random.default_rng(5)
    counts = rng.poisson(3.0, size=(4, 6))
    a, na, ta = O.deredundancy_dispatch_indices(counts, 0, 2, 3)
    b, nb, tb = O.permute_indices(counts.reshape(-1), 4, 6)
    assert a.tolist() == b.tolist() and na.tolist() == nb.tolist() and ta == tb


# ---------------------------------------------------------------- activity mask

def test_masked_routing_brute_force_and_token_mask_broadcast():
    rng = np.random.default_rng(21)
    T, K, E = 9, 3, 5
    ids = _rand_ids(rng, T, K, E + 1)
    mask = rng.random((T, K)) < 0.6
    si, rm, tpe, off = O.permute_routing(ids, E, 1, active_mask=mask)
    # brute force: a masked slot is treated like a slot of a non-dispatched id
    hidden = ids.copy()
    hidden[~mask] = -1
    flat = [int(v) for v in hidden.reshape(-1)]
    counts = [sum(1 for v in flat if v == e) for e in range(E)]
    assert tpe.tolist() == counts
    for f, v in enumerate(flat):
        if 0 <= v < E:
            assert rm[f] == off[v] + sum(1 for g in range(f) if flat[g] == v)
        else:
            assert rm[f] == -1
    tok_mask = rng.random(T) < 0.5
    a = O.permute_routing(ids, E, 1, active_mask=tok_mask)
    b = O.permute_routing(ids, E, 1, active_mask=np.repeat(tok_mask[:, None], K, axis=1))
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_masked_combine_equals_zero_scale():
    """A slot masked off contributes what a slot of scale 0 contributes."""
    rng = np.random.default_rng(22)
    T, K, E, H = 6, 3, 4, 8
    ids = _rand_ids(rng, T, K, E + 3)
    si, rm, _, _ = O.permute_routing(ids, E, 3)
    Y = rng.standard_normal((len(si), H))
    s = rng.random((T, K))
    ori, sh = rng.standard_normal((T, H)), rng.standard_normal((T, H))
    a1, a2, v = rng.random((1, H)), rng.random((1, H)), rng.standard_normal((1, H))
    mask = rng.random((T, K)) < 0.5
    got = O.combine(Y, rm, ids, s, sh, ori, E, 1, 1, 1, a1, a2, v, "f64", active_mask=mask)
    want = O.combine(Y, rm, ids, np.where(mask, s, 0.0), sh, ori, E, 1, 1, 1, a1, a2, v, "f64")
    assert np.allclose(got, want, atol=1e-14)


# ---------------------------------------------------------------- bf16 storage rounding of the MLP

def _tbf16(t):
    """torch's own float32 -> bfloat16 conversion (round to nearest even),
    back to float64: an implementation of the storage rounding that shares
    nothing with the oracle's round_to_bf16."""
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def _mlp_case(seed, E=3, H=16, I=24, rows=(5, 0, 9)):
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(rows)])
    X = O.round_to_bf16(rng.standard_normal((int(off[-1]), H)))
    Wg = O.round_to_bf16(rng.standard_normal((E, I, H)) * 0.3)
    Wu = O.round_to_bf16(rng.standard_normal((E, I, H)) * 0.3)
    Wd = O.round_to_bf16(rng.standard_normal((E, H, I)) * 0.3)
    return off, X, Wg, Wu, Wd


def test_expert_mlp_bf16_rounds_exactly_act_and_expanded():
    """The "bf16" branch of expert_mlp rounds the stored tensors, act before
    the down projection and the expanded output, and nothing else (reading
    R7): a per-expert loop in torch float64 that rounds with torch's bf16
    conversion at those two points gives the same bits.  Dropping the act
    rounding changes the output, so the pin sees that rounding point."""
    off, X, Wg, Wu, Wd = _mlp_case(21)
    act, out, g, u = O.expert_mlp(X, off, Wg, Wu, Wd, "bf16")
    tX = torch.from_numpy(X)
    for e in range(len(off) - 1):
        lo, hi = int(off[e]), int(off[e + 1])
        if lo == hi:
            continue
        tg = tX[lo:hi] @ torch.from_numpy(Wg[e]).T
        tu = tX[lo:hi] @ torch.from_numpy(Wu[e]).T
        ta = _tbf16(torch.nn.functional.silu(tg) * tu)
        ty = _tbf16(ta @ torch.from_numpy(Wd[e]).T)
        assert np.array_equal(act[lo:hi], ta.numpy())
        assert np.array_equal(out[lo:hi], ty.numpy())
        assert np.allclose(g[lo:hi], tg.numpy(), rtol=1e-14, atol=0)     # unrounded
        unrounded_act = _tbf16((torch.nn.functional.silu(tg) * tu) @ torch.from_numpy(Wd[e]).T)
        assert not np.array_equal(out[lo:hi], unrounded_act.numpy())


def test_expert_mlp_grad_bf16_rounds_exactly_the_stored_gradients():
    """The "bf16" branch of expert_mlp_grad rounds dg and du (stored between
    the down dgrad and the gate/up GEMMs), d_permuted and the three weight
    gradients, and nothing else: the same chain rule in torch float64 with
    torch's bf16 conversion at those points gives the same bits.  Feeding the
    unrounded dg, du to the gate/up dgrad changes d_permuted, so the pin sees
    that rounding point."""
    off, X, Wg, Wu, Wd = _mlp_case(22)
    rng = np.random.default_rng(23)
    act, _, _, _ = O.expert_mlp(X, off, Wg, Wu, Wd, "bf16")
    dY = O.round_to_bf16(rng.standard_normal((X.shape[0], X.shape[1])))
    dX, dWg, dWu, dWd = O.expert_mlp_grad(dY, X, act, off, Wg, Wu, Wd, "bf16")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
    for e in range(len(off) - 1):
        lo, hi = int(off[e]), int(off[e + 1])
        if lo == hi:
            assert not dWg[e].any() and not dWu[e].any() and not dWd[e].any()
            continue
        x, dy, a = t(X[lo:hi]), t(dY[lo:hi]), t(act[lo:hi])
        g, u = x @ t(Wg[e]).T, x @ t(Wu[e]).T
        s = torch.sigmoid(g)
        dA = dy @ t(Wd[e])
        dg_raw = dA * u * s * (1 + g * (1 - s))
        du_raw = dA * torch.nn.functional.silu(g)
        dg, du = _tbf16(dg_raw), _tbf16(du_raw)
        assert np.array_equal(dX[lo:hi], _tbf16(dg @ t(Wg[e]) + du @ t(Wu[e])).numpy())
        assert np.array_equal(dWd[e], _tbf16(dy.T @ a).numpy())
        assert np.array_equal(dWg[e], _tbf16(dg.T @ x).numpy())
        assert np.array_equal(dWu[e], _tbf16(du.T @ x).numpy())
        unrounded = _tbf16(dg_raw @ t(Wg[e]) + du_raw @ t(Wu[e])).numpy()
        assert not np.array_equal(dX[lo:hi], unrounded)


# ---------------------------------------------------------------- whiteboard combine

def test_whiteboard_combine_hand_case():
    """Three dispatched rows of a five-row gathered buffer, worked by hand:
    row i of the expert outputs is scaled by the coefficient of gathered row
    d[i] and lands at row d[i]; the other rows stay zero."""
    rows = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])
    d = np.array([4, 0, 2])
    coeff = np.array([0.5, 9.0, -1.0, 9.0, 2.0])        # per gathered row
    want = np.array([[1.5, 2.0], [0.0, 0.0], [-5.0, -6.0], [0.0, 0.0], [2.0, 4.0]])
    assert np.array_equal(O.whiteboard_combine(rows, d, coeff, 5, "f64"), want)
    assert np.array_equal(O.whiteboard_combine(rows, d, None, 5, "f64")[4], [1.0, 2.0])


def test_scatter_add_first_dim_accumulates_repeated_rows():
    src = np.array([[1.0], [2.0], [4.0], [8.0]])
    got = O.scatter_add_first_dim(src, np.array([1, 3, 1, 1]), 4)
    assert np.array_equal(got, [[0.0], [13.0], [0.0], [2.0]])


def test_scale_by_router_coeff_rules():
    rows = np.arange(6.0).reshape(3, 2)
    assert np.array_equal(O.scale_by_router_coeff(rows, None), rows)
    assert np.array_equal(O.scale_by_router_coeff(rows, [1.0, -2.0, 0.5]),
                          [[0.0, 1.0], [-4.0, -6.0], [2.0, 2.5]])
    with pytest.raises(ValueError):
        O.scale_by_router_coeff(rows, [1.0, 2.0])


def test_whiteboard_combine_on_dispatch_indices_is_the_k1_unpermute():
    """On the deredundancy dispatch indices (distinct rows of the gathered
    buffer) the scatter-add whiteboard equals the weighted gather of the
    unpermute with one slot per gathered row, weight = its coefficient and
    row_map = the inverse of the dispatch indices (-1 for rows not
    dispatched)."""
    rng = np.random.default_rng(24)
    counts = rng.poisson(3.0, size=(4, 12))
    idx, _, n = O.deredundancy_dispatch_indices(counts, 4, 2, 3)
    total = int(counts.sum())
    Y = rng.standard_normal((n, 5))
    coeff = rng.random(total)
    wb = O.whiteboard_combine(Y, idx, coeff, total, "f64")
    rm = np.full(total, -1)
    rm[idx] = np.arange(n)
    assert np.allclose(wb, O.unpermute(Y, rm, coeff.reshape(total, 1), total, 1, "f64"), atol=0)
