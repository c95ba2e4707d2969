"""Plain CPU oracle of the single-GPU MoE expert layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, helpers, tables or
constant generators) and imports nothing from it.

Every function is the plain definition of one step, written for a reader who
checks it against the source pages by eye: numpy, float64 arithmetic, loops
where a loop is the definition, library primitives (a matmul, a stable sort,
a bincount) as single steps, and no blocking, fusion or reordering.

Sources (cited by page title and section):
  [EP]  hyper_parallel ``expert_parallel.py`` coverage page: the docstring and
        body of ``_generate_permute_indices``, ``_permute`` and ``_unpermute``.
  [CMB] torch_npu ``npu_moe_distribute_combine_v2`` API reference: the
        "function description" formulas (combine and special experts), the
        parameter list (``expert_ids``, ``expert_scales``,
        ``shared_expert_x``, ``ori_x``, ``const_expert_*``, special-expert id
        ranges) and the constraints section (K range).
  [UNP] Ascend/pytorch PR #42584 "Update moe token unpermute DTensor
        support", change summary: the sharding rules of
        ``npu_moe_token_unpermute`` and ``npu_moe_token_unpermute_grad_v2``
        (hidden-dim sharding of the tokens, ``Partial`` grad of the probs).
  [GMM] modelscope/twinkle PR #252 "NPU EP experts forward uses NPU grouped
        matmul", description: the per-expert loop replaced by grouped matmul
        + SwiGLU on stacked expert weights; ``permute`` as ``x[idx]`` whose
        backward accumulates duplicate indices.

Readings where the pages are silent:
  R1 unpermute forward = probability-weighted gather-sum over the K slots.
  R2 ``sorted_indices`` uses the gather convention of [EP]: entry i is the
     flat slot f = t*K + k whose row lands at permuted row i.
  R3 ties inside one expert keep increasing f (stable).
  R4 ``shared_expert_x`` is added once, after the weighted sum.
  R5 special-expert outputs are weighted by ``expert_scales`` like any expert.
  R6 ``const_expert_alpha_1/2`` and ``const_expert_v`` are [const_num, H] and
     act element-wise.
  R7 stored tensors (act, expanded, outputs, dgu, grads) are rounded once to
     the storage dtype; every sum before that is exact here (float64).
  R8 SwiGLU(g, u) = silu(g) * u with silu(x) = x * sigmoid(x).
  R9 special ids (>= E) are not dispatched: they get no permuted row and
     ``row_map`` = -1.
  R10 index dtype is int32 on the GPU; values equal the int64 of [EP].

parity pinned: every function below has a ``-m "not gpu"`` pin in
``tests/test_oracle_pins.py`` (brute force, closed forms, finite differences,
adjoint identities, library special cases); none is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "round_to_bf16",
    "round_to_f32",
    "round_to",
    "silu",
    "validate_expert_ids",
    "permute_routing",
    "permute_rows",
    "expert_mlp",
    "unpermute",
    "unpermute_grad",
    "combine",
    "permute_indices",
    "deredundancy_dispatch_indices",
    "scale_by_router_coeff",
    "scatter_add_first_dim",
    "whiteboard_combine",
    "permute_grad",
    "expert_mlp_grad",
]


# --------------------------------------------------------------------------
# Storage rounding (reading R7)
# --------------------------------------------------------------------------

def round_to_f32(x):
    """Round float64 values to the nearest float32 (IEEE ties-to-even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to_bf16(x):
    """Round to the nearest bfloat16, ties to even, returned as float64.

    bfloat16 keeps the upper 16 bits of an IEEE float32.  Rounding the low 16
    bits to nearest-even: add 0x7FFF plus the lowest kept bit, then clear the
    low half.  The input is first rounded to float32 (the GPU accumulates in
    float32 and stores bf16 from there).  Finite inputs only.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + keep_lsb) & np.uint64(0xFFFF0000)
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def round_to(x, dtype: str):
    """Round to the storage dtype: "bf16", "f32", or "f64" (no rounding)."""
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f32":
        return round_to_f32(x)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def silu(x):
    """silu(x) = x * sigmoid(x) = x / (1 + exp(-x))  (reading R8)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def _sigmoid(x):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


# --------------------------------------------------------------------------
# Step a1-a3: routing (histogram, scan, stable expert-major rank)
# --------------------------------------------------------------------------

def validate_expert_ids(expert_ids, num_experts: int, num_special: int = 0):
    """Check the id rules of [CMB] parameter ``expert_ids`` and constraints.

    Values lie in [0, E + num_special) and the K ids of one row are distinct;
    0 < K <= 16 and K <= E + num_special.  Raises ValueError otherwise.
    """
    ids = np.asarray(expert_ids)
    if ids.ndim != 2:
        raise ValueError("expert_ids must be [T, K]")
    T, K = ids.shape
    total = num_experts + num_special
    if not (0 < K <= 16) or K > total:
        raise ValueError(f"K={K} outside (0, min(16, {total})]")
    if ids.size and (ids.min() < 0 or ids.max() >= total):
        raise ValueError("expert id out of range")
    for t in range(T):
        if len(set(ids[t].tolist())) != K:
            raise ValueError(f"row {t} repeats an expert id")


def _active(active_mask, T: int, K: int):
    """[CMB] ``x_active_mask``: [T] per token or [T, K] per slot; None = all
    active.  Returns a flat [T*K] bool array."""
    if active_mask is None:
        return np.ones(T * K, dtype=bool)
    m = np.asarray(active_mask).astype(bool)
    if m.shape == (T,):
        m = np.repeat(m, K)
    elif m.shape != (T, K):
        raise ValueError("active mask must be [T] or [T, K]")
    return m.reshape(-1)


def permute_routing(expert_ids, num_experts: int, num_special: int = 0, active_mask=None):
    """Expert-major routing of the T*K slots ([EP] ``_generate_permute_indices``
    docstring: the expert-major buffer holds all rows of expert 0, then all of
    expert 1, ...; readings R2, R3, R9).

    Returns (sorted_indices[N], row_map[T*K], tokens_per_expert[E],
    expert_offsets[E+1]) as int64, with N = number of slots whose id < E.
      tokens_per_expert[e] = #{f : id_f == e}
      expert_offsets       = exclusive prefix sum of tokens_per_expert
      sorted_indices       = stable argsort of the flat ids (dispatched slots)
      row_map[f]           = position of slot f in the permuted buffer, or -1
    A slot masked off by ``active_mask`` ([CMB] ``x_active_mask``) takes no
    part: it is not dispatched.
    """
    validate_expert_ids(expert_ids, num_experts, num_special)
    T, K = np.asarray(expert_ids).shape
    flat = np.asarray(expert_ids, dtype=np.int64).reshape(-1)
    dispatched = np.nonzero((flat < num_experts) & _active(active_mask, T, K))[0]
    order = np.argsort(flat[dispatched], kind="stable")
    sorted_indices = dispatched[order].astype(np.int64)
    tokens_per_expert = np.bincount(flat[dispatched], minlength=num_experts).astype(np.int64)
    expert_offsets = np.zeros(num_experts + 1, dtype=np.int64)
    expert_offsets[1:] = np.cumsum(tokens_per_expert)
    row_map = np.full(flat.shape[0], -1, dtype=np.int64)
    row_map[sorted_indices] = np.arange(sorted_indices.shape[0], dtype=np.int64)
    return sorted_indices, row_map, tokens_per_expert, expert_offsets


def permute_rows(tokens, sorted_indices, K: int):
    """Step a4: ``permuted[i] = tokens[sorted_indices[i] // K]`` — the row
    gather ``x[permuted_indices]`` of [EP] ``_permute`` and of [GMM]'s
    ``permute`` fix.  An exact copy (no arithmetic)."""
    tokens = np.asarray(tokens)
    idx = np.asarray(sorted_indices, dtype=np.int64)
    return tokens[idx // K]


# --------------------------------------------------------------------------
# Steps a5-a6: expert MLP (the per-expert loop that [GMM] replaces)
# --------------------------------------------------------------------------

def expert_mlp(permuted, expert_offsets, W_gate, W_up, W_down, dtype: str):
    """Per-expert SwiGLU MLP over the expert-major rows ([GMM]; R7, R8).

    For rows X_e = permuted[off[e]:off[e+1]]:
        g = X_e @ W_gate[e]^T,  u = X_e @ W_up[e]^T           ([M_e, I])
        act_e = round(silu(g) * u)                            (stored tensor)
        expanded_e = round(act_e @ W_down[e]^T)               ([M_e, H])
    Weights are [E, I, H] (gate, up) and [E, H, I] (down), nn.Linear style.
    Rows at or past off[E] are left zero.
    Returns (act[N, I], expanded[N, H], gate[N, I], up[N, I]) in float64;
    gate/up are the unrounded pre-activations.
    """
    X = np.asarray(permuted, dtype=np.float64)
    Wg = np.asarray(W_gate, dtype=np.float64)
    Wu = np.asarray(W_up, dtype=np.float64)
    Wd = np.asarray(W_down, dtype=np.float64)
    off = np.asarray(expert_offsets, dtype=np.int64)
    N = X.shape[0]
    E, I, H = Wg.shape
    act = np.zeros((N, I))
    expanded = np.zeros((N, H))
    gate = np.zeros((N, I))
    up = np.zeros((N, I))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        Xe = X[lo:hi]
        g = Xe @ Wg[e].T
        u = Xe @ Wu[e].T
        a = round_to(silu(g) * u, dtype)
        gate[lo:hi] = g
        up[lo:hi] = u
        act[lo:hi] = a
        expanded[lo:hi] = round_to(a @ Wd[e].T, dtype)
    return act, expanded, gate, up


# --------------------------------------------------------------------------
# Step a7: unpermute forward;  a8: unpermute backward
# --------------------------------------------------------------------------

def unpermute(expanded, row_map, probs, T: int, K: int, dtype: str):
    """out[t] = round( sum_{k=0..K-1} probs[t,k] * expanded[row_map[t*K+k]] )

    Reading R1: the weighted gather-sum that inverts [EP] ``_unpermute``'s
    scatter and matches [CMB]'s ``Sum(expert_scales * ata_out)``.  ``probs``
    None means weight 1 (the plain inverse permutation).  Slots with
    row_map = -1 contribute nothing.
    """
    Y = np.asarray(expanded, dtype=np.float64)
    rm = np.asarray(row_map, dtype=np.int64).reshape(T, K)
    H = Y.shape[1]
    out = np.zeros((T, H))
    for k in range(K):
        rows = rm[:, k]
        live = rows >= 0
        w = np.ones(T) if probs is None else np.asarray(probs, dtype=np.float64).reshape(T, K)[:, k]
        contrib = np.zeros((T, H))
        contrib[live] = w[live, None] * Y[rows[live]]
        out += contrib
    return round_to(out, dtype)


def unpermute_grad(grad_out, permuted_tokens, row_map, probs, T: int, K: int, dtype: str):
    """Backward of :func:`unpermute` ([UNP]: the tokens' grad shards on the
    hidden dim like the tokens, the probs' grad is ``Partial`` i.e. a sum of
    per-hidden-column terms).

        grad_permuted[row_map[f]] = round(probs[f] * grad_out[t])
        grad_probs[t, k]          = round_f32( sum_h permuted_tokens[row_map[f], h] * grad_out[t, h] )

    with f = t*K + k.  Rows of grad_permuted no slot maps to stay zero;
    grad_probs of an undispatched slot (row_map = -1) is 0.
    """
    G = np.asarray(grad_out, dtype=np.float64)
    P = np.asarray(permuted_tokens, dtype=np.float64)
    rm = np.asarray(row_map, dtype=np.int64).reshape(T, K)
    pr = np.ones((T, K)) if probs is None else np.asarray(probs, dtype=np.float64).reshape(T, K)
    grad_permuted = np.zeros_like(P)
    grad_probs = np.zeros((T, K))
    for k in range(K):
        rows = rm[:, k]
        live = rows >= 0
        grad_permuted[rows[live]] = pr[live, k, None] * G[live]
        grad_probs[live, k] = np.sum(P[rows[live]] * G[live], axis=1)
    return round_to(grad_permuted, dtype), round_to_f32(grad_probs)


# --------------------------------------------------------------------------
# Step a9: combine with shared expert and zero / copy / const experts
# --------------------------------------------------------------------------

def combine(expanded, row_map, expert_ids, scales, shared_x, ori_x, num_experts: int,
            zero_num: int, copy_num: int, const_num: int,
            alpha1, alpha2, const_v, dtype: str, active_mask=None):
    """[CMB] function description: x = Sum_k(expert_scales * y_k) + shared_expert_x,

    where y_k, the expert output for slot (t, k) with id e, is
      e <  E                 : expanded[row_map[t*K+k]]          (routed expert)
      E <= e < E+Z           : 0                                  (zero expert)
      E+Z <= e < E+Z+C       : ori_x[t]                           (copy expert)
      E+Z+C <= e < E+Z+C+Cn  : alpha1[j]*ori_x[t] + alpha2[j]*v[j], j = e-E-Z-C
                                                                  (const expert)
    The id ranges follow [CMB] ``zero_expert_num`` / ``copy_expert_num`` /
    ``const_expert_num``.  Readings R4, R5, R6.  shared_x None adds nothing.
    A slot masked off by ``active_mask`` ([CMB] ``x_active_mask``) adds
    nothing (reading R18); the shared term is still added.
    """
    ids = np.asarray(expert_ids, dtype=np.int64)
    T, K = ids.shape
    validate_expert_ids(ids, num_experts, zero_num + copy_num + const_num)
    Y = np.asarray(expanded, dtype=np.float64)
    H = Y.shape[1]
    rm = np.asarray(row_map, dtype=np.int64).reshape(T, K)
    s = np.asarray(scales, dtype=np.float64).reshape(T, K)
    ox = None if ori_x is None else np.asarray(ori_x, dtype=np.float64)
    a1 = None if alpha1 is None else np.asarray(alpha1, dtype=np.float64)
    a2 = None if alpha2 is None else np.asarray(alpha2, dtype=np.float64)
    cv = None if const_v is None else np.asarray(const_v, dtype=np.float64)
    zero_lo = num_experts
    copy_lo = zero_lo + zero_num
    const_lo = copy_lo + copy_num
    const_hi = const_lo + const_num
    act = _active(active_mask, T, K).reshape(T, K)
    x = np.zeros((T, H))
    for t in range(T):
        acc = np.zeros(H)
        for k in range(K):
            if not act[t, k]:
                continue
            e = ids[t, k]
            if e < zero_lo:
                y = Y[rm[t, k]]
            elif e < copy_lo:
                y = np.zeros(H)
            elif e < const_lo:
                y = ox[t]
            elif e < const_hi:
                j = e - const_lo
                y = a1[j] * ox[t] + a2[j] * cv[j]
            else:
                raise ValueError("expert id out of range")
            acc = acc + s[t, k] * y
        x[t] = acc
    if shared_x is not None:
        x = x + np.asarray(shared_x, dtype=np.float64).reshape(T, H)
    return round_to(x, dtype)


# --------------------------------------------------------------------------
# Step a10: rank-major -> expert-major permute indices
# --------------------------------------------------------------------------

def permute_indices(counts, num_ranks: int, experts_per_rank: int):
    """[EP] ``_generate_permute_indices``, as its docstring states it.

    ``counts[r*E + e]`` rows arrive from rank r for local expert e, laid out
    rank-major: block (r=0,e=0), (0,1), ..., (1,0), ...  The expert-major
    buffer visits blocks (e=0,r=0), (0,1), ..., (1,0), ...; the output entry
    for destination i is the rank-major source position of that row.
    Restated as a double loop: for e, for r, for j < counts[r*E+e], emit
    start_rm(r, e) + j, where start_rm is the exclusive prefix sum of counts
    in rank-major order.

    Returns (indices[total] int64, tokens_per_expert[E] int64, total int);
    total == 0 returns an empty index array.
    """
    R, E = int(num_ranks), int(experts_per_rank)
    c = np.asarray(counts, dtype=np.int64).reshape(-1)
    if c.shape[0] != R * E:
        raise ValueError("counts must have num_ranks * experts_per_rank entries")
    if c.size and c.min() < 0:
        raise ValueError("negative count")
    start_rm = np.zeros(R * E, dtype=np.int64)
    running = 0
    for b in range(R * E):
        start_rm[b] = running
        running += int(c[b])
    out = []
    for e in range(E):
        for r in range(R):
            s = int(start_rm[r * E + e])
            for j in range(int(c[r * E + e])):
                out.append(s + j)
    tokens_per_expert = np.array([sum(int(c[r * E + e]) for r in range(R)) for e in range(E)],
                                 dtype=np.int64)
    return np.array(out, dtype=np.int64), tokens_per_expert, len(out)


def deredundancy_dispatch_indices(counts, expert_start: int, iep_size: int,
                                  num_local_experts: int):
    """[EP] ``_generate_deredundency_dispatch_indices``.

    ``counts[o, e]`` rows of expert e sit in source o's expert-major buffer;
    the sources' buffers are concatenated (source 0 first), so block (o, e)
    starts after every block (o', e') that precedes it in (o, e) order.  The
    output selects the outer expert range [expert_start, expert_start +
    iep_size * num_local_experts) and orders its rows as [iep destination d,
    local expert l, source o] (expert e = expert_start + d * L + l), each
    block keeping its rows in order.  Also returns, per (d, l), the rows of
    that expert summed over the sources.
    """
    c = np.asarray(counts, dtype=np.int64)
    if c.ndim != 2:
        raise ValueError("counts must be [sources, experts]")
    O, NE = c.shape
    L, D = int(num_local_experts), int(iep_size)
    if expert_start < 0 or expert_start + D * L > NE:
        raise ValueError("expert range outside the experts")
    if c.size and c.min() < 0:
        raise ValueError("negative count")
    start = np.zeros((O, NE), dtype=np.int64)
    running = 0
    for o in range(O):
        for e in range(NE):
            start[o, e] = running
            running += int(c[o, e])
    out = []
    per_dest_expert = []
    for d in range(D):
        for l in range(L):
            e = expert_start + d * L + l
            n = 0
            for o in range(O):
                out.extend(range(int(start[o, e]), int(start[o, e] + c[o, e])))
                n += int(c[o, e])
            per_dest_expert.append(n)
    return np.array(out, dtype=np.int64), np.array(per_dest_expert, dtype=np.int64), len(out)


# --------------------------------------------------------------------------
# The deredundancy dispatcher's combine ([EP] _scale_by_router_coeff,
# _scatter_add_first_dim and the combine that calls them)
# --------------------------------------------------------------------------

def scale_by_router_coeff(rows, router_coeff):
    """[EP] ``_scale_by_router_coeff``: each routed expert-output row times
    its own router coefficient; no coefficients leave the rows unchanged.
    The coefficient vector must have one entry per row (ValueError
    otherwise)."""
    Y = np.asarray(rows, dtype=np.float64)
    if router_coeff is None:
        return Y
    c = np.asarray(router_coeff, dtype=np.float64).reshape(-1)
    if c.shape[0] != Y.shape[0]:
        raise ValueError("router_coeff length must match the number of routed rows")
    return Y * c.reshape((-1,) + (1,) * (Y.ndim - 1))


def scatter_add_first_dim(src, indices, n_rows: int):
    """[EP] ``_scatter_add_first_dim``: a zero buffer of ``n_rows`` rows to
    which row i of ``src`` is added at row ``indices[i]`` (rows named more
    than once accumulate)."""
    S = np.asarray(src, dtype=np.float64)
    out = np.zeros((int(n_rows),) + S.shape[1:])
    for i, j in enumerate(np.asarray(indices, dtype=np.int64).reshape(-1)):
        out[j] += S[i]
    return out


def whiteboard_combine(expert_rows, dispatch_indices, gathered_coeff, n_gathered: int,
                       dtype: str):
    """The deredundancy combine on one outer-EP rank ([EP], the combine of
    the deredundancy dispatcher with an outer-EP size of 1, so no
    reduce-scatter follows): the dispatch gathered rows ``dispatch_indices``
    of the gathered buffer (with their router coefficients
    ``gathered_coeff[dispatch_indices]``); the combine scales the expert
    outputs of those rows by their coefficients and scatter-adds them back to
    the same positions of a zero [n_gathered, H] whiteboard, in that order.
    ``gathered_coeff`` None means no scaling."""
    idx = np.asarray(dispatch_indices, dtype=np.int64).reshape(-1)
    coeff = None if gathered_coeff is None else np.asarray(gathered_coeff, dtype=np.float64)[idx]
    weighted = scale_by_router_coeff(expert_rows, coeff)
    return round_to(scatter_add_first_dim(weighted, idx, n_gathered), dtype)


# --------------------------------------------------------------------------
# Step a11: permute backward
# --------------------------------------------------------------------------

def permute_grad(grad_permuted, row_map, T: int, K: int, dtype: str):
    """Backward of the row gather ``x[idx]`` ([GMM]: the gather's backward is
    an index_put that accumulates duplicate indices):

        grad_tokens[t] = round( sum_{k} grad_permuted[row_map[t*K+k]] )

    slots with row_map = -1 contribute nothing.
    """
    G = np.asarray(grad_permuted, dtype=np.float64)
    rm = np.asarray(row_map, dtype=np.int64).reshape(T, K)
    H = G.shape[1]
    out = np.zeros((T, H))
    for k in range(K):
        rows = rm[:, k]
        live = rows >= 0
        contrib = np.zeros((T, H))
        contrib[live] = G[rows[live]]
        out += contrib
    return round_to(out, dtype)


# --------------------------------------------------------------------------
# Step a12: expert MLP backward
# --------------------------------------------------------------------------

def expert_mlp_grad(grad_expanded, permuted, act, expert_offsets, W_gate, W_up, W_down,
                    dtype: str):
    """Backward of :func:`expert_mlp` by the textbook chain rule (R7, R8).

    Per expert e with rows X = permuted_e, dY = grad_expanded_e and the
    stored activation A = act_e:
        g = X Wg^T, u = X Wu^T, s = sigmoid(g)
        dA  = dY Wd                                   (d of act, [M, I])
        dg  = round(dA * u * s * (1 + g (1 - s)))     (d silu(g)/dg = s(1+g(1-s)))
        du  = round(dA * g * s)                       (= dA * silu(g))
        dX  = round(dg Wg + du Wu)                    ([M, H])
        dWd = round(dY^T A)    dWg = round(dg^T X)    dWu = round(du^T X)
    Experts with no rows get zero weight grads.  dg/du are rounded as the
    stored gradient of the pre-activations.
    Returns (d_permuted[N,H], dW_gate[E,I,H], dW_up[E,I,H], dW_down[E,H,I]).
    """
    X = np.asarray(permuted, dtype=np.float64)
    dY_all = np.asarray(grad_expanded, dtype=np.float64)
    A_all = np.asarray(act, dtype=np.float64)
    Wg = np.asarray(W_gate, dtype=np.float64)
    Wu = np.asarray(W_up, dtype=np.float64)
    Wd = np.asarray(W_down, dtype=np.float64)
    off = np.asarray(expert_offsets, dtype=np.int64)
    E, I, H = Wg.shape
    d_perm = np.zeros_like(X)
    dWg = np.zeros_like(Wg)
    dWu = np.zeros_like(Wu)
    dWd = np.zeros_like(Wd)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        Xe, dY, A = X[lo:hi], dY_all[lo:hi], A_all[lo:hi]
        g = Xe @ Wg[e].T
        u = Xe @ Wu[e].T
        s = _sigmoid(g)
        dA = dY @ Wd[e]
        dg = round_to(dA * u * s * (1.0 + g * (1.0 - s)), dtype)
        du = round_to(dA * g * s, dtype)
        d_perm[lo:hi] = round_to(dg @ Wg[e] + du @ Wu[e], dtype)
        dWd[e] = round_to(dY.T @ A, dtype)
        dWg[e] = round_to(dg.T @ Xe, dtype)
        dWu[e] = round_to(du.T @ Xe, dtype)
    return d_perm, dWg, dWu, dWd
