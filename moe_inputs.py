"""Seeded synthetic inputs for the MoE expert-layer workloads.

This module only draws random inputs: it holds none of the layer's arithmetic
(no routing, permutation, GEMM, SwiGLU, unpermute or combine).  Both the CUDA
library's tests/benchmark and the CPU oracle consume exactly the tensors it
returns, so the two sides see identical bytes.

Every draw uses numpy's PCG64 generator (platform independent) seeded by the
caller.  bf16 tensors are drawn in float32 and rounded to nearest-even by
torch's dtype conversion.  All tensors are returned on the CPU.

Workloads (sizes are parameters so tests can shrink them):
  tiny_fp32_layer      T=64 H=128 E=8 K=2 I=256, fp32, uniform distinct ids
  permute_unpermute    T=16384 H=4096 E=64 K=8, bf16 tokens, fp32 probs,
                       bf16 grad_out
  layer_forward_zipf   T=8192 H=2048 E=256 K=8 I=512, Zipf(1.2) routing with
                       8 experts that receive no token
  layer_fwd_bwd        T=4096 H=2048 E=128 K=8 I=768, uniform routing,
                       bf16 grad_out
  index_combine        counts[16 x 16] ~ Poisson(64); combine T=4096 H=7168
                       K=8 over 256 real + 4 zero + 4 copy + 4 const experts
"""

from __future__ import annotations

import numpy as np
import torch


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal(rng, shape, std=1.0, dtype=torch.bfloat16) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return torch.from_numpy(x).to(dtype)


def _uniform(rng, shape, lo=0.0, hi=1.0, dtype=torch.bfloat16) -> torch.Tensor:
    x = rng.uniform(lo, hi, size=shape).astype(np.float32)
    return torch.from_numpy(x).to(dtype)


def uniform_distinct_ids(rng, T: int, K: int, num_ids: int) -> torch.Tensor:
    """K distinct ids per row, each K-subset of [0, num_ids) equally likely,
    in random order: the first K columns of a random ranking of all ids."""
    ranks = np.argsort(rng.random((T, num_ids)), axis=1, kind="stable")[:, :K]
    return torch.from_numpy(ranks.astype(np.int32))


def zipf_distinct_ids(rng, T: int, K: int, E: int, s: float = 1.2,
                      num_empty: int = 8) -> torch.Tensor:
    """Zipf(s)-skewed distinct ids: rank r (0-based) has weight (r+1)^-s, the
    last ``num_empty`` ranks have weight 0, ranks map to experts through a
    seeded random permutation.  K distinct ids are sampled without
    replacement by Gumbel-top-K on log(weight)."""
    ranks = np.arange(E, dtype=np.float64)
    w = (ranks + 1.0) ** (-s)
    if num_empty:
        w[E - num_empty:] = 0.0
    rank_to_expert = rng.permutation(E)
    logw = np.full(E, -np.inf)
    logw[rank_to_expert] = np.log(np.where(w > 0, w, 1.0))
    logw[rank_to_expert[w == 0]] = -np.inf
    gumbel = -np.log(-np.log(rng.random((T, E))))
    score = logw[None, :] + gumbel
    ids = np.argsort(-score, axis=1, kind="stable")[:, :K]
    return torch.from_numpy(ids.astype(np.int32))


def softmax_probs(rng, T: int, K: int) -> torch.Tensor:
    """fp32 router weights: softmax over the K selected slots of N(0,1)
    logits (each row sums to 1)."""
    logits = rng.standard_normal((T, K))
    logits -= logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    return torch.from_numpy(p.astype(np.float32))


def tiny_fp32_layer(seed: int = 0, T: int = 64, H: int = 128, E: int = 8, K: int = 2,
                    I: int = 256) -> dict:
    rng = _rng(seed)
    return dict(
        T=T, H=H, E=E, K=K, I=I, dtype="f32",
        expert_ids=uniform_distinct_ids(rng, T, K, E),
        probs=softmax_probs(rng, T, K),
        W_gate=_normal(rng, (E, I, H), 0.02, torch.float32),
        W_up=_normal(rng, (E, I, H), 0.02, torch.float32),
        W_down=_normal(rng, (E, H, I), 0.02, torch.float32),
        tokens=_normal(rng, (T, H), 1.0, torch.float32),
    )


def permute_unpermute(seed: int = 0, T: int = 16384, H: int = 4096, E: int = 64,
                      K: int = 8) -> dict:
    rng = _rng(seed)
    return dict(
        T=T, H=H, E=E, K=K, dtype="bf16",
        expert_ids=uniform_distinct_ids(rng, T, K, E),
        probs=softmax_probs(rng, T, K),
        tokens=_normal(rng, (T, H)),
        grad_out=_normal(rng, (T, H)),
    )


def layer_forward_zipf(seed: int = 0, T: int = 8192, H: int = 2048, E: int = 256, K: int = 8,
                       I: int = 512, num_empty: int = 8) -> dict:
    rng = _rng(seed)
    return dict(
        T=T, H=H, E=E, K=K, I=I, dtype="bf16",
        expert_ids=zipf_distinct_ids(rng, T, K, E, 1.2, num_empty),
        probs=softmax_probs(rng, T, K),
        W_gate=_normal(rng, (E, I, H), 0.02),
        W_up=_normal(rng, (E, I, H), 0.02),
        W_down=_normal(rng, (E, H, I), 0.02),
        tokens=_normal(rng, (T, H)),
    )


def layer_fwd_bwd(seed: int = 0, T: int = 4096, H: int = 2048, E: int = 128, K: int = 8,
                  I: int = 768) -> dict:
    rng = _rng(seed)
    return dict(
        T=T, H=H, E=E, K=K, I=I, dtype="bf16",
        expert_ids=uniform_distinct_ids(rng, T, K, E),
        probs=softmax_probs(rng, T, K),
        W_gate=_normal(rng, (E, I, H), 0.02),
        W_up=_normal(rng, (E, I, H), 0.02),
        W_down=_normal(rng, (E, H, I), 0.02),
        tokens=_normal(rng, (T, H)),
        grad_out=_normal(rng, (T, H)),
    )


def index_counts(seed: int = 0, R: int = 16, E_local: int = 16, lam: float = 64.0) -> dict:
    rng = _rng(seed)
    counts = rng.poisson(lam, size=R * E_local).astype(np.int32)
    return dict(R=R, E=E_local, counts=torch.from_numpy(counts))


def index_combine(seed: int = 0, R: int = 16, E_local: int = 16, T: int = 4096, H: int = 7168,
                  K: int = 8, zero_num: int = 4, copy_num: int = 4, const_num: int = 4) -> dict:
    """Index generation plus combine.  The combine has E = R * E_local real
    experts followed by the zero, copy and const id ranges; ids are uniform
    distinct over all of them.  ``expanded`` has one N(0,1) row per slot
    whose id is a real expert (the expert outputs, in expert-major order)."""
    rng = _rng(seed)
    E = R * E_local
    counts = rng.poisson(64.0, size=R * E_local).astype(np.int32)
    total_ids = E + zero_num + copy_num + const_num
    ids = uniform_distinct_ids(rng, T, K, total_ids)
    n_real = int((ids < E).sum())
    return dict(
        R=R, E_local=E_local, counts=torch.from_numpy(counts),
        T=T, H=H, K=K, E=E, zero_num=zero_num, copy_num=copy_num, const_num=const_num,
        dtype="bf16",
        expert_ids=ids,
        scales=softmax_probs(rng, T, K),
        expanded=_normal(rng, (n_real, H)),
        shared_x=_normal(rng, (T, H)),
        ori_x=_normal(rng, (T, H)),
        alpha1=_uniform(rng, (const_num, H)),
        alpha2=_uniform(rng, (const_num, H)),
        const_v=_normal(rng, (const_num, H)),
    )
