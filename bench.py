#!/usr/bin/env python
"""Benchmark of the single-GPU MoE expert layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-components]

One step is one pass of the layer's hot path over one batch of synthetic
input that is already resident in HBM (seeded generators of moe_inputs.py):

  layer_fwd_bwd      T=4096 H=2048 E=128 K=8 I=768 bf16, uniform routing:
                     permute -> gate/up GEMM + SwiGLU -> down GEMM ->
                     unpermute -> unpermute backward -> expert-MLP backward
                     (dgrad + wgrad) -> permute backward
  permute_unpermute  T=16384 H=4096 E=64 K=8 bf16: permute -> unpermute ->
                     unpermute backward -> permute backward

The default workload is layer_fwd_bwd.  ``components`` adds the kernels of
the other workloads, measured the same way after the timed region:
permute_unpermute (permute/unpermute HBM GB/s), layer_forward (T=8192 H=2048
E=256 K=8 I=512 with Zipf(1.2) routing: grouped GEMM TFLOP/s) and
index_combine (index generation from counts[16 x 16] and the combine of
T=4096 H=7168 K=8 with 12 special experts).  The metric is tokens/s of the whole job
(all ranks).  The timed steps carry CUDA events around the dominant call
alone (picked from the warm-up steps), which give its achieved HBM GB/s or
TFLOP/s for the ``roofline`` object against the measured peaks in
MEASURED_PEAKS.json; ``kernels`` lists every call's figures from a separate
pass of as many steps with events around each call.
Inputs are larger than L2 (129 MB) for both workloads, so no L2 flush runs
between steps.

``e2e`` measures the same steps through the same C-ABI calls with the step's
inputs copied from pinned host memory and its results copied back inside the
timed region.  ``cpu_baseline`` times the CPU oracle on a bounded sample of
the same workload (rank 0, N=1 only), on all host cores and, in a child
process limited to one thread, on one.  ``--impl reference`` times the oracle
alone (the reference arm: there is no runnable reference implementation).

Multi-GPU: the layer's token batches are independent, so N GPUs run N
replicas (weak scaling) with no collective on the data path; ranks only meet
at the barriers around the timed region and in the max-over-ranks of the
elapsed time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import moe_inputs  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "MoE layer tokens/s on 1 GB300; permute/unpermute HBM GB/s; GMM TFLOP/s"


# ---------------------------------------------------------------- environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, device) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step: int, steps: int, world: int, max_elapsed_ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (weak scaling: each rank runs its own batch)."""
    return units_per_step * steps * world / (max_elapsed_ms / 1e3)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock/throttle samples every 50 ms; the samples whose
    timestamps fall inside the timed region are kept."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t_begin=None, t_end=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                except (ValueError, IndexError):
                    ts = None
                if t_begin is not None and ts is not None and not (t_begin - 0.05 <= ts <= t_end + 0.05):
                    continue
                try:
                    sm.append(float(parts[2]))
                    smax.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[6:10]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- traffic records

def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "unpermute_moe_permute_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_profile(workload: str, call: str):
    """The committed ncu record of one call of a workload
    (profiles/traffic.json, keyed by workload and call: DRAM bytes and the
    kernels' duration per launch), or None when there is no record or the
    kernel's sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(workload, {}).get(call)
    if not rec:
        return None
    if source_digest(rec["sources"]) != rec["digest"]:
        return None
    return rec


def recorded_traffic(workload: str, call: str):
    """DRAM bytes (read + written) per launch of one call, from the
    committed ncu record, or None (see recorded_profile)."""
    rec = recorded_profile(workload, call)
    return None if rec is None else rec["bytes_per_launch"]


# ---------------------------------------------------------------- workloads

class Timers:
    """CUDA events around each library call of a step, on the launch stream;
    with `only`, around that one call alone (an event record between two
    calls delays the second, so the timed steps carry as few as possible)."""

    def __init__(self, only=None):
        self.pending = {}
        self.enabled = False
        self.only = only

    def __call__(self, name):
        timers = self
        on = lambda: timers.enabled and timers.only in (None, name)  # noqa: E731

        class _Ctx:
            def __enter__(self_):
                if on():
                    self_.a = torch.cuda.Event(enable_timing=True)
                    self_.a.record()

            def __exit__(self_, *exc):
                if on():
                    b = torch.cuda.Event(enable_timing=True)
                    b.record()
                    timers.pending.setdefault(name, []).append((self_.a, b))
        return _Ctx()

    def summary(self):
        out = {}
        for name, pairs in self.pending.items():
            ms = [a.elapsed_time(b) for a, b in pairs]
            out[name] = {"launches": len(ms), "avg_ms": sum(ms) / len(ms), "total_ms": sum(ms),
                         "median_ms": statistics.median(ms)}
        return out


class PermuteUnpermute:
    name = "permute_unpermute"

    def __init__(self, lib, dev, seed=0, T=16384, H=4096, E=64, K=8):
        d = moe_inputs.permute_unpermute(seed, T=T, H=H, E=E, K=K)
        self.lib, self.dev = lib, dev
        self.T, self.H, self.E, self.K = T, H, E, K
        self.host = {k: d[k] for k in ("tokens", "expert_ids", "probs", "grad_out")}
        self.x = {k: v.to(dev) for k, v in self.host.items()}
        TK = T * K
        bf = torch.bfloat16
        self.permuted = torch.empty((TK, H), dtype=bf, device=dev)
        self.sorted = torch.empty(TK, dtype=torch.int32, device=dev)
        self.row_map = torch.empty(TK, dtype=torch.int32, device=dev)
        self.tpe = torch.empty(E, dtype=torch.int32, device=dev)
        self.off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.ws = torch.empty(max(lib.moe_permute_workspace_size(T, K, E), 16), dtype=torch.uint8,
                              device=dev)
        self.out = torch.empty((T, H), dtype=bf, device=dev)
        self.grad_perm = torch.empty((TK, H), dtype=bf, device=dev)
        self.grad_probs = torch.empty((T, K), dtype=torch.float32, device=dev)
        self.grad_tokens = torch.empty((T, H), dtype=bf, device=dev)
        rows = T * H * 2
        perm_rows = TK * H * 2
        idx = TK * 4
        # algorithmic bytes per launch of each timed call
        self.bytes = {
            "permute": rows + perm_rows + 4 * idx + 2 * 4 * (E + 1),
            "unpermute": perm_rows + rows + idx + TK * 4,
            "unpermute_grad": rows + 2 * perm_rows + idx + 2 * TK * 4,
            "permute_grad": perm_rows + rows + idx,
        }
        self.flops = {}
        self.kernel_sources = {
            "permute": ["route.cu", "common.cuh"],
            "unpermute": ["gather.cu", "common.cuh"],
            "unpermute_grad": ["gather.cu", "common.cuh"],
            "permute_grad": ["gather.cu", "common.cuh"],
        }
        self.config = {"workload": "permute_unpermute_bwd: T=16384 H=4096 E=64 K=8 bf16, fp32 "
                                   "probs, uniform distinct ids",
                       "T": T, "H": H, "E": E, "K": K, "l2": "inputs larger than L2, no flush"}

    def step(self, t: Timers, x=None):
        lib, x = self.lib, (x or self.x)
        T, K, E = self.T, self.K, self.E
        with t("permute"):
            lib.moe_permute(x["tokens"], x["expert_ids"], E, 0, permuted=self.permuted,
                            sorted_indices=self.sorted, row_map=self.row_map,
                            tokens_per_expert=self.tpe, expert_offsets=self.off,
                            workspace=self.ws)
        with t("unpermute"):
            lib.moe_unpermute(self.permuted, self.row_map, x["probs"], T, K, out=self.out)
        with t("unpermute_grad"):
            lib.moe_unpermute_grad(x["grad_out"], self.permuted, self.row_map, x["probs"], K,
                                   grad_permuted=self.grad_perm, grad_probs=self.grad_probs)
        with t("permute_grad"):
            lib.moe_permute_grad(self.grad_perm, self.row_map, T, K, out=self.grad_tokens)

    def results(self):
        return [self.out, self.grad_tokens, self.grad_probs]

    result_names = ("out", "grad_tokens", "grad_probs")

    units_per_step = property(lambda self: self.T)

    def oracle_sample(self, O, n_tokens: int, seed: int = 1):
        """Oracle on the first n_tokens tokens of the same workload."""
        d = self.host
        T, K, E = n_tokens, self.K, self.E
        ids = d["expert_ids"][:T].numpy()
        tok = d["tokens"][:T].float().numpy().astype(np.float64)
        probs = d["probs"][:T].numpy()
        gout = d["grad_out"][:T].float().numpy().astype(np.float64)
        si, rm, tpe, off = O.permute_routing(ids, E)
        perm = O.permute_rows(tok, si, K)
        out = O.unpermute(perm, rm, probs, T, K, "bf16")
        gp, gprob = O.unpermute_grad(gout, perm, rm, probs, T, K, "bf16")
        gt = O.permute_grad(gp, rm, T, K, "bf16")
        return out, gt, gprob


def _gemm_bytes(T, H, E_active, E, K, I, bf=2, fused=False):
    """Algorithmic bytes and flops of each call of the bf16 layer (each
    operand read once, each result written once; weights of experts that
    have rows are read, weight grads of every expert are written).  fused:
    the permute only routes, and the gate/up GEMMs read the [T, H] token
    matrix (their gathered operand) instead of the [N, H] permuted copy."""
    N = T * K
    idx = N * 4
    w_gu, w_d = E_active * 2 * I * H * bf, E_active * H * I * bf
    x_rows = T if fused else N  # rows of the gate/up GEMMs' token operand
    by = {
        "permute": 4 * idx if fused else T * H * bf + N * H * bf + 4 * idx,
        "gate_up_swiglu": x_rows * H * bf + w_gu + N * I * bf + N * 2 * I * bf,
        "gate_up_swiglu_nosave": x_rows * H * bf + w_gu + N * I * bf,
        "down_proj": N * I * bf + w_d + N * H * bf,
        "unpermute": N * H * bf + T * H * bf + idx + N * 4,
        "unpermute_grad": T * H * bf + 2 * N * H * bf + idx + 2 * N * 4,
        "down_dgrad_swiglu": N * H * bf + w_d + 2 * N * 2 * I * bf,
        "gate_up_dgrad": N * 2 * I * bf + w_gu + N * H * bf,
        "down_wgrad": N * H * bf + N * I * bf + E * H * I * bf,
        "gate_up_wgrad": N * 2 * I * bf + x_rows * H * bf + E * 2 * I * H * bf,
        "permute_grad": N * H * bf + T * H * bf + idx,
    }
    fl = {
        "gate_up_swiglu": 2.0 * N * H * 2 * I,
        "gate_up_swiglu_nosave": 2.0 * N * H * 2 * I,
        "down_proj": 2.0 * N * I * H,
        "down_dgrad_swiglu": 2.0 * N * H * I,
        "gate_up_dgrad": 2.0 * N * 2 * I * H,
        "down_wgrad": 2.0 * N * H * I,
        "gate_up_wgrad": 2.0 * N * 2 * I * H,
    }
    return by, fl


class LayerFwdBwd:
    """T=4096 H=2048 E=128 K=8 I=768 bf16: forward and backward of the layer."""

    name = "layer_fwd_bwd"
    oracle_start_tokens = 256  # amortises the oracle's per-expert weight reads
    # True: the permute's row copy fused into the gate/up GEMMs (they gather
    # the token rows themselves).  Off by default: on GB300 at these shapes
    # the gathering GEMMs are slower than the row copy plus the plain GEMMs.
    FUSED_PERMUTE = False

    @staticmethod
    def available(lib):
        return True

    def __init__(self, lib, dev, seed=0, gen=moe_inputs.layer_fwd_bwd, backward=True, **kw):
        d = gen(seed, **kw)
        self.lib, self.dev, self.backward = lib, dev, backward
        self.fused = self.FUSED_PERMUTE
        T, H, E, K, I = d["T"], d["H"], d["E"], d["K"], d["I"]
        self.T, self.H, self.E, self.K, self.I = T, H, E, K, I
        keys = ("tokens", "expert_ids", "probs") + (("grad_out",) if backward else ())
        self.host = {k: d[k] for k in keys}
        self.x = {k: v.to(dev) for k, v in self.host.items()}
        self.Wg, self.Wu, self.Wd = d["W_gate"].to(dev), d["W_up"].to(dev), d["W_down"].to(dev)
        N = T * K
        bf = torch.bfloat16
        e = lambda *shape, dt=bf: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
        self.permuted = None if self.fused else e(N, H)
        self.sorted, self.row_map = e(N, dt=torch.int32), e(N, dt=torch.int32)
        self.tpe, self.off = e(E, dt=torch.int32), e(E + 1, dt=torch.int32)
        self.ws = e(max(lib.moe_permute_workspace_size(T, K, E), 16), dt=torch.uint8)
        self.act, self.expanded, self.out = e(N, I), e(N, H), e(T, H)
        self.gu = e(N, 2 * I) if backward else None
        if backward:
            self.gexp, self.gprobs, self.dgu, self.dperm = e(N, H), e(T, K, dt=torch.float32), e(N, 2 * I), e(N, H)
            self.dWg, self.dWu, self.dWd = torch.empty_like(self.Wg), torch.empty_like(self.Wu), torch.empty_like(self.Wd)
            self.gtok = e(T, H)
        counts = np.bincount(d["expert_ids"].numpy().reshape(-1), minlength=E)
        self.E_active = int((counts > 0).sum())
        by, fl = _gemm_bytes(T, H, self.E_active, E, K, I, fused=self.fused)
        if not backward:
            by["gate_up_swiglu"], fl["gate_up_swiglu"] = by["gate_up_swiglu_nosave"], fl["gate_up_swiglu_nosave"]
        self.bytes, self.flops = by, fl
        self.config = {"workload": f"{'layer_fwd_bwd' if backward else 'layer_forward'}: "
                                   f"T={T} H={H} E={E} K={K} I={I} bf16, fp32 probs",
                       "T": T, "H": H, "E": E, "K": K, "I": I, "experts_with_rows": self.E_active,
                       "permute": ("routing only; the gate/up GEMMs gather the token rows "
                                   "(cp.async row gathers)") if self.fused else "routing + row copy",
                       "l2": "inputs larger than L2 (weights alone exceed it), no flush"}

    @classmethod
    def host_only(cls, seed=0):
        """The workload's host inputs only (no GPU): for the CPU oracle."""
        w = cls.__new__(cls)
        d = moe_inputs.layer_fwd_bwd(seed)
        w.T, w.H, w.E, w.K, w.I, w.backward = d["T"], d["H"], d["E"], d["K"], d["I"], True
        w.host = {k: d[k] for k in ("tokens", "expert_ids", "probs", "grad_out")}
        w.Wg, w.Wu, w.Wd = d["W_gate"], d["W_up"], d["W_down"]
        w.config = {"workload": f"layer_fwd_bwd: T={w.T} H={w.H} E={w.E} K={w.K} I={w.I} bf16, "
                                "fp32 probs"}
        return w

    def step(self, t: Timers, x=None):
        lib, x = self.lib, (x or self.x)
        T, K, E = self.T, self.K, self.E
        with t("permute"):
            lib.moe_permute(None if self.fused else x["tokens"], x["expert_ids"], E, 0,
                            permuted=self.permuted, sorted_indices=self.sorted,
                            row_map=self.row_map, tokens_per_expert=self.tpe,
                            expert_offsets=self.off, workspace=self.ws)
        with t("gate_up_swiglu"):
            if self.fused:
                lib.moe_gate_up_swiglu_gather(x["tokens"], self.sorted, K, self.off, self.Wg,
                                              self.Wu, act=self.act, gate_up_save=self.gu)
            else:
                lib.moe_gate_up_swiglu(self.permuted, self.off, self.Wg, self.Wu, act=self.act,
                                       gate_up_save=self.gu)
        with t("down_proj"):
            lib.moe_down_proj(self.act, self.off, self.Wd, expanded=self.expanded)
        with t("unpermute"):
            lib.moe_unpermute(self.expanded, self.row_map, x["probs"], T, K, out=self.out)
        if not self.backward:
            return
        with t("unpermute_grad"):
            lib.moe_unpermute_grad(x["grad_out"], self.expanded, self.row_map, x["probs"], K,
                                   grad_permuted=self.gexp, grad_probs=self.gprobs)
        with t("down_dgrad_swiglu"):
            lib.moe_down_dgrad_swiglu(self.gexp, self.gu, self.off, self.Wd, dgu=self.dgu)
        with t("gate_up_dgrad"):
            lib.moe_gate_up_dgrad(self.dgu, self.off, self.Wg, self.Wu, d_permuted=self.dperm)
        with t("down_wgrad"):
            lib.moe_down_wgrad(self.gexp, self.act, self.off, dW_down=self.dWd)
        with t("gate_up_wgrad"):
            if self.fused:
                lib.moe_gate_up_wgrad_gather(self.dgu, x["tokens"], self.sorted, K, self.off,
                                             dW_gate=self.dWg, dW_up=self.dWu)
            else:
                lib.moe_gate_up_wgrad(self.dgu, self.permuted, self.off, dW_gate=self.dWg,
                                      dW_up=self.dWu)
        with t("permute_grad"):
            lib.moe_permute_grad(self.dperm, self.row_map, T, K, out=self.gtok)

    def results(self):
        return [getattr(self, n) for n in self.result_names]

    @property
    def result_names(self):
        return ("out", "gtok", "gprobs") if self.backward else ("out",)

    units_per_step = property(lambda self: self.T)

    def oracle_sample(self, O, n_tokens: int, reached_only: bool = False, cache={}):
        """Oracle forward (and backward) of the first n_tokens tokens.  With
        reached_only, the sample is the sub-problem over the experts those
        tokens reach (ids renumbered in expert order, so the permuted order
        is the full problem's): the same outputs and the same weight
        gradients of those experts, without the exact zeros of the others."""
        key = (id(self), n_tokens if reached_only else None)
        if key not in cache:  # bf16 -> float64 decode of the weights, done once
            cache.clear()
            ids = self.host["expert_ids"][:n_tokens].numpy()
            sel = np.unique(ids) if reached_only else np.arange(self.E)
            cache[key] = (sel,) + tuple(w[torch.from_numpy(sel).long().to(w.device)].float().cpu().numpy()
                                        .astype(np.float64) for w in (self.Wg, self.Wu, self.Wd))
        sel, Wg, Wu, Wd = cache[key]
        d = self.host
        T, K, E = n_tokens, self.K, len(sel)
        ids = np.searchsorted(sel, d["expert_ids"][:T].numpy()).astype(np.int32)
        tok = d["tokens"][:T].float().numpy().astype(np.float64)
        probs = d["probs"][:T].numpy()
        si, rm, tpe, off = O.permute_routing(ids, E)
        perm = O.permute_rows(tok, si, K)
        act, y, _, _ = O.expert_mlp(perm, off, Wg, Wu, Wd, "bf16")
        out = O.unpermute(y, rm, probs, T, K, "bf16")
        if not self.backward:
            return out
        gout = d["grad_out"][:T].float().numpy().astype(np.float64)
        gy, gp = O.unpermute_grad(gout, y, rm, probs, T, K, "bf16")
        dperm, dWg, dWu, dWd = O.expert_mlp_grad(gy, perm, act, off, Wg, Wu, Wd, "bf16")
        return out, O.permute_grad(dperm, rm, T, K, "bf16"), gp


class LayerForward(LayerFwdBwd):
    """T=8192 H=2048 E=256 K=8 I=512 bf16 forward, Zipf(1.2) routing."""

    name = "layer_forward"

    def __init__(self, lib, dev, seed=0, **kw):
        super().__init__(lib, dev, seed, gen=moe_inputs.layer_forward_zipf, backward=False, **kw)


class SharedExpertOverlap:
    """T=4096 H=2048 E=128 K=8 I=768 bf16 forward plus a shared expert
    (I=1536) whose output the combine adds: one stream, or the shared expert
    on a second stream concurrently with the routed path."""

    name = "shared_expert_overlap"

    def __init__(self, lib, dev, seed=0, I_shared=1536):
        d = moe_inputs.layer_fwd_bwd(seed)
        s = moe_inputs.layer_fwd_bwd(seed + 1, T=1, H=d["H"], E=1, K=1, I=I_shared)
        self.lib, self.dev = lib, dev
        T, H, E, K, I = d["T"], d["H"], d["E"], d["K"], d["I"]
        self.T, self.E, self.K = T, E, K
        self.x = {k: d[k].to(dev) for k in ("tokens", "expert_ids", "probs")}
        self.Wg, self.Wu, self.Wd = d["W_gate"].to(dev), d["W_up"].to(dev), d["W_down"].to(dev)
        self.Sg, self.Su, self.Sd = (s["W_gate"][0].to(dev), s["W_up"][0].to(dev),
                                     s["W_down"][0].to(dev))
        N, bf = T * K, torch.bfloat16
        e = lambda *shape, dt=bf: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
        self.permuted, self.sorted, self.row_map = e(N, H), e(N, dt=torch.int32), e(N, dt=torch.int32)
        self.tpe, self.off = e(E, dt=torch.int32), e(E + 1, dt=torch.int32)
        self.ws = e(max(lib.moe_permute_workspace_size(T, K, E), 16), dt=torch.uint8)
        self.act, self.expanded, self.out = e(N, I), e(N, H), e(T, H)
        self.s_act, self.shared = e(T, I_shared), e(T, H)
        self.side = torch.cuda.Stream(device=dev)
        self.config = {"workload": f"layer forward T={T} H={H} E={E} K={K} I={I} plus a shared "
                                   f"expert I={I_shared}, bf16"}

    def _shared(self):
        self.lib.moe_shared_expert_mlp(self.x["tokens"], self.Sg, self.Su, self.Sd,
                                       act=self.s_act, out=self.shared)

    def _routed(self):
        lib, x = self.lib, self.x
        lib.moe_permute(x["tokens"], x["expert_ids"], self.E, 0, permuted=self.permuted,
                        sorted_indices=self.sorted, row_map=self.row_map,
                        tokens_per_expert=self.tpe, expert_offsets=self.off, workspace=self.ws)
        lib.moe_gate_up_swiglu(self.permuted, self.off, self.Wg, self.Wu, act=self.act)
        lib.moe_down_proj(self.act, self.off, self.Wd, expanded=self.expanded)

    def _combine(self):
        x = self.x
        self.lib.moe_combine(self.expanded, self.row_map, x["expert_ids"], x["probs"], self.E,
                             shared_x=self.shared, out=self.out)

    def step(self, overlapped: bool):
        main = torch.cuda.current_stream(self.dev)
        if not overlapped:
            self._shared()
            self._routed()
        else:
            ready = torch.cuda.Event()
            ready.record(main)
            with torch.cuda.stream(self.side):
                self.side.wait_event(ready)
                self._shared()
                done = torch.cuda.Event()
                done.record(self.side)
            self._routed()
            main.wait_event(done)
        self._combine()

    def measure(self, steps=20, warmup=3):
        res = {}
        for overlapped in (False, True):
            for _ in range(warmup):
                self.step(overlapped)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(steps):
                self.step(overlapped)
            b.record()
            torch.cuda.synchronize()
            res["overlapped_us" if overlapped else "one_stream_us"] = a.elapsed_time(b) / steps * 1e3
        return res


class IndexCombine:
    """Permute-index generation from counts[16 x 16] and the combine of
    T=4096 H=7168 K=8 over 256 real + 4 zero + 4 copy + 4 const experts."""

    name = "index_combine"

    def __init__(self, lib, dev, seed=0):
        d = moe_inputs.index_combine(seed)
        self.lib = lib
        self.d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in d.items()}
        T, K, H = d["T"], d["K"], d["H"]
        self.R, self.El = d["R"], d["E_local"]
        self.total = int(d["counts"].sum())
        self.idx = torch.empty(self.total, dtype=torch.int32, device=dev)
        self.tpe = torch.empty(self.El, dtype=torch.int32, device=dev)
        self.tot = torch.empty(1, dtype=torch.int32, device=dev)
        nsp = d["zero_num"] + d["copy_num"] + d["const_num"]
        self.routing = lib.moe_permute(None, self.d["expert_ids"], d["E"], nsp)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        n_real = d["expanded"].shape[0]
        ids = d["expert_ids"].numpy()
        n_ori = int(((ids >= d["E"] + d["zero_num"]).any(axis=1)).sum())
        self.bytes = {"combine": n_real * H * 2 + n_ori * H * 2 + 2 * T * H * 2 + T * K * 12,
                      "permute_indices": self.R * self.El * 4 * 2 + self.total * 4}
        self.flops = {}

    def step(self, t: Timers, x=None):
        d, lib = self.d, self.lib
        with t("permute_indices"):
            lib.moe_permute_indices(d["counts"], self.R, self.El, self.total, indices=self.idx,
                                    tokens_per_expert=self.tpe, total=self.tot)
        with t("combine"):
            lib.moe_combine(d["expanded"], self.routing.row_map, d["expert_ids"], d["scales"], d["E"],
                            shared_x=d["shared_x"], ori_x=d["ori_x"], zero_num=d["zero_num"],
                            copy_num=d["copy_num"], const_num=d["const_num"], alpha1=d["alpha1"],
                            alpha2=d["alpha2"], const_v=d["const_v"], out=self.out)


WORKLOADS = {"permute_unpermute": PermuteUnpermute, "layer_fwd_bwd": LayerFwdBwd,
             "layer_forward": LayerForward}


def pick_workload(lib, requested: str):
    if requested != "auto":
        return WORKLOADS[requested]
    return WORKLOADS["layer_fwd_bwd"]


def kernel_table(per, work, peaks):
    """Per-call figures from CUDA-event times: GB/s and TFLOP/s of the
    algorithmic bytes/flops, their fractions of the measured peaks, and the
    bound (the larger of flops/peak and bytes/bandwidth)."""
    total = max(sum(v["total_ms"] for v in per.values()), 1e-9)
    out = {}
    for name, s in per.items():
        sec = s["avg_ms"] * 1e-3
        e = {"launches": s["launches"], "avg_us": s["avg_ms"] * 1e3, "share": s["total_ms"] / total}
        if "median_ms" in s:
            e["median_us"] = s["median_ms"] * 1e3
        by, fl = work.bytes.get(name), work.flops.get(name)
        if by:
            e["gbs"] = by / sec / 1e9
            e["hbm_frac"] = e["gbs"] / peaks["hbm_gbs"]
        rec = recorded_profile(getattr(work, "name", ""), name)
        if rec is not None:
            # ncu, per launch (profiles/traffic.json): DRAM bytes, and the
            # kernels' own duration (cold caches, no launch gaps; the event
            # times above include the gap an event record adds before a call)
            e["dram_bytes"] = rec["bytes_per_launch"]
            e["ncu_us"] = rec["ncu_duration_ns"] / 1e3
            if by:
                e["dram_over_algorithmic"] = rec["bytes_per_launch"] / by
                e["ncu_hbm_frac"] = by / (rec["ncu_duration_ns"] * 1e-9) / 1e9 / peaks["hbm_gbs"]
        if fl:
            e["tflops"] = fl / sec / 1e12
            e["tensor_frac"] = e["tflops"] / peaks["bf16_tflops_sustained"]
            t_tc = fl / (peaks["bf16_tflops_sustained"] * 1e12)
            t_hbm = (by or 0) / (peaks["hbm_gbs"] * 1e9)
            e["bound"] = "tensor" if t_tc >= t_hbm else "hbm"
            e["roofline_frac"] = max(t_tc, t_hbm) / sec
        else:
            e["bound"] = "hbm"
            if by:
                e["roofline_frac"] = e["hbm_frac"]
        out[name] = e
    return out


def measure(work, steps, warmup, sync_barrier=False):
    t = Timers()
    for _ in range(warmup):
        work.step(t)
    torch.cuda.synchronize()
    t.enabled = True
    for _ in range(steps):
        work.step(t)
    torch.cuda.synchronize()
    return t.summary()


def run_components(lib, dev, peaks, steps=50, warmup=5):
    """The other workloads' headline kernels, measured the same way (50
    steps after 5 warm-up steps; every input is larger than L2, so no flush
    runs between steps)."""
    comps = {}
    for cls in (PermuteUnpermute, LayerForward, IndexCombine):
        w = cls(lib, dev)
        per = measure(w, steps, warmup)
        comps[w.name if hasattr(w, "name") else cls.__name__] = {
            "config": getattr(w, "config", {}).get("workload", cls.__doc__.strip().splitlines()[0] if cls.__doc__ else ""),
            "kernels": kernel_table(per, w, peaks)}
        del w
        torch.cuda.empty_cache()
    w = SharedExpertOverlap(lib, dev)
    comps[w.name] = {"config": w.config["workload"], "forward_us": w.measure()}
    del w
    torch.cuda.empty_cache()
    return comps


# ---------------------------------------------------------------- CPU oracle timing

def time_oracle(work, budget_s: float = 12.0, start_tokens: int = None, max_tokens: int = 2048):
    """Time the oracle on growing samples until one sample takes a few
    seconds, then repeat that sample within the budget.  Returns
    (tokens/s, cores, sample description)."""
    from oracle import moe_oracle as O
    n = start_tokens or getattr(work, "oracle_start_tokens", 64)
    t0 = time.perf_counter()
    work.oracle_sample(O, n)
    dt = time.perf_counter() - t0
    while dt < budget_s / 6 and n < max_tokens:
        n = min(max_tokens, n * 2)
        t0 = time.perf_counter()
        work.oracle_sample(O, n)
        dt = time.perf_counter() - t0
    done, spent = 0, 0.0
    while spent < budget_s / 2 or done == 0:
        t0 = time.perf_counter()
        work.oracle_sample(O, n)
        spent += time.perf_counter() - t0
        done += n
    cores = os.cpu_count() or 1
    return done / spent, cores, f"{n}-token prefix of the same workload, {done // n} run(s), float64 numpy"


def time_oracle_single_thread(budget_s: float = 12.0):
    """The same oracle timing in a child process whose BLAS and OpenMP pools
    are limited to one thread (the variables must be set before numpy
    loads).  Returns (tokens/s, sample description), or None if the child
    failed."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-child", str(budget_s)]
    try:
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=30 * budget_s)
        line = [ln for ln in res.stdout.splitlines() if ln.startswith("{")][-1]
        rec = json.loads(line)
        return rec["value"], rec["sample"]
    except Exception:  # noqa: BLE001 - a missing baseline must not fail the bench
        return None


def oracle_child(budget_s: float):
    """Entry of the single-thread oracle timing (see time_oracle_single_thread)."""
    work = LayerFwdBwd.host_only(0)
    v, _, sample = time_oracle(work, budget_s=budget_s, start_tokens=16)
    print(json.dumps({"value": v, "sample": sample}), flush=True)


# ---------------------------------------------------------------- main

def run_ours(args, world, rank, local):
    from unpermute_moe_permute_gb300 import binding as lib
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    W = pick_workload(lib, args.workload)
    work = W(lib, dev)
    peaks, peak_kind = load_peaks()
    # The warm-up steps after the first carry events around every call; they
    # pick the dominant call, which alone is bracketed by events in the
    # timed steps.
    warm = Timers()

    clocks = ClockSampler(local)
    clocks.start()  # started before the warm-up so that it samples the whole timed region
    for i in range(args.warmup):
        warm.enabled = i > 0
        work.step(warm)
    warm.enabled = False
    torch.cuda.synchronize()
    warm_per = warm.summary()
    dom = max(warm_per, key=lambda n: warm_per[n]["total_ms"])
    timers = Timers(only=dom)
    time.sleep(0.2)
    barrier()
    torch.cuda.synchronize()

    timers.enabled = True
    launches0 = lib.moe_kernel_launches()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    start.record()
    for _ in range(args.steps):
        work.step(timers)
    end.record()
    torch.cuda.synchronize()
    t_end = time.time()
    launches = lib.moe_kernel_launches() - launches0
    timers.enabled = False
    clk = clocks.stop(t_begin, t_end)
    barrier()
    elapsed_ms = start.elapsed_time(end)
    max_ms = reduce_max(elapsed_ms, dev)
    value = job_throughput(work.units_per_step, args.steps, world, max_ms)

    # per-call figures: a separate pass of as many steps with events around
    # every call; the dominant call's own figures come from the timed steps
    per = measure(work, args.steps, 0)
    kernels = kernel_table(per, work, peaks)
    k = kernel_table(timers.summary(), work, peaks)[dom]
    if k.get("bound") == "tensor":
        achieved, peak = k["tflops"], peaks["bf16_tflops_sustained"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        achieved, peak = k["gbs"], peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    roof["frac"] = achieved / peak
    roof["kernel"] = dom
    roof["peak_source"] = ("measured (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback")
    roof["traffic"] = recorded_traffic(work.name, dom)
    roof["algorithmic_bytes"] = work.bytes.get(dom)
    roof["algorithmic_flops"] = work.flops.get(dom)

    # end to end through the same calls with host buffers
    e2e = run_e2e(work, args, dev, world)

    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": max_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded moe_inputs generators)",
        "config": dict(work.config, parallelism=f"replicas{world}"),
        "roofline": roof,
        "kernels": kernels,
        "kernels_pass": "per-call CUDA events in a separate pass of the same number of steps "
                        "after the timed region (the timed steps bracket only the dominant call)",
        "gpu_launches": int(launches),
        "clocks": clk,
        "e2e": e2e,
    }
    if not args.no_components and world == 1:
        result["components"] = run_components(lib, dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = time_oracle(work)
        result["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores,
                                  "kind": "oracle", "sample": sample}
        one = time_oracle_single_thread()
        if one is not None:
            result["cpu_baseline"]["single_thread"] = {"value": one[0], "unit": "tokens/s",
                                                       "cores": 1, "sample": one[1]}
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_e2e(work, args, dev, world):
    """Same steps through the same calls, with every step's inputs copied in
    from pinned host memory and its results copied back to pinned host
    memory inside the timed region.  As a training loop would, the copies
    run on two copy streams and overlap the neighbouring steps' compute:
    inputs and results are double-buffered (slot = step % 2), and events
    order each copy against the compute that produces or consumes it."""
    host_in = {k: v.pin_memory() for k, v in work.host.items()}
    names = list(work.result_names)
    slots = [{n: getattr(work, n) for n in names},
             {n: torch.empty_like(getattr(work, n)) for n in names}]
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host_in.items()} for _ in range(2)]
    host_out = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in sl.items()}
                for sl in slots]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    compute = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    off = Timers()

    def run(n_steps):
        for i in range(n_steps):
            sl = i % 2
            if i >= 2:
                s_in.wait_event(in_free[sl])          # step i-2 finished reading this slot
            with torch.cuda.stream(s_in):
                for k in dev_in[sl]:
                    dev_in[sl][k].copy_(host_in[k], non_blocking=True)
                in_ready[sl].record(s_in)
            compute.wait_event(in_ready[sl])
            if i >= 2:
                compute.wait_event(out_free[sl])      # step i-2's results were copied out
            for n in names:
                setattr(work, n, slots[sl][n])
            work.step(off, dev_in[sl])
            in_free[sl].record(compute)
            out_ready[sl].record(compute)
            s_out.wait_event(out_ready[sl])
            with torch.cuda.stream(s_out):
                for n in names:
                    host_out[sl][n].copy_(slots[sl][n], non_blocking=True)
                out_free[sl].record(s_out)
        for n in names:
            setattr(work, n, slots[0][n])

    run(max(2, args.warmup))
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    run(args.steps)
    torch.cuda.synchronize()
    dt = reduce_max(time.perf_counter() - t0, dev)
    barrier()
    return {"value": work.units_per_step * args.steps * world / dt, "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "double-buffered copies on two copy streams, overlapping neighbouring steps"}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle timed on bounded samples of the same
    workload (one sample per step)."""
    if rank != 0:
        return
    from oracle import moe_oracle as O
    work = LayerFwdBwd.host_only(0)
    # Tokens per step: the first n of the batch, over the experts they reach.
    # The cost is dominated by the reached experts' weight gradients, so n
    # is halved (down to 1) until the timed steps fit in about two minutes.
    budget_s = 120.0
    n = 8
    while True:
        work.oracle_sample(O, n, reached_only=True)  # decodes the sample's weights once
        t0 = time.perf_counter()
        work.oracle_sample(O, n, reached_only=True)
        if n == 1 or (time.perf_counter() - t0) * args.steps <= budget_s:
            break
        n //= 2
    for _ in range(max(0, args.warmup - 2)):
        work.oracle_sample(O, n, reached_only=True)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        work.oracle_sample(O, n, reached_only=True)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    cores = os.cpu_count() or 1
    sample = (f"first {n} tokens of the layer_fwd_bwd batch per step (forward + backward over "
              "the experts they reach, whose weight gradients it computes), float64 numpy oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded moe_inputs generators)",
        "config": dict(work.config, parallelism="cpu"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-components", action="store_true")
    ap.add_argument("--oracle-child", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--fused-permute", action="store_true",
                    help="layer workloads: the gate/up GEMMs gather the token rows themselves "
                         "(default: the permute writes the permuted copy they read)")
    args = ap.parse_args(argv)
    if args.oracle_child is not None:
        oracle_child(args.oracle_child)
        return
    if args.fused_permute:
        LayerFwdBwd.FUSED_PERMUTE = True
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
