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

The default workload is layer_fwd_bwd when the bf16 expert-MLP kernels are
available, else permute_unpermute.  The metric is tokens/s of the whole job
(all ranks).  Per-kernel CUDA-event times inside the timed region give each
kernel's achieved HBM GB/s or TFLOP/s; the dominant kernel goes into the
``roofline`` object against the measured peaks in MEASURED_PEAKS.json.
Inputs are larger than L2 (129 MB) for both workloads, so no L2 flush runs
between steps.

``e2e`` measures the same steps through the same C-ABI calls with the step's
inputs copied from pinned host memory and its results copied back inside the
timed region.  ``cpu_baseline`` times the CPU oracle on a bounded sample of
the same workload (rank 0, N=1 only).  ``--impl reference`` times the oracle
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


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
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
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
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


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    if source_digest(rec["sources"]) != rec["digest"]:
        return None
    return rec["bytes_per_launch"]


# ---------------------------------------------------------------- workloads

class Timers:
    """CUDA events around each library call of a step, on the launch stream."""

    def __init__(self):
        self.pending = {}
        self.enabled = False

    def __call__(self, name):
        timers = self

        class _Ctx:
            def __enter__(self_):
                if timers.enabled:
                    self_.a = torch.cuda.Event(enable_timing=True)
                    self_.a.record()

            def __exit__(self_, *exc):
                if timers.enabled:
                    b = torch.cuda.Event(enable_timing=True)
                    b.record()
                    timers.pending.setdefault(name, []).append((self_.a, b))
        return _Ctx()

    def summary(self):
        out = {}
        for name, pairs in self.pending.items():
            ms = [a.elapsed_time(b) for a, b in pairs]
            out[name] = {"launches": len(ms), "avg_ms": sum(ms) / len(ms), "total_ms": sum(ms)}
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


WORKLOADS = {"permute_unpermute": PermuteUnpermute}


def pick_workload(lib, requested: str):
    if requested != "auto":
        return WORKLOADS[requested]
    if "layer_fwd_bwd" in WORKLOADS and getattr(WORKLOADS["layer_fwd_bwd"], "available",
                                                lambda lib: False)(lib):
        return WORKLOADS["layer_fwd_bwd"]
    return WORKLOADS["permute_unpermute"]


# ---------------------------------------------------------------- CPU oracle timing

def time_oracle(work, budget_s: float = 12.0, start_tokens: int = 64, max_tokens: int = 2048):
    """Time the oracle on growing samples until one sample takes a few
    seconds, then repeat that sample within the budget.  Returns
    (tokens/s, cores, sample description)."""
    from oracle import moe_oracle as O
    n = start_tokens
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


# ---------------------------------------------------------------- main

def run_ours(args, world, rank, local):
    from unpermute_moe_permute_gb300 import binding as lib
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    W = pick_workload(lib, args.workload)
    work = W(lib, dev)
    peaks, peak_kind = load_peaks()
    timers = Timers()

    for _ in range(args.warmup):
        work.step(timers)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    timers.enabled = True
    launches0 = lib.moe_kernel_launches()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(args.steps):
        work.step(timers)
    end.record()
    torch.cuda.synchronize()
    launches = lib.moe_kernel_launches() - launches0
    timers.enabled = False
    clk = clocks.stop()
    barrier()
    elapsed_ms = start.elapsed_time(end)
    max_ms = reduce_max(elapsed_ms, dev)
    units = work.units_per_step * args.steps * world
    value = units / (max_ms / 1e3)

    # per-kernel figures and the dominant kernel
    per = timers.summary()
    kernels = {}
    for name, s in per.items():
        entry = {"launches": s["launches"], "avg_us": s["avg_ms"] * 1e3,
                 "share": s["total_ms"] / max(sum(v["total_ms"] for v in per.values()), 1e-9)}
        if name in work.flops:
            entry["tflops"] = work.flops[name] / (s["avg_ms"] * 1e-3) / 1e12
        if name in work.bytes:
            entry["gbs"] = work.bytes[name] / (s["avg_ms"] * 1e-3) / 1e9
        kernels[name] = entry
    dom = max(per, key=lambda n: per[n]["total_ms"])
    if dom in work.flops and work.flops[dom] / work.bytes.get(dom, 1) > 300:
        achieved = kernels[dom]["tflops"]
        peak = peaks["bf16_tflops_sustained"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        achieved = kernels[dom]["gbs"]
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    roof["frac"] = achieved / peak
    roof["kernel"] = dom
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    tr = recorded_traffic(dom)
    roof["traffic"] = tr
    roof["algorithmic_bytes"] = work.bytes.get(dom)

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
        "gpu_launches": int(launches),
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = time_oracle(work)
        result["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores,
                                  "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_e2e(work, args, dev, world):
    """Same steps, inputs copied in from pinned host memory and results
    copied back to pinned host memory inside the timed region."""
    host_in = {k: v.pin_memory() for k, v in work.host.items()}
    dev_in = {k: torch.empty_like(v, device=dev) for k, v in host_in.items()}
    host_out = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in work.results()]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(r.numel() * r.element_size() for r in host_out)
    off = Timers()

    def one():
        for k in dev_in:
            dev_in[k].copy_(host_in[k], non_blocking=True)
        work.step(off, dev_in)
        for h, r in zip(host_out, work.results()):
            h.copy_(r, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        one()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    torch.cuda.synchronize()
    dt = reduce_max(time.perf_counter() - t0, dev)
    barrier()
    return {"value": work.units_per_step * args.steps * world / dt, "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle timed on bounded samples."""
    if rank != 0:
        return
    from oracle import moe_oracle as O

    class _Host:
        pass

    work = PermuteUnpermute.__new__(PermuteUnpermute)
    d = moe_inputs.permute_unpermute(0)
    work.T, work.H, work.E, work.K = d["T"], d["H"], d["E"], d["K"]
    work.host = {k: d[k] for k in ("tokens", "expert_ids", "probs", "grad_out")}
    n = 256
    for _ in range(args.warmup):
        work.oracle_sample(O, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        work.oracle_sample(O, n)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    cores = os.cpu_count() or 1
    sample = f"{n}-token prefix of permute_unpermute_bwd per step, float64 numpy oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded moe_inputs generators)",
        "config": {"workload": "permute_unpermute_bwd: T=16384 H=4096 E=64 K=8 (oracle sample)",
                   "parallelism": "cpu"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
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
