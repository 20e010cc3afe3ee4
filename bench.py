"""Benchmark of the verification step on GB300.

Default workload: sampling verification, B=64 requests, K=4 drafts, V=128256,
fp32 logits, T=0.7 (the configuration the headline metric is quoted on).
One step = one spec_verify_sample call over the resident batch: both passes
(logits stream + decide, residual + draw).  Metric: verified draft tokens/s
(B K per step) and the HBM bandwidth implied by reading logits + q once.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (torchrun): every rank verifies its own batch (requests are
independent, no collective on the data path; replicas, weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/s and HBM GB/s vs ~8 TB/s peak (B=64, K=4, V=128256)"
UNIT = "verified draft tokens/s"
WORKLOAD = "sampling verify B=64 K=4 V=128256 fp32 logits T=0.7"
L2_FLUSH_BYTES = 256 << 20
NOMINAL_PEAK_GBS = 8000.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_11_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(kernel)
        if rec and rec.get("source_hash") == _source_hash():
            return rec["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


class Clocks:
    """Samples nvidia-smi every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _cpu_sample(batch, target_s=10.0):
    """The oracle as it stands on a bounded sample of the workload: the first
    16 requests, repeated until ~target_s of host time."""
    import oracle
    n_req = 16
    rows = n_req * (batch.K + 1)
    z, q = batch.logits[:rows], batch.q[: n_req * batch.K]
    x, u = batch.draft[: n_req * batch.K], batch.uniforms[:rows]
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.verify_fixed(z, q, x, u, n_req, batch.K, batch.temperature)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return {"value": reps * n_req * batch.K / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {n_req} of 64 requests, {reps} repetitions, {el:.1f} s, fp64 C, 1 thread"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    from speculative_decoding_verification_11_gb300 import workloads as W
    import oracle
    oracle.build()
    batch = W.sampling()
    n_req = 8
    rows = n_req * (batch.K + 1)
    z, q = batch.logits[:rows], batch.q[: n_req * batch.K]
    x, u = batch.draft[: n_req * batch.K], batch.uniforms[:rows]
    for _ in range(args.warmup):
        oracle.verify_fixed(z, q, x, u, n_req, batch.K, batch.temperature)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify_fixed(z, q, x, u, n_req, batch.K, batch.temperature)
    el = time.perf_counter() - t0
    value = args.steps * n_req * batch.K / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "B": 64, "K": 4, "V": 128256},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{n_req} of 64 requests per step, fp64 C oracle, 1 thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from speculative_decoding_verification_11_gb300 import binding as B_, build as build_mod, workloads as W
    build_mod.build()
    B_.load()

    batch = W.sampling(seed=1002 + rank)
    Bn, K, V, T = batch.B, batch.K, batch.V, batch.temperature
    R = batch.rows
    logits = batch.logits.to(dev)
    q = batch.q.to(dev)
    draft = batch.draft.to(dev)
    uni = batch.uniforms.to(dev)
    out = torch.empty(R, dtype=torch.int32, device=dev)
    al = torch.empty(Bn, dtype=torch.int32, device=dev)
    ws = B_.workspace(B_.spec_verify_workspace_size(Bn, R, V), dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        B_.spec_verify_sample(logits, q, Bn, K, V, T, draft, uni, out, al, ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for evs in ev:  # torch creates an event on its first record; the library re-records them
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    launches = 0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        flush.fill_(float(i))
        s0, s1, k0, k1 = ev[i]
        B_.spec_profile_set_events(k0, k1)
        s0.record(stream)
        step()
        s1.record(stream)
        launches += B_.spec_last_launch_count()
    B_.spec_profile_set_events(None, None)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b, _, _ in ev]
    k_ms = [c.elapsed_time(d) for _, _, c, d in ev]
    ms = statistics.mean(step_ms)
    kms = statistics.mean(k_ms)
    if world > 1:
        t = torch.tensor([ms, kms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms, kms = t.tolist()

    # outcome of the step (same every step: same inputs)
    al_h = al.cpu()
    n_reject = int((al_h <= K).sum())
    units = Bn * K
    value = world * units / (ms * 1e-3)
    nominal = W.nominal_bytes(batch)
    logits_bytes = R * V * 4
    gathers = Bn * K * 16 + R * 4 + Bn * 4
    pass1_alg = logits_bytes + gathers
    step_alg = pass1_alg + n_reject * V * 4
    peak, peak_kind = _peaks()
    achieved = pass1_alg / (kms * 1e-3) / 1e9

    # end to end through the public API: pinned host inputs in, results out
    pin = {k: v.pin_memory() for k, v in
           (("logits", batch.logits), ("q", batch.q), ("draft", batch.draft), ("uni", batch.uniforms))}
    out_h = torch.empty(R, dtype=torch.int32).pin_memory()
    al_hh = torch.empty(Bn, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = out_h.numel() * 4 + al_hh.numel() * 4

    def e2e_step():
        logits.copy_(pin["logits"], non_blocking=True)
        q.copy_(pin["q"], non_blocking=True)
        draft.copy_(pin["draft"], non_blocking=True)
        uni.copy_(pin["uni"], non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
        al_hh.copy_(al, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(args.steps, 20))
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = t.item()

    cpu = _cpu_sample(batch) if (rank == 0 and world == 1 and not args.no_cpu) else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": Bn, "K": K, "V": V, "T": T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (256 MB write); inputs 295.5 MB > L2"},
        "hbm_gbs_nominal": world * nominal / (ms * 1e-3) / 1e9,
        "frac_of_8tbs_nominal": nominal / (ms * 1e-3) / 1e9 / NOMINAL_PEAK_GBS,
        "step_algorithmic_bytes": step_alg,
        "step_gbs_algorithmic": step_alg / (ms * 1e-3) / 1e9,
        "mean_accept_len": float(al_h.float().mean()),
        "emitted_tokens_per_s": world * float(al_h.sum()) / (ms * 1e-3),
        "roofline": {"kernel": "stats_decide_kernel (logits stream)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _traffic("stats_decide_kernel"),
                     "algorithmic_bytes_per_launch": pass1_alg, "ms_per_launch": kms},
        "cpu_baseline": cpu,
        "e2e": {"value": world * units / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "clocks": clk,
        "gpu_launches": launches,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
