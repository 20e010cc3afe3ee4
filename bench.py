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


# the sources each profiled kernel is built from (its own file and the shared device headers)
KERNEL_SOURCES = {
    "fused_kernel": ("verify.cu", "sv_args.cuh", "sv_device.cuh", "sv_draw.cuh", "sv_host.h"),
    "lmhead_gemm_kernel": ("lmhead.cu", "sv_device.cuh", "sv_draw.cuh", "sv_host.h", "sv_slice.cuh"),
    "cluster_kernel": ("cluster.cu", "sv_args.cuh", "sv_device.cuh", "sv_draw.cuh", "sv_host.h", "sv_slice.cuh"),
}
KERNEL_SOURCES["fused_kernel_ragged"] = KERNEL_SOURCES["fused_kernel"]  # the same kernel, its ragged capture
KERNEL_SOURCES["lmhead_gemm_kernel_draft"] = KERNEL_SOURCES["lmhead_gemm_kernel"]  # the draft head's capture
KERNEL_SOURCES["ngram_kernel"] = ("ngram.cu", "sv_device.cuh", "sv_host.h")


def _source_hash(kernel: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_11_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the kernel's current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(kernel)
        if rec and rec.get("source_hash") == _source_hash(kernel):
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


def _max_over_ranks(values, device):
    """Each rank's timings -> the maximum over ranks of each (the slowest rank
    sets the job's time); a no-op on one rank."""
    import torch
    if int(os.environ.get("WORLD_SIZE", "1")) <= 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def _job_value(world, units_per_rank, ms):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (ms * 1e-3)


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


def _cpu_sample_all_cores(batch, target_s=10.0):
    """The same oracle on every host core: one thread per core, each verifying
    the same 16 requests repeatedly for ~target_s (the C oracle keeps no shared
    state, and ctypes releases the GIL during the call)."""
    import concurrent.futures as cf
    import oracle
    n_req = 16
    rows = n_req * (batch.K + 1)
    z, q = batch.logits[:rows], batch.q[: n_req * batch.K]
    x, u = batch.draft[: n_req * batch.K], batch.uniforms[:rows]
    cores = os.cpu_count() or 1
    oracle.verify_fixed(z, q, x, u, n_req, batch.K, batch.temperature)  # builds and loads the library once
    t0 = time.perf_counter()
    deadline = t0 + target_s

    def work():
        reps = 0
        while time.perf_counter() < deadline:
            oracle.verify_fixed(z, q, x, u, n_req, batch.K, batch.temperature)
            reps += 1
        return reps

    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        reps = sum(f.result() for f in [ex.submit(work) for _ in range(cores)])
    el = time.perf_counter() - t0
    return {"value": reps * n_req * batch.K / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {n_req} of 64 requests on each of {cores} threads, {reps} verifications in "
                      f"{el:.1f} s, fp64 C"}


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

    # Default: the K steps run back to back between one pair of events (the
    # kernel is the whole step, launched with programmatic stream serialization,
    # so nothing may sit between two launches).  With --l2-flush every step is
    # bracketed by its own events, its flush outside them.
    n_ev = args.steps if args.l2_flush else 1
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
    for evs in ev:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    # The same C call every step, marshalled once, so that the host stays ahead of the
    # GPU.  Without a flush, consecutive steps read different resident copies of the
    # inputs: the kernel keeps some logits rows in L2 for its own residual pass, and
    # the next step must not find them there.
    copies = [(logits, q)]
    if not args.l2_flush:
        for _ in range(args.copies - 1):
            copies.append((logits.clone(), q.clone()))
    calls = [B_.bind_spec_verify_sample(lg, qq, Bn, K, V, T, draft, uni, out, al, ws, stream=stream)
             for lg, qq in copies]
    call = calls[0]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    if args.l2_flush:
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
    else:
        for c in calls:  # touch every copy once outside the timed region
            c()
        ev[0][0].record(stream)
        for i in range(args.steps):
            calls[i % len(calls)]()
        ev[0][1].record(stream)
    launches = args.steps * B_.spec_last_launch_count()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if args.l2_flush:
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    else:
        ms = ev[0][0].elapsed_time(ev[0][1]) / args.steps
    kms = ms * args.steps / launches  # one kernel per step: its mean duration, launch gap included
    ms, kms = _max_over_ranks([ms, kms], dev)

    # outcome of the step (same every step: same inputs)
    al_h = al.cpu()
    n_reject = int((al_h <= K).sum())
    units = Bn * K
    value = _job_value(world, units, ms)
    nominal = W.nominal_bytes(batch)
    logits_bytes = R * V * 4
    gathers = Bn * K * 16 + R * 4 + Bn * 4
    # one fused kernel runs the whole step: logits once, the drafts' gathers,
    # and the q row of every request that rejected (re-reading the selected
    # logits row for the residual is the method's second pass, not counted)
    step_alg = logits_bytes + gathers + n_reject * V * 4
    kernel_alg = step_alg
    peak, peak_kind = _peaks()
    achieved = kernel_alg / (kms * 1e-3) / 1e9

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
    e2e_ms = _max_over_ranks([e2e_ms], dev)[0]

    cpu = _cpu_sample(batch) if (rank == 0 and world == 1 and not args.no_cpu) else None
    cpu_all = _cpu_sample_all_cores(batch) if (rank == 0 and world == 1 and not args.no_cpu) else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": Bn, "K": K, "V": V, "T": T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": ("flushed between steps (256 MB write)" if args.l2_flush else
                          f"no flush: steps run back to back over {len(calls)} resident copies of the inputs "
                          f"({len(calls) * 295.5:.0f} MB), so no step reads what the step before it read")},
        "hbm_gbs_nominal": world * nominal / (ms * 1e-3) / 1e9,
        "frac_of_8tbs_nominal": nominal / (ms * 1e-3) / 1e9 / NOMINAL_PEAK_GBS,
        "step_algorithmic_bytes": step_alg,
        "step_gbs_algorithmic": step_alg / (ms * 1e-3) / 1e9,
        "mean_accept_len": float(al_h.float().mean()),
        "emitted_tokens_per_s": world * float(al_h.sum()) / (ms * 1e-3),
        "roofline": {"kernel": "fused_kernel (whole step)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _traffic("fused_kernel"),
                     "algorithmic_bytes_per_launch": kernel_alg, "ms_per_launch": kms},
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": {"value": _job_value(world, units, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "clocks": clk,
        "gpu_launches": launches,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_lmhead(args):
    """Fused LM-head + verify, B=16 K=7 (128 rows) d=8192 V=128256, T=1, plus
    the pages' speedup closed form from measured times."""
    import torch
    import oracle
    from oracle import speedup as SP
    from speculative_decoding_verification_11_gb300 import binding as B_, build as build_mod, workloads as W
    world, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build_mod.build()
    B_.load()
    batch = W.lmhead()
    Bn, K, V, T = batch.B, batch.K, batch.V, batch.temperature
    d = batch.hidden.shape[1]
    M = batch.rows
    h, w = batch.hidden.to(dev), batch.w_vocab_t.to(dev)
    q, x, u = batch.q.to(dev), batch.draft.to(dev), batch.uniforms.to(dev)
    out = torch.empty(M, dtype=torch.int32, device=dev)
    al = torch.empty(Bn, dtype=torch.int32, device=dev)
    ws = B_.workspace(B_.spec_lmhead_workspace_size(Bn, K, d, V), dev)
    stream = torch.cuda.current_stream(dev)
    # plain decoding step of the same batch: one row per request (K = 0)
    h0 = h.view(Bn, K + 1, d)[:, 0].contiguous()
    u0 = u.view(Bn, K + 1)[:, 0].contiguous()
    out0 = torch.empty(Bn, dtype=torch.int32, device=dev)
    al0 = torch.empty(Bn, dtype=torch.int32, device=dev)
    x0 = torch.empty(0, dtype=torch.int32, device=dev)
    ws0 = B_.workspace(B_.spec_lmhead_workspace_size(Bn, 0, d, V), dev)
    # stand-in draft model step: the draft head GEMM at M = B (cuBLAS) + softmax
    hd = torch.randn(Bn, 2048, device=dev).to(torch.bfloat16)
    wd = (torch.randn(V, 2048, device=dev) * 0.02).to(torch.bfloat16)

    def spec_step():
        B_.spec_lmhead_verify(h, w, d, q, Bn, K, V, T, x, u, out, al, ws, stream=stream)

    def plain_step():
        B_.spec_lmhead_verify(h0, w, d, None, Bn, 0, V, T, x0, u0, out0, al0, ws0, stream=stream)

    def draft_step():
        torch.softmax((hd @ wd.T).float(), dim=-1)

    def timed(fn, n, prof=False):
        """n steps back to back between one pair of events (W, 2.1 GB, is far
        beyond L2); with prof, the GEMM of every step is bracketed by its own
        events through the library's profiling hook.  Returns ([mean step ms],
        [GEMM ms per step])."""
        ks_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for a, b in ks_ev:
            a.record(stream)
            b.record(stream)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            if prof:
                B_.spec_profile_set_events(ks_ev[i][0], ks_ev[i][1])
            fn()
        e1.record(stream)
        if prof:
            B_.spec_profile_set_events(None, None)
        torch.cuda.synchronize()
        ks = [a.elapsed_time(b) for a, b in ks_ev] if prof else []
        return [e0.elapsed_time(e1) / n], ks

    for fn in (spec_step, plain_step, draft_step):
        for _ in range(max(args.warmup, 3)):
            fn()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    ts, _ = timed(spec_step, args.steps)  # events inside the step would serialise it: step time alone
    _, ks = timed(spec_step, args.steps, prof=True)
    clk = clocks.stop()
    ms = statistics.mean(ts)
    kms = statistics.mean(ks)
    t_plain = statistics.median(timed(plain_step, max(5, args.steps // 2))[0])
    t_draft1 = statistics.median(timed(draft_step, max(5, args.steps // 2))[0])
    al_mean = float(al.float().mean())
    # directly timed: round(AL) plain steps against one speculative step + K draft steps
    n_plain = max(1, int(round(al_mean)))

    def plain_loop():
        for _ in range(n_plain):
            plain_step()

    def spec_cycle():
        for _ in range(K):
            draft_step()
        spec_step()

    t_plain_loop = statistics.median(timed(plain_loop, 5)[0])
    t_spec_cycle = statistics.median(timed(spec_cycle, 5)[0])
    w_bytes = V * d * 2
    gemm_bytes = w_bytes + M * d * 2 + M * V * 4 + M * ((V + 255) // 256) * 8
    flops = 2.0 * M * d * V
    peak, pk = _peaks()
    tpk, tpk_kind = _peak_tflops()
    achieved = gemm_bytes / (kms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": Bn * K / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 GEMM, f32 verify", "data": "synthetic",
        "config": {"workload": "fused LM-head + verify B=16 K=7 (128 rows) d=8192 V=128256 T=1", "B": Bn,
                   "K": K, "V": V, "d": d, "l2": "inputs 2.1 GB > L2"},
        "roofline": {"kernel": "lmhead_gemm_kernel (tcgen05, W stream)", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "peak_kind": pk, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": _traffic("lmhead_gemm_kernel"), "algorithmic_bytes_per_launch": gemm_bytes,
                     "ms_per_launch": kms,
                     "tensor": {"achieved_tflops": flops / (kms * 1e-3) / 1e12, "peak_tflops": tpk,
                                "peak_kind": tpk_kind, "frac": flops / (kms * 1e-3) / 1e12 / tpk}},
        "speedup_model": {
            "T_verif_B_ms": t_plain, "T_verif_B1D_ms": ms, "T_draft_ms": K * t_draft1, "AL": al_mean,
            "closed_form": SP.measured_speedup(t_plain, ms, K * t_draft1, al_mean),
            "direct": {"plain_steps": n_plain, "plain_loop_ms": t_plain_loop, "spec_cycle_ms": t_spec_cycle,
                       "ratio": t_plain_loop / t_spec_cycle},
            "draft_stand_in": "draft head GEMM (B x 2048 . 2048 x V, bf16, cuBLAS) + softmax per drafted token"},
        "clocks": clk,
        "gpu_launches": 3 * args.steps,
    }
    if not args.no_cpu:
        t0 = time.perf_counter()
        oracle.lmhead_verify(batch.hidden, batch.w_vocab_t, batch.q, batch.draft, batch.uniforms, Bn, K, T)
        el = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": Bn * K / el, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"whole batch once: fp64 GEMM (numpy BLAS, all cores) + C verify, {el:.1f} s"}
    print(json.dumps(line), flush=True)
    return 0


def _alg_bytes(batch, al, n_rows_out):
    """Algorithmic bytes of one verification call: every logit once, 16 B per
    draft (z[x], q[x], x, u), the q row of every request that rejected (its
    residual), and 4 B per output row and request."""
    import torch
    esize = 2 if batch.logits.dtype == torch.bfloat16 else 4
    R, V = batch.rows, batch.V
    nq = R - batch.B
    k_i = (batch.row_offsets[1:] - batch.row_offsets[:-1] - 1).to(al.device)
    rejected = int((al.to(torch.int64) <= k_i).sum()) if batch.q is not None else 0
    return R * V * esize + nq * 16 + rejected * V * 4 + (n_rows_out + batch.B) * 4


def run_config(args):
    """The other workloads of the scope table, each a single JSON line:
    greedy (B=32 K=5 V=32000 bf16), ragged (B=256, K_i ~ U{0..8}, V=151936),
    tiny (B=1 K=4 V=1024: 1000 calls captured in one CUDA graph, and the same
    1000 requests as one call)."""
    import torch
    from speculative_decoding_verification_11_gb300 import build, binding as B_, workloads as W
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    batch = {"greedy": W.greedy, "ragged": W.ragged, "tiny": W.tiny}[args.config]()
    Bn, V, R = batch.B, batch.V, batch.rows
    logits = batch.logits.to(dev)
    draft = batch.draft.to(dev)
    q = batch.q.to(dev) if batch.q is not None else None
    uni = batch.uniforms.to(dev) if batch.uniforms is not None else None
    offs = batch.row_offsets.to(dev)
    out = torch.empty(R, dtype=torch.int32, device=dev)
    al = torch.empty(Bn, dtype=torch.int32, device=dev)
    ws = B_.workspace(B_.spec_verify_workspace_size(Bn, R, V), dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (logits, q) if t is not None)
    small = in_bytes < 2 * (129 << 20)
    # inputs smaller than twice L2: steps rotate over enough copies that no step finds the bytes
    # an earlier step read in L2 (or, with --l2-flush, L2 is flushed before every timed call)
    n_copies = 1 if (not small or args.l2_flush) else -(-2 * (129 << 20) // in_bytes) + 1
    copies = [(logits, q)] + [(logits.clone(), q.clone() if q is not None else None) for _ in range(n_copies - 1)]
    k_step = [0]

    def step_on(st):
        lg, qq = copies[k_step[0] % n_copies]
        k_step[0] += 1
        if args.config == "greedy":
            B_.spec_verify_greedy(lg, draft, Bn, batch.K, V, out, al, ws, stream=st)
        elif args.config == "ragged":
            B_.spec_verify_ragged(lg, qq, offs, Bn, R, V, batch.temperature, draft, uni, out, al, ws,
                                  stream=st)
        else:
            B_.spec_verify_sample(lg, qq, Bn, batch.K, V, batch.temperature, draft, uni, out, al, ws,
                                  stream=st)

    def step():
        step_on(stream)

    # inputs that fit in L2 are evicted before every timed call: a 256 MB write,
    # then a 256 MB read so that no dirty line is left to be written back inside
    # the timed call
    flush = small and args.l2_flush
    fw = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    fr = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    for _ in range(max(args.warmup, 3, n_copies)):
        step()
    torch.cuda.synchronize()
    n0 = B_.spec_last_launch_count()
    kernel_used = B_.spec_last_kernel()
    clocks = Clocks(0)
    clocks.start()
    if flush:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            fw.fill_(float(i))
            fr.sum()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        l2 = f"inputs {in_bytes / 1e6:.1f} MB < L2: 256 MB write then 256 MB read before every call, outside its events"
    else:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        l2 = (f"inputs {in_bytes / 1e6:.1f} MB > L2 (129 MB), no flush: calls back to back" if not small else
              f"inputs {in_bytes / 1e6:.1f} MB x {n_copies} rotating copies > 2 x L2, no flush: calls back to back")
        if small:
            # a short kernel can be limited by the host's launch rate: the same steps (same copies,
            # same launches) captured in one CUDA graph and replayed time the device alone
            ms_stream = ms
            gs = torch.cuda.Stream(dev)
            gs.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gs):
                k_step[0] = 0
                for _ in range(args.steps):
                    step_on(gs)
            g.replay()  # on the current stream
            torch.cuda.synchronize()
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            l2 += f"; the {args.steps} steps replayed from one CUDA graph ({ms_stream * 1e3:.2f} us per step when launched one by one)"
    clk = clocks.stop()
    alg = _alg_bytes(batch, al, R)
    drafts = R - Bn
    peak, peak_kind = _peaks()
    achieved = alg / (ms * 1e-3) / 1e9
    line = {
        "metric": "verified draft tokens/s", "value": drafts / (ms * 1e-3), "unit": "verified draft tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if logits.dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": {"workload": f"{args.config} verify B={Bn} rows={R} V={V} T={batch.temperature}", "l2": l2},
        "mean_accept_len": float(al.float().mean()),
        "roofline": {"kernel": {"small": "sk::small_kernel", "cluster": "cv::cluster_kernel", "stream": "fused_kernel",
                                "scalar": "stats_scalar_kernel + residual_kernel"}.get(kernel_used, kernel_used) +
                               " (whole step)", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     # committed captures exist for the greedy workload (cluster kernel) and the ragged
                     # one (streaming kernel); tiny has none
                     "traffic": (_traffic("cluster_kernel") if (args.config == "greedy" and kernel_used == "cluster")
                                 else _traffic("fused_kernel_ragged") if (args.config == "ragged" and kernel_used == "stream")
                                 else None),
                     "algorithmic_bytes_per_launch": alg, "ms_per_launch": ms},
        "clocks": clk, "gpu_launches": args.steps * n0,
    }
    if args.config == "tiny":
        # 1000 B=1 calls captured in one CUDA graph, replayed: latency per call
        n_req = Bn
        ws1 = B_.workspace(B_.spec_verify_workspace_size(1, 5, V), dev)
        gs = torch.cuda.Stream(dev)
        out1 = torch.empty(R, dtype=torch.int32, device=dev)
        al1 = torch.empty(n_req, dtype=torch.int32, device=dev)
        calls = [B_.bind_spec_verify_sample(logits[5 * i:5 * i + 5], q[4 * i:4 * i + 4], 1, 4, V,
                                            batch.temperature, draft[4 * i:4 * i + 4], uni[5 * i:5 * i + 5],
                                            out1[5 * i:5 * i + 5], al1[i:i + 1], ws1, stream=gs)
                 for i in range(n_req)]
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            for c in calls[:3]:
                c()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            for c in calls:
                c()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out1, out) and torch.equal(al1, al), "graph of B=1 calls differs from one B=1000 call"
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * n_req)
        line["graph_b1"] = {"calls": n_req, "us_per_call": us, "verified_draft_tokens_per_s": 4 / (us * 1e-6),
                            "note": "1000 B=1 calls in one CUDA graph, replayed 5 times; inputs stay in L2"}
    print(json.dumps(line), flush=True)
    return 0


def run_kv(args):
    """KV-cache bookkeeping after verification: spec_kv_reserve then
    spec_kv_rollback with every draft rejected (accept length 1: the most
    blocks returned), which leaves the cache as it was, so steps repeat on the
    same state.  K = 4 drafts per request, 16-token blocks, lengths up to 4096."""
    import numpy as np
    import torch
    from speculative_decoding_verification_11_gb300 import build, binding as B_
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    clocks = Clocks(0)
    clocks.start()
    for Bn in (64, 4096):
        rng = np.random.default_rng(7 + Bn)
        bs, K, max_blocks = 16, 4, 264
        seq = rng.integers(1, 4096, size=Bn).astype(np.int32)
        n_ids = Bn * max_blocks
        ids = rng.permutation(n_ids).astype(np.int32)
        bt = np.full((Bn, max_blocks), -1, dtype=np.int32)
        k = 0
        for b in range(Bn):
            nb = -(-int(seq[b]) // bs)
            bt[b, :nb] = ids[k:k + nb]
            k += nb
        free = np.full(n_ids, -1, dtype=np.int32)
        free[:n_ids - k] = ids[k:]
        g_bt = torch.from_numpy(bt).to(dev)
        g_seq = torch.from_numpy(seq).to(dev)
        g_free = torch.from_numpy(free).to(dev)
        g_fc = torch.tensor([n_ids - k], dtype=torch.int32, device=dev)
        g_K = torch.full((Bn,), K, dtype=torch.int32, device=dev)
        g_al = torch.ones(Bn, dtype=torch.int32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)

        def step():
            B_.spec_kv_reserve(g_bt, g_seq, g_free, g_fc, g_K, bs, st, stream=stream)
            B_.spec_kv_rollback(g_bt, g_seq, g_free, g_fc, g_K, g_al, bs, st, stream=stream)

        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize()
        # launch-bound: the K steps are captured in one CUDA graph
        g = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        with torch.cuda.graph(g, stream=gs):
            for _ in range(args.steps):
                B_.spec_kv_reserve(g_bt, g_seq, g_free, g_fc, g_K, bs, st, stream=gs)
                B_.spec_kv_rollback(g_bt, g_seq, g_free, g_fc, g_K, g_al, bs, st, stream=gs)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        assert st.item() == 0 and np.array_equal(g_bt.cpu().numpy(), bt), "state must return to itself"
        new_blocks = sum(-(-(int(s) + K) // bs) - (-(-int(s) // bs)) for s in seq)
        # bytes: lengths and counts read twice, accept lengths, touched table entries
        # (checked, then written), free-list slots (read, then written)
        alg = Bn * 4 * 5 + new_blocks * 4 * 6
        res[f"B={Bn}"] = {"us_per_step": ms * 1e3, "blocks_moved_per_step": 2 * new_blocks,
                          "algorithmic_bytes": alg, "achieved_gbs": alg / (ms * 1e-3) / 1e9}
    clk = clocks.stop()
    peak, peak_kind = _peaks()
    head = res["B=64"]
    line = {
        "metric": "KV bookkeeping steps/s (reserve + rollback)", "value": 1e6 / head["us_per_step"],
        "unit": "steps/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": head["us_per_step"] * 1e-3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": "paged KV reserve + rollback, B=64 and 4096, K=4, 16-token blocks, "
                               "every draft rejected", "l2": "state stays in L2 (launch-bound, one CTA)"},
        "roofline": {"kernel": "kvb::reserve_kernel + kvb::rollback_kernel", "bound": "hbm",
                     "achieved": head["achieved_gbs"], "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": head["achieved_gbs"] / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": head["algorithmic_bytes"] / 2,
                     "ms_per_launch": head["us_per_step"] * 1e-3 / 2,
                     "note": "latency-bound: one CTA and two dependent launches per step"},
        "batches": res, "clocks": clk, "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_draft(args):
    """Draft head + draft sampling at the fused workload's draft head: M = 128
    rows (16 requests x 8 positions), d = 2048, V = 128256, T = 1: the tcgen05
    GEMM writes fp32 logits into q's buffer, then one CTA per row turns them
    into q and draws x with Philox."""
    import torch
    from speculative_decoding_verification_11_gb300 import build, binding as B_
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    M, d, V, T = 128, 2048, 128256, 1.0
    g = torch.Generator().manual_seed(1005)
    h = torch.randn(M, d, generator=g).to(torch.bfloat16).to(dev)
    w = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16).to(dev)
    q = torch.empty(M, V, device=dev)
    x = torch.empty(M, dtype=torch.int32, device=dev)
    ws = B_.workspace(B_.spec_draft_workspace_size(M, d, V), dev)
    for i in range(max(args.warmup, 3)):
        B_.spec_draft_sample(h, w, T, 1005, i * M, q, x, ws, stream=stream)
    torch.cuda.synchronize()
    # steps back to back between one pair of events (W, 525 MB, is beyond L2); the GEMM's own time
    # from a second pass with the library's profiling events around every GEMM launch (events
    # between the two launches of a step would serialise it)
    clocks = Clocks(0)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        B_.spec_draft_sample(h, w, T, 1005, (100 + i) * M, q, x, ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in kev:  # torch measures only events it has recorded itself once
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        B_.spec_profile_set_events(kev[i][0], kev[i][1])
        B_.spec_draft_sample(h, w, T, 1005, (100 + i) * M, q, x, ws, stream=stream)
    B_.spec_profile_set_events(None, None)
    torch.cuda.synchronize()
    clk = clocks.stop()
    gms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    peak, peak_kind = _peaks()
    tpk, tpk_kind = _peak_tflops()
    gemm_bytes = V * d * 2 + M * d * 2 + M * V * 4  # W, hidden, fp32 logits written
    flops = 2 * M * d * V
    finish_bytes = 2 * M * V * 4                     # logits read, q written
    line = {
        "metric": "drafted tokens/s (draft head GEMM + q + Philox draw)", "value": M / (ms * 1e-3),
        "unit": "drafted tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"draft head M={M} d={d} V={V} T={T} bf16 weights, fp32 q",
                   "l2": "inputs 525 MB > L2, no flush"},
        "roofline": {"kernel": "lmhead_gemm_kernel (draft head)", "bound": "hbm",
                     "achieved": gemm_bytes / (gms * 1e-3) / 1e9, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": gemm_bytes / (gms * 1e-3) / 1e9 / peak,
                     "traffic": _traffic("lmhead_gemm_kernel_draft"),
                     "algorithmic_bytes_per_launch": gemm_bytes, "ms_per_launch": gms,
                     "tensor": {"achieved_tflops": flops / (gms * 1e-3) / 1e12, "peak_tflops": tpk,
                                "peak_kind": tpk_kind, "frac": flops / (gms * 1e-3) / 1e12 / tpk}},
        "finish": {"ms": ms - gms, "algorithmic_bytes": finish_bytes,
                   "achieved_gbs": finish_bytes / ((ms - gms) * 1e-3) / 1e9},
        "clocks": clk, "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ngram(args):
    """Model-free n-gram (prompt lookup) drafting over synthetic streams with
    repetition: B = 256 contexts of L tokens (L = 8192 and 32768), K = 8,
    n in [1, 4].  The contexts fit in L2, so calls rotate over copies whose
    total exceeds twice L2, replayed back to back from a CUDA graph."""
    import torch
    from speculative_decoding_verification_11_gb300 import build, binding as B_, workloads as W
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    fw = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if args.l2_flush else None
    fr = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if args.l2_flush else None
    res = {}
    B, K, n_min, n_max = 256, 8, 1, 4
    clocks = Clocks(0)
    clocks.start()
    for L in (8192, 32768):
        tokens, offs = W.repetitive_streams(seed=1006, B=B, L=L)
        t = torch.from_numpy(tokens).to(dev)
        o = torch.from_numpy(offs).to(dev)
        d = torch.empty(B, K, dtype=torch.int32, device=dev)
        k = torch.empty(B, dtype=torch.int32, device=dev)
        # the contexts fit in L2: calls rotate over enough copies that none finds bytes an earlier
        # call read, and the calls are replayed from one CUDA graph (each call's own launch is short
        # next to the host's launch rate); with --l2-flush, L2 is flushed before every timed call
        in_bytes = t.numel() * 4
        n_copies = 1 if args.l2_flush else -(-2 * (129 << 20) // in_bytes) + 1
        copies = [t] + [t.clone() for _ in range(n_copies - 1)]
        for i in range(max(args.warmup, 3, n_copies)):
            B_.spec_ngram_draft(copies[i % n_copies], o, K, n_min, n_max, d, k, stream=stream)
        torch.cuda.synchronize()
        if args.l2_flush:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for i in range(args.steps):
                fw.fill_(float(i))
                fr.sum()
                ev[i][0].record(stream)
                B_.spec_ngram_draft(t, o, K, n_min, n_max, d, k, stream=stream)
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        else:
            gs = torch.cuda.Stream(dev)
            gs.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gs):
                for i in range(args.steps):
                    B_.spec_ngram_draft(copies[i % n_copies], o, K, n_min, n_max, d, k, stream=gs)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
        kh = k.cpu()
        alg = B * L * 4 + (B + 1) * 4 + B * K * 4 + B * 4
        res[f"L={L}"] = {"us_per_call": ms * 1e3, "requests_per_s": B / (ms * 1e-3),
                         "mean_draft_len": float(kh.float().mean()), "with_proposal": float((kh > 0).float().mean()),
                         "algorithmic_bytes": alg, "achieved_gbs": alg / (ms * 1e-3) / 1e9}
    clk = clocks.stop()
    peak, peak_kind = _peaks()
    head = res["L=8192"]
    line = {
        "metric": "n-gram drafting requests/s", "value": head["requests_per_s"], "unit": "requests/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": head["us_per_call"] * 1e-3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": f"prompt-lookup drafting B={B} K={K} n={n_min}..{n_max} over repetitive streams",
                   "l2": ("contexts < L2: 256 MB write then 256 MB read before every call, outside its events"
                          if args.l2_flush else
                          "contexts < L2: calls rotate over copies > 2 x L2, replayed back to back from a CUDA graph")},
        "roofline": {"kernel": "ng::ngram_kernel", "bound": "hbm", "achieved": head["achieved_gbs"], "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": head["achieved_gbs"] / peak, "traffic": _traffic("ngram_kernel"),
                     "algorithmic_bytes_per_launch": head["algorithmic_bytes"],
                     "ms_per_launch": head["us_per_call"] * 1e-3},
        "lengths": res, "clocks": clk, "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_dynk(args):
    """Dynamic-K controller after verification (goodput rule, 10-result rings,
    K in [1, 8], row offsets for the next ragged verification), B = 64 and
    4096, captured in a CUDA graph (the update is launch-bound)."""
    import torch
    from speculative_decoding_verification_11_gb300 import build, binding as B_
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    clocks = Clocks(0)
    clocks.start()
    for Bn in (64, 4096):
        g = torch.Generator().manual_seed(Bn)
        al = torch.randint(1, 6, (Bn,), generator=g, dtype=torch.int32).to(dev)
        ku = torch.full((Bn,), 5, dtype=torch.int32, device=dev)
        hist = torch.zeros(Bn, 10, 2, dtype=torch.int32, device=dev)
        count = torch.zeros(Bn, dtype=torch.int32, device=dev)
        kn = torch.empty(Bn, dtype=torch.int32, device=dev)
        offs = torch.empty(Bn + 1, dtype=torch.int32, device=dev)
        itl = (10.0 + 1.5 * torch.arange(9, dtype=torch.float32)).to(dev)
        for _ in range(max(args.warmup, 3)):
            B_.spec_dynk_update(al, ku, hist, count, B_.SV_DYNK_GOODPUT, 1, 8, kn, itl=itl, row_offsets=offs,
                                stream=stream)
        torch.cuda.synchronize()
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(args.steps):
                B_.spec_dynk_update(al, ku, hist, count, B_.SV_DYNK_GOODPUT, 1, 8, kn, itl=itl, row_offsets=offs,
                                    stream=gs)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / args.steps
        alg = Bn * (4 * 4 + 10 * 8 + 8) + 9 * 4  # AL, K used, count, k_next; the ring read (and one pair written); offsets
        res[f"B={Bn}"] = {"us_per_update": us, "algorithmic_bytes": alg, "achieved_gbs": alg / (us * 1e-6) / 1e9,
                          "mean_k_next": float(kn.float().mean())}
    clk = clocks.stop()
    peak, peak_kind = _peaks()
    head = res["B=64"]
    line = {
        "metric": "dynamic-K controller updates/s", "value": 1e6 / head["us_per_update"], "unit": "updates/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": head["us_per_update"] * 1e-3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32/f32", "data": "synthetic",
        "config": {"workload": "goodput rule, W=10, K in [1, 8], B=64 and 4096, offsets for ragged verification",
                   "l2": "state stays in L2 (launch-bound, one CTA)"},
        "roofline": {"kernel": "dk::dynk_kernel", "bound": "hbm", "achieved": head["achieved_gbs"], "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": head["achieved_gbs"] / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": head["algorithmic_bytes"],
                     "ms_per_launch": head["us_per_update"] * 1e-3,
                     "note": "latency-bound: one CTA per update, in a CUDA graph"},
        "batches": res, "clocks": clk, "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--l2-flush", action="store_true",
                    help="write a 256 MB buffer before every timed step (its dirty lines are written back "
                         "during the next step); by default the inputs, larger than L2, stand in for a flush")
    ap.add_argument("--copies", type=int, default=3,
                    help="resident copies of the inputs the back-to-back steps rotate over (no flush)")
    ap.add_argument("--config", choices=["sampling", "lmhead", "greedy", "ragged", "tiny", "kv", "draft", "ngram", "dynk"], default="sampling",
                    help="sampling: the headline workload; lmhead: the fused LM-head front end; "
                         "greedy / ragged / tiny: the other verification workloads")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.config == "lmhead":
        return run_lmhead(args)
    if args.config in ("greedy", "ragged", "tiny"):
        return run_config(args)
    if args.config == "kv":
        return run_kv(args)
    if args.config == "draft":
        return run_draft(args)
    if args.config == "ngram":
        return run_ngram(args)
    if args.config == "dynk":
        return run_dynk(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
