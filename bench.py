"""Benchmark of the verification step on GB300.

Default workload (the configuration the headline metric is quoted on):
sampling verification, B=64 requests, K=4 drafts, V=128256, fp32 logits,
T=0.7.  One step = one spec_verify_sample call over the resident batch (the
whole hot path: logits stream, decisions, residual, draw).  Metric: verified
draft tokens/s (B K per step) and the HBM bandwidth implied by reading logits
+ q once.

The default run prints ONE JSON line: the headline's measurement, and under
"workloads" every other configuration of the scope (tiny, greedy, fused
LM-head, ragged) and the serving-loop steps around it (KV rollback, draft
head, n-gram drafting, dynamic K), each with its own step time, roofline,
clock samples and a parity count of a bounded sample of its outputs against
the oracle (the sample its cpu_baseline times).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config NAME]   (one workload alone, one line)

N > 1 (torchrun): every rank verifies its own batch (requests are
independent, no collective on the data path; replicas, weak scaling); the
other workloads run on one GPU only.
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
L2_BYTES = 129 << 20
L2_FLUSH_BYTES = 256 << 20
NOMINAL_PEAK_GBS = 8000.0
SUSTAIN_S = 2.0          # headline: seconds of back-to-back steps ahead of the timed K steps (--sustain)
SUSTAIN_S_OTHER = 0.4    # every other workload (scaled with --sustain)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


# the sources each profiled kernel is built from (its own file and the shared device headers)
KERNEL_SOURCES = {
    "fused_kernel": ("verify.cu", "sv_args.cuh", "sv_device.cuh", "sv_draw.cuh", "sv_host.h"),
    "lmhead_gemm_kernel": ("lmhead.cu", "sv_args.cuh", "sv_device.cuh", "sv_draw.cuh", "sv_host.h", "sv_slice.cuh"),
    "cluster_kernel": ("cluster.cu", "sv_args.cuh", "sv_device.cuh", "sv_draw.cuh", "sv_host.h", "sv_slice.cuh"),
}
KERNEL_SOURCES["fused_kernel_ragged"] = KERNEL_SOURCES["fused_kernel"]  # the same kernel, its ragged capture
KERNEL_SOURCES["lmhead_gemm_kernel_draft"] = KERNEL_SOURCES["lmhead_gemm_kernel"]  # the draft head's capture
KERNEL_SOURCES["ngram_kernel"] = ("ngram.cu", "sv_args.cuh", "sv_device.cuh", "sv_host.h")
KERNEL_SOURCES["small_kernel"] = ("small.cu", "sv_args.cuh", "sv_device.cuh", "sv_draw.cuh", "sv_host.h")


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
    """Samples nvidia-smi every 200 ms while a measured region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

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
        return self

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
        sm, smax, reasons, busy = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                busy += float(parts[9]) > 0
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "samples_busy": busy}


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


def _events(n=1):
    import torch
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]


def _spacer(us=60.0):
    """Keeps the GPU busy for ~us (a spin kernel on the current stream) ahead of a
    timed region's start event, so that by the time the GPU reaches the event
    the host has already enqueued the first timed launches: the host's launch
    latency then stays outside the region.  No-op where torch lacks the spin."""
    import torch
    try:
        torch.cuda._sleep(int(us * 2100))  # SM cycles at ~2.1 GHz
    except Exception:
        pass


def _time_back_to_back(fn, n, stream):
    """n calls of fn back to back between one pair of events: ms per call."""
    import torch
    (e0, e1), = _events()
    _spacer()
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


_SUSTAIN_SCALE = [1.0]


def _sustain(fn, stream, seconds, calls_per_fn=1):
    """About `seconds` of back-to-back calls of fn (the steps of the timed
    region, or a graph replaying them), so that the clock record holds samples
    under load; returns its own step time (None when --sustain 0)."""
    seconds *= _SUSTAIN_SCALE[0]
    if seconds <= 0:
        return None
    t1 = _time_back_to_back(fn, 3, stream)
    n = max(3, min(200000, int(seconds * 1e3 / max(t1, 1e-4))))
    ms = _time_back_to_back(fn, n, stream)
    return {"seconds": n * ms * 1e-3, "steps": n * calls_per_fn, "ms_per_step": ms / calls_per_fn}


def _graph_of(steps_fn, stream):
    """A CUDA graph of the launches steps_fn(stream) issues (replayed for
    launch-bound workloads: the device time of the same steps without the
    host's launch rate)."""
    import torch
    gs = torch.cuda.Stream(stream.device)
    gs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        steps_fn(gs)
    g.replay()
    torch.cuda.synchronize()
    return g


def _roof(kernel, alg_bytes, ms, traffic=None, bound="hbm", note=None):
    peak, kind = _peaks()
    ach = alg_bytes / (ms * 1e-3) / 1e9
    r = {"kernel": kernel, "bound": bound, "achieved": ach, "peak": peak, "peak_kind": kind, "unit": "GB/s",
         "frac": ach / peak, "traffic": traffic, "algorithmic_bytes_per_launch": alg_bytes, "ms_per_launch": ms}
    if note:
        r["note"] = note
    return r


def _decision_parity(out, al, orc, row_offsets, n_req, greedy_ties=None):
    """Requests of the sample whose accepted length and tokens match the
    oracle's, counted: mismatches outside near ties, near ties (the oracle's
    flags; in greedy mode greedy_ties, or none), mismatches among them."""
    import numpy as np
    out, al = np.asarray(out), np.asarray(al)
    ro = np.asarray(row_offsets, dtype=np.int64)
    mism = ties = tie_mism = 0
    for b in range(n_req):
        r0, r1 = ro[b], ro[b + 1]
        same = al[b] == orc["accept_len"][b] and np.array_equal(out[r0:r1], orc["out_tokens"][r0:r1])
        if greedy_ties is not None:
            tie = bool(greedy_ties[b])
        else:
            tie = bool(orc["near_tie_accept"][b] or orc["near_tie_sample"][b]) if "near_tie_accept" in orc else False
        ties += tie
        if not same:
            if tie:
                tie_mism += 1
            else:
                mism += 1
    return {"requests": n_req, "mismatch": mism, "near_ties": ties, "near_tie_mismatch": tie_mism}


def _oracle_timed(fn, min_s=1.0):
    """Runs the oracle call fn until ~min_s of host time: (last result, seconds per call, calls)."""
    reps, t0 = 0, time.perf_counter()
    while True:
        res = fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_s:
            return res, el / reps, reps


def _cpu_sample(batch, target_s=10.0):
    """The oracle as it stands on a bounded sample of the workload: the first
    16 requests, repeated until ~target_s of host time."""
    import oracle
    n_req = 16
    rows = n_req * (batch.K + 1)
    z, q = batch.logits[:rows], batch.q[: n_req * batch.K]
    x, u = batch.draft[: n_req * batch.K], batch.uniforms[:rows]
    res, per, reps = _oracle_timed(lambda: oracle.verify_fixed(z, q, x, u, n_req, batch.K, batch.temperature),
                                   target_s)
    return {"value": n_req * batch.K / per, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {n_req} of 64 requests, {reps} repetitions, {per * reps:.1f} s, fp64 C, 1 thread"}, res


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


def _headline_config(world, args):
    """The headline workload's config, the same dict on both arms (the reference arm times the oracle
    on the workload this arm's GPU steps run, so it reports this arm's config)."""
    n = 1 if args.l2_flush else args.copies
    return {"workload": WORKLOAD, "B": 64, "K": 4, "V": 128256, "T": 0.7,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": ("flushed between steps (256 MB write)" if args.l2_flush else
                   f"no flush: steps run back to back over {n} resident copies of the inputs "
                   f"({n * 295.5:.0f} MB), so no step reads what the step before it read")}


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
            "data": "synthetic", "config": _headline_config(world, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{n_req} of 64 requests per step, fp64 C oracle, 1 thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# The headline workload
# ---------------------------------------------------------------------------
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
    ev = _events(n_ev)
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
    rot = [0]

    def rotating():
        calls[rot[0] % len(calls)]()
        rot[0] += 1

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    # ~2 s of the same steps back to back first: the clock record then holds samples under load,
    # and the timed K steps that follow run on a GPU in its sustained state
    sustained = None if args.l2_flush else _sustain(rotating, stream, SUSTAIN_S)
    if args.l2_flush:
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
    else:
        _spacer()
        ev[0][0].record(stream)
        for i in range(args.steps):
            rotating()
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
    out_h_last = out.cpu()
    units = Bn * K
    value = _job_value(world, units, ms)
    nominal = W.nominal_bytes(batch)
    # one fused kernel runs the whole step.  Algorithmic bytes (the scope table's per-step figure,
    # _alg_bytes): every logit once, the drafts' gathers, and per request its selected logits row (the
    # residual or bonus pass needs the row's normaliser first, so the method reads that row twice)
    # and, after a rejection, that position's q row.  The one-pass count leaves out the second read.
    step_alg = _alg_bytes(batch, al_h, R)
    strict_alg = step_alg - Bn * V * 4
    kernel_alg = step_alg

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
    n_e2e = max(3, min(args.steps, 20))
    e2e_ms = _time_back_to_back(e2e_step, n_e2e, stream)
    e2e_ms = _max_over_ranks([e2e_ms], dev)[0]

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _headline_config(world, args),
        "hbm_gbs_nominal": world * nominal / (ms * 1e-3) / 1e9,
        "frac_of_8tbs_nominal": nominal / (ms * 1e-3) / 1e9 / NOMINAL_PEAK_GBS,
        "step_algorithmic_bytes": step_alg,
        "step_gbs_algorithmic": step_alg / (ms * 1e-3) / 1e9,
        "step_bytes_one_pass": strict_alg,
        "frac_one_pass": strict_alg / (kms * 1e-3) / 1e9 / _peaks()[0],
        "mean_accept_len": float(al_h.float().mean()),
        "emitted_tokens_per_s": world * float(al_h.sum()) / (ms * 1e-3),
        "roofline": _roof("fused_kernel (whole step)", kernel_alg, kms, _traffic("fused_kernel")),
        "sustained": sustained,
        "e2e": {"value": _job_value(world, units, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "clocks": clk,
        "gpu_launches": launches,
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        # the oracle's sample (the first 16 requests), timed as the CPU baseline; its outputs are
        # compared with the timed steps' outputs for the same requests
        line["cpu_baseline"], orc = _cpu_sample(batch)
        line["cpu_baseline_all_cores"] = _cpu_sample_all_cores(batch)
        line["parity"] = _decision_parity(out_h_last.numpy(), al_h.numpy(), orc, batch.row_offsets[:17], 16)
    if world > 1:
        torch.distributed.destroy_process_group()
    del copies, calls, logits, q, flush
    return line


# ---------------------------------------------------------------------------
# The other verification workloads
# ---------------------------------------------------------------------------
def _alg_bytes(batch, al, n_rows_out):
    """Algorithmic bytes of one verification call (the scope table's figure):
    every logit once, 16 B per draft (z[x], q[x], x, u), 4 B per output row and
    request, and in sampling mode each request's selected logits row a second
    time (the residual or bonus pass needs the row's normaliser first) plus the
    q row of every request that rejected."""
    import torch
    esize = 2 if batch.logits.dtype == torch.bfloat16 else 4
    R, V = batch.rows, batch.V
    nq = R - batch.B
    k_i = (batch.row_offsets[1:] - batch.row_offsets[:-1] - 1).to(al.device)
    sampling = batch.q is not None
    rejected = int((al.to(torch.int64) <= k_i).sum()) if sampling else 0
    second = batch.B * V * esize if sampling else 0
    return R * V * esize + nq * 16 + second + rejected * V * 4 + (n_rows_out + batch.B) * 4


KERNEL_NAMES = {"small": "sk::small_kernel", "cluster": "cv::cluster_kernel", "stream": "fused_kernel",
                "scalar": "stats_scalar_kernel + residual_kernel"}


def run_config(args, name):
    """greedy (B=32 K=5 V=32000 bf16), ragged (B=256, K_i ~ U{0..8}, V=151936),
    tiny (B=1 K=4 V=1024, 1000 independent steps: one call over the 1000
    requests, and the same requests as 1000 B=1 calls captured in one CUDA
    graph)."""
    import numpy as np
    import torch
    from speculative_decoding_verification_11_gb300 import build, binding as B_, workloads as W
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    batch = {"greedy": W.greedy, "ragged": W.ragged, "tiny": W.tiny}[name]()
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
    small = in_bytes < 2 * L2_BYTES
    # inputs smaller than twice L2: steps rotate over enough copies that no step finds the bytes
    # an earlier step read in L2 (or, with --l2-flush, L2 is flushed before every timed call)
    n_copies = 1 if (not small or args.l2_flush) else -(-2 * L2_BYTES // in_bytes) + 1
    copies = [(logits, q)] + [(logits.clone(), q.clone() if q is not None else None) for _ in range(n_copies - 1)]
    k_step = [0]

    def step_on(st):
        lg, qq = copies[k_step[0] % n_copies]
        k_step[0] += 1
        if name == "greedy":
            B_.spec_verify_greedy(lg, draft, Bn, batch.K, V, out, al, ws, stream=st)
        elif name == "ragged":
            B_.spec_verify_ragged(lg, qq, offs, Bn, R, V, batch.temperature, draft, uni, out, al, ws, stream=st)
        else:
            B_.spec_verify_sample(lg, qq, Bn, batch.K, V, batch.temperature, draft, uni, out, al, ws, stream=st)

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
    clocks = Clocks(0).start()
    sustained = None
    if flush:
        ev = _events(args.steps)
        for i in range(args.steps):
            fw.fill_(float(i))
            fr.sum()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        l2 = f"inputs {in_bytes / 1e6:.1f} MB < L2: 256 MB write then 256 MB read before every call, outside its events"
    elif not small:
        sustained = _sustain(step, stream, SUSTAIN_S_OTHER)
        ms = _time_back_to_back(step, args.steps, stream)
        l2 = f"inputs {in_bytes / 1e6:.1f} MB > L2 (129 MB), no flush: calls back to back"
    else:
        # a short kernel is limited by the host's launch rate: the same steps (same copies, same
        # launches) captured in one CUDA graph and replayed time the device alone
        ms_stream = _time_back_to_back(step, args.steps, stream)

        def steps_fn(st):
            k_step[0] = 0
            for _ in range(args.steps):
                step_on(st)

        g = _graph_of(steps_fn, stream)
        sustained = _sustain(g.replay, stream, SUSTAIN_S_OTHER, calls_per_fn=args.steps)
        ms = _time_back_to_back(g.replay, 1, stream) / args.steps
        l2 = (f"inputs {in_bytes / 1e6:.1f} MB x {n_copies} rotating copies > 2 x L2, no flush: the {args.steps} "
              f"steps replayed from one CUDA graph ({ms_stream * 1e3:.2f} us per step when launched one by one)")
    clk = clocks.stop()
    torch.cuda.synchronize()
    alg = _alg_bytes(batch, al, R)
    drafts = R - Bn
    traffic = (_traffic("cluster_kernel") if (name == "greedy" and kernel_used == "cluster")
               else _traffic("fused_kernel_ragged") if (name == "ragged" and kernel_used == "stream")
               else _traffic("small_kernel") if (name == "tiny" and kernel_used == "small") else None)
    line = {
        "metric": "verified draft tokens/s", "value": drafts / (ms * 1e-3), "unit": "verified draft tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if logits.dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": {"workload": f"{name} verify B={Bn} rows={R} V={V} T={batch.temperature}", "l2": l2},
        "mean_accept_len": float(al.float().mean()),
        "roofline": _roof(KERNEL_NAMES.get(kernel_used, kernel_used) + " (whole step)", alg, ms, traffic),
        "sustained": sustained, "clocks": clk, "gpu_launches": args.steps * n0,
    }
    out_h, al_h = out.cpu().numpy(), al.cpu().numpy()
    if name == "tiny":
        # 1000 B=1 calls captured in one CUDA graph, replayed: latency per call
        n_req = Bn
        ws1 = B_.workspace(B_.spec_verify_workspace_size(1, 5, V), dev)
        out1 = torch.empty(R, dtype=torch.int32, device=dev)
        al1 = torch.empty(n_req, dtype=torch.int32, device=dev)

        def b1_calls(st):
            for i in range(n_req):
                B_.spec_verify_sample(logits[5 * i:5 * i + 5], q[4 * i:4 * i + 4], 1, 4, V, batch.temperature,
                                      draft[4 * i:4 * i + 4], uni[5 * i:5 * i + 5], out1[5 * i:5 * i + 5],
                                      al1[i:i + 1], ws1, stream=st)

        b1_calls(stream)
        torch.cuda.synchronize()
        g1 = _graph_of(b1_calls, stream)
        assert torch.equal(out1, out) and torch.equal(al1, al), "graph of B=1 calls differs from one B=1000 call"
        us = _time_back_to_back(g1.replay, 5, stream) * 1e3 / n_req
        line["graph_b1"] = {"calls": n_req, "us_per_call": us, "verified_draft_tokens_per_s": 4 / (us * 1e-6),
                            "note": "1000 B=1 calls in one CUDA graph, replayed 5 times; inputs stay in L2"}
    if not args.no_cpu:
        import oracle
        n_req = {"tiny": 100, "greedy": Bn, "ragged": 32}[name]
        ro = batch.row_offsets[:n_req + 1]
        r1 = int(ro[-1])
        nd = r1 - n_req
        greedy = name == "greedy"
        fn = lambda: oracle.verify(batch.logits[:r1], None if greedy else batch.q[:nd], batch.draft[:nd],  # noqa: E731
                                   None if greedy else batch.uniforms[:r1], ro, batch.temperature, greedy=greedy)
        orc, per, reps = _oracle_timed(fn)
        line["cpu_baseline"] = {"value": nd / per, "unit": "verified draft tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"first {n_req} of {Bn} requests, {reps} repetitions, fp64 C, 1 thread"}
        line["parity"] = _decision_parity(out_h, al_h, orc, ro, n_req, greedy_ties=np.zeros(n_req) if greedy else None)
    return line


# ---------------------------------------------------------------------------
# Fused LM-head + verify, and the speedup closed form on the repo's own draft head
# ---------------------------------------------------------------------------
def run_lmhead(args):
    """Fused LM-head + verify, B=16 K=7 (128 rows) d=8192 V=128256, T=1, plus
    the pages' speedup closed form from measured times, the draft step being
    the repo's own draft head (spec_draft_sample at M = B, d = 2048)."""
    import numpy as np
    import torch
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
    # one draft step: the draft head (hidden B x 2048, W 2048 x V, the workload's draft head shape) on the
    # library's own tcgen05 GEMM, q in place and a Philox draw per request
    gd = torch.Generator().manual_seed(1005)
    d_draft = 2048
    hd = torch.randn(Bn, d_draft, generator=gd).to(torch.bfloat16).to(dev)
    wd = (torch.randn(V, d_draft, generator=gd) * 0.02).to(torch.bfloat16).to(dev)
    qd = torch.empty(Bn, V, device=dev)
    xd = torch.empty(Bn, dtype=torch.int32, device=dev)
    wsd = B_.workspace(B_.spec_draft_workspace_size(Bn, d_draft, V), dev)
    n_draft_calls = [0]

    def spec_step():
        B_.spec_lmhead_verify(h, w, d, q, Bn, K, V, T, x, u, out, al, ws, stream=stream)

    def plain_step():
        B_.spec_lmhead_verify(h0, w, d, None, Bn, 0, V, T, x0, u0, out0, al0, ws0, stream=stream)

    def draft_step():
        B_.spec_draft_sample(hd, wd, T, 1005, n_draft_calls[0] * Bn, qd, xd, wsd, stream=stream)
        n_draft_calls[0] += 1

    for fn in (spec_step, plain_step, draft_step):
        for _ in range(max(args.warmup, 3)):
            fn()
    torch.cuda.synchronize()
    clocks = Clocks(local).start()
    sustained = _sustain(spec_step, stream, SUSTAIN_S_OTHER)
    ms = _time_back_to_back(spec_step, args.steps, stream)  # events inside the step would serialise it
    # the GEMM's own time: a second pass with the library's profiling events around every GEMM launch
    ks_ev = _events(args.steps)
    for a, b in ks_ev:  # torch measures only events it has recorded itself once
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        B_.spec_profile_set_events(ks_ev[i][0], ks_ev[i][1])
        spec_step()
    B_.spec_profile_set_events(None, None)
    torch.cuda.synchronize()
    clk = clocks.stop()
    kms = statistics.mean(a.elapsed_time(b) for a, b in ks_ev)
    n_side = max(5, args.steps // 2)
    t_plain = _time_back_to_back(plain_step, n_side, stream)
    t_draft1 = _time_back_to_back(draft_step, n_side, stream)
    al_h, out_h = al.cpu().numpy(), out.cpu().numpy()
    al_mean = float(al_h.mean())
    # directly timed: round(AL) plain steps against one speculative cycle (K draft steps + verify)
    n_plain = max(1, int(round(al_mean)))

    def plain_loop():
        for _ in range(n_plain):
            plain_step()

    def spec_cycle():
        for _ in range(K):
            draft_step()
        spec_step()

    t_plain_loop = _time_back_to_back(plain_loop, 5, stream)
    t_spec_cycle = _time_back_to_back(spec_cycle, 5, stream)
    closed = SP.measured_speedup(t_plain, ms, K * t_draft1, al_mean)
    direct_ratio = t_plain_loop / t_spec_cycle
    # the same comparison with AL's fraction kept: round(AL) plain steps stand for AL of them
    direct_scaled = direct_ratio * al_mean / n_plain
    w_bytes = V * d * 2
    gemm_bytes = w_bytes + M * d * 2 + M * V * 4 + M * ((V + 255) // 256) * 8
    flops = 2.0 * M * d * V
    tpk, tpk_kind = _peak_tflops()
    roof = _roof("lmhead_gemm_kernel (tcgen05, W stream)", gemm_bytes, kms, _traffic("lmhead_gemm_kernel"))
    roof["tensor"] = {"achieved_tflops": flops / (kms * 1e-3) / 1e12, "peak_tflops": tpk, "peak_kind": tpk_kind,
                      "frac": flops / (kms * 1e-3) / 1e12 / tpk}
    line = {
        "metric": METRIC, "value": Bn * K / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 GEMM, f32 verify", "data": "synthetic",
        "config": {"workload": "fused LM-head + verify B=16 K=7 (128 rows) d=8192 V=128256 T=1", "B": Bn,
                   "K": K, "V": V, "d": d, "l2": "inputs 2.1 GB > L2, no flush: steps back to back"},
        "mean_accept_len": al_mean,
        "roofline": roof,
        "speedup_model": {
            "T_verif_B_ms": t_plain, "T_verif_B1D_ms": ms, "T_draft_ms": K * t_draft1, "AL": al_mean,
            "closed_form": closed,
            "direct": {"plain_steps": n_plain, "plain_loop_ms": t_plain_loop, "spec_cycle_ms": t_spec_cycle,
                       "ratio": direct_ratio, "ratio_at_AL": direct_scaled,
                       "closed_form_vs_direct_at_AL": closed / direct_scaled},
            "draft_step": f"spec_draft_sample at M={Bn}, d={d_draft}, V={V}, T={T} (tcgen05 GEMM, q in place, "
                          "Philox draw), K of them per cycle"},
        "sustained": sustained, "clocks": clk,
        "gpu_launches": 2 * args.steps,
    }
    if not args.no_cpu:
        # the oracle's sample: the first 2 requests (16 rows), with near-tie bands derived from the
        # GEMM's accumulation bound over those rows (oracle/gemm_bound.py)
        import oracle
        from oracle import gemm_bound as G
        n_req = 2
        rows = n_req * (K + 1)
        hs = batch.hidden[:rows]

        def fn():
            bands = G.bands(hs, batch.w_vocab_t, T)
            return oracle.lmhead_verify(hs, batch.w_vocab_t, batch.q[:n_req * K], batch.draft[:n_req * K],
                                        batch.uniforms[:rows], n_req, K, T, bands=bands)

        orc, per, reps = _oracle_timed(fn, 0.1)
        line["cpu_baseline"] = {"value": n_req * K / per, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"first {n_req} of {Bn} requests: fp64 GEMM (torch, all cores), its "
                                          f"accumulation bound, C verify; {per:.1f} s"}
        line["parity"] = _decision_parity(out_h, al_h, orc, np.arange(n_req + 1) * (K + 1), n_req)
        line["parity"]["bands"] = "derived from the GEMM's accumulation bound"
    return line


# ---------------------------------------------------------------------------
# The serving-loop steps around verification
# ---------------------------------------------------------------------------
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
    clocks = Clocks(0).start()
    parity = None
    sustained = None
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
        if Bn == 64 and not args.no_cpu:
            # bit-exact parity of one reserve (the state after it) against the oracle, timed as the CPU baseline
            from oracle import kv_blocks as kv
            B_.spec_kv_reserve(g_bt, g_seq, g_free, g_fc, g_K, bs, st, stream=stream)
            got_bt, got_fc = g_bt.cpu().numpy(), int(g_fc.item())
            (o_bt, o_fc, o_st), per, reps = _oracle_timed(lambda: kv.reserve(bt, seq, free, n_ids - k, np.full(Bn, K), bs),
                                                          0.5)
            B_.spec_kv_rollback(g_bt, g_seq, g_free, g_fc, g_K, g_al, bs, st, stream=stream)
            ok = np.array_equal(got_bt, o_bt) and got_fc == o_fc and o_st == kv.OK
            parity = {"requests": Bn, "mismatch": 0 if ok else 1, "near_ties": 0, "near_tie_mismatch": 0,
                      "what": "block table and free count after one reserve, bit-exact"}
            cpu = {"value": 1.0 / per, "unit": "reserves/s", "cores": 1, "kind": "oracle",
                   "sample": f"reserve of the B=64 state, {reps} repetitions, numpy/Python"}

        def steps_fn(s, n=args.steps):
            for _ in range(n):
                B_.spec_kv_reserve(g_bt, g_seq, g_free, g_fc, g_K, bs, st, stream=s)
                B_.spec_kv_rollback(g_bt, g_seq, g_free, g_fc, g_K, g_al, bs, st, stream=s)

        for _ in range(max(args.warmup, 3)):
            steps_fn(stream, 1)
        torch.cuda.synchronize()
        # launch-bound: the K steps are captured in one CUDA graph
        g = _graph_of(steps_fn, stream)
        if Bn == 64:
            sustained = _sustain(g.replay, stream, SUSTAIN_S_OTHER, calls_per_fn=args.steps)
        ms = _time_back_to_back(g.replay, 1, stream) / args.steps
        assert st.item() == 0 and np.array_equal(g_bt.cpu().numpy(), bt), "state must return to itself"
        new_blocks = sum(-(-(int(s) + K) // bs) - (-(-int(s) // bs)) for s in seq)
        # bytes: lengths and counts read twice, accept lengths, touched table entries
        # (checked, then written), free-list slots (read, then written)
        alg = Bn * 4 * 5 + new_blocks * 4 * 6
        res[f"B={Bn}"] = {"us_per_step": ms * 1e3, "blocks_moved_per_step": 2 * new_blocks,
                          "algorithmic_bytes": alg, "achieved_gbs": alg / (ms * 1e-3) / 1e9}
    clk = clocks.stop()
    head = res["B=64"]
    line = {
        "metric": "KV bookkeeping steps/s (reserve + rollback)", "value": 1e6 / head["us_per_step"],
        "unit": "steps/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": head["us_per_step"] * 1e-3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": "paged KV reserve + rollback, B=64 and 4096, K=4, 16-token blocks, "
                               "every draft rejected", "l2": "state stays in L2 (launch-bound, one CTA)"},
        "roofline": _roof("kvb::reserve_kernel + kvb::rollback_kernel", head["algorithmic_bytes"] / 2,
                          head["us_per_step"] * 1e-3 / 2,
                          note="latency-bound: one CTA and two dependent launches per step"),
        "batches": res, "sustained": sustained, "clocks": clk, "gpu_launches": 2 * args.steps,
    }
    if parity is not None:
        line["parity"], line["cpu_baseline"] = parity, cpu
    return line


def run_draft(args):
    """Draft head + draft sampling at the fused workload's draft head: M = 128
    rows (16 requests x 8 positions), d = 2048, V = 128256, T = 1: the tcgen05
    GEMM writes fp32 logits into q's buffer, then one CTA per row turns them
    into q and draws x with Philox."""
    import numpy as np
    import torch
    from speculative_decoding_verification_11_gb300 import build, binding as B_
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    M, d, V, T = 128, 2048, 128256, 1.0
    g = torch.Generator().manual_seed(1005)
    h_host = torch.randn(M, d, generator=g).to(torch.bfloat16)
    w_host = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16)
    h, w = h_host.to(dev), w_host.to(dev)
    q = torch.empty(M, V, device=dev)
    x = torch.empty(M, dtype=torch.int32, device=dev)
    ws = B_.workspace(B_.spec_draft_workspace_size(M, d, V), dev)
    calls = [0]

    def step():
        B_.spec_draft_sample(h, w, T, 1005, calls[0] * M, q, x, ws, stream=stream)
        calls[0] += 1

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    # steps back to back between one pair of events (W, 525 MB, is beyond L2); the GEMM's own time
    # from a second pass with the library's profiling events around every GEMM launch (events
    # between the two launches of a step would serialise it)
    clocks = Clocks(0).start()
    sustained = _sustain(step, stream, SUSTAIN_S_OTHER)
    ms = _time_back_to_back(step, args.steps, stream)
    kev = _events(args.steps)
    for a, b in kev:  # torch measures only events it has recorded itself once
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        B_.spec_profile_set_events(kev[i][0], kev[i][1])
        step()
    B_.spec_profile_set_events(None, None)
    torch.cuda.synchronize()
    clk = clocks.stop()
    gms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    tpk, tpk_kind = _peak_tflops()
    gemm_bytes = V * d * 2 + M * d * 2 + M * V * 4  # W, hidden, fp32 logits written
    flops = 2 * M * d * V
    finish_bytes = 2 * M * V * 4                     # logits read, q written
    roof = _roof("lmhead_gemm_kernel (draft head)", gemm_bytes, gms, _traffic("lmhead_gemm_kernel_draft"))
    roof["tensor"] = {"achieved_tflops": flops / (gms * 1e-3) / 1e12, "peak_tflops": tpk, "peak_kind": tpk_kind,
                      "frac": flops / (gms * 1e-3) / 1e12 / tpk}
    line = {
        "metric": "drafted tokens/s (draft head GEMM + q + Philox draw)", "value": M / (ms * 1e-3),
        "unit": "drafted tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"draft head M={M} d={d} V={V} T={T} bf16 weights, fp32 q",
                   "l2": "inputs 525 MB > L2, no flush"},
        "roofline": roof,
        "finish": {"ms": ms - gms, "algorithmic_bytes": finish_bytes,
                   "achieved_gbs": finish_bytes / ((ms - gms) * 1e-3) / 1e9},
        "sustained": sustained, "clocks": clk, "gpu_launches": 2 * args.steps,
    }
    if not args.no_cpu:
        # the last call's first 8 rows against the oracle, with bands derived from the GEMM's
        # accumulation bound (oracle/gemm_bound.py): u bit-exact, q within e_p, x outside near ties
        from oracle import draft as D
        from oracle import gemm_bound as G
        n = 8
        offset = (calls[0] - 1) * M
        qg, xg = q[:n].cpu().numpy(), x[:n].cpu().numpy()

        def fn():
            bands = G.bands(h_host[:n], w_host, T)
            return bands, D.draft_sample(h_host[:n], w_host, T, 1005, offset, bands=bands)

        (bands, orc), per, reps = _oracle_timed(fn, 0.1)
        big = orc["q"] > 1e-30
        ratio = float((np.abs(qg[big] - orc["q"][big]) / orc["q"][big] / bands.e_p[big]).max())
        same = xg == orc["x"]
        line["parity"] = {"requests": n, "mismatch": int((~same & ~orc["near_tie"]).sum()),
                          "near_ties": int(orc["near_tie"].sum()), "near_tie_mismatch": int((~same & orc["near_tie"]).sum()),
                          "q_err_over_bound": ratio, "bands": "derived from the GEMM's accumulation bound"}
        line["cpu_baseline"] = {"value": n / per, "unit": "drafted tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"first {n} of {M} rows: fp64 GEMM (torch, all cores), its accumulation "
                                          f"bound, softmax and draw; {per:.1f} s"}
    return line


def run_ngram(args):
    """Model-free n-gram (prompt lookup) drafting over synthetic streams with
    repetition: B = 256 contexts of L tokens (L = 8192 and 32768), K = 8,
    n in [1, 4].  The contexts fit in L2, so calls rotate over copies whose
    total exceeds twice L2, replayed back to back from a CUDA graph."""
    import numpy as np
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
    clocks = Clocks(0).start()
    parity = cpu = sustained = None
    for L in (8192, 32768):
        tokens, offs = W.repetitive_streams(seed=1006, B=B, L=L)
        t = torch.from_numpy(tokens).to(dev)
        o = torch.from_numpy(offs).to(dev)
        dd = torch.empty(B, K, dtype=torch.int32, device=dev)
        k = torch.empty(B, dtype=torch.int32, device=dev)
        # the contexts fit in L2: calls rotate over enough copies that none finds bytes an earlier
        # call read, and the calls are replayed from one CUDA graph (each call's own launch is short
        # next to the host's launch rate); with --l2-flush, L2 is flushed before every timed call
        in_bytes = t.numel() * 4
        n_copies = 1 if args.l2_flush else -(-2 * L2_BYTES // in_bytes) + 1
        copies = [t] + [t.clone() for _ in range(n_copies - 1)]
        for i in range(max(args.warmup, 3, n_copies)):
            B_.spec_ngram_draft(copies[i % n_copies], o, K, n_min, n_max, dd, k, stream=stream)
        torch.cuda.synchronize()
        if args.l2_flush:
            ev = _events(args.steps)
            for i in range(args.steps):
                fw.fill_(float(i))
                fr.sum()
                ev[i][0].record(stream)
                B_.spec_ngram_draft(t, o, K, n_min, n_max, dd, k, stream=stream)
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        else:
            def steps_fn(s):
                for i in range(args.steps):
                    B_.spec_ngram_draft(copies[i % n_copies], o, K, n_min, n_max, dd, k, stream=s)

            g = _graph_of(steps_fn, stream)
            if L == 8192:
                sustained = _sustain(g.replay, stream, SUSTAIN_S_OTHER, calls_per_fn=args.steps)
            ms = _time_back_to_back(g.replay, 1, stream) / args.steps
        kh = k.cpu()
        alg = B * L * 4 + (B + 1) * 4 + B * K * 4 + B * 4
        res[f"L={L}"] = {"us_per_call": ms * 1e3, "requests_per_s": B / (ms * 1e-3),
                         "mean_draft_len": float(kh.float().mean()), "with_proposal": float((kh > 0).float().mean()),
                         "algorithmic_bytes": alg, "achieved_gbs": alg / (ms * 1e-3) / 1e9}
        if L == 8192 and not args.no_cpu:
            from oracle import ngram as NG
            n_req = 32
            ctxs = [tokens[offs[b]:offs[b + 1]].tolist() for b in range(n_req)]
            (od, ok_), per, reps = _oracle_timed(lambda: NG.propose_batch(ctxs, K, n_min, n_max), 0.1)
            gd_, gk_ = dd[:n_req].cpu().numpy(), kh[:n_req].numpy()
            mism = int(sum(not (np.array_equal(gd_[b], od[b]) and gk_[b] == ok_[b]) for b in range(n_req)))
            parity = {"requests": n_req, "mismatch": mism, "near_ties": 0, "near_tie_mismatch": 0,
                      "what": "proposed tokens and lengths, bit-exact"}
            cpu = {"value": n_req / per, "unit": "requests/s", "cores": 1, "kind": "oracle",
                   "sample": f"first {n_req} of {B} contexts (L=8192), pure Python, {per:.2f} s"}
    clk = clocks.stop()
    head = res["L=8192"]
    line = {
        "metric": "n-gram drafting requests/s", "value": head["requests_per_s"], "unit": "requests/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": head["us_per_call"] * 1e-3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": f"prompt-lookup drafting B={B} K={K} n={n_min}..{n_max} over repetitive streams",
                   "l2": ("contexts < L2: 256 MB write then 256 MB read before every call, outside its events"
                          if args.l2_flush else
                          "contexts < L2: calls rotate over copies > 2 x L2, replayed back to back from a CUDA graph")},
        "roofline": _roof("ng::ngram_kernel", head["algorithmic_bytes"], head["us_per_call"] * 1e-3,
                          _traffic("ngram_kernel")),
        "lengths": res, "sustained": sustained, "clocks": clk, "gpu_launches": 2 * args.steps,
    }
    if parity is not None:
        line["parity"], line["cpu_baseline"] = parity, cpu
    return line


def run_dynk(args):
    """Dynamic-K controller after verification (goodput rule, 10-result rings,
    K in [1, 8], row offsets for the next ragged verification), B = 64 and
    4096, captured in a CUDA graph (the update is launch-bound)."""
    import numpy as np
    import torch
    from speculative_decoding_verification_11_gb300 import build, binding as B_
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    clocks = Clocks(0).start()
    parity = cpu = sustained = None
    for Bn in (64, 4096):
        g = torch.Generator().manual_seed(Bn)
        al = torch.randint(1, 6, (Bn,), generator=g, dtype=torch.int32).to(dev)
        ku = torch.full((Bn,), 5, dtype=torch.int32, device=dev)
        hist = torch.zeros(Bn, 10, 2, dtype=torch.int32, device=dev)
        count = torch.zeros(Bn, dtype=torch.int32, device=dev)
        kn = torch.empty(Bn, dtype=torch.int32, device=dev)
        offs = torch.empty(Bn + 1, dtype=torch.int32, device=dev)
        itl = (10.0 + 1.5 * torch.arange(9, dtype=torch.float32)).to(dev)
        if Bn == 64 and not args.no_cpu:
            # one update from empty rings, bit-exact against the oracle (timed as the CPU baseline)
            from oracle import dynk as DK
            B_.spec_dynk_update(al, ku, hist, count, B_.SV_DYNK_GOODPUT, 1, 8, kn, itl=itl, row_offsets=offs,
                                stream=stream)
            got_k, got_o = kn.cpu().numpy(), offs.cpu().numpy()
            al_h, ku_h, itl_h = al.cpu().numpy(), ku.cpu().numpy(), itl.cpu().numpy()

            def fn():
                return DK.update(al_h, ku_h, np.zeros((Bn, 10, 2), np.int32), np.zeros(Bn, np.int32), 10,
                                 DK.GOODPUT, 1.5, 1, 8, itl=itl_h)

            (ok_, oo), per, reps = _oracle_timed(fn, 0.1)
            parity = {"requests": Bn, "mismatch": int((got_k != ok_).sum()) + int(not np.array_equal(got_o, oo)),
                      "near_ties": 0, "near_tie_mismatch": 0, "what": "next K and row offsets, bit-exact"}
            cpu = {"value": 1.0 / per, "unit": "updates/s", "cores": 1, "kind": "oracle",
                   "sample": f"one B=64 update, {reps} repetitions, numpy/Python"}
            hist.zero_()
            count.zero_()

        def steps_fn(s, n=args.steps):
            for _ in range(n):
                B_.spec_dynk_update(al, ku, hist, count, B_.SV_DYNK_GOODPUT, 1, 8, kn, itl=itl, row_offsets=offs,
                                    stream=s)

        for _ in range(max(args.warmup, 3)):
            steps_fn(stream, 1)
        torch.cuda.synchronize()
        graph = _graph_of(steps_fn, stream)
        if Bn == 64:
            sustained = _sustain(graph.replay, stream, SUSTAIN_S_OTHER, calls_per_fn=args.steps)
        us = _time_back_to_back(graph.replay, 1, stream) * 1e3 / args.steps
        alg = Bn * (4 * 4 + 10 * 8 + 8) + 9 * 4  # AL, K used, count, k_next; the ring read (and one pair written); offsets
        res[f"B={Bn}"] = {"us_per_update": us, "algorithmic_bytes": alg, "achieved_gbs": alg / (us * 1e-6) / 1e9,
                          "mean_k_next": float(kn.float().mean())}
    clk = clocks.stop()
    head = res["B=64"]
    line = {
        "metric": "dynamic-K controller updates/s", "value": 1e6 / head["us_per_update"], "unit": "updates/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": head["us_per_update"] * 1e-3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32/f32", "data": "synthetic",
        "config": {"workload": "goodput rule, W=10, K in [1, 8], B=64 and 4096, offsets for ragged verification",
                   "l2": "state stays in L2 (launch-bound, one CTA)"},
        "roofline": _roof("dk::dynk_kernel", head["algorithmic_bytes"], head["us_per_update"] * 1e-3,
                          note="latency-bound: one CTA per update, in a CUDA graph"),
        "batches": res, "sustained": sustained, "clocks": clk, "gpu_launches": args.steps,
    }
    if parity is not None:
        line["parity"], line["cpu_baseline"] = parity, cpu
    return line


OTHER = {
    "tiny": lambda a: run_config(a, "tiny"),
    "greedy": lambda a: run_config(a, "greedy"),
    "lmhead": run_lmhead,
    "ragged": lambda a: run_config(a, "ragged"),
    "kv": run_kv,
    "draft": run_draft,
    "ngram": run_ngram,
    "dynk": run_dynk,
}

# keys of a workload's own line carried into the headline's "workloads" block
_ENTRY_KEYS = ("metric", "value", "unit", "ms_per_step", "steps", "dtype", "config", "roofline", "mean_accept_len",
               "sustained", "clocks", "gpu_launches", "parity", "cpu_baseline", "speedup_model", "graph_b1", "finish",
               "lengths", "batches")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baselines and parity samples")
    ap.add_argument("--l2-flush", action="store_true",
                    help="write a 256 MB buffer before every timed step (its dirty lines are written back "
                         "during the next step); by default the inputs, larger than L2, stand in for a flush")
    ap.add_argument("--sustain", type=float, default=SUSTAIN_S,
                    help="seconds of back-to-back headline steps run ahead of the timed steps so that the clock "
                         "record holds samples under load (the other workloads get a fifth of it); 0 skips them, "
                         "e.g. under a profiler.  The timed steps are the same either way")
    ap.add_argument("--copies", type=int, default=3,
                    help="resident copies of the inputs the back-to-back steps rotate over (no flush)")
    ap.add_argument("--config", choices=["all", "sampling"] + list(OTHER), default="all",
                    help="all (default): the headline workload's line with every other workload under "
                         "'workloads'; sampling: the headline alone; any other name: that workload alone")
    args = ap.parse_args()
    _SUSTAIN_SCALE[0] = args.sustain / SUSTAIN_S if SUSTAIN_S > 0 else 0.0
    if args.impl == "reference":
        return run_reference(args)
    if args.config in OTHER:
        print(json.dumps(OTHER[args.config](args)), flush=True)
        return 0
    line = run_ours(args)
    world, rank, _ = _dist()
    if args.config == "all" and world == 1:
        import torch
        line["workloads"] = {}
        for name, fn in OTHER.items():
            torch.cuda.empty_cache()
            try:
                w = fn(args)
                line["workloads"][name] = {k: w[k] for k in _ENTRY_KEYS if k in w}
            except Exception as e:  # a failing side workload is reported, not hidden
                line["workloads"][name] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
