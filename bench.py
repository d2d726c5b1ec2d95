#!/usr/bin/env python3
"""Benchmark of the confidence-driven variable-length verify step.

One step = dspark_score_compact (steps a1-a4 in one launch: what
dspark_score_budget + dspark_compact compute) + dspark_verify (C ABI, one
stream) over one batch of the mixed-traffic workload: B=256 requests,
gamma=16, V=129280, d=7168, bf16, c=0.35, cap T=768, sampling at Tm=1.

* value: steps/s over all ranks, from CUDA events around each timed step;
  inputs are resident in HBM; several input sets are cycled and L2 is flushed
  (256 MiB write, outside the events) before every timed step.
* roofline: the verify kernel's algorithmic bytes per launch (ragged target
  rows + kept draft rows, read once) over its event-timed duration, against
  the measured HBM copy bandwidth.  The early-exit count (rows only up to
  each request's first rejection) is reported beside it: the kernel skips
  bonus rows of requests it already knows to reject, so its reads fall
  between the two.
* e2e: the same metric through the C ABI with host inputs: every step copies
  its inputs from pinned host memory and reads the results back.
* cpu_baseline: the CPU oracle (single thread) on the same workload;
  cpu_baseline_omp: its OpenMP build over all host cores; parity: the GPU's
  outputs of input set 0 against the oracle, with the near-tie counts.
* cap_accept_arm: the audit arm on the same inputs -- the full block
  verified, the confidence-driven window committed -- with its step time and
  the utilization against the ceiling (accepted drafts kept / accepted drafts
  the full verify finds).
* entropy_arm: the step with the entropy-confidence variant of the score
  (conf = exp(-H) of each draft row at theta = 0.3): step time, the score
  kernel's time and bandwidth over the B*gamma*V draft logits it streams.
* sts_fit: the STS temperatures fitted to the logged confidences, lengths
  and accept lengths of the timed step's input sets, with the fit's time.
* latency_b1: the B=1 DeepSeek-class greedy step, microseconds per step with
  plain launches and replayed as CUDA graphs; input sets cycled so that they
  exceed L2 (no flush).
* --impl reference: the CPU oracle as the reference arm, full steps of the
  same configuration.

Multi-GPU runs are independent replicas (the step has no cross-request
exchange without a cross-rank cap); the slowest rank sets the time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ragged verify steps/s & HBM GB/s (% of peak) at B=256, gamma=16, V=129280"
DEFAULT_WORKLOAD = "mixed_B256_g16_V129280_d7168_bf16"
FLUSH_BYTES = 256 << 20
L2_BYTES = 129_000_000  # GB300 L2, nominal size
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILE_FILE = os.path.join(ROOT, "profiles", "verify_kernel_mixed_B256.json")
KERNEL_SOURCES = ["confidence_driven_speculative_gb300/csrc/verify.cu",
                  "confidence_driven_speculative_gb300/csrc/dspark_internal.cuh"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--sets", type=int, default=4, help="input sets cycled through the steps")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-latency", action="store_true")
    ap.add_argument("--no-audit-arm", action="store_true")
    ap.add_argument("--no-entropy-arm", action="store_true")
    ap.add_argument("--no-sts-fit", action="store_true")
    ap.add_argument("--no-fixed-arm", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--l2", choices=["inputs", "flush"], default="inputs",
                    help="between timed steps: rely on inputs larger than L2 (each step reads "
                         "its own input set, the sets cycled), or write a 256 MiB buffer")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------- #
# distributed plumbing (replicas)
# --------------------------------------------------------------------------- #
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int, device="cpu") -> float:
    """Maximum of x over ranks (x itself when there is one rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(steps_per_rank: int, world: int, max_total_ms: float) -> float:
    """Steps per second of the whole job: all ranks' steps over the slowest rank's time."""
    return steps_per_rank * world / (max_total_ms / 1000.0)


# --------------------------------------------------------------------------- #
# clocks during the timed region
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.gpu = vis.split(",")[local_rank] if vis else str(local_rank)
        self.samples = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.gpu],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._reader, daemon=True).start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5.0:
            time.sleep(0.05)

    def _reader(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        win = [p for t, p in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not win:
            win = [p for _, p in self.samples[-3:]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        mx = [num(p[1]) for p in win if num(p[1]) is not None]
        pw = [num(p[2]) for p in win if num(p[2]) is not None]
        reasons = sorted({r for p in win for r, v in zip(self.REASONS, p[3:7]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(win)}


# --------------------------------------------------------------------------- #
# byte model
# --------------------------------------------------------------------------- #
def verify_bytes(B: int, sum_L: int, V: int, logit_size: int, sampling: bool, gamma: int) -> int:
    """Algorithmic bytes of one verify launch: every packed target row
    (sum L + B) and, when sampling, every kept draft row (sum L), read once;
    plus the small integer/float inputs and outputs."""
    rows = (sum_L + B) + (sum_L if sampling else 0)
    small = 4 * (B * gamma + 5 * B + 2 * (B + 1) + 2 * B * (gamma + 1)) + 8 * sum_L
    return rows * V * logit_size + small


def early_exit_bytes(accept_len, L, V: int, logit_size: int, sampling: bool) -> int:
    """The secondary, early-exit count of a verify launch's logit bytes: rows
    only up to each request's first rejection.  Target rows 0..a_b; when
    sampling, the draft rows of the drafts tested (min(a_b + 1, L_b))."""
    import torch
    a = accept_len.to(torch.int64)
    tgt = int((a + 1).sum().item())
    drf = int(torch.minimum(a + 1, L.to(torch.int64)).sum().item()) if sampling else 0
    return (tgt + drf) * V * logit_size


def score_bytes(B: int, gamma: int, d: int, hidden_size: int) -> int:
    """Algorithmic bytes of one score_budget launch: the hidden block once,
    the head weight, and the small outputs."""
    return B * gamma * d * hidden_size + 4 * d + 4 * (B + gamma) + 4 * (3 * B * gamma + 4 * B)


# GB300 HBM3e nominal bandwidth (vendor figure), reported beside the
# measured copy bandwidth.
SPEC_HBM_GBS = 7900.0


def measured_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per verify launch from the committed ncu figures, if they
    were taken on the current kernel source; else None."""
    try:
        with open(PROFILE_FILE) as f:
            vals = json.load(f)
    except (OSError, ValueError):
        return None
    if vals.get("source_sha256") != source_hash():
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def prepare_set(W, binding, w, step: int, fixed_budget: int = -1, entropy_theta=None):
    import torch
    kw = {"fixed_budget": fixed_budget}
    if fixed_budget >= 0:
        kw["cap_T"] = -1
    inp = W.make_inputs(w, step, device="cuda", **kw)
    bufs = binding.StepBuffers(inp["B"], inp["gamma"], inp["V"], inp["d"])
    commit = inp["seq_lens"].clone()
    bufs.bind(inp, seq_lens_commit=commit)
    if entropy_theta is None:
        binding.dspark_score_compact(bufs.step)
    else:
        binding.dspark_score_entropy(bufs.step, entropy_theta)
        binding.dspark_compact(bufs.step)
    torch.cuda.synchronize()
    n_rows = int(bufs.row_off[inp["B"]].item())
    # Stand-in for the target forward over the packed rows (not timed).
    tgt = W.ragged_target_rows(inp["target_dense"], bufs.row_req, bufs.row_k, n_rows).contiguous()
    bufs.bind_target(tgt)
    binding.dspark_verify(bufs.step)
    torch.cuda.synchronize()
    sum_L = int(bufs.L.sum().item())
    ee = early_exit_bytes(bufs.accept_len, bufs.L, inp["V"], tgt.element_size(),
                          inp["temperature"] > 0)
    return {"inp": inp, "bufs": bufs, "tgt": tgt, "sum_L": sum_L, "early_exit_bytes": ee,
            "L_ref": bufs.L.clone(), "commit": commit}


def prepare_audit(W, binding, w, step: int, window_set):
    """The cap-accept audit arm on the same inputs: the full block (static,
    every L_b = gamma) is verified and the window ``window_set`` (the
    confidence-driven step on the same inputs) is committed."""
    import torch
    st = prepare_set(W, binding, w, step, fixed_budget=w.gamma)
    st["window"] = window_set
    st["accept_full"] = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    st["totals"] = torch.zeros(2, dtype=torch.int32, device="cuda")
    binding.dspark_verify_cap_accept(st["bufs"].step, window_set["bufs"].L, st["accept_full"],
                                     st["totals"])
    torch.cuda.synchronize()
    return st


class L2Policy:
    """What happens between timed steps.  ``inputs``: nothing -- every step
    reads its own input set (~0.5 GB, several times L2) and the sets are
    cycled, so no step finds its inputs in L2.  ``flush``: a 256 MiB write
    outside the events; it leaves L2 full of dirty lines whose write-back then
    lands inside the next timed step."""

    def __init__(self, mode: str, buf):
        self.mode = mode
        self.buf = buf

    def zero_(self):
        if self.mode == "flush":
            self.buf.zero_()

    def describe(self, set_bytes: float) -> str:
        if self.mode == "flush":
            return "256 MiB write before every timed step (outside the events)"
        return (f"inputs larger than L2: each step reads its own input set "
                f"(~{set_bytes / 1e9:.2f} GB), the sets cycled; no flush")


def audit_loop(binding, audit, K, W_, flush, stream):
    """Warm-up, then K timed audit steps: the confidence-driven budget (the
    window), the static budget and packing, the cap-accept verify."""
    import torch
    P = len(audit)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(W_ + K):
        st = audit[i % P]
        s, win = st["bufs"].step, st["window"]["bufs"]
        flush.zero_()
        e = ev[i - W_] if i >= W_ else None
        if e:
            e[0].record()
        binding.dspark_score_budget(win.step, stream)
        binding.dspark_score_compact(s, stream)
        if e:
            e[1].record()
        binding.dspark_verify_cap_accept(s, win.L, st["accept_full"], st["totals"], stream)
        if e:
            e[2].record()
    torch.cuda.synchronize()
    return ev


ENTROPY_THETA = 0.3


def entropy_loop(binding, sets, K, W_, flush, stream, theta):
    """Warm-up, then K timed steps of the entropy-confidence variant:
    score_entropy, compact, verify (events around the score kernel and the
    whole step)."""
    import torch
    P = len(sets)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(W_ + K):
        s = sets[i % P]["bufs"].step
        flush.zero_()
        e = ev[i - W_] if i >= W_ else None
        if e:
            e[0].record()
        binding.dspark_score_entropy(s, theta, stream)
        if e:
            e[1].record()
        binding.dspark_compact(s, stream)
        binding.dspark_verify(s, stream)
        if e:
            e[2].record()
    torch.cuda.synchronize()
    return ev


def run_steps(binding, sets, K, W_, flush, stream):
    """Warm up, then time exactly K steps with events (flush outside them)."""
    import torch
    P = len(sets)
    for i in range(W_):
        s = sets[i % P]["bufs"].step
        flush.zero_()
        binding.dspark_score_compact(s, stream)
        binding.dspark_verify(s, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    return ev


def timed_loop(binding, sets, ev, flush, stream):
    P = len(sets)
    for i, (e0, e1, e2) in enumerate(ev):
        s = sets[i % P]["bufs"].step
        flush.zero_()
        e0.record()
        binding.dspark_score_compact(s, stream)
        e1.record()
        binding.dspark_verify(s, stream)
        e2.record()


def run_e2e(binding, W, st, steps, stream):
    """Steps through the C ABI with host inputs: H2D of every input from pinned
    memory, the step's calls, D2H of the results, inside the timed region.
    (Spreading the copies over several streams measured no faster.)"""
    import torch
    inp, bufs = st["inp"], st["bufs"]
    names = ["hidden", "head_w", "head_bias", "sts_tau", "draft_tokens", "draft_logits",
             "last_tokens", "seq_lens"]
    host = {k: inp[k].cpu().pin_memory() for k in names}
    host["target"] = st["tgt"].cpu().pin_memory()
    dev = {k: inp[k] for k in names}
    dev["target"] = st["tgt"]
    outs = [bufs.accept_len, bufs.num_emitted, bufs.out_tokens]
    host_out = [o.cpu().pin_memory() for o in outs]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    times = []
    for i in range(steps + 2):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        binding.dspark_score_compact(bufs.step, stream)
        binding.dspark_verify(bufs.step, stream)
        for o, h in zip(outs, host_out):
            h.copy_(o, non_blocking=True)
        e1.record()
        e1.synchronize()
        if i >= 2:
            times.append(e0.elapsed_time(e1))
    return statistics.mean(times), h2d, d2h


def run_latency(binding, W, steps: int = 200):
    """The B=1 latency step (DeepSeek-class shapes, greedy): microseconds per
    step with plain launches and as replayed CUDA graphs (median of per-step
    CUDA events).  No step finds its inputs in L2: enough input sets of this
    small shape are cycled that they exceed L2 twice over (a flush before
    each step would leave dirty lines whose write-back lands in the next
    ~15 us step)."""
    import math
    import torch
    first = prepare_set(W, binding, W.LATENCY_B1, 0)
    inp = first["inp"]
    set_bytes = sum(t.numel() * t.element_size() for t in (
        inp["hidden"], inp["draft_logits"], first["tgt"]))
    n_sets = max(2, min(64, math.ceil(2 * L2_BYTES / max(set_bytes, 1))))
    sets = [first] + [prepare_set(W, binding, W.LATENCY_B1, i) for i in range(1, n_sets)]

    def one(st):
        binding.dspark_score_compact(st["bufs"].step)
        binding.dspark_verify(st["bufs"].step)

    def timed(fns):
        for i in range(2 * len(fns)):
            fns[i % len(fns)]()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        for i, (e0, e1) in enumerate(ev):
            e0.record()
            fns[i % len(fns)]()
            e1.record()
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) * 1000.0

    out = {"workload": W.LATENCY_B1.name, "steps": steps,
           "l2": f"{n_sets} input sets of {set_bytes / 1e6:.1f} MB cycled (> 2x L2); no flush",
           "us_per_step_plain": timed([lambda st=st: one(st) for st in sets])}
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graphs = []
        with torch.cuda.stream(side):
            for st in sets:
                one(st)  # warm-up on the capture stream
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    one(st)
                graphs.append(g)
        torch.cuda.current_stream().wait_stream(side)
        out["us_per_step_graph"] = timed([g.replay for g in graphs])
        assert all(st["bufs"].device_status() == 0 for st in sets)
    except Exception as e:  # report the reason, not a number
        out["us_per_step_graph"] = None
        out["graph_error"] = str(e).splitlines()[0][:200]
    return out


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip()
                if key in ("model name", "Model"):
                    return line.split(":", 1)[1].strip()
                if key == "CPU part":
                    return f"{platform.machine()} CPU part {line.split(':', 1)[1].strip()}"
    except OSError:
        pass
    return platform.machine()


def cpu_baseline_oracle(W, st, seconds: float, threads: int = 1):
    """The CPU oracle (C, fp64) on full steps of input set 0: single-threaded
    as it stands, or (threads > 1) its OpenMP build with the requests of the
    verify spread over the host's threads."""
    import oracle
    npi = W.to_numpy(st["inp"])
    oracle.build(omp=threads > 1)
    if threads > 1:
        threads = oracle.omp_threads(threads)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.step(npi, threads=threads)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "steps/s", "cores": threads,
            "kind": "oracle" if threads == 1 else "oracle_openmp_over_requests",
            "cpu": cpu_model(),
            "sample": f"{n} full steps of input set 0 ({npi['workload']}), {dt:.1f} s"}


def parity_of_set0(W, st):
    """The GPU's outputs of input set 0 (its last timed step) against the
    oracle, with the counts of decisions left open by near ties."""
    from tests.gpu_harness import compare_with_oracle, outputs_of
    try:
        stats = compare_with_oracle(W.to_numpy(st["inp"]), outputs_of(st["bufs"]))
        return {"input_set": 0, "ok": True, **stats}
    except AssertionError as e:
        return {"input_set": 0, "ok": False, "error": str(e).splitlines()[0][:200]}


def workload_config(w) -> dict:
    """The keys naming the workload, the same in both arms' lines."""
    return {"workload": w.name, "B": w.B, "gamma": w.gamma, "V": w.V, "d": w.d,
            "storage": w.dtype + " logits and hidden states",
            "temperature": w.temperature, "cost_c": w.cost_c, "cap_T": w.cap_T}


def mean_L_of(sets, B):
    return statistics.mean(st["sum_L"] / B for st in sets)


def run_ours(args, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    from confidence_driven_speculative_gb300 import _build, binding
    from confidence_driven_speculative_gb300 import workloads as W
    _build.build()
    binding.load()
    w = W.WORKLOADS[args.workload]
    sampling = w.temperature > 0
    ls = 2 if w.dtype == "bf16" else 4
    stream = torch.cuda.current_stream().cuda_stream

    sets = [prepare_set(W, binding, w, s) for s in range(args.sets)]
    fixed = [] if args.no_fixed_arm else [prepare_set(W, binding, w, s, fixed_budget=5)
                                         for s in range(args.sets)]
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush = L2Policy(args.l2, flush_buf)
    sampler = ClockSampler(local)
    if not args.no_clocks:
        sampler.start()

    ev = run_steps(binding, sets, args.steps, args.warmup, flush, stream)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    timed_loop(binding, sets, ev, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    step_ms = [e0.elapsed_time(e2) for e0, _, e2 in ev]
    ver_ms = [e1.elapsed_time(e2) for _, e1, e2 in ev]
    sb_ms = [e0.elapsed_time(e1) for e0, e1, _ in ev]
    for st in sets:  # the step is deterministic: the ragged target still matches
        assert torch.equal(st["bufs"].L, st["L_ref"]), "verify lengths changed between runs"
        assert st["bufs"].device_status() == 0
    total_ms = reduce_max(sum(step_ms), world, "cuda")
    value = whole_job_rate(args.steps, world, total_ms)

    B, g, V, d = w.B, w.gamma, w.V, w.d
    P = len(sets)
    vb = [verify_bytes(B, sets[i % P]["sum_L"], V, ls, sampling, g) for i in range(args.steps)]
    sbb = score_bytes(B, g, d, ls)
    peak, peak_kind = measured_peak()
    ver_mean = statistics.mean(ver_ms)
    achieved = statistics.mean(vb) / (ver_mean * 1e-3) / 1e9
    step_bytes = statistics.mean(vb) + sbb
    ms_per_step = statistics.mean(step_ms)

    fixed_arm = None
    if fixed:
        evf = run_steps(binding, fixed, args.steps, args.warmup, flush, stream)
        timed_loop(binding, fixed, evf, flush, stream)
        torch.cuda.synchronize()
        fms = statistics.mean(e0.elapsed_time(e2) for e0, _, e2 in evf)
        fixed_arm = {"fixed_budget": 5, "ms_per_step": fms, "steps_per_s": 1000.0 / fms,
                     "verify_ms": statistics.mean(e1.elapsed_time(e2) for _, e1, e2 in evf),
                     "mean_L": statistics.mean(st["sum_L"] / B for st in fixed),
                     "committed_tokens_per_step": statistics.mean(
                         float(st["bufs"].num_emitted.sum().item()) for st in fixed)}

    audit_arm = None
    if not args.no_audit_arm:
        audit = [prepare_audit(W, binding, w, s, sets[s]) for s in range(len(sets))]
        eva = audit_loop(binding, audit, args.steps, args.warmup, flush, stream)
        tot = [st["totals"].tolist() for st in audit]
        same = sum(int(torch.equal(st["bufs"].out_tokens, st["window"]["bufs"].out_tokens))
                   for st in audit)
        same_req = sum(int((st["bufs"].out_tokens == st["window"]["bufs"].out_tokens)
                           .all(dim=1).sum().item()) for st in audit)
        ams = statistics.mean(e0.elapsed_time(e2) for e0, _, e2 in eva)
        avm = statistics.mean(e1.elapsed_time(e2) for _, e1, e2 in eva)
        avb = verify_bytes(B, B * g, V, ls, sampling, g)
        audit_arm = {
            "mode": "cap-accept: static block (L_b = gamma) verified, confidence-driven "
                    "window committed",
            "ms_per_step": ams, "steps_per_s": 1000.0 / ams,
            "verify_ms": avm,
            "verify_bytes_per_launch": avb,
            "verify_gbs": avb / (avm * 1e-3) / 1e9,
            "verify_frac": avb / (avm * 1e-3) / 1e9 / peak,
            "utilization": sum(t[1] for t in tot) / max(1, sum(t[0] for t in tot)),
            "accepted_full_per_step": statistics.mean(t[0] for t in tot),
            "accepted_committed_per_step": statistics.mean(t[1] for t in tot),
            "trimmed_away_per_step": statistics.mean(t[0] - t[1] for t in tot),
            "mean_window": mean_L_of(sets, B),
            "commit_equals_compact_sets": f"{same}/{len(audit)}",
            "commit_equals_compact_requests": f"{same_req}/{len(audit) * B}"}

    entropy_arm = None
    if not args.no_entropy_arm:
        ent = [prepare_set(W, binding, w, s, entropy_theta=ENTROPY_THETA) for s in range(len(sets))]
        eve = entropy_loop(binding, ent, args.steps, args.warmup, flush, stream, ENTROPY_THETA)
        for st in ent:
            assert torch.equal(st["bufs"].L, st["L_ref"]), "entropy verify lengths changed"
            assert st["bufs"].device_status() == 0
        ems = statistics.mean(e0.elapsed_time(e2) for e0, _, e2 in eve)
        sms = statistics.mean(e0.elapsed_time(e1) for e0, e1, _ in eve)
        sbytes = B * g * V * ls + 4 * (2 * B * g + 4 * B + 2)
        entropy_arm = {
            "theta": ENTROPY_THETA, "ms_per_step": ems, "steps_per_s": 1000.0 / ems,
            "score_entropy_us": sms * 1000.0, "score_entropy_bytes_per_launch": sbytes,
            "score_entropy_gbs": sbytes / (sms * 1e-3) / 1e9,
            "score_entropy_frac": sbytes / (sms * 1e-3) / 1e9 / peak,
            "mean_L": mean_L_of(ent, B),
            "committed_tokens_per_step": statistics.mean(
                float(st["bufs"].num_emitted.sum().item()) for st in ent)}

    sts_fit = None
    if not args.no_sts_fit:
        # STS temperatures fitted to the logs of the timed step (conf, L and
        # accept lengths of every input set), timed with events.
        conf = torch.cat([st["bufs"].conf for st in sets])
        Lg = torch.cat([st["bufs"].L for st in sets])
        ag = torch.cat([st["bufs"].accept_len for st in sets])
        tu = sets[0]["inp"]["sts_tau"]
        tau = torch.empty(g, dtype=torch.float32, device="cuda")
        nobs = torch.empty(g, dtype=torch.int32, device="cuda")
        for _ in range(3):
            binding.dspark_fit_sts_tau(conf, tu, Lg, ag, tau, n_obs=nobs)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        f0.record()
        for _ in range(reps):
            binding.dspark_fit_sts_tau(conf, tu, Lg, ag, tau, n_obs=nobs)
        f1.record()
        torch.cuda.synchronize()
        sts_fit = {"logged_request_steps": int(conf.shape[0]),
                   "us_per_fit": f0.elapsed_time(f1) * 1000.0 / reps,
                   "tau_used": [round(float(v), 4) for v in tu.tolist()],
                   "tau_fit": [round(float(v), 4) for v in tau.tolist()],
                   "observations": nobs.tolist()}

    latency = None
    if not args.no_latency:
        # one B=1 step's inputs (~5 MB) fit in L2: flush before every step
        latency = run_latency(binding, W)

    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = run_e2e(binding, W, sets[0], args.e2e_steps, stream)
        e2e_total = reduce_max(e2e_ms, world, "cuda")
        e2e = {"value": world * 1000.0 / e2e_total, "unit": "steps/s",
               "ms_per_step": e2e_total, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps}

    cpu = cpu_omp = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_oracle(W, sets[0], args.cpu_seconds)
        cpu_omp = cpu_baseline_oracle(W, sets[0], args.cpu_seconds, threads=os.cpu_count() or 1)
        parity = parity_of_set0(W, sets[0])

    if rank != 0:
        return None
    mean_L = mean_L_of(sets, B)
    return {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {**workload_config(w),
                   "input_sets": P, "parallelism": "replicas" if world > 1 else "single",
                   "l2": flush.describe(step_bytes),
                   "timing": "CUDA events around score_compact+verify per step"},
        "us_per_step": ms_per_step * 1000.0,
        "hbm_gbs_step": step_bytes / (ms_per_step * 1e-3) / 1e9,
        "hbm_frac_step": step_bytes / (ms_per_step * 1e-3) / 1e9 / peak,
        "hbm_frac_step_of_spec": step_bytes / (ms_per_step * 1e-3) / 1e9 / SPEC_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     # the committed capture is of the default workload only
                     "traffic": profiled_traffic() if w.name == DEFAULT_WORKLOAD else None,
                     "kernel": "verify_kernel", "peak_kind": peak_kind,
                     "frac_of_spec": achieved / SPEC_HBM_GBS, "spec_peak": SPEC_HBM_GBS,
                     "bytes_per_launch": statistics.mean(vb), "launch_us": ver_mean * 1000.0,
                     "early_exit_logit_bytes_per_launch": statistics.mean(
                         sets[i % P]["early_exit_bytes"] for i in range(args.steps))},
        "score_budget_compact_us": statistics.mean(sb_ms) * 1000.0,
        "cpu_baseline": cpu, "cpu_baseline_omp": cpu_omp, "parity": parity,
        "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clocks,
        "mean_L": mean_L,
        "committed_tokens_per_step": statistics.mean(
            float(st["bufs"].num_emitted.sum().item()) for st in sets),
        "fixed_budget_arm": fixed_arm,
        "cap_accept_arm": audit_arm,
        "entropy_arm": entropy_arm,
        "sts_fit": sts_fit,
        "latency_b1": latency,
    }


# --------------------------------------------------------------------------- #
# reference arm: the CPU oracle
# --------------------------------------------------------------------------- #
def run_reference(args, rank, world):
    """The oracle on the metric's own configuration: input set 0 of the
    workload, every request, the cap as configured; each step a full step."""
    if rank != 0:
        return None
    import oracle
    from confidence_driven_speculative_gb300 import workloads as W
    oracle.build()
    w = W.WORKLOADS[args.workload]
    inp = W.to_numpy(W.make_inputs(w, 0))
    for _ in range(args.warmup):
        oracle.step(inp)
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.step(inp)
        t.append(time.perf_counter() - t0)
    step_s = statistics.mean(t)
    value = 1.0 / step_s
    sample = (f"each step: the oracle on the full input set 0 ({w.B} requests, "
              f"cap {w.cap_T}), single thread, {args.steps} steps after {args.warmup} warm-up")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1000.0, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": 1, "kind": "oracle",
                             "cpu": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
