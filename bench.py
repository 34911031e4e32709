"""Benchmark of the fused P-EAGLE drafting step (verify + rebuild + assemble).

One step = one pe_step launch over one batch of seeded synthetic inputs
already resident in HBM.  Default workload: large-batch decode, B=256 requests,
K'=7, K=7, H=2048, V=151936, bf16 (the configuration whose HBM-bandwidth
target is stated).  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, same metric

Timing: W untimed steps, then K steps, each bracketed by CUDA events on the
launching stream; between steps the L2 is flushed by writing a buffer of
twice its size (outside the events; --l2-flush write-read adds a read of
another such buffer, so that no dirty line of the flush is left for the step
to write back).  Multi-GPU (torchrun): every rank runs
its own independent requests (weak scaling, no collective on the data path);
the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from speculative_decoding_pe_gb300 import workloads as wl  # noqa: E402

METRIC = "verify+rebuild+assemble draft rows/s"
DTYPE_NAME = {torch.bfloat16: "bf16", torch.float32: "f32"}  # the JSON line's "dtype"
UNIT = "rows/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("speculative_decoding_pe_gb300/csrc/pe_step.cu",
                  "speculative_decoding_pe_gb300/csrc/pe_internal.cuh",
                  "speculative_decoding_pe_gb300/csrc/pe_tma.cuh",
                  "speculative_decoding_pe_gb300/csrc/pe_workspace.cuh")
SAMPLED_SOURCES = ("speculative_decoding_pe_gb300/csrc/pe_sampled.cu",
                   "speculative_decoding_pe_gb300/csrc/pe_internal.cuh")


# ------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    """Largest value of ``x`` across ranks (the timing reduction)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(rows_this_rank: float, ms_this_rank: float, world: int, device):
    """Whole-job throughput: rows of all ranks over the slowest rank's time."""
    ms = max_over_ranks(ms_this_rank, world, device)
    rows = sum_over_ranks(rows_this_rank, world, device)
    return rows / (ms / 1e3), ms, rows


def rank_seed(workload: str, rank: int) -> int:
    """Each rank draws its own independent requests."""
    return 5000 + 97 * (list(wl.SPECS).index(workload) + 1) + rank


# ------------------------------------------------------------ byte counts

def algorithmic_bytes(spec: wl.WorkloadSpec, R: int, logits_rows: int | None = None) -> dict:
    """Bytes one step must move at minimum (each byte counted once).

    logits: every row read once; hidden: every target row read once;
    emb: one table row per verified / prompt slot plus the MASK row (the
    repeated MASK-row reads hit L2); X: written once; metadata: 18 bytes per
    output slot (token, position, two masks, slot id) plus the per-row and
    per-request integers.  With early exit, ``logits_rows`` is the number of
    rows a greedy verifier must read (rows 0..a_b of each request)."""
    B, Kp, K, V, H = spec.B, spec.Kp, spec.K, spec.V, spec.H
    elt = torch.tensor([], dtype=spec.dtype).element_size()
    Rl = B * (Kp + 1) if logits_rows is None else logits_rows
    T = R + B * (K - 1)
    parts = {
        "logits": Rl * V * elt,
        "hidden": R * H * elt,
        "emb": (R + 1) * H * elt,
        "X": T * 2 * H * elt,
        "metadata": 18 * T + 12 * R + 4 * (B + 1) + 8 * B + 4 * B * K + 4 * Rl,
    }
    parts["total"] = sum(parts.values())
    return parts


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C / CUDA source without comments, trailing blanks and empty lines:
    what the compiler sees, so that a comment edit keeps a profile current.
    (String literals holding comment markers are not special-cased; the
    kernel sources have none.)"""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    """Hash of the kernel sources' code (comments ignored)."""
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "pe_step", sources=KERNEL_SOURCES):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel, workload))
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16\s*=\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch\s*=\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(sources):
        return None
    return int(m_bytes.group(1))


# ------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running.

    Started before the warm-up (nvidia-smi takes a moment to print its first
    sample); ``stop(t0, t1)`` keeps the samples taken between t0 and t1
    (wall clock), waiting briefly for one past t1 to arrive."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    @staticmethod
    def _stamp(text: str) -> float:
        whole, _, frac = text.strip().partition(".")
        ts = time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S"))
        return ts + (float("0." + frac) if frac.isdigit() else 0.0)

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(max(0.0, min(0.5, t1 + 0.3 - time.time())))  # let a sample past t1 land
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for rec in csv.reader(io.StringIO(out)):
            if len(rec) < 10:
                continue
            try:
                rows.append((self._stamp(rec[0]), [r.strip() for r in rec]))
            except ValueError:
                continue
        inside = [r for ts, r in rows if t0 <= ts <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4)
                          if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


def soak(step, flush, seconds: float, device):
    """Run the same (flush, step) pair, untimed, for about ``seconds`` after
    the timed region, so that the clock samples see the GPU under this load
    even when the timed region itself is too short to sample."""
    t_end = time.time() + seconds
    n = 0
    while time.time() < t_end:
        for _ in range(20):
            flush()
            step()
        n += 20
        torch.cuda.synchronize(device)
    return n


# ------------------------------------------------------------ CPU oracle

def sub_workload(w, nreq: int):
    """The first ``nreq`` requests of a workload, on the host."""
    import dataclasses
    spec = w.spec.with_(B=nreq)
    rows = nreq * (w.Kp + 1)
    if w.in_offsets is not None:
        R = int(w.in_offsets[nreq])
        offs = w.in_offsets[:nreq + 1].cpu()
    else:
        R = rows
        offs = None
    return dataclasses.replace(
        w, spec=spec, logits=w.logits[:rows].cpu().contiguous(), in_offsets=offs,
        in_tokens=w.in_tokens[:R].cpu(), in_positions=w.in_positions[:R].cpu(),
        block_table=w.block_table[:nreq].cpu(), emb=w.emb.cpu(), hidden=w.hidden[:R].cpu(),
        h_shared=w.h_shared.cpu(), planted_accept=w.planted_accept[:nreq],
        planted_bonus=w.planted_bonus[:nreq])


def time_oracle(sub, budget_s: float, min_runs: int = 1):
    """Run the oracle step on ``sub`` until ``budget_s`` seconds have passed."""
    import oracle
    times = []
    start = time.perf_counter()
    while len(times) < min_runs or time.perf_counter() - start < budget_s:
        t0 = time.perf_counter()
        oracle.step(sub)
        times.append(time.perf_counter() - t0)
    return times


def pick_sample_requests(w, per_step_s: float) -> int:
    probe = sub_workload(w, 1)
    t = min(time_oracle(probe, 0.0, min_runs=2))
    return max(1, min(w.B, int(per_step_s / max(t, 1e-6))))


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ------------------------------------------------------------ arms

def config_of(spec, extra=None, l2_mode="write") -> dict:
    c = {"workload": spec.name, "description": spec.description, "B": spec.B,
         "Kp": spec.Kp, "K": spec.K, "H": spec.H, "V": spec.V,
         "dtype": str(spec.dtype).replace("torch.", ""),
         "l2": L2Flush.describe_mode(l2_mode),
         "parallelism": "requests sharded across ranks, no data-path collective"}
    if extra:
        c.update(extra)
    return c


class L2Flush:
    """Evicts the L2 between timed steps, outside the events.  "write" (the
    default) writes a buffer twice the L2's size.  That leaves the L2 full of
    the flush's dirty lines, which the next step then writes back to HBM
    while it streams (about 6 us of a B=256 step).  "write-read" follows the
    write with a read of another such buffer, so no dirty line is left and
    the step is timed on a clean, cold L2."""

    def __init__(self, device, mode="write"):
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.mode = mode
        self.buf = torch.empty(2 * l2, dtype=torch.uint8, device=device)
        if mode == "write-read":
            self.rbuf = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
            self.acc = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.zero_()
        if self.mode == "write-read":
            torch.sum(self.rbuf, dim=0, out=self.acc)

    @staticmethod
    def describe_mode(mode: str) -> str:
        if mode == "write-read":
            return "flushed between timed steps (write of 2x L2, then a read of 2x L2)"
        return "flushed between timed steps (write of 2x L2)"

    def describe(self) -> str:
        return self.describe_mode(self.mode)


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    spec = wl.SPECS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = wl.make_workload(spec, rank_seed(args.workload, 0), device=dev)
    per_step = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    nreq = pick_sample_requests(w, per_step)
    sub = sub_workload(w, nreq)
    import oracle
    for _ in range(args.warmup):
        oracle.step(sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.step(sub)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    T = sub.R + nreq * (spec.K - 1)
    value = T / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype":
        DTYPE_NAME[spec.dtype], "data": "synthetic",
        "config": config_of(spec),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "first %d of %d requests per step (%d draft rows), "
                                   "single-threaded C oracle on %s" % (
                                       nreq, spec.B, T, cpu_model())},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    rank, world, local = dist_env()
    if world != args.gpus:
        raise SystemExit("--gpus %d but WORLD_SIZE=%d" % (args.gpus, world))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    from speculative_decoding_pe_gb300 import _native, harness
    _native.load()  # fails loudly when the CUDA library is missing
    if args.tuning:
        _native.set_tuning(**json.loads(args.tuning))

    sampler = ClockSampler(local)
    spec = wl.SPECS[args.workload]
    w = wl.make_workload(spec, rank_seed(args.workload, rank), device=device)
    out, ws, err = harness.allocate(w, device)
    packed = harness.pack(w, out, ws, err)
    flush = L2Flush(device, args.l2_flush)
    stream = torch.cuda.current_stream(device)

    run_step = _native.step_early_exit_packed if args.early_exit else _native.step_packed

    def step():
        run_step(packed, stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(device)
    if int(err.item()) != 0:
        raise SystemExit("device error word %d on warm-up" % int(err.item()))

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    torch.cuda.nvtx.range_push("timed")
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(device)
    barrier(world)
    soak_steps = soak(step, flush, args.clock_soak, device)
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1)
    clocks["window"] = ("the timed region, then %d more flush+step pairs (untimed, %.1f s) "
                        "of the same step" % (soak_steps, args.clock_soak))
    if int(err.item()) != 0:
        raise SystemExit("device error word %d after the timed steps" % int(err.item()))
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    mean_ms = sum(step_ms) / len(step_ms)
    T = w.T
    value, mean_ms_max, rows_all = aggregate(float(T), mean_ms, world, device)

    needed = None
    if args.early_exit:  # rows 0..a_b of each request, a_b as planted
        needed = int((w.planted_accept.long() + 1).sum())
    bytes_ = algorithmic_bytes(spec, w.R, needed)
    peak, peak_kind = measured_peak()
    achieved = bytes_["total"] / (mean_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": profiled_traffic(args.workload,
                                            "pe_step_early_exit" if args.early_exit else "pe_step"),
                "peak_source": peak_kind, "algorithmic_bytes_per_launch": bytes_["total"],
                "kernel": "pe::step_kernel<%s, early_exit=%s>" % (
                    "bf16" if spec.dtype == torch.bfloat16 else "f32",
                    "true" if args.early_exit else "false")}

    e2e = measure_e2e(w, out, ws, err, packed, stream, device, args) if args.e2e else None
    if e2e is not None:
        e2e_ms = max_over_ranks(e2e["ms"], world, device)
        e2e = {"value": rows_all / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
               "ms_per_step": e2e_ms, "scope": E2E_SCOPE}

    graph = measure_graph(spec, args, device, run_step) if args.graph else None

    workloads = None
    if args.workloads and not args.early_exit and args.workload == "decode_b256":
        workloads = measure_workloads(args, device, flush, rank)

    cpu = None
    if rank == 0 and world == 1 and args.cpu_baseline:
        cpu = measure_cpu_baseline(w, args.cpu_budget)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_NAME[spec.dtype], "data": "synthetic",
            "config": config_of(spec, {"T_per_rank": T, "R_per_rank": w.R,
                                       "early_exit": bool(args.early_exit),
                                       "logits_rows_needed": needed,
                                       "median_us": statistics.median(step_ms) * 1e3,
                                       "min_us": min(step_ms) * 1e3,
                                       "p99_us": sorted(step_ms)[int(0.99 * (len(step_ms) - 1))] * 1e3,
                                       "max_us": max(step_ms) * 1e3,
                                       "tuning": _native.get_tuning()}, l2_mode=flush.mode),
            "us_per_step": mean_ms_max * 1e3,
            "hbm_gbs": achieved,
            "roofline": roofline,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": args.steps,
            "clocks": clocks,
        }
        if graph is not None:
            line["graph"] = graph
        if workloads is not None:
            line["workloads"] = workloads
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


SAMPLED_METRIC = "rejection-sampling verification logits rows/s"
SAMPLED_SHAPE = {"B": 256, "Kp": 7, "V": 151936}  # the large-batch decode shape


def sampled_bytes(B, Kp, V, elt, rejected: int) -> dict:
    """Bytes the two-pass rejection-sampling verification must move: every
    target and draft row once (statistics, probabilities, bonus-row draw),
    then the target and draft row at the rejected position of each request
    with a rejection again (the residual needs both rows' normalisers before
    it can be drawn), plus tokens, coins and the two outputs."""
    rows = B * (Kp + 1) + B * Kp
    parts = {"logits": rows * V * elt, "residual_reread": rejected * 2 * V * elt,
             "metadata": 4 * B * (Kp + 1) + 4 * B * Kp + 8 * B}
    parts["total"] = sum(parts.values())
    return parts


def sampled_setup(device, rank, temperature):
    """Inputs, outputs and the launch of one pe_verify_sampled call on the
    large-batch decode shape."""
    from speculative_decoding_pe_gb300 import _native
    B, Kp, V = SAMPLED_SHAPE["B"], SAMPLED_SHAPE["Kp"], SAMPLED_SHAPE["V"]
    s = wl.make_sampled_inputs(B, Kp, V, dtype=torch.bfloat16, seed=7100 + rank, device=device)
    acc = torch.empty(B, dtype=torch.int32, device=device)
    bon = torch.empty(B, dtype=torch.int32, device=device)
    ws = torch.zeros(_native.workspace_bytes_sampled(B, Kp), dtype=torch.uint8, device=device)
    err = _native.new_error_word(device)
    stream = torch.cuda.current_stream(device)

    def step():
        _native.verify_sampled(s.target_logits, s.draft_logits, Kp, s.tokens, s.u_accept,
                               temperature, 1234 + rank, acc, bon, ws, err, stream)
    return s, acc, bon, ws, err, step


def sampled_entry(args, device, flush, rank, steps, warm):
    peak, _ = measured_peak()
    B, Kp, V = SAMPLED_SHAPE["B"], SAMPLED_SHAPE["Kp"], SAMPLED_SHAPE["V"]
    s, acc, bon, ws, err, step = sampled_setup(device, rank, args.temperature)
    ms = time_steps(step, flush, torch.cuda.current_stream(device), steps, warm)
    if int(err.item()) != 0 or int(ws.count_nonzero()) != 0:
        raise SystemExit("sampled: device error word or workspace not zero")
    rejected = int((acc < Kp).sum())
    return _entry(ms, sampled_bytes(B, Kp, V, 2, rejected)["total"], peak,
                  {"entry": "pe_verify_sampled", "rejecting_requests": rejected,
                   "temperature": args.temperature})


def run_sampled(args):
    """Time pe_verify_sampled (two launches per step) on the large-batch
    decode shape: B=256, K'=7, V=151936, bf16, temperature --temperature."""
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    from speculative_decoding_pe_gb300 import _native
    _native.load()
    sampler = ClockSampler(local)
    B, Kp, V = SAMPLED_SHAPE["B"], SAMPLED_SHAPE["Kp"], SAMPLED_SHAPE["V"]
    s, acc, bon, ws, err, step = sampled_setup(device, rank, args.temperature)
    flush = L2Flush(device, args.l2_flush)
    stream = torch.cuda.current_stream(device)
    T = args.temperature

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(device)
    if int(err.item()) != 0 or int(ws.count_nonzero()) != 0:
        raise SystemExit("device error word or workspace not zero after warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    torch.cuda.nvtx.range_push("timed")
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(device)
    barrier(world)
    soak(step, flush, args.clock_soak, device)
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1)
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    mean_ms = sum(step_ms) / len(step_ms)
    rows = B * (Kp + 1) + B * Kp
    value, mean_ms_max, _ = aggregate(float(rows), mean_ms, world, device)
    rejected = int((acc < Kp).sum())
    bytes_ = sampled_bytes(B, Kp, V, 2, rejected)
    peak, peak_kind = measured_peak()
    achieved = bytes_["total"] / (mean_ms / 1e3) / 1e9

    cpu = None
    if rank == 0 and world == 1 and args.cpu_baseline:
        import oracle  # CPU baseline leg only
        host = s.to("cpu")
        nreq = 4
        sub = wl.SampledInputs(B=nreq, Kp=Kp, V=V,
                               target_logits=host.target_logits[:nreq * (Kp + 1)],
                               draft_logits=host.draft_logits[:nreq * Kp],
                               tokens=host.tokens[:nreq * (Kp + 1)],
                               u_accept=host.u_accept[:nreq * Kp])
        times = []
        t_end = time.time() + args.cpu_budget
        while len(times) < 3 or time.time() < t_end:
            t0 = time.perf_counter()
            oracle.verify_sampled(sub.target_logits, sub.draft_logits, nreq, Kp, sub.tokens,
                                  sub.u_accept, T, 1234)
            times.append(time.perf_counter() - t0)
        t = statistics.median(times)
        cpu = {"value": nreq * (2 * Kp + 1) / t, "unit": "rows/s", "cores": 1,
               "kind": "oracle",
               "sample": "first %d of %d requests, %d runs, median %.1f ms, "
                         "single-threaded C oracle on %s" % (
                             nreq, B, len(times), t * 1e3, cpu_model())}
    if rank == 0:
        print(json.dumps({
            "metric": SAMPLED_METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "rejection-sampling verification B=%d K'=%d V=%d bf16 "
                                   "T=%g" % (B, Kp, V, T),
                       "accepted_len_histogram": torch.bincount(
                           acc.long().cpu(), minlength=Kp + 1).tolist(),
                       "l2": flush.describe(),
                       "median_us": statistics.median(step_ms) * 1e3,
                       "min_us": min(step_ms) * 1e3},
            "us_per_step": mean_ms_max * 1e3,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": profiled_traffic("decode_b256", "pe_verify_sampled",
                                                     SAMPLED_SOURCES),
                         "peak_source": peak_kind,
                         "algorithmic_bytes_per_launch": bytes_["total"],
                         "bytes": bytes_,
                         "kernel": "pe::sampled_stats_kernel + pe::sampled_residual_kernel "
                                   "(one call, two launches)"},
            "cpu_baseline": cpu, "gpu_launches": 2 * args.steps, "clocks": clocks}))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


READOUT_METRIC = "greedy drafter readout rows/s"
READOUT_SHAPE = {"B": 256, "K": 7, "V": 151936}  # the large-batch decode shape


def readout_setup(device, rank):
    """Drafter logits for B*K sampled rows, outputs, and the launch of one
    pe_draft_readout call."""
    from speculative_decoding_pe_gb300 import _native
    B, K, V = READOUT_SHAPE["B"], READOUT_SHAPE["K"], READOUT_SHAPE["V"]
    n = B * K
    g = torch.Generator(device=device)
    g.manual_seed(7300 + rank)
    logits = (torch.randn(n, V, generator=g, device=device) * 2.0).to(torch.bfloat16)
    out = torch.empty(n, dtype=torch.int32, device=device)
    ws = _native.new_workspace(n, n, device)
    err = _native.new_error_word(device)
    stream = torch.cuda.current_stream(device)

    def step():
        _native.draft_readout(logits, out, ws, err, None, stream)
    return logits, out, ws, err, step


def readout_entry(args, device, flush, rank, steps, warm):
    peak, _ = measured_peak()
    logits, out, ws, err, step = readout_setup(device, rank)
    ms = time_steps(step, flush, torch.cuda.current_stream(device), steps, warm)
    if int(err.item()) != 0 or int(ws.count_nonzero()) != 0:
        raise SystemExit("readout: device error word or workspace not zero")
    n, V = logits.shape
    return _entry(ms, n * V * 2 + 4 * n, peak, {"entry": "pe_draft_readout"})


def run_readout(args):
    """Time pe_draft_readout (one launch) on the drafter's logits for the K
    sampled rows of each of B requests: argmax of B*K rows of V columns,
    bf16, N(0, 2), the drafter computing only the sampled rows."""
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    from speculative_decoding_pe_gb300 import _native
    _native.load()
    sampler = ClockSampler(local)
    B, K, V = READOUT_SHAPE["B"], READOUT_SHAPE["K"], READOUT_SHAPE["V"]
    n = B * K
    logits, out, ws, err, step = readout_setup(device, rank)
    flush = L2Flush(device, args.l2_flush)
    stream = torch.cuda.current_stream(device)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(device)
    if int(err.item()) != 0 or int(ws.count_nonzero()) != 0:
        raise SystemExit("device error word or workspace not zero after warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    torch.cuda.nvtx.range_push("timed")
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(device)
    barrier(world)
    soak(step, flush, args.clock_soak, device)
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1)
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    mean_ms = sum(step_ms) / len(step_ms)
    value, mean_ms_max, _ = aggregate(float(n), mean_ms, world, device)
    total = n * V * 2 + 4 * n  # logits read once, tokens written
    peak, peak_kind = measured_peak()
    achieved = total / (mean_ms / 1e3) / 1e9

    cpu = None
    if rank == 0 and world == 1 and args.cpu_baseline:
        import oracle  # CPU baseline leg only
        rows = 64
        host = logits[:rows].cpu()
        times = []
        t_end = time.time() + args.cpu_budget
        while len(times) < 3 or time.time() < t_end:
            t0 = time.perf_counter()
            oracle.draft_readout(host)
            times.append(time.perf_counter() - t0)
        t = statistics.median(times)
        cpu = {"value": rows / t, "unit": "rows/s", "cores": 1, "kind": "oracle",
               "sample": "first %d of %d rows, %d runs, median %.1f ms, single-threaded C "
                         "oracle on %s" % (rows, n, len(times), t * 1e3, cpu_model())}
    if rank == 0:
        print(json.dumps({
            "metric": READOUT_METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "greedy drafter readout B=%d K=%d V=%d bf16" % (B, K, V),
                       "l2": flush.describe(),
                       "median_us": statistics.median(step_ms) * 1e3,
                       "min_us": min(step_ms) * 1e3,
                       "tuning": _native.get_tuning()},
            "us_per_step": mean_ms_max * 1e3,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": profiled_traffic("decode_b256", "pe_draft_readout"),
                         "peak_source": peak_kind, "algorithmic_bytes_per_launch": total,
                         "kernel": "pe::step_kernel<bf16> (readout: argmax units only)"},
            "cpu_baseline": cpu, "gpu_launches": args.steps, "clocks": clocks}))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


E2E_SCOPE = ("every input the step reads that changes from step to step (logits, target "
             "hidden rows, input tokens and positions, block table, prompt offsets) copied "
             "in from pinned host memory, and every output (accepted lengths, bonus tokens, "
             "per-row argmax, offsets, tokens, positions, masks, hidden map, slot mapping, "
             "sample_idx and X) copied back, every step; the embedding table and h_shared "
             "stay resident")


def measure_e2e(w, out, ws, err, packed, stream, device, args):
    """The same step through the public API with its per-step inputs copied
    in from pinned host memory and all of its outputs copied back, every
    step (see E2E_SCOPE)."""
    from speculative_decoding_pe_gb300 import _native, harness
    per_step = [w.logits, w.hidden, w.in_tokens, w.in_positions, w.block_table]
    if w.in_offsets is not None:
        per_step.append(w.in_offsets)
    host = []
    for t in per_step:
        if t.dim() == 2 and t.stride(0) != t.shape[1]:
            base = t.as_strided((t.shape[0], t.stride(0)), (t.stride(0), 1))
            host.append((base, base.cpu().pin_memory()))
        else:
            host.append((t, t.cpu().pin_memory()))
    res_dev = [getattr(out, k) for k in harness.OUTPUT_KEYS if getattr(out, k) is not None]
    res_host = [torch.empty_like(r, device="cpu").pin_memory() for r in res_dev]
    h2d = sum(h.numel() * h.element_size() for _, h in host)
    d2h = sum(r.numel() * r.element_size() for r in res_host)
    n = max(3, min(args.steps, args.e2e_steps))

    run_step = _native.step_early_exit_packed if args.early_exit else _native.step_packed

    def one():
        for d, h in host:
            d.copy_(h, non_blocking=True)
        run_step(packed, stream)
        for d, h in zip(res_dev, res_host):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        one()
    e1.record(stream)
    torch.cuda.synchronize(device)
    return {"ms": e0.elapsed_time(e1) / n, "h2d": h2d, "d2h": d2h}


def time_steps(step, flush, stream, steps: int, warmup: int):
    """Per-step milliseconds of ``step`` (CUDA events on ``stream``, the L2
    flushed before each step, outside the events)."""
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


def time_graph(fn_list, stream, reps: int):
    """Microseconds per captured call: ``fn_list`` (launches on the current
    stream) captured once in a CUDA graph, replayed ``reps`` times."""
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        for f in fn_list:
            f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for f in fn_list:
            f()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(reps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * len(fn_list))


def _entry(step_ms, total_bytes, peak, extra=None):
    mean = sum(step_ms) / len(step_ms)
    achieved = total_bytes / (mean / 1e3) / 1e9
    e = {"us_per_step": mean * 1e3, "median_us": statistics.median(step_ms) * 1e3,
         "min_us": min(step_ms) * 1e3, "algorithmic_bytes": total_bytes,
         "achieved_gbs": achieved, "roofline_frac": achieved / peak}
    if extra:
        e.update(extra)
    return e


def measure_workloads(args, device, flush, rank):
    """Every other workload and every further entry point, each timed like
    the headline (CUDA events per launch, L2 flushed between launches):
    decode_b1 / decode_b64 / prefill_b8 / tiny through pe_step; decode_b1
    also inside a CUDA graph, against the latency floor (an empty launch of
    the step's grid, and the same plus one dependent global round trip);
    early exit at B=256 (against the bytes of the rows it needs); the
    drafter readout; rejection sampling; the no-allocation step."""
    from speculative_decoding_pe_gb300 import _native, harness
    peak, _ = measured_peak()
    stream = torch.cuda.current_stream(device)
    steps, warm = args.workload_steps, max(3, args.warmup)
    res = {}
    for name in ("decode_b1", "decode_b64", "prefill_b8", "tiny"):
        spec = wl.SPECS[name]
        w = wl.make_workload(spec, rank_seed(name, rank), device=device)
        out, ws, err = harness.allocate(w, device)
        packed = harness.pack(w, out, ws, err)
        ms = time_steps(lambda: _native.step_packed(packed, stream), flush, stream, steps, warm)
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise SystemExit("device error word %d (%s)" % (int(err.item()), name))
        b = algorithmic_bytes(spec, w.R)["total"]
        res[name] = _entry(ms, b, peak, {"rows_per_s": w.T / (sum(ms) / len(ms) / 1e3),
                                         "entry": "pe_step"})
        if name == "decode_b1":
            # the same step captured 16 times (16 input sets) in one graph
            ws_list = [wl.make_workload(spec, 9100 + i, device=device) for i in range(16)]
            wsp = _native.new_workspace(spec.B * (spec.Kp + 1), spec.B, device)
            bufs = [harness.allocate(x, device) for x in ws_list]
            packs = [harness.pack(x, o, wsp, e) for x, (o, _, e) in zip(ws_list, bufs)]
            res[name]["graph_us_per_step"] = time_graph(
                [lambda a=a: _native.step_packed(a) for a in packs], stream, 50)
            grid = torch.cuda.get_device_properties(device).multi_processor_count * \
                _native.get_tuning()["ctas_per_sm"]
            chain = torch.zeros(1, dtype=torch.int32, device=device)
            sink = torch.zeros(1, dtype=torch.int32, device=device)
            empty = time_steps(lambda: _native.latency_floor(grid, 0, stream=stream), flush,
                               stream, steps, warm)
            hop = time_steps(lambda: _native.latency_floor(grid, 1, chain, sink, stream),
                             flush, stream, steps, warm)
            res[name]["floor"] = {
                "grid_ctas": grid,
                "empty_launch_us": statistics.median(empty) * 1e3,
                "empty_plus_one_round_trip_us": statistics.median(hop) * 1e3,
                "empty_launch_graph_us": time_graph(
                    [lambda: _native.latency_floor(grid, 0)] * 16, stream, 50),
                "empty_plus_one_round_trip_graph_us": time_graph(
                    [lambda: _native.latency_floor(grid, 1, chain, sink)] * 16, stream, 50),
                "note": "launched: the L2 flushed before each launch, so the round trip "
                        "goes to HBM; in the graph it hits L2"}
            del ws_list, bufs, packs
        del w, out, ws, err, packed
        torch.cuda.empty_cache()
    # early exit at B=256: rows 0..a_b of each request are what it must read
    spec = wl.SPECS["decode_b256"]
    w = wl.make_workload(spec, rank_seed("decode_b256", rank), device=device)
    out, ws, err = harness.allocate(w, device)
    packed = harness.pack(w, out, ws, err)
    ms = time_steps(lambda: _native.step_early_exit_packed(packed, stream), flush, stream,
                    steps, warm)
    needed = int((w.planted_accept.long() + 1).sum())
    res["early_exit_decode_b256"] = _entry(
        ms, algorithmic_bytes(spec, w.R, needed)["total"], peak,
        {"entry": "pe_step_early_exit", "logits_rows_needed": needed,
         "logits_rows": w.B * (w.Kp + 1)})
    # the no-allocation step (its scratch cleared by a memset each call)
    lib = _native.load()
    import ctypes
    nb = algorithmic_bytes(spec, w.R)["total"]
    def noalloc_call(args_):
        if lib.pe_step_noalloc(ctypes.byref(args_), ctypes.c_void_p(stream.cuda_stream)) != 0:
            raise SystemExit("pe_step_noalloc rejected its arguments")

    ms = time_steps(lambda: noalloc_call(packed), flush, stream, steps, warm)
    res["noalloc_decode_b256"] = _entry(ms, nb, peak, {"entry": "pe_step_noalloc"})
    del w, out, ws, err, packed
    w1 = wl.make_workload("decode_b1", rank_seed("decode_b1", rank), device=device)
    out1, ws1, err1 = harness.allocate(w1, device)
    p1 = harness.pack(w1, out1, ws1, err1)
    ms = time_steps(lambda: noalloc_call(p1), flush, stream, steps, warm)
    res["noalloc_decode_b1"] = _entry(ms, algorithmic_bytes(w1.spec, w1.R)["total"], peak,
                                      {"entry": "pe_step_noalloc"})
    del w1, out1, ws1, err1, p1
    torch.cuda.empty_cache()
    # drafter readout and rejection sampling (their own bench modes)
    res["readout_decode_b256"] = readout_entry(args, device, flush, rank, steps, warm)
    res["sampled_decode_b256"] = sampled_entry(args, device, flush, rank, steps, warm)
    return res


def measure_graph(spec, args, device, run_step):
    """N steps, each over its own input set, captured in one CUDA graph and
    replayed; events around whole replays.  No L2 flush: the N input sets
    are distinct (for the large workloads they are far larger than L2)."""
    from speculative_decoding_pe_gb300 import _native, harness
    n = args.graph
    ws_list = [wl.make_workload(spec, 9000 + i, device=device) for i in range(n)]
    ws = _native.new_workspace(spec.B * (spec.Kp + 1), spec.B, device)
    bufs = [harness.allocate(w, device) for w in ws_list]
    packed = [harness.pack(w, out, ws, err) for w, (out, _, err) in zip(ws_list, bufs)]
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for a in packed:
            run_step(a, s)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for a in packed:
            run_step(a, torch.cuda.current_stream(device))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(device)
    reps = max(3, args.steps // n)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(device)
    e0.record(cur)
    for _ in range(reps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize(device)
    us = e0.elapsed_time(e1) * 1e3 / (reps * n)
    return {"steps_per_graph": n, "replays": reps, "us_per_step": us,
            "value": float(ws_list[0].T) / (us * 1e-6), "unit": UNIT,
            "inputs": "%d distinct input sets, no flush between steps" % n}


def measure_cpu_baseline(w, budget_s: float):
    nreq = pick_sample_requests(w, budget_s / 20)
    sub = sub_workload(w, nreq)
    times = time_oracle(sub, budget_s, min_runs=3)
    T = sub.R + nreq * (w.K - 1)
    t = statistics.median(times)
    return {"value": T / t, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "first %d of %d requests (%d draft rows), %d runs, median %.1f ms, "
                      "single-threaded C oracle on %s" % (
                          nreq, w.B, T, len(times), t * 1e3, cpu_model())}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(wl.SPECS), default="decode_b256")
    ap.add_argument("--tuning", default="", help="JSON launch-shape knobs")
    ap.add_argument("--l2-flush", choices=["write", "write-read"], default="write",
                    help="how the L2 is evicted between timed steps (see L2Flush)")
    ap.add_argument("--graph", type=int, default=0,
                    help="also time N steps captured in one CUDA graph")
    ap.add_argument("--early-exit", action="store_true",
                    help="time pe_step_early_exit (rows after each request's first "
                         "mismatch are not read)")
    ap.add_argument("--readout", action="store_true",
                    help="time the greedy drafter readout (B=256 x K=7 rows, V=151936)")
    ap.add_argument("--sampled", action="store_true",
                    help="time rejection-sampling verification (pe_verify_sampled) "
                         "instead of the fused greedy step")
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the extra per-workload entries of the default line")
    ap.add_argument("--workload-steps", type=int, default=50,
                    help="timed launches per extra workload entry")
    ap.add_argument("--clock-soak", type=float, default=1.0,
                    help="seconds of untimed steps after the timed region, sampled "
                         "for the clocks record")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.sampled:
        return run_sampled(args)
    if args.readout:
        return run_readout(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
