#!/usr/bin/env python
"""Benchmark of the fused SwiGLU up-projection; prints ONE JSON line.

Workload (one "step"): the bf16 decode sweep -- one call for each
M in {1, 2, 4, 8, 16} at d=4096, d_ff=14336, weights N(0, 1/d) -- the
configuration the headline metric (HBM GB/s at M <= 16) is quoted on.
value = algorithmic bytes of all calls of all ranks / max-over-ranks time.
Algorithmic bytes per call = 2 (2 d d_ff + M d + M d_ff) (weights read once,
x read once, h written once).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--split replicas|columns]
With --gpus N > 1 outside torchrun the script re-launches itself under
torch.distributed.run with N local ranks.  Each rank runs its own replica of
the sweep (weak scaling, no collective on the data path), or with
--split columns its 64-aligned share of the d_ff columns of both weight
matrices (strong scaling, still no collective); the max time over ranks is
reported.

Besides the GPU timings, rank 0 runs the CPU oracle on bounded samples: the
headline cpu_baseline (all host cores and one core) and, for every timed
up-projection configuration, the oracle on a set of rows of the same call,
whose time is extrapolated to the whole call and whose result checks the GPU
output of the timed call (max error, normwise error, mismatch %).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

D, D_FF = 4096, 14336
SWEEP = (1, 2, 4, 8, 16)
WORKLOAD = "bf16_decode_d4096 (M in {1,2,4,8,16}, d=4096, d_ff=14336)"
METRIC = "SwiGLU up-proj: HBM GB/s at M≤16, TFLOP/s at M≥512, % of roofline"
L2_BYTES = 129 * 2 ** 20          # nominal; the measured value is read from the device


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the secondary per-config measurements")
    ap.add_argument("--extra-iters", type=int, default=30)
    ap.add_argument("--split", choices=["replicas", "columns"], default="replicas",
                    help="multi-rank data path: a replica of the sweep per rank, or each "
                         "rank's share of the d_ff columns")
    ap.add_argument("--no-oracle", action="store_true",
                    help="skip the CPU oracle leg (baseline timings and accuracy)")
    return ap.parse_args()


def quantiles(xs):
    """Median, 10th and 90th percentile of a list of times (nearest rank)."""
    xs = sorted(xs)
    if not xs:
        return {"median": None, "p10": None, "p90": None}
    pick = lambda q: xs[min(len(xs) - 1, max(0, int(round(q * (len(xs) - 1)))))]
    return {"median": statistics.median(xs), "p10": pick(0.10), "p90": pick(0.90)}


def bench_config():
    """The `config` both arms print (identical, so the two lines describe the
    same workload)."""
    return {"workload": WORKLOAD,
            "weights": "N(0,1/d) bf16, seed 0; the library arm reads them packed once "
                       "(step a0: gate and up 64-column blocks interleaved) outside the "
                       "timed region",
            "l2": "inputs larger than L2: 235 MB of weights per call, distinct weight "
                  "copies rotated per call, at least 2 GiB of them (no call finds an "
                  "earlier call's weights in L2)"}


def torchrun_argv(args, argv):
    """Command that re-runs this script under torch.distributed.run with
    args.gpus local ranks (used when --gpus N > 1 is given outside torchrun)."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            "--nproc-per-node", str(args.gpus), "--master-addr", "127.0.0.1",
            "--master-port", str(port), os.path.abspath(__file__)] + list(argv)


def max_over_ranks(value, world, device=None):
    """Largest `value` over all ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


TRAFFIC_FILE = os.path.join("profiles", "skinny_decode_traffic.json")


# Distinct weight bytes rotated through in every timed loop.  Weights are
# streamed with an L2 evict-first hint, and on GB300 a part of a weight set
# read two calls earlier was measured to still hit in L2 when fewer than
# about 1 GB of other weights came in between (the decode call at d = 4096,
# M = 1: 36.2 us with 2 copies of 235 MB, 38.4 us from 8 copies on; plain
# loads show no such effect).  A model's layers each read their own weights
# once per token, so the timed loops rotate at least 2 GiB of copies.
WEIGHT_FOOTPRINT = 2 << 30


def copies_for(l2, nbytes):
    """Weight copies rotated per call: at least 3 L2 capacities and
    WEIGHT_FOOTPRINT bytes of distinct weights, so that no call finds the
    weights of an earlier one in L2."""
    nbytes = max(int(nbytes), 1)
    return max(2, math.ceil(3 * l2 / nbytes), math.ceil(WEIGHT_FOOTPRINT / nbytes))


def profiled_traffic():
    """Mean DRAM bytes per launch of the decode kernel from the committed ncu
    capture, or None when the kernel sources changed since that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, TRAFFIC_FILE)) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for rel in rec["source_files"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["source_sha256"]:
            return None
        return int(rec["traffic_bytes_per_launch_mean"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """Polls SM clock, max SM clock and clock-event reasons every ~10 ms
    through NVML (read-only queries, via ctypes); falls back to nvidia-smi."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid):
        self.uuid = uuid
        self.samples = []          # (time, sm_mhz, max_mhz, reasons_bitmask)
        self.stop_evt = threading.Event()
        self.thread = None
        self.proc = None
        self.source = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if not self.uuid or lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
            if lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                raise OSError("no NVML device handle")
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, get_reasons

    def start(self):
        try:
            lib, h, get_reasons = self._nvml()
            self.source = "nvml"
        except (OSError, AttributeError):
            return self._start_smi()
        import ctypes

        def run():
            clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            while not self.stop_evt.is_set():
                if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                        get_reasons(h, ctypes.byref(rs)) == 0:
                    self.samples.append((time.time(), float(clk.value), float(mx.value), rs.value))
                time.sleep(0.01)
        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()

    def _start_smi(self):
        self.source = "nvidia-smi"
        cmd = ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd.insert(1, "--id=" + self.uuid)
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return

        def read():
            for line in self.proc.stdout:
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append((time.time(), float(parts[0]), float(parts[1]),
                                         int(parts[2], 16)))
                except (ValueError, IndexError):
                    continue
        self.thread = threading.Thread(target=read, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_evt.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1, settle0):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if len(inside) < 3:
            inside = [s for s in self.samples if settle0 <= s[0] <= t1]
            window = "settle+timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "source": self.source}
        bits = 0
        for s in inside:
            bits |= s[3]
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b)
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "window": window, "source": self.source}


def gpu_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle on the same workload
# ---------------------------------------------------------------------------

_ORACLE_INPUTS = {}


def _oracle_inputs(cols):
    """Seeded sweep inputs (x per M, first `cols` weight columns), drawn once."""
    if cols not in _ORACLE_INPUTS:
        from swiglu_mlp_projection_gb300 import inputs
        _, wg, wu = inputs.make_inputs(1, D, D_FF, "bf16", seed=0)
        xs = {M: inputs.raw_bits(inputs.make_inputs(M, D, D_FF, "bf16", seed=0, x_only=True)[0])
              for M in SWEEP}
        _ORACLE_INPUTS[cols] = (xs, inputs.raw_bits(wg[:, :cols]), inputs.raw_bits(wu[:, :cols]))
    return _ORACLE_INPUTS[cols]


ORACLE_COLS = 2048     # columns of the decode sweep in the oracle's timed sample


def oracle_sweep(cols, reps_budget_s, threads=None):
    """Time the oracle on the decode sweep restricted to the first `cols`
    columns (full K), repeated until `reps_budget_s` seconds have been spent;
    returns (GB/s, seconds, calls, threads)."""
    import oracle
    from swiglu_mlp_projection_gb300 import workload
    xs, wg_s, wu_s = _oracle_inputs(cols)
    threads = threads or oracle.default_threads()
    total_bytes, t_total, calls = 0, 0.0, 0
    while True:
        for M in SWEEP:
            t0 = time.perf_counter()
            oracle.swiglu_up(xs[M], wg_s, wu_s, oracle.BF16, nthreads=threads)
            t_total += time.perf_counter() - t0
            total_bytes += workload.algorithmic_bytes(M, D, cols, "bf16")
            calls += 1
        if t_total >= reps_budget_s:
            break
    return total_bytes / t_total / 1e9, t_total, calls, threads


def oracle_sample_text(cols, budget_s):
    return ("decode sweep M in {1,2,4,8,16}, d=4096, first %d of 14336 columns (all K), "
            "repeated for >= %.1f s" % (cols, budget_s))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # bounded: about 90 s of CPU work for the whole run, whatever K and W are;
    # the same sample (columns of the sweep) as our arm's cpu_baseline
    cols = ORACLE_COLS
    budget = min(2.0, max(0.05, 90.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        oracle_sweep(cols, 0.0)
    vals, times = [], []
    for _ in range(args.steps):
        gbs, t, calls, threads = oracle_sweep(cols, budget)
        vals.append(gbs)
        times.append(t)
    value = statistics.median(vals)
    sample = oracle_sample_text(cols, budget) + " per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "step_GB/s": {k: round(v, 3) for k, v in quantiles(vals).items()},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    import swiglu_mlp_projection_gb300 as swg
    from swiglu_mlp_projection_gb300 import inputs, sharding, workload

    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    swg._lib.load()
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    num_sms = props.multi_processor_count
    l2 = getattr(props, "L2_cache_size", L2_BYTES) or L2_BYTES
    oracle_leg = rank == 0 and not args.no_oracle

    # this rank's columns of both weight matrices: all of them (a replica of
    # the sweep per rank), or its 64-aligned share (--split columns)
    c0, c1 = (0, D_FF) if args.split == "replicas" else sharding.column_range(D_FF, rank, world)
    n_cols = c1 - c0
    # weights: enough distinct copies that no call finds an earlier call's
    # weights in L2 (copies_for)
    w_bytes = 2 * D * max(n_cols, 1) * 2
    n_copies = copies_for(l2, w_bytes)
    _, wg_h, wu_h = inputs.make_inputs(1, D, D_FF, "bf16", seed=0)
    wg_s, wu_s = wg_h[:, c0:c1].contiguous(), wu_h[:, c0:c1].contiguous()
    # The sweep reads each copy in the packed layout of step a0 (the pages'
    # gate|up interleave: 64-column blocks of W_gate and W_up alternating),
    # written once per copy by swiglu_pack_weights outside every timed
    # region; packed weights measured 0.7-3.8 % faster per call.  The same
    # sweep on unpacked [d, d_ff] weights is reported as "sweep_unpacked".
    packs = []
    for _ in range(n_copies):
        a, b = wg_s.to(dev), wu_s.to(dev)
        packs.append(swg.pack_weights(a, b))
        del a, b
    torch.cuda.synchronize(dev)
    # one step's activations and outputs, each as one contiguous buffer with a
    # view per call (so the end-to-end loop moves them in one copy each way)
    xs_host = {M: inputs.make_inputs(M, D, D_FF, "bf16", seed=0, x_only=True)[0] for M in SWEEP}
    x_all_host = torch.cat([xs_host[M] for M in SWEEP], 0)
    x_all = x_all_host.to(dev)
    h_all = torch.empty(sum(SWEEP), n_cols, dtype=torch.bfloat16, device=dev)
    offs = {M: sum(SWEEP[:i]) for i, M in enumerate(SWEEP)}
    xs = {M: x_all[offs[M]:offs[M] + M] for M in SWEEP}
    hs = {M: h_all[offs[M]:offs[M] + M] for M in SWEEP}
    stream = torch.cuda.current_stream(dev)
    step_bytes = sum(workload.algorithmic_bytes(M, D, n_cols, "bf16") for M in SWEEP)
    plans = {M: swg.plan(M, D, n_cols, "bf16", "auto", num_sms) for M in SWEEP}
    launches_per_step = sum(p["launches"] for p in plans.values())

    counter = [0]

    def call(M, st=None):
        wp = packs[counter[0] % n_copies]
        counter[0] += 1
        swg.swiglu_up_packed(xs[M], wp, n_cols, out=hs[M], stream=st if st is not None else stream)

    def step():
        for M in SWEEP:
            call(M)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(gpu_uuid(dev))
    sampler.start()
    for _ in range(max(args.warmup, 3)):
        step()
    # keep the GPU busy ~1 s before timing so clock samples reflect load
    torch.cuda.synchronize(dev)
    settle0 = time.time()
    settle_steps = 0
    while time.time() - settle0 < 1.0:
        for _ in range(20):
            step()
        settle_steps += 20
        torch.cuda.synchronize(dev)

    # ---- timed region: K steps back to back; events only at its ends.  It
    # holds only launches of the kernel the sweep dispatches to, so its time
    # per launch is that kernel's average launch duration.
    start_ev, end_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    wall0 = time.time()
    start_ev.record(stream)
    for _ in range(args.steps):
        step()
    end_ev.record(stream)
    barrier()
    wall1 = time.time()
    total_ms = max_over_ranks(start_ev.elapsed_time(end_ev), world, dev)
    ms_per_step = total_ms / args.steps
    # the job's bytes: every rank's algorithmic bytes (with --split columns
    # each rank reads x and its share of the weights, and writes its share of h)
    job_bytes = sum(workload.algorithmic_bytes(M, D, hi - lo, "bf16")
                    for r in range(world) for M in SWEEP
                    for lo, hi in [(0, D_FF) if args.split == "replicas"
                                   else sharding.column_range(D_FF, r, world)])
    value = job_bytes / (ms_per_step * 1e-3) / 1e9
    achieved = step_bytes * args.steps / (total_ms * 1e-3) / 1e9
    avg_launch_us = 1e3 * total_ms / (args.steps * launches_per_step)
    clocks = sampler.summary(wall0, wall1, settle0)

    # ---- distribution of the step time (outside the timed region above,
    # whose value is taken with events at its two ends only): 30 repetitions
    # of 10 steps back to back, an event at each repetition's boundary, so
    # the calls inside a repetition overlap as in the timed region
    step_ms = quantiles(timed_reps(lambda i: step(), 10, 30, stream))

    # ---- end to end through the public API with pinned host buffers.  Every
    # step copies its inputs (x for every M) host->device in one copy, makes
    # the five calls, and copies its results (h for every M) back in one
    # copy.  As a serving loop would, the copies run on their own streams
    # with two buffer sets, so step i's calls overlap the upload of step
    # i+1's inputs and the download of step i-1's results; every copy of
    # every step is inside the timed region.
    x_pin = [x_all_host.pin_memory() for _ in range(2)]
    h_pin = [torch.empty(sum(SWEEP), n_cols, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = x_pin[0].numel() * 2
    d2h = h_pin[0].numel() * 2
    xb = [x_all, torch.empty_like(x_all)]
    hb = [h_all, torch.empty_like(h_all)]
    xv = [{M: xb[j][offs[M]:offs[M] + M] for M in SWEEP} for j in range(2)]
    hv = [{M: hb[j][offs[M]:offs[M] + M] for M in SWEEP} for j in range(2)]
    up_st, down_st = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
    uploaded, computed, downloaded = ev(), ev(), ev()

    def upload(j, after=None):
        if after is not None:
            up_st.wait_event(after)
        up_st.wait_event(computed[j])            # the calls that read this x buffer
        with torch.cuda.stream(up_st):
            xb[j].copy_(x_pin[j], non_blocking=True)
        uploaded[j].record(up_st)

    def e2e_steps(n, start=None):
        upload(0, start)
        for i in range(n):
            j = i % 2
            if i + 1 < n:
                upload(1 - j)
            stream.wait_event(uploaded[j])
            stream.wait_event(downloaded[j])     # the download of this h buffer
            for M in SWEEP:
                wp = packs[counter[0] % n_copies]
                counter[0] += 1
                swg.swiglu_up_packed(xv[j][M], wp, n_cols, out=hv[j][M], stream=stream)
            computed[j].record(stream)
            down_st.wait_event(computed[j])
            with torch.cuda.stream(down_st):
                h_pin[j].copy_(hb[j], non_blocking=True)
            downloaded[j].record(down_st)
        stream.wait_event(downloaded[(n - 1) % 2])

    for _ in range(3):
        e2e_steps(4)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(args.steps, start=e0)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = job_bytes * args.steps / (e2e_ms * 1e-3) / 1e9
    sampler.stop()

    # ---- per-M breakdown (diagnostic, outside the timed region): each M
    # back to back, per-call times, the latency of one isolated call, and
    # CUDA-graph replay
    sweep = {}
    for M in SWEEP:
        b = workload.algorithmic_bytes(M, D, n_cols, "bf16")
        per = timed_reps(lambda i: call(M), 20, 10, stream)
        ms = sum(per) / len(per)
        q = quantiles(per)
        lat = []
        for _ in range(20):
            l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            l0.record(stream)
            call(M)
            l1.record(stream)
            torch.cuda.synchronize(dev)
            lat.append(l0.elapsed_time(l1))
        # the same calls captured into a CUDA graph (as a serving loop would
        # replay them), on a side stream
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            call(M, gs)
            with torch.cuda.graph(graph, stream=gs):
                for _ in range(20):
                    call(M, gs)
        stream.wait_stream(gs)
        graph.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(3):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = g0.elapsed_time(g1) / 60
        del graph
        sweep[str(M)] = {"us": round(ms * 1e3, 2), "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                         "frac": round(b / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         "us_median": round(q["median"] * 1e3, 2),
                         "us_p10": round(q["p10"] * 1e3, 2), "us_p90": round(q["p90"] * 1e3, 2),
                         "isolated_call_us": round(statistics.median(lat) * 1e3, 2),
                         "graph_us": round(graph_ms * 1e3, 2),
                         "path": plans[M]["path"]}

    # ---- oracle leg on the sweep's own outputs (every output of every M,
    # this rank's columns), outside every timed region
    if oracle_leg:
        torch.cuda.synchronize(dev)
        for M in SWEEP:
            chk = oracle_check(xs_host[M], wg_s, wu_s, hs[M].cpu(), list(range(M)), "bf16",
                               M, D, n_cols)
            sweep[str(M)]["accuracy"] = chk["accuracy"]
            sweep[str(M)]["oracle"] = chk["oracle"]
    del wg_h, wu_h

    # ---- the same calls on unpacked [d, d_ff] weights (swiglu_up), per M
    del packs
    torch.cuda.synchronize(dev)
    plain = [(wg_s.to(dev), wu_s.to(dev)) for _ in range(n_copies)]
    sweep_unpacked = {}
    for M in SWEEP:
        b = workload.algorithmic_bytes(M, D, n_cols, "bf16")
        k = [0]

        def plain_call(i, M=M):
            wgc, wuc = plain[k[0] % n_copies]
            k[0] += 1
            swg.swiglu_up(xs[M], wgc, wuc, out=hs[M], stream=stream)
        for i in range(3):
            plain_call(i)
        per = timed_reps(plain_call, 20, 10, stream)
        ms = sum(per) / len(per)
        q = quantiles(per)
        sweep_unpacked[str(M)] = {"us": round(ms * 1e3, 2), "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                                  "frac": round(b / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                  "us_median": round(q["median"] * 1e3, 2),
                                  "us_p10": round(q["p10"] * 1e3, 2),
                                  "us_p90": round(q["p90"] * 1e3, 2)}
    del plain

    extra = next_rows = fp8_rows = None
    if not args.no_extra:
        xs_sampler = ClockSampler(gpu_uuid(dev))
        xs_sampler.start()
        extra = other_configs(dev, peaks, l2, args.extra_iters, oracle_leg, xs_sampler)
        next_rows = down_and_mlp(dev, peaks, l2, args.extra_iters, xs_sampler)
        fp8_rows = fp8_configs(dev, peaks, l2, args.extra_iters, xs_sampler)
        xs_sampler.stop()

    if rank == 0:
        cpu = cpu_baseline() if oracle_leg else None
        kernels = sorted(set(p["path"] for p in plans.values()))
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak" if args.split == "replicas" else "strong",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": bench_config(),
            "split": args.split if world > 1 else None,
            "weight_copies": n_copies, "clock_settle_steps": settle_steps,
            "step_ms": {k: round(v, 5) for k, v in step_ms.items()},
            "step_ms_note": "median / p10 / p90 of the mean step time of 30 repetitions of 10 "
                            "steps back to back (after the timed region; ms_per_step is the "
                            "timed region's mean)",
            "roofline": {"bound": "hbm",
                         "kernel": "skinny_tc_kernel" if kernels == ["skinny"] else "+".join(kernels),
                         "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": profiled_traffic() if kernels == ["skinny"] and n_cols == D_FF
                         else None,
                         "traffic_source": TRAFFIC_FILE + " (ncu, mean of the 5 sweep "
                                           "launches; null if the kernel changed since)",
                         "algorithmic_bytes_per_launch": step_bytes // launches_per_step,
                         "avg_launch_us": round(avg_launch_us, 2),
                         "peak_source": peaks["source"] + " hbm_gbs (copy, burst)",
                         "timing": "CUDA events on the launching stream around the timed region, "
                                   "which holds only this kernel's launches"},
            "sweep": sweep,
            "sweep_unpacked": sweep_unpacked,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "note": "every step: one H2D copy of the step's x rows and one D2H copy "
                            "of its h rows (pinned host buffers), on copy streams with two "
                            "buffer sets so they overlap the neighbouring steps' calls; "
                            "weights resident in HBM"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if extra is not None:
            line["other_configs"] = extra
        if next_rows is not None:
            line["down_and_mlp"] = next_rows
        if fp8_rows is not None:
            line["fp8"] = fp8_rows
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def timed_reps(fn, iters, reps=10, stream=None):
    """Mean per-call time (ms) of each of `reps` repetitions of `iters` calls
    back to back, with events only at the repetitions' boundaries (an event
    between two calls would cut the programmatic overlap of one call's set-up
    with the previous call's tail, and for calls of a few microseconds it
    would time the host); for the median / p10 / p90 of a configuration."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    evs[0].record(stream)
    k = 0
    for r in range(reps):
        for _ in range(iters):
            fn(k)
            k += 1
        evs[r + 1].record(stream)
    torch.cuda.synchronize()
    return [evs[r].elapsed_time(evs[r + 1]) / iters for r in range(reps)]


def add_quantiles(entry, per_ms):
    q = quantiles(per_ms)
    entry["us_median"] = round(q["median"] * 1e3, 2)
    entry["us_p10"] = round(q["p10"] * 1e3, 2)
    entry["us_p90"] = round(q["p90"] * 1e3, 2)
    return entry


def other_configs(dev, peaks, l2, iters, oracle_leg=False, sampler=None):
    """Secondary measurements of the other workloads (not the headline):
    `iters` calls back to back after 3 warm-up calls, weight copies rotated so
    that the weights read by each call are not in L2 (mean from events at the
    two ends; median / p10 / p90 from a second pass with an event per call);
    then the same calls replayed from a CUDA graph.  With `oracle_leg`, the
    oracle evaluates rows of each call (check_rows) and the GPU's output of
    the timed calls is compared with it."""
    import torch
    import swiglu_mlp_projection_gb300 as swg
    from swiglu_mlp_projection_gb300 import inputs, workload
    out = {}
    for cfg in workload.CONFIGS:
        if cfg.name == "bf16_decode_d4096":
            continue
        _, wg, wu = inputs.make_inputs(1, cfg.d, cfg.d_ff, cfg.dtype, seed=0)
        w_bytes = 2 * wg.numel() * wg.element_size()
        n_copies = copies_for(l2, w_bytes)
        copies = [(wg.to(dev), wu.to(dev)) for _ in range(n_copies)]
        for M in cfg.Ms:
            x_h = inputs.make_inputs(M, cfg.d, cfg.d_ff, cfg.dtype, seed=0, x_only=True)[0]
            x = x_h.to(dev)
            h = torch.empty(M, cfg.d_ff, dtype=x.dtype, device=dev)
            k = [0]

            def call():
                a, b = copies[k[0] % n_copies]
                k[0] += 1
                swg.swiglu_up(x, a, b, out=h)
            for _ in range(3):
                call()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            w0 = time.time()
            e0.record()
            for _ in range(iters):
                call()
            e1.record()
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / iters
            per = timed_reps(lambda i: call(), iters)
            w1 = time.time()
            # the same calls captured once into a CUDA graph and replayed:
            # no host work per call
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(iters):
                    call()
            g.replay()
            torch.cuda.synchronize(dev)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize(dev)
            ms_graph = e0.elapsed_time(e1) / iters
            del g
            by = workload.algorithmic_bytes(M, cfg.d, cfg.d_ff, cfg.dtype)
            fl = workload.flops(M, cfg.d, cfg.d_ff)
            gbs = by / (ms * 1e-3) / 1e9
            tfs = fl / (ms * 1e-3) / 1e12
            key = "%s/M=%d" % (cfg.name, M)
            dplan = swg.plan(M, cfg.d, cfg.d_ff, cfg.dtype, "auto", 0)   # as this GPU serves it
            entry = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "TFLOP/s": round(tfs, 2),
                     "graph_us": round(ms_graph * 1e3, 2),
                     "graph_GB/s": round(by / (ms_graph * 1e-3) / 1e9, 1),
                     "path": dplan["path"], "cluster": dplan["cluster"]}
            add_quantiles(entry, per)
            if sampler is not None:
                # SM clock while this configuration ran (both timing passes):
                # calls of milliseconds of dense tensor work run under the
                # power cap at lower clocks
                cs = sampler.summary(w0, w1, w0)
                entry["clocks"] = {"sm_mhz": cs["sm_mhz"], "reasons": cs["reasons"],
                                   "samples": cs.get("samples", 0)}
            if oracle_leg:
                rows = check_rows(M, cfg.d, cfg.d_ff)
                torch.cuda.synchronize(dev)
                entry.update(oracle_check(x_h, wg, wu, h[rows].cpu(), rows, cfg.dtype,
                                          M, cfg.d, cfg.d_ff))
            if M <= 16 or cfg.dtype == "f32":
                entry["frac_hbm"] = round(gbs / peaks["hbm_gbs"], 4)
            else:
                entry["frac_bf16"] = round(tfs / peaks["bf16_tflops"], 4)
                # calls of milliseconds run under the power cap: also against
                # the sustained (seconds-long cuBLAS loop) peak
                entry["frac_bf16_sustained"] = round(tfs / peaks["bf16_tflops_sustained"], 4)
            out[key] = entry
            del x, x_h, h
        del copies, wg, wu
        torch.cuda.empty_cache()
    return out


def clocks_of(sampler, w0, w1):
    """Median SM clock and throttle reasons sampled between wall times w0, w1."""
    if sampler is None:
        return None
    cs = sampler.summary(w0, w1, w0)
    return {"sm_mhz": cs["sm_mhz"], "reasons": cs["reasons"], "samples": cs.get("samples", 0)}




def fp8_configs(dev, peaks, l2, iters, sampler=None):
    """The FP8 (e4m3) up projection at d=4096, d_ff=14336: the decode sweep
    and the prefill call, back to back with weight copies rotated per call
    (copies_for); then the FP8 down projection and the FP8 MLP (both
    projections, with the residual) at M = 1, 16, 4096.  GB/s counts fp8_bytes; TFLOP/s is against the FP8
    dense peak taken as 2x the measured bf16 peak (the nominal FP8 : BF16
    ratio, 4.5 : 2.25 PFLOP/s)."""
    import torch
    import swiglu_mlp_projection_gb300 as swg
    from swiglu_mlp_projection_gb300 import inputs, workload
    d, d_ff = D, D_FF
    _, wg, wu = inputs.make_inputs(1, d, d_ff, "bf16", seed=0)
    wgd, wud = wg.to(dev), wu.to(dev)
    nq = copies_for(l2, 2 * d * d_ff)
    qs = [swg.quantize_weights_fp8(wgd, wud) for _ in range(nq)]
    del wg, wu, wgd, wud
    torch.cuda.synchronize(dev)
    out = {}
    fp8_peak = 2 * peaks["bf16_tflops"]
    for M in SWEEP + (4096,):
        x = inputs.make_inputs(M, d, 8, "bf16", seed=M, x_only=True)[0].to(dev)
        h = torch.empty(M, d_ff, dtype=torch.bfloat16, device=dev)
        for i in range(3):
            swg.swiglu_up_fp8(x, qs[i % nq], out=h)
        torch.cuda.synchronize(dev)
        w0 = time.time()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(iters):
            swg.swiglu_up_fp8(x, qs[i % nq], out=h)
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / iters
        per = timed_reps(lambda i: swg.swiglu_up_fp8(x, qs[i % nq], out=h), iters)
        w1 = time.time()
        by = workload.fp8_bytes(M, d, d_ff)
        fl = workload.flops(M, d, d_ff)
        e = {"us": round(ms * 1e3, 2), "GB/s": round(by / ms / 1e6, 1),
             "TFLOP/s": round(fl / ms / 1e9, 2), "path": swg.plan(M, d, d_ff)["path"],
             "launches": 2}
        add_quantiles(e, per)
        e["clocks"] = clocks_of(sampler, w0, w1)
        if M <= 16:
            e["frac_hbm"] = round(by / ms / 1e6 / peaks["hbm_gbs"], 4)
        else:
            e["frac_fp8"] = round(fl / ms / 1e9 / fp8_peak, 4)
        out["fp8_d4096/M=%d" % M] = e
        del x, h
    # the FP8 down projection and the whole FP8 MLP (both projections e4m3)
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=1)
    wdd = wd.to(dev)
    nqd = copies_for(l2, d * d_ff)
    qds = [swg.quantize_weight_fp8(wdd) for _ in range(nqd)]
    del wd, wdd
    for M in (1, 16, 4096):
        x = inputs.make_inputs(M, d, 8, "bf16", seed=M, x_only=True)[0].to(dev)
        hb = torch.empty(M, d_ff, dtype=torch.bfloat16, device=dev)
        y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        swg.swiglu_up_fp8(x, qs[0], out=hb)
        for name, fn, by, fl in (
                ("fp8_down_d4096", lambda i: swg.swiglu_down_fp8(hb, qds[i % nqd], residual=x, out=y),
                 workload.fp8_down_bytes(M, d_ff, d), workload.down_flops(M, d_ff, d)),
                ("fp8_mlp_d4096", lambda i: (swg.swiglu_up_fp8(x, qs[i % nq], out=hb),
                                             swg.swiglu_down_fp8(hb, qds[i % nqd], residual=x, out=y)),
                 workload.fp8_bytes(M, d, d_ff) + workload.fp8_down_bytes(M, d_ff, d),
                 workload.flops(M, d, d_ff) + workload.down_flops(M, d_ff, d))):
            for i in range(3):
                fn(i)
            torch.cuda.synchronize(dev)
            w0 = time.time()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(iters):
                fn(i)
            e1.record()
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / iters
            e = add_quantiles({"us": round(ms * 1e3, 2), "GB/s": round(by / ms / 1e6, 1),
                               "TFLOP/s": round(fl / ms / 1e9, 2)}, timed_reps(fn, iters))
            e["clocks"] = clocks_of(sampler, w0, time.time())
            if M <= 16:
                e["frac_hbm"] = round(by / ms / 1e6 / peaks["hbm_gbs"], 4)
            else:
                e["frac_fp8"] = round(fl / ms / 1e9 / fp8_peak, 4)
            out["%s/M=%d" % (name, M)] = e
        del x, hb, y
    del qs, qds
    torch.cuda.empty_cache()
    return out


def down_and_mlp(dev, peaks, l2, iters, sampler=None):
    """The down projection y = h.W_down + r and the two-kernel MLP at the
    decode and prefill shapes of d=4096, d_ff=14336 (back to back); the down
    projection also at M = 64 and 128, which its skinny path serves."""
    import torch
    import swiglu_mlp_projection_gb300 as swg
    from swiglu_mlp_projection_gb300 import inputs, workload
    d, d_ff = D, D_FF
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=1)
    _, wg, wu = inputs.make_inputs(1, d, d_ff, "bf16", seed=0)
    n_copies = copies_for(l2, 2 * d * d_ff)   # the down projection's weights alone
    wds = [wd.to(dev) for _ in range(n_copies)]
    wgs = [(wg.to(dev), wu.to(dev)) for _ in range(n_copies)]
    del wd, wg, wu
    out = {}
    per_call = []
    walls = []

    def timed(fn):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize(dev)
        walls.append(time.time())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(iters):
            fn(i)
        e1.record()
        torch.cuda.synchronize(dev)
        per_call.append(timed_reps(fn, iters))
        walls.append(time.time())
        return e0.elapsed_time(e1) / iters

    for M in (1, 16, 64, 128, 4096):
        h = inputs.make_inputs(M, d_ff, 8, "bf16", seed=2, x_only=True)[0].to(dev)
        x = inputs.make_inputs(M, d, 8, "bf16", seed=3, x_only=True)[0].to(dev)
        y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        hb = torch.empty(M, d_ff, dtype=torch.bfloat16, device=dev)
        ms = timed(lambda i: swg.swiglu_down(h, wds[i % n_copies], residual=x, out=y))
        by = workload.down_bytes(M, d_ff, d, "bf16")
        fl = workload.down_flops(M, d_ff, d)
        e = {"us": round(ms * 1e3, 2), "GB/s": round(by / ms / 1e6, 1),
             "TFLOP/s": round(fl / ms / 1e9, 2),
             "path": swg.down_plan(M, d_ff, d, "bf16", "auto", 0)["path"],
             "cluster": swg.down_plan(M, d_ff, d, "bf16", "auto", 0)["cluster"]}
        add_quantiles(e, per_call[-1])
        e["clocks"] = clocks_of(sampler, walls[-2], walls[-1])
        if e["path"] == "skinny":   # M FLOP per weight byte: below the ridge, HBM-bound
            e["frac_hbm"] = round(by / ms / 1e6 / peaks["hbm_gbs"], 4)
        else:
            e["frac_bf16"] = round(fl / ms / 1e9 / peaks["bf16_tflops"], 4)
            e["frac_bf16_sustained"] = round(fl / ms / 1e9 / peaks["bf16_tflops_sustained"], 4)
        out["down_d4096/M=%d" % M] = e
        if M not in (1, 16, 4096):
            del h, x, y, hb
            continue
        ms = timed(lambda i: swg.swiglu_mlp(x, wgs[i % n_copies][0], wgs[i % n_copies][1],
                                             wds[i % n_copies], residual=x, h=hb, out=y))
        by = workload.algorithmic_bytes(M, d, d_ff, "bf16") + workload.down_bytes(M, d_ff, d, "bf16")
        fl = workload.flops(M, d, d_ff) + workload.down_flops(M, d_ff, d)
        e = add_quantiles({"us": round(ms * 1e3, 2), "GB/s": round(by / ms / 1e6, 1),
                           "TFLOP/s": round(fl / ms / 1e9, 2)}, per_call[-1])
        e["clocks"] = clocks_of(sampler, walls[-2], walls[-1])
        if M <= 16:
            e["frac_hbm"] = round(by / ms / 1e6 / peaks["hbm_gbs"], 4)
        else:
            e["frac_bf16"] = round(fl / ms / 1e9 / peaks["bf16_tflops"], 4)
            e["frac_bf16_sustained"] = round(fl / ms / 1e9 / peaks["bf16_tflops_sustained"], 4)
        out["mlp_d4096/M=%d" % M] = e
        del h, x, y, hb
    del wds, wgs
    torch.cuda.empty_cache()
    return out


def cpu_baseline():
    """The oracle, as it stands, on a bounded sample of the headline workload
    (the same sample as the reference arm): on all host cores, then on one."""
    import oracle
    try:
        gbs, t, calls, threads = oracle_sweep(ORACLE_COLS, 10.0)
        gbs1, t1, calls1, _ = oracle_sweep(ORACLE_COLS, 5.0, threads=1)
    except Exception as e:  # the baseline must not sink the GPU measurement
        return {"value": None, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                "sample": "failed: %s" % e}
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": oracle_sample_text(ORACLE_COLS, 10.0) + ": %d calls over %.1f s" % (calls, t),
            "single_thread": {"value": round(gbs1, 3), "unit": "GB/s", "cores": 1,
                              "sample": oracle_sample_text(ORACLE_COLS, 5.0) +
                              ": %d calls over %.1f s" % (calls1, t1)},
            "host_cores": os.cpu_count(), "oracle_threads_default": oracle.default_threads()}


def check_rows(M, d=0, d_ff=0):
    """Rows of an M-row call the oracle leg evaluates: all of them up to 64
    rows or 4e9 multiply-adds per matrix, else 8 rows from different 128-row
    blocks and 32-row quarters, including the first and the last row."""
    if M <= 64 or M * d * d_ff <= 4e9:
        return list(range(M))
    blocks = (M + 127) // 128
    picks = {0, M - 1}
    for i, frac in enumerate((0.0, 0.2, 0.4, 0.6, 0.8, 1.0)):
        b = min(blocks - 1, int(frac * (blocks - 1)))
        picks.add(min(M - 1, b * 128 + 32 * (i % 4) + 5 * i))
    return sorted(picks)


def oracle_check(x, wg, wu, h_rows, rows, dtype, M, d, d_ff):
    """The oracle leg for one timed call: the oracle on `rows` of x (timed on
    all host cores; the time is extrapolated linearly in M to the whole call,
    rows being independent), and the GPU's h on those rows compared with it.
    x, wg, wu: the call's host inputs; h_rows: the GPU result on `rows`."""
    import numpy as np
    import oracle
    import torch
    from swiglu_mlp_projection_gb300 import inputs, workload
    from tests.parity import compare
    raw = inputs.raw_bits
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    xr = x[rows].contiguous()
    t0 = time.perf_counter()
    h64, _, sens = oracle.swiglu_up(raw(xr), raw(wg), raw(wu), od)
    t = time.perf_counter() - t0
    res = compare(h_rows.to(torch.float64).numpy(), h64, sens, dtype, d)
    full_s = t * M / len(rows)
    by = workload.algorithmic_bytes(M, d, d_ff, dtype)
    fl = workload.flops(M, d, d_ff)
    return {
        "accuracy": {"rows_checked": len(rows), "all_rows": len(rows) == M, "ok": res["ok"],
                     "max_err": float("%.3g" % res["max_err"]),
                     "normwise": float("%.3g" % res["normwise"]),
                     "mismatch_pct": round(res["mismatch_pct"], 4),
                     "mismatch_pct_above_1e-3max": round(res["mismatch_pct_above_1e-3max"], 4)},
        "oracle": {"rows": len(rows), "s": round(t, 3), "threads": oracle.default_threads(),
                   "call_s": round(full_s, 3),
                   "GB/s": round(by / full_s / 1e9, 4), "TFLOP/s": round(fl / full_s / 1e12, 6),
                   "extrapolated": len(rows) != M},
    }


def main():
    args = parse()
    rank, world, _ = dist_env()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU: re-run under torch.distributed.run
        if args.impl == "ours":
            import torch
            if torch.cuda.device_count() < args.gpus:
                print("bench.py: --gpus %d asked for, %d CUDA devices visible"
                      % (args.gpus, torch.cuda.device_count()), file=sys.stderr)
                return 2
        return subprocess.call(torchrun_argv(args, sys.argv[1:]))
    if world != args.gpus:
        print("bench.py: --gpus %d but WORLD_SIZE=%d" % (args.gpus, world), file=sys.stderr)
        return 2
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
