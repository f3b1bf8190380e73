"""Benchmark of the CAT forward (circular-convolutional attention) on GB300.

One step = one cat_forward over one batch of the workload: score
projection, softmax over the tokens, spectrum of z*, and the circulant
product IFFT(FFT(z*) ⊙ FFT(V)) for every column (the hot path of the CAT
notes page, section 方法详解).  Inputs are seeded synthetic tensors already
resident in HBM; X + V + O are larger than L2, so no flush is needed
between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--config long16k] [--no-secondary] [--no-short] [--no-backward]
                    [--backward-only]

The line also carries the backward pass (cat_backward: dX, dW_A, dV for an
upstream gradient) at the long-sequence and the short workloads, with its
roofline fraction; --backward-only times just that on --config.  It also
carries the 2-D (BCCB) circulant attention of a second page on its token-grid
workloads (--no-grid2d leaves them out) and the fused value-and-score
projection (cat_forward_fused, --no-fused leaves it out).

Prints ONE JSON line (rank 0).  With --impl reference the fp64 CPU oracle
is timed instead, on a bounded sample of the same workload.
"""
import argparse
import json
import math
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

import synth  # noqa: E402

METRIC = "CAT attention tokens·heads/s at N=16384 & 131072; % of HBM/FP32 roofline"
UNIT = "tokens·heads/s"
PRIMARY = "long16k"
SECONDARY = "long128k"

# FP32 peak = SMs x 128 FP32 lanes x 2 flops (FMA) x maximum SM clock.  The
# SM count is read from the device and the clock from the measured-peaks
# file (else the GB300's 2070 MHz) when the GPU arm starts; 152 SMs until then.
FP32_LANES, DEFAULT_MAX_SM_MHZ = 128, 2070.0
FP32_PEAK_TFLOPS = 152 * FP32_LANES * 2 * DEFAULT_MAX_SM_MHZ * 1e6 / 1e12
FP32_PEAK_SOURCE = "FP32: 152 SMs x 128 lanes x 2 x 2070 MHz"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per launch of the dominant kernel (pass B of the
# fast path), from an ncu capture of the same kernel sources, committed with
# its command under profiles/.  Keyed by (workload, hash of the kernel
# sources): any change to those sources makes the figure stale, and the
# bench then reports null.  ncu flushes L2 before each captured launch, so
# the figure is cold-cache traffic (the scratch refilled from DRAM), an upper
# bound on the traffic of a launch inside the overlapped schedule.
NCU_TRAFFIC = {
    # the launch-list captures: the median of their pass-B launches (8 at
    # long16k, 16 at long128k)
    ("long16k", "43d02c8c03ce"): 34773632,
    ("long128k", "43d02c8c03ce"): 35691264,
}
KERNEL_SOURCES = ["fourstep_fast.cu", "fft_reg.cuh", "fft_device.cuh", "bulk.cuh", "elem.cuh"]
# Pass B's transforms: per (pair, k2) signal one forward and one inverse DFT
# of length N1 = 512, counted as 5·N1·log2(N1) flops each.
PASS_B_N1 = 512


def set_fp32_peak(device):
    """FP32 peak of `device` from its SM count and the maximum SM clock."""
    global FP32_PEAK_TFLOPS, FP32_PEAK_SOURCE
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz, src = DEFAULT_MAX_SM_MHZ, "GB300 maximum"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz, src = float(json.load(f)["sm_max_mhz"]), "measured-peaks file"
    except Exception:
        pass
    FP32_PEAK_TFLOPS = sms * FP32_LANES * 2 * mhz * 1e6 / 1e12
    FP32_PEAK_SOURCE = ("FP32: %d SMs (device) x %d lanes x 2 x %.0f MHz (%s); derived "
                        "from unit counts and the maximum SM clock" % (sms, FP32_LANES, mhz, src))


def kernel_hash():
    import hashlib
    h = hashlib.sha1()
    base = os.path.join(ROOT, "fft_circulant_attention_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(base, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def cfg_of(name):
    c = dict(synth.CONFIGS[name])
    c["es"] = 2 if c["dtype"] == "bf16" else 4
    return c


def fft_flops(N):
    return 5.0 * N * math.log2(N) if N > 1 else 0.0


def algorithmic(c):
    """Bytes and FFT flops of one forward, and of its circulant-product stage."""
    B, N, D, H, es = c["B"], c["N"], c["D"], c["H"], c["es"]
    npair = (D // H + 1) // 2
    pair_tf = 2 * B * H * npair          # forward + inverse per packed pair
    conv_flops = pair_tf * fft_flops(N)
    total_flops = conv_flops + B * H * fft_flops(N)   # + spectrum of z*
    conv_bytes = 2 * B * N * D * es       # V read, O written
    total_bytes = 3 * B * N * D * es + D * H * es
    return dict(conv_flops=conv_flops, total_flops=total_flops, conv_bytes=conv_bytes,
                total_bytes=total_bytes, score_flops=2.0 * B * N * D * H)


def algorithmic_backward(c):
    """Bytes and FFT flops of one backward: X, V, dO read, dX, dV written (W_A
    read, dW_A written); transforms of length N: dV's circulant product (a
    forward and an inverse per packed pair, plus the spectrum of z*) and the
    correlation (a forward per packed pair of dO and of V, one inverse per
    (b, h))."""
    B, N, D, H, es = c["B"], c["N"], c["D"], c["H"], c["es"]
    npair = (D // H + 1) // 2
    transforms = 4 * B * H * npair + 2 * B * H
    return dict(flops=transforms * fft_flops(N),
                bytes=5 * B * N * D * es + 2 * D * H * es,
                dense_flops=3 * 2.0 * B * N * D * H)


class ClockSampler:
    """nvidia-smi clock and throttle sampling while the timed loop runs."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(", ") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[4:8]):
                    if v.strip() == "Active":
                        reasons.add(n)
            except Exception:
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "gb300" and torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle

def oracle_sample(c, heads):
    """A bounded sample of the workload for the fp64 oracle: batch 0 and the
    first `heads` heads (their W_A columns and value columns)."""
    X, WA, V = synth.make_inputs(1, c["N"], c["D"], c["H"], c["dtype"], seed=0)
    dh = c["D"] // c["H"]
    WAs = WA[:, :heads].contiguous()
    Vs = V[:, :, : heads * dh].contiguous()
    # The head split only needs D/H = dh: keep dh columns per sampled head.
    return X, WAs, Vs


def time_oracle(c, heads, reps=1):
    import oracle
    X, WAs, Vs = oracle_sample(c, heads)
    X64, W64, V64 = (t.double().numpy() for t in (X, WAs, Vs))
    units = c["N"] * heads
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        _forward_sample(oracle, X64, W64, V64, heads)
        times.append(time.perf_counter() - t0)
    return units, times, oracle.num_threads()


def _forward_sample(oracle, X, WA, V, heads):
    # z* for the sampled heads from the full X rows, then the circulant
    # product of each sampled head's columns (the oracle's FFT mode).
    zs = oracle.zstar(X, WA)                  # [1, heads, N]
    return oracle.circ_fft(zs, V)             # V holds heads·dh columns


def sample_heads(c):
    # All heads of batch 0: a few seconds of fp64 work on a many-core host.
    return c["H"]


def host_cores():
    """Cores of the host and the CPU affinity of this process."""
    try:
        aff = sorted(os.sched_getaffinity(0))
    except Exception:
        aff = list(range(os.cpu_count() or 1))
    # Compress the mask into ranges: [0, 1, 2, 5] -> "0-2,5".
    parts, i = [], 0
    while i < len(aff):
        j = i
        while j + 1 < len(aff) and aff[j + 1] == aff[j] + 1:
            j += 1
        parts.append(str(aff[i]) if i == j else "%d-%d" % (aff[i], aff[j]))
        i = j + 1
    return {"nproc": os.cpu_count(), "affinity": ",".join(parts), "affinity_cores": len(aff)}


def time_slice_131072(heads=(0, 15)):
    """The 131072-token workload's O(N^2) definition on its 4096-row slice
    (rows 32·r) for the value columns of `heads`, all host cores: the
    oracle's direct-product check of that workload, timed on its own."""
    import oracle
    c = cfg_of("long128k")
    X, WA, V = synth.make_inputs(c["B"], c["N"], c["D"], c["H"], c["dtype"], seed=0)
    dh = c["D"] // c["H"]
    cols = np.concatenate([np.arange(h * dh, (h + 1) * dh) for h in heads])
    t0 = time.perf_counter()
    zs = oracle.zstar(X, WA)
    t1 = time.perf_counter()
    Vs = np.ascontiguousarray(V.double().numpy()[:, :, cols])
    zss = np.ascontiguousarray(zs[:, list(heads)])
    rows = list(range(0, c["N"], 32))
    t2 = time.perf_counter()
    oracle.circ_direct_rows(zss, Vs, rows)
    t3 = time.perf_counter()
    outputs = len(rows) * cols.size
    return {"workload": "long128k", "rows": len(rows), "columns": int(cols.size),
            "heads": list(heads), "zstar_s": t1 - t0, "direct_s": t3 - t2,
            "multiply_adds": float(outputs) * c["N"],
            "outputs_per_s": outputs / (t3 - t2), "threads": oracle.num_threads()}


def cpu_baseline_leg(c, heads):
    """The fp64 oracle on the host cores: FFT mode on batch 0 of the workload
    with all cores (the reported value) and with one thread, and the
    131072-token row slice of the direct product."""
    import oracle
    cores_all = oracle.num_threads()
    units, times, cores = time_oracle(c, heads)
    oracle.set_num_threads(1)
    try:
        units1, times1, _ = time_oracle(c, heads)
    finally:
        oracle.set_num_threads(cores_all)
    sl = time_slice_131072()
    return {"value": units / times[0], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "batch 0, head%s 0..%d of %s: z* from the full rows and the fp64 "
                      "FFT-mode circulant product of those heads' columns"
                      % ("s" if heads > 1 else "", heads - 1, c["name"]),
            "seconds": times[0],
            "single_thread": {"value": units1 / times1[0], "unit": UNIT, "cores": 1,
                              "seconds": times1[0]},
            "host": host_cores(),
            "slice_131072_direct": sl}


def workload_config(c, name, world):
    """The `config` object of the JSON line; the same in both arms."""
    return {"workload": name, "B": c["B"], "N": c["N"], "D": c["D"], "H": c["H"],
            "storage": c["dtype"],
            "l2": "inputs larger than L2 (X+V+O %.0f MB), no flush"
                  % (3 * c["B"] * c["N"] * c["D"] * c["es"] / 1e6),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    c = cfg_of(args.config)
    c["name"] = args.config
    heads = args.sample_heads or sample_heads(c)
    for _ in range(args.warmup):
        time_oracle(c, heads)
    times = []
    for _ in range(args.steps):
        units, t, cores = time_oracle(c, heads)
        times.extend(t)
    tot = sum(times)
    value = units * len(times) / tot
    sample = ("batch 0, heads 0..%d of %s (B=%d N=%d D=%d H=%d %s): z* from the full rows, "
              "fp64 FFT-mode circulant product of %d value columns"
              % (heads - 1, args.config, c["B"], c["N"], c["D"], c["H"], c["dtype"],
                 heads * (c["D"] // c["H"])))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(c, args.config, world),
        "timed_sample": sample,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample, "host": host_cores()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ GPU path

def measure_workload(name, steps, warmup, device, world, sampler=None):
    import fft_circulant_attention_gb300 as cat
    c = cfg_of(name)
    X, WA, V = synth.make_inputs(c["B"], c["N"], c["D"], c["H"], c["dtype"], seed=0)
    Xd, Wd, Vd = (t.to(device) for t in (X, WA, V))
    Od = torch.empty_like(Vd)
    stream = torch.cuda.current_stream(device)
    plan = cat.Plan(c["B"], c["N"], c["D"], c["H"], c["dtype"], stream=stream)
    for _ in range(warmup):
        plan.forward(Xd, Wd, Vd, Od)
    plan.sync()
    barrier(world)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        plan.forward(Xd, Wd, Vd, Od)
    e1.record(stream)
    torch.cuda.synchronize(device)
    clocks = sampler.stop() if sampler else None
    barrier(world)
    ms_total = e0.elapsed_time(e1)
    plan.sync()
    desc = plan.describe()
    launches = int(desc.split("launches=")[1].split()[0])
    # Stage times: the library's CUDA events on the plan's stream around each
    # stage; with timing armed the forward runs its stages one after another
    # (no cross-stream overlap), so each stage is timed on its own.
    stage_steps = max(3, min(steps, 50))
    plan.timing(stage_steps)
    for _ in range(stage_steps):
        plan.forward(Xd, Wd, Vd, Od)
    stage_ms, ncalls = plan.stage_times()
    pass_ms, pass_launches = plan.pass_times() if "path=fast" in desc else ([0.0] * 3, 0)
    plan.timing(0)
    ms_total = max_over_ranks(ms_total, world, device)

    # End to end through the C ABI with pinned host buffers: every step
    # copies X, W_A, V in and O out inside the timed region.
    Xp, Wp, Vp = (t.pin_memory() for t in (X, WA, V))
    Op = torch.empty_like(Vp).pin_memory()
    e2e_steps = max(3, min(steps, 20))
    plan.forward_host(Xp, Wp, Vp, Op)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        plan.forward_host(Xp, Wp, Vp, Op)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, device)
    plan.close()
    del Xd, Vd, Od
    torch.cuda.empty_cache()

    units = c["B"] * c["N"] * c["H"]
    ms_step = ms_total / steps
    a = algorithmic(c)
    hbm, hbm_kind = load_peaks()
    # Roofline of the dominant kernel, pass B: its average launch duration
    # from the library's CUDA events around every pass-B launch of the
    # recorded (serialised) forwards, against its algorithmic flops per
    # launch: chunk_bh·N2 (b, h, k2) columns × npair signals × two length-512
    # transforms.
    chunk = int(desc.split("chunk_bh=")[1].split()[0]) if "chunk_bh=" in desc else 0
    n2 = c["N"] // PASS_B_N1
    npair = (c["D"] // c["H"] + 1) // 2
    b_ms = pass_ms[1] / max(pass_launches, 1)
    b_flops = chunk * n2 * npair * 2 * fft_flops(PASS_B_N1)
    b_tflops = b_flops / (b_ms * 1e-3) / 1e12 if b_ms > 0 else 0.0
    roof = {
        "kernel": "fsf_pass_b: per (b, h, k2) and 16 column pairs, the length-512 DFT over n1, "
                  "the product with FFT(z*)/N and the inverse DFT, on the L2-resident scratch; "
                  "one launch = one chunk of %d (b, h) rows" % chunk,
        "bound": "alu",
        "achieved": b_tflops,
        "peak": FP32_PEAK_TFLOPS,
        "unit": "TFLOP/s",
        "frac": b_tflops / FP32_PEAK_TFLOPS,
        "traffic": NCU_TRAFFIC.get((name, kernel_hash())),
        "peak_source": FP32_PEAK_SOURCE,
        "traffic_note": "ncu DRAM read+write per launch, cold cache (L2 flushed before the "
                        "captured launch): the scratch refilled from DRAM, an upper bound "
                        "on a launch inside the overlapped schedule; null when the kernel "
                        "sources changed since the capture",
        "flops_per_launch": b_flops,
        "ms_per_launch": b_ms,
        "launches_timed": pass_launches,
    }
    pass_ms_launch = {k: v / max(pass_launches, 1) for k, v in zip("ABC", pass_ms)}
    t_roof = max(a["total_bytes"] / (hbm * 1e9), a["total_flops"] / (FP32_PEAK_TFLOPS * 1e12))
    e2e_val = world * units * e2e_steps / e2e_s
    es = c["es"]
    return {
        "name": name, "c": c, "value": world * units / (ms_step * 1e-3), "ms_per_step": ms_step,
        "stage_ms": [s / max(ncalls, 1) for s in stage_ms], "roofline": roof,
        "pass_ms_per_launch": pass_ms_launch,
        "path_roofline_frac": t_roof / (ms_step * 1e-3), "t_roof_us": t_roof * 1e6,
        "launches": launches, "desc": desc, "clocks": clocks,
        "e2e": {"value": e2e_val, "unit": UNIT,
                "h2d_bytes_per_step": 2 * c["B"] * c["N"] * c["D"] * es + c["D"] * c["H"] * es,
                "d2h_bytes_per_step": c["B"] * c["N"] * c["D"] * es,
                "ms_per_step": 1e3 * e2e_s / e2e_steps},
    }


def measure_backward(name, device, reps, warmup=3):
    """ms per cat_backward (resident inputs and upstream gradient, plan's
    stream, CUDA events) with its whole-pass roofline fraction."""
    import fft_circulant_attention_gb300 as cat
    c = cfg_of(name)
    X, WA, V = (t.to(device) for t in synth.make_inputs(c["B"], c["N"], c["D"], c["H"],
                                                         c["dtype"], seed=0))
    G = synth.make_grad(c["B"], c["N"], c["D"], c["dtype"], seed=0).to(device)
    dX, dWA, dV = torch.empty_like(X), torch.empty_like(WA), torch.empty_like(V)
    stream = torch.cuda.current_stream(device)
    with cat.Plan(c["B"], c["N"], c["D"], c["H"], c["dtype"], stream=stream) as plan:
        for _ in range(warmup):
            plan.backward(X, WA, V, G, dX, dWA, dV)
        plan.sync()
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            plan.backward(X, WA, V, G, dX, dWA, dV)
        e1.record(stream)
        torch.cuda.synchronize(device)
        plan.sync()
    ms = e0.elapsed_time(e1) / reps
    a = algorithmic_backward(c)
    hbm, _ = load_peaks()
    t_roof = max(a["bytes"] / (hbm * 1e9), a["flops"] / (FP32_PEAK_TFLOPS * 1e12))
    del X, V, G, dX, dV
    torch.cuda.empty_cache()
    return {"workload": name, "B": c["B"], "N": c["N"], "D": c["D"], "H": c["H"],
            "storage": c["dtype"], "ms_per_step": ms,
            "value": c["B"] * c["N"] * c["H"] / (ms * 1e-3), "unit": UNIT,
            "path_roofline_frac": t_roof / (ms * 1e-3), "t_roof_us": t_roof * 1e6,
            "algorithmic_bytes": a["bytes"], "fft_flops": a["flops"], "reps": reps}


def measure_grid2d(name, device, reps=20, warmup=3):
    """ms per cat2d_forward (2-D circulant attention on a token grid;
    resident inputs, plan's stream, CUDA events)."""
    import fft_circulant_attention_gb300 as cat
    c = dict(synth.GRID_CONFIGS[name])
    B, h, w, D, H = c["B"], c["h"], c["w"], c["D"], c["H"]
    Q, K, V = (t.to(device) for t in synth.make_qkv(B, h * w, D, c["dtype"], seed=0))
    O = torch.empty_like(V)
    stream = torch.cuda.current_stream(device)
    with cat.Plan2D(B, h, w, D, H, c["dtype"], stream=stream) as plan:
        for _ in range(warmup):
            plan.forward(Q, K, V, O)
        plan.sync()
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            plan.forward(Q, K, V, O)
        e1.record(stream)
        torch.cuda.synchronize(device)
        plan.sync()
        desc = plan.describe()
    ms = e0.elapsed_time(e1) / reps
    N = h * w
    es = 2 if c["dtype"] == "bf16" else 4
    npair = (D // H + 1) // 2
    # Q, K, V read and O written; transforms: a forward per Q and K pair, one
    # inverse per (b, h) for the scores, then the product (a forward and an
    # inverse per V pair, one forward of σ(a)), each 5·N·log2(N) flops.
    nbytes = 4 * B * N * D * es
    flops = (4 * B * H * npair + 2 * B * H) * fft_flops(N)
    hbm, _ = load_peaks()
    t_roof = max(nbytes / (hbm * 1e9), flops / (FP32_PEAK_TFLOPS * 1e12))
    return {"workload": name, "B": B, "grid": [h, w], "D": D, "H": H, "storage": c["dtype"],
            "ms_per_step": ms, "value": B * N * H / (ms * 1e-3), "unit": UNIT,
            "path_roofline_frac": t_roof / (ms * 1e-3), "t_roof_us": t_roof * 1e6,
            "plan": desc, "reps": reps}


def measure_fused(name, device, reps=20, warmup=3):
    """ms per cat_forward_fused (V = X·W_V and the scores from one pass over
    X on the tensor cores, then the forward), with the projection alone
    (cat_project) and, as context, a library GEMM for V (torch.matmul, i.e.
    cuBLAS) followed by cat_forward.  Resident bf16 inputs, CUDA events."""
    import fft_circulant_attention_gb300 as cat
    c = cfg_of(name)
    B, N, D, H = c["B"], c["N"], c["D"], c["H"]
    X, WA, _ = synth.make_inputs(B, N, D, H, "bf16", seed=0)
    WV = synth.make_wv(D, "bf16", seed=0)
    Xd, WAd, WVd = X.to(device), WA.to(device), WV.to(device)
    V = torch.empty_like(Xd)
    O = torch.empty_like(Xd)
    zs = torch.empty((B, H, N), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps

    with cat.Plan(B, N, D, H, "bf16", stream=stream) as plan:
        t_fused = timed(lambda: plan.forward_fused(Xd, WVd, WAd, V, O))
        t_proj = timed(lambda: cat.cat_project(plan.handle, Xd, WVd, WAd, V, zs, B, N, D, H,
                                               "bf16"))
        t_lib = timed(lambda: (torch.matmul(Xd, WVd, out=V), plan.forward(Xd, WAd, V, O)))
        plan.sync()
    gemm_flops = 2.0 * B * N * D * (D + H)
    del Xd, V, O
    torch.cuda.empty_cache()
    return {"workload": name, "B": B, "N": N, "D": D, "H": H, "storage": "bf16",
            "ms_fused_forward": t_fused, "ms_projection": t_proj,
            "projection_tflops": gemm_flops / (t_proj * 1e-3) / 1e12,
            "ms_library_gemm_then_forward": t_lib,
            "value": B * N * H / (t_fused * 1e-3), "unit": UNIT, "reps": reps}


# The short-sequence configurations of the workload table (parity cases of
# the tests; timed here so that every path has a measured figure).
SHORT = ["tiny", "vit196", "gpt2_f32", "gpt2_bf16"]


def measure_short(name, device, reps=200, warmup=20):
    """ms per forward of one short configuration (resident inputs, plan's
    stream, CUDA events) with its whole-step roofline fraction."""
    import fft_circulant_attention_gb300 as cat
    c = cfg_of(name)
    X, WA, V = (t.to(device) for t in synth.make_inputs(c["B"], c["N"], c["D"], c["H"],
                                                         c["dtype"], seed=0))
    O = torch.empty_like(V)
    stream = torch.cuda.current_stream(device)
    with cat.Plan(c["B"], c["N"], c["D"], c["H"], c["dtype"], stream=stream) as plan:
        for _ in range(warmup):
            plan.forward(X, WA, V, O)
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            plan.forward(X, WA, V, O)
        e1.record(stream)
        torch.cuda.synchronize(device)
        desc = plan.describe()
    ms = e0.elapsed_time(e1) / reps
    a = algorithmic(c)
    hbm, _ = load_peaks()
    t_roof = max(a["total_bytes"] / (hbm * 1e9), a["total_flops"] / (FP32_PEAK_TFLOPS * 1e12))
    return {"workload": name, "B": c["B"], "N": c["N"], "D": c["D"], "H": c["H"],
            "storage": c["dtype"], "ms_per_step": ms,
            "value": c["B"] * c["N"] * c["H"] / (ms * 1e-3),
            "path_roofline_frac": t_roof / (ms * 1e-3), "plan": desc}


def profile_range(args, device):
    """Steady-state forwards of --config bracketed by cudaProfilerStart/Stop
    (after --warmup untimed ones), for a range capture of the whole forward:
        ncu --profile-from-start off --replay-mode app-range --clock-control none \
            --metrics dram__bytes_read.sum,dram__bytes_write.sum \
            python bench.py --config long16k --profile-range 4
    DRAM bytes per forward = the range's totals / --profile-range."""
    import fft_circulant_attention_gb300 as cat
    stream = torch.cuda.current_stream(device)
    if args.config in synth.GRID_CONFIGS:
        # A 2-D (token-grid) workload: cat2d_forward on Q, K, V.
        c = dict(synth.GRID_CONFIGS[args.config])
        B, h, w = c["B"], c["h"], c["w"]
        A, K, V = (t.to(device) for t in synth.make_qkv(B, h * w, c["D"], c["dtype"], seed=0))
        plan = cat.Plan2D(B, h, w, c["D"], c["H"], c["dtype"], stream=stream)
        run = lambda: plan.forward(A, K, V, O)   # noqa: E731
    else:
        c = cfg_of(args.config)
        if args.batches:
            # A smaller case of the same workload (its first batches), for
            # captures that replay each kernel many times.
            c["B"] = min(c["B"], args.batches)
        A, K, V = (t.to(device) for t in synth.make_inputs(c["B"], c["N"], c["D"], c["H"],
                                                            c["dtype"], seed=0))
        plan = cat.Plan(c["B"], c["N"], c["D"], c["H"], c["dtype"], stream=stream)
        run = lambda: plan.forward(A, K, V, O)   # noqa: E731
    O = torch.empty_like(V)
    with plan:
        for _ in range(args.warmup):
            run()
        plan.sync()
        torch.cuda.synchronize(device)
        torch.cuda.profiler.start()
        for _ in range(args.profile_range):
            run()
        torch.cuda.synchronize(device)
        torch.cuda.profiler.stop()
        plan.sync()
        desc = plan.describe()
    print(json.dumps({"profile_range": args.profile_range, "workload": args.config,
                      "plan": desc}), flush=True)


def dft_probe(args, device):
    """One length-32 DFT stage on the FP32 pipe against the same stage as a
    dense contraction on the tensor cores (cat_probe_dft32): time per stage
    per signal with CUDA events, and the error of one stage against an fp64
    DFT (numpy), for 2 and 3 bf16 terms.
        python bench.py --dft-probe"""
    import fft_circulant_attention_gb300 as cat
    nsig, rounds = 152 * 128 * 8, 64
    rng = np.random.default_rng(0)
    xh = rng.standard_normal((nsig, 32, 2)).astype(np.float32)
    x = torch.from_numpy(xh).to(device)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(device)
    ref = np.fft.fft(xh[..., 0].astype(np.float64) + 1j * xh[..., 1], axis=1) / np.sqrt(32)
    out = {"signals": nsig, "rounds": rounds}
    for mode, name in ((0, "fp32_pipe"), (1, "tensor_2terms"), (2, "tensor_3terms")):
        cat.cat_probe_dft32(x, y, nsig, mode, 1, stream)
        torch.cuda.synchronize(device)
        g = y.cpu().double().numpy()
        err = np.abs(g[..., 0] + 1j * g[..., 1] - ref).max() / np.abs(ref).max()
        for _ in range(3):
            cat.cat_probe_dft32(x, y, nsig, mode, rounds, stream)
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cat.cat_probe_dft32(x, y, nsig, mode, rounds, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1)
        out[name] = {"ms": ms, "ns_per_stage_per_signal": ms * 1e6 / (nsig * rounds),
                     "stages_per_s": nsig * rounds / (ms * 1e-3),
                     "max_rel_error_one_stage": float(err)}
    print(json.dumps({"dft32_stage_probe": out}), flush=True)


def run_gb300(args, world, rank, local):
    import fft_circulant_attention_gb300 as cat
    from fft_circulant_attention_gb300 import build
    build.build()
    cat.lib()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    set_fp32_peak(device)
    if args.profile_range:
        profile_range(args, device)
        return
    if args.dft_probe:
        dft_probe(args, device)
        return
    if args.backward_only:
        bw = measure_backward(args.config, device, max(args.steps, 1), args.warmup)
        if rank == 0:
            print(json.dumps({"backward": bw}), flush=True)
        return
    sampler = ClockSampler(local) if rank == 0 else None
    prim = measure_workload(args.config, args.steps, args.warmup, device, world, sampler)
    sec = None
    if not args.no_secondary and args.config != SECONDARY:
        sec = measure_workload(SECONDARY, max(3, args.steps // 4), args.warmup, device, world)
    short = [] if args.no_short else [measure_short(n, device) for n in SHORT]
    grid2d = []
    if not args.no_grid2d:
        # The 2-D (BCCB) circulant attention of the token-grid workloads; a
        # failure is recorded in its entry.
        for n in synth.GRID_CONFIGS:
            try:
                grid2d.append(measure_grid2d(n, device))
            except Exception as exc:
                grid2d.append({"workload": n, "error": "%s: %s" % (type(exc).__name__, exc)})
    fused = []
    if not args.no_fused:
        for n in (PRIMARY, "gpt2_bf16"):
            try:
                fused.append(measure_fused(n, device))
            except Exception as exc:
                fused.append({"workload": n, "error": "%s: %s" % (type(exc).__name__, exc)})
    backward = []
    if not args.no_backward:
        # The backward pass at the two long workloads and the short ones; a
        # failure is recorded in its entry instead of losing the line.
        for n, r in ((PRIMARY, 20), (SECONDARY, 5), ("tiny", 50), ("vit196", 20),
                     ("gpt2_f32", 20), ("gpt2_bf16", 20)):
            try:
                backward.append(measure_backward(n, device, r))
            except Exception as exc:   # reported, not fatal to the forward's line
                backward.append({"workload": n, "error": "%s: %s" % (type(exc).__name__, exc)})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        c = cfg_of(args.config)
        c["name"] = args.config
        cpu = cpu_baseline_leg(c, args.sample_heads or sample_heads(c))
    if rank != 0:
        return
    c = prim["c"]
    line = {
        "metric": METRIC, "value": prim["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": prim["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(c, args.config, world),
        "plan": prim["desc"],
        "roofline": prim["roofline"],
        "path_roofline_frac": prim["path_roofline_frac"],
        "stage_ms_serialised": {"score": prim["stage_ms"][0],
                                "softmax_spectrum": prim["stage_ms"][1],
                                "circulant_product": prim["stage_ms"][2]},
        "pass_ms_per_launch_serialised": prim["pass_ms_per_launch"],
        "e2e": prim["e2e"],
        "gpu_launches": prim["launches"] * args.steps,
        "clocks": prim["clocks"],
        "cpu_baseline": cpu,
    }
    if sec is not None:
        sc = sec["c"]
        line["secondary"] = {
            "workload": SECONDARY, "B": sc["B"], "N": sc["N"], "D": sc["D"], "H": sc["H"],
            "value": sec["value"], "ms_per_step": sec["ms_per_step"],
            "path_roofline_frac": sec["path_roofline_frac"], "roofline": sec["roofline"],
            "stage_ms_serialised": sec["stage_ms"],
            "pass_ms_per_launch_serialised": sec["pass_ms_per_launch"],
            "e2e": sec["e2e"], "plan": sec["desc"]}
    if short:
        line["short_configs"] = short
    if backward:
        line["backward"] = backward
    if grid2d:
        line["grid2d"] = grid2d
    if fused:
        line["fused_projection"] = fused
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default=PRIMARY,
                    choices=sorted(synth.CONFIGS) + sorted(synth.GRID_CONFIGS),
                    help="workload (the 2-D grid ones only with --profile-range)")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-short", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-grid2d", action="store_true")
    ap.add_argument("--no-fused", action="store_true")
    ap.add_argument("--dft-probe", action="store_true",
                    help="time one DFT-32 stage on the FP32 pipe and on the tensor cores, "
                         "print it and exit")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only cat_backward on --config (--steps calls) and print it")
    ap.add_argument("--sample-heads", type=int, default=0)
    ap.add_argument("--batches", type=int, default=0,
                    help="with --profile-range: run only the first this-many batches of --config")
    ap.add_argument("--profile-range", type=int, default=0,
                    help="run this many forwards of --config between cudaProfilerStart and "
                         "cudaProfilerStop (for an ncu range capture) and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.config in synth.GRID_CONFIGS and not args.profile_range:
        ap.error("the 2-D grid workloads are timed in the grid2d entries; "
                 "--config takes them only with --profile-range")
    world, rank, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gb300(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
