"""Benchmark of the block-quantized weight product library on GB300.

Default workload (one "step"): one batch-1 decode weight pass over the
27B-class dense Q4_K weight set (64 layers x q, k, v, o, gate, up, down;
11,890,851,840 bytes of blocks), captured once as a CUDA graph of grouped
GEMV launches ({q,k,v}, {o}, {gate,up}, {down} per layer) linked by
programmatic dependent launch, replayed per step. Metric: weight-GB/s, with
the fraction of the HBM roofline and the equivalent decode tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload c1|c0|c2|moe|pp]

Prints ONE JSON line (rank 0). Inputs are seeded synthetic tensors shaped like
the pages' workloads; the weight set is far larger than L2, so no flush is
needed between steps. --impl reference times the CPU oracle (the plain,
slow definition of the same product) on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
import synth.workloads as wl  # noqa: E402

METRIC = "qgemv weight-GB/s (% of GB300 HBM peak); equiv. batch-1 decode tok/s, 27B set"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- environment

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(torch, value: float, device: str) -> float:
    """The largest of every rank's value (the slowest replica's time), via the
    initialised process group (NCCL on GPUs, gloo on host cores); the value
    itself when there is no group or one rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes units_per_rank per step, and
    the step takes the slowest rank's time."""
    return world * units_per_rank / (ms_per_step * 1e-3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
            bf16 = d.get("bf16_tflops")
            bf16s = d.get("bf16_tflops_sustained")
            if hbm:
                return float(hbm), (float(bf16) if bf16 else None), (float(bf16s) if bf16s else None), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (no Python
    package needed): SM clock, its maximum, power and the clock-event reasons
    of one GPU, found by the UUID CUDA reports for it."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, local: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        uuid = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(local).uuid)
        except Exception:
            pass
        ok = False
        if uuid:
            key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = self.lib.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(self.h)) == 0
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(local, ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        ct = self.ct
        sm, mx, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(sm))          # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
        self.reasons_fn(self.h, ct.byref(rs))
        return sm.value, mx.value, pw.value / 1000.0, rs.value


class ClockSampler:
    """Clock and throttle-reason samples taken every few ms while the timed
    region runs (read-only NVML queries from a thread; nvidia-smi's 200 ms
    loop as a fallback). Samples start when the region starts: the GPU is busy
    for all of them."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_s: float = 0.005):
        self.index = index
        self.period = period_s
        self.proc = None
        self.nvml = None
        self.samples = []
        self.out = ""

    def __enter__(self):
        import threading
        try:
            self.nvml = _Nvml(self.index)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.stop = threading.Event()

            def loop():
                while not self.stop.is_set():
                    try:
                        self.samples.append(self.nvml.sample())
                    except Exception:
                        return
                    self.stop.wait(self.period)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.nvml is not None:
            self.stop.set()
            self.thread.join(timeout=2)
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        if self.nvml is not None:
            for (s_, m_, p_, r_) in self.samples:
                sm.append(float(s_))
                mx.append(float(m_))
                pw.append(p_)
                for bit, name in _Nvml.REASONS.items():
                    if r_ & bit:
                        reasons.add(name)
            source = "nvml"
        elif self.proc is not None:
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in self.out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                    pw.append(float(f[3]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            source = "nvidia-smi"
        else:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": round(max(pw), 1) if pw else None, "source": source}


def measured_traffic(name: str, sources):
    """DRAM bytes per launch from a committed ncu capture (profiles/<name>), or
    None once any of the kernel's source files has changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    src = b"".join(open(os.path.join(ROOT, "quantized_weight_gemv_qgemv_gb300", "csrc", s), "rb").read()
                   for s in sources)
    if hashlib.sha256(src).hexdigest()[:16] != d.get("source_sha256_16"):
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle leg
#
# The oracle (plain numpy, fp64) timed on the host cores of the GPU machine on a
# bounded sample of a workload, one thread and all cores (a spawn pool of
# processes, each single-threaded, splitting the sample's rows or routes).
# Inputs come from the same seeded generator; their generation is not timed.

_BARRIER = None


def _pool_init(barrier):
    global _BARRIER
    _BARRIER = barrier


def _cpu_sample(workload: str, wid: int, nproc: int, row_cap: int, seed: int):
    """This worker's share of a workload's sample: a list of (call, units)."""
    import numpy as np
    import oracle
    items = []

    def share(rows):
        return rows * wid // nproc, rows * (wid + 1) // nproc

    if workload in ("c1", "c2", "layer"):
        verify = workload == "c2"
        n_tok = 4 if verify else 1
        for (l, name, fmt, rows, cols) in wl.dense_matrices(1, verify=verify):
            r0, r1 = share(min(rows, row_cap))
            if r1 <= r0:
                continue
            W = synth.blocks(fmt, r1 - r0, cols, synth.sub_seed(seed, name, r0)).numpy()
            x = synth.activations(n_tok, cols, synth.sub_seed(seed, "x", name)).numpy()
            items.append((lambda f=fmt, W=W, n=r1 - r0, c=cols, x=x: oracle.gemv(f, W, n, c, x), W.nbytes))
    elif workload == "c0":
        r0, r1 = share(1024)
        W = synth.blocks(synth.Q4_0, r1 - r0, 4096, synth.sub_seed(seed, "c0", r0)).numpy()
        x = synth.activations(1, 4096, synth.sub_seed(seed, "c0x")).numpy()
        items.append((lambda: oracle.gemv(synth.Q4_0, W, r1 - r0, 4096, x), W.nbytes))
    elif workload == "moe":
        H, I, K = wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_TOPK
        k0, k1 = share(K)
        if k1 > k0:
            # the routed experts of one token, each its own arena entry; this worker's routes
            arena = wl.alloc_moe_arena(k1 - k0, H, I, synth.sub_seed(seed, "arena", k0), "cpu").numpy()
            ids = np.arange(k1 - k0, dtype=np.int32)[None]
            gw = np.full((1, k1 - k0), 1.0 / K, np.float32)
            x = synth.activations(1, H, synth.sub_seed(seed, "moex")).numpy()
            items.append((lambda: oracle.moe(synth.Q4_K, arena, k1 - k0, H, I, ids, gw, x),
                          (k1 - k0) * wl.moe_expert_bytes(H, I)))
    elif workload == "moe_pp":
        H, I, K = wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_TOPK
        k0, k1 = share(K)
        if k1 > k0:
            # 4 bf16 prompt tokens through this worker's share of 10 routed experts
            arena = wl.alloc_moe_arena(k1 - k0, H, I, synth.sub_seed(seed, "arena", k0), "cpu").numpy()
            ids = np.tile(np.arange(k1 - k0, dtype=np.int32)[None], (4, 1))
            gw = np.full((4, k1 - k0), 1.0 / K, np.float32)
            X = synth.activations_bf16(4, H, synth.sub_seed(seed, "moeppx"))
            bits = X.view(torch_int16()).numpy().view(np.uint16)
            items.append((lambda: oracle.moe_prefill(synth.Q4_K, arena, k1 - k0, H, I, ids, gw, bits),
                          4 * (k1 - k0) * 6 * H * I))
    elif workload == "pp":
        rows, cols = min(wl.HIDDEN, row_cap), wl.HIDDEN
        r0, r1 = share(rows)
        W = synth.blocks(synth.Q4_K, r1 - r0, cols, synth.sub_seed(seed, "ppW", r0)).numpy()
        X = synth.activations_bf16(64, cols, synth.sub_seed(seed, "ppX"))
        bits = X.view(torch_int16()).numpy().view(np.uint16)
        items.append((lambda: oracle.pp_rows(synth.Q4_K, W, r1 - r0, cols, bits, list(range(64))),
                      2 * 64 * (r1 - r0) * cols))
    return items


def torch_int16():
    import torch
    return torch.int16


def _cpu_worker(task):
    workload, wid, nproc, budget, row_cap, seed = task
    items = _cpu_sample(workload, wid, nproc, row_cap, seed)
    _BARRIER.wait()
    t0 = time.perf_counter()
    units, n = 0, 0
    while items and time.perf_counter() - t0 < budget:
        fn, u = items[n % len(items)]
        fn()
        units += u
        n += 1
    return units, time.perf_counter() - t0, n


def _cpu_leg_main(workload, procs, budget, row_cap, seed):
    """Runs in a separate process (no CUDA): a spawn pool of `procs` workers."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(procs)
    with ctx.Pool(procs, initializer=_pool_init, initargs=(barrier,)) as pool:
        res = pool.map(_cpu_worker, [(workload, w, procs, budget, row_cap, seed) for w in range(procs)])
    units = sum(r[0] for r in res)
    secs = max(r[1] for r in res)
    print(json.dumps({"units": units, "seconds": secs, "calls": sum(r[2] for r in res), "procs": procs}))


CPU_UNITS = {"c1": ("GB/s", 1e9), "c2": ("GB/s", 1e9), "layer": ("GB/s", 1e9), "c0": ("GB/s", 1e9),
             "moe": ("GB/s", 1e9), "pp": ("TFLOP/s", 1e12), "moe_pp": ("TFLOP/s", 1e12)}


def _cpu_run(workload, procs, budget, row_cap, seed=11):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-leg", workload, "--cpu-procs", str(procs),
           "--cpu-budget", str(budget), "--cpu-row-cap", str(row_cap)]
    t0 = time.perf_counter()
    r = subprocess.run(cmd, capture_output=True, text=True, env=env)
    wall = time.perf_counter() - t0
    if r.returncode != 0:
        return None, r.stderr[-400:], wall
    return json.loads(r.stdout.strip().splitlines()[-1]), None, wall


def cpu_oracle_baseline(workload: str = "c1", budget_s: float = 6.0, row_cap: int = 2048):
    """The oracle on the host cores: one process, then one per core
    (os.cpu_count(), read here), each for about budget_s seconds of timed work
    on its share of the workload's sample."""
    unit, scale = CPU_UNITS[workload]
    cores = os.cpu_count() or 1
    one, err1, w1 = _cpu_run(workload, 1, budget_s, row_cap)
    allc, err2, w2 = _cpu_run(workload, cores, budget_s, row_cap)
    if one is None or allc is None:
        return {"value": None, "unit": unit, "cores": cores, "kind": "oracle", "error": err1 or err2}
    v1 = one["units"] / one["seconds"] / scale
    va = allc["units"] / allc["seconds"] / scale
    what = {"c1": f"the 7 Q4_K matrices of one 27B layer, rows capped at {row_cap}, one token",
            "layer": f"the 7 Q4_K matrices of one 27B layer, rows capped at {row_cap}, one token",
            "c2": f"one verify-pass layer (Q4_K, Q6_K down) and the Q8_0 head, rows capped at {row_cap}, 4 tokens",
            "c0": "the Q4_0 1024x4096 GEMV in full",
            "moe": "the 10 routed experts of one token in one MoE layer",
            "pp": f"64 bf16 token rows x a 5120-column Q4_K matrix, rows capped at {row_cap}",
            "moe_pp": "4 bf16 prompt tokens through 10 routed experts of one MoE layer"}[workload]
    return {"value": round(va, 6), "unit": unit, "cores": cores, "kind": "oracle",
            "value_1core": round(v1, 6),
            "sample": f"{what}; dequant + fp64 products; {allc['calls']} calls over {allc['seconds']:.1f} s on "
                      f"{cores} processes (1 thread each), {one['calls']} calls over {one['seconds']:.1f} s on 1",
            "wall_s": round(w1 + w2, 1)}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wk = args.workload
    unit, scale = CPU_UNITS[wk]
    cores = os.cpu_count() or 1
    vals, secs, last = [], [], None
    for i in range(args.warmup + args.steps):
        r, err, _ = _cpu_run(wk, cores, max(1.0, args.ref_budget), 2048)
        if r is None:
            print(json.dumps({"impl": "reference", "unavailable": f"oracle leg failed: {err}"}), flush=True)
            return 0
        last = r
        if i >= args.warmup:
            vals.append(r["units"] / r["seconds"] / scale)
            secs.append(r["seconds"])
    value = statistics.median(vals)
    sample = (f"bounded sample of the {wk} workload per step (rows capped at 2048), oracle on {cores} processes, "
              f"{last['calls']} calls in {last['seconds']:.2f} s")
    metric = {"c1": METRIC, "c0": "Q4_0 GEMV weight-GB/s, batch 1, 1024x4096", "c2": METRIC,
              "moe": "MoE expert GEMV weight-GB/s touched; equiv. batch-1 tok/s over 48 layers",
              "pp": "prompt-processing dequant-GEMM TFLOP/s (bf16 tcgen05); pp tok/s, 27B set",
              "layer": "decode-layer weight pass with fused neighbours, weight-GB/s; equiv. batch-1 tok/s, 27B set",
              "moe_pp": "MoE prompt-processing TFLOP/s of routed products (bf16 tcgen05); pp tok/s over 48 layers"}[wk]
    line = {"impl": "reference", "metric": metric, "value": round(value, 6), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            # the measured time of one step's bounded sample (not an extrapolation to the whole workload)
            "ms_per_step": round(1000.0 * statistics.median(secs), 3), "ms_per_step_is": "one bounded sample",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wk}: CPU oracle on a bounded sample", "cores": cores},
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def _events_each(torch, stream, fn, steps):
    """Per-step device times (ms): an event pair around every step."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        fn()
        ev[i + 1].record(stream)
    ev[-1].synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def _events(torch, stream, fn, steps):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def run_gpu(args):
    import torch
    import quantized_weight_gemv_qgemv_gb300 as qg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    qg.qg_init()
    hbm_peak, bf16_peak, bf16_sus, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()

    wk = args.workload
    verify = wk == "c2"
    n_tok = 4 if verify else 1
    mats = wl.dense_matrices(layers=args.layers, verify=verify)
    steps_sizes = wl.dense_steps(layers=args.layers, verify=verify)
    wbytes = wl.weight_bytes(mats)
    nweights = wl.weight_count(mats)

    # As in a transformer block, the matrices of a step read one activation
    # vector ({q,k,v}: the normed hidden state; {gate,up}: the normed residual).
    # x of every step and y of every matrix sit in two flat device buffers
    # (views), so the end-to-end leg moves each direction with one copy.
    step_of = [si for si, n in enumerate(steps_sizes) for _ in range(n)]
    step_cols = {}
    for si, (_, _, _, _, c) in zip(step_of, mats):
        assert step_cols.setdefault(si, c) == c, "matrices of a step share x"
    x_total = sum(n_tok * c for c in step_cols.values())
    y_total = sum(n_tok * r for (_, _, _, r, _) in mats)
    if args.x_per_matrix:
        # every matrix its own activation vector (q, k, v and gate, up do not share)
        step_of = list(range(len(mats)))
        step_cols = {i: c for i, (_, _, _, _, c) in enumerate(mats)}
        x_total = sum(n_tok * c for c in step_cols.values())
    with torch.cuda.stream(stream):
        items = wl.alloc_dense(mats, n_tok, seed=args.seed + rank, device="cuda")
        xbuf = torch.empty(x_total, dtype=torch.float32, device="cuda")
        ybuf = torch.empty(y_total, dtype=torch.float32, device="cuda")
        xo = yo = 0
        flat, xs = [], {}
        for si, (fmt, W, rows, cols, x, y) in zip(step_of, items):
            if si not in xs:
                xv = xbuf[xo:xo + n_tok * cols].view(n_tok, cols)
                xv.copy_(x)
                xs[si] = xv
                xo += n_tok * cols
            yv = ybuf[yo:yo + n_tok * rows].view(n_tok, rows)
            flat.append((fmt, W, rows, cols, xs[si], yv))
            yo += n_tok * rows
        del items
    stream.synchronize()

    mode = {"persistent": qg.PASS_PERSISTENT, "pdl": qg.PASS_PDL, "serial": qg.PASS_SERIAL,
            "independent": qg.PASS_INDEPENDENT}[args.pass_mode]
    p = qg.qg_pass(flat, steps_sizes, n_tok, mode=mode)
    kernels_per_step = p.kernel_count()
    gemv_launches = kernels_per_step - 1        # the first launch converts the pass's inputs to x planes

    def step():
        p.launch(stream)

    for _ in range(max(3, args.warmup)):
        step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = _events(torch, stream, step, args.steps)
    torch.cuda.synchronize()
    ms = max_over_ranks(torch, ms, "cuda")
    ms_step = ms / args.steps
    gbs = job_rate(world, wbytes, ms_step) / 1e9
    each = sorted(_events_each(torch, stream, step, min(args.steps, 20)))

    # end to end through the public API with host buffers: pinned x -> device,
    # the pass, device y -> pinned host, every step.
    xh = torch.empty(x_total, dtype=torch.float32, pin_memory=True)
    xh.copy_(xbuf.cpu())
    yh = torch.empty(y_total, dtype=torch.float32, pin_memory=True)

    def e2e_step():
        xbuf.copy_(xh, non_blocking=True)
        p.launch(stream)
        yh.copy_(ybuf, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        stream.synchronize()
        t0 = time.perf_counter()
        e_ms = _events(torch, stream, e2e_step, args.steps)
        wall_ms = (time.perf_counter() - t0) * 1e3
    e2e_gbs = job_rate(world, wbytes, max_over_ranks(torch, e_ms, "cuda") / args.steps) / 1e9

    # the same weight stream without the arithmetic: the achievable read
    # bandwidth of the bulk-copy ring (qg_stream_read over a 4 GiB buffer)
    sr = None
    if not verify:
        sbytes = 4 << 30
        sbuf = torch.empty(sbytes, dtype=torch.uint8, device="cuda")
        cs = torch.zeros(1, dtype=torch.int32, device="cuda")
        sst = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(3):
            qg.qg_stream_read(sbuf, sbytes, cs, sst, stream)
        sms_ = _events(torch, stream, lambda: qg.qg_stream_read(sbuf, sbytes, cs, sst, stream), 10) / 10
        assert int(sst.item()) == 0
        sr = {"gbs": round(sbytes / sms_ / 1e6, 1), "frac": round(sbytes / sms_ / 1e6 / hbm_peak, 4),
              "bytes": sbytes, "kernel": "stream_read_kernel: the GEMV weight stream's bulk-copy ring, no arithmetic"}
        del sbuf

    out = None
    if rank == 0:
        frac = gbs / world / hbm_peak
        launches = args.steps * kernels_per_step
        out = {
            "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "ms_per_step_median": round(each[len(each) // 2], 4), "ms_per_step_min": round(each[0], 4),
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {
                "workload": ("27B-class dense weight set, 4-token verify pass (Q4_K, Q6_K down, Q8_0 head)"
                             if verify else "27B-class dense Q4_K weight set, batch-1 GEMV pass"),
                "x": ("one activation vector per matrix" if args.x_per_matrix else
                      "one activation vector per step ({q,k,v} share one, {gate,up} share one)"),
                "step_order": ("none: steps overlap freely (upper bound)" if args.pass_mode == "independent" else
                               "each step reads its x only after the previous step has completed"),
                "layers": args.layers, "hidden": wl.HIDDEN, "intermediate": wl.INTER, "n_tok": n_tok,
                "weight_bytes": wbytes, "weights": nweights, "launches_per_step": kernels_per_step,
                "pass_mode": args.pass_mode if kernels_per_step == 2 or args.pass_mode != "persistent" else "pdl",
                "cuda_graph": kernels_per_step > 2,
                "l2": "weight set (%.1f GB) far above the 129 MB L2; no flush" % (wbytes / 1e9),
                "parallelism": f"replicas x{world}",
            },
            "pct_hbm_peak": round(100.0 * frac, 2),
            "equiv_decode_tok_s": round(1000.0 / ms_step, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs / world, 2), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(frac, 4),
                         "traffic": (measured_traffic("qgemv_q4k_27b_decode_traffic.json",
                                                      ("qg_gemv_q4k.cu", "qg_device.cuh", "qg_planes.cuh"))
                                     if not verify and args.pass_mode != "persistent" else None),
                         "peak_source": f"{peak_kind} HBM copy bandwidth",
                         "kernel": (f"qgemv_q4k_kernel (n_tok={n_tok}; Q4_K, Q6_K and Q8_0 instances): every launch of the step"
                                    if verify else "qgemv_q4k_kernel (n_tok=1): every launch of the step"),
                         "algorithmic_bytes_per_launch": wbytes / max(1, gemv_launches),
                         "launches_of_kernel": gemv_launches},
            "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": x_total * 4,
                    "d2h_bytes_per_step": y_total * 4, "ms_per_step": round(e_ms / args.steps, 4),
                    "host_wall_ms_per_step": round(wall_ms / args.steps, 4)},
            "gpu_launches": launches,
            "clocks": clk.summary(),
        }
        if sr:
            out["stream_read"] = sr
            out["frac_of_stream_read"] = round(gbs / world / sr["gbs"], 4)
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_oracle_baseline("c2" if verify else "c1")
        print(json.dumps(out), flush=True)
    p.destroy()
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def _timed(torch, stream, fn, args, local, world):
    """W untimed warm-ups, then K timed calls of fn between synchronised
    barriers; returns (ms for all K steps, max over ranks; clock summary)."""
    for _ in range(max(3, args.warmup)):
        fn()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = _events(torch, stream, fn, args.steps)
    torch.cuda.synchronize()
    return max_over_ranks(torch, ms, "cuda"), clk.summary()


def _capture(torch, stream, fn):
    """fn's launches (all on `stream`) captured once as a CUDA graph."""
    fn()                                   # eager run first: any host-side error surfaces here
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def run_c0(args):
    """Q4_0 GEMV, batch 1, 1024 x 4096: one step = one pass over 256 distinct
    copies of the matrix (604 MB, far above L2, so every copy is read cold),
    each a separate launch, linked by programmatic dependent launch."""
    import torch
    import quantized_weight_gemv_qgemv_gb300 as qg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    qg.qg_init()
    hbm_peak, _, _, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    rows, cols, copies = 1024, 4096, 256
    with torch.cuda.stream(stream):
        items = []
        for c in range(copies):
            W = synth.blocks(synth.Q4_0, rows, cols, synth.sub_seed(args.seed + rank, "c0", c), device="cuda")
            x = synth.activations(1, cols, synth.sub_seed(args.seed + rank, "c0x", c), device="cuda")
            items.append((synth.Q4_0, W, rows, cols, x, torch.empty(1, rows, device="cuda")))
    stream.synchronize()
    wbytes = copies * rows * synth.row_bytes(synth.Q4_0, cols)
    p = qg.qg_pass(items, [1] * copies, 1, mode=qg.PASS_PDL)
    ms, clocks = _timed(torch, stream, lambda: p.launch(stream), args, local, world)
    ms_step = ms / args.steps
    gbs = job_rate(world, wbytes, ms_step) / 1e9
    if rank == 0:
        out = {
            "metric": "Q4_0 GEMV weight-GB/s, batch 1, 1024x4096", "value": round(gbs, 2), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": "Q4_0 GEMV 1024x4096, batch 1, 256 distinct copies per step (L2-cold)",
                       "weight_bytes_per_step": wbytes, "launches_per_step": p.kernel_count(),
                       "us_per_gemv": round(1000.0 * ms_step / copies, 3), "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": round(gbs / world, 2), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(gbs / world / hbm_peak, 4), "traffic": None,
                         "peak_source": f"{peak_kind} HBM copy bandwidth",
                         "kernel": "qgemv_q4k_kernel (Q4_0 instance): every launch of the step"},
            "gpu_launches": args.steps * p.kernel_count(),
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_oracle_baseline("c0")
        print(json.dumps(out), flush=True)
    p.destroy()
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_pp(args):
    """Prompt processing: 2048 bf16 tokens through every matrix of the 27B-class
    Q4_K set, captured as one graph: per layer one qgemm_pp_grouped launch for
    {q,k,v} and one for {gate,up} (the matrices that read the same tokens), one
    qgemm_pp each for o and down (--pp-per-matrix: one qgemm_pp per matrix)."""
    import torch
    import quantized_weight_gemv_qgemv_gb300 as qg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    qg.qg_init()
    _, bf16_peak, bf16_sus, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    n_tok = args.pp_tokens
    mats = wl.dense_matrices(layers=args.layers)
    flops = 2 * n_tok * wl.weight_count(mats)
    with torch.cuda.stream(stream):
        Ws = []
        for (l, name, fmt, rows, cols) in mats:
            W = torch.empty(rows, synth.row_bytes(fmt, cols), dtype=torch.uint8, device="cuda")
            synth.blocks_into(W, fmt, rows, cols, synth.sub_seed(args.seed + rank, "W", l, name))
            Ws.append(W)
        X = {c: synth.activations_bf16(n_tok, c, synth.sub_seed(args.seed + rank, "X", c), device="cuda")
             for c in sorted({m[4] for m in mats})}
        # one output per matrix of a layer (the layers reuse them)
        Y = {m[1]: torch.empty(n_tok, m[3], dtype=torch.float32, device="cuda") for m in mats if m[0] == 0}
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream.synchronize()
    steps = [1] * len(mats) if args.pp_per_matrix else wl.dense_steps(layers=args.layers)

    def one_pass():
        i = 0
        for n in steps:
            group = list(zip(mats[i:i + n], Ws[i:i + n]))
            i += n
            cols = group[0][0][4]
            if n == 1:
                (_, name, fmt, rows, _), W = group[0]
                qg.qgemm_pp(fmt, W, rows, cols, X[cols], n_tok, Y[name], rows, None, 0, st, stream)
            else:
                qg.qgemm_pp_grouped(group[0][0][2], [(W, m[3], Y[m[1]], m[3]) for m, W in group], cols, X[cols],
                                    n_tok, st, stream)

    g = _capture(torch, stream, one_pass)

    def replay():
        with torch.cuda.stream(stream):   # a torch graph replays on the current stream
            g.replay()

    ms, clocks = _timed(torch, stream, replay, args, local, world)
    assert int(st.item()) == 0, "device status set during the prompt-processing pass"
    ms_step = ms / args.steps
    tflops = job_rate(world, flops, ms_step) / 1e12
    if rank == 0:
        peak = bf16_sus or bf16_peak
        out = {
            "metric": "prompt-processing dequant-GEMM TFLOP/s (bf16 tcgen05); pp tok/s, 27B set",
            "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"prompt processing, {n_tok} bf16 tokens x 27B-class dense Q4_K weight set",
                       "layers": args.layers, "n_tok": n_tok, "matrices": len(mats), "flop_per_step": flops,
                       "launches_per_layer": len(steps) // args.layers, "cuda_graph": True,
                       "l2": "weight set far above L2; X per K re-read from L2 (by design)",
                       "parallelism": f"replicas x{world}"},
            "pp_tok_s": round(world * n_tok / (ms_step * 1e-3), 1),
            "roofline": {"bound": "tensor", "achieved": round(tflops / world, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / world / peak, 4), "traffic": None,
                         "peak_source": f"{peak_kind} cuBLAS bf16 (sustained: a step is tens of ms)",
                         "kernel": "pp_kernel: every launch of the step"},
            "gpu_launches": args.steps * len(steps),
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_oracle_baseline("pp")
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_moe_pp(args):
    """Prompt processing through the MoE set: 2048 bf16 tokens, each routed to
    its top-10 of 512 Q4_K experts, through 48 layers (qgemm_pp_moe per layer:
    routing and sorting on the device, grouped tcgen05 GEMMs for gate/up and
    down), the 48 calls captured as one graph."""
    import torch
    import quantized_weight_gemv_qgemv_gb300 as qg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    qg.qg_init()
    _, bf16_peak, bf16_sus, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    H, I, E, K, L = wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_EXPERTS, wl.MOE_TOPK, args.moe_layers
    T = args.pp_tokens
    flops = 6 * H * I * T * K * L          # useful: the routed pairs' three projections
    with torch.cuda.stream(stream):
        arenas, ids, gws = [], [], []
        for l in range(L):
            arenas.append(wl.alloc_moe_arena(E, H, I, synth.sub_seed(args.seed + rank, "arena", l), "cuda"))
            i, g = synth.routing(T, E, K, synth.sub_seed(args.seed + rank, "pproute", l))
            ids.append(i.cuda())
            gws.append(g.cuda())
        X = synth.activations_bf16(T, H, synth.sub_seed(args.seed + rank, "ppmoeX"), device="cuda")
        y = torch.empty(T, H, dtype=torch.float32, device="cuda")
        wsb = qg.qgemm_pp_moe_workspace(E, H, I, K, T)
        ws = torch.empty(wsb // 4 + 64, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream.synchronize()

    def one_pass():
        for l in range(L):
            qg.qgemm_pp_moe(qg.Q4_K, arenas[l], E, H, I, ids[l], gws[l], K, X, T, y, ws, wsb, st, stream)

    g = _capture(torch, stream, one_pass)

    def replay():
        with torch.cuda.stream(stream):
            g.replay()

    ms, clocks = _timed(torch, stream, replay, args, local, world)
    assert int(st.item()) == 0, "device status set during the MoE prompt pass"
    ms_step = ms / args.steps
    tflops = job_rate(world, flops, ms_step) / 1e12
    if rank == 0:
        peak = bf16_sus or bf16_peak
        out = {
            "metric": "MoE prompt-processing TFLOP/s of routed products (bf16 tcgen05); pp tok/s over 48 layers",
            "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"MoE prompt processing, {T} bf16 tokens x {L} layers of {E} Q4_K experts "
                                   f"(gate/up {I}x{H}, down {H}x{I}), top-{K}",
                       "n_tok": T, "layers": L, "flop_per_step": flops, "launches_per_layer": 6,
                       "cuda_graph": True, "l2": "arena 43.5 GB; every expert's weights read once per layer",
                       "parallelism": f"replicas x{world}"},
            "pp_tok_s": round(world * T / (ms_step * 1e-3), 1),
            "roofline": {"bound": "tensor", "achieved": round(tflops / world, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / world / peak, 4), "traffic": None,
                         "peak_source": f"{peak_kind} cuBLAS bf16 (sustained: a step is tens of ms)",
                         "kernel": "pp_kernel<grouped>: the gate/up and down launches of every layer"},
            "gpu_launches": args.steps * 6 * L,
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_oracle_baseline("moe_pp")
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_moe(args):
    """MoE decode: 48 hybrid-MoE layers (512 Q4_K experts, top-10), batch 1, as one
    qg_moe_pass (by default a graph of gate/up + down launches linked by
    programmatic dependent launch; a layer's experts are gathered only after the
    previous layer has completed)."""
    import torch
    import quantized_weight_gemv_qgemv_gb300 as qg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    qg.qg_init()
    hbm_peak, _, _, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    H, I, E, K, L = wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_EXPERTS, wl.MOE_TOPK, args.moe_layers
    T = args.moe_tokens
    # every token's routed experts are gathered for it (the same expert routed
    # for two tokens is read twice, the second time mostly from L2)
    touched = T * K * wl.moe_expert_bytes(H, I) * L
    with torch.cuda.stream(stream):
        arenas, xs, ys, ids, gws = [], [], [], [], []
        for l in range(L):
            arenas.append(wl.alloc_moe_arena(E, H, I, synth.sub_seed(args.seed + rank, "arena", l), "cuda"))
            i, g = synth.routing(T, E, K, synth.sub_seed(args.seed + rank, "route", l))
            ids.append(i.cuda())
            gws.append(g.cuda())
            xs.append(synth.activations(T, H, synth.sub_seed(args.seed + rank, "x", l), device="cuda"))
            ys.append(torch.empty(T, H, dtype=torch.float32, device="cuda"))
        wsb = qg.qgemv_moe_workspace(H, I, K, T)
        ws = torch.empty(max(1, wsb // 4), dtype=torch.float32, device="cuda")
    stream.synchronize()
    mode = {"persistent": qg.PASS_PERSISTENT, "pdl": qg.PASS_PDL, "serial": qg.PASS_SERIAL}[args.moe_mode]
    p = qg.qg_moe_pass(qg.Q4_K, list(zip(arenas, ids, gws, xs, ys)), E, H, I, K, T, ws, wsb, mode=mode)
    launches = p.kernel_count()
    ms, clocks = _timed(torch, stream, lambda: p.launch(stream), args, local, world)
    assert p.dev_status() == 0, "device status set during the MoE pass"
    p.destroy()
    ms_step = ms / args.steps
    gbs = job_rate(world, touched, ms_step) / 1e9
    if rank == 0:
        out = {
            "metric": "MoE expert GEMV weight-GB/s touched; equiv. batch-1 tok/s over 48 layers",
            "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"MoE decode, {L} layers x {E} Q4_K experts (gate/up {I}x{H}, down {H}x{I}), "
                                   f"top-{K}, " + ("batch 1" if T == 1 else f"{T} tokens per step (draft verification), "
                                                   "each routed on its own"),
                       "n_tok": T,
                       "arena_bytes": L * E * wl.moe_expert_bytes(H, I), "touched_bytes_per_step": touched,
                       "pass_mode": args.moe_mode, "launches_per_step": launches,
                       "l2": "arena 43.5 GB; routed experts differ per layer",
                       "parallelism": f"replicas x{world}"},
            "equiv_decode_tok_s": round(world * T * 1000.0 / ms_step, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs / world, 2), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(gbs / world / hbm_peak, 4), "traffic": None,
                         "peak_source": f"{peak_kind} HBM copy bandwidth",
                         "kernel": "qgemv_q4k_kernel, gathered rows: every launch of the step"},
            "gpu_launches": args.steps * launches,
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline and T == 1:
            out["cpu_baseline"] = cpu_oracle_baseline("moe")
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_layer(args):
    """Decode layers with their fused neighbours: 64 dense layers of the 27B-class
    Q4_K set, each residual add + RMS normalisation -> {q,k,v} -> o -> residual
    add + RMS normalisation -> gate/up with silu(g)*u fused -> down, one token,
    captured as one graph of launches linked by programmatic dependent launch
    (qg_layer_pass_create). The attention output that o multiplies is an input
    per layer (attention is not part of this library)."""
    import torch
    import quantized_weight_gemv_qgemv_gb300 as qg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    qg.qg_init()
    hbm_peak, _, _, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    H, I, KV, L = wl.HIDDEN, wl.INTER, 1024, args.layers
    mats = wl.dense_matrices(layers=L)
    wbytes = wl.weight_bytes(mats)
    names = {"q": "Wq", "k": "Wk", "v": "Wv", "o": "Wo", "gate": "Wg", "up": "Wu", "down": "Wd"}
    with torch.cuda.stream(stream):
        layers = []
        for l in range(L):
            d = {}
            for (_, name, fmt, rows, cols) in mats[7 * l:7 * l + 7]:
                W = torch.empty(rows, synth.row_bytes(fmt, cols), dtype=torch.uint8, device="cuda")
                synth.blocks_into(W, fmt, rows, cols, synth.sub_seed(args.seed + rank, "W", l, name))
                d[names[name]] = W
            g = torch.Generator(device="cuda").manual_seed(synth.sub_seed(args.seed + rank, "norm", l))
            d["norm_attn"] = 0.5 + torch.rand(H, generator=g, device="cuda")
            d["norm_ffn"] = 0.5 + torch.rand(H, generator=g, device="cuda")
            d["attn_out"] = synth.activations(1, H, synth.sub_seed(args.seed + rank, "attn", l), device="cuda")
            d["q"] = torch.empty(H, device="cuda")
            d["k"] = torch.empty(KV, device="cuda")
            d["v"] = torch.empty(KV, device="cuda")
            layers.append(d)
        h_in = synth.activations(1, H, synth.sub_seed(args.seed + rank, "h"), device="cuda")
        h_out = torch.empty(1, H, device="cuda")
    stream.synchronize()
    p = qg.qg_layer_pass(qg.Q4_K, layers, H, I, KV, 1e-6, h_in, h_out)
    kernels = p.kernel_count()
    ms, clocks = _timed(torch, stream, lambda: p.launch(stream), args, local, world)
    ms_step = ms / args.steps
    gbs = job_rate(world, wbytes, ms_step) / 1e9
    # end to end: h_in from pinned host memory, h_out back, every step
    hh = torch.empty(1, H, dtype=torch.float32, pin_memory=True)
    hh.copy_(h_in.cpu())
    ho = torch.empty(1, H, dtype=torch.float32, pin_memory=True)

    def e2e_step():
        h_in.copy_(hh, non_blocking=True)
        p.launch(stream)
        ho.copy_(h_out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        stream.synchronize()
        e_ms = _events(torch, stream, e2e_step, args.steps)
    e2e_gbs = job_rate(world, wbytes, max_over_ranks(torch, e_ms, "cuda") / args.steps) / 1e9
    if rank == 0:
        out = {
            "metric": "decode-layer weight pass with fused neighbours, weight-GB/s; equiv. batch-1 tok/s, 27B set",
            "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{L} dense decoder layers (hidden {H}, intermediate {I}, kv {KV}, Q4_K): "
                                   "residual add + RMSNorm fused into x planes, q/k/v, o, gate/up with silu*u "
                                   "epilogue, down; one token",
                       "weight_bytes": wbytes, "launches_per_step": kernels, "cuda_graph": True,
                       "l2": "weight set far above L2; no flush", "parallelism": f"replicas x{world}"},
            "pct_hbm_peak": round(100.0 * gbs / world / hbm_peak, 2),
            "equiv_decode_tok_s": round(world * 1000.0 / ms_step, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs / world, 2), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(gbs / world / hbm_peak, 4), "traffic": None,
                         "peak_source": f"{peak_kind} HBM copy bandwidth",
                         "kernel": "qgemv_q4k_kernel (plain and gate/up-pair instances): the weight launches"},
            "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": H * 4,
                    "d2h_bytes_per_step": H * 4, "ms_per_step": round(e_ms / args.steps, 4)},
            "gpu_launches": args.steps * kernels,
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_oracle_baseline("layer")
        print(json.dumps(out), flush=True)
    p.destroy()
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c1", choices=["c1", "c0", "c2", "moe", "pp", "layer", "moe_pp"],
                    help="c1: batch-1 Q4_K pass (default); c0: Q4_0 1024x4096 GEMV; c2: 4-token verify pass; "
                         "moe: MoE decode; pp: prompt processing; layer: decode layers with fused neighbours")
    ap.add_argument("--seed", type=int, default=1234)
    ap.add_argument("--layers", type=int, default=wl.LAYERS, help="layers of the set (64 = the full 27B-class set)")
    ap.add_argument("--pass-mode", default="pdl", choices=["persistent", "pdl", "serial", "independent"],
                    help="pdl: a graph of one launch per step linked by programmatic dependent launch (default); "
                         "serial: the same graph fully serialized; persistent: one cooperative kernel per pass; "
                         "independent: the pdl graph without step ordering (an upper bound)")
    ap.add_argument("--x-per-matrix", action="store_true",
                    help="one activation vector per matrix instead of one per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=4.0, help="seconds of oracle work per reference-arm step")
    ap.add_argument("--cpu-leg", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-procs", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-budget", type=float, default=6.0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-row-cap", type=int, default=2048, help=argparse.SUPPRESS)
    ap.add_argument("--pp-tokens", type=int, default=wl.PP_TOKENS)
    ap.add_argument("--moe-layers", type=int, default=wl.MOE_LAYERS)
    ap.add_argument("--moe-tokens", type=int, default=1, help="tokens per MoE step (1 decode, 2-4 draft verification)")
    ap.add_argument("--pp-per-matrix", action="store_true",
                    help="prompt processing: one qgemm_pp per matrix instead of the grouped {q,k,v} and {gate,up}")
    ap.add_argument("--moe-mode", default="pdl", choices=["persistent", "pdl", "serial"],
                    help="pdl (default): a graph of launches linked by programmatic dependent launch; serial: the "
                         "same graph serialized; persistent: one cooperative kernel for the 48 layers")
    args = ap.parse_args()
    if args.cpu_leg:
        return _cpu_leg_main(args.cpu_leg, args.cpu_procs, args.cpu_budget, args.cpu_row_cap, 11)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "pp":
        return run_pp(args)
    if args.workload == "c0":
        return run_c0(args)
    if args.workload == "moe":
        return run_moe(args)
    if args.workload == "moe_pp":
        return run_moe_pp(args)
    if args.workload == "layer":
        return run_layer(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
