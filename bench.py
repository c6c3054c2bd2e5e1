"""Benchmark of the VQ3 Hadamard-rotated vector-LUT MLP block on GB300.

Default workload: one SwiGLU block at the 27B-dense shape (hidden 5120,
intermediate 17408), T = 8 speculative-verify rows, seed 1. One step is one
full block forward (rotate x, gate/up with SiLU*mul, rotate h, down) through
the library's C ABI. Weights stream from HBM: the timed loop cycles through
enough independent weight sets (>= 4x L2) that no step finds its weights in L2.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle instead
(the reference arm of this repository, on the host cores).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import inputs as S  # noqa: E402

HIDDEN, INTER = S.HIDDEN, S.INTERMEDIATE
BLOCK_BYTES = 3 * S.stream_bytes(HIDDEN, INTER) + 2 * (2 * INTER + HIDDEN) + 3 * 64 * 2 * 2  # 100,350,720
FLOP_PER_ROW = 2 * (2 * HIDDEN * INTER + INTER * HIDDEN)  # 534,773,760
METRIC = "VQ3 Hadamard-MLP rows/s; weight GB/s vs HBM peak @T=8; TFLOP/s @prefill"
REF_BUDGET_S = 100.0
# DRAM bytes (read + write) of one persistent_kernel launch at T=8, from one ncu capture of
# the kernel (dram__bytes_read.sum + dram__bytes_write.sum); None when the kernel has changed
# since that capture.
TRAFFIC_PER_LAUNCH = 104_139_008


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(v: float, world: int, device=None) -> float:
    """The largest of every rank's v (each rank passes its own); v itself when world == 1."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units all ranks processed per second of the slowest rank (replicas: same work on each rank)."""
    return world * units_per_rank / seconds


def blas_threads():
    """Threads of the BLAS that numpy calls: threadpoolctl when it is installed, else the
    OpenBLAS thread-count entry point of the library loaded into this process, else None."""
    np.ones((4, 4)) @ np.ones((4, 4))  # make sure the BLAS is loaded
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"), default=0)
        if n:
            return n
    except Exception:
        pass
    try:
        import ctypes
        paths = sorted({ln.split()[-1] for ln in open("/proc/self/maps") if "openblas" in ln.lower() and ".so" in ln})
        for path in paths:
            lib = ctypes.CDLL(path)
            for name in ("openblas_get_num_threads", "openblas_get_num_threads64_", "scipy_openblas_get_num_threads64_",
                         "scipy_openblas_get_num_threads"):
                f = getattr(lib, name, None)
                if f is not None:
                    f.restype = ctypes.c_int
                    return int(f())
    except Exception:
        pass
    return None


def cpu_cores() -> dict:
    try:
        aff = len(os.sched_getaffinity(0))
    except AttributeError:
        aff = os.cpu_count()
    return {"cpu_count": os.cpu_count(), "affinity": aff, "blas_threads": blas_threads()}


# ------------------------------------------------------------------ oracle (CPU baseline / reference arm)

class OracleSample:
    """A bounded sample of one block for the CPU oracle. A step dequantises and
    applies a fraction `f` of every matrix's output channels (gate and up rows
    [0, n_gu), down rows [0, n_dn)) in FP64, as the oracle does for a whole
    block. Both rotations (the oracle's explicit block-matrix products) and h for
    the down rows are computed once at set-up, untimed. A step counts as
    T * (its share of the block's three weight products' multiply-adds) rows."""

    def __init__(self, rows: int, f: float, outliers: bool = False):
        from oracle import vq3_oracle as O
        self.O = O
        self.wl = S.mlp_prefill_outliers(seed=2, rows=rows) if outliers else S.mlp_27b(seed=1, rows=rows)
        blk = self.wl.layers[0]
        self.xr = O.rotate(self.wl.x.astype(np.float64), blk.gate.block, blk.gate.signs)
        # set-up only (untimed): h of every intermediate channel, output ranges on host threads
        workers = os.cpu_count() or 1
        g = O.linear_f64(self.wl.x, blk.gate, workers=workers)
        u = O.linear_f64(self.wl.x, blk.up, workers=workers)
        self.hr = O.rotate(O.silu(g) * u, blk.down.block, blk.down.signs)
        self.set_fraction(f)

    def set_fraction(self, f: float):
        self.n_gu = max(2, 2 * int(round(INTER * f / 2)))
        self.n_dn = max(2, 2 * int(round(HIDDEN * f / 2)))
        macs = 2 * self.n_gu * HIDDEN + self.n_dn * INTER
        self.share = macs / (3 * HIDDEN * INTER)

    def step(self) -> float:
        O, blk = self.O, self.wl.layers[0]
        Wg = O.dense_weight(blk.gate.stream, blk.gate.codebook, blk.gate.scales, HIDDEN, INTER, rows=(0, self.n_gu))
        Wu = O.dense_weight(blk.up.stream, blk.up.codebook, blk.up.scales, HIDDEN, INTER, rows=(0, self.n_gu))
        _ = O.silu(self.xr @ Wg.T) * (self.xr @ Wu.T)
        Wd = O.dense_weight(blk.down.stream, blk.down.codebook, blk.down.scales, INTER, HIDDEN, rows=(0, self.n_dn))
        _ = self.hr @ Wd.T
        return self.wl.x.shape[0] * self.share


def oracle_config_rates(budget_s: float = 3.0) -> dict:
    """Rows/s of the oracle as it stands on the three single-block workloads: the 256 -> 256
    linear (seed 0, 8 rows: whole calls), the block at 8 rows (seed 1) and the 64-row chunk with
    outlier channels (seed 2) (a sampled fraction of each matrix's channels per step, sized to
    about budget_s / 2 per step, two steps, scaled to whole rows). Run once with the host's
    cores and once in a child process pinned to one BLAS and OpenMP thread."""
    from oracle import vq3_oracle as O
    res = {}
    wl = S.linear_256(seed=0, rows=8)
    n, t0 = 0, time.perf_counter()
    while n < 3 or time.perf_counter() - t0 < budget_s:
        O.linear_f64(wl.x, wl.layers[0])
        n += 1
    res["linear_256x256_T8"] = round(8 * n / (time.perf_counter() - t0), 2)
    for name, rows, outl in (("mlp_5120x17408_T8", 8, False), ("mlp_5120x17408_T64_outliers", 64, True)):
        smp = OracleSample(rows, 1.0 / 256, outliers=outl)
        t0 = time.perf_counter()
        smp.step()
        t_small = time.perf_counter() - t0
        smp.set_fraction(min(0.25, max(1.0 / 2048, (budget_s / 2) / max(t_small, 1e-6) / 256)))
        units, t0 = 0.0, time.perf_counter()
        for _ in range(2):
            units += smp.step()
        res[name] = round(units / (time.perf_counter() - t0), 4)
    return res


def oracle_config_baseline() -> dict:
    """oracle_config_rates on all host cores, and in a child process with one BLAS/OpenMP thread."""
    all_cores = oracle_config_rates()
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    one = None
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-config-rates"], env=env,
                           capture_output=True, text=True, timeout=600)
        one = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal
        one = {"error": str(e)[:200]}
    return {"all_cores": all_cores, "all_cores_blas_threads": blas_threads(), "one_thread": one,
            "unit": "rows/s"}


def time_oracle(rows: int, f: float, steps: int, warmup: int):
    smp = OracleSample(rows, f)
    for _ in range(warmup):
        smp.step()
    t0 = time.perf_counter()
    units = 0.0
    for _ in range(steps):
        units += smp.step()
    dt = time.perf_counter() - t0
    return units / dt, dt, smp


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples (the JSON line carries their summary); VQ3_BENCH_OUT picks the folder
        out_dir = os.environ.get("VQ3_BENCH_OUT", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out_dir, f"clocks_bench_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self) -> dict:
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ our arm

def run_ours(args) -> dict | None:
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from bit_vector_lut_gb300 import vq3

    rows = args.rows
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(2, math.ceil(4 * l2 / BLOCK_BYTES))
    sets = []
    for k in range(n_sets):
        wl = S.mlp_27b(seed=1 + 1000 * k, rows=rows)
        sets.append(vq3.MLP.from_block(wl.layers[0], dev))
        if k == 0:
            x_host = wl.x
    x = torch.from_numpy(x_host).to(dev)
    out = torch.empty_like(x)
    ws = vq3.workspace(vq3.mlp_workspace_bytes(rows, sets[0]), dev)
    torch.cuda.synchronize(dev)
    # a side stream: CUDA graphs cannot be captured on the legacy default stream
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        return _run_ours_on(args, torch, vq3, dev, stream, rows, sets, x_host, x, out, ws, l2, n_sets, rank, world,
                            local)


def _run_ours_on(args, torch, vq3, dev, stream, rows, sets, x_host, x, out, ws, l2, n_sets, rank, world, local):

    def step(i):
        vq3.mlp_forward(x, sets[i % n_sets], out=out, ws=ws, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    # CUDA graphs: one per weight set (one block forward each) and one for a whole cycle of the
    # n_sets sets; the timed loop replays cycles, then single steps for the remainder, so it
    # runs exactly `steps` blocks and each replay submits n_sets of them
    graphs = []
    for i in range(n_sets):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            step(i)
        graphs.append(gph)
    cycle = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cycle, stream=stream):
        for i in range(n_sets):
            step(i)
    torch.cuda.synchronize(dev)
    for gph in graphs:
        gph.replay()
    cycle.replay()
    torch.cuda.synchronize(dev)
    steps = args.steps

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # nvidia-smi start-up
        barrier()
        e0.record(stream)
        for _ in range(steps // n_sets):
            cycle.replay()
        for i in range(steps % n_sets):
            graphs[i].replay()
        e1.record(stream)
        barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_per_step = ms / steps
    value = whole_job_rate(rows * steps, world, ms / 1e3)

    # dominant kernel: the block's one launch (persistent_kernel). Every launch in the timed
    # region is this kernel, so its average duration there is the region's time per launch.
    # For reference, the median of 60 launches each bracketed by events on the stream.
    launches_per_step = vq3.mlp_kernel_launches(rows, sets[0])
    k_ms = ms_per_step / launches_per_step
    durs = []
    for i in range(n_sets + 60):
        ga = torch.cuda.Event(enable_timing=True)
        gb = torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        vq3.mlp_forward(x, sets[i % n_sets], out=out, ws=ws, stream=stream)
        gb.record(stream)
        gb.synchronize()
        if i >= n_sets:
            durs.append(ga.elapsed_time(gb))
    k_ms_isolated = float(np.median(durs))
    pk = peaks()
    achieved = BLOCK_BYTES / (k_ms / 1e3) / 1e9
    traffic = args.traffic if args.traffic is not None else TRAFFIC_PER_LAUNCH
    roofline = {"bound": "hbm", "kernel": "persistent_kernel (whole MLP block, one launch)",
                "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": f"{pk['source']} (HBM copy, burst)", "ms_per_launch": round(k_ms, 5),
                "algorithmic_bytes_per_launch": BLOCK_BYTES,
                "ms_per_launch_isolated": round(k_ms_isolated, 5)}

    # end to end through the host-buffer entry point (copies in the timed region)
    hws = vq3.workspace(vq3.mlp_host_workspace_bytes(rows, sets[0]), dev, stream)
    xh = torch.from_numpy(x_host).pin_memory().numpy()
    yh = torch.empty((rows, HIDDEN), dtype=torch.float16).pin_memory().numpy()
    e2e_steps = max(n_sets, min(steps, 2000))
    for i in range(n_sets):
        vq3.mlp_forward_host(xh, sets[i % n_sets], hws, out=yh, stream=stream)
    barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        vq3.mlp_forward_host(xh, sets[i % n_sets], hws, out=yh, stream=stream)
    dt = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e = {"value": round(whole_job_rate(rows * e2e_steps, world, dt), 1), "unit": "rows/s",
           "h2d_bytes_per_step": int(x_host.nbytes), "d2h_bytes_per_step": int(rows * HIDDEN * 2),
           "api": "vq3_mlp_forward_host (pageable->pinned host buffers)"}

    extra, stack, fmts, mixers = {}, {}, {}, {}
    if not args.quick and rank == 0:
        extra = prefill_sweep(vq3, dev, stream, pk, l2)
        extra["config_outliers_T64"] = prefill_outliers_line(vq3, dev, stream, pk, l2)
        fp16_matmul_reference(extra, dev, stream)
        extra["config_linear_256_T8"] = linear256_line(vq3, dev, stream)
        stack = stack64(vq3, dev, stream, pk)
        fmts = format_lines(vq3, dev, stream, pk, l2)
        mixers = token_mixer_lines(vq3, dev, stream, pk, l2)
        mixers.update(delta_rule_lines(vq3, dev, stream))

    launches = vq3.mlp_kernel_launches(rows, sets[0]) * steps
    line = None
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world, "steps": steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f16 (fp32 accumulate)", "data": "synthetic",
                "config": {"workload": f"mlp_5120x17408_T{rows}", "hidden": HIDDEN, "intermediate": INTER,
                           "rows": rows, "rotation_block": 1024, "seed": 1, "weight_sets": n_sets,
                           "l2": f"weights rotate over {n_sets} independent sets "
                                 f"({n_sets * BLOCK_BYTES / 1e6:.0f} MB > 4x L2 {l2 / 1e6:.0f} MB)",
                           "timing": "CUDA graphs of whole weight-set cycles (then single steps for the remainder); "
                                     "CUDA events on the launching stream",
                           "parallelism": f"replicas x{world}"},
                "clocks": clk.summary(), "e2e": e2e, "gpu_launches": launches, "roofline": roofline}
        if extra:
            line["prefill_sweep"] = extra
        if stack:
            line["stack64"] = stack
        if fmts:
            line["formats"] = fmts
        if mixers:
            line["token_mixers"] = mixers
        if world == 1 and not args.no_cpu_baseline:
            rate, dt, smp = time_oracle(rows, 1.0 / args.oracle_frac, args.oracle_steps, 1)
            line["cpu_baseline"] = {"value": round(rate, 3), "unit": "rows/s", "cores": cpu_cores(),
                                    "kind": "oracle",
                                    "sample": f"{args.oracle_steps} oracle steps at T={rows}, each {smp.n_gu} gate "
                                              f"and up channels and {smp.n_dn} down channels "
                                              f"({smp.share:.4f} of the block's multiply-adds; rotations untimed), "
                                              f"{dt:.1f} s, scaled to whole rows"}
            if not args.quick:
                line["cpu_baseline"]["per_config"] = oracle_config_baseline()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def format_bytes(fmt: str) -> int:
    """Algorithmic bytes of one block in another index format: packed indices, scales, codebooks."""
    _, vec, entries = S.FORMATS[fmt]
    return (3 * S.stream_bytes(HIDDEN, INTER, fmt) + 2 * (2 * INTER + HIDDEN) + 3 * entries * vec * 2)


def format_lines(vq3, dev, stream, pk, l2) -> dict:
    """The block in the previous release's formats (two-bit vector LUT, four-bit scalar LUT): T = 8
    through a CUDA graph cycling weight sets that together exceed 4x L2 (weight GB/s against the HBM
    copy peak), and the 2048-row prefill (TFLOP/s)."""
    import torch
    res = {}
    for fmt in ("2x16", "lut4"):
        nbytes = format_bytes(fmt)
        n_sets = max(2, math.ceil(4 * l2 / nbytes))
        sets = [vq3.MLP.from_block(S.mlp_block(S.rng(S.FORMAT_SEEDS[fmt] + 1000 * k, 1), HIDDEN, INTER, 1024, fmt),
                                   dev) for k in range(n_sets)]
        x = torch.from_numpy(S.activations(S.rng(S.FORMAT_SEEDS[fmt], 0), 8, HIDDEN)).to(dev)
        out = torch.empty_like(x)
        ws = vq3.workspace(vq3.mlp_workspace_bytes(8, sets[0]), dev, stream)
        for i in range(n_sets):
            vq3.mlp_forward(x, sets[i], out=out, ws=ws, stream=stream)
        gph = torch.cuda.CUDAGraph()
        reps = 20 * n_sets
        with torch.cuda.graph(gph, stream=stream):
            for i in range(reps):
                vq3.mlp_forward(x, sets[i % n_sets], out=out, ws=ws, stream=stream)
        gph.replay()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            gph.replay()
        b.record(stream)
        b.synchronize()
        ms8 = a.elapsed_time(b) / (3 * reps)
        gbs = nbytes / (ms8 / 1e3) / 1e9
        rows = 2048
        xp = torch.from_numpy(S.activations(S.rng(S.FORMAT_SEEDS[fmt], 0), rows, HIDDEN)).to(dev)
        outp = torch.empty_like(xp)
        wsp = vq3.workspace(vq3.mlp_workspace_bytes(rows, sets[0]), dev, stream)
        for _ in range(2):
            vq3.mlp_forward(xp, sets[0], out=outp, ws=wsp, stream=stream)
        a.record(stream)
        for _ in range(3):
            vq3.mlp_forward(xp, sets[0], out=outp, ws=wsp, stream=stream)
        b.record(stream)
        b.synchronize()
        msp = a.elapsed_time(b) / 3
        tf = FLOP_PER_ROW * rows / (msp / 1e3) / 1e12
        res[fmt] = {"bits_per_weight": S.FORMATS[fmt][0] // S.FORMATS[fmt][1],
                    "algorithmic_bytes": nbytes, "T8_us": round(ms8 * 1e3, 2), "T8_rows_per_s": round(8 / (ms8 / 1e3), 1),
                    "T8_weight_gbs": round(gbs, 1), "T8_frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                    "T2048_ms": round(msp, 4), "T2048_tflops": round(tf, 2),
                    "T2048_frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                    "status": vq3.workspace_status(ws) | vq3.workspace_status(wsp)}
    return res


# token-mixer projections: the pages give their formats (two-bit vector LUT in layers 0-23, four-bit
# LUT in 24-63, rank-64 FP16 factors, 1024-wide input rotations) but not their shapes: these are synthetic
TOKEN_MIXERS = (("in_proj_5120x12288", 5120, 12288), ("out_proj_6144x5120", 6144, 5120))


def token_mixer_lines(vq3, dev, stream, pk, l2) -> dict:
    """One projection per (shape, format) with rank-64 factors at T = 8 and T = 64, through a CUDA
    graph cycling copies of the layer that together exceed 4x L2 (as for the block's formats):
    every launch of the rotation, the factor kernels and the decode kernel is in the graph."""
    import torch
    res = {}
    for name, d_in, d_out in TOKEN_MIXERS:
        for fmt in ("2x16", "lut4"):
            m = S.matrix(S.rng(80, 1), d_in, d_out, 1024, fmt)
            S.add_lowrank(S.rng(80, 3), m, 64, 0.02)
            nbytes = S.stream_bytes(d_in, d_out, fmt) + 2 * d_out + 2 * S.FORMATS[fmt][2] * S.FORMATS[fmt][1] \
                + 2 * 64 * (d_in + d_out)
            n_sets = max(2, math.ceil(4 * l2 / nbytes))
            lins = [vq3.Linear.from_matrix(m, dev) for _ in range(n_sets)]
            for rows in (8, 64):
                x = torch.from_numpy(S.activations(S.rng(80, 0), rows, d_in)).to(dev)
                out = torch.empty((rows, d_out), dtype=torch.float16, device=dev)
                ws = vq3.workspace(vq3.linear_workspace_bytes(rows, lins[0]), dev, stream)
                for lin in lins:
                    vq3.linear_forward(x, lin, out=out, ws=ws, stream=stream)
                gph = torch.cuda.CUDAGraph()
                reps = 4 * n_sets
                with torch.cuda.graph(gph, stream=stream):
                    for i in range(reps):
                        vq3.linear_forward(x, lins[i % n_sets], out=out, ws=ws, stream=stream)
                gph.replay()
                torch.cuda.synchronize(dev)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(3):
                    gph.replay()
                b.record(stream)
                b.synchronize()
                ms = a.elapsed_time(b) / (3 * reps)
                gbs = nbytes / (ms / 1e3) / 1e9
                res[f"{name}_{fmt}_T{rows}"] = {"us": round(ms * 1e3, 2), "weight_bytes": nbytes,
                                               "weight_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                                               "tflops": round(2 * d_in * d_out * rows / (ms / 1e3) / 1e12, 2),
                                               "weight_copies": n_sets, "status": vq3.workspace_status(ws)}
            del lins
    return res


def delta_rule_lines(vq3, dev, stream) -> dict:
    """The gated delta-rule block (16 heads, d_k = d_v = 128: synthetic sizes) at 8 tokens (one
    verify block) and 64 tokens (a prefill chunk): mean of 50 calls in a CUDA graph."""
    import torch
    res = {}
    for tokens in (8, 64):
        w = S.delta_rule_inputs(seed=12, tokens=tokens, heads=16, d_k=128, d_v=128)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        q, k, v, be, al, st0 = t(w.q), t(w.k), t(w.v), t(w.beta), t(w.alpha), t(w.state)
        state = st0.clone()
        out = torch.empty((tokens, 16, 128), dtype=torch.float16, device=dev)
        vq3.delta_rule_forward(q, k, v, be, al, state, out=out, stream=stream)
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            for _ in range(50):
                vq3.delta_rule_forward(q, k, v, be, al, state, out=out, stream=stream)
        gph.replay()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            gph.replay()
        b.record(stream)
        b.synchronize()
        us = a.elapsed_time(b) / 150 * 1e3
        res[f"delta_rule_16x128x128_T{tokens}"] = {"us": round(us, 2), "tokens_per_s": round(tokens / (us / 1e6), 1)}
    return res


def graph_block_us(vq3, torch, dev, stream, x, sets, rows, min_blocks) -> tuple[float, int]:
    """Microseconds per block: a CUDA graph of one cycle through the weight sets (one block per
    set, each set's weights streamed from HBM) replayed until at least `min_blocks` blocks ran,
    timed with CUDA events on the launching stream; and the workspace status."""
    out = torch.empty((rows, HIDDEN), dtype=torch.float16, device=dev)
    ws = vq3.workspace(vq3.mlp_workspace_bytes(rows, sets[0]), dev, stream)
    for lay in sets:  # warm-up: module load, tensor maps, first touches
        vq3.mlp_forward(x, lay, out=out, ws=ws, stream=stream)
    gph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gph, stream=stream):
        for lay in sets:
            vq3.mlp_forward(x, lay, out=out, ws=ws, stream=stream)
    gph.replay()
    torch.cuda.synchronize(dev)
    reps = max(1, math.ceil(min_blocks / len(sets)))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        gph.replay()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) * 1e3 / (reps * len(sets)), vq3.workspace_status(ws, stream)


def weight_sets(vq3, dev, seed: int, l2: int) -> list:
    """Independent weight sets of one block (seeds seed + 1000 k) that together exceed 4x L2."""
    n = max(2, math.ceil(4 * l2 / BLOCK_BYTES))
    return [vq3.MLP.from_block(S.mlp_block(S.rng(seed + 1000 * k, 1), HIDDEN, INTER, 1024), dev) for k in range(n)]


def prefill_sweep(vq3, dev, stream, pk, l2) -> dict:
    """The row sweep of one block (seed 4): T in {1, 8, 64, 512, 2048, 4096}. Each T runs through
    a CUDA graph cycling independent weight sets (> 4x L2, so weights stream from HBM at every T),
    at least 24 blocks per T (12 at 2048 and 4096 rows). TFLOP/s against the measured bf16 peak,
    weight GB/s against the measured HBM copy peak."""
    import torch
    res = {}
    sets = weight_sets(vq3, dev, 4, l2)
    for rows in S.SWEEP_ROWS:
        x = torch.from_numpy(S.activations(S.rng(4, 0), rows, HIDDEN)).to(dev)
        us, st = graph_block_us(vq3, torch, dev, stream, x, sets, rows, 12 if rows >= 2048 else 24)
        tf = FLOP_PER_ROW * rows / (us / 1e6) / 1e12
        gbs = BLOCK_BYTES / (us / 1e6) / 1e9
        res[f"T{rows}"] = {"us": round(us, 2), "tflops": round(tf, 2), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                           "weight_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                           "rows_per_s": round(rows / (us / 1e6), 1),
                           "launches_per_block": vq3.mlp_kernel_launches(rows, sets[0]), "status": st}
    res["weight_sets"] = len(sets)
    return res


def fp16_matmul_reference(sweep: dict, dev, stream) -> None:
    """A second denominator for the sweep's TFLOP/s: cuBLAS's dense FP16 GEMM (torch.matmul,
    8192 x 8192 x 8192, FP32 accumulate) timed in the same run on the same stream, 3 warm-up
    and 10 timed calls. Each sweep point and the outlier chunk get their fraction of it."""
    import torch
    n = 8192
    try:
        g = torch.Generator(device=dev).manual_seed(5)
        a = torch.randn((n, n), device=dev, dtype=torch.float16, generator=g)
        b = torch.randn((n, n), device=dev, dtype=torch.float16, generator=g)
        stream.wait_stream(torch.cuda.current_stream(dev))
    except RuntimeError as e:  # a reference figure only: the line keeps the reason
        sweep["fp16_matmul_tflops"] = {"error": str(e)[:200]}
        return
    with torch.cuda.stream(stream):
        c = torch.matmul(a, b)
        for _ in range(2):
            torch.matmul(a, b, out=c)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            torch.matmul(a, b, out=c)
        e1.record(stream)
    e1.synchronize()
    tflops = 2.0 * n ** 3 * 10 / (e0.elapsed_time(e1) / 1e3) / 1e12
    sweep["fp16_matmul_tflops"] = round(tflops, 1)
    for k, v in sweep.items():
        if isinstance(v, dict) and "tflops" in v:
            v["frac_of_fp16_matmul"] = round(v["tflops"] / tflops, 4)
    del a, b, c


def prefill_outliers_line(vq3, dev, stream, pk, l2) -> dict:
    """The 64-row prefill chunk with outlier channels: seed 2, X ~ N(0,1) FP16 with 51 of the 5120
    channels (1%) scaled x50, weights cycling through independent sets (> 4x L2) in a CUDA graph."""
    import torch
    sets = weight_sets(vq3, dev, 2, l2)
    wl = S.mlp_prefill_outliers(seed=2, rows=64)
    x = torch.from_numpy(wl.x).to(dev)
    us, st = graph_block_us(vq3, torch, dev, stream, x, sets, 64, 48)
    tf = FLOP_PER_ROW * 64 / (us / 1e6) / 1e12
    gbs = BLOCK_BYTES / (us / 1e6) / 1e9
    return {"workload": "mlp_5120x17408_T64_outliers", "us": round(us, 2), "rows_per_s": round(64 / (us / 1e6), 1),
            "tflops": round(tf, 2), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
            "weight_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
            "roof_us": {"tensor": round(FLOP_PER_ROW * 64 / (pk["bf16_tflops"] * 1e12) * 1e6, 2),
                        "hbm": round(BLOCK_BYTES / (pk["hbm_gbs"] * 1e9) * 1e6, 2)},
            "weight_sets": len(sets), "status": st}


def linear256_line(vq3, dev, stream) -> dict:
    """The single 256 -> 256 VQ3 linear (seed 0, 8 rows, one 256-point rotation block): a
    launch-latency-bound case, so microseconds per call (mean of 200 calls in a CUDA graph)."""
    import torch
    wl = S.linear_256(seed=0, rows=8)
    lin = vq3.Linear.from_matrix(wl.layers[0], dev)
    x = torch.from_numpy(wl.x).to(dev)
    out = torch.empty((8, 256), dtype=torch.float16, device=dev)
    ws = vq3.workspace(vq3.linear_workspace_bytes(8, lin), dev, stream)
    vq3.linear_forward(x, lin, out=out, ws=ws, stream=stream)
    gph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gph, stream=stream):
        for _ in range(200):
            vq3.linear_forward(x, lin, out=out, ws=ws, stream=stream)
    gph.replay()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(3):
        gph.replay()
    b.record(stream)
    b.synchronize()
    us = a.elapsed_time(b) * 1e3 / 600
    return {"workload": "linear_256x256_T8", "us": round(us, 3), "rows_per_s": round(8 / (us / 1e6), 1),
            "launches_per_call": 1, "status": vq3.workspace_status(ws, stream)}


def stack64(vq3, dev, stream, pk) -> dict:
    """The 64-layer stack at T = 8: per layer a residual add + RMSNorm and one MLP block
    (6.42 GB of packed weights, so every layer streams from HBM), one CUDA graph of all
    64 layers, timed with events on its stream over 5 replays after 2 warm-up replays.
    Each layer is one vq3_mlp_prenorm_step call: RMSNorm from the previous layer's
    partial sums of squares, the block, and the residual add with the next partial sums
    in the block's output step (two residual and two partial-sum buffers)."""
    import torch
    seed, rows, layers_n = 3, 8, 64
    x = torch.from_numpy(S.activations(S.rng(seed, 0), rows, HIDDEN)).to(dev)
    g = S.rng(seed, 1)
    layers = [vq3.MLP.from_block(S.mlp_block(g, HIDDEN, INTER, 1024), dev) for _ in range(layers_n)]
    res = [torch.empty_like(x), torch.empty_like(x)]
    ss = [torch.empty((rows, HIDDEN // 16), dtype=torch.float32, device=dev) for _ in range(2)]
    out = torch.empty_like(x)
    ws = vq3.workspace(vq3.mlp_workspace_bytes(rows, layers[0]), dev, stream)

    def run():
        res[0].copy_(x)
        for li, layer in enumerate(layers):
            vq3.mlp_prenorm_step(res[li % 2], layer, out, res[(li + 1) % 2], ss=ss[li % 2] if li > 0 else None,
                                 ss_next=ss[(li + 1) % 2], ws=ws, stream=stream)

    run()
    torch.cuda.synchronize(dev)
    gph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gph, stream=stream):
        run()
    for _ in range(2):
        gph.replay()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    reps = 5
    a.record(stream)
    for _ in range(reps):
        gph.replay()
    b.record(stream)
    b.synchronize()
    ms = a.elapsed_time(b) / reps
    gbs = layers_n * BLOCK_BYTES / (ms / 1e3) / 1e9
    return {"ms_per_stack": round(ms, 4), "rows_per_s": round(rows / (ms / 1e3), 1),
            "weight_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
            "status": vq3.workspace_status(ws, stream)}


def run_profile_case(args) -> None:
    """A small case for profiler captures, untimed: --steps calls at --rows rows on one weight
    set of the MLP block (~100 MB on the device), or with --case of the 5120 -> 12288
    projection with rank-64 factors (two-bit format), or of the delta-rule block (16 heads,
    128 x 128, --rows tokens)."""
    import torch
    from bit_vector_lut_gb300 import vq3
    dev = torch.device("cuda:0")
    if args.case == "lowrank":
        m = S.matrix(S.rng(80, 1), 5120, 12288, 1024, "2x16")
        S.add_lowrank(S.rng(80, 3), m, 64, 0.02)
        lin = vq3.Linear.from_matrix(m, dev)
        x = torch.from_numpy(S.activations(S.rng(80, 0), args.rows, 5120)).to(dev)
        out = torch.empty((args.rows, 12288), dtype=torch.float16, device=dev)
        ws = vq3.workspace(vq3.linear_workspace_bytes(args.rows, lin), dev)
        for _ in range(args.steps):
            vq3.linear_forward(x, lin, out=out, ws=ws)
        torch.cuda.synchronize(dev)
        print(json.dumps({"profile_case": f"linear_5120x12288_2x16_rank64_T{args.rows}", "calls": args.steps,
                          "launches_per_call": vq3.linear_kernel_launches(args.rows, lin),
                          "status": vq3.workspace_status(ws)}), flush=True)
        return
    if args.case == "delta":
        w = S.delta_rule_inputs(seed=12, tokens=args.rows, heads=16, d_k=128, d_v=128)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        q, k, v, be, al, state = t(w.q), t(w.k), t(w.v), t(w.beta), t(w.alpha), t(w.state)
        out = torch.empty((args.rows, 16, 128), dtype=torch.float16, device=dev)
        for _ in range(args.steps):
            vq3.delta_rule_forward(q, k, v, be, al, state, out=out)
        torch.cuda.synchronize(dev)
        print(json.dumps({"profile_case": f"delta_rule_16x128x128_T{args.rows}", "calls": args.steps}), flush=True)
        return
    wl = S.mlp_27b(seed=1, rows=args.rows)
    layer = vq3.MLP.from_block(wl.layers[0], dev)
    x = torch.from_numpy(wl.x).to(dev)
    out = torch.empty_like(x)
    ws = vq3.workspace(vq3.mlp_workspace_bytes(args.rows, layer), dev)
    for _ in range(args.steps):
        vq3.mlp_forward(x, layer, out=out, ws=ws)
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_case": f"mlp_5120x17408_T{args.rows}", "blocks": args.steps,
                      "launches_per_block": vq3.mlp_kernel_launches(args.rows, layer),
                      "status": vq3.workspace_status(ws)}), flush=True)


def run_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    rows = args.rows
    # size each step so that warm-up + timed steps take about REF_BUDGET_S of host time
    smp = OracleSample(rows, 1.0 / 64)
    t0 = time.perf_counter()
    smp.step()
    t64 = time.perf_counter() - t0
    per_step = REF_BUDGET_S / (args.steps + args.warmup)
    f = min(0.25, max(1e-6, per_step / t64 / 64))
    rate, dt, smp = time_oracle(rows, f, args.steps, args.warmup)
    sample = (f"each step: {smp.n_gu} gate and up channels and {smp.n_dn} down channels of one block at T={rows} "
              f"({smp.share:.6f} of its multiply-adds, FP64; rotations untimed), scaled to whole rows")
    return {"impl": "reference", "metric": METRIC, "value": round(rate, 3), "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"mlp_5120x17408_T{rows}", "hidden": HIDDEN, "intermediate": INTER, "rows": rows,
                       "rotation_block": 1024, "seed": 1},
            "cpu_baseline": {"value": round(rate, 3), "unit": "rows/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(rate, 3), "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--rows", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="skip the prefill sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-frac", type=int, default=8)
    ap.add_argument("--oracle-steps", type=int, default=32)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture, if current")
    ap.add_argument("--oracle-config-rates", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--profile-case", action="store_true",
                    help="run --steps untimed blocks at --rows on one weight set (a small case for ncu) and exit")
    ap.add_argument("--case", choices=["mlp", "lowrank", "delta"], default="mlp",
                    help="with --profile-case: the MLP block, the 5120 -> 12288 projection with rank-64 factors, "
                         "or the delta-rule block")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    if args.oracle_config_rates:  # the one-thread leg of the CPU baseline (a child process)
        print(json.dumps(dict(oracle_config_rates(), blas_threads=blas_threads())), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
