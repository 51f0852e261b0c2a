"""Benchmark of the NVFP4 skinny projection on GB300.

Metric: NVFP4 weight-stream GB/s (and fraction of the measured HBM peak) at
M = 1 / 16 / 17 / 32 on the square 5120 x 5120 projection.  Bytes per call =
N*K/2 + N*K/16 + 2*M*K + 2*M*N (codes + block scales + bf16 x + bf16 y).

One step = for each M in (1, 16, 17, 32): one call on each of R rotating weight
copies (R * 16.4 MB > 3 x L2, so every launch reads cold weights), each M-block
replayed as one CUDA graph.  Inputs are resident in HBM when the timed region
starts.  `e2e` repeats the step through the public call with pinned host
activations copied in and the output copied back, every call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling); the time is the max over ranks and `value` sums all ranks' bytes.

`other_workloads` adds the other projection shapes, the 64-layer decode round and the prefill
projection (M = 64 / 256 / 1024, TFLOP/s against the dense bf16 tensor peak); `kernel_ab` times
the two mma.sync kernels on the same shapes: the register-direct one everywhere and on the
round, the cluster-split one on the shapes it takes (the plans' default is the tcgen05 kernel).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 skinny-GEMM weight-stream GB/s and % of GB300 HBM peak at M=1/16/17/32"
HEAD_MS = (1, 16, 17, 32)
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("nvfp4_skinny_gb300/csrc/nvfp4_skinny.cu", "nvfp4_skinny_gb300/csrc/skinny_kernels.cuh",
                  "nvfp4_skinny_gb300/csrc/gemv_kernels.cuh", "nvfp4_skinny_gb300/csrc/cluster_kernels.cuh",
                  "nvfp4_skinny_gb300/csrc/ptx.cuh")
# DRAM bytes per launch measured with ncu, one JSON object per line (written from a capture's
# dram__bytes_read.sum + dram__bytes_write.sum, keyed by the kernel sources' hash)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_records.txt")


def call_bytes(N, K, M, out_bytes=2):
    return N * K // 2 + N * K // 16 + 2 * M * K + out_bytes * M * N


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(N, K, M):
    """DRAM bytes per launch of the projection kernel from the traffic records, if one was taken
    on the current kernel sources for this shape and M; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            recs = [json.loads(ln) for ln in f if ln.strip().startswith("{")]
    except Exception:
        return None
    for rec in recs:
        try:
            if (rec.get("kernel_source_hash") == kernel_source_hash() and int(rec["N"]) == N
                    and int(rec["K"]) == K and int(rec["M"]) == M):
                return int(rec["dram_bytes_per_launch"])
        except (KeyError, ValueError, TypeError):
            continue
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        # the raw samples go to $NVFP4_CLOCKS_DIR when set (the summary is in the JSON line)
        out_dir = os.environ.get("NVFP4_CLOCKS_DIR", "")
        self.path = (os.path.join(out_dir, "clocks_rank%d.csv" % device_index) if out_dir and os.path.isdir(out_dir)
                     else "/tmp/nvfp4_clocks_%d_%d.csv" % (device_index, os.getpid()))

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        if not sm:
            return None
        loaded = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- our implementation

class Projection:
    """R rotating weight copies of one [N, K] shape, resident on the device, plus a plan."""

    def __init__(self, N, K, seed, copies, f32_out=False, flags=0):
        import torch
        from nvfp4_skinny_gb300 import binding as nb
        from nvfp4_skinny_gb300 import synth
        self.N, self.K, self.f32_out = N, K, f32_out
        self.plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_F32 if f32_out else nb.NVFP4_OUT_BF16, flags)
        self.w = [synth.weights(N, K, seed + 7919 * i, device="cuda") for i in range(copies)]
        self.out_dtype = torch.float32 if f32_out else torch.bfloat16
        self.out_bytes = 4 if f32_out else 2


def make_graph(calls, stream):
    """Capture a list of zero-argument callables into one CUDA graph on `stream`."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c in calls:
            c()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c()
    return g


def run_ours(args, rank, world):
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    from nvfp4_skinny_gb300 import build as nbuild
    from nvfp4_skinny_gb300 import synth

    nbuild.build()
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    peak, peak_src = hbm_peak()

    # ---------------- headline: square projection, M sweep, rotating cold weights
    sq = synth.WORKLOADS["square"].projections[0]
    per_copy = call_bytes(sq.N, sq.K, 1)
    copies = max(args.copies, -(-3 * L2_BYTES // per_copy))
    proj = Projection(sq.N, sq.K, sq.seed + 1000 * rank, copies)
    x_all = synth.activations(32, sq.K, sq.seed + 1000 * rank, device="cuda")
    ys = {M: torch.empty((M, sq.N), dtype=torch.bfloat16, device="cuda") for M in HEAD_MS}
    xs = {M: x_all[:M].contiguous() for M in HEAD_MS}

    def call(M, i, s=stream):
        c, sc, gs = proj.w[i]
        return lambda: nb.nvfp4_skinny_linear(proj.plan, xs[M], M, c, sc, gs, ys[M], stream=s)

    graphs = {M: make_graph([call(M, i) for i in range(copies)], stream) for M in HEAD_MS}
    step_bytes = {M: copies * call_bytes(sq.N, sq.K, M) for M in HEAD_MS}

    def one_step(ev=None):
        with torch.cuda.stream(stream):
            for j, M in enumerate(HEAD_MS):
                if ev is not None:
                    ev[j].record(stream)
                graphs[M].replay()
            if ev is not None:
                ev[len(HEAD_MS)].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if nb.nvfp4_plan_check(proj.plan, stream) != nb.NVFP4_OK:
        raise RuntimeError("kernel reported an error during warm-up")

    clocks = ClockSampler(dev)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(HEAD_MS) + 1)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        one_step(events[k])
    t_stop.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_stop)
    step_m_ms = {M: [events[k][j].elapsed_time(events[k][j + 1]) for k in range(args.steps)]
                 for j, M in enumerate(HEAD_MS)}
    per_m_ms = {M: sum(v) for M, v in step_m_ms.items()}
    status = nb.nvfp4_plan_check(proj.plan, stream)
    if status != nb.NVFP4_OK:
        raise RuntimeError("kernel reported %s in the timed region" % nb.nvfp4_status_string(status))
    total_ms = max_over_ranks(total_ms, world)
    bytes_per_step = sum(step_bytes.values())
    value = bytes_per_step * args.steps * world / (total_ms * 1e-3) / 1e9
    launches_per_step = copies * len(HEAD_MS) * nb.nvfp4_plan_get_info(proj.plan)["launches_per_call"]

    per_m = {}
    for M in HEAD_MS:
        t_call = per_m_ms[M] / (args.steps * copies)  # ms per call
        gbs = call_bytes(sq.N, sq.K, M) / (t_call * 1e-3) / 1e9
        q = statistics.quantiles([v / copies * 1e3 for v in step_m_ms[M]], n=10) if args.steps > 1 else None
        per_m[str(M)] = {"us_per_call": round(t_call * 1e3, 3), "GBps": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 4),
                         "us_per_call_p10_p50_p90_over_steps": [round(q[0], 3), round(q[4], 3), round(q[8], 3)] if q
                         else None}

    # roofline of the dominant kernel: algorithmic bytes per call / average call time over the timed region
    avg_call_ms = total_ms / (args.steps * copies * len(HEAD_MS))
    avg_bytes = bytes_per_step / (copies * len(HEAD_MS))
    achieved = avg_bytes / (avg_call_ms * 1e-3) / 1e9
    traffic = recorded_traffic(sq.N, sq.K, 16)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one M=16 launch of the "
                                  "projection kernel (the traffic records under profiles/); null once the kernel "
                                  "sources change",
                "algorithmic_bytes_per_launch": int(avg_bytes), "peak_source": peak_src,
                "timing": "CUDA events on the launching stream over the timed region; a call is the "
                          "plan's launches (one skinny_kernel for this shape; back-to-back calls overlap "
                          "through programmatic dependent launch)"}

    # ---------------- e2e through the public call: pinned host x in, host y out, every call
    e2e = run_e2e(args, proj, x_all, stream, world)

    # ---------------- other workloads (reported alongside, not the headline)
    others = {} if args.quick else run_other_workloads(stream, rank, peak)
    # ---------------- the two mma.sync kernels on the same shapes (A/B against the default tcgen05)
    ab = {} if args.quick else {
        "mma_sync": {
            "kernel": "register-direct mma.sync (NVFP4_PLAN_KERNEL_MMA_SYNC); the default plans run tcgen05",
            "square 5120x5120": run_square_ab(stream, rank, peak, nb.NVFP4_PLAN_KERNEL_MMA_SYNC),
            **run_other_workloads(stream, rank, peak, flags=nb.NVFP4_PLAN_KERNEL_MMA_SYNC, Ms=HEAD_MS,
                                  with_prefill=False)},
        "cluster": {
            "kernel": "cluster-split mma.sync, one launch (NVFP4_PLAN_KERNEL_CLUSTER); only the shapes it takes",
            "square 5120x5120": run_square_ab(stream, rank, peak, nb.NVFP4_PLAN_KERNEL_CLUSTER),
            **run_other_workloads(stream, rank, peak, flags=nb.NVFP4_PLAN_KERNEL_CLUSTER, Ms=HEAD_MS,
                                  with_prefill=False, with_round=False)}}

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": "square 5120x5120 NVFP4 projection (N=5120, K=5120), M in {1,16,17,32}, "
                               "%d rotating weight copies per M (%.0f MB > L2), each M-block one CUDA graph"
                               % (copies, copies * per_copy / 1e6),
                   "N": sq.N, "K": sq.K, "Ms": list(HEAD_MS), "weight_copies": copies,
                   "l2": "inputs larger than L2 (rotating weight copies)", "parallelism": "replicas"},
        "frac_of_peak": round(value / world / peak, 4),
        "per_m": per_m,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "other_workloads": others,
        "kernel_ab": ab,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return out


def run_e2e(args, proj, x_all, stream, world):
    """Public call with host buffers: H2D of x from pinned memory, the call, D2H of y, around every
    call.  The step is timed as one CUDA graph of those copies and calls (how a serving loop
    issues it; the copies move host memory on every replay) and, for comparison, eagerly from
    Python."""
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    N, K = proj.N, proj.K
    hx = {M: x_all[:M].cpu().pin_memory() for M in HEAD_MS}
    hy = {M: torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for M in HEAD_MS}
    dx = {M: torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for M in HEAD_MS}
    dy = {M: torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for M in HEAD_MS}
    copies = len(proj.w)
    steps = max(3, args.steps // 20)

    def step():
        with torch.cuda.stream(stream):
            for M in HEAD_MS:
                for i in range(copies):
                    c, sc, gs = proj.w[i]
                    dx[M].copy_(hx[M], non_blocking=True)
                    nb.nvfp4_skinny_linear(proj.plan, dx[M], M, c, sc, gs, dy[M], stream=stream)
                    hy[M].copy_(dy[M], non_blocking=True)

    def timed(run, n):
        # everything (the graph replays included) runs on `stream`, between its two events
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(n):
                run()
            b.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b), world)

    byts = sum(copies * call_bytes(N, K, M) for M in HEAD_MS)
    h2d = sum(copies * M * K * 2 for M in HEAD_MS)
    d2h = sum(copies * M * N * 2 for M in HEAD_MS)
    step()
    ms_eager = timed(step, steps)
    g = make_graph([step], stream)
    with torch.cuda.stream(stream):
        g.replay()
    ms_graph = timed(lambda: g.replay(), steps)
    rate = lambda ms: round(byts * steps * world / (ms * 1e-3) / 1e9, 1)
    return {"value": rate(ms_graph), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps,
            "how": "public calls with pinned host x copied in and y copied out around every call, the step "
                   "replayed as one CUDA graph",
            "eager": {"value": rate(ms_eager), "unit": "GB/s",
                      "how": "the same step issued eagerly from Python, call by call"}}


def run_square_ab(stream, rank, peak, flags):
    """The headline square projection on plans made with `flags` (another kernel), each M as in
    other_workloads."""
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    from nvfp4_skinny_gb300 import synth
    sq = synth.WORKLOADS["square"].projections[0]
    copies = max(2, -(-3 * L2_BYTES // call_bytes(sq.N, sq.K, 1)))
    proj = Projection(sq.N, sq.K, sq.seed + 1000 * rank, copies, False, flags)
    x_all = synth.activations(32, sq.K, sq.seed, device="cuda")
    entry = {}
    for M in HEAD_MS:
        xm = x_all[:M].contiguous()
        y = torch.empty((M, sq.N), dtype=torch.bfloat16, device="cuda")
        calls = [(lambda c=c, sc=sc, gs=gs: nb.nvfp4_skinny_linear(proj.plan, xm, M, c, sc, gs, y, stream=stream))
                 for (c, sc, gs) in proj.w]
        t_call = _time_graph(make_graph(calls, stream), stream, 10) / copies
        gbs = call_bytes(sq.N, sq.K, M) / (t_call * 1e-3) / 1e9
        entry[str(M)] = {"us_per_call": round(t_call * 1e3, 3), "GBps": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 4)}
    assert nb.nvfp4_plan_check(proj.plan, stream) == nb.NVFP4_OK
    del proj
    torch.cuda.empty_cache()
    return entry


def _time_graph(g, stream, reps, warm=3):
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def run_other_workloads(stream, rank, peak, flags=0, Ms=None, with_prefill=True, with_round=True):
    """QKV / down, wide gate|up / head (fp32 out), and the full 64-layer decode round (on plans
    made with `flags`; each shape at its workload's Ms, or at `Ms`).  A shape the flags' kernel
    does not take is reported as such."""
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    from nvfp4_skinny_gb300 import synth
    res = {}
    for wl in ("qkv_down", "wide_head"):
        w = synth.WORKLOADS[wl]
        for pj in w.projections:
            per_copy = call_bytes(pj.N, pj.K, 1, 4 if pj.f32_out else 2)
            copies = max(2, -(-3 * L2_BYTES // per_copy))
            name = "%s %dx%d%s" % (pj.name, pj.N, pj.K, " f32-out" if pj.f32_out else "")
            try:
                nb.nvfp4_plan_create_flags(pj.N, pj.K, nb.NVFP4_OUT_BF16, flags).destroy()
            except nb.Nvfp4Error as e:
                res[name] = {"not_planned": str(e)}
                continue
            proj = Projection(pj.N, pj.K, pj.seed + 1000 * rank, copies, pj.f32_out, flags)
            x_all = synth.activations(32, pj.K, pj.seed, device="cuda", outlier_frac=w.outlier_frac)
            entry = {}
            for M in (Ms or w.Ms):
                xm = x_all[:M].contiguous()
                y = torch.empty((M, pj.N), dtype=proj.out_dtype, device="cuda")
                calls = [(lambda c=c, sc=sc, gs=gs: nb.nvfp4_skinny_linear(proj.plan, xm, M, c, sc, gs, y,
                                                                           stream=stream))
                         for (c, sc, gs) in proj.w]
                t_call = _time_graph(make_graph(calls, stream), stream, 10) / copies
                byts = call_bytes(pj.N, pj.K, M, proj.out_bytes)
                gbs = call_bytes(pj.N, pj.K, M) / (t_call * 1e-3) / 1e9
                entry[str(M)] = {"us_per_call": round(t_call * 1e3, 3), "GBps": round(gbs, 1),
                                 "frac_of_peak": round(gbs / peak, 4),
                                 "GBps_actual_out_bytes": round(byts / (t_call * 1e-3) / 1e9, 1)}
            res[name] = entry
            assert nb.nvfp4_plan_check(proj.plan, stream) == nb.NVFP4_OK
            del proj
            torch.cuda.empty_cache()
    if with_round:
        res["round"] = run_round(stream, rank, peak, flags)
    if with_prefill:
        res["prefill"] = run_prefill(stream, rank)
    return res


def bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s (the fp16 MMAs of the prefill run at the same rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback"


PREFILL_MS = (64, 256, 1024)


def run_prefill(stream, rank):
    """The prefill projection (row counts above the skinny band) on the stated projection shapes:
    time per call over rotating cold weight copies, TFLOP/s against the dense bf16 tensor peak."""
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    from nvfp4_skinny_gb300 import synth
    tpeak, tsrc = bf16_peak()
    out = {"peak_tflops": tpeak, "peak_source": tsrc,
           "timing": "CUDA graph of back-to-back calls (activation preparation, projection and, when the "
                     "k-range is split, the reduction), rotating weight copies > 2x L2"}
    for name, N, K in (("square", 5120, 5120), ("qkv", 7168, 5120), ("gate_up", 34816, 5120),
                       ("down", 5120, 17408)):
        per_copy = call_bytes(N, K, 1)
        copies = min(16, max(2, -(-2 * L2_BYTES // per_copy)))
        ws = [synth.weights(N, K, 300 + 7919 * i + 1000 * rank, device="cuda") for i in range(copies)]
        plan = nb.nvfp4_prefill_plan_create(N, K, max(PREFILL_MS))
        entry = {}
        for M in PREFILL_MS:
            x = synth.activations(M, K, 5, device="cuda")
            y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            calls = [(lambda c=c, sc=sc, gs=gs: nb.nvfp4_prefill_linear(plan, x, M, c, sc, gs, y, stream=stream))
                     for (c, sc, gs) in ws]
            t_call = _time_graph(make_graph(calls, stream), stream, 5) / copies  # ms
            tf = 2.0 * M * N * K / (t_call * 1e-3) / 1e12
            g = nb.nvfp4_prefill_plan_get_info(plan, M)
            entry[str(M)] = {"us_per_call": round(t_call * 1e3, 2), "TFLOPs": round(tf, 1),
                             "frac_of_peak": round(tf / tpeak, 4), "bm": g["bm"], "m_tiles": g["m_tiles"],
                             "splits": g["splits"], "grid": g["grid"], "launches": g["launches_per_call"]}
        assert nb.nvfp4_prefill_plan_check(plan, stream) == nb.NVFP4_OK
        out["%s %dx%d" % (name, N, K)] = entry
        del ws, plan
        torch.cuda.empty_cache()
    return out


def run_round(stream, rank, peak, flags=0):
    """64 layers x {qkv, o, gate|up, down}: 256 calls back to back, eager and as one CUDA graph."""
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    from nvfp4_skinny_gb300 import synth
    w = synth.WORKLOADS["round"]
    plans = {}
    weights = []
    for pj in w.projections:
        key = (pj.N, pj.K)
        if key not in plans:
            plans[key] = nb.nvfp4_plan_create_flags(pj.N, pj.K, nb.NVFP4_OUT_BF16, flags)
        weights.append((pj, synth.weights(pj.N, pj.K, pj.seed + 100000 * rank, device="cuda")))
    total_w = sum(pj.N * pj.K // 2 + pj.N * pj.K // 16 for pj, _ in weights)
    out = {"launches": len(weights), "weight_bytes": total_w}
    for M in w.Ms:
        xs = {K: synth.activations(M, K, 1, device="cuda") for K in (5120, 17408)}
        ys = {N: torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for N in (5120, 7168, 34816)}

        def round_calls():
            for pj, (c, sc, gs) in weights:
                nb.nvfp4_skinny_linear(plans[(pj.N, pj.K)], xs[pj.K], M, c, sc, gs, ys[pj.N], stream=stream)

        byts = sum(call_bytes(pj.N, pj.K, M) for pj, _ in weights)
        with torch.cuda.stream(stream):
            round_calls()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                round_calls()
            b.record(stream)
        torch.cuda.synchronize()
        t_eager = a.elapsed_time(b) / reps
        t_graph = _time_graph(make_graph([round_calls], stream), stream, reps, warm=2)
        out[str(M)] = {"eager_ms": round(t_eager, 4), "graph_ms": round(t_graph, 4),
                       "graph_GBps": round(byts / (t_graph * 1e-3) / 1e9, 1),
                       "graph_frac_of_peak": round(byts / (t_graph * 1e-3) / 1e9 / peak, 4),
                       "eager_GBps": round(byts / (t_eager * 1e-3) / 1e9, 1)}
    for p in plans.values():
        assert nb.nvfp4_plan_check(p, stream) == nb.NVFP4_OK
    return out


# ----------------------------------------------------------------------------- CPU oracle

_ORACLE_INPUTS = {}


def _oracle_inputs():
    """Seeded square-workload inputs on the host (generated once)."""
    if not _ORACLE_INPUTS:
        import numpy as np
        import torch
        from nvfp4_skinny_gb300 import synth
        sq = synth.WORKLOADS["square"].projections[0]
        codes, scales, gs = synth.weights(sq.N, sq.K, sq.seed)
        x = synth.activations(32, sq.K, sq.seed)
        _ORACLE_INPUTS.update(N=sq.N, K=sq.K, gs=gs, codes=codes.numpy(), scales=scales.numpy(),
                              xb=x.contiguous().view(torch.int16).numpy().view(np.uint16))
    return _ORACLE_INPUTS


def _oracle_sample(seconds_target, M_list=HEAD_MS):
    """Time the oracle on a bounded sample of the square workload: for each M, all outputs of
    a subset of weight rows.  Returns (GB/s in the metric's bytes, seconds, sample text, threads)."""
    import oracle
    d = _oracle_inputs()
    N, K, gs = d["N"], d["K"], d["gs"]
    orc = oracle.default()
    threads = orc.max_threads()
    if "per_row_m" not in d:
        t0 = time.perf_counter()
        orc.linear(d["xb"][:1], d["codes"][:64], d["scales"][:64], gs)
        d["per_row_m"] = max((time.perf_counter() - t0) / 64, 1e-7)
    rows = int(max(8, min(N, seconds_target / (d["per_row_m"] * sum(M_list)))))
    elapsed = 0.0
    byts = 0.0
    for M in M_list:
        t0 = time.perf_counter()
        orc.linear(d["xb"][:M], d["codes"][:rows], d["scales"][:rows], gs)
        elapsed += time.perf_counter() - t0
        byts += call_bytes(N, K, M) * rows / N  # the metric's bytes for the covered fraction of the call
    sample = ("oracle (fp64, OpenMP over weight rows) on the square 5120x5120 workload: the first %d of %d "
              "weight rows against all M activation rows, for each M in %s; bytes = the call's bytes x %d/%d"
              % (rows, N, list(M_list), rows, N))
    return byts / elapsed / 1e9, elapsed, sample, threads


def _oracle_configs(seconds_each):
    """The oracle on every other single-projection shape and on one layer of the decode round
    (the round is 64 such layers): for M = 1 and 32, a bounded sample of weight rows, in the
    metric's bytes for the covered fraction.  Timing does not depend on the values, so each
    shape's sample rows are generated on their own (2048 rows, the shape's K)."""
    import numpy as np
    import torch
    import oracle
    from nvfp4_skinny_gb300 import synth
    orc = oracle.default()
    shapes = (("qkv", 7168, 5120, 2, 3), ("o", 5120, 5120, 2, 2), ("down", 5120, 17408, 2, 4),
              ("gate_up", 34816, 5120, 2, 5), ("head", 152064, 5120, 4, 6))
    out, layer_t, layer_b = {}, {1: 0.0, 32: 0.0}, {1: 0.0, 32: 0.0}
    for name, N, K, ob, seed in shapes:
        codes, scales, gs = synth.weights(2048, K, seed)
        c, sc = codes.numpy(), scales.numpy()
        xb = synth.activations(32, K, seed).contiguous().view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        orc.linear(xb[:1], c[:16], sc[:16], gs)
        per_row_m = max((time.perf_counter() - t0) / 16, 1e-7)
        entry = {}
        for M in (1, 32):
            rows = int(max(8, min(2048, seconds_each / 2 / (per_row_m * M))))
            t0 = time.perf_counter()
            orc.linear(xb[:M], c[:rows], sc[:rows], gs)
            dt = time.perf_counter() - t0
            gbs = call_bytes(N, K, M, ob) * rows / N / dt / 1e9
            entry[str(M)] = {"GBps": round(gbs, 6), "rows": rows, "seconds": round(dt, 3)}
            if name != "head":  # a decode-round layer is qkv, o, gate|up and down
                layer_t[M] += dt * N / rows
                layer_b[M] += call_bytes(N, K, M, ob)
        out["%s %dx%d%s" % (name, N, K, " f32-out" if ob == 4 else "")] = entry
    out["round layer (x64 for the round)"] = {str(M): {"GBps": round(layer_b[M] / layer_t[M] / 1e9, 6),
                                                       "round_seconds_estimate": round(64 * layer_t[M], 1)}
                                              for M in (1, 32)}
    return out


def cpu_baseline(seconds_target):
    gbs, elapsed, sample, threads = _oracle_sample(seconds_target)
    return {"value": round(gbs, 6), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
            "seconds": round(elapsed, 2),
            "other_configs": _oracle_configs(max(0.5, seconds_target / 10))}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, as it stands, on bounded samples of the same workload."""
    if rank != 0:
        return None
    per_step = max(0.002, min(5.0, args.cpu_seconds / max(1, args.steps)))
    for _ in range(args.warmup):
        _oracle_sample(per_step / 4)
    tot_b, tot_t = 0.0, 0.0
    sample = ""
    threads = 1
    for _ in range(args.steps):
        gbs, el, sample, threads = _oracle_sample(per_step)
        tot_b += gbs * el
        tot_t += el
    value = tot_b / tot_t
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "square 5120x5120 NVFP4 projection (N=5120, K=5120), M in {1,16,17,32}; "
                                   "each step a bounded sample of weight rows", "N": 5120, "K": 5120,
                       "Ms": list(HEAD_MS)},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_shape(args):
    """Calls of one shape on rotating cold weights (> 2x L2), for ncu captures: for each M in
    turn (N,K,M1:M2:...), --warmup then --steps calls."""
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    from nvfp4_skinny_gb300 import build as nbuild
    from nvfp4_skinny_gb300 import synth
    nbuild.build()
    parts = args.profile_shape.split(",")
    N, K = int(parts[0]), int(parts[1])
    Ms = [int(v) for v in parts[2].split(":")]
    f32 = len(parts) > 3 and parts[3] == "f32"
    copies = max(2, -(-2 * L2_BYTES // call_bytes(N, K, 1)))
    proj = Projection(N, K, 77, copies, f32, nb.NVFP4_PLAN_KERNEL_MMA_SYNC if args.mma else 0)
    x_all = synth.activations(max(Ms), K, 77, device="cuda")
    torch.cuda.synchronize()
    i = 0
    for M in Ms:
        x = x_all[:M].contiguous()
        y = torch.empty((M, N), dtype=proj.out_dtype, device="cuda")
        for _ in range(args.warmup + args.steps):
            c, sc, gs = proj.w[i % copies]
            nb.nvfp4_skinny_linear(proj.plan, x, M, c, sc, gs, y)
            i += 1
        torch.cuda.synchronize()
    st = nb.nvfp4_plan_check(proj.plan)
    if st != nb.NVFP4_OK:
        raise RuntimeError(nb.nvfp4_status_string(st))
    print("profiled shape N=%d K=%d Ms=%s copies=%d calls per M=%d kernel=%s" % (
        N, K, Ms, copies, args.warmup + args.steps, "mma" if args.mma else "tcgen05"))


def profile_round(args):
    """The 64-layer decode round (qkv, o, gate|up, down per layer), --warmup then --steps rounds
    at one M, issued eagerly, for an ncu launch list (the per-launch times of all 256 calls)."""
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    from nvfp4_skinny_gb300 import build as nbuild
    from nvfp4_skinny_gb300 import synth
    nbuild.build()
    M = int(args.profile_round)
    w = synth.WORKLOADS["round"]
    plans = {}
    weights = []
    for pj in w.projections:
        if (pj.N, pj.K) not in plans:
            plans[(pj.N, pj.K)] = nb.nvfp4_plan_create(pj.N, pj.K)
        weights.append((pj, synth.weights(pj.N, pj.K, pj.seed, device="cuda")))
    xs = {K: synth.activations(M, K, 1, device="cuda") for K in (5120, 17408)}
    ys = {N: torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for N in (5120, 7168, 34816)}
    torch.cuda.synchronize()
    for _ in range(args.warmup + args.steps):
        for pj, (c, sc, gs) in weights:
            nb.nvfp4_skinny_linear(plans[(pj.N, pj.K)], xs[pj.K], M, c, sc, gs, ys[pj.N])
    torch.cuda.synchronize()
    for p in plans.values():
        if nb.nvfp4_plan_check(p) != nb.NVFP4_OK:
            raise RuntimeError("kernel reported an error")
    print("profiled round M=%d calls per round=%d rounds=%d" % (M, len(weights), args.warmup + args.steps))


def profile_prefill(args):
    """A few prefill calls of one shape on rotating cold weights (> 2x L2), for ncu captures."""
    import torch
    from nvfp4_skinny_gb300 import binding as nb
    from nvfp4_skinny_gb300 import build as nbuild
    from nvfp4_skinny_gb300 import synth
    nbuild.build()
    N, K, M = (int(v) for v in args.profile_prefill.split(","))
    copies = max(2, -(-2 * L2_BYTES // call_bytes(N, K, 1)))
    ws = [synth.weights(N, K, 77 + 7919 * i, device="cuda") for i in range(copies)]
    plan = nb.nvfp4_prefill_plan_create(N, K, M)
    x = synth.activations(M, K, 77, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    for i in range(args.warmup + args.steps):
        c, sc, gs = ws[i % copies]
        nb.nvfp4_prefill_linear(plan, x, M, c, sc, gs, y)
    torch.cuda.synchronize()
    st = nb.nvfp4_prefill_plan_check(plan)
    if st != nb.NVFP4_OK:
        raise RuntimeError(nb.nvfp4_status_string(st))
    print("profiled prefill N=%d K=%d M=%d copies=%d calls=%d geometry=%s" % (
        N, K, M, copies, args.warmup + args.steps, nb.nvfp4_prefill_plan_get_info(plan, M)))


# ----------------------------------------------------------------------------- distributed plumbing

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("NVFP4_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--copies", type=int, default=32, help="rotating weight copies per M (raised to > 3x L2)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip the other workloads")
    ap.add_argument("--profile-shape", default=None, metavar="N,K,M[:M2...][,f32]",
                    help="profiling driver: for each M, run --warmup then --steps calls of one shape on cold "
                         "weights, no JSON")
    ap.add_argument("--mma", action="store_true", help="--profile-shape on register-direct mma.sync plans")
    ap.add_argument("--profile-round", default=None, metavar="M",
                    help="run the 64-layer decode round at one M eagerly (for ncu launch lists), then exit")
    ap.add_argument("--profile-prefill", default=None, metavar="N,K,M",
                    help="run a few prefill calls of one shape (for ncu) and exit")
    args = ap.parse_args(argv)
    if args.profile_shape:
        return profile_shape(args)
    if args.profile_prefill:
        return profile_prefill(args)
    if args.profile_round:
        return profile_round(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world = dist_init()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
