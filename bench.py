#!/usr/bin/env python
"""Throughput of the MiTA attention forward pass on GB300, one JSON line.

A step is one full forward pass (landmark pooling, landmark pass with the
shared expert, top-k expert sets, routing, bucketing, expert attention fused
with the merge) over one batch of synthetic inputs already resident in HBM, through
the C ABI ``mita_forward``. The default workload is the 32k-token long-context
case (B=2, H=16, N=32768, d=128, m=128, k=256, s=2, bf16). Inputs (805 MB)
are larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 oracle on the host cores

Under torchrun every rank runs the same workload on its own GPU (weak
scaling, no collective on the data path); a gloo barrier brackets the timed
region and rank 0 prints the job-wide line (max time over ranks).
"""
import argparse
import json
import statistics
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MiTA fwd query-tokens/sec·head and % roofline at N=32k bf16, 1×GB300"
UNIT = "query-tokens/s·head"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the dominant kernel on the 32k long-context workload, from an ncu capture of
# a smaller head count scaled to 32 heads. It is tied to the kernel source it
# was taken on (sha256 of csrc/tc.cu, first 16 hex digits); once that source
# changes, the figure no longer describes the kernel and the line reports null.
EXPERT_TRAFFIC = {"kernel": "k_expert_res", "src_sha16": "cca051e6f4bbed89", "bytes_per_launch": 128.2e6 * 32 / 6,
                  "how": "ncu dram__bytes.sum of one launch on the 6-head case (128.2 MB), scaled by 32 / 6 heads"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def work_counts(w):
    """Algorithmic flops and compulsory bytes of one forward pass."""
    elem = 2 if w.dtype == "bf16" else 4
    F = 4.0 * w.BH * w.N * w.d * (2 * w.m + w.s * w.k)
    Bytes = 4.0 * w.BH * w.N * w.d * elem
    return F, Bytes


def expert_flops(w):
    """Algorithmic flops of one expert-attention launch: q . k and p . v over
    the s * k routed slots of every query (the shared slots run in the routing
    pass, or with more than 128 landmarks in a pass of their own)."""
    return 4.0 * w.BH * w.N * w.d * w.s * w.k


def expert_src_sha16():
    """Hash of the expert kernel's source (tc.cu from its tile descriptor to
    the host code): the stored traffic figure belongs to that source only."""
    import hashlib
    with open(os.path.join(ROOT, "compressed_attention_adaptive_gb300", "csrc", "tc.cu")) as f:
        src = f.read()
    a = src.index("struct ResTile {")
    b = src.index("// ------------------------------------------------------------------ host", a)
    return hashlib.sha256(src[a:b].encode()).hexdigest()[:16]


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.gpu = gpu_index
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [ln.strip().split(", ") for ln in self.f.read().splitlines() if ln.strip()]
        self.f.close()
        os.unlink(self.f.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")
        return dist, dist.get_rank(), ws
    return None, 0, 1


def job_max(dist, x):
    """Max of a float over ranks (gloo, CPU)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class OracleSample:
    """The fp64 oracle (unchanged, one head per host thread) on a bounded
    sample of a workload: n_heads heads. The inputs are generated once, outside
    every timed region."""

    def __init__(self, w, n_heads, seed=0):
        from compressed_attention_adaptive_gb300 import synth
        Qn, Kn, Vn = synth.make_inputs(w, seed=seed, heads=list(range(n_heads)))
        f = lambda a: synth.widen(a, w.dtype)
        self.w, self.n_heads = w, n_heads
        self.Q, self.K, self.V = f(Qn), f(Kn), f(Vn)

    def run(self, q_ids=None, threads=None, heads=None):
        """Seconds for the oracle forward on `heads` of the sample (all by
        default), the queries q_ids (all if None) of each."""
        import oracle
        w = self.w
        sl = slice(None) if heads is None else slice(0, heads)
        t0 = time.perf_counter()
        oracle.forward(self.Q[sl], self.K[sl], self.V[sl], w.m, w.k, w.s, grid=w.grid, lm=w.lm, q_ids=q_ids,
                       threads=threads or self.n_heads)
        return time.perf_counter() - t0


def reference_arm(args, w, rank):
    """The oracle timed as the reference implementation (rank 0 only).

    A step is `cores` whole heads (every query), one head per thread, when
    (K + W) such steps fit in about four minutes. Otherwise a step is the same
    heads at a stride of queries, and the per-head time of the whole workload
    is assembled from two timed parts: the head's fixed work (a run with one
    query: pooling, landmark pass, expert sets; timed once before the steps)
    and the step's per-query work (its run minus the fixed part, per query),
    so that the fixed part counts once per head as in the full workload, not
    once per sampled block of queries."""
    if rank != 0:
        return
    import numpy as np
    cores = os.cpu_count() or 1
    n_heads = min(w.BH, cores)
    S = OracleSample(w, n_heads)
    t_full = S.run()  # calibration run (untimed in the line): one step of whole heads
    steps = args.steps + args.warmup
    if steps * t_full <= 240.0:
        mode, stride = "whole heads", 1
    else:
        mode = "strided queries"
        stride = 2
        while stride < 4096 and steps * (0.2 * t_full + t_full / stride) > 150.0:
            stride *= 2
    q_sparse = np.arange(0, w.N, stride)
    t_fixed = S.run(q_ids=np.array([0])) if mode != "whole heads" else 0.0  # calibration, untimed
    total_t, est = 0.0, []
    for i in range(steps):
        if mode == "whole heads":
            t = S.run()
            per_head = t
        else:
            t = S.run(q_ids=q_sparse)
            per_query = max(0.0, t - t_fixed) / max(1, len(q_sparse) - 1)
            per_head = t_fixed + (w.N - 1) * per_query
        if i >= args.warmup:
            total_t += t
            est.append(per_head)
    per_head = sum(est) / len(est)  # wall seconds for n_heads whole heads on n_heads threads
    value = n_heads * w.N / per_head
    if mode == "whole heads":
        sample = "%d of %d heads, all %d queries each, one head per thread (%d threads), fp64 oracle" % (
            n_heads, w.BH, w.N, n_heads)
    else:
        sample = ("%d of %d heads, one head per thread (%d threads), fp64 oracle; per step one run with every "
                  "%d-th query (%d per head); the whole-head time is the fixed per-head work (a run with one "
                  "query per head, timed once before the steps) plus N - 1 times the per-query time each step "
                  "measured") % (
            n_heads, w.BH, n_heads, stride, len(q_sparse))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "m": w.m, "k": w.k, "s": w.s},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_heads, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model(), "host_cpus": cores},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(w):
    """The oracle on the host cores, bounded sample: `cores` whole heads, one
    per thread; plus one head on one thread (the per-core rate)."""
    cores = os.cpu_count() or 1
    n_heads = min(w.BH, cores)
    S = OracleSample(w, n_heads)
    t = S.run()
    t1 = S.run(heads=1, threads=1)
    return {"value": n_heads * w.N / t, "unit": UNIT, "cores": n_heads, "kind": "oracle",
            "sample": "%d of %d heads, all %d queries each, fp64 oracle, one head per thread" % (n_heads, w.BH, w.N),
            "seconds": t, "cpu_model": cpu_model(), "host_cpus": cores,
            "one_head_one_thread": {"seconds": t1, "value": w.N / t1, "unit": UNIT}}


def expert_roofline(w, phase_ms, pk, pk_src, ms_step):
    """Roofline of the dominant kernel, the expert attention: algorithmic
    flops of one launch over its average duration (CUDA events recorded on the
    launching stream around the launch, inside the timed region), against the
    measured burst bf16 peak (the step is milliseconds long, not a sustained
    seconds-long loop); the sustained peak is given beside it."""
    phase = "expert_res"
    flops = expert_flops(w)
    ms = phase_ms[phase]
    achieved = flops / (ms * 1e-3) / 1e12
    kernel = "k_expert_res"
    traffic = None
    if EXPERT_TRAFFIC["kernel"] == kernel and EXPERT_TRAFFIC["src_sha16"] == expert_src_sha16() \
            and w.name == "longctx_n32k":
        traffic = EXPERT_TRAFFIC["bytes_per_launch"]
    peak = pk["bf16_tflops"]
    sus = pk.get("bf16_tflops_sustained")
    return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": traffic,
            "traffic_how": EXPERT_TRAFFIC["how"] if traffic else "no capture of the current kernel source",
            "peak_source": "%s bf16 burst (MEASURED_PEAKS.json)" % pk_src,
            "frac_of_sustained": achieved / sus if sus else None,
            "algorithmic_flops_per_launch": flops,
            "flops_counted": "4*B*H*N*d*s*k (routed slots)",
            "avg_launch_ms": ms, "share_of_step": ms / ms_step}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mita", choices=["mita", "reference"])
    ap.add_argument("--workload", default="longctx_n32k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--B", type=int, default=None, help="override the batch (small profiling cases)")
    ap.add_argument("--H", type=int, default=None, help="override the heads (small profiling cases)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every configuration (vision, 32k, 131k and the m/k/s sweep) against its roofline, "
                         "one JSON line each, instead of the benchmark line")
    ap.add_argument("--context", action="store_true",
                    help="time dense softmax attention (torch scaled_dot_product_attention, bf16) beside the MiTA "
                         "forward over N = 4k .. 128k at the long-context head shape, one JSON line per N")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (CUDA cores, fp32) on the long-context head shape at B=1, H=2")
    ap.add_argument("--causal", action="store_true",
                    help="time the causal variant on the long-context workload against its own roofline")
    ap.add_argument("--inference-mk", action="store_true",
                    help="time the MiTA forward on one fixed input while m and k grow beyond the training values "
                         "(the pages' inference-time knob), one JSON line per (m, k)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed steps
    if args.sweep:
        sweep(args)
        return
    if args.context:
        context(args)
        return
    if args.inference_mk:
        inference_mk(args)
        return
    if args.backward:
        backward_arm(args)
        return
    if args.causal:
        causal_arm(args)
        return

    from compressed_attention_adaptive_gb300 import synth
    w = synth.get(args.workload)
    if args.B or args.H:
        w = w.with_(B=args.B or w.B, H=args.H or w.H)
    dist, rank, world = _dist()
    if args.impl == "reference":
        reference_arm(args, w, rank)
        return

    import numpy as np
    import torch
    import compressed_attention_adaptive_gb300 as mita

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    Qn, Kn, Vn = synth.make_inputs(w, seed=0)
    tt = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev) if w.dtype == "bf16" \
        else torch.from_numpy(a).to(dev)
    Q, K, V = tt(Qn), tt(Kn), tt(Vn)
    O = torch.empty_like(Q)
    p = mita.params_for(Q, w.m, w.k, w.s, w.grid, w.lm)
    ws = mita.workspace(p, dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        mita.mita_forward(p, Q, K, V, O, ws)
    torch.cuda.synchronize(dev)
    mita.mita_device_status(ws)

    # The timed region replays one forward pass captured as a CUDA graph: all K
    # steps are queued at once, so a stall of the host process cannot leave
    # the GPU idle inside the region (eager launches can: the launch queue
    # fills and the host then feeds it step by step).
    graph, per_step_launches = capture_forward(mita, torch, p, Q, K, V, O, ws)
    graph.replay()
    torch.cuda.synchronize(dev)
    mita.mita_device_status(ws)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    mita.mita_device_status(ws)
    launches = per_step_launches * args.steps
    ms_step = job_max(dist, e0.elapsed_time(e1) / args.steps)
    # phases (and the expert kernel's launch time for the roofline): a separate
    # eager pass, one profile per step, median over the steps
    phase_ms = profile_phases(mita, lambda: mita.mita_forward(p, Q, K, V, O, ws), min(args.steps, 30))
    mita.mita_device_status(ws)
    value = world * w.BH * w.N / (ms_step * 1e-3)

    pk, pk_src = peaks()
    F, Bytes = work_counts(w)
    t_roof = max(F / (pk["bf16_tflops"] * 1e12), Bytes / (pk["hbm_gbs"] * 1e9))
    uses_tc = mita.mita_uses_tensor_cores(p) == 1
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "m": w.m, "k": w.k, "s": w.s,
                       "path": "tcgen05" if uses_tc else "cuda-core", "l2": "inputs larger than L2 (no flush)",
                       "parallelism": "replicas x%d" % world},
            "roofline": expert_roofline(w, phase_ms, pk, pk_src, ms_step)
            if "expert_res" in phase_ms else None,
            "path_roofline": {"t_roof_us": t_roof * 1e6, "frac": t_roof / (ms_step * 1e-3),
                              "flops": F, "compulsory_bytes": Bytes,
                              "peaks": {"bf16_tflops": pk["bf16_tflops"], "hbm_gbs": pk["hbm_gbs"],
                                        "source": pk_src}},
            "phases_ms": phase_ms, "phases_how": "separate eager pass, median per phase over %d profiled steps"
            % min(args.steps, 30), "timed_as": "one forward pass captured as a CUDA graph, replayed once per step",
            "gpu_launches": launches, "clocks": clk}

    if not args.no_e2e:
        line["e2e"] = e2e_run(mita, p, Qn, Kn, Vn, w, dev, max(30, min(args.steps, 50)), dist, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def sweep(args):
    """Per configuration: step time (CUDA events over --steps replays of the
    forward pass captured as a CUDA graph, after --warmup eager passes),
    t_roof = max(F / bf16 peak, bytes / HBM peak) and their ratio."""
    import numpy as np
    import torch
    import compressed_attention_adaptive_gb300 as mita
    from compressed_attention_adaptive_gb300 import synth
    dev = torch.device("cuda", 0)
    pk, pk_src = peaks()
    names = ["vision_128x128", "longctx_n32k", "n131k"] + [w.name for w in synth.sweep_workloads()]
    for name in names:
        w = synth.get(name)
        Qn, Kn, Vn = synth.make_inputs(w, seed=0)
        tt = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev) if w.dtype == "bf16" \
            else torch.from_numpy(a).to(dev)
        Q, K, V = tt(Qn), tt(Kn), tt(Vn)
        O = torch.empty_like(Q)
        p = mita.params_for(Q, w.m, w.k, w.s, w.grid, w.lm)
        ws = mita.workspace(p, dev)
        ms = _time_cuda(lambda: mita.mita_forward(p, Q, K, V, O, ws), args.steps, args.warmup)
        mita.mita_device_status(ws)
        F, Bytes = work_counts(w)
        t_f, t_b = F / (pk["bf16_tflops"] * 1e12), Bytes / (pk["hbm_gbs"] * 1e9)
        t_roof = max(t_f, t_b)
        print(json.dumps({"workload": name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "m": w.m, "k": w.k, "s": w.s,
                          "ms_per_step": ms, "value": w.BH * w.N / (ms * 1e-3), "unit": UNIT,
                          "flops": F, "compulsory_bytes": Bytes, "bound": "tensor" if t_f >= t_b else "hbm",
                          "t_roof_us": t_roof * 1e6, "frac": t_roof / (ms * 1e-3), "peaks": pk_src,
                          "path": "tcgen05" if mita.mita_uses_tensor_cores(p) == 1 else "cuda-core"}), flush=True)
        del Q, K, V, O, ws
        torch.cuda.empty_cache()


def pinned_host(nbytes, torch):
    """A page-locked host buffer (torch uint8 tensor) for the end-to-end run:
    anonymous memory advised for transparent huge pages (fewer, larger pages
    for the device's DMA engines to map), page-locked with cudaHostRegister;
    torch's pin_memory() when that is unavailable."""
    import mmap
    try:
        mm = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        if hasattr(mmap, "MADV_HUGEPAGE"):
            mm.madvise(mmap.MADV_HUGEPAGE)
        t = torch.frombuffer(mm, dtype=torch.uint8)
        t.zero_()  # touch every page before registering
        rc = torch.cuda.cudart().cudaHostRegister(t.data_ptr(), nbytes, 0)
        if int(rc) != 0:
            raise RuntimeError("cudaHostRegister failed: %s" % rc)
        t._mita_mmap = mm  # keeps the mapping alive with the tensor
        return t, "mmap+MADV_HUGEPAGE+cudaHostRegister"
    except Exception:
        return torch.empty(nbytes, dtype=torch.uint8).pin_memory(), "torch pin_memory"


def capture_forward(mita, torch, p, Q, K, V, O, ws):
    """One mita_forward on the current stream captured as a CUDA graph, and the
    number of this library's kernels in it (counted by the library during the
    capture; every replay launches the same kernels)."""
    n0 = mita.mita_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        mita.mita_forward(p, Q, K, V, O, ws)
    return graph, mita.mita_launch_count() - n0


def profile_phases(mita, fn, steps):
    """Per-phase milliseconds of fn() (the library's phase events), profiled
    step by step; the median of each phase over `steps` steps."""
    per = {}
    for _ in range(steps):
        mita.mita_profile_begin(64)
        fn()
        for k, v in mita.mita_profile_end().items():
            per.setdefault(k, []).append(v)
    return {k: statistics.median(v) for k, v in per.items()}


def _time_cuda(fn, steps, warmup):
    """Mean milliseconds of fn() over `steps` calls after `warmup`, CUDA events;
    fn is captured once as a CUDA graph and the graph replayed, so that the
    whole timed region is queued at once (no host stall inside it)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        fn()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def context(args):
    """Dense softmax attention against the MiTA forward over N at the
    long-context head shape (B=1, H=16, d=128; MiTA m=128, k=256, s=2):
    the measured counterpart of the pages' speed-up over standard attention.
    The dense arm is PyTorch's scaled_dot_product_attention in bf16 (a library
    flash-attention kernel), non-causal; inputs are the clustered synthetic
    long-context draws. Neither arm is part of the other."""
    import numpy as np
    import torch
    import torch.nn.functional as F
    import compressed_attention_adaptive_gb300 as mita
    from compressed_attention_adaptive_gb300 import synth
    dev = torch.device("cuda", 0)
    base = synth.WORKLOADS["longctx_n32k"]
    for N in (4096, 8192, 16384, 32768, 65536, 131072):
        w = base.with_(B=1, H=16, N=N)
        Qn, Kn, Vn = synth.make_inputs(w, seed=0)
        tt = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        Q, K, V = tt(Qn), tt(Kn), tt(Vn)
        O = torch.empty_like(Q)
        p = mita.params_for(Q, w.m, w.k, w.s)
        ws = mita.workspace(p, dev)
        steps = max(3, min(args.steps, 20 if N <= 32768 else 5))
        t_mita = _time_cuda(lambda: mita.mita_forward(p, Q, K, V, O, ws), steps, args.warmup)
        mita.mita_device_status(ws)
        t_sdpa = _time_cuda(lambda: F.scaled_dot_product_attention(Q, K, V), steps, args.warmup)
        print(json.dumps({"N": N, "B": w.B, "H": w.H, "d": w.d, "m": w.m, "k": w.k, "s": w.s, "dtype": "bf16",
                          "mita_ms": t_mita, "sdpa_ms": t_sdpa, "speedup": t_sdpa / t_mita,
                          "dense_flops": 4.0 * w.BH * N * N * w.d,
                          "mita_flops": 4.0 * w.BH * N * w.d * (2 * w.m + w.s * w.k)}), flush=True)
        del Q, K, V, O, ws
        torch.cuda.empty_cache()


def inference_mk(args):
    """One fixed input (the long-context draw at B=1, H=16, N=32768), the
    MiTA forward with m and k raised beyond the training values (m=128,
    k=256): time per forward, the roofline of each point, and the change of
    the output against the training setting (relative Frobenius distance)."""
    import numpy as np
    import torch
    import compressed_attention_adaptive_gb300 as mita
    from compressed_attention_adaptive_gb300 import synth
    dev = torch.device("cuda", 0)
    pk, pk_src = peaks()
    w0 = synth.WORKLOADS["longctx_n32k"].with_(B=1, H=16)
    Qn, Kn, Vn = synth.make_inputs(w0, seed=0)
    tt = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    Q, K, V = tt(Qn), tt(Kn), tt(Vn)
    ref = None
    for m, k in ((128, 256), (128, 512), (128, 1024), (256, 256), (256, 512), (256, 1024), (512, 512),
                 (512, 1024), (512, 2048)):
        w = w0.with_(m=m, k=k)
        O = torch.empty_like(Q)
        p = mita.params_for(Q, m, k, w.s)
        ws = mita.workspace(p, dev)
        ms = _time_cuda(lambda: mita.mita_forward(p, Q, K, V, O, ws), max(3, min(args.steps, 20)), args.warmup)
        mita.mita_device_status(ws)
        Of = O.float()
        if ref is None:
            ref = Of.clone()
        F_, B_ = work_counts(w)
        t_roof = max(F_ / (pk["bf16_tflops"] * 1e12), B_ / (pk["hbm_gbs"] * 1e9))
        print(json.dumps({"m": m, "k": k, "s": w.s, "N": w.N, "B": w.B, "H": w.H, "d": w.d, "ms": ms,
                          "value": w.BH * w.N / (ms * 1e-3), "unit": UNIT, "t_roof_us": t_roof * 1e6,
                          "frac": t_roof / (ms * 1e-3),
                          "rel_change_vs_m128_k256": float((Of - ref).norm() / ref.norm())}), flush=True)
        del O, ws
        torch.cuda.empty_cache()


def causal_arm(args):
    """The causal variant on the long-context workload (B=2, H=16, N=32768,
    m=128, k=256, s=2): time per forward and its roofline with the causal
    variant's own algorithmic flops: the shared expert of landmark i over the
    keys before its bin's end, the first floor((t + 1) m / N) shared slots of
    query t, and of each routed expert the keys at or before t (counted on the
    sets and routes this forward chose)."""
    import numpy as np
    import torch
    import compressed_attention_adaptive_gb300 as mita
    from compressed_attention_adaptive_gb300 import synth
    dev = torch.device("cuda", 0)
    pk, pk_src = peaks()
    w = synth.get("longctx_n32k")
    Qn, Kn, Vn = synth.make_inputs(w, seed=0)
    tt = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    Q, K, V = tt(Qn), tt(Kn), tt(Vn)
    O = torch.empty_like(Q)
    p = mita.params_for(Q, w.m, w.k, w.s)
    p.flags |= mita.FLAG_CAUSAL
    ws = mita.workspace(p, dev)
    idx = torch.empty((w.BH, w.m, w.k), dtype=torch.int32, device=dev)
    route = torch.empty((w.BH, w.N, w.s), dtype=torch.int32, device=dev)
    mita.mita_forward(p, Q, K, V, O, ws, idx_out=idx, route_out=route)
    torch.cuda.synchronize()
    mita.mita_device_status(ws)
    fwd = lambda: mita.mita_forward(p, Q, K, V, O, ws)
    ms = _time_cuda(fwd, max(3, min(args.steps, 50)), args.warmup)
    phases = profile_phases(mita, fwd, max(3, min(args.steps, 30)))
    mita.mita_device_status(ws)
    # algorithmic flops of the causal variant (4 d per query-key pair: q.k and p.v)
    N, m, d = w.N, w.m, w.d
    hi = np.minimum(N, ((np.arange(m) + 1) * N + m - 1) // m)  # landmark bins' ends
    shared_expert = 4.0 * d * hi.sum()
    t = np.arange(N)
    shared_slots = 4.0 * d * ((t + 1) * m // N).sum()
    routed = 0.0
    tq = torch.arange(N, device=dev, dtype=torch.int32)
    for bh in range(w.BH):
        rows = idx[bh][route[bh].long()]  # [N, s, k] ascending key indices of each routed expert
        routed += 4.0 * d * float(torch.searchsorted(rows.reshape(N * w.s, w.k).contiguous(),
                                                     tq.repeat_interleave(w.s).reshape(-1, 1),
                                                     right=True).sum())
    F = w.BH * (shared_expert + shared_slots) + routed
    _, Bytes = work_counts(w)
    t_roof = max(F / (pk["bf16_tflops"] * 1e12), Bytes / (pk["hbm_gbs"] * 1e9))
    print(json.dumps({"workload": "longctx_n32k causal", "B": w.B, "H": w.H, "N": N, "d": d, "m": m, "k": w.k,
                      "s": w.s, "ms": ms, "value": w.BH * N / (ms * 1e-3), "unit": UNIT, "flops": F,
                      "flops_non_causal": work_counts(w)[0], "t_roof_us": t_roof * 1e6,
                      "frac": t_roof / (ms * 1e-3), "phases_ms": phases,
                      "timed_as": "CUDA graph replays of the forward pass"}), flush=True)


def backward_arm(args):
    """The backward pass (mita_backward, CUDA cores in fp32) on the long-context
    head shape at B=1, H=2, N=32768, for the sets and routes of one forward
    pass: time per call (CUDA events) and its arithmetic against the fp32 FMA
    peak of the CUDA cores (152 SMs x 128 lanes x 2 flops x the SM clock)."""
    import numpy as np
    import torch
    import compressed_attention_adaptive_gb300 as mita
    from compressed_attention_adaptive_gb300 import synth
    dev = torch.device("cuda", 0)
    w = synth.WORKLOADS["longctx_n32k"].with_(B=1, H=2)
    Qn, Kn, Vn = synth.make_inputs(w, seed=0)
    tt = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    Q, K, V = tt(Qn), tt(Kn), tt(Vn)
    dO = torch.randn_like(Q)
    O, idx, route, _ = mita.forward(Q, K, V, w.m, w.k, w.s, return_sets=True)
    p = mita.params_for(Q, w.m, w.k, w.s)
    ws = torch.empty(mita.mita_backward_workspace_size(p), dtype=torch.uint8, device=dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    steps = max(3, min(args.steps, 10))
    bwd = lambda: mita.mita_backward(p, Q, K, V, dO, idx, route, dQ, dK, dV, ws)
    ms = _time_cuda(bwd, steps, args.warmup)
    phases = profile_phases(mita, bwd, steps)
    mita.mita_device_status(ws)
    slots = w.m + w.s * w.k
    flops = w.BH * w.N * (2.0 * 2 * slots * w.d + 2.0 * 3 * slots * w.d) + w.BH * 8.0 * 2 * w.m * w.N * w.d
    sm_mhz = 2070.0
    peak = 152 * 128 * 2 * sm_mhz * 1e6 / 1e12
    print(json.dumps({"workload": "longctx_n32k B1 H2 (backward)", "ms": ms, "unit": "ms per backward",
                      "flops": flops, "achieved_tflops": flops / (ms * 1e-3) / 1e12, "bound": "alu",
                      "peak_tflops": peak, "frac": flops / (ms * 1e-3) / 1e12 / peak,
                      "peak_source": "152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz",
                      "phases_ms": phases}), flush=True)


def e2e_run(mita, p, Qn, Kn, Vn, w, dev, steps, dist, world):
    """The same metric through mita_forward_host: pinned host buffers, copies
    in, forward, copy out, all inside the timed region (one call captured as a
    CUDA graph and replayed per step). Per-step CUDA events give the spread
    (median, min, max); the raw copy rate of the same buffers is measured
    beside it."""
    import numpy as np
    import torch
    nbytes = Qn.nbytes
    hb = []
    for a in (Qn, Kn, Vn):
        t, how = pinned_host(nbytes, torch)
        t.copy_(torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8)))
        hb.append(t)
    hO, _ = pinned_host(nbytes, torch)
    buf = torch.empty(mita.mita_host_buffer_size(p), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(5):
        mita.mita_forward_host(p, hb[0], hb[1], hb[2], hO, buf)
    torch.cuda.synchronize(dev)
    # one call (its copies in, forward and copy out) captured as a CUDA graph and
    # replayed per step, as in the device-resident timing: the whole timed region
    # is queued at once, so a stall of the host process leaves no gap in it
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        mita.mita_forward_host(p, hb[0], hb[1], hb[2], hO, buf)
    graph.replay()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        graph.replay()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    seq = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    per = sorted(seq)
    ms = job_max(dist, ev[0].elapsed_time(ev[steps]) / steps)
    # raw copy rates of the same pinned buffers (the floor of the end-to-end step)
    c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    c0.record(stream)
    for i in range(3):
        buf[i * nbytes:(i + 1) * nbytes].copy_(hb[i], non_blocking=True)
    c1.record(stream)
    hO.copy_(buf[:nbytes], non_blocking=True)
    c2.record(stream)
    torch.cuda.synchronize(dev)
    h2d_gbs = 3 * nbytes / (c0.elapsed_time(c1) * 1e-3) / 1e9
    d2h_gbs = nbytes / (c1.elapsed_time(c2) * 1e-3) / 1e9
    return {"value": world * w.BH * w.N / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": 3 * nbytes,
            "d2h_bytes_per_step": nbytes, "ms_per_step": ms, "steps": steps,
            "ms_median": per[len(per) // 2], "ms_min": per[0], "ms_max": per[-1],
            "slowest_step": int(max(range(steps), key=lambda i: seq[i])),
            "host_buffers": how, "timed_as": "one mita_forward_host call captured as a CUDA graph, replayed per step",
            "copy_only_h2d_gbs": h2d_gbs, "copy_only_d2h_gbs": d2h_gbs}


if __name__ == "__main__":
    main()
