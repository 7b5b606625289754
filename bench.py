#!/usr/bin/env python
"""Throughput of the MiTA attention forward pass on GB300, one JSON line.

A step is one full forward pass (landmark pooling, landmark pass with the
shared expert, top-k expert sets, routing, bucketing, expert attention with
the merge) over one batch of synthetic inputs already resident in HBM, through
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
# dram__bytes_read.sum + dram__bytes_write.sum of one expert-attention launch
# (k_expert_res) on the 32k long-context workload: a 6-head capture (157.9 MB)
# scaled by 32 / 6 heads (profiles/k_expert_res_longctx_6heads.md).
EXPERT_TRAFFIC_BYTES = 8.42e8


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
    expert_F = 4.0 * w.BH * w.N * w.d * (w.s * w.k + w.m)  # routed slots + shared slots
    return F, Bytes, expert_F


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


def oracle_sample(w, n_heads, q_stride, threads, seed=0):
    """Times the fp64 oracle on n_heads heads (one per thread), every
    q_stride-th query. Returns (seconds, query-tokens*heads processed)."""
    import numpy as np
    import oracle
    from compressed_attention_adaptive_gb300 import synth
    heads = list(range(n_heads))
    Qn, Kn, Vn = synth.make_inputs(w, seed=seed, heads=heads)
    f = lambda a: synth.widen(a, w.dtype)
    Q, K, V = f(Qn), f(Kn), f(Vn)
    q_ids = None if q_stride == 1 else np.arange(0, w.N, q_stride)
    t0 = time.perf_counter()
    oracle.forward(Q, K, V, w.m, w.k, w.s, grid=w.grid, lm=w.lm, q_ids=q_ids, threads=threads)
    dt = time.perf_counter() - t0
    nq = w.N if q_ids is None else len(q_ids)
    return dt, n_heads * nq


def reference_arm(args, w, rank):
    """The oracle timed as the reference implementation (rank 0 only)."""
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    n_heads = min(w.BH, cores)
    # per step about 150 s / (K + W), at least one landmark pass per head
    budget = 150.0 / max(1, args.steps + args.warmup)
    stride = 1
    while stride < 64 and 2.5 + 8.6 / stride > budget:
        stride *= 2
    for _ in range(args.warmup):
        oracle_sample(w, n_heads, stride, cores)
    total_t, total_q = 0.0, 0
    for _ in range(args.steps):
        t, q = oracle_sample(w, n_heads, stride, cores)
        total_t += t
        total_q += q
    value = total_q / total_t
    sample = "%d of %d heads, every %d-th query (%d per head), %d threads, fp64 oracle" % (
        n_heads, w.BH, stride, w.N // stride, cores)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "m": w.m, "k": w.k, "s": w.s},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


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
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed steps
    if args.sweep:
        sweep(args)
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

    mita.mita_profile_begin(12 * args.steps + 16)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n0 = mita.mita_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        mita.mita_forward(p, Q, K, V, O, ws)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    launches = mita.mita_launch_count() - n0
    clk = clocks.stop()
    phases = mita.mita_profile_end()
    mita.mita_device_status(ws)
    ms_step = job_max(dist, e0.elapsed_time(e1) / args.steps)
    value = world * w.BH * w.N / (ms_step * 1e-3)

    pk, pk_src = peaks()
    F, Bytes, expert_F = work_counts(w)
    tensor_peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    t_roof = max(F / (pk["bf16_tflops"] * 1e12), Bytes / (pk["hbm_gbs"] * 1e9))
    phase_ms = {k: v / args.steps for k, v in phases.items()}
    uses_tc = mita.mita_uses_tensor_cores(p) == 1
    dom = "expert" if "expert" in phase_ms else max(phase_ms, key=phase_ms.get)
    dom_ms = phase_ms[dom]
    achieved = expert_F / (dom_ms * 1e-3) / 1e12
    kname = "k_expert_res (expert attention)" if "merge" in phase_ms else "k_expert_ws (expert attention + merge)"
    roof = {"kernel": kname if dom == "expert" else dom,
            "bound": "tensor", "achieved": achieved, "peak": tensor_peak, "unit": "TFLOP/s",
            "frac": achieved / tensor_peak,
            "traffic": EXPERT_TRAFFIC_BYTES if (dom == "expert" and w.name == "longctx_n32k" and "merge" in phase_ms)
            else None,
            "peak_source": "%s bf16 sustained (MEASURED_PEAKS.json)" % pk_src,
            "algorithmic_flops_per_launch": expert_F, "avg_launch_ms": dom_ms}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "m": w.m, "k": w.k, "s": w.s,
                       "path": "tcgen05" if uses_tc else "cuda-core", "l2": "inputs larger than L2 (no flush)",
                       "parallelism": "replicas x%d" % world},
            "roofline": roof,
            "path_roofline": {"t_roof_us": t_roof * 1e6, "frac": t_roof / (ms_step * 1e-3),
                              "flops": F, "compulsory_bytes": Bytes,
                              "peaks": {"bf16_tflops": pk["bf16_tflops"], "hbm_gbs": pk["hbm_gbs"],
                                        "source": pk_src}},
            "phases_ms": phase_ms, "gpu_launches": launches, "clocks": clk}

    if not args.no_e2e:
        line["e2e"] = e2e_run(mita, p, Qn, Kn, Vn, w, dev, min(args.steps, 10), dist, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        n_heads = min(w.BH, cores)
        t, q = oracle_sample(w, n_heads, 1, cores)
        line["cpu_baseline"] = {"value": q / t, "unit": UNIT, "cores": min(cores, n_heads), "kind": "oracle",
                                "sample": "%d of %d heads, all %d queries each, fp64 oracle, one head per thread"
                                          % (n_heads, w.BH, w.N), "seconds": t}
    if rank == 0:
        print(json.dumps(line), flush=True)


def sweep(args):
    """Per configuration: step time (CUDA events over --steps steps after
    --warmup), t_roof = max(F / bf16 peak, bytes / HBM peak) and their ratio."""
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
        stream = torch.cuda.current_stream(dev)
        for _ in range(args.warmup):
            mita.mita_forward(p, Q, K, V, O, ws)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            mita.mita_forward(p, Q, K, V, O, ws)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        mita.mita_device_status(ws)
        ms = e0.elapsed_time(e1) / args.steps
        F, Bytes, _ = work_counts(w)
        t_f, t_b = F / (pk["bf16_tflops"] * 1e12), Bytes / (pk["hbm_gbs"] * 1e9)
        t_roof = max(t_f, t_b)
        print(json.dumps({"workload": name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "m": w.m, "k": w.k, "s": w.s,
                          "ms_per_step": ms, "value": w.BH * w.N / (ms * 1e-3), "unit": UNIT,
                          "flops": F, "compulsory_bytes": Bytes, "bound": "tensor" if t_f >= t_b else "hbm",
                          "t_roof_us": t_roof * 1e6, "frac": t_roof / (ms * 1e-3), "peaks": pk_src,
                          "path": "tcgen05" if mita.mita_uses_tensor_cores(p) == 1 else "cuda-core"}), flush=True)
        del Q, K, V, O, ws
        torch.cuda.empty_cache()


def e2e_run(mita, p, Qn, Kn, Vn, w, dev, steps, dist, world):
    """The same metric through mita_forward_host: pinned host buffers, copies
    in, forward, copy out, all inside the timed region."""
    import numpy as np
    import torch
    hb = [torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8)).pin_memory() for a in (Qn, Kn, Vn)]
    hO = torch.empty_like(hb[0]).pin_memory()
    buf = torch.empty(mita.mita_host_buffer_size(p), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):
        mita.mita_forward_host(p, hb[0], hb[1], hb[2], hO, buf)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        mita.mita_forward_host(p, hb[0], hb[1], hb[2], hO, buf)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = job_max(dist, e0.elapsed_time(e1) / steps)
    nbytes = hb[0].numel()
    return {"value": world * w.BH * w.N / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": 3 * nbytes,
            "d2h_bytes_per_step": nbytes, "ms_per_step": ms, "steps": steps}


if __name__ == "__main__":
    main()
