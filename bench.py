"""Benchmark of the GB300 fused MoE expert layer.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one full layer forward (routing, permutation + activation
quantisation, GEMM1 + SwiGLU + requantisation, GEMM2, combine) over one batch
of synthetic tokens, through the library's C ABI.  Inputs are resident in HBM
when the timed region starts; the timed region is bracketed by a barrier and
torch.cuda.synchronize() on both sides and timed with CUDA events on the
launching stream.  Every step streams the weights of all touched experts
(larger than the 129 MB L2 for every workload), so no L2 flush is needed.

Multi-GPU: the layer does not shard (one GPU, no collectives), so N GPUs run
N independent replicas under torchrun (replicas only); value is the total
tokens of all ranks over the slowest rank's time.

--impl reference times the CPU oracle (the only reference implementation this
project has) on the host cores, each step a bounded sample of the workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

# The largest single-GPU configuration, the one the metric's prefill
# fraction is about: NVFP4, T=8192, H=7168, I=2048, E=384, top-8, Zipf(1.1)
# expert popularity.  The other workloads run with --workload.
DEFAULT_WORKLOAD = "nvfp4_prefill"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=0, help="0: enough for ~3 s of timed work")
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--tokens", type=int, default=0, help="override T (decode sweep)")
    p.add_argument("--experts", type=int, default=0,
                   help="override E (small cases for profiler captures)")
    p.add_argument("--act", default="", choices=["", "swiglu", "relu2"],
                   help="expert activation (default: the workload's; relu2 drops the clamp)")
    p.add_argument("--combine", default="gather", choices=["gather", "reduce", "fused"],
                   help="sum of the K expert outputs: combine kernel (deterministic), "
                        "in-kernel atomic reduce, or the deterministic gather fused into "
                        "GEMM2's epilogue")
    p.add_argument("--max-ctas", type=int, default=0,
                   help="cap on the CTAs of each GEMM launch (0: one per SM)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


def workload_spec(args):
    s = workloads.spec(args.workload)
    if args.tokens:
        s["T"] = args.tokens
    if args.experts:
        s["E"] = args.experts
    s["combine"] = args.combine
    if args.act:
        s["act"] = args.act
        if args.act == "relu2":
            s["clamp"] = 0.0
    return s


def describe(s):
    return "%s: T=%d H=%d I=%d E=%d top-%d %s %s%s, logits %s%s" % (
        s["name"], s["T"], s["H"], s["I"], s["E"], s["K"], s["fmt"], s.get("act", "swiglu"),
        (", clamp %g" % s["clamp"]) if s["clamp"] else "", s["logits"],
        {"reduce": ", in-kernel reduce", "fused": ", combine fused into GEMM2"}.get(
            s.get("combine"), ""))


def dtype_of(s):
    return {"bf16": "bf16", "mxfp8": "e4m3 (mxfp8)", "nvfp4": "e2m1 (nvfp4)"}[s["fmt"]]


NOMINAL_DENSE_TFLOPS = {"bf16": 2250.0, "mxfp8": 4500.0, "nvfp4": 13500.0}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- roofline
def algorithmic_bytes(s, counts):
    """Bytes one launch of each GEMM must move at least: the touched experts'
    weights (codes + block scales) once, its activation input and its output.
    Returns dict kernel -> bytes, and the number of touched experts."""
    H, I, fmt = s["H"], s["I"], s["fmt"]
    touched = int((counts > 0).sum())
    R = int(counts.sum())
    if fmt == "nvfp4":
        wb = lambda n, k: n * k // 2 + n * k // 16          # noqa: E731
        ab = lambda k: k // 2 + k // 16                     # noqa: E731
    elif fmt == "mxfp8":
        wb = lambda n, k: n * k + n * k // 32               # noqa: E731
        ab = lambda k: k + k // 32                          # noqa: E731
    else:
        wb = lambda n, k: 2 * n * k                         # noqa: E731
        ab = lambda k: 2 * k                                # noqa: E731
    g1 = touched * wb(workloads.w13_rows(s), H) + R * ab(H) + R * ab(I)
    g2 = touched * wb(H, I) + R * ab(I) + R * 2 * H
    return {"gemm1_swiglu": g1, "gemm2": g2}, touched


def source_digest(path):
    """SHA-1 of a C++/CUDA source with comments and whitespace removed, so
    that edits of comments alone do not mark a capture as stale."""
    import hashlib
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha1(" ".join(text.split()).encode()).hexdigest()


def ncu_traffic(s, touched, kernel, alg_bytes):
    """DRAM bytes per launch of `kernel` from the committed ncu captures
    (profiles/gemm_traffic.json), scaled from the captured case to this run:
    by the number of touched experts where every expert's weights are read
    once (decode, bf16: the weights dominate the traffic), or by the
    algorithmic bytes where the captured case is a reduced-E prefill whose
    experts span several chunks (traffic / algorithmic bytes of the capture
    times this run's algorithmic bytes).  None when the workload was not
    captured or the kernel sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    try:
        tab = json.load(open(path))
        for src, digest in tab["sources_sha1"].items():
            if source_digest(os.path.join(ROOT, src)) != digest:
                return None, "kernel changed since the ncu capture"
        name = s["name"]
        per = tab.get("per_touched_expert_bytes", {}).get(name, {}).get(kernel)
        if per is not None:
            return int(per * touched), "ncu capture: " + tab["captures"][name] + \
                ", scaled by touched experts"
        ratio = tab["traffic_per_algorithmic_byte"][name][kernel]
    except (OSError, KeyError, ValueError):
        return None, "no ncu capture for this workload and kernel"
    return int(ratio * alg_bytes), "ncu capture: " + tab["captures"][name] + \
        ", DRAM bytes per algorithmic byte of that case times this run's algorithmic bytes"


# ---------------------------------------------------------------- ranks
def rank_env():
    """(world, rank, local_rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(x, device="cpu"):
    """The largest value of x over all ranks (x itself on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, slowest_seconds):
    """Replicas: every rank processes the same units; the job's rate is the
    units of all ranks over the slowest rank's time."""
    return units_per_rank * world / slowest_seconds


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import moe_expert_layer_histogram_gb300 as moe

    world, rank, local = rank_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    s = workload_spec(args)
    T = s["T"]

    case = workloads.make_case(s, seed=0, device=dev)
    layer = moe.MoELayer(T, s["H"], s["I"], s["E"], s["K"], s["fmt"], s["clamp"], s["act"],
                         s["combine"], max_ctas=args.max_ctas)
    layer.prepare_weights(case["weights"])
    torch.cuda.synchronize()
    gemm_ctas = moe.moe_gemm_ctas(layer.handle, T > 1024)
    w_sample = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle's bounded sample: the first n tokens of this very
        # workload and the experts they touch, copied off the device
        import oracle
        n = cpu_sample_tokens(s)
        ids, _ = oracle.route(case["logits"][:n].cpu().numpy(), s["K"])
        w_sample = (n, workloads.host_weights(s, ids.reshape(-1), source=case["weights"]))
    del case["weights"]
    torch.cuda.empty_cache()
    hidden, logits = case["hidden"], case["logits"]
    out = torch.empty_like(hidden)
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 3)):
        layer.forward(hidden, logits, out=out)
    torch.cuda.synchronize()
    _, _, off, _ = layer.routing()
    counts = np.diff(off.cpu().numpy())
    st = layer.status()
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)

    # step count: ~3 s of timed work unless given
    t0 = time.perf_counter()
    for _ in range(5):
        layer.forward(hidden, logits, out=out)
    torch.cuda.synchronize()
    per = (time.perf_counter() - t0) / 5
    steps = args.steps or int(min(20000, max(20, 3.0 / max(per, 1e-6))))

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        moe.moe_forward(layer.handle, hidden, logits, out, T, stream.cuda_stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop()
    launches = moe.moe_last_launch_count(layer.handle) * steps
    st = layer.status()
    if st != 0:
        raise RuntimeError("device status %d after timed region" % st)
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    value = whole_job_rate(T * steps, world, elapsed_ms / 1e3)

    # per-kernel durations: a second timed pass with CUDA events recorded
    # around every kernel (kept out of the pass above: events between kernels
    # also stop consecutive kernels from overlapping their launch)
    prof_steps = min(steps, 2000)
    moe.moe_timing_start(layer.handle, prof_steps)
    torch.cuda.synchronize()
    for _ in range(prof_steps):
        moe.moe_forward(layer.handle, hidden, logits, out, T, stream.cuda_stream)
    torch.cuda.synchronize()
    kern_ms, nrec = moe.moe_timing_stop(layer.handle)

    # roofline of the dominant kernel (decode batches run both GEMMs in one
    # launch, timed in the GEMM1 slot: its bytes are both GEMMs')
    alg, touched = algorithmic_bytes(s, counts)
    nlaunch = moe.moe_last_launch_count(layer.handle)
    if nlaunch == 1:
        # decode batches: the whole layer in one kernel (timed in the GEMM1
        # slot); its bytes are both GEMMs'
        alg["decode_layer"] = alg["gemm1_swiglu"] + alg["gemm2"]
        kern_ms["decode_layer"] = kern_ms["gemm1_swiglu"]
        dom = "decode_layer"
    elif nlaunch == 3:
        alg["gemm1_gemm2_fused"] = alg["gemm1_swiglu"] + alg["gemm2"]
        kern_ms["gemm1_gemm2_fused"] = kern_ms["gemm1_swiglu"]
        dom = "gemm1_gemm2_fused"
    else:
        dom = max(("gemm1_swiglu", "gemm2"), key=lambda k: kern_ms[k])
    avg_ms = kern_ms[dom] / max(nrec, 1)
    peak, peak_src = measured_peaks()
    achieved = alg[dom] / (avg_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
            "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": None, "algorithmic_bytes": alg[dom], "avg_launch_us": round(avg_ms * 1e3, 2)}
    kern_ms.pop("gemm1_gemm2_fused", None)
    if kern_ms.pop("decode_layer", None) is not None:
        kern_ms = {"decode_layer": kern_ms["gemm1_swiglu"]}
    roof["traffic"], roof["traffic_source"] = ncu_traffic(s, touched, dom, alg[dom])
    roof["frac_of_8tbs"] = round(achieved / 8000.0, 4)
    layer_bytes = alg["gemm1_swiglu"] + alg["gemm2"]
    ms_step = elapsed_ms / steps

    # the tensor-pipe side: the layer's FLOPs against this GPU's measured
    # rate for the format's MMA kind (tcgen05 microbenchmark in the library)
    flops = 2.0 * int(counts.sum()) * s["H"] * (workloads.w13_rows(s) + s["I"])
    mma_peak = moe.moe_measure_mma_rate(s["fmt"], 256, iters=8000)
    tensor = {"flops_per_step": flops,
              "achieved_tflops": round(flops / (ms_step / 1e3) / 1e12, 1),
              "peak_tflops": round(mma_peak, 1),
              "peak_source": "measured: tcgen05.mma %s 128x256 loop on smem-resident operands"
                             % s["fmt"],
              "frac": round(flops / (ms_step / 1e3) / 1e12 / mma_peak, 4)}
    binding_ms = max(layer_bytes / (peak * 1e9), flops / (mma_peak * 1e12)) * 1e3
    tensor["binding_roofline_frac"] = round(binding_ms / ms_step, 4)
    # the same FLOPs against the nominal dense rate of the format (GB300:
    # 2.25 PFLOP/s BF16, 4.5 FP8, 13.5 FP4), which single-CTA 128 x 256 MMAs
    # do not reach; the measured loop above is what this kernel's MMAs can do
    nominal = NOMINAL_DENSE_TFLOPS[s["fmt"]]
    tensor["nominal_tflops"] = nominal
    tensor["frac_of_nominal"] = round(flops / (ms_step / 1e3) / 1e12 / nominal, 4)

    # the same forward captured once in a CUDA graph and replayed
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            moe.moe_forward(layer.handle, hidden, logits, out, T,
                            torch.cuda.current_stream().cuda_stream)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        g_steps = max(10, min(steps, 2000))
        gs0 = torch.cuda.Event(enable_timing=True)
        gs1 = torch.cuda.Event(enable_timing=True)
        gs0.record()
        for _ in range(g_steps):
            g.replay()
        gs1.record()
        torch.cuda.synchronize()
        g_ms = gs0.elapsed_time(gs1) / g_steps
        graph = {"value": round(whole_job_rate(T, world, g_ms / 1e3), 1), "unit": "tokens/s",
                 "ms_per_step": round(g_ms, 5), "steps": g_steps}
        del g
    except Exception as exc:  # capture unsupported: report, do not fail the bench
        graph = {"error": str(exc)[:200]}
    if layer.status() != 0:
        raise RuntimeError("device status %d after graph replay" % layer.status())

    # end to end: host buffers through the C ABI, every step's copies inside
    # the timed region.  moe_forward_host_async pipelines consecutive steps
    # (step i+1's input copy and step i-1's output copy overlap step i's
    # layer); the clock stops once the last step's output is in host memory.
    # The synchronous moe_forward_host (one step at a time) is reported too.
    e2e = None
    if not args.no_e2e:
        hid_h = hidden.cpu().pin_memory()
        lg_h = logits.cpu().pin_memory()
        out_h = torch.empty_like(hid_h).pin_memory()
        e_steps = max(10, min(steps, 2000))

        def host_loop(fn, n):
            torch.cuda.synchronize()
            barrier()
            t0 = time.perf_counter()
            for _ in range(n):
                fn(layer.handle, hid_h, lg_h, out_h, T, stream.cuda_stream)
            stream.synchronize()
            return max_over_ranks(time.perf_counter() - t0, dev)

        for fn in (moe.moe_forward_host_async, moe.moe_forward_host):
            host_loop(fn, 3)
        e_s = host_loop(moe.moe_forward_host_async, e_steps)
        sync_s = host_loop(moe.moe_forward_host, e_steps)
        if layer.status() != 0:
            raise RuntimeError("device status %d after the host-buffer steps" % layer.status())
        e2e = {"value": round(whole_job_rate(T * e_steps, world, e_s), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": T * s["H"] * 2 + T * s["E"] * 4,
               "d2h_bytes_per_step": T * s["H"] * 2,
               "ms_per_step": round(e_s / e_steps * 1e3, 4),
               "api": "moe_forward_host_async (pinned host buffers; copies on copy engines, "
                      "overlapping the neighbouring steps' layer work)",
               "synchronous": {"value": round(whole_job_rate(T * e_steps, world, sync_s), 1),
                               "ms_per_step": round(sync_s / e_steps * 1e3, 4),
                               "api": "moe_forward_host (one step at a time)"}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(s, case, w_sample)

    layer.close()
    if rank == 0:
        line = {
            "metric": "MoE-layer tokens/s at 1 GB300 (" + s["name"] + ")",
            "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype_of(s), "data": "synthetic (seeded; weights drawn and quantised on device)",
            "config": {"workload": describe(s), "T": T, "H": s["H"], "I": s["I"], "E": s["E"],
                       "top_k": s["K"], "format": s["fmt"], "clamp": s["clamp"],
                       "touched_experts": touched, "max_rows_per_expert": int(counts.max()),
                       "empty_experts": int((counts == 0).sum()),
                       "gemm_ctas": gemm_ctas,
                       "l2": "no flush: every step streams %.2f GB of touched-expert weights, "
                             "larger than the 129 MB L2" % (layer_bytes / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roof,
            "layer_hbm_frac": round(layer_bytes / (ms_step / 1e3) / 1e9 / peak, 4),
            "tensor": tensor,
            "graph": graph,
            "kernels_us": {k: round(v / max(nrec, 1) * 1e3, 2) for k, v in kern_ms.items()},
            "kernels_note": "per-kernel averages from a second pass of %d steps with events "
                            "around each kernel" % nrec,
            "gpu_launches": launches,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- oracle arm
def oracle_cost_core_s(s, n):
    """Rough core-seconds of one oracle forward over n tokens: the dot
    products plus decoding every touched expert's weights once."""
    E, K, H, I = s["E"], s["K"], s["H"], s["I"]
    touched = E * (1.0 - (1.0 - K / E) ** n)
    dec = {"bf16": 1e-9, "mxfp8": 3e-9, "nvfp4": 4e-9}[s["fmt"]]
    return n * K * 3 * H * I * 1.2e-9 + touched * 3 * H * I * dec


def cpu_sample_tokens(s, core_seconds=20.0):
    """Tokens of the workload the oracle runs for its bounded sample (about
    10-30 s of CPU work on the host cores)."""
    n = 1
    while n < s["T"] and oracle_cost_core_s(s, n + 1) <= core_seconds:
        n += 1
    return n


def _cfg(s):
    return dict(H=s["H"], I=s["I"], E=s["E"], K=s["K"], fmt=s["fmt"], clamp=s["clamp"],
                act=s.get("act", "swiglu"))


def cpu_baseline(s, case, w_sample):
    import oracle
    import torch
    n, wh = w_sample
    hid = case["hidden"][:n].cpu().view(torch.int16).numpy().view("uint16")
    lg = case["logits"][:n].cpu().numpy()
    t0 = time.perf_counter()
    oracle.forward(_cfg(s), wh, hid, lg)
    dt = time.perf_counter() - t0
    return {"value": round(n / dt, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "first %d of %d tokens of the same workload and the %d experts they touch "
                      "(weights copied from the device), one oracle forward, %.1f s wall"
                      % (n, s["T"], len(set(oracle.route(lg, s["K"])[0].reshape(-1).tolist())), dt)}


def run_reference(args):
    """The oracle as it stands, timed on the host cores.  Each step is one
    oracle forward over the first n tokens of the workload, n sized so the
    whole --warmup/--steps run stays within a few minutes."""
    world, rank, _ = rank_env()
    if rank != 0:
        return
    import oracle
    import torch
    s = workload_spec(args)
    steps = args.steps or 3
    warm = args.warmup
    budget_core_s = 120.0 * oracle.num_threads() / max(1, steps + warm)
    n = max(1, min(cpu_sample_tokens(s, budget_core_s), s["T"]))
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = workloads.make_case(s, seed=0, device=dev, weights=False)
    lg = case["logits"][:n].cpu().numpy()
    hid = case["hidden"][:n].cpu().view(torch.int16).numpy().view("uint16")
    ids, _ = oracle.route(lg, s["K"])
    wh = workloads.host_weights(s, ids.reshape(-1), device=dev)
    for _ in range(warm):
        oracle.forward(_cfg(s), wh, hid, lg)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.forward(_cfg(s), wh, hid, lg)
    dt = time.perf_counter() - t0
    value = n * steps / dt
    line = {"impl": "reference", "metric": "MoE-layer tokens/s at 1 GB300 (" + s["name"] + ")",
            "value": round(value, 3), "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": round(dt / steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype_of(s), "data": "synthetic (seeded)",
            "config": {"workload": describe(s), "T": s["T"]},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s",
                             "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": "first %d of %d tokens per step, the experts they touch"
                                       % (n, s["T"])},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
