"""Benchmark of the VC-Attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--mode step|schedule|sweep|preproc|fill|hybrid]

Default (mode=step): the Wan2.2-shaped workload (B=1, H=40, N=75,600, d=128,
k=256).  One step = one grouping denoising step of the whole path: warm-started
k-means (1 Lloyd iteration) + stable counting sort, the fused quantizer, and
the FP8 attention with ExpCast and the V-Smooth mean restore.  The headline
metric is FP8 attention TFLOPS, 4 B H N^2 d per step divided by the step time
(the whole step is timed, so grouping and quantization count against it).
Inputs (2.3 GB) are larger than the 129 MB L2, so no flush is needed between
steps.  Under torchrun every rank runs the full workload on its own GPU (weak
scaling, no collective on the data path); the time is the max over ranks.

--mode sweep times the attention kernel alone over N = 4,096 ... 131,072
(H = 24, d = 128) for each of ExpCast / exp-then-cast and V-Smooth on / off.
--mode schedule runs 50 denoising steps of the Wan2.2 shape with the
first-quarter, 1-in-4 clustering schedule and reports the clustering share.

--mode preproc times the quantizer with the rotary transform and the Hadamard
rotation of Q/K fused in (vc_quantize_ex) against the same computation run as
the unfused chain of kernels (vc_quantize_staged), on the Wan2.2 shape with a
21 x 45 x 80 rotary grid, plus the plain quantizer for reference.

--mode fill compares the plain permutation (stable argsort of the k-means
labels) with the block-fill permutation (vc_cluster_ex): grouping time, the
relative error of the dequantized V', and the attention output against an
fp64 reference on sampled query rows.

--mode hybrid times the attention kernel with ExpCast bytes, range-adaptive
ExpCast bytes (a beta per pair of codes of the octave), exp-then-cast bytes
and the hybrid bytes (exact exponent on high-weight tiles) at several
margins, with the attention error against an fp64 reference on sampled rows.

--mode v4 compares the 8-bit and the 4-bit V residual (E2M1 with a
power-of-two scale per 32 tokens): quantizer and attention time and the
attention output against an fp64 reference on sampled query rows.

--impl reference times the CPU oracle (the only other implementation of the
method that exists) on a bounded sample of the same workload.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 attention TFLOPS at N=75,600 H=40 d=128; % of GB300 dense FP8 peak"
FP8_PER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="step", choices=["step", "schedule", "sweep", "preproc", "fill", "hybrid", "v4"])
    ap.add_argument("--expcast", type=int, default=1)
    ap.add_argument("--vsmooth", type=int, default=1)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-numa-bind", action="store_true",
                    help="allocate the pinned e2e buffers without binding to the GPU's NUMA node")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="profiling aid: run the workload with this many heads instead of its own")
    ap.add_argument("--arm", default="all", choices=["all", "plain", "fused", "unfused"],
                    help="profiling aid for --mode preproc: time only this arm")
    return ap.parse_args()


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        loaded = [s for s in sm if mx is None or s >= 0.3 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        cl = d.get("clocks_under_load") or {}
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sustained_sm_mhz": cl.get("sm_mhz_median"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sustained_sm_mhz": None,
            "source": "fallback"}


def fp8_peak_for(peaks, clocks):
    """The dense FP8 peak a tensor-bound kernel is compared with, from the
    measured bf16 GEMM peaks (x2, the nominal fp8/bf16 ratio).

    The burst figure applies when the kernel ran at full clock without the
    power cap (no sw_power_cap sample and a median SM clock within 3 % of the
    maximum); otherwise the sustained one, which the GEMM loop reached under
    the power cap.  Also returned: the fraction against the sustained figure
    and against the sustained figure scaled to the clock this kernel ran at
    (GEMM throughput per clock x the kernel's clock)."""
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    capped = "sw_power_cap" in clocks.get("reasons", [])
    full_clock = sm is not None and mx is not None and sm >= 0.97 * mx
    burst = peaks["bf16_tflops"] * FP8_PER_BF16
    sustained = peaks["bf16_tflops_sustained"] * FP8_PER_BF16
    use_burst = full_clock and not capped
    clock_matched = None
    if sm and peaks.get("sustained_sm_mhz"):
        clock_matched = sustained * sm / peaks["sustained_sm_mhz"]
    return {"peak": burst if use_burst else sustained, "which": "burst" if use_burst else "sustained",
            "burst": burst, "sustained": sustained, "clock_matched": clock_matched}


def dist_setup(args):
    """Returns (rank, world, local_rank, pg_ready)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return rank, world, local, True
    return rank, world, local, False


def max_over_ranks(x, pg_ready):
    """Max of a float over ranks (identity without a process group)."""
    if not pg_ready:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world, flops_per_rank, ms_max):
    """Whole-job TFLOPS: every rank does the same work; the slowest rank sets the time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def barrier(pg_ready):
    if pg_ready:
        import torch.distributed as dist
        dist.barrier()


def attn_flops(B, H, N, d):
    return 4.0 * B * H * N * N * d


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for name in ("vc_attn.cu", "vc_device.cuh"):
        with open(os.path.join(ROOT, "bit_fp8_attention_means_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch_full_size")


def cpu_baseline_sample(Qc, Kc, Vc, perm_h0, N, d, target_s=15.0):
    """The oracle, as it stands, on a bounded sample: attention rows of head 0."""
    import numpy as np

    import oracle
    from bit_fp8_attention_means_gb300 import inputs
    u16 = inputs.to_u16
    qz = oracle.quantize(u16(Qc), u16(Kc), u16(Vc), perm_h0, 1)
    rng = np.random.default_rng(0)
    # calibrate on a sample large enough that the per-call overhead does not dominate
    probe = np.sort(rng.choice(N, 512, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attn(qz, N, rows=probe)
    per_row = (time.perf_counter() - t0) / probe.size
    R = int(max(512, min(N, target_s / max(per_row, 1e-9))))
    rows = np.sort(rng.choice(N, R, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attn(qz, N, rows=rows)
    dt = time.perf_counter() - t0
    flops = 4.0 * R * N * d
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "oracle attention (ExpCast, V-Smooth) on %d random query rows of head 0 against all "
                      "%d keys, inputs quantized by the oracle from the same bf16 tensors; %.1f s" % (R, N, dt)}


def run_ours(args):
    import torch

    from bit_fp8_attention_means_gb300 import inputs, schedule, vc
    rank, world, local, pg = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = inputs.WORKLOADS["wan"]
    B, H, N, d, k = w.B, (args.heads or w.H), w.N, w.d, w.k
    warm_iters = 1
    ec, vs = args.expcast, args.vsmooth
    Q, K, V = inputs.make_qkv(w, dev, seed=w.seed + rank, H=H)
    state = schedule.GroupingState()
    qz, O = schedule.run_step(state, Q, K, V, 0, 1, k, w.iters, warm_iters, expcast=ec, vsmooth=vs,
                              force_cluster=True)
    stream = torch.cuda.current_stream()

    def step(times):
        nonlocal qz, O
        qz, O = schedule.run_step(state, Q, K, V, 1, 1, k, w.iters, warm_iters, qz=qz, O=O, expcast=ec,
                                  vsmooth=vs, times=times, force_cluster=True)

    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    barrier(pg)
    times = schedule.StepTimes()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step(times)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(pg)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, pg)
    schedule.collect(times)
    attn_ms = statistics.mean(times.attn_ms)
    flops = attn_flops(B, H, N, d)
    peaks = measured_peaks()
    clocks = clk.summary()
    pk = fp8_peak_for(peaks, clocks)
    fp8_peak = pk["peak"]
    achieved = flops / (attn_ms * 1e-3) / 1e12
    # k-means iteration: assignment, histogram, scan, scatter, update (5 kernels;
    # k <= 256 takes the tensor-core assignment, which needs no norm kernel)
    launches_per_step = (5 * warm_iters if vs else 0) + 3 + 1
    result = {
        "metric": METRIC,
        "value": weak_scaling_value(world, flops, ms_max),
        "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
        "data": "synthetic: seeded Wan2.2-shaped Q/K/V (Q,K ~ N(0,1) + per-channel bias N(0,2); V a 256-centroid "
                "mixture with 1% outlier tokens x20)",
        "config": {"workload": "wan2.2-shaped B=%d H=%d N=%d d=%d, k=%d" % (B, H, N, d, k),
                   "step": "grouping step: k-means (warm, %d iteration) + stable sort + fused quantizer + FP8 "
                           "attention (expcast=%d, vsmooth=%d)" % (warm_iters, ec, vs),
                   "expcast": ec, "vsmooth": vs, "l2": "inputs 2.3 GB > 129 MB L2; no flush needed",
                   "parallelism": "replicas x%d (weak scaling, no collective on the data path)" % world},
        "attn_tflops": achieved,
        "pct_fp8_peak": 100.0 * achieved / fp8_peak,
        "pct_fp8_nominal": 100.0 * achieved / 4500.0,
        "breakdown_ms": {"cluster": statistics.mean(times.cluster_ms), "quantize": statistics.mean(times.quantize_ms),
                         "attn": attn_ms},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp8_peak, "traffic": ncu_traffic("attn_fwd_kernel"),
                     "kernel": "attn_fwd_kernel<128,expcast,vsmooth>",
                     "peak_which": pk["which"],
                     "peak_source": "%s bf16 %s %.1f TFLOP/s x %.0f (nominal fp8/bf16 ratio); burst applies when "
                                    "the timed region ran at full clock with no power cap"
                                    % (peaks["source"], pk["which"], fp8_peak / FP8_PER_BF16, FP8_PER_BF16),
                     "frac_vs_sustained": achieved / pk["sustained"],
                     "frac_vs_clock_matched": (achieved / pk["clock_matched"]) if pk["clock_matched"] else None},
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
    }
    if not args.no_e2e:
        def run_on(Qd, Kd, Vd, Od):
            nonlocal qz
            qz, Onew = schedule.run_step(state, Qd, Kd, Vd, 1, 1, k, w.iters, warm_iters, qz=qz, O=Od, expcast=ec,
                                         vsmooth=vs, force_cluster=True)
            return Onew

        result["e2e"] = e2e_run(args, Q, K, V, run_on)
    if rank == 0 and world == 1 and not args.no_cpu:
        Qc, Kc, Vc = (t[:, :, :1].cpu() for t in (Q, K, V))
        result["cpu_baseline"] = cpu_baseline_sample(Qc, Kc, Vc, state.perm[:, :1].cpu().numpy(), N, d)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if pg:
        import torch.distributed as dist
        dist.destroy_process_group()


def _cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        lo, _, hi = part.partition("-")
        cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def gpu_host_node(dev_index):
    """NUMA node of the host CPUs attached to the GPU (sysfs, via its PCI address),
    or None.  On Grace machines the GPU's own memory shows up as further nodes
    without CPUs; only a node with CPUs is returned."""
    import torch
    props = torch.cuda.get_device_properties(dev_index)
    try:
        addr = "%04x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        with open("/sys/bus/pci/devices/%s/numa_node" % addr) as f:
            node = int(f.read())
        with open("/sys/devices/system/node/node%d/cpulist" % node) as f:
            cpus = _cpulist(f.read())
    except (AttributeError, OSError, ValueError):
        return None, set()
    return (node, cpus) if node >= 0 and cpus else (None, set())


def pinned_pages_nodes(ptr):
    """Host NUMA nodes holding the pages of the mapping that contains ptr, from
    /proc/self/numa_maps ({node: pages}), or None if the kernel does not say."""
    try:
        with open("/proc/self/maps") as f:
            start = next(int(a, 16) for a, b in (ln.split()[0].split("-") for ln in f)
                         if int(a, 16) <= ptr < int(b, 16))
        with open("/proc/self/numa_maps") as f:
            for ln in f:
                fields = ln.split()
                if int(fields[0], 16) == start:
                    out = {int(k[1:]): int(v) for k, v in (x.split("=") for x in fields if x[:1] == "N" and "=" in x)}
                    return out or None
    except (OSError, StopIteration, ValueError):
        return None
    return None


def e2e_run(args, Q, K, V, run_on):
    """Same metric through the public API with host buffers, pipelined the way a
    serving loop would run it: every step copies its Q/K/V from pinned host
    memory (2.32 GB) and reads its O back (0.77 GB) on a copy stream, the H2D
    of step i+1 and the D2H of step i overlapping the compute of step i
    (two device buffer sets).  The timed region runs from before the first
    H2D to after the last D2H.  run_on(Qd, Kd, Vd, Od) launches one step on
    the current stream and returns its O."""
    import torch
    n_steps = max(2, args.steps)
    # pinned buffers on the host memory next to the GPU: allocate them from the
    # CPUs of the GPU's NUMA node (first touch places the pages there)
    node, cpus = gpu_host_node(Q.device.index or 0)
    allowed = os.sched_getaffinity(0)
    bound = bool(cpus & allowed) and not args.no_numa_bind
    if bound:
        os.sched_setaffinity(0, cpus & allowed)
    try:
        hQ, hK, hV = (t.cpu().pin_memory() for t in (Q, K, V))
        hO = [torch.empty(Q.shape, dtype=Q.dtype).pin_memory() for _ in range(2)]
    finally:
        if bound:
            os.sched_setaffinity(0, allowed)
    host_numa = {"gpu_node": node, "bound": bound, "pages_of_Q": pinned_pages_nodes(hQ.data_ptr()),
                 "pages_of_O": pinned_pages_nodes(hO[0].data_ptr())}
    bufs = [(Q, K, V, torch.empty_like(Q)), tuple(torch.empty_like(t) for t in (Q, K, V, Q))]
    comp = torch.cuda.current_stream()
    cp = torch.cuda.Stream()     # host -> device
    cp_out = torch.cuda.Stream()  # device -> host (the link is full duplex)
    ev = lambda: torch.cuda.Event()
    ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def h2d(b):
        with torch.cuda.stream(cp):
            cp.wait_event(ev_done[b])  # the step that last read buffer set b has finished
            for dst, src in zip(bufs[b][:3], (hQ, hK, hV)):
                dst.copy_(src, non_blocking=True)
            ev_in[b].record(cp)

    def d2h(b, O):
        with torch.cuda.stream(cp_out):
            cp_out.wait_event(ev_done[b])
            hO[b].copy_(O, non_blocking=True)
            ev_out[b].record(cp_out)

    def run(steps, e0=None):
        if e0 is not None:
            cp.wait_event(e0)
            cp_out.wait_event(e0)
        for b in range(2):
            ev_done[b].record(comp)
            ev_out[b].record(comp)
        h2d(0)
        last = 0
        for i in range(steps):
            b = i % 2
            if i + 1 < steps:
                h2d(1 - b)
            comp.wait_event(ev_in[b])
            comp.wait_event(ev_out[b])  # this set's O has been read back
            O = run_on(*bufs[b])
            ev_done[b].record(comp)
            d2h(b, O)
            last = b
        comp.wait_event(ev_out[last])
        comp.wait_event(ev_out[1 - last])

    run(2)
    torch.cuda.synchronize()
    # the link's own speed, for the record: one H2D of the inputs, one D2H of O
    t0, t1, t2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    t0.record(comp)
    for dst, src in zip(bufs[0][:3], (hQ, hK, hV)):
        dst.copy_(src, non_blocking=True)
    t1.record(comp)
    hO[0].copy_(bufs[0][3], non_blocking=True)
    t2.record(comp)
    torch.cuda.synchronize()
    h2d_bytes, d2h_bytes = 3 * Q.numel() * Q.element_size(), Q.numel() * Q.element_size()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    run(n_steps, e0)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_steps
    B, N, H, d = Q.shape
    return {"value": attn_flops(B, H, N, d) / (ms * 1e-3) / 1e12, "unit": "TFLOPS", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "steps": n_steps,
            "h2d_gbs": h2d_bytes / (t0.elapsed_time(t1) * 1e-3) / 1e9,
            "d2h_gbs": d2h_bytes / (t1.elapsed_time(t2) * 1e-3) / 1e9,
            "overlap": "H2D of step i+1 and D2H of step i on two copy streams during step i",
            "host_numa": host_numa}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample per step.

    Each step = oracle grouping (1 warm Lloyd iteration) + stable sort + quantizer
    for head 0 of the Wan2.2-shaped workload, then oracle attention on R query
    rows of that head against all N keys; the metric credits the attention
    FLOPs of those rows (4 R N d) per step time.
    """
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    from bit_fp8_attention_means_gb300 import inputs
    w = inputs.WORKLOADS["wan"]
    N, d, k = w.N, w.d, w.k
    Q, K, V = inputs.make_qkv(w, "cpu", H=1)
    q, kk, v = (inputs.to_u16(t) for t in (Q, K, V))
    cent, lab = oracle.kmeans(v, k, 1)                      # setup: a first (cold) clustering
    rng = np.random.default_rng(0)
    R = 64
    rows = np.sort(rng.choice(N, R, replace=False)).astype(np.int32)

    def step():
        nonlocal cent
        cent, lab = oracle.kmeans(v, k, 1, centroids=cent)
        perm = oracle.argsort_labels(lab, k)
        qz = oracle.quantize(q, kk, v, perm, 1)
        oracle.attn(qz, N, rows=rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    val = 4.0 * R * N * d / dt / 1e12
    sample = ("per step: oracle k-means (1 warm Lloyd iteration, k=%d) + argsort + quantizer on head 0 of the "
              "Wan2.2-shaped workload (N=%d, d=%d), then oracle attention on %d query rows against all keys; "
              "credited FLOPs = 4*R*N*d" % (k, N, d, R))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle; fp32 where codes are decided)",
        "data": "synthetic: seeded Wan2.2-shaped head",
        "config": {"workload": "wan2.2-shaped B=%d H=%d N=%d d=%d, k=%d" % (w.B, w.H, N, d, k),
                   "step": "bounded CPU sample, see cpu_baseline.sample"},
        "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_schedule(args):
    """Amortized denoising schedule: 50 steps, clustering only where the schedule says."""
    import torch

    from bit_fp8_attention_means_gb300 import inputs, schedule
    dev = torch.device("cuda", 0)
    w = inputs.WORKLOADS["wan"]
    S = 50
    Q, K, V = inputs.make_qkv(w, dev)
    state = schedule.GroupingState()
    times = schedule.StepTimes()
    qz = O = None
    for s in range(S):
        if s > 0:
            V = inputs.drift_v(V, s, w.seed)
            Q, K, _ = inputs.make_qkv(w, dev, seed=w.seed + 100 + s, H=w.H)
        qz, O = schedule.run_step(state, Q, K, V, s, S, w.k, w.iters, 1, qz=qz, O=O, times=times)
        torch.cuda.synchronize()
        schedule.collect(times)
    tot = sum(times.cluster_ms) + sum(times.quantize_ms) + sum(times.attn_ms)
    flops = attn_flops(w.B, w.H, w.N, w.d)
    print(json.dumps({
        "mode": "schedule", "metric": METRIC, "steps": S, "clusterings": state.clusterings,
        "cluster_steps": [s for s in range(S) if schedule.clusters_at(s, S)],
        "cluster_share_of_path": sum(times.cluster_ms) / tot,
        "cluster_ms_per_grouping_step": sum(times.cluster_ms[1:]) / max(1, state.clusterings - 1),
        "cold_cluster_ms": times.cluster_ms[0],
        "quantize_ms_mean": statistics.mean(times.quantize_ms), "attn_ms_mean": statistics.mean(times.attn_ms),
        "amortized_tflops": S * flops / (tot * 1e-3) / 1e12,
        "config": {"workload": "wan2.2-shaped 50-step schedule, V drift N(0,0.05), Q/K redrawn"}}), flush=True)


def run_sweep(args):
    """Attention kernel alone, H=24, N in {4K..128K}, ExpCast x V-Smooth on/off."""
    import torch

    from bit_fp8_attention_means_gb300 import inputs, vc
    dev = torch.device("cuda", 0)
    rows = []
    for N in (4096, 16384, 32768, 65536, 131072):
        w = inputs.sweep_workload(N)
        Q, K, V = inputs.make_qkv(w, dev)
        perm = vc.vc_cluster(V, w.k, w.iters)[2]
        s = vc.shape_of(Q)
        O = torch.empty_like(Q)
        flops = attn_flops(w.B, w.H, N, w.d)
        for vs in (0, 1):
            qz = vc.vc_quantize(Q, K, V, perm if vs else None, vs)
            for ec in (0, 1):
                for _ in range(2):
                    vc.vc_attn_fwd(qz, s, expcast=ec, vsmooth=vs, O=O)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = max(2, int(2e14 // flops))
                e0.record()
                for _ in range(reps):
                    vc.vc_attn_fwd(qz, s, expcast=ec, vsmooth=vs, O=O)
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / reps
                rows.append({"N": N, "expcast": ec, "vsmooth": vs, "ms": ms, "tflops": flops / ms / 1e9})
        del Q, K, V, qz, O
        torch.cuda.empty_cache()
    print(json.dumps({"mode": "sweep", "metric": "attention kernel TFLOPS, H=24 d=128", "rows": rows}), flush=True)


def run_preproc(args):
    """Fused vs unfused preprocessing chain (rotary, gather, block means,
    Hadamard, FP8 quantization of Q/K/V) on the Wan2.2 shape."""
    import torch

    from bit_fp8_attention_means_gb300 import inputs, vc
    dev = torch.device("cuda", 0)
    w = inputs.WORKLOADS["wan"]
    H = args.heads or w.H
    Q, K, V = inputs.make_qkv(w, dev, H=H)
    perm = vc.vc_cluster(V, w.k, w.iters)[2]
    rope = torch.from_numpy(inputs.rope_table(w.N, w.d, inputs.WAN_GRID)).to(dev)
    s = vc.shape_of(Q)
    out = vc.alloc_quantized(s, dev, 1)
    ws = torch.empty(vc.quantize_workspace_bytes(s), dtype=torch.uint8, device=dev)
    ws_staged = torch.empty(vc.quantize_staged_workspace_bytes(s), dtype=torch.uint8, device=dev)
    arms = {
        "plain": lambda: vc.vc_quantize(Q, K, V, perm, 1, out=out, workspace=ws),
        "fused": lambda: vc.vc_quantize_ex(Q, K, V, perm, 1, rope=rope, hadamard=1, out=out, workspace=ws),
        "unfused": lambda: vc.vc_quantize_staged(Q, K, V, perm, 1, rope=rope, hadamard=1, out=out,
                                                 workspace=ws_staged),
    }
    if args.arm != "all":
        arms = {args.arm: arms[args.arm]}
    reps = max(3, args.steps)
    res = {}
    for name, fn in arms.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / reps
    if args.arm != "all":
        print(json.dumps({"mode": "preproc", "arm": args.arm, "ms": res[args.arm], "heads": H}), flush=True)
        return
    elems = w.B * w.N * H * w.d
    # algorithmic bytes: Q, K, V read once (bf16), codes written (E4M3), the
    # rotary table read once; scales, means and pi are < 1 %
    alg = 3 * 2 * elems + 3 * elems + rope.numel() * 4
    peak = measured_peaks()
    print(json.dumps({
        "mode": "preproc",
        "metric": "Q/K/V preprocessing chain ms (rotary + gather + block means + Hadamard + FP8 quantization)",
        "fused_ms": res["fused"], "unfused_ms": res["unfused"], "plain_quantizer_ms": res["plain"],
        "fused_speedup": res["unfused"] / res["fused"],
        "fused_gbs": alg / (res["fused"] * 1e-3) / 1e9, "algorithmic_bytes": alg,
        "hbm_peak_gbs": peak["hbm_gbs"], "peak_source": peak["source"],
        "unfused_workspace_bytes": ws_staged.numel(), "reps": reps,
        "config": {"workload": "wan2.2-shaped B=1 H=%d N=75600 d=128, rotary grid 21x45x80, k=256 pi" % H,
                   "l2": "inputs 2.3 GB > L2, no flush"}}), flush=True)


def run_fill(args):
    """Plain vs block-fill permutation on the Wan2.2 shape: grouping cost, V'
    reconstruction error, attention error against fp64 on sampled rows."""
    import torch

    from bit_fp8_attention_means_gb300 import inputs, vc
    dev = torch.device("cuda", 0)
    w = inputs.WORKLOADS["wan"]
    H = args.heads or w.H
    Q, K, V = inputs.make_qkv(w, dev, H=H)
    cent0, _, _ = vc.vc_cluster(V, w.k, w.iters)
    s = vc.shape_of(Q)
    res = {}
    g = torch.Generator(device="cpu").manual_seed(7)
    rows = torch.randperm(w.N, generator=g)[:256].to(dev)
    heads = list(range(0, H, max(1, H // 4)))[:4]
    ref = fp64_rows(Q, K, V, rows, heads, w.d)
    for fill in (0, 1):
        cent = cent0.clone()
        fn = lambda: vc.vc_cluster(V, w.k, 1, warm_start=True, centroids=cent.copy_(cent0), block_fill=fill)
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, args.steps)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        _, _, perm = fn()
        qz = vc.vc_quantize(Q, K, V, perm, 1)
        O = vc.vc_attn_fwd(qz, s)
        torch.cuda.synchronize()
        # V' reconstruction: R codes * s_v + block mean, against V gathered by pi
        Rq = qz["V8T"].view(torch.float8_e4m3fn).float() * qz["sv"][..., None]       # [B,H,d,Npad]
        mu = qz["mu"].view(torch.bfloat16).float().repeat_interleave(128, dim=2)     # [B,H,Npad,d]
        Vr = Rq.transpose(2, 3)[:, :, :w.N] + mu[:, :, :w.N]
        Vp = torch.gather(V.permute(0, 2, 1, 3).float(), 2, perm.long()[..., None].expand(-1, -1, -1, w.d))
        verr = float((Vr - Vp).norm() / Vp.norm())
        mres = float((Vp - mu[:, :, :w.N]).norm() / Vp.norm())
        oerr = [float((O[0, rows, h].double() - ref[h]).norm() / ref[h].norm()) for h in heads]
        res[fill] = {"cluster_ms": ms, "v_rel_err": verr, "residual_energy": mres ** 2,
                     "o_rel_err_vs_fp64": sum(oerr) / len(oerr)}
    print(json.dumps({
        "mode": "fill", "metric": "V' reconstruction error and attention error vs fp64, plain vs block-fill pi",
        "plain": res[0], "block_fill": res[1],
        "v_err_reduction": 1 - res[1]["v_rel_err"] / res[0]["v_rel_err"],
        "fill_overhead_ms": res[1]["cluster_ms"] - res[0]["cluster_ms"],
        "config": {"workload": "wan2.2-shaped B=1 H=%d N=75600 d=128 k=256, warm k-means step (1 iteration)" % H,
                   "sampled_rows": 256, "sampled_heads": heads}}), flush=True)


def fp64_rows(Q, K, V, rows, heads, d):
    """softmax(q K^T / sqrt d) V in fp64 (torch, on the device) for sampled rows."""
    import torch
    ref = {}
    for h in heads:
        q = Q[0, rows, h].double()
        p = torch.softmax(q @ K[0, :, h].double().T / math.sqrt(d), dim=-1)
        ref[h] = p @ V[0, :, h].double()
    return ref


def run_hybrid(args):
    """Attention with ExpCast / adaptive-beta / exp-then-cast / hybrid bytes on the Wan2.2 shape:
    kernel time and error against fp64 on sampled rows."""
    import torch

    from bit_fp8_attention_means_gb300 import inputs, vc
    dev = torch.device("cuda", 0)
    w = inputs.WORKLOADS["wan"]
    H = args.heads or w.H
    Q, K, V = inputs.make_qkv(w, dev, H=H)
    perm = vc.vc_cluster(V, w.k, w.iters)[2]
    qz = vc.vc_quantize(Q, K, V, perm, 1)
    s = vc.shape_of(Q)
    O = torch.empty_like(Q)
    g = torch.Generator(device="cpu").manual_seed(7)
    rows = torch.randperm(w.N, generator=g)[:256].to(dev)
    heads = list(range(0, H, max(1, H // 4)))[:4]
    ref = fp64_rows(Q, K, V, rows, heads, w.d)
    flops = attn_flops(w.B, H, w.N, w.d)
    arms = [("expcast", dict(expcast=1)), ("adaptive_beta", dict(expcast=3)), ("hybrid_m1", dict(exact_margin=1.0)),
            ("hybrid_m2", dict(exact_margin=2.0)), ("hybrid_m3", dict(exact_margin=3.0)),
            ("hybrid_m5", dict(exact_margin=5.0)), ("exp_then_cast", dict(expcast=0))]
    out = []
    for name, kw in arms:
        fn = lambda: vc.vc_attn_fwd(qz, s, O=O, **kw)
        for _ in range(max(2, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, args.steps)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        err = [float((O[0, rows, h].double() - ref[h]).norm() / ref[h].norm()) for h in heads]
        out.append({"arm": name, **{k: v for k, v in kw.items()}, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                    "o_rel_err_vs_fp64": sum(err) / len(err)})
    print(json.dumps({"mode": "hybrid", "metric": "attention kernel ms and O error vs fp64 per probability-byte mode",
                      "rows": out,
                      "config": {"workload": "wan2.2-shaped B=1 H=%d N=75600 d=128, vsmooth=1, k=256 pi" % H,
                                 "sampled_rows": 256, "sampled_heads": heads}}), flush=True)


def run_v4(args):
    """8-bit against 4-bit V residual on the Wan2.2 shape: quantizer and attention
    time (CUDA events) and O against fp64 on sampled rows, V-Smooth on."""
    import torch

    from bit_fp8_attention_means_gb300 import inputs, vc
    dev = torch.device("cuda", 0)
    w = inputs.WORKLOADS["wan"]
    H = args.heads or w.H
    Q, K, V = inputs.make_qkv(w, dev, H=H)
    perm = vc.vc_cluster(V, w.k, w.iters)[2]
    s = vc.shape_of(Q)
    O = torch.empty_like(Q)
    g = torch.Generator(device="cpu").manual_seed(7)
    rows = torch.randperm(w.N, generator=g)[:256].to(dev)
    heads = list(range(0, H, max(1, H // 4)))[:4]
    ref = fp64_rows(Q, K, V, rows, heads, w.d)
    flops = attn_flops(w.B, H, w.N, w.d)
    out = []
    for vbits in (8, 4):
        qz = vc.vc_quantize(Q, K, V, perm, 1, vbits=vbits)

        def timed(fn):
            for _ in range(max(2, args.warmup)):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(3, args.steps)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        q_ms = timed(lambda: vc.vc_quantize(Q, K, V, perm, 1, out=qz, vbits=vbits))
        a_ms = timed(lambda: vc.vc_attn_fwd(qz, s, O=O))
        err = [float((O[0, rows, h].double() - ref[h]).norm() / ref[h].norm()) for h in heads]
        out.append({"vbits": vbits, "quantize_ms": q_ms, "attn_ms": a_ms,
                    "attn_tflops": flops / (a_ms * 1e-3) / 1e12, "o_rel_err_vs_fp64": sum(err) / len(err),
                    "v_bytes_4bit_packed": (w.B * H * w.d * vc.nblk_of(w.N) * 128) // 2 if vbits == 4 else None})
    print(json.dumps({"mode": "v4", "metric": "quantizer and attention ms, O error vs fp64: 8-bit vs 4-bit V residual",
                      "rows": out,
                      "config": {"workload": "wan2.2-shaped B=1 H=%d N=75600 d=128, vsmooth=1, k=256 pi" % H,
                                 "sampled_rows": 256, "sampled_heads": heads}}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.mode == "step":
        run_ours(args)
    elif args.mode == "schedule":
        run_schedule(args)
    elif args.mode == "preproc":
        run_preproc(args)
    elif args.mode == "fill":
        run_fill(args)
    elif args.mode == "hybrid":
        run_hybrid(args)
    elif args.mode == "v4":
        run_v4(args)
    else:
        run_sweep(args)


if __name__ == "__main__":
    main()
