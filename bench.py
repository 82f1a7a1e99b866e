"""Benchmark of the GB300 GPTQ GEMM library; prints ONE JSON line (rank 0).

Workload (the headline): Llama-7B-shaped decode GEMV, A fp16 [1, 4096] x W [4096, 11008] 4-bit,
group 128, GPTQv2 -- metric "M=1 decode weight GB/s" with algorithmic bytes = qweight + scales +
qzeros + A.  One step = one gptq_gemm launch on one batch (M = 1 token).  Steps run as CUDA-graph
replays over S rotating copies of the weights whose total size is more than 3x the L2 cache, so
every step reads its weights from HBM.  The same line carries the secondary figure of the
metric (M = 4096 prefill TFLOP/s, A bf16 [4096, 4096] x W [4096, 14336] 4-bit g128) and a
per-configuration section: every one of the five workload configurations at its exact shape
(decode at each of its token counts, act-order through gptq_gemm and prepacked, the three
prefill variants), the standalone dequant and the mixture-of-experts layer, each timed as the
median of 10 graph replays (a first replay discarded) with its roofline fraction.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, one thread) on the host cores, each step a
bounded column sample of the same workload.  Under torchrun (N > 1) every rank runs its own
replica on its own GPU (the path has no exchange step); rank 0 prints the aggregate.
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gptq_inputs  # noqa: E402

DECODE = gptq_inputs.WORKLOADS["llama7b_decode_4bit_g128"]
PREFILL = gptq_inputs.WORKLOADS["prefill_4bit_g128"]
METRIC = "M=1 decode weight GB/s (% of 8 TB/s HBM); M=4096 prefill TFLOP/s (% peak)"
L2_BYTES_FALLBACK = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def algorithmic_bytes(wl, M):
    """qweight + scales + qzeros + A (+ g_idx): every byte the GEMM must read once."""
    qweight = wl.K * wl.bits // 32 * wl.N * 4
    scales = wl.G * wl.N * 2
    qzeros = wl.G * (wl.N * wl.bits // 32) * 4
    acts = M * wl.K * 2
    gidx = wl.K * 4 if wl.act_order else 0
    return qweight + scales + qzeros + acts + gidx


def grouped_bytes(mw, offsets):
    """Mixture of experts: every expert that holds rows reads its whole weight (qweight, scales,
    qzeros) once; plus the grouped activations and the offsets."""
    active = int(np.count_nonzero(np.diff(offsets)))
    per_expert = (mw.K * mw.bits // 32 * mw.N * 4 + mw.G * mw.N * 2 + mw.G * (mw.N * mw.bits // 32) * 4)
    return active * per_expert + int(offsets[-1]) * mw.K * 2 + (mw.E + 1) * 4, active


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


def load_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    source of the kernel (matching hash); otherwise None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        entry = t[kernel_key]
        h = hashlib.sha256()
        for rel in entry["sources"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != entry["source_hash"]:
            return None
        return float(entry["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        window = "timed"
        sel = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        if not sel:
            sel, window = rows, "warmup+timed"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "unavailable"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": float(np.median([r[1] for r in sel])), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel), "window": window}


# ------------------------------------------------------------------------------------ host
def host_info():
    """Core count and CPU model of the host the CPU legs run on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model, "machine": platform.machine()}


# ------------------------------------------------------------------------------------ ranks
def max_over_ranks(x, dist, device):
    """The largest value of x over all ranks (x itself on one rank)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, bytes_per_step, steps, seconds):
    """Throughput of the whole job: every rank processed `steps` steps of `bytes_per_step`
    (weak scaling: per-rank work is fixed), timed by the slowest rank."""
    return world * bytes_per_step * steps / seconds / 1e9


# ------------------------------------------------------------------------------------ timing
def replay_median(torch, stream, graph, launches, replays=11):
    """Per-launch time of a captured graph of `launches` launches: `replays` replays, each timed
    with CUDA events on the launching stream; the first is discarded and the median of the rest
    is returned (ms per launch), with the spread (min, max) of those replays."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
    with torch.cuda.stream(stream):
        for st, en in evs:
            st.record(stream)
            graph.replay()
            en.record(stream)
    stream.synchronize()
    ms = [st.elapsed_time(en) / launches for st, en in evs[1:]]
    return float(np.median(ms)), float(min(ms)), float(max(ms))


def capture(torch, stream, launch, n):
    """Run `launch(i)` for i < n once (kernel attributes are set outside capture), then capture n
    launches in one CUDA graph."""
    with torch.cuda.stream(stream):
        for i in range(n):
            launch(i)
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for i in range(n):
            launch(i)
    return gr


def roofline(achieved, peak, unit, bound, source, traffic=None):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": source}


# ------------------------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import gptq_bit_weight_gemm_gb300 as g
    from gptq_bit_weight_gemm_gb300 import build as lib_build

    lib_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK
    peaks = load_peaks()
    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    uuid = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(local_rank)
    sampler = ClockSampler(uuid)

    # ---- inputs: seeded draws -> device -> GPU round-to-nearest checkpoint writer
    wl, M = DECODE, 1
    draw = gptq_inputs.draw_weights(wl)
    W = torch.from_numpy(draw.W).to(dev)
    qw, qz, sc = g.quantize_rtn(W, bits=wl.bits, group=wl.group, fmt=g.V2)
    del W
    A = gptq_inputs.draw_activations(wl, M).to(dev)
    set_bytes = algorithmic_bytes(wl, M)
    S = max(2, int(np.ceil(3 * l2 / set_bytes)))
    sets = [(qw.clone(), qz.clone(), sc.clone(), A.clone(), torch.empty((M, wl.N), dtype=A.dtype, device=dev))
            for _ in range(S)]
    torch.cuda.synchronize()

    def launch(i):
        q, z, s, a, c = sets[i % S]
        g.gemm(a, q, z, s, bits=wl.bits, group=wl.group, fmt=g.V2, out=c, stream=stream)

    # ---- CUDA graphs of R launches (and one of the remainder) replayed for exact step counts
    R = S * max(1, 256 // S)
    main_graph = capture(torch, stream, launch, R)
    rem_graphs = {}
    for n in (args.warmup, args.steps):   # every graph is captured before anything is timed
        if n % R and n % R not in rem_graphs:
            rem_graphs[n % R] = capture(torch, stream, launch, n % R)

    def run_steps(n):
        for _ in range(n // R):
            main_graph.replay()
        if n % R:
            rem_graphs[n % R].replay()

    # kernel figure the replay way: median of 10 replays of R launches (first replay discarded),
    # and one launch on its own
    med_ms, min_ms, max_ms = replay_median(torch, stream, main_graph, R)
    single = []
    with torch.cuda.stream(stream):
        for i in range(12):
            st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            st.record(stream)
            launch(i)
            en.record(stream)
            stream.synchronize()
            single.append(st.elapsed_time(en))
    single_ms = float(np.median(single[2:]))

    with torch.cuda.stream(stream):
        run_steps(args.warmup)
    stream.synchronize()
    # clock window: the timed region of a short run lasts well under the sampler's 100 ms period,
    # so the same graph keeps the GPU busy for about a second right before it
    tc0 = time.time()
    with torch.cuda.stream(stream):
        while time.time() - tc0 < 1.2:
            main_graph.replay()
            stream.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        # a short GPU sleep queued ahead of the start event: the graph launches are enqueued while
        # it runs, so the timed region holds the K steps back to back and no host launch latency
        torch.cuda._sleep(200000)
        start.record(stream)
        run_steps(args.steps)
        end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    ms_total = max_over_ranks(start.elapsed_time(end), dist, dev)
    ms_per_step = ms_total / args.steps
    value = whole_job_gbs(world, set_bytes, args.steps, ms_total * 1e-3)   # GB/s over all ranks
    kernel_gbs = set_bytes / (ms_per_step * 1e-3) / 1e9                 # per launch, this GPU
    clocks = sampler.summary(tc0, t1)
    clocks["window"] = "timed region and the 1.2 s of the same graph replays before it"

    # ---- end to end through the public API: gptq_gemm_host with A in pinned host memory and C
    # returned to pinned host memory (the copies, the GEMM and the wait inside the call)
    a_host = A.cpu().pin_memory()
    c_host = torch.empty((M, wl.N), dtype=A.dtype).pin_memory()
    n_e2e = max(1, min(args.steps, 2000))

    # each weight set's call prepared once (g.HostGemm on a named stream: gptq_gemm_host captured
    # into a graph); a step is one gptq_host_plan_run call
    host_calls = [g.HostGemm(a_host, a, q, z, s, bits=wl.bits, group=wl.group, fmt=g.V2, C_dev=c,
                             C_host=c_host, stream=stream) for (q, z, s, a, c) in sets]

    def host_step(i):
        host_calls[i % S]()

    with torch.cuda.stream(stream):
        for i in range(min(50, n_e2e)):
            host_step(i)
        barrier()
        te0 = time.perf_counter()
        for i in range(n_e2e):
            host_step(i)
        te1 = time.perf_counter()
    e2e_s = max_over_ranks(te1 - te0, dist, dev)
    e2e_value = whole_job_gbs(world, set_bytes, n_e2e, e2e_s)
    del sets, host_calls, main_graph, rem_graphs
    torch.cuda.synchronize()

    # ---- the secondary figure (M = 4096 prefill) and the per-configuration section
    configs = None if args.skip_configs else run_configs(g, torch, dev, stream, peaks, l2, args.config_filter)
    sampler.stop()
    prefill = None
    if configs is not None:
        prefill = next((r for r in configs if r["workload"] == PREFILL.name and r["path"] == "gptq_gemm"), None)
    sweep = run_sweep(g, torch, dev, stream, hbm_peak, bf16_peak, l2, args.sweep_filter) if args.all else None
    torch.cuda.synchronize()
    assert g.device_status(stream) == 0, "device status word reported an error"

    traffic = load_traffic("decode_m1_4bit")
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded N(0,0.02) weights quantized on the GPU by round-to-nearest; N(0,1) activations)",
        "config": {"workload": "llama7b_decode_4bit_g128", "M": M, "K": wl.K, "N": wl.N,
                   "bits": wl.bits, "group": wl.group, "fmt": "v2", "act_dtype": "fp16",
                   "accumulate": "fp32", "bytes_per_step": set_bytes,
                   "l2": "inputs rotate over %d weight sets = %.0f MB > 3x L2 (%.0f MB)" % (
                       S, S * set_bytes / 1e6, l2 / 1e6),
                   "timing": "CUDA events on the launching stream around CUDA-graph replays of the K "
                             "steps, queued behind a short GPU sleep so that no host launch latency "
                             "falls inside the timed region",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline(kernel_gbs, hbm_peak, "GB/s", "hbm", peak_src + " (hbm_gbs)", traffic),
        "kernel_replays": {"us_median": round(med_ms * 1e3, 3), "us_min": round(min_ms * 1e3, 3),
                           "us_max": round(max_ms * 1e3, 3), "launches_per_replay": R, "replays": 10,
                           "GB/s": round(set_bytes / (med_ms * 1e-3) / 1e9, 1),
                           "frac": round(set_bytes / (med_ms * 1e-3) / 1e9 / hbm_peak, 4),
                           "single_launch_us": round(single_ms * 1e3, 3),
                           "note": "median of 10 replays of one graph (a first replay discarded); "
                                   "single launch: event pair around one launch, synchronized"},
        "e2e": {"value": round(e2e_value, 3), "unit": "GB/s", "h2d_bytes_per_step": M * wl.K * 2,
                "d2h_bytes_per_step": M * wl.N * 2,
                "note": "weights resident on the device (the model); per step one gptq_host_plan_run "
                        "call (gptq_gemm_host captured once per weight set): A host->device, gptq_gemm, "
                        "C device->host, stream synchronize"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if prefill is not None:
        line["prefill"] = prefill
    if configs is not None:
        line["configs"] = configs
    if sweep is not None:
        line["all_workloads"] = sweep
    return line


# ------------------------------------------------------------------------------------ configs
def _checkpoint(g, torch, dev, wl, fmt=None):
    draw = gptq_inputs.draw_weights(wl)
    W = torch.from_numpy(draw.W).to(dev)
    gi = None if draw.g_idx is None else torch.from_numpy(draw.g_idx).to(dev)
    f = fmt if fmt is not None else g.V2
    qw, qz, sc = g.quantize_rtn(W, bits=wl.bits, group=wl.group, g_idx=gi, sym=wl.sym, fmt=f)
    del W
    return draw, qw, qz, sc, gi


def time_gemm(g, torch, dev, stream, wl, M, l2, path="gemm", fmt=None, reps=200):
    """Median per-launch time of one GEMM call on one workload: a CUDA graph of launches over S
    rotating copies of every input (S x bytes > 3x L2 where one copy is smaller), replayed 11
    times, the first replay discarded.  path: "gemm" (gptq_gemm; act-order: g_idx with the
    workspace in which the rows are sorted by group on the device), "rows" (gptq_gemm with g_idx
    and the per-row-group kernels),
    "perm" (act-order rows sorted on the host, gptq_gemm_perm), "il" (qweight in the interleaved
    layout, gptq_gemm_interleaved; act-order checkpoints sorted first, through perm) or "dequant"
    (gptq_dequant)."""
    f = fmt if fmt is not None else g.V2
    draw, qw, qz, sc, gi = _checkpoint(g, torch, dev, wl, f)
    perm = ws = None
    if path in ("perm", "il") and draw.g_idx is not None:
        qw2, p = g.prepack_act_order(qw.cpu().numpy(), draw.g_idx, K=wl.K, N=wl.N, bits=wl.bits,
                                     group=wl.group)
        qw, perm, gi = torch.from_numpy(qw2).to(dev), torch.from_numpy(p).to(dev), None
        ws = torch.empty(max(1, g.gemm_perm_workspace_size(M, wl.K)), dtype=torch.uint8, device=dev)
    if path == "il":
        qw = torch.from_numpy(g.prepack_interleave(qw.cpu().numpy(), K=wl.K, N=wl.N, bits=wl.bits)).to(dev)
    A = gptq_inputs.draw_activations(wl, M).to(dev) if path != "dequant" else None
    if path == "dequant":
        out_shape, out_dt = (wl.K, wl.N), torch.float16 if wl.act_dtype == "f16" else torch.bfloat16
        nbytes = algorithmic_bytes(wl, 0) - (wl.K * 4 if wl.act_order else 0) + wl.K * wl.N * 2
    else:
        out_shape, out_dt = (M, wl.N), A.dtype
        nbytes = algorithmic_bytes(wl, M)
    per_set = nbytes + (0 if path == "dequant" else M * wl.N * 2)
    # the caller's workspace: act-order rows sorted on the device, or bf16 activations through the
    # tensor-core kernel (fp16 copy of A)
    gws = None
    if path in ("gemm", "rows") and A is not None:
        size = g.act_order_workspace_size(M, wl.K, wl.N, wl.bits, wl.group) if (
            path == "gemm" and draw.g_idx is not None) else 0
        if size == 0 and A.dtype == torch.bfloat16:
            size = g.workspace_size(M, wl.K, wl.N, wl.bits, wl.group)
        if size:
            gws = torch.empty(size, dtype=torch.uint8, device=dev)
    S = max(1, min(256, int(np.ceil(3 * l2 / per_set))))
    sets = [(qw.clone(), qz.clone(), sc.clone(), None if A is None else A.clone(),
             torch.empty(out_shape, dtype=out_dt, device=dev)) for _ in range(S)]
    # the copies ran on the current stream; the launches go to `stream`, which (a PyTorch pool
    # stream) does not wait for it
    torch.cuda.synchronize()
    n = S * max(1, reps // S) if (M <= 64 and path != "dequant") else S * max(1, 8 // S)

    def launch(i):
        q, z, s_, a, c = sets[i % S]
        if path == "perm":
            g.gemm_perm(a, perm, q, z, s_, bits=wl.bits, group=wl.group, fmt=f, out=c, workspace=ws,
                        stream=stream)
        elif path == "il":
            g.gemm_interleaved(a, q, z, s_, perm, N=wl.N, bits=wl.bits, group=wl.group, fmt=f, out=c,
                               workspace=ws, stream=stream)
        elif path == "dequant":
            g.dequant(q, z, s_, gi, K=wl.K, bits=wl.bits, group=wl.group, fmt=f, dtype=out_dt, out=c,
                      stream=stream)
        else:
            g.gemm(a, q, z, s_, gi, bits=wl.bits, group=wl.group, fmt=f, out=c, workspace=gws,
                   sort_rows=(path == "gemm"), stream=stream)

    gr = capture(torch, stream, launch, n)
    ms, ms_min, ms_max = replay_median(torch, stream, gr, n)
    del sets, gr
    return ms, nbytes, S


def time_device_prepack(g, torch, dev, stream, wl, l2, reps=64):
    """Median per-call time of gptq_prepack_act_order_device (sort, repack, ordering kernel) on an
    act-order workload, a CUDA graph of calls over rotating copies of qweight and g_idx.  Bytes:
    qweight and g_idx read, the sorted qweight and perm written."""
    import ctypes
    draw, qw, qz, sc, gi = _checkpoint(g, torch, dev, wl)
    nbytes = 2 * qw.numel() * 4 + 2 * wl.K * 4
    S = max(1, min(256, int(np.ceil(3 * l2 / nbytes))))
    wsb = g.prepack_act_order_device_workspace_size(wl.K, wl.bits, wl.group)
    sets = [(qw.clone(), gi.clone(), torch.empty_like(qw), torch.empty(wl.K, dtype=torch.int32, device=dev),
             torch.empty(wsb, dtype=torch.uint8, device=dev)) for _ in range(S)]
    torch.cuda.synchronize()                   # the copies ran on another stream than the calls
    n = S * max(1, reps // S)
    p = lambda t: ctypes.c_void_p(t.data_ptr())

    def launch(i):
        q, gix, out, perm, ws = sets[i % S]
        rc = g.lib().gptq_prepack_act_order_device(p(q), p(gix), wl.K, wl.N, wl.bits, wl.group, p(out), p(perm),
                                                   p(ws), wsb, ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, g.strerror(rc)

    gr = capture(torch, stream, launch, n)
    ms, _, _ = replay_median(torch, stream, gr, n)
    del sets, gr
    return ms, nbytes, S


def run_configs(g, torch, dev, stream, peaks, l2, only=""):
    """Every workload configuration at its exact shape, with its roofline fraction."""
    hbm_peak, bf16_peak, _, src = peaks
    W = gptq_inputs.WORKLOADS
    plan = [
        # (config, workload, M, path, label)
        ("1", "tiny_4bit_g64", 4, "gemm", "correctness case"),
        ("2", "llama7b_decode_4bit_g128", 1, "gemm", ""),
        ("2", "llama7b_decode_4bit_g128", 8, "gemm", ""),
        ("2", "llama7b_decode_4bit_g128", 16, "gemm", ""),
        ("2", "llama7b_decode_4bit_g128", 1, "il", "interleaved layout, gptq_gemm_interleaved"),
        ("2", "llama7b_decode_4bit_g128", 16, "il", "interleaved layout, gptq_gemm_interleaved"),
        ("3", "lowbit_2bit_g64", 1, "gemm", ""),
        ("3", "lowbit_2bit_g64", 8, "gemm", ""),
        ("3", "lowbit_2bit_g64", 32, "gemm", ""),
        ("4", "act_order_3bit_g128", 16, "gemm", "g_idx through gptq_gemm, rows sorted by group on the device"),
        ("4", "act_order_3bit_g128", 16, "rows", "g_idx through gptq_gemm, per-row groups"),
        ("4", "act_order_3bit_g128", 1, "gemm", "one token, rows sorted by group on the device"),
        ("4", "act_order_3bit_g128", 1, "rows", "one token, per-row groups"),
        ("4", "act_order_3bit_g128", 4096, "gemm", "4096 tokens, rows sorted by group on the device"),
        ("4", "act_order_3bit_g128", 16, "perm", "rows sorted on the host, gptq_gemm_perm"),
        ("4", "act_order_3bit_g128", 16, "il", "rows sorted, then interleaved, gptq_gemm_interleaved"),
        ("4", "act_order_3bit_g128", 0, "devprep", "gptq_prepack_act_order_device: rows sorted on the device "
                                                   "once per weight (qweight and g_idx read, sorted copy and perm written)"),
        ("5", "prefill_4bit_g128", 4096, "gemm", ""),
        ("5", "prefill_8bit_sym_g128", 4096, "gemm", ""),
        ("5", "prefill_4bit_gall", 4096, "gemm", ""),
        ("5", "prefill_4bit_g128", 0, "dequant", "gptq_dequant to bf16"),
        ("2", "llama7b_decode_4bit_g128", 0, "dequant", "gptq_dequant to fp16"),
    ]
    rows = []
    for cfg, name, M, path, label in plan:
        if only and only not in name:
            continue
        wl = W[name]
        if path == "devprep":
            ms, nbytes, S = time_device_prepack(g, torch, dev, stream, wl, l2)
        else:
            ms, nbytes, S = time_gemm(g, torch, dev, stream, wl, M, l2, path=path)
        row = {"config": cfg, "workload": name, "M": M, "path": {"gemm": "gptq_gemm", "perm": "gptq_gemm_perm",
                                                                 "rows": "gptq_gemm (per-row groups)",
                                                                 "il": "gptq_gemm_interleaved",
                                                                 "dequant": "gptq_dequant",
                                                                 "devprep": "gptq_prepack_act_order_device"}[path],
               "us": round(ms * 1e3, 3)}
        if label:
            row["note"] = label
        if path not in ("dequant", "devprep") and M > g.DECODE_MAX_M:
            tflops = 2.0 * M * wl.N * wl.K / (ms * 1e-3) / 1e12
            key = {"prefill_4bit_g128": "prefill_4bit"}.get(name)
            row.update(value=round(tflops, 2), unit="TFLOP/s",
                       roofline=roofline(tflops, bf16_peak, "TFLOP/s", "tensor", src + " (bf16_tflops, burst)",
                                         load_traffic(key) if key else None))
        else:
            gbs = nbytes / (ms * 1e-3) / 1e9
            key = {("llama7b_decode_4bit_g128", 1): "decode_m1_4bit"}.get((name, M)) if path == "gemm" else None
            row.update(value=round(gbs, 1), unit="GB/s", bytes=nbytes,
                       roofline=roofline(gbs, hbm_peak, "GB/s", "hbm", src + " (hbm_gbs)",
                                         load_traffic(key) if key else None))
        row["inputs"] = "%d rotating copies (%.0f MB)" % (S, S * nbytes / 1e6)
        rows.append(row)
        print(json.dumps(row), file=sys.stderr, flush=True)
    for name, mw in gptq_inputs.MOE_WORKLOADS.items():
        if only and only not in name:
            continue
        for T in mw.Ts:
            ms, nbytes, active, nrows, max_m = time_grouped(g, torch, dev, stream, mw, T, l2)
            gbs = nbytes / (ms * 1e-3) / 1e9
            row = {"config": "moe", "workload": name, "M": T, "path": "gptq_gemm_grouped", "rows": nrows,
                   "experts_active": active, "us": round(ms * 1e3, 3), "value": round(gbs, 1), "unit": "GB/s",
                   "bytes": nbytes, "roofline": roofline(gbs, hbm_peak, "GB/s", "hbm", src + " (hbm_gbs)")}
            rows.append(row)
            print(json.dumps(row), file=sys.stderr, flush=True)
    return rows


# ------------------------------------------------------------------------------------ sweep
def time_grouped(g, torch, dev, stream, mw, T, l2, reps=200):
    """Median per-launch time of gptq_gemm_grouped on a mixture-of-experts layer: T tokens routed
    to top-k experts (rows grouped by expert), CUDA graph of launches over expert-weight copies
    whose total exceeds 3x L2."""
    r = gptq_inputs.draw_routing(mw, T)
    toks = gptq_inputs.draw_token_activations(mw, T)
    A = toks[torch.from_numpy(r.row_token).long()].contiguous().to(dev)
    offsets = torch.from_numpy(r.offsets).to(dev)
    max_m = int(np.diff(r.offsets).max())
    qws, qzs, scs = [], [], []
    for e in range(mw.E):
        W = torch.from_numpy(gptq_inputs.draw_expert_weights(mw, e)).to(dev)
        qw, qz, sc = g.quantize_rtn(W, bits=mw.bits, group=mw.group, fmt=g.V2)
        qws.append(qw); qzs.append(qz); scs.append(sc)
        del W
    qw, qz, sc = torch.stack(qws), torch.stack(qzs), torch.stack(scs)
    del qws, qzs, scs
    nbytes, active = grouped_bytes(mw, r.offsets)
    weight_bytes = qw.numel() * 4 + qz.numel() * 4 + sc.numel() * 2
    S = max(1, min(64, int(np.ceil(3 * l2 / weight_bytes))))
    sets = [(qw.clone(), qz.clone(), sc.clone(), torch.empty((A.shape[0], mw.N), dtype=A.dtype, device=dev))
            for _ in range(S)]
    del qw, qz, sc
    torch.cuda.synchronize()                   # the copies ran on another stream than the calls
    n = max(S, (reps // S) * S)

    def launch(i):
        q, z, s_, c = sets[i % S]
        g.gemm_grouped(A, offsets, q, z, s_, bits=mw.bits, group=mw.group, max_m=max_m, fmt=g.V2, out=c,
                       stream=stream)

    gr = capture(torch, stream, launch, n)
    ms, _, _ = replay_median(torch, stream, gr, n)
    del sets, gr
    return ms, nbytes, active, int(r.offsets[-1]), max_m


def run_sweep(g, torch, dev, stream, hbm_peak, bf16_peak, l2, only=""):
    """--all: every workload x token count x checkpoint format (v1 and v2), gptq_gemm and, for
    act-order, the prepacked call."""
    rows = []
    for name, wl in gptq_inputs.WORKLOADS.items():
        if only not in name:
            continue
        variants = [(fmt, False) for fmt in wl.fmts]
        if wl.act_order:
            variants += [(fmt + "+prepacked", True) for fmt in wl.fmts]
        for M in wl.Ms:
            for fmt, pre in variants:
                if pre and M > g.DECODE_MAX_M:
                    continue
                f = g.V2 if fmt.startswith("v2") else g.V1
                ms, nbytes, _ = time_gemm(g, torch, dev, stream, wl, M, l2, path="perm" if pre else "gemm", fmt=f)
                gbs = nbytes / (ms * 1e-3) / 1e9
                tflops = 2.0 * M * wl.N * wl.K / (ms * 1e-3) / 1e12
                row = {"workload": name, "M": M, "fmt": fmt, "us": round(ms * 1e3, 3),
                       "GB/s": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
                       "TFLOP/s": round(tflops, 2), "tensor_frac": round(tflops / bf16_peak, 4)}
                rows.append(row)
                print(json.dumps(row), file=sys.stderr, flush=True)
    return rows


# ------------------------------------------------------------------------------------ CPU oracle
def oracle_checkpoint(wl):
    import oracle
    draw = gptq_inputs.draw_weights(wl)
    return oracle.make_checkpoint(draw.W, wl.bits, wl.group, draw.g_idx, wl.sym, oracle.V2)


def oracle_sample(ck, wl, ncols):
    """A column slice [0, ncols) of the checkpoint: a smaller GEMM of the same recipe."""
    zw = ncols * wl.bits // 32
    return (np.ascontiguousarray(ck["qweight"][:, :ncols]), np.ascontiguousarray(ck["qzeros"][:, :zw]),
            np.ascontiguousarray(ck["scales"][:, :ncols]))


def time_oracle_step(ck, wl, A16, ncols, dtype_code=None):
    import oracle
    qw, qz, sc = oracle_sample(ck, wl, ncols)
    t = time.perf_counter()
    oracle.gemm(A16, oracle.F16 if dtype_code is None else dtype_code, qw, qz, sc, ck["g_idx"], ncols,
                wl.bits, wl.group, oracle.V2)
    return time.perf_counter() - t


def sample_bytes(wl, M, ncols):
    sub = gptq_inputs.Workload("s", wl.K, ncols, wl.bits, wl.group, wl.act_dtype, (M,), ("v2",), 0)
    return algorithmic_bytes(sub, M)


def cpu_baseline(budget_s=8.0):
    """The oracle as it stands (one thread) on a bounded column sample of the decode workload,
    and on 64 rows of the M = 4096 prefill workload (extrapolated to all 4096 rows)."""
    import oracle
    wl, M = DECODE, 1
    ck = oracle_checkpoint(wl)
    A16 = gptq_inputs.bits16(gptq_inputs.draw_activations(wl, M))
    t32 = time_oracle_step(ck, wl, A16, 32 * 8)
    ncols = int(min(wl.N, max(256, (budget_s / 4) / max(t32, 1e-6) * 256)) // 32 * 32)
    time_oracle_step(ck, wl, A16, ncols)                 # discarded first run (cold caches)
    reps, total, t_end = 0, 0.0, time.perf_counter() + budget_s
    while time.perf_counter() < t_end or reps == 0:
        total += time_oracle_step(ck, wl, A16, ncols)
        reps += 1
    per = total / reps
    gbs = sample_bytes(wl, M, ncols) / per / 1e9
    host = host_info()
    out = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "host": host,
           "sample": "decode M=1, K=4096, first %d of 11008 columns (4-bit g128 v2), %d runs after one "
                     "discarded, %.2f s each (unpack + fp32 dequant + fp32 GEMM, single thread)" % (ncols, reps, per)}
    # prefill leg: 64 seeded rows of the M = 4096 problem, all N; time x 64 for the whole problem
    pw = PREFILL
    pck = oracle_checkpoint(pw)
    A = gptq_inputs.draw_activations(pw, pw.Ms[0])
    rows = np.sort(np.random.default_rng(64).choice(pw.Ms[0], size=64, replace=False)).astype(np.int32)
    A64 = gptq_inputs.bits16(A)[rows]
    t = time.perf_counter()
    oracle.gemm(A64, oracle.BF16, pck["qweight"], pck["qzeros"], pck["scales"], None, pw.N, pw.bits, pw.group,
                oracle.V2)
    dt = time.perf_counter() - t
    tflops = 2.0 * 64 * pw.N * pw.K / dt / 1e12
    out["prefill"] = {"value": round(tflops, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                      "seconds_64_rows": round(dt, 3), "seconds_extrapolated_4096_rows": round(dt * 64, 1),
                      "sample": "prefill_4bit_g128: 64 seeded rows of A [4096, 4096] x W [4096, 14336] "
                                "(4-bit g128 v2, bf16), all columns; the full problem is 64x this time"}
    return out


def run_reference(args):
    wl, M = DECODE, 1
    ck = oracle_checkpoint(wl)
    A16 = gptq_inputs.bits16(gptq_inputs.draw_activations(wl, M))
    t_probe = time_oracle_step(ck, wl, A16, 256)
    budget = 150.0 / max(1, args.steps + args.warmup)
    ncols = int(min(wl.N, max(32, budget / max(t_probe, 1e-6) * 256)) // 32 * 32)
    ncols = max(32, ncols)
    for _ in range(args.warmup):
        time_oracle_step(ck, wl, A16, ncols)
    total = 0.0
    for _ in range(args.steps):
        total += time_oracle_step(ck, wl, A16, ncols)
    per = total / args.steps
    gbs = sample_bytes(wl, M, ncols) / per / 1e9
    sample = "decode M=1, K=4096, first %d of 11008 columns per step (4-bit g128 v2)" % ncols
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded, same recipe as our arm; checkpoint written by the oracle)",
        "config": {"workload": "llama7b_decode_4bit_g128", "M": M, "K": wl.K, "N": wl.N,
                   "bits": wl.bits, "group": wl.group, "fmt": "v2", "sample_columns": ncols},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_info()},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile_target(args):
    """--profile WORKLOAD:M[:PATH]: just `warmup + steps` eager launches of one call on one
    workload (PATH gemm, rows, perm, il or dequant; a mixture-of-experts workload with M tokens
    runs gptq_gemm_grouped), for a profiler to capture; prints one short line."""
    import torch
    import gptq_bit_weight_gemm_gb300 as g
    from gptq_bit_weight_gemm_gb300 import build as lib_build
    lib_build.build()
    parts = args.profile.split(":")
    if parts[0] in gptq_inputs.MOE_WORKLOADS:
        mw, T = gptq_inputs.MOE_WORKLOADS[parts[0]], int(parts[1])
        dev = torch.device("cuda", 0)
        stream = torch.cuda.Stream()
        r = gptq_inputs.draw_routing(mw, T)
        toks = gptq_inputs.draw_token_activations(mw, T)
        A = toks[torch.from_numpy(r.row_token).long()].contiguous().to(dev)
        offsets = torch.from_numpy(r.offsets).to(dev)
        max_m = int(np.diff(r.offsets).max())
        qws, qzs, scs = [], [], []
        for e in range(mw.E):
            W = torch.from_numpy(gptq_inputs.draw_expert_weights(mw, e)).to(dev)
            qw, qz, sc = g.quantize_rtn(W, bits=mw.bits, group=mw.group, fmt=g.V2)
            qws.append(qw); qzs.append(qz); scs.append(sc)
            del W
        qw, qz, sc = torch.stack(qws), torch.stack(qzs), torch.stack(scs)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup + args.steps):
                g.gemm_grouped(A, offsets, qw, qz, sc, bits=mw.bits, group=mw.group, max_m=max_m, fmt=g.V2,
                               stream=stream)
        stream.synchronize()
        assert g.device_status(stream) == 0
        print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps}))
        return
    wl, M = gptq_inputs.WORKLOADS[parts[0]], int(parts[1])
    path = parts[2] if len(parts) > 2 else "gemm"
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream()
    draw, qw, qz, sc, gi = _checkpoint(g, torch, dev, wl)
    perm = ws = None
    if path in ("perm", "il") and draw.g_idx is not None:
        qw2, p = g.prepack_act_order(qw.cpu().numpy(), draw.g_idx, K=wl.K, N=wl.N, bits=wl.bits, group=wl.group)
        qw, perm, gi = torch.from_numpy(qw2).to(dev), torch.from_numpy(p).to(dev), None
        ws = torch.empty(max(1, g.gemm_perm_workspace_size(M, wl.K)), dtype=torch.uint8, device=dev)
    if path == "il":
        qw = torch.from_numpy(g.prepack_interleave(qw.cpu().numpy(), K=wl.K, N=wl.N, bits=wl.bits)).to(dev)
    A = gptq_inputs.draw_activations(wl, max(M, 1)).to(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup + args.steps):
            if path == "perm":
                g.gemm_perm(A, perm, qw, qz, sc, bits=wl.bits, group=wl.group, workspace=ws, stream=stream)
            elif path == "il":
                g.gemm_interleaved(A, qw, qz, sc, perm, N=wl.N, bits=wl.bits, group=wl.group, workspace=ws,
                                   stream=stream)
            elif path == "dequant":
                g.dequant(qw, qz, sc, gi, K=wl.K, bits=wl.bits, group=wl.group, stream=stream,
                          dtype=torch.float16 if wl.act_dtype == "f16" else torch.bfloat16)
            else:
                g.gemm(A, qw, qz, sc, gi, bits=wl.bits, group=wl.group, sort_rows=(path != "rows"), stream=stream)
    stream.synchronize()
    assert g.device_status(stream) == 0
    print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-configs", action="store_true",
                    help="leave out the per-configuration section (and with it the prefill figure)")
    ap.add_argument("--config-filter", default="",
                    help="only the configurations whose workload name contains this string")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--all", action="store_true",
                    help="also time every workload, token count and format (per-launch us, GB/s, TFLOP/s)")
    ap.add_argument("--sweep-filter", default="",
                    help="with --all: only the workloads whose name contains this string")
    ap.add_argument("--profile", default="",
                    help="WORKLOAD:M[:gemm|perm|il|dequant]: only launch that call warmup+steps times "
                         "(for a profiler), no timing")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    if args.profile:
        run_profile_target(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu = cpu_baseline()
    line = run_ours(args, rank, world, local_rank)
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
