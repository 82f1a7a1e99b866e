"""Benchmark of the GB300 GPTQ GEMM library; prints ONE JSON line (rank 0).

Workload (the headline): Llama-7B-shaped decode GEMV, A fp16 [1, 4096] x W [4096, 11008] 4-bit,
group 128, GPTQv2 -- metric "M=1 decode weight GB/s" with algorithmic bytes = qweight + scales +
qzeros + A.  One step = one gptq_gemm launch on one batch (M = 1 token).  Steps run as CUDA-graph
replays over S rotating copies of the weights whose total size is more than 3x the L2 cache, so
every step reads its weights from HBM.  The same line carries the secondary figure of the
metric: M = 4096 prefill TFLOP/s (A bf16 [4096, 4096] x W [4096, 14336] 4-bit g128).

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
    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

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
    with torch.cuda.stream(stream):
        for i in range(2 * S):
            launch(i)   # sets kernel attributes before capture
    stream.synchronize()

    def capture(n):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(n):
                launch(i)
        return gr

    main_graph = capture(R)
    rem_graphs = {}

    for n in (args.warmup, args.steps):   # every graph is captured before anything is timed
        if n % R and n % R not in rem_graphs:
            rem_graphs[n % R] = capture(n % R)

    def run_steps(n):
        for _ in range(n // R):
            main_graph.replay()
        if n % R:
            rem_graphs[n % R].replay()

    uuid = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(local_rank)
    sampler = ClockSampler(uuid)
    with torch.cuda.stream(stream):
        run_steps(args.warmup)
    stream.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
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

    # ---- end to end through the public API: A from pinned host memory, C read back
    a_host = A.cpu().pin_memory()
    c_host = torch.empty((M, wl.N), dtype=A.dtype).pin_memory()
    n_e2e = max(1, min(args.steps, 2000))
    with torch.cuda.stream(stream):
        for i in range(min(50, n_e2e)):
            q, z, s, a, c = sets[i % S]
            a.copy_(a_host, non_blocking=True)
            launch(i)
            c_host.copy_(c, non_blocking=True)
            stream.synchronize()
        barrier()
        te0 = time.perf_counter()
        for i in range(n_e2e):
            q, z, s, a, c = sets[i % S]
            a.copy_(a_host, non_blocking=True)
            launch(i)
            c_host.copy_(c, non_blocking=True)
            stream.synchronize()
        te1 = time.perf_counter()
    e2e_s = max_over_ranks(te1 - te0, dist, dev)
    e2e_value = whole_job_gbs(world, set_bytes, n_e2e, e2e_s)
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    # ---- secondary figure: M = 4096 prefill TFLOP/s
    prefill = run_prefill(g, torch, dev, stream, bf16_peak, peak_src, l2) if not args.skip_prefill else None
    sweep = run_sweep(g, torch, dev, stream, hbm_peak, bf16_peak, l2, args.sweep_filter) if args.all else None
    del sets
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
                   "timing": "CUDA events on the launching stream around CUDA-graph replays",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(kernel_gbs, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(kernel_gbs / hbm_peak, 4),
                     "traffic": traffic, "peak_source": peak_src + " (hbm_gbs)"},
        "e2e": {"value": round(e2e_value, 3), "unit": "GB/s", "h2d_bytes_per_step": M * wl.K * 2,
                "d2h_bytes_per_step": M * wl.N * 2,
                "note": "weights resident on the device (the model); per step: A host->device, "
                        "gptq_gemm, C device->host, stream synchronize"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if prefill is not None:
        line["prefill"] = prefill
    if sweep is not None:
        line["all_workloads"] = sweep
    return line


def run_prefill(g, torch, dev, stream, bf16_peak, peak_src, l2):
    wl = PREFILL
    M = wl.Ms[0]
    draw = gptq_inputs.draw_weights(wl)
    W = torch.from_numpy(draw.W).to(dev)
    qw, qz, sc = g.quantize_rtn(W, bits=wl.bits, group=wl.group, fmt=g.V2)
    del W
    A = gptq_inputs.draw_activations(wl, M).to(dev)
    C = torch.empty((M, wl.N), dtype=A.dtype, device=dev)
    flop = 2.0 * M * wl.N * wl.K
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.gemm(A, qw, qz, sc, bits=wl.bits, group=wl.group, out=C, stream=stream)
        stream.synchronize()
        n = 10
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(n):
            g.gemm(A, qw, qz, sc, bits=wl.bits, group=wl.group, out=C, stream=stream)
        e.record(stream)
    stream.synchronize()
    ms = s.elapsed_time(e) / n
    tflops = flop / (ms * 1e-3) / 1e12
    return {"workload": "prefill_4bit_g128", "M": M, "K": wl.K, "N": wl.N, "value": round(tflops, 2),
            "unit": "TFLOP/s", "ms_per_launch": ms,
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": round(tflops / bf16_peak, 4),
                         "traffic": load_traffic("prefill_4bit"),
                         "peak_source": peak_src + " (bf16_tflops, burst)"},
            "note": "A (33.5 MB) and W (29 MB) fit in L2 but are re-read per tile; timed back to back"}


# ------------------------------------------------------------------------------------ sweep
def time_workload(g, torch, dev, stream, wl, M, fmt, l2, reps=200, prepacked=False):
    """Per-launch time of gptq_gemm on one workload: CUDA graph of `reps` launches over weight
    copies whose total exceeds 3x L2 (or the whole problem when one copy is larger).
    prepacked: an act-order checkpoint with its rows sorted by group (gptq_prepack_act_order),
    multiplied by gptq_gemm_perm."""
    draw = gptq_inputs.draw_weights(wl)
    W = torch.from_numpy(draw.W).to(dev)
    gi = None if draw.g_idx is None else torch.from_numpy(draw.g_idx).to(dev)
    f = g.V2 if fmt == "v2" else g.V1
    qw, qz, sc = g.quantize_rtn(W, bits=wl.bits, group=wl.group, g_idx=gi, sym=wl.sym, fmt=f)
    del W
    perm = None
    if prepacked:
        qw2, p = g.prepack_act_order(qw.cpu().numpy(), draw.g_idx, K=wl.K, N=wl.N, bits=wl.bits,
                                     group=wl.group)
        qw, perm = torch.from_numpy(qw2).to(dev), torch.from_numpy(p).to(dev)
        ws = torch.empty(max(1, g.gemm_perm_workspace_size(M, wl.K)), dtype=torch.uint8, device=dev)
    A = gptq_inputs.draw_activations(wl, M).to(dev)
    nbytes = algorithmic_bytes(wl, M)
    S = max(1, min(256, int(np.ceil(3 * l2 / nbytes))))   # > 3x L2 of weights (the tiny case: L2)
    sets = [(qw.clone(), qz.clone(), sc.clone(), A.clone(),
             torch.empty((M, wl.N), dtype=A.dtype, device=dev)) for _ in range(S)]
    n = max(S, (reps // S) * S) if M <= 64 else S * max(1, 8 // S)

    def launch(i):
        q, z, s_, a, c = sets[i % S]
        if prepacked:
            g.gemm_perm(a, perm, q, z, s_, bits=wl.bits, group=wl.group, fmt=f, out=c, workspace=ws,
                        stream=stream)
        else:
            g.gemm(a, q, z, s_, gi, bits=wl.bits, group=wl.group, fmt=f, out=c, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(2 * S):
            launch(i)
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for i in range(n):
            launch(i)
    with torch.cuda.stream(stream):
        gr.replay()
        st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        st.record(stream)
        for _ in range(3):
            gr.replay()
        en.record(stream)
    stream.synchronize()
    ms = st.elapsed_time(en) / (3 * n)
    del sets, gr
    return ms, nbytes


def time_grouped(g, torch, dev, stream, mw, T, l2, reps=200):
    """Per-launch time of gptq_gemm_grouped on a mixture-of-experts layer: T tokens routed to
    top-k experts (rows grouped by expert), CUDA graph of launches over expert-weight copies
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
    n = max(S, (reps // S) * S)

    def launch(i):
        q, z, s_, c = sets[i % S]
        g.gemm_grouped(A, offsets, q, z, s_, bits=mw.bits, group=mw.group, max_m=max_m, fmt=g.V2, out=c,
                       stream=stream)

    with torch.cuda.stream(stream):
        for i in range(2 * S):
            launch(i)
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for i in range(n):
            launch(i)
    with torch.cuda.stream(stream):
        gr.replay()
        st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        st.record(stream)
        for _ in range(3):
            gr.replay()
        en.record(stream)
    stream.synchronize()
    ms = st.elapsed_time(en) / (3 * n)
    del sets, gr
    return ms, nbytes, active, int(r.offsets[-1]), max_m


def run_sweep(g, torch, dev, stream, hbm_peak, bf16_peak, l2, only=""):
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
                ms, nbytes = time_workload(g, torch, dev, stream, wl, M, fmt.split("+")[0], l2,
                                           prepacked=pre)
                gbs = nbytes / (ms * 1e-3) / 1e9
                tflops = 2.0 * M * wl.N * wl.K / (ms * 1e-3) / 1e12
                row = {"workload": name, "M": M, "fmt": fmt, "us": round(ms * 1e3, 3),
                       "GB/s": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
                       "TFLOP/s": round(tflops, 2), "tensor_frac": round(tflops / bf16_peak, 4)}
                rows.append(row)
                print(json.dumps(row), file=sys.stderr, flush=True)
    for name, mw in gptq_inputs.MOE_WORKLOADS.items():
        if only not in name:
            continue
        for T in mw.Ts:
            ms, nbytes, active, nrows, max_m = time_grouped(g, torch, dev, stream, mw, T, l2)
            gbs = nbytes / (ms * 1e-3) / 1e9
            row = {"workload": name, "M": T, "fmt": "v2 grouped", "rows": nrows, "experts_active": active,
                   "max_m": max_m, "us": round(ms * 1e3, 3), "GB/s": round(gbs, 1),
                   "hbm_frac": round(gbs / hbm_peak, 4),
                   "TFLOP/s": round(2.0 * nrows * mw.N * mw.K / (ms * 1e-3) / 1e12, 2), "tensor_frac": None}
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


def time_oracle_step(ck, wl, A16, ncols):
    import oracle
    qw, qz, sc = oracle_sample(ck, wl, ncols)
    t = time.perf_counter()
    oracle.gemm(A16, oracle.F16, qw, qz, sc, ck["g_idx"], ncols, wl.bits, wl.group, oracle.V2)
    return time.perf_counter() - t


def sample_bytes(wl, M, ncols):
    sub = gptq_inputs.Workload("s", wl.K, ncols, wl.bits, wl.group, wl.act_dtype, (M,), ("v2",), 0)
    return algorithmic_bytes(sub, M)


def cpu_baseline(budget_s=12.0):
    """The oracle as it stands (one thread) on a bounded column sample of the decode workload."""
    wl, M = DECODE, 1
    ck = oracle_checkpoint(wl)
    A16 = gptq_inputs.bits16(gptq_inputs.draw_activations(wl, M))
    t32 = time_oracle_step(ck, wl, A16, 32 * 8)
    ncols = int(min(wl.N, max(256, (budget_s / 4) / max(t32, 1e-6) * 256)) // 32 * 32)
    reps, total, t_end = 0, 0.0, time.perf_counter() + budget_s
    while time.perf_counter() < t_end or reps == 0:
        total += time_oracle_step(ck, wl, A16, ncols)
        reps += 1
    per = total / reps
    gbs = sample_bytes(wl, M, ncols) / per / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "decode M=1, K=4096, first %d of 11008 columns (4-bit g128 v2), %d runs, "
                      "%.2f s each (unpack + fp32 dequant + fp32 GEMM, single thread)" % (ncols, reps, per)}


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
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--all", action="store_true",
                    help="also time every workload and M (per-launch us, GB/s, TFLOP/s)")
    ap.add_argument("--sweep-filter", default="",
                    help="with --all: only the workloads whose name contains this string")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

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
