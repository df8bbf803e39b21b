"""Benchmark of the GGUF block-quantized matmul on GB300.

Workload (one "step"): the L2-defeating decode sweep -- for each weight type
(Q4_K and Q8_0) eight distinct 28672 x 8192 weight buffers (132 MB and 250 MB
each, more than the 129 MB L2) rotated call by call, for activation batches
M in {1, 2, 4, 8} and both QMatMul forms (int8_act: activations quantized per
row inside the launch; f32_act: f32 activations times in-kernel dequantized
weights).  128 qmm_matmul calls per step, inputs resident in HBM.

Printed JSON line: value = weight bytes streamed per second (GB/s, whole
job), roofline of the streaming kernel against the measured HBM copy
bandwidth, the oracle's throughput on the host cores on a bounded sample, an
end-to-end figure through the public API with pinned host buffers (each step
copies its activation batches in and all 128 outputs out), SM clocks sampled during the timed region,
and a per-(type, form, M) breakdown.  A prefill section times the Llama-shaped
GEMMs in both forms (4096 x 4096 and 14336 x 4096 weights, M = 16, 37, 64, 256,
1024) as TOPS, with the tensor work of the three f16 passes against the
measured bf16 peak.

--impl reference times the CPU oracle (the only reference there is: the pages
publish no code) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import qmm_synth  # noqa: E402

METRIC = "decode GEMV weight GB/s (% of HBM peak); prefill int8 GEMM TOPS (% of peak)"
N_DEC, K_DEC = 28672, 8192
BUFFERS = 8
MS = (1, 2, 4, 8)
TYPES = ("q4_k", "q8_0")
MODES = ("int8_act", "f32_act")
WORKLOAD = (f"L2-defeating decode sweep: {BUFFERS} distinct {N_DEC}x{K_DEC} weight buffers per type "
            f"(Q4_K 132 MB, Q8_0 250 MB each) rotated per call; activations M in {list(MS)} x {K_DEC} N(0,1); "
            "int8_act and f32_act; 128 qmm_matmul calls per step")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# source files that define each kernel (its traffic figure is void once they change)
KERNEL_SOURCES = {
    "qmm_gemv_kernel": ["qmm_gemv.cuh", "qmm_device.cuh"],
    "qmm_dmma_kernel": ["qmm_dmma.cuh", "qmm_device.cuh"],
    "qmm_stream_kernel": ["qmm_stream.cuh", "qmm_device.cuh"],
    "qmm_tc_kernel": ["qmm_tc.cuh", "qmm_device.cuh"],
}


def kernel_hash(kernel: str) -> str:
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "gguf_block_quantized_qmatmul_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(cs, f), "rb").read())
    return h.hexdigest()[:16]


def kernel_of(wtype: str, mode: str, M: int) -> str:
    """The streaming kernel qmm_matmul dispatches to for a decode shape (the
    library's own rule): Q8_0 int8_act with M = 1 -> per-thread dp4a GEMV;
    other M <= 16 -> 16-row tensor-core decode kernel (after an activation-
    preparing kernel for large weight matrices); larger M -> the GEMMs."""
    if mode == "int8_act" and wtype == "q8_0" and M <= 1:
        return "qmm_gemv_kernel"
    return "qmm_dmma_kernel" if M <= 16 else "qmm_tc_kernel"


def ncu_traffic(kernel: str):
    """DRAM bytes per algorithmic byte of `kernel` from the committed ncu
    summary (profiles/traffic.json), or None if the kernel changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("source_hash") != kernel_hash(kernel):
        return None
    return d


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        # nvidia-smi takes a moment to start: begin the timed region once it samples
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init(backend: str | None = None):
    """Rank, world and local rank from the launcher's environment; one
    process group when world > 1 (NCCL on GPUs; gloo when asked or when no
    GPU is present, as in the CPU tests of this multi-rank plumbing)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allmax(world, v: float) -> float:
    """The largest v over the ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_sample(rows: int, wq_host: dict, xs: dict):
    """One pass of the step's structure over `rows` weight rows of one buffer
    per type (instead of 8 full buffers).  Returns (weight bytes, seconds)."""
    import oracle
    t0 = time.perf_counter()
    nbytes = 0
    for M in MS:
        for wtype in TYPES:
            wq = wq_host[wtype][:rows]
            for mode in MODES:
                oracle.matmul(wtype, mode, wq, xs[M])
                nbytes += wq.nbytes
    return nbytes, time.perf_counter() - t0


def host_sample_inputs(rows: int):
    """The sampled weight rows, quantized by the oracle (the reference arm may
    not use the CUDA path), and the activations."""
    import oracle
    w = qmm_synth.weights(rows, K_DEC, seed=0)
    wq = {t: oracle.quantize(t, w) for t in TYPES}
    xs = {M: qmm_synth.activations(M, K_DEC) for M in MS}
    return wq, xs


def run_reference(args):
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return
    import oracle
    rows = args.ref_rows
    wq, xs = host_sample_inputs(rows)
    for _ in range(args.warmup):
        oracle_sample(rows, wq, xs)
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b, s = oracle_sample(rows, wq, xs)
        tot_b += b
        tot_s += s
    v = tot_b / tot_s / 1e9
    sample = f"{rows} of {N_DEC} rows of one buffer per type, all M and both forms, per step"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def make_buffers(q, torch, wtype: str, seed0: int):
    cols = torch.from_numpy(qmm_synth.outlier_columns(K_DEC)).cuda()
    out = []
    for b in range(BUFFERS):
        g = torch.Generator(device="cuda").manual_seed(seed0 + b)
        w = torch.randn((N_DEC, K_DEC), generator=g, device="cuda") * 0.02
        w[:, cols] *= 8.0
        out.append(q.quantize_weights(w, wtype))
        del w
    torch.cuda.synchronize()
    return out


def next_types(q, torch, stream, K=K_DEC, N=N_DEC, Ms=(1, 8), reps=10):
    """The weight types beyond the headline pair (Q4_0, Q5_0, Q6_K) on the
    decode shape, both forms: weight GB/s over reps calls rotating two buffers
    of each type (each buffer larger than half of L2; the pair exceeds it)."""
    out = {}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for t in ("q4_0", "q5_0", "q6_k"):
        bufs = []
        for b in range(2):
            g = torch.Generator(device="cuda").manual_seed(500 + b)
            bufs.append(q.quantize_weights(torch.randn((N, K), generator=g, device="cuda") * 0.02, t))
        for M in Ms:
            x = torch.from_numpy(qmm_synth.activations(M, K)).cuda()
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            for mode in MODES:
                ws = torch.empty(max(q.matmul_workspace(t, mode, M, N, K), 16), dtype=torch.uint8, device="cuda")
                for i in range(4):
                    q.matmul(bufs[i % 2], x, t, mode, N=N, out=y, workspace=ws)
                torch.cuda.synchronize()
                ev0.record(stream)
                for i in range(reps):
                    q.matmul(bufs[i % 2], x, t, mode, N=N, out=y, workspace=ws)
                ev1.record(stream)
                torch.cuda.synchronize()
                us = ev0.elapsed_time(ev1) / reps * 1e3
                out[f"{t}/{mode}/M{M}/{N}x{K}"] = {"us_per_call": round(us, 1),
                                                   "weight_GBps": round(bufs[0].numel() / (us * 1e3), 1)}
        del bufs
    return out


def small_configs(q, torch, stream):
    """Latency-bound configurations: one Q8_0 GEMV 576x576 (M=1), the Q4_K
    576x1536 GEMV (M = 1, 2, 4, 8), and the 211-matmul SmolLM2-135M-shaped
    decode step (all Q8_0, M=1), each in both forms.  The step is timed with
    the L2 flushed before every step (a 2 x L2 buffer written, then read back
    so that no dirty line of it is written back inside the timed step):
    eagerly and replayed from a CUDA graph (211 launches), and as one
    qmm_matmul_batch call; then the same step with the weight types of the
    model's Q4_K_M file as one qmm_matmul_batch_typed call."""
    out = {}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def time_calls(fn, reps=200):
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(reps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / reps * 1e3  # us

    for wtype, N, K, Ms in (("q8_0", 576, 576, (1,)), ("q4_k", 576, 1536, (1, 2, 4, 8))):
        wq = q.quantize_weights(torch.from_numpy(qmm_synth.weights(N, K)).cuda(), wtype)
        for M in Ms:
            x = torch.from_numpy(qmm_synth.activations(M, K)).cuda()
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            for mode in MODES:
                us = time_calls(lambda: q.matmul(wq, x, wtype, mode, N=N, out=y))
                out[f"{wtype} {N}x{K} M{M} {mode}"] = {"us_per_call": round(us, 2),
                                                      "weight_GBps": round(wq.numel() / (us * 1e3), 1)}
    # SmolLM2-135M-shaped decode step: 211 Q8_0 matmuls, M = 1
    lins = qmm_synth.smollm2_linears()
    wqs = []
    for i, (_, N, K) in enumerate(lins):
        g = torch.Generator(device="cuda").manual_seed(1000 + i)
        w = torch.randn((N, K), generator=g, device="cuda") * 0.02
        wqs.append((q.quantize_weights(w, "q8_0"), N, K))
    step_bytes = sum(w.numel() for w, _, _ in wqs)
    xs = {K: torch.from_numpy(qmm_synth.activations(1, K)).cuda() for K in (576, 1536)}
    ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, N, _ in wqs]
    flush = torch.empty(2 * 129 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty(1, dtype=torch.float32, device="cuda")

    def flush_l2():
        # write a 2 x L2 buffer, then read it back: L2 then holds clean lines of the
        # flush buffer, so the timed step pays no write-back of the flush's dirty lines
        flush.fill_(1.0)
        sink.copy_(flush.sum().reshape(1))

    for mode in MODES:
        def step():
            for (w, N, K), y in zip(wqs, ys):
                q.matmul(w, xs[K], "q8_0", mode, N=N, out=y)
        step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        res = {}
        for name, fn in (("eager", step), ("graph", graph.replay)):
            tot = 0.0
            reps = 20
            for _ in range(reps + 3):
                flush_l2()
                ev0.record(stream)
                fn()
                ev1.record(stream)
                torch.cuda.synchronize()
                tot += ev0.elapsed_time(ev1)
            ms = tot / (reps + 3)
            res[name] = {"ms_per_step": round(ms, 4), "weight_GBps": round(step_bytes / (ms * 1e6), 1)}
        out[f"smollm2_step_211_matmuls q8_0 M1 {mode} (L2 flushed)"] = res
        # the same step as one qmm_matmul_batch call (one launch for all 211 items),
        # its descriptor table built once; called directly and replayed from a graph
        batch = q.MatmulBatch([(w, xs[K], y) for (w, N, K), y in zip(wqs, ys)], "q8_0", mode)
        batch.run()
        torch.cuda.synchronize()
        bgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(bgraph):
            batch.run()
        torch.cuda.synchronize()
        for name, fn in (("batched", batch.run), ("batched_graph", bgraph.replay)):
            tot = 0.0
            reps = 20
            for _ in range(reps + 3):
                flush_l2()
                ev0.record(stream)
                fn()
                ev1.record(stream)
                torch.cuda.synchronize()
                tot += ev0.elapsed_time(ev1)
            ms = tot / (reps + 3)
            res[name] = {"ms_per_step": round(ms, 4), "weight_GBps": round(step_bytes / (ms * 1e6), 1), "launches": 1}
    out["smollm2_step_weight_bytes"] = step_bytes
    # the same step with the weight types of the model's Q4_K_M file (Q5_0, Q8_0,
    # Q4_K, Q6_K): 211 qmm_matmul calls replayed from a graph, and one
    # qmm_matmul_batch_typed launch (direct and from a graph)
    tl = qmm_synth.smollm2_q4_k_m_linears()
    twq = []
    for i, (_, N, K, t) in enumerate(tl):
        g = torch.Generator(device="cuda").manual_seed(2000 + i)
        twq.append((t, q.quantize_weights(torch.randn((N, K), generator=g, device="cuda") * 0.02, t), N, K))
    tbytes = sum(w.numel() for _, w, _, _ in twq)
    tys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, _, N, _ in twq]
    for mode in MODES:
        def tstep():
            for (t, w, N, K), y in zip(twq, tys):
                q.matmul(w, xs[K], t, mode, N=N, out=y)
        tstep()
        torch.cuda.synchronize()
        tgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tgraph):
            tstep()
        tb = q.MatmulBatchTyped([(t, w, xs[K], y) for (t, w, N, K), y in zip(twq, tys)], mode)
        tb.run()
        torch.cuda.synchronize()
        tbgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tbgraph):
            tb.run()
        torch.cuda.synchronize()
        res = {}
        for name, fn in (("graph", tgraph.replay), ("batched", tb.run), ("batched_graph", tbgraph.replay)):
            tot = 0.0
            reps = 20
            for _ in range(reps + 3):
                flush_l2()
                ev0.record(stream)
                fn()
                ev1.record(stream)
                torch.cuda.synchronize()
                tot += ev0.elapsed_time(ev1)
            ms = tot / (reps + 3)
            res[name] = {"ms_per_step": round(ms, 4), "weight_GBps": round(tbytes / (ms * 1e6), 1),
                         "launches": 1 if name.startswith("batched") else len(twq)}
        out[f"smollm2_step_211_matmuls q4_k_m M1 {mode} (L2 flushed)"] = res
    out["smollm2_q4_k_m_step_weight_bytes"] = tbytes
    assert q.last_device_error() == 0
    return out


def dequant_all_case(q, torch, stream, wq, t, N, K, Ms=(16, 256, 1024)):
    """The dequantize-all serving form as a comparison point: the weights
    dequantized once (the library's dequantize kernel, timed on its own) and
    kept as dense f32 or bf16, then one cuBLAS GEMM per call (f32 with TF32
    off, or bf16 operands with f32 accumulation).  TOPS = 2 M N K / time."""
    res = {}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, reps=10):
        fn()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(reps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / reps

    w32 = torch.empty((N, K), dtype=torch.float32, device="cuda")
    res["dequantize_ms"] = round(timed(lambda: q.dequantize(wq, t, K, out=w32)), 4)
    w16 = w32.to(torch.bfloat16)
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        for M in Ms:
            x = torch.from_numpy(qmm_synth.activations(M, K, outlier_channels=4)).cuda()
            x16 = x.to(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            y16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            ms32 = timed(lambda: torch.matmul(x, w32.t(), out=y))
            ms16 = timed(lambda: torch.matmul(x16, w16.t(), out=y16))
            res[f"M{M}"] = {"f32_gemm_ms": round(ms32, 4), "f32_gemm_TOPS": round(2.0 * M * N * K / ms32 / 1e9, 1),
                            "bf16_gemm_ms": round(ms16, 4), "bf16_gemm_TOPS": round(2.0 * M * N * K / ms16 / 1e9, 1)}
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32
    return res


PREFILL_SHAPES = ((4096, 4096), (14336, 4096))
PREFILL_MS = (16, 37, 64, 256, 1024)
PREFILL_HEADLINE = "q8_0/int8_act/M1024/14336x4096"
PREFILL_HEADLINE_F32 = "q8_0/f32_act/M1024/14336x4096"
PREFILL_HEADLINE_Q4_K = "q4_k/int8_act/M1024/14336x4096"
WARP_MMA_F16_PEAK = 605.0  # TFLOP/s, legacy warp-level f16 MMA on this GPU (register-only probe)


def prefill_kernel(t: str, mode: str, M: int) -> str:
    """The kernel qmm_matmul runs for a prefill shape with K % 256 = 0 (the
    library's dispatch): the Metal form on the three-pass tcgen05 GEMM, up to
    64 rows on the exact-code GEMM with two activation pieces; the CPU form,
    whose bound needs exact integer block sums, on the exact tcgen05 GEMM; up
    to 16 rows, the decode kernel."""
    if M <= 16:
        return "qmm_dmma_kernel"
    if mode == "f32_act" and (M > 64 or t in ("q4_0", "q5_0")):
        return "qmm_tc_kernel"
    return "qmm_tcx_kernel"


def prefill_section(q, torch, stream, hbm_peak, bf16_peak):
    """Config 4: the Llama-shaped prefill GEMMs (4096 x 4096 and 14336 x 4096
    weights; Q8_0, Q4_K at M = 16, 37, 64, 256, 1024, and Q6_K and Q5_0 as
    next types at M = 37, 256, 1024; both forms).  Each point runs calls back to back over distinct quantized
    weight buffers that together exceed twice the L2 (so every call streams
    its weights from HBM), timed with CUDA events over the whole run.
    Reported per point: the kernel; algorithmic TOPS = 2 M N K / t and its
    fraction of the measured bf16 tensor peak (tcgen05 f16 MMAs run at the
    bf16 rate) and, for the warp-MMA kernels, of the legacy warp-level f16
    MMA's rate; weight GB/s and its fraction of the measured HBM bandwidth;
    the roofline time max(2 M N K / peak, bytes / HBM) with bytes = weights +
    x + y, and roofline_frac = roofline time / measured time.  The tcgen05
    GEMM's three f16 passes are reported beside it as tensor_TFLOPs.
    Returns (points, the dequantize-all comparison)."""
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0) or 129 * 1024 * 1024
    points, deq = {}, {}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    K = 4096
    cols = torch.from_numpy(qmm_synth.outlier_columns(K)).cuda()
    for t in ("q8_0", "q4_k", "q6_k", "q5_0"):
        for N, _ in PREFILL_SHAPES:
            wbytes = N * q.row_bytes(t, K)
            nbuf = max(3, -(-2 * l2 // wbytes) + 1)
            bufs = []
            for b in range(nbuf):
                g = torch.Generator(device="cuda").manual_seed(7000 + b)
                w = torch.randn((N, K), generator=g, device="cuda") * 0.02
                w[:, cols] *= 8.0
                bufs.append(q.quantize_weights(w, t))
                del w
            Ms = PREFILL_MS if t in ("q8_0", "q4_k") else (37, 256, 1024)
            for mode in MODES:
                for M in Ms:
                    x = torch.from_numpy(qmm_synth.activations(M, K, outlier_channels=4)).cuda()
                    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
                    wsp = torch.empty(max(q.matmul_workspace(t, mode, M, N, K), 16), dtype=torch.uint8, device="cuda")
                    for i in range(3):
                        q.matmul(bufs[i % nbuf], x, t, mode, N=N, out=y, workspace=wsp)
                    reps = max(2 * nbuf, 12)
                    torch.cuda.synchronize()
                    ev0.record(stream)
                    for i in range(reps):
                        q.matmul(bufs[i % nbuf], x, t, mode, N=N, out=y, workspace=wsp)
                    ev1.record(stream)
                    torch.cuda.synchronize()
                    sec = ev0.elapsed_time(ev1) / reps / 1e3
                    ops = 2.0 * M * N * K
                    nbytes = wbytes + 4.0 * M * K + 4.0 * M * N
                    roof = max(ops / (bf16_peak * 1e12), nbytes / (hbm_peak * 1e9))
                    kern = prefill_kernel(t, mode, M)
                    pt = {"kernel": kern, "us": round(sec * 1e6, 2), "TOPS": round(ops / sec / 1e12, 1),
                          "frac_of_bf16_peak": round(ops / sec / 1e12 / bf16_peak, 4),
                          "weight_GBps": round(wbytes / sec / 1e9, 1),
                          "frac_of_hbm": round(nbytes / sec / 1e9 / hbm_peak, 4),
                          "bound": "tensor" if ops / (bf16_peak * 1e12) > nbytes / (hbm_peak * 1e9) else "hbm",
                          "roofline_us": round(roof * 1e6, 2), "roofline_frac": round(roof / sec, 4),
                          "buffers": nbuf, "launches_per_call": q.matmul_launches(t, mode, M, N, K)}
                    if kern == "qmm_tc_kernel":  # three f16 passes
                        pt["tensor_TFLOPs"] = round(3 * ops / sec / 1e12, 1)
                    else:
                        pt["frac_of_warp_mma_f16_peak"] = round(ops / sec / 1e12 / WARP_MMA_F16_PEAK, 4)
                    points[f"{t}/{mode}/M{M}/{N}x{K}"] = pt
            if t == "q8_0":
                deq[f"{N}x{K}"] = dequant_all_case(q, torch, stream, bufs[0], t, N, K)
            del bufs
            torch.cuda.empty_cache()
    return points, deq


def oracle_configs():
    """The oracle timed on the host cores beside the GPU configurations:
    configs 1 and 2 on one thread (single calls), the SmolLM2-135M-shaped step
    and the prefill shapes on all cores (the prefill on a sample of weight
    rows, scaled to TOPS).  Inputs are synthetic, quantized by the oracle."""
    import oracle
    out = {"cores_all": None, "configs": {}}
    res = out["configs"]

    def timed(fn, min_s=0.2):
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            el = time.perf_counter() - t0
            if el >= min_s:
                return el / n

    oracle.set_num_threads(1)
    try:
        for t, N, K, Ms in (("q8_0", 576, 576, (1,)), ("q4_k", 576, 1536, (1, 2, 4, 8))):
            wq = oracle.quantize(t, qmm_synth.weights(N, K))
            for M in Ms:
                x = qmm_synth.activations(M, K)
                for mode in MODES:
                    s = timed(lambda: oracle.matmul(t, mode, wq, x))
                    res[f"{t} {N}x{K} M{M} {mode}"] = {"us_per_call": round(s * 1e6, 1), "threads": 1}
    finally:
        oracle.set_num_threads(0)
    out["cores_all"] = oracle.num_threads()
    lins = qmm_synth.smollm2_linears()
    wqs = [(oracle.quantize("q8_0", qmm_synth.weights(N, K, seed=1000 + i)), K) for i, (_, N, K) in enumerate(lins)]
    xs = {K: qmm_synth.activations(1, K, seed=K) for K in (576, 1536)}
    for mode in MODES:
        t0 = time.perf_counter()
        for wq, K in wqs:
            oracle.matmul("q8_0", mode, wq, xs[K])
        s = time.perf_counter() - t0
        res[f"smollm2_step_211_matmuls q8_0 M1 {mode}"] = {"ms_per_step": round(s * 1e3, 2),
                                                            "threads": out["cores_all"]}
    tl = qmm_synth.smollm2_q4_k_m_linears()
    twq = [(t, oracle.quantize(t, qmm_synth.weights(N, K, seed=2000 + i)), K) for i, (_, N, K, t) in enumerate(tl)]
    for mode in MODES:
        t0 = time.perf_counter()
        for t, wq, K in twq:
            oracle.matmul(t, mode, wq, xs[K])
        s = time.perf_counter() - t0
        res[f"smollm2_step_211_matmuls q4_k_m M1 {mode}"] = {"ms_per_step": round(s * 1e3, 2),
                                                              "threads": out["cores_all"]}
    rows = 512
    K = 4096
    for t in ("q8_0", "q4_k"):
        wq = oracle.quantize(t, qmm_synth.weights(rows, K, seed=7))
        for mode in MODES:
            for M in PREFILL_MS:
                x = qmm_synth.activations(M, K, outlier_channels=4)
                t0 = time.perf_counter()
                oracle.matmul(t, mode, wq, x)
                s = time.perf_counter() - t0
                res[f"{t}/{mode}/M{M}/prefill K{K}"] = {
                    "TOPS": round(2.0 * M * rows * K / s / 1e12, 4), "sample": f"{rows} weight rows",
                    "threads": out["cores_all"]}
    return out


def run_ours(args):
    import torch

    import gguf_block_quantized_qmatmul_gb300 as q

    world, rank, local = dist_init()
    torch.cuda.set_device(local)
    hbm_peak, bf16_peak, peak_src = peaks()
    stream = torch.cuda.current_stream()

    wqs = {t: make_buffers(q, torch, t, seed0=100 * rank + (0 if t == "q4_k" else 50)) for t in TYPES}
    xs = {M: torch.from_numpy(qmm_synth.activations(M, K_DEC)).cuda() for M in MS}
    ys = {M: torch.empty((M, N_DEC), dtype=torch.float32, device="cuda") for M in MS}
    ws_need = max(q.matmul_workspace(t, m, M, N_DEC, K_DEC) for t in TYPES for m in MODES for M in MS)
    ws = torch.empty(max(ws_need, 16), dtype=torch.uint8, device="cuda")
    wbytes = {t: wqs[t][0].numel() for t in TYPES}

    calls = [(M, t, mode, b) for M in MS for t in TYPES for mode in MODES for b in range(BUFFERS)]

    def call(M, t, mode, b):
        q.matmul(wqs[t][b], xs[M], t, mode, N=N_DEC, out=ys[M], workspace=ws)

    def step():
        for c in calls:
            call(*c)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)

    # The timed region: exactly K steps.  Consecutive calls of one (type, form, M) group
    # (its 8 rotated buffers) run back to back with nothing recorded between them, so
    # each call's grids are scheduled while the previous call finishes (programmatic
    # dependent launch), as in a model's step; an event after each group (on the
    # launching stream) attributes its time to the one kernel the group runs.
    groups = [calls[i:i + BUFFERS] for i in range(0, len(calls), BUFFERS)]
    assert all(len({(M, t, mode) for (M, t, mode, _) in g}) == 1 for g in groups)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(groups) + 1)] for _ in range(args.steps)]
    clocks = Clocks(local)
    clocks.start()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    start.record(stream)
    for s in range(args.steps):
        ev[s][0].record(stream)
        for gi, g in enumerate(groups):
            for c in g:
                call(*c)
            ev[s][gi + 1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    ck = clocks.stop()
    barrier(world)
    elapsed_ms = allmax(world, start.elapsed_time(stop))
    bytes_per_step = sum(wbytes[t] for (_, t, _, _) in calls)
    value = world * bytes_per_step * args.steps / (elapsed_ms / 1e3) / 1e9

    # group durations -> per-kernel roofline and breakdown
    per = {}
    kern = {}  # kernel -> [algorithmic bytes, ms, launches]
    for s in range(args.steps):
        for gi, g in enumerate(groups):
            M, t, mode, _ = g[0]
            d = ev[s][gi].elapsed_time(ev[s][gi + 1])
            ab = len(g) * (wbytes[t] + M * K_DEC * 4 + M * N_DEC * 4)
            k = kern.setdefault(kernel_of(t, mode, M), [0.0, 0.0, 0])
            k[0] += ab
            k[1] += d
            k[2] += len(g)
            per.setdefault((t, mode, M), []).append((len(g) * wbytes[t], d))
    sweep = {f"{t}/{mode}/M{M}": round(sum(b for b, _ in v) / (sum(d for _, d in v) / 1e3) / 1e9, 1)
             for (t, mode, M), v in sorted(per.items())}
    dom = max(kern, key=lambda k: kern[k][1])
    alg_bytes, dur_ms, nl = kern[dom]
    achieved = alg_bytes / (dur_ms / 1e3) / 1e9
    tr = ncu_traffic(dom)
    traffic = None if tr is None else tr["dram_bytes_per_alg_byte"] * alg_bytes / nl
    kernels = {k: {"GBps": round(v[0] / (v[1] / 1e3) / 1e9, 1), "frac": round(v[0] / (v[1] / 1e3) / 1e9 / hbm_peak, 4),
                   "time_share": round(v[1] / sum(x[1] for x in kern.values()), 3), "launches": v[2]}
               for k, v in kern.items()}
    launches = sum(q.matmul_launches(t, mode, M, N_DEC, K_DEC) for (M, t, mode, _) in calls)

    # end to end through the public API with pinned host buffers: each step copies its
    # activation batches in (one copy per M), runs the 128 calls, each into its own
    # slice of one output buffer, and reads all 128 outputs back with one copy
    xh = {M: xs[M].cpu().pin_memory() for M in MS}
    xd = {M: torch.empty_like(xs[M]) for M in MS}
    offs, o = [], 0
    for (M, _, _, _) in calls:
        offs.append(o)
        o += M * N_DEC
    y_all = torch.empty(o, dtype=torch.float32, device="cuda")
    y_host = torch.empty(o, dtype=torch.float32).pin_memory()
    y_views = [y_all[a:a + M * N_DEC].view(M, N_DEC) for a, (M, _, _, _) in zip(offs, calls)]
    h2d = sum(xh[M].numel() * 4 for M in MS)
    d2h = y_host.numel() * 4

    def e2e_step():
        for M in MS:
            xd[M].copy_(xh[M], non_blocking=True)
        for (M, t, mode, b), yv in zip(calls, y_views):
            q.matmul(wqs[t][b], xd[M], t, mode, N=N_DEC, out=yv, workspace=ws)
        y_host.copy_(y_all, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = allmax(world, time.perf_counter() - t0)
    e2e = world * bytes_per_step * args.steps / e2e_s / 1e9

    # prefill (config 4, Llama-shaped, both forms) on weights rotated through buffers
    # that together exceed 2 x L2, with the algorithmic roofline per point
    prefill, prefill_points, dequant_all = {}, {}, {}
    if not args.no_prefill:
        prefill_points, dequant_all = prefill_section(q, torch, stream, hbm_peak, bf16_peak)
        head = prefill_points.get(PREFILL_HEADLINE)
        hf = prefill_points.get(PREFILL_HEADLINE_F32)
        if head:
            prefill = {"point": PREFILL_HEADLINE, "kernel": head["kernel"], "TOPS": head["TOPS"],
                       "frac_of_bf16_peak": head["frac_of_bf16_peak"],
                       "frac_of_warp_mma_f16_peak": head.get("frac_of_warp_mma_f16_peak"),
                       "roofline_frac": head["roofline_frac"], "peak_TFLOPs": bf16_peak,
                       "f32_act_point": PREFILL_HEADLINE_F32, "f32_act_TOPS": hf["TOPS"] if hf else None,
                       "f32_act_frac_of_bf16_peak": hf["frac_of_bf16_peak"] if hf else None,
                       "l2": "weights rotated over distinct buffers totalling > 2 x L2"}
            hk = prefill_points.get(PREFILL_HEADLINE_Q4_K)
            if hk:  # the same int8_act GEMM on the other headline weight type
                prefill.update({"q4_k_point": PREFILL_HEADLINE_Q4_K, "q4_k_TOPS": hk["TOPS"],
                                "q4_k_frac_of_bf16_peak": hk["frac_of_bf16_peak"]})

    small = small_configs(q, torch, stream) if not args.no_small else {}
    nxt = next_types(q, torch, stream) if not args.no_small else {}

    # oracle on the host cores, bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        rows = N_DEC
        wq_h = {t: wqs[t][0][:rows].cpu().numpy() for t in TYPES}
        xs_h = {M: xs[M].cpu().numpy() for M in MS}
        b, s = oracle_sample(rows, wq_h, xs_h)
        cpu = {"value": b / s / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{rows} of {N_DEC} rows of one buffer per type, all M and both forms ({s:.1f} s)"}

    oracle_cfg = oracle_configs() if (rank == 0 and world == 1 and not args.no_cpu) else None

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "s8xs8->s32 (int8_act), f16xf16->f32 (f32_act)",
                "data": "synthetic",
                "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (8 distinct weight buffers per type, "
                           "each >= 132 MB, rotated per call)", "parallelism": f"replicas x{world}"},
                "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                             "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                             "kernel": dom, "peak_source": f"{peak_src} hbm_gbs",
                             "alg_bytes": "weights + x f32 + y f32 per call; a call's duration includes its "
                                          "activation-preparing launch",
                             "durations": "CUDA events in the timed region after each group of 8 calls "
                                          "of one type, form and M (one kernel per group)"},
                "kernels": kernels,
                "dequantize_all": dequant_all,
                "cpu_baseline": cpu,
                "e2e": {"value": round(e2e, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": launches * args.steps,
                "clocks": ck, "sweep_GBps": sweep, "prefill": prefill, "prefill_points": prefill_points,
                "small_configs": small, "next_types": nxt, "oracle_configs": oracle_cfg}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_case(spec: str, launches: int):
    """A few launches of one configuration, for ncu: spec = wtype:mode:M:N:K, or
    smollm2_batch:wtype:mode for the 211-item SmolLM2-135M decode step as one
    qmm_matmul_batch call (M = 1)."""
    import torch

    import gguf_block_quantized_qmatmul_gb300 as q
    if spec.startswith("q4_k_m_batch:"):
        _, mode = spec.split(":")
        items = []
        xs = {K: torch.from_numpy(qmm_synth.activations(1, K)).cuda() for K in (576, 1536)}
        for i, (_, N, K, t) in enumerate(qmm_synth.smollm2_q4_k_m_linears()):
            g = torch.Generator(device="cuda").manual_seed(2000 + i)
            w = q.quantize_weights(torch.randn((N, K), generator=g, device="cuda") * 0.02, t)
            items.append((t, w, xs[K], torch.empty((1, N), dtype=torch.float32, device="cuda")))
        batch = q.MatmulBatchTyped(items, mode)
        for _ in range(launches):
            batch.run()
        torch.cuda.synchronize()
        assert q.last_device_error() == 0
        print(f"profile case {spec}: {launches} launches ok")
        return
    if spec.startswith("smollm2_batch:"):
        _, wtype, mode = spec.split(":")
        wqs = []
        for i, (_, N, K) in enumerate(qmm_synth.smollm2_linears()):
            g = torch.Generator(device="cuda").manual_seed(1000 + i)
            wqs.append((q.quantize_weights(torch.randn((N, K), generator=g, device="cuda") * 0.02, wtype), N, K))
        xs = {K: torch.from_numpy(qmm_synth.activations(1, K)).cuda() for K in (576, 1536)}
        ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _, N, _ in wqs]
        batch = q.MatmulBatch([(w, xs[K], y) for (w, N, K), y in zip(wqs, ys)], wtype, mode)
        for _ in range(launches):
            batch.run()
        torch.cuda.synchronize()
        assert q.last_device_error() == 0
        print(f"profile case {spec}: {launches} launches ok")
        return
    wtype, mode, M, N, K = spec.split(":")
    M, N, K = int(M), int(N), int(K)
    g = torch.Generator(device="cuda").manual_seed(0)
    w = torch.randn((N, K), generator=g, device="cuda") * 0.02
    wq = q.quantize_weights(w, wtype)
    del w
    x = torch.from_numpy(qmm_synth.activations(M, K, outlier_channels=4 if M >= 16 else 0)).cuda()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    need = q.matmul_workspace(wtype, mode, M, N, K)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    for _ in range(launches):
        q.matmul(wq, x, wtype, mode, N=N, out=y, workspace=ws)
    torch.cuda.synchronize()
    assert q.last_device_error() == 0
    print(f"profile case {spec}: {launches} launches ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=4096)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-small", action="store_true")
    ap.add_argument("--profile", default=None, help="wtype:mode:M:N:K, smollm2_batch:wtype:mode or q4_k_m_batch:mode -- run a few launches for ncu and exit")
    ap.add_argument("--launches", type=int, default=4)
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args.profile, args.launches)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
