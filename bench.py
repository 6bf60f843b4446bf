"""Benchmark of the quantized-linear hot path on GB300.

Headline workload (the configuration the metric is quoted on): the W4A16
decode GEMM at the Llama-3.1-8B MLP shape, K = 4096, N = 14336, activations
bf16 M in {1, 4, 16} ~ N(0,1) with 1% channels x20, weights N(0, 0.02)
quantized to symmetric INT4 with one bf16 scale per 128 along K.

One step = one decode pass over 8 distinct weight copies (think 8 layers) at
each of M = 1, 4 and 16: 24 GEMM launches, 8 x 30.3 MB = 242 MB of weights,
more than L2 (so every step streams its weights from HBM; no flush needed).

value  = algorithmic bytes of the step (packed weights + scales + A + Y) / time,
         GB/s, inputs resident in HBM, CUDA events on the launching stream.
e2e    = the same metric through the public API with host buffers: per step the
         activations of the three batch sizes are copied in from pinned host memory,
         the same 24 qz_gemm_w4a16 calls run eagerly, and all 24 outputs are copied
         back to pinned host memory, inside the timed region.
Secondary measurements of the other rows (quantizers, KV write, FP8/NVFP4/MXFP4
GEMMs, the Qwen3-0.6B decode step) are reported beside the headline under
"rows", each timed on its own with CUDA events.

`--impl reference` times the CPU oracle (single-threaded C, test
infrastructure) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16 decode GEMM HBM GB/s; FP8/NVFP4 GEMM TFLOPS; % of GB300 roofline"
K_DIM, N_DIM = 4096, 14336
MS = (1, 4, 16)
COPIES = 8
WORKLOAD = "W4A16 decode GEMM, Llama-3.1-8B MLP 4096x14336, INT4 g128 bf16 scales, M in {1,4,16}"


# ------------------------------------------------------------------ shared

def step_bytes(M: int, K: int = K_DIM, N: int = N_DIM) -> int:
    """Algorithmic bytes of one W4A16 GEMM: packed INT4 weights, bf16 scales, A, Y."""
    return K * N // 2 + (K // 128) * N * 2 + M * K * 2 + M * N * 2


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current source of the kernel (its file hash is recorded beside the number)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path, encoding="utf-8"):
        f = line.split("#", 1)[0].split()
        if len(f) == 5 and f[0] == kernel and f[1] == workload:
            src = os.path.join(ROOT, "bit_quantized_linear_quantizers_gb300", "csrc", f[3])
            if os.path.exists(src) and hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] == f[4]:
                return float(f[2])
    return None


def dist_setup(n_gpus: int):
    """(rank, world, local_rank). One process per GPU under torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("QZ_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
        return dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def reduce_max(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- GPU arm

class Timer:
    """Kernel time per call: `reps` calls captured in one CUDA graph on the launching
    stream, replayed `replays` (>= 20) times after warm-up, each replay timed with CUDA
    events on that stream. Returns the median over the replays of the time per call;
    `last` keeps the median, the mean and the replay count of the latest measurement."""

    def __init__(self, stream, replays: int = 20):
        import torch
        self.torch = torch
        self.stream = stream
        self.replays = max(20, replays)
        self.last = {}

    def __call__(self, fn, reps: int, warm: int = 3) -> float:
        """fn(i) runs call i; rows rotate i over input copies whose total exceeds L2."""
        torch = self.torch
        with torch.cuda.stream(self.stream):
            fn(0)                                      # first call outside capture (sets attributes)
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(reps):
                fn(i)
        with torch.cuda.stream(self.stream):
            for _ in range(warm):
                g.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(self.replays + 1)]
        with torch.cuda.stream(self.stream):
            ev[0].record(self.stream)
            for r in range(self.replays):
                g.replay()
                ev[r + 1].record(self.stream)
        torch.cuda.synchronize()
        per_call = [ev[r].elapsed_time(ev[r + 1]) * 1e3 / reps for r in range(self.replays)]
        self.last = {"median_us": statistics.median(per_call), "mean_us": statistics.fmean(per_call),
                     "replays": self.replays, "calls_per_replay": reps}
        return self.last["median_us"]


def gpu_arm(args, rank, world, local_rank):
    import numpy as np
    import torch

    import bit_quantized_linear_quantizers_gb300 as qz
    import synthetic as syn

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    pk = peaks()

    # ---- inputs (seeded, generated once on the host, resident in HBM)
    _, w = syn.w4a16_decode_inputs(M=1, seed=0)
    with torch.cuda.stream(stream):
        qw, sc, _ = qz.qz_quantize_int4_g128(torch.from_numpy(w).to(dev))
    stream.synchronize()
    del w
    weights = [(qw.clone(), sc.clone()) for _ in range(COPIES)]
    del qw, sc
    # The e2e step's inputs live in one contiguous buffer (device and pinned host): one
    # copy in per step. Its outputs live in one buffer ordered by weight copy, so the
    # outputs of the first half of the weight copies are one contiguous range: they go
    # back on a second stream while the second half computes, the rest after it.
    acts, outs, outs_all = {}, {}, {}
    n_a, per_copy = sum(M * K_DIM for M in MS), sum(M * N_DIM for M in MS)
    dev_a = torch.empty(n_a, dtype=torch.bfloat16, device=dev)
    host_a = torch.empty(n_a, dtype=torch.bfloat16).pin_memory()
    dev_y = torch.empty(COPIES * per_copy, dtype=torch.bfloat16, device=dev)
    host_y = torch.empty(COPIES * per_copy, dtype=torch.bfloat16).pin_memory()
    oa = oy = 0
    for M in MS:
        a_bits, _ = syn.w4a16_decode_inputs(M=M, seed=0, N=128)      # same A recipe; tiny W discarded
        a_t = torch.from_numpy(a_bits.view(np.int16)).view(torch.bfloat16)
        host_a[oa:oa + M * K_DIM].copy_(a_t.reshape(-1))
        acts[M] = dev_a[oa:oa + M * K_DIM].view(M, K_DIM)
        acts[M].copy_(a_t)
        outs[M] = torch.empty((M, N_DIM), dtype=torch.bfloat16, device=dev)
        outs_all[M] = [dev_y[i * per_copy + oy:i * per_copy + oy + M * N_DIM].view(M, N_DIM) for i in range(COPIES)]
        oa, oy = oa + M * K_DIM, oy + M * N_DIM
    half = (COPIES // 2) * per_copy
    copy_stream = torch.cuda.Stream(device=dev)
    ev_half, ev_back = torch.cuda.Event(), torch.cuda.Event()

    def step():
        for i in range(COPIES):
            q, s = weights[i]
            for M in MS:
                qz.qz_gemm_w4a16(acts[M], q, s, Y=outs[M], stream=stream)

    def step_e2e():
        # the step's inputs in (one pinned copy), the same 24 calls, every GEMM's
        # output back to pinned host memory: the first half's outputs on copy_stream
        # while the second half computes, the rest on the stream; the stream then waits
        # for copy_stream, so the step ends when all its outputs are on the host (and
        # the next step's GEMMs cannot overwrite outputs still being read)
        dev_a.copy_(host_a, non_blocking=True)
        for i in range(COPIES):
            if i == COPIES // 2:
                ev_half.record(stream)
                copy_stream.wait_event(ev_half)
                with torch.cuda.stream(copy_stream):
                    host_y[:half].copy_(dev_y[:half], non_blocking=True)
                ev_back.record(copy_stream)
            q, s = weights[i]
            for M in MS:
                qz.qz_gemm_w4a16(acts[M], q, s, Y=outs_all[M][i], stream=stream)
        host_y[half:].copy_(dev_y[half:], non_blocking=True)
        stream.wait_event(ev_back)

    bytes_per_step = COPIES * sum(step_bytes(M) for M in MS)
    launches_per_step = COPIES * len(MS)

    # ---- the step as one CUDA graph (24 launches, no host overhead between them)
    with torch.cuda.stream(stream):
        step()                                         # first calls outside capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()

    # ---- warm-up, then exactly K timed steps between barriers + synchronize
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    t_ms = ev0.elapsed_time(ev1)
    t_ms = reduce_max(t_ms, world, dev)
    ms_per_step = t_ms / args.steps
    value = world * bytes_per_step * args.steps / (t_ms * 1e-3) / 1e9

    # ---- e2e through the public API with pinned host buffers
    with torch.cuda.stream(stream):
        for _ in range(2):
            step_e2e()
    torch.cuda.synchronize()
    barrier(world)
    e_steps = max(3, args.steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e_steps):
            step_e2e()
        e1.record(stream)
    torch.cuda.synchronize()
    wall_s = reduce_max(time.perf_counter() - w0, world, dev)
    te_ms = reduce_max(e0.elapsed_time(e1), world, dev)
    e2e_value = world * bytes_per_step * e_steps / (te_ms * 1e-3) / 1e9
    e2e_wall = world * bytes_per_step * e_steps / wall_s / 1e9
    h2d = host_a.numel() * host_a.element_size()
    d2h = host_y.numel() * host_y.element_size()

    # ---- roofline of the dominant kernel: w4a16_bulk_kernel (M <= 8 tokens, two thirds of
    # the step's launches). Each M is timed on its own as a CUDA graph of 200 launches
    # over the rotating weight copies, CUDA events on the launching stream; the roofline
    # object is the M = 1 decode case, per_M lists every M (M = 16 runs w4a16_kernel).
    timer = Timer(stream)
    per_m = {}
    for M in MS:
        def one(i, M=M):
            q, s = weights[i % COPIES]
            qz.qz_gemm_w4a16(acts[M], q, s, Y=outs[M], stream=stream)
        us = timer(one, reps=200, warm=10)
        per_m[M] = {"kernel": "w4a16_bulk_kernel" if M <= 8 else "w4a16_kernel", "us": round(us, 3),
                    "us_mean": round(timer.last["mean_us"], 3), "replays": timer.last["replays"],
                    "algorithmic_bytes": step_bytes(M), "gbps": round(step_bytes(M) / us / 1e3, 1),
                    "frac_of_hbm": round(step_bytes(M) / us / 1e3 / pk["hbm_gbs"], 4)}
    achieved = per_m[1]["gbps"]
    roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": kernel_traffic("w4a16_bulk_kernel", "llama_mlp_M1"),
                "kernel": "w4a16_bulk_kernel", "workload": "M=1, K=4096, N=14336",
                "peak_source": pk["source"], "algorithmic_bytes_per_launch": step_bytes(1),
                "avg_launch_us": per_m[1]["us"],
                "step_avg_launch_us": round(t_ms * 1e3 / (args.steps * launches_per_step), 3), "per_M": per_m}

    rows = {}
    if not args.no_rows:
        rows = secondary_rows(qz, syn, stream, dev, pk, set(args.rows.split(",")))

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int4xbf16->f32acc", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": list(MS), "K": K_DIM, "N": N_DIM, "weight_copies": COPIES,
                   "l2": "inputs larger than L2 (8 rotating weight copies, 242 MB)",
                   "parallelism": f"replicas{world}"},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "host_wall_value": round(e2e_wall, 1),
                "timing": "value: CUDA events on the stream; host_wall_value: host clock around the same "
                          "steps, synchronised on both sides (includes enqueue cost)"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roofline,
        "clocks": clk.summary(),
        "rows": rows,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def secondary_rows(qz, syn, stream, dev, pk, which):
    """The other hot-path rows, each timed on its own (CUDA events, inputs resident).
    `which` selects among fp8 (config 3), fp4 (config 4), roundtrip (config 1), kv and
    qwen (config 5)."""
    import numpy as np
    import torch

    timer = Timer(stream)
    rows = {}
    ws = qz.Workspace(dev)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    fp8_peak = 2.0 * pk["bf16_tflops"]          # FP8 dense = 2 x bf16 (nominal 4.5 / 2.25 PF)
    fp4_peak = 6.0 * pk["bf16_tflops"]          # FP4 dense = 6 x bf16 (nominal 13.5 / 2.25 PF)

    q = {}
    if "fp8" in which:
        fp8_rows(qz, syn, stream, dev, pk, timer, ws, bf, rows, q, fp8_peak)
    if "fp4" in which:
        fp4_rows(qz, syn, stream, dev, pk, timer, ws, bf, rows, q, fp4_peak)
    if "roundtrip" in which:
        roundtrip_rows(qz, syn, dev, timer, ws, rows, stream)
    if "kv" in which:
        kv_rows(qz, syn, stream, pk, timer, ws, bf, q)
    if q:
        rows["quantizers"] = q
    if "qwen" in which:
        rows["qwen3_decode_step"] = qwen3_step(qz, syn, stream, dev, pk, timer, ws)
    if "next" in which:
        rows["variants"] = next_rows(qz, syn, stream, dev, pk, timer, ws, bf, rows)
    return rows


def copies_for(nbytes: int, l2_bytes: int = 126 << 20) -> int:
    """Copies of an input of nbytes needed for the copies together to exceed 2 x L2."""
    return max(2, -(-2 * l2_bytes // max(1, nbytes)))


def fp8_rows(qz, syn, stream, dev, pk, timer, ws, bf, rows, q, fp8_peak):
    import torch
    # config 3: FP8 1x128 activations, 128x128 weights, block-scaled GEMM
    a, bt = syn.fp8_block_gemm_inputs(seed=0)
    a_d, bt_d = bf(a), bf(bt)
    del a, bt
    M3, K3 = a_d.shape
    N3 = bt_d.shape[0]
    na = copies_for(a_d.numel() * 3)
    A = [a_d] + [a_d.clone() for _ in range(na - 1)]
    outa = [qz.qz_quantize_fp8(x, qz.FP8_GROUP_1x128, stream=stream)[:2] for x in A]
    us = timer(lambda i: qz.qz_quantize_fp8(A[i % na], qz.FP8_GROUP_1x128, codes=outa[i % na][0],
                                            scales=outa[i % na][1], stream=stream), 4 * na)
    by = M3 * K3 * 2 + M3 * K3 + M3 * (K3 // 128) * 4
    q["fp8_1x128_A_2048x4096_bf16"] = {"us": round(us, 2), "gbps": round(by / us / 1e3, 1),
                                       "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3)}
    nb = copies_for(bt_d.numel() * 3)
    B = [bt_d] + [bt_d.clone() for _ in range(nb - 1)]
    outb = [qz.qz_quantize_fp8(x, qz.FP8_BLOCK_128x128, stream=stream)[:2] for x in B]
    us = timer(lambda i: qz.qz_quantize_fp8(B[i % nb], qz.FP8_BLOCK_128x128, codes=outb[i % nb][0],
                                            scales=outb[i % nb][1], stream=stream), 4 * nb)
    by = N3 * K3 * 2 + N3 * K3 + (N3 // 128) * (K3 // 128) * 4
    q["fp8_128x128_Bt_14336x4096_bf16"] = {"us": round(us, 2), "gbps": round(by / us / 1e3, 1),
                                           "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3)}
    del A, B
    try:
        # GEMM operands rotate over copies (A + B codes exceed 2 x L2 together)
        ng = copies_for(M3 * K3 + N3 * K3 + M3 * N3 * 2)
        ops = [(outa[i % len(outa)][0], outa[i % len(outa)][1], outb[i % len(outb)][0], outb[i % len(outb)][1])
               for i in range(ng)]
        ys = [torch.empty((M3, N3), dtype=torch.bfloat16, device=dev) for _ in range(ng)]
        us = timer(lambda i: qz.qz_gemm_fp8_block(*ops[i % ng], Y=ys[i % ng], ws=ws, stream=stream), 4 * ng)
        fl = 2.0 * M3 * N3 * K3
        rows["fp8_block_gemm_2048x14336x4096"] = {"us": round(us, 2), "tflops": round(fl / us / 1e6, 1),
                                                  "peak_tflops": fp8_peak,
                                                  "frac": round(fl / us / 1e6 / fp8_peak, 4)}
    except qz.QZError as e:
        rows["fp8_block_gemm_2048x14336x4096"] = {"unavailable": str(e)}


def fp4_rows(qz, syn, stream, dev, pk, timer, ws, bf, rows, q, fp4_peak):
    import torch
    # config 4: NVFP4 / MXFP4 quantize + GEMM
    a, bt = syn.fp4_gemm_inputs(seed=0)
    a_d, bt_d = bf(a), bf(bt)
    del a, bt
    M4, K4 = a_d.shape
    N4 = bt_d.shape[0]
    na = copies_for(a_d.numel() * 2)
    A = [a_d] + [a_d.clone() for _ in range(na - 1)]
    nvA = [qz.qz_quantize_nvfp4(x, ws=ws, stream=stream)[:3] for x in A]
    mxA = [qz.qz_quantize_mxfp4(x, stream=stream)[:2] for x in A]
    nvB = qz.qz_quantize_nvfp4(bt_d, ws=ws, stream=stream)[:3]
    mxB = qz.qz_quantize_mxfp4(bt_d, stream=stream)[:2]
    us = timer(lambda i: qz.qz_quantize_nvfp4(A[i % na], codes=nvA[i % na][0], scale_e4m3=nvA[i % na][1],
                                              global_scale=nvA[i % na][2], ws=ws, stream=stream), 4 * na)
    by = M4 * K4 * 2 + M4 * K4 // 2 + M4 * K4 // 16 + 4
    q["nvfp4_A_8192x4096_bf16"] = {"us": round(us, 2), "gbps": round(by / us / 1e3, 1),
                                   "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3)}
    us = timer(lambda i: qz.qz_quantize_mxfp4(A[i % na], codes=mxA[i % na][0], scale_e8m0=mxA[i % na][1],
                                              stream=stream), 4 * na)
    by = M4 * K4 * 2 + M4 * K4 // 2 + M4 * K4 // 32
    q["mxfp4_A_8192x4096_bf16"] = {"us": round(us, 2), "gbps": round(by / us / 1e3, 1),
                                   "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3)}
    del A
    fl = 2.0 * M4 * N4 * K4
    # the na copies of A's codes (plus B and the output) exceed 2 x L2 together
    ys = [torch.empty((M4, N4), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    for name, fn in (("nvfp4_gemm_8192x4096x4096",
                      lambda i: qz.qz_gemm_nvfp4(*nvA[i % na], *nvB, Y=ys[i % 2], ws=ws, stream=stream)),
                     ("mxfp4_gemm_8192x4096x4096",
                      lambda i: qz.qz_gemm_mxfp4(*mxA[i % na], *mxB, Y=ys[i % 2], ws=ws, stream=stream))):
        try:
            us = timer(fn, 4 * na)
            rows[name] = {"us": round(us, 2), "tflops": round(fl / us / 1e6, 1), "peak_tflops": fp4_peak,
                          "frac": round(fl / us / 1e6 / fp4_peak, 4)}
        except qz.QZError as e:
            rows[name] = {"unavailable": str(e)}
    # f1 for NVFP4: the GEMM's output leaves as NVFP4 codes + block scales (tensor amax
    # given: the plain GEMM's own output amax), against the GEMM then the quantizer
    if "nvfp4_gemm_8192x4096x4096" in rows and "us" in rows["nvfp4_gemm_8192x4096x4096"]:
        with torch.cuda.stream(stream):
            qz.qz_gemm_nvfp4(*nvA[0], *nvB, Y=ys[0], ws=ws, stream=stream)
            amax = ys[0].float().abs().max().reshape(1)
            yq = qz.qz_gemm_nvfp4_quant(*nvA[0], *nvB, amax, ws=ws, stream=stream)
            sep = qz.qz_quantize_nvfp4(ys[1], global_amax_in=amax, stream=stream)[:3]
        us_fused = timer(lambda i: qz.qz_gemm_nvfp4_quant(*nvA[i % na], *nvB, amax, y_codes=yq[0], y_scales=yq[1],
                                                          y_global=yq[2], ws=ws, stream=stream), 4 * na)

        def separate(i):
            qz.qz_gemm_nvfp4(*nvA[i % na], *nvB, Y=ys[1], ws=ws, stream=stream)
            qz.qz_quantize_nvfp4(ys[1], codes=sep[0], scale_e4m3=sep[1], global_scale=sep[2], global_amax_in=amax,
                                 stream=stream)
        us_sep = timer(separate, 4 * na)
        rows["nvfp4_gemm_with_nvfp4_output_8192x4096x4096"] = {
            "fused_us": round(us_fused, 2), "gemm_then_quantizer_us": round(us_sep, 2),
            "tflops_fused": round(fl / us_fused / 1e6, 1), "frac_of_fp4_peak_fused": round(fl / us_fused / 1e6 / fp4_peak, 4),
            "hbm_bytes_saved_per_call": M4 * N4 * 2 * 2,
            "note": "fused: NVFP4 codes + block scales with a given tensor amax; separate: bf16 output written, "
                    "read back and quantized with the same amax"}
    if "mxfp4_gemm_8192x4096x4096" in rows and "us" in rows["mxfp4_gemm_8192x4096x4096"]:
        with torch.cuda.stream(stream):
            yq = qz.qz_gemm_mxfp4_quant(*mxA[0], *mxB, ws=ws, stream=stream)
            sep = qz.qz_quantize_mxfp4(ys[1], stream=stream)[:2]
        us_fused = timer(lambda i: qz.qz_gemm_mxfp4_quant(*mxA[i % na], *mxB, y_codes=yq[0], y_e8m0=yq[1], ws=ws,
                                                          stream=stream), 4 * na)

        def separate_mx(i):
            qz.qz_gemm_mxfp4(*mxA[i % na], *mxB, Y=ys[1], ws=ws, stream=stream)
            qz.qz_quantize_mxfp4(ys[1], codes=sep[0], scale_e8m0=sep[1], stream=stream)
        us_sep = timer(separate_mx, 4 * na)
        rows["mxfp4_gemm_with_mxfp4_output_8192x4096x4096"] = {
            "fused_us": round(us_fused, 2), "gemm_then_quantizer_us": round(us_sep, 2),
            "tflops_fused": round(fl / us_fused / 1e6, 1), "frac_of_fp4_peak_fused": round(fl / us_fused / 1e6 / fp4_peak, 4),
            "hbm_bytes_saved_per_call": M4 * N4 * 2 * 2,
            "note": "fused: MXFP4 codes + E8M0 scales; separate: bf16 output written, read back and quantized"}
    del a_d, bt_d


def roundtrip_rows(qz, syn, dev, timer, ws, rows, stream):
    import torch
    # config 1: the six quantizer paths on the 1024 x 1024 fp32 weight (4 MiB, launch-bound: us);
    # 128 copies rotate so that each call reads its input from HBM
    x0 = torch.from_numpy(syn.quant_roundtrip_input(seed=0)).to(dev)
    n = copies_for(x0.numel() * 4)
    X = [x0] + [x0.clone() for _ in range(n - 1)]
    c1 = {}
    for nm, g in (("fp8_per_tensor", 0), ("fp8_per_row", 1), ("fp8_128x128", 2), ("fp8_1x128", 3)):
        outs = [qz.qz_quantize_fp8(x, g, dequant=True, ws=ws, stream=stream) for x in X]
        c1[nm] = round(timer(lambda i, g=g, outs=outs: qz.qz_quantize_fp8(
            X[i % n], g, codes=outs[i % n][0], scales=outs[i % n][1], dequant=outs[i % n][2], ws=ws,
            stream=stream), 2 * n), 2)
    outs = [qz.qz_quantize_mxfp4(x, dequant=True, stream=stream) for x in X]
    c1["mxfp4"] = round(timer(lambda i: qz.qz_quantize_mxfp4(
        X[i % n], codes=outs[i % n][0], scale_e8m0=outs[i % n][1], dequant=outs[i % n][2], stream=stream), 2 * n), 2)
    outs = [qz.qz_quantize_nvfp4(x, dequant=True, ws=ws, stream=stream) for x in X]
    c1["nvfp4"] = round(timer(lambda i: qz.qz_quantize_nvfp4(
        X[i % n], codes=outs[i % n][0], scale_e4m3=outs[i % n][1], global_scale=outs[i % n][2],
        dequant=outs[i % n][3], ws=ws, stream=stream), 2 * n), 2)
    outs = [qz.qz_quantize_int4_g128(x, dequant=True, stream=stream) for x in X]
    c1["int4_g128"] = round(timer(lambda i: qz.qz_quantize_int4_g128(
        X[i % n], qweight=outs[i % n][0], scale_bf16=outs[i % n][1], dequant=outs[i % n][2], stream=stream),
        2 * n), 2)
    rows["quantize_roundtrip_1024x1024_f32_us"] = c1


def kv_rows(qz, syn, stream, pk, timer, ws, bf, q):
    # config 5: FP8 KV write of K, V bf16 [1, 8, 4096, 128] (8 MiB each), rotating copies
    k, v = syn.kv_cache_inputs(seed=0)
    k_d, v_d = bf(k), bf(v)
    n = copies_for(k.size * 2 * 3)
    KV = [(k_d, v_d)] + [(k_d.clone(), v_d.clone()) for _ in range(n - 1)]
    outs = [qz.qz_kv_write_fp8(a, b, ws=ws, stream=stream) for a, b in KV]
    us = timer(lambda i: qz.qz_kv_write_fp8(*KV[i % n], k_codes=outs[i % n][0], v_codes=outs[i % n][1],
                                            k_scale=outs[i % n][2], v_scale=outs[i % n][3], ws=ws,
                                            stream=stream), 2 * n)
    by = 2 * (k.size * 2 + k.size) + 8
    q["kv_write_fp8_2x8x4096x128_bf16"] = {"us": round(us, 2), "gbps": round(by / us / 1e3, 1),
                                           "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3)}


def qwen3_step(qz, syn, stream, dev, pk, timer, ws):
    """Config 5: one decode step of a random-init Qwen3-0.6B-shaped decoder at 64
    tokens, all 196 linears (a) in W4A16 as one grouped launch and (b) in NVFP4 as
    grouped launches over prepared weight scales; the activations' NVFP4 quantization
    timed apart, per linear and as one grouped call (two launches for all 196)."""
    import numpy as np
    import torch
    probs, nv_probs, nv_acts = [], [], []
    wbytes = nvbytes = 0
    for layer, name, A, w in syn.qwen3_decode_linears(layers=28, tokens=64, seed=0):
        K, N = w.shape
        with torch.cuda.stream(stream):
            w_d = torch.from_numpy(w).to(dev)
            qw, sc, _ = qz.qz_quantize_int4_g128(w_d, stream=stream)
            bt = w_d.t().contiguous().to(torch.bfloat16)                  # weights as B^T [N, K]
            cb, sb, gb, _ = qz.qz_quantize_nvfp4(bt, ws=ws, stream=stream)
            sbp = qz.qz_prepare_fp4_scales(sb, K, nv=True, stream=stream)
        a_d = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).to(dev)
        Y = torch.empty((64, N), dtype=torch.bfloat16, device=dev)
        probs.append((a_d, qw, sc, Y))
        wbytes += K * N // 2 + (K // 128) * N * 2 + 64 * K * 2 + 64 * N * 2
        with torch.cuda.stream(stream):
            ca, sa, ga, _ = qz.qz_quantize_nvfp4(a_d, ws=ws, stream=stream)
        Yn = torch.empty((64, N), dtype=torch.bfloat16, device=dev)
        nv_probs.append((ca, sa, ga, cb, sbp, gb, Yn))
        nv_acts.append((a_d, ca, sa, ga))
        nvbytes += N * K // 2 + N * K // 16 + 64 * K // 2 + 64 * K // 16 + 64 * N * 2 + 8
        stream.synchronize()
        del w_d, bt, sb
    us = timer(lambda i: qz.qz_gemm_w4a16_grouped(probs, stream=stream), 20)
    out = {"w4a16_grouped_196_linears_us": round(us, 2), "w4a16_gbps": round(wbytes / us / 1e3, 1),
           "w4a16_frac_of_hbm": round(wbytes / us / 1e3 / pk["hbm_gbs"], 3)}
    nws = qz.Workspace(dev)
    us = timer(lambda i: qz.qz_gemm_nvfp4_grouped(nv_probs, ws=nws, stream=stream), 20)
    out.update({"nvfp4_grouped_196_linears_us": round(us, 2), "nvfp4_gbps": round(nvbytes / us / 1e3, 1),
                "nvfp4_frac_of_hbm": round(nvbytes / us / 1e3 / pk["hbm_gbs"], 3),
                "nvfp4_bytes": nvbytes})

    def quant_all(i):
        for a_d, ca, sa, ga in nv_acts:
            qz.qz_quantize_nvfp4(a_d, codes=ca, scale_e4m3=sa, global_scale=ga, ws=ws, stream=stream)
    us = timer(quant_all, 3)
    out["nvfp4_activation_quant_per_linear_196_calls_us"] = round(us, 2)
    xs = [a for a, _, _, _ in nv_acts]
    outs = [(ca, sa, ga) for _, ca, sa, ga in nv_acts]
    gws = qz.Workspace(dev)
    us = timer(lambda i: qz.qz_quantize_nvfp4_grouped(xs, outs=outs, ws=gws, stream=stream), 20)
    out["nvfp4_activation_quant_grouped_us"] = round(us, 2)

    # the whole step as one CUDA graph: every linear of the 28 layers plus the FP8 KV write
    # (the NVFP4 GEMMs read the activation codes the grouped quantizer writes in the same graph)
    k, v = syn.kv_cache_inputs(seed=0)
    k_d = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).to(dev)
    v_d = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(dev)
    kws = qz.Workspace(dev)
    kv_out = qz.qz_kv_write_fp8(k_d, v_d, ws=kws, stream=stream)
    kv_bytes = 2 * (k.size * 2 + k.size) + 8

    def kv(i):
        qz.qz_kv_write_fp8(k_d, v_d, k_codes=kv_out[0], v_codes=kv_out[1], k_scale=kv_out[2], v_scale=kv_out[3],
                           ws=kws, stream=stream)

    def step_w4(i):
        qz.qz_gemm_w4a16_grouped(probs, stream=stream)
        kv(i)

    def step_nv(i):
        qz.qz_quantize_nvfp4_grouped(xs, outs=outs, ws=gws, stream=stream)
        qz.qz_gemm_nvfp4_grouped(nv_probs, ws=nws, stream=stream)
        kv(i)
    us = timer(step_w4, 10)
    out["w4a16_step_with_kv_one_graph_us"] = round(us, 2)
    out["w4a16_step_with_kv_frac_of_hbm"] = round((wbytes + kv_bytes) / us / 1e3 / pk["hbm_gbs"], 3)
    act_bytes = sum(x.numel() * 2 + x.numel() // 2 + x.numel() // 16 + 4 for x in xs)
    us = timer(step_nv, 10)
    out["nvfp4_step_with_act_quant_and_kv_one_graph_us"] = round(us, 2)
    out["nvfp4_step_with_act_quant_and_kv_frac_of_hbm"] = round(
        (nvbytes + act_bytes + kv_bytes) / us / 1e3 / pk["hbm_gbs"], 3)
    return out


def next_rows(qz, syn, stream, dev, pk, timer, ws, bf, rows):
    """The variants beyond the base formats: INT4 with zero points and weight-only FP4 at
    the decode shape, the per-head and per-channel-zero-point KV writes, SmoothQuant INT8
    W8A8 at the prefill shape, the FP8 GEMM with its output quantized in the epilogue, and
    W4A16 at prefill batch sizes (against cuBLAS bf16 and the FP8 GEMM)."""
    import numpy as np
    import torch
    out = {}
    fp16_peak = pk["bf16_tflops"]                 # the fp16 tensor rate equals the bf16 one
    fp8_peak = 2.0 * pk["bf16_tflops"]

    # ---- decode shape (Llama-3.1-8B MLP 4096 x 14336): zero points and weight-only FP4
    _, w = syn.w4a16_decode_inputs(M=1, seed=0)
    w_d = torch.from_numpy(w).to(dev)
    del w
    with torch.cuda.stream(stream):
        zq = qz.qz_quantize_int4_g128_zp(w_d, stream=stream)[:3]
        bt = w_d.t().contiguous().to(torch.bfloat16)
        nvw = qz.qz_quantize_nvfp4(bt, ws=ws, stream=stream)[:3]
        mxw = qz.qz_quantize_mxfp4(bt, stream=stream)[:2]
    stream.synchronize()
    del w_d, bt
    zc = [tuple(t.clone() for t in zq) for _ in range(COPIES)]
    nvc = [tuple(t.clone() for t in nvw) for _ in range(COPIES)]
    mxc = [tuple(t.clone() for t in mxw) for _ in range(COPIES)]
    for M in (1, 16):
        a_bits, _ = syn.w4a16_decode_inputs(M=M, seed=0, N=128)
        A = bf(a_bits)
        Y = torch.empty((M, N_DIM), dtype=torch.bfloat16, device=dev)
        io = M * K_DIM * 2 + M * N_DIM * 2
        cases = (
            ("w4a16_zp", K_DIM * N_DIM // 2 + (K_DIM // 128) * N_DIM * 3 + io,
             lambda i: qz.qz_gemm_w4a16_zp(A, *zc[i % COPIES], Y=Y, stream=stream)),
            ("w4a16_nvfp4", K_DIM * N_DIM // 2 + K_DIM * N_DIM // 16 + 4 + io,
             lambda i: qz.qz_gemm_w4a16_nvfp4(A, *nvc[i % COPIES], Y=Y, stream=stream)),
            ("w4a16_mxfp4", K_DIM * N_DIM // 2 + K_DIM * N_DIM // 32 + io,
             lambda i: qz.qz_gemm_w4a16_mxfp4(A, *mxc[i % COPIES], Y=Y, stream=stream)))
        for name, by, fn in cases:
            us = timer(fn, 8 * COPIES)
            out[f"{name}_llama_mlp_M{M}"] = {"us": round(us, 3), "gbps": round(by / us / 1e3, 1),
                                             "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3),
                                             "algorithmic_bytes": by}
    del zc, nvc, mxc

    # ---- KV variants, 2 x [1, 8, 4096, 128] bf16
    k, v = syn.kv_cache_inputs(seed=0)
    n = copies_for(k.size * 2 * 3)
    KV = [(bf(k), bf(v)) for _ in range(n)]
    ph = [qz.qz_kv_write_fp8_per_head(a, b, ws=ws, stream=stream) for a, b in KV]
    us = timer(lambda i: qz.qz_kv_write_fp8_per_head(*KV[i % n], k_codes=ph[i % n][0], v_codes=ph[i % n][1],
                                                     k_scale=ph[i % n][2], v_scale=ph[i % n][3], ws=ws,
                                                     stream=stream), 2 * n)
    by = 2 * (k.size * 2 + k.size) + 2 * 8 * 4
    out["kv_write_fp8_per_head_2x8x4096x128"] = {"us": round(us, 2), "gbps": round(by / us / 1e3, 1),
                                                 "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3)}
    cz = [qz.qz_kv_write_fp8_channel_zp(a, b, ws=ws, stream=stream) for a, b in KV]
    us = timer(lambda i: qz.qz_kv_write_fp8_channel_zp(*KV[i % n], *cz[i % n], ws=ws, stream=stream), 2 * n)
    by = 2 * (k.size * 2 + k.size) + 8 * 128 * 8 + 8 * 4096 * 4
    out["kv_write_fp8_k_channel_zp_v_token_2x8x4096x128"] = {"us": round(us, 2), "gbps": round(by / us / 1e3, 1),
                                                             "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3)}
    del KV, ph, cz

    # ---- SmoothQuant INT8 W8A8 at the prefill shape 2048 x 14336 x 4096
    a, bt = syn.fp8_block_gemm_inputs(seed=0)
    a_d, bt_d = bf(a), bf(bt)
    M3, K3 = a_d.shape
    N3 = bt_d.shape[0]
    with torch.cuda.stream(stream):
        s = qz.qz_smooth_factors(qz.qz_col_amax(a_d, ws=ws, stream=stream), qz.qz_col_amax(bt_d, ws=ws, stream=stream),
                                 stream=stream)
        qa, sa, _ = qz.qz_quantize_int8_rows(a_d, s, qz.SMOOTH_DIVIDE, stream=stream)
        qb, sb, _ = qz.qz_quantize_int8_rows(bt_d, s, qz.SMOOTH_MULTIPLY, stream=stream)
    stream.synchronize()
    na = copies_for(a_d.numel() * 3)
    As = [a_d] + [a_d.clone() for _ in range(na - 1)]
    qas = [(torch.empty_like(qa), torch.empty_like(sa)) for _ in range(na)]
    us = timer(lambda i: qz.qz_quantize_int8_rows(As[i % na], s, qz.SMOOTH_DIVIDE, codes=qas[i % na][0],
                                                  scales=qas[i % na][1], stream=stream), 2 * na)
    by = M3 * K3 * 2 + M3 * K3 + M3 * 4 + K3 * 4
    out["int8_smooth_quantize_A_2048x4096_bf16"] = {"us": round(us, 2), "gbps": round(by / us / 1e3, 1),
                                                    "frac_of_hbm": round(by / us / 1e3 / pk["hbm_gbs"], 3)}
    del As, qas
    ng = copies_for(M3 * K3 + N3 * K3 + M3 * N3 * 2)
    ops = [(qa, sa, qb.clone(), sb) for _ in range(ng)]
    ys = [torch.empty((M3, N3), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    us = timer(lambda i: qz.qz_gemm_int8(*ops[i % ng], Y=ys[i % 2], stream=stream), 2 * ng)
    fl = 2.0 * M3 * N3 * K3
    out["int8_w8a8_gemm_2048x14336x4096"] = {"us": round(us, 2), "tops": round(fl / us / 1e6, 1),
                                             "peak_tflops_fp16_tensor": fp16_peak,
                                             "frac_of_fp16_peak": round(fl / us / 1e6 / fp16_peak, 4)}
    del ops

    # ---- FP8 GEMM with the output quantized in the epilogue, against GEMM + 1x128 quantizer
    ca, sca, _ = qz.qz_quantize_fp8(a_d, qz.FP8_GROUP_1x128, stream=stream)
    cb, scb, _ = qz.qz_quantize_fp8(bt_d, qz.FP8_BLOCK_128x128, stream=stream)
    del a_d, bt_d
    cbs = [cb] + [cb.clone() for _ in range(ng - 1)]
    yq = qz.qz_gemm_fp8_block_quant(ca, sca, cb, scb, stream=stream)
    us_fused = timer(lambda i: qz.qz_gemm_fp8_block_quant(ca, sca, cbs[i % ng], scb, y_codes=yq[0], y_scales=yq[1],
                                                          stream=stream), 2 * ng)
    ysep = torch.empty((M3, N3), dtype=torch.bfloat16, device=dev)
    sep_out = qz.qz_quantize_fp8(ysep, qz.FP8_GROUP_1x128, stream=stream)

    def separate(i):
        qz.qz_gemm_fp8_block(ca, sca, cbs[i % ng], scb, Y=ysep, stream=stream)
        qz.qz_quantize_fp8(ysep, qz.FP8_GROUP_1x128, codes=sep_out[0], scales=sep_out[1], stream=stream)
    us_sep = timer(separate, 2 * ng)
    out["fp8_gemm_with_quantized_output_2048x14336x4096"] = {
        "fused_us": round(us_fused, 2), "gemm_then_quantizer_us": round(us_sep, 2),
        "tflops_fused": round(fl / us_fused / 1e6, 1), "frac_of_fp8_peak_fused": round(fl / us_fused / 1e6 / fp8_peak, 4),
        "hbm_bytes_saved_per_call": M3 * N3 * 2 * 2,
        "note": "fused: codes + scales only; separate: bf16 output written, read back and quantized"}
    del cbs

    # ---- W4A16 at prefill batch sizes: 2048 tokens as 32 slices of 64 through the grouped
    # tcgen05 kernel (same weight, re-read from L2), against cuBLAS bf16 and the FP8 GEMM
    _, wq = syn.w4a16_decode_inputs(M=1, seed=0)
    wq_d = torch.from_numpy(wq).to(dev)
    del wq
    qw, sc, _ = qz.qz_quantize_int4_g128(wq_d, stream=stream)
    wb = wq_d.to(torch.bfloat16)
    del wq_d
    Ap = bf(syn.fp8_block_gemm_inputs(seed=0, N=256)[0])
    Yp = torch.empty((M3, N_DIM), dtype=torch.bfloat16, device=dev)
    slices = [(Ap[i * 64:(i + 1) * 64], qw, sc, Yp[i * 64:(i + 1) * 64]) for i in range(M3 // 64)]
    us_w4 = timer(lambda i: qz.qz_gemm_w4a16_grouped(slices, stream=stream), 4)
    with torch.cuda.stream(stream):
        torch.matmul(Ap, wb, out=Yp)
    us_bf16 = timer(lambda i: torch.matmul(Ap, wb, out=Yp), 4)
    out["w4a16_prefill_2048x14336x4096"] = {
        "w4a16_us": round(us_w4, 2), "w4a16_tflops": round(fl / us_w4 / 1e6, 1),
        "cublas_bf16_us": round(us_bf16, 2), "cublas_bf16_tflops": round(fl / us_bf16 / 1e6, 1),
        "fp8_block_gemm_us": rows.get("fp8_block_gemm_2048x14336x4096", {}).get("us"),
        "note": "W4A16 runs the 2048 tokens as 32 grouped slices of 64 (the kernel's widest token tile)"}
    return out


# ---------------------------------------------------------- CPU baseline

_CPU_CACHE = {}


def _cpu_inputs():
    """The oracle's own INT4 quantization of the workload weight (setup, untimed)."""
    if not _CPU_CACHE:
        import oracle
        import synthetic as syn
        _, w = syn.w4a16_decode_inputs(M=1, seed=0)
        qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
        acts = {M: syn.w4a16_decode_inputs(M=M, seed=0, N=128)[0] for M in MS}
        _CPU_CACHE.update(qw=qw, sc=sc, acts=acts)
    return _CPU_CACHE


def cpu_baseline(budget_s: float = 12.0):
    """The oracle's W4A16 reference (single-threaded C, FP64 accumulation) timed on
    this host on a bounded sample: chunks of 64 output columns at every M in
    {1, 4, 16}, until the time budget is spent. Bytes are counted as for the GPU
    (the sampled columns' share of each GEMM's algorithmic bytes)."""
    with _one_core() as core:
        done_bytes, spent, n_cols = _oracle_w4a16_sample(budget_s)
    return {"value": round(done_bytes / spent / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_cols} of {N_DIM} output columns at each M in {list(MS)} (K={K_DIM}); "
                      f"{spent:.1f} s of single-threaded oracle time",
            "host": {**host_cpu(), "pinned_core": core}}


def _oracle_w4a16_sample(budget_s: float):
    """(algorithmic bytes covered, oracle seconds, output columns) of the oracle's W4A16
    reference run over chunks of 64 output columns at every M until the budget is spent."""
    import numpy as np
    import oracle
    c = _cpu_inputs()
    done_bytes, spent, n_cols = 0.0, 0.0, 0
    while spent < budget_s and n_cols < N_DIM:
        cols = np.arange(n_cols, n_cols + 64)
        for M in MS:
            ii = np.repeat(np.arange(M), cols.size)
            jj = np.tile(cols, M)
            t0 = time.perf_counter()
            oracle.gemm_w4a16(c["acts"][M], c["qw"], c["sc"], ii, jj)
            spent += time.perf_counter() - t0
            done_bytes += step_bytes(M) * cols.size / N_DIM
        n_cols += cols.size
    return done_bytes, spent, n_cols


def host_cpu(cpuinfo: str = "/proc/cpuinfo"):
    """Core count and CPU model of this host: /proc/cpuinfo's model name, or on Arm
    hosts (which list none) the implementer and part numbers of the first core."""
    fields = {}
    try:
        with open(cpuinfo, encoding="utf-8", errors="replace") as f:
            for line in f:
                key, _, val = line.partition(":")
                key, val = key.strip().lower(), val.strip()
                if key and val and key not in fields:
                    fields[key] = val
    except OSError:
        pass
    if "model name" in fields:
        model = fields["model name"]
    elif "cpu part" in fields:
        model = f"implementer {fields.get('cpu implementer', '?')} part {fields['cpu part']}"
    else:
        model = platform.processor() or platform.machine()
    return {"nproc": os.cpu_count(), "cpu": model, "machine": platform.machine()}


class _one_core:
    """Pins this process to one of its allowed cores while the oracle is timed (the
    oracle is single-threaded), restoring the previous affinity afterwards; yields
    the core, or None where affinity cannot be set."""

    def __enter__(self):
        self.prev = None
        try:
            self.prev = os.sched_getaffinity(0)
            core = min(self.prev)
            os.sched_setaffinity(0, {core})
            return core
        except (AttributeError, OSError, ValueError):
            self.prev = None
            return None

    def __exit__(self, *exc):
        if self.prev is not None:
            os.sched_setaffinity(0, self.prev)


def oracle_per_config():
    """Wall time of the oracle (single-threaded C, pinned to one core) per workload: each
    part timed on a bounded sample of its workload, with the share of the full workload
    the sample covers and the time extrapolated to all of it (the oracle's cost is
    linear in the elements it quantizes and in the output points it computes)."""
    import numpy as np
    import oracle
    import synthetic as syn

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    def part(seconds, share, sample):
        return {"seconds": round(seconds, 3), "share": share, "sample": sample,
                "extrapolated_seconds": round(seconds / share, 1)}

    def points(M, N, n, seed):
        rng = np.random.default_rng(seed)
        return rng.integers(0, M, n), rng.integers(0, N, n)

    out = {}
    with _one_core() as core:
        x = syn.quant_roundtrip_input(seed=0)
        out["1_quantize_roundtrip_1024x1024_f32"] = part(timed(lambda: (
            [oracle.quant_fp8(x, g) for g in range(4)], oracle.quant_mxfp4(x), oracle.quant_nvfp4(x),
            oracle.quant_int4_g128(x))), 1.0, "the seven quantizer paths on the whole tensor")
        _, spent, n_cols = _oracle_w4a16_sample(5.0)
        out["2_w4a16_decode_M1_4_16"] = part(spent, n_cols / N_DIM,
                                             f"{n_cols} of {N_DIM} output columns at each M in {list(MS)}")

        a, bt = syn.fp8_block_gemm_inputs(seed=0, M=128, N=256)
        qa, sa, _ = oracle.quant_fp8(a, oracle.FP8_GROUP_1x128, want_deq=False)
        qb, sb, _ = oracle.quant_fp8(bt, oracle.FP8_BLOCK_128x128, want_deq=False)
        ii, jj = points(128, 256, 4096, 3)
        out["3_fp8_quantize_A_2048x4096"] = part(timed(
            lambda: oracle.quant_fp8(a, oracle.FP8_GROUP_1x128, want_deq=False)), 128 / 2048, "128 of 2048 rows")
        out["3_fp8_quantize_Bt_14336x4096"] = part(timed(
            lambda: oracle.quant_fp8(bt, oracle.FP8_BLOCK_128x128, want_deq=False)), 256 / 14336, "256 of 14336 rows")
        out["3_fp8_block_gemm_2048x14336x4096"] = part(timed(
            lambda: oracle.gemm_fp8_block(qa, sa, qb, sb, ii, jj)), 4096 / (2048 * 14336), "4096 output points")

        a, bt = syn.fp4_gemm_inputs(seed=0, M=128, N=256)
        ca, sca, ga, _ = oracle.quant_nvfp4(a, want_deq=False)
        cb, scb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
        ma, ea, _ = oracle.quant_mxfp4(a, want_deq=False)
        mb, eb, _ = oracle.quant_mxfp4(bt, want_deq=False)
        ii, jj = points(128, 256, 4096, 4)
        out["4_nvfp4_quantize_A_8192x4096"] = part(timed(
            lambda: oracle.quant_nvfp4(a, want_deq=False)), 128 / 8192, "128 of 8192 rows")
        out["4_mxfp4_quantize_A_8192x4096"] = part(timed(
            lambda: oracle.quant_mxfp4(a, want_deq=False)), 128 / 8192, "128 of 8192 rows")
        out["4_nvfp4_gemm_8192x4096x4096"] = part(timed(
            lambda: oracle.gemm_nvfp4(ca, sca, ga, cb, scb, gb, ii, jj)), 4096 / (8192 * 4096), "4096 output points")
        out["4_mxfp4_gemm_8192x4096x4096"] = part(timed(
            lambda: oracle.gemm_mxfp4(ma, ea, mb, eb, ii, jj)), 4096 / (8192 * 4096), "4096 output points")

        w4_s = nv_s = 0.0
        n_pts, full_pts = 0, 0
        for _, name, a_bits, w in syn.qwen3_decode_linears(layers=1, tokens=64, seed=0):
            K, N = w.shape
            qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
            ca, sca, ga, _ = oracle.quant_nvfp4(a_bits, want_deq=False)
            cb, scb, gb, _ = oracle.quant_nvfp4(syn.to_bf16_bits(np.ascontiguousarray(w.T)), want_deq=False)
            ii, jj = points(64, N, 512, K + N)
            w4_s += timed(lambda: oracle.gemm_w4a16(a_bits, qw, sc, ii, jj))
            nv_s += timed(lambda: oracle.gemm_nvfp4(ca, sca, ga, cb, scb, gb, ii, jj))
            n_pts += ii.size
            full_pts += 64 * N
        share = n_pts / (28 * full_pts)
        out["5_qwen3_step_w4a16_196_linears"] = part(w4_s, share, "512 output points of each linear of one layer")
        out["5_qwen3_step_nvfp4_196_linears"] = part(nv_s, share, "512 output points of each linear of one layer")
        k, v = syn.kv_cache_inputs(seed=0)
        out["5_kv_write_fp8_2x8x4096x128"] = part(timed(lambda: oracle.kv_write_fp8(k, v)), 1.0, "the whole K and V")
    return {"oracle_per_config": out, "host": {**host_cpu(), "pinned_core": core}}


def reference_arm(args, rank, world):
    """--impl reference: the CPU oracle as it stands, timed on this host's cores, on a
    bounded sample of the same workload each step. Rank 0 alone runs it."""
    if rank != 0:
        return
    per_step_budget = max(0.5, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(budget_s=per_step_budget / 4)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(budget_s=per_step_budget))
    elapsed = time.perf_counter() - t0
    value = statistics.median(v["value"] for v in vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed * 1e3 / args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": list(MS), "K": K_DIM, "N": N_DIM,
                       "parallelism": "cpu single thread"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": vals[-1]["sample"], "host": vals[-1].get("host")},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


ROW_NAMES = ("fp8", "fp4", "roundtrip", "kv", "qwen", "next")


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["qz", "reference"], default="qz")
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary per-row measurements")
    ap.add_argument("--rows", default="fp8,fp4,roundtrip,kv,qwen,next",
                    help="secondary rows to measure (comma list of fp8, fp4, roundtrip, kv, qwen, next)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--oracle-per-config", action="store_true",
                    help="only time the CPU oracle on a sample of every workload (no GPU) and print it")
    return ap


def main(argv=None):
    ap = build_parser()
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    unknown = set(args.rows.split(",")) - set(ROW_NAMES)
    if unknown:
        ap.error(f"unknown rows: {sorted(unknown)}")
    if args.oracle_per_config:
        print(json.dumps(oracle_per_config()), flush=True)
        return
    rank, world, local_rank = dist_setup(args.gpus)
    if args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        gpu_arm(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
