"""Benchmark of the BitLinear forward on B300.

Default workload (N=1): decode, M = 1 token, over the four BitLinear
projections of a 2B-class layer (q/o 2560->2560, k/v 2560->640, FFN up
2560->6912, FFN down 6912->2560) for 30 independent layers: 120 independent
problems, each with its own weights and its own input row. One step = the 120
BitLinear forwards (per-token int8 quantization, packed ternary GEMV, dequant),
issued as one bitlinear_forward_batch call (one quantization launch for all
120 inputs, then one GEMV launch over all 120 weight matrices), captured once
in a CUDA graph and replayed. The packed weights of one step (327 MB)
exceed the 126 MB L2, so no flush is needed between steps. Metric: GB/s of
packed weights streamed. The same 120 forwards issued as dependent
bitlinear_forward calls (each waits for the previous one, as consecutive
layers of a model would) are timed too and reported under "chained".

Multi-GPU (torchrun): each rank runs an independent replica (weak scaling);
value = all ranks' bytes / the slowest rank's time.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the oracle is the reference arm; it is not tuned).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BitLinear decode GB/s of packed weights (% HBM peak); prefill int8 TOPS (% peak)"
UNIT = "GB/s"
SHAPE_ORDER = ["qo", "kv", "up", "down"]


def rank_info():
    r = int(os.environ.get("RANK", "0"))
    w = int(os.environ.get("WORLD_SIZE", "1"))
    lr = int(os.environ.get("LOCAL_RANK", str(r)))
    return r, w, lr


def slowest_rank_seconds(torch, seconds: float, world: int, device) -> float:
    """The job's time: the maximum over the ranks (all-reduce MAX; the
    identity on one rank)."""
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_step: int, steps: int, world: int, slowest_s: float) -> float:
    """Whole-job throughput: the bytes all ranks streamed (each rank runs its
    own replica of the step) over the slowest rank's time, in GB/s."""
    return bytes_per_step * steps * world / slowest_s / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.lines = []
            import threading

            def reader():
                for line in self.proc.stdout:
                    self.lines.append((time.time(), line.strip()))
            self.th = threading.Thread(target=reader, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.1 <= r[0] <= (self.t1 or r[0]) + 0.1]
        use = inside if inside else rows[-3:]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in use if num(p[1]) is not None]
        smax = [num(p[2]) for _, p in use if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in use for i in range(4) if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# --------------------------------------------------------- decode workload
def build_decode(torch, BL, WL, layers: int, device):
    """Packs the 30x4 weight matrices and draws the 120 activation rows. The
    inputs of all problems live end to end in one device buffer and the
    outputs in another (each row 16-byte aligned), as a caller of the batched
    call keeps them, so one copy moves all inputs and one all outputs."""
    specs = [(layer, shape) + WL.SHAPES_2B[shape] for layer in range(layers) for shape in SHAPE_ORDER]
    x_flat = torch.empty(sum(K for _, _, K, _ in specs), dtype=torch.float32, device=device)
    y_flat = torch.empty(sum(N for _, _, _, N in specs), dtype=torch.float32, device=device)
    mats = []
    xo = yo = 0
    for layer, shape, K, N in specs:
        W = torch.from_numpy(WL.decode_weights(shape, layer)).to(device)
        packed, s_w = BL.pack(W)
        del W
        X = x_flat[xo:xo + K].view(1, K)
        X.copy_(torch.from_numpy(WL.decode_activations(shape, layer)))
        Y = y_flat[yo:yo + N].view(1, N)
        xo += K
        yo += N
        mats.append({"shape": shape, "layer": layer, "K": K, "N": N, "packed": packed, "s_w": s_w, "X": X,
                     "Y": Y})
    torch.cuda.synchronize()
    return mats, x_flat, y_flat


# DRAM bytes (read + write) of one launch of the dominant kernel, from the ncu
# capture summarised in profiles/gemv_batch_decode_m1_x12.md (12 layers). They
# hold only for the kernel source they were taken on: a changed gemv.cu gives
# traffic = null until it is profiled again.
TRAFFIC = {"source": "ternary_weight_linear_06_b300/csrc/gemv.cu", "sha256_prefix": "dcebfd9a1121beeb",
           "bytes": 135634432.0, "layers": 12}


def traffic_per_launch(layers: int):
    import hashlib
    with open(os.path.join(ROOT, TRAFFIC["source"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != TRAFFIC["sha256_prefix"]:
            return None
    return TRAFFIC["bytes"] * layers / TRAFFIC["layers"]


def packed_bytes(mats):
    return sum(m["N"] * m["K"] // 4 for m in mats)


def gemv_algorithmic_bytes(mats, M=1):
    # packed weights + int8 activations + fp32 outputs + the per-token scale
    return sum(m["N"] * m["K"] // 4 + M * m["K"] + 4 * M * m["N"] + 4 * M for m in mats)


def time_graph(torch, g, steps, warmup, stream):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def run_ours(args):
    import torch
    import torch.distributed as dist

    import ternary_weight_linear_06_b300 as BL
    from ternary_weight_linear_06_b300 import workloads as WL

    rank, world, local_rank = rank_info()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    peaks, peak_src = measured_peaks()

    mats, x_flat, y_flat = build_decode(torch, BL, WL, args.layers, device)
    ws = BL.Workspace(1 << 16, device)
    stream = torch.cuda.Stream(device)
    bytes_step = packed_bytes(mats)
    problems = [(m["X"], m["packed"], m["s_w"], m["Y"]) for m in mats]

    # ---- the step: the 120 independent forwards of one decode token in one
    #      bitlinear_forward_batch call (quantization launch + GEMV launch)
    with torch.cuda.stream(stream):
        descs = BL.forward_batch(problems, workspace=ws)        # first call outside capture
    torch.cuda.synchronize()

    def step():
        BL.forward_batch(problems, workspace=ws, descs=descs)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()

    # ---- the same work as 120 dependent bitlinear_forward calls (stream order,
    #      programmatic dependent launch): each waits for the previous one
    def chained():
        for m in mats:
            BL.forward(m["X"], m["packed"], m["s_w"], out=m["Y"], workspace=ws)

    with torch.cuda.stream(stream):
        chained()
    torch.cuda.synchronize()
    gc = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gc, stream=stream):
        chained()
    torch.cuda.synchronize()

    # ---- the GEMV alone (the dominant kernel): the same 120 problems given
    #      already quantized, so the call launches only the GEMV
    qms = [BL.quant_act(m["X"]) for m in mats]
    y_q8 = [torch.empty_like(m["Y"]) for m in mats]
    problems_q8 = [(q, m["packed"], m["s_w"], y, None, mm) for (q, mm), m, y in zip(qms, mats, y_q8)]
    with torch.cuda.stream(stream):
        descs_q8 = BL.forward_batch(problems_q8, workspace=ws)
    torch.cuda.synchronize()
    gq = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gq, stream=stream):
        BL.forward_batch(problems_q8, workspace=ws, descs=descs_q8)
    torch.cuda.synchronize()

    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[local_rank]
                    if os.environ.get("CUDA_VISIBLE_DEVICES") else local_rank)
    clocks = ClockSampler(gpu_index)
    time.sleep(0.3)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    if world > 1:
        dist.barrier()
    elapsed = e0.elapsed_time(e1) / 1e3
    elapsed_max = slowest_rank_seconds(torch, elapsed, world, device)
    clk = clocks.stop()

    # dominant kernel: the GEMV launch alone, timed on the launching stream
    with torch.cuda.stream(stream):
        gemv_s = time_graph(torch, gq, args.steps, args.warmup, stream)
    launch_s = gemv_s / args.steps
    alg_bytes_launch = gemv_algorithmic_bytes(mats)
    achieved = alg_bytes_launch / launch_s / 1e9
    same = all(torch.equal(a["Y"], b) for a, b in zip(mats, y_q8))
    traffic = traffic_per_launch(args.layers)
    traffic = round(traffic) if traffic is not None else None

    chained_steps = max(20, args.steps // 5)
    with torch.cuda.stream(stream):
        chained_s = time_graph(torch, gc, chained_steps, 3, stream)

    # end-to-end: pinned host X -> device (one copy of the 120 input rows), the
    # batched call, device Y -> pinned host (one copy of the 120 output rows)
    x_host = x_flat.cpu().pin_memory()
    y_host = torch.empty_like(y_flat, device="cpu").pin_memory()
    h2d = x_host.numel() * 4
    d2h = y_host.numel() * 4
    e_steps = max(1, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(2):
            x_flat.copy_(x_host, non_blocking=True)
            g.replay()
            y_host.copy_(y_flat, non_blocking=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e_steps):
            x_flat.copy_(x_host, non_blocking=True)
            g.replay()
            y_host.copy_(y_flat, non_blocking=True)
        stream.synchronize()
        e2e_s = time.perf_counter() - t0
    e2e_value = bytes_step * e_steps / e2e_s / 1e9 * world

    assert BL.workspace_status(ws) == 0, "device-side status word set"
    prefill = None if args.no_prefill else prefill_leg(torch, BL, WL, device, peaks, peak_src, stream)

    value = job_value(bytes_step, args.steps, world, elapsed_max)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_max / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": f"decode M=1, 2B-class projections (q/o 2560x2560, k/v 2560x640, up 2560x6912, "
                               f"down 6912x2560) x {args.layers} layers", "M": 1, "layers": args.layers,
                   "forwards_per_step": len(mats), "packed_bytes_per_step": bytes_step,
                   "l2": "inputs larger than L2 (packed weights per step exceed 126 MB)",
                   "launch": "one bitlinear_forward_batch call per step (120 independent problems: one "
                             "quantization launch + one GEMV launch), CUDA graph",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel (M=1, 120 problems per launch)",
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "peak_source": f"{peak_src} hbm_gbs (burst copy)", "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "traffic_source": "ncu capture of 12 layers scaled by layers (profiles/gemv_batch_decode_m1_x12.md)",
                     "alg_bytes_per_launch": round(alg_bytes_launch), "avg_launch_us": round(launch_s * 1e6, 3),
                     "how": "the GEMV launch alone (the 120 problems given pre-quantized, one graph per step), "
                            "CUDA events on the launching stream", "matches_step_output": same},
        "chained": {"value": round(bytes_step * chained_steps / chained_s / 1e9, 2), "unit": UNIT,
                    "ms_per_step": round(chained_s / chained_steps * 1e3, 4), "launches_per_step": len(mats),
                    "how": "the same 120 forwards as dependent bitlinear_forward calls in stream order "
                           "(programmatic dependent launch), CUDA graph"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "pinned host -> device copy of the 120 input rows (one buffer), graph replay, device -> "
                       "pinned host copy of the 120 output rows (one buffer), every step"},
        "gpu_launches": 2 * args.steps,
        "prefill": prefill,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(mats, args.cpu_seconds)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


# --------------------------------------------------------- prefill leg
def time_each(torch, fn, iters, stream, flush=None):
    """Mean device time of fn() over iters calls, each bracketed by CUDA events
    on `stream`; L2 is flushed (a write larger than L2) between calls."""
    tot = 0.0
    for _ in range(iters):
        if flush is not None:
            flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1) / 1e3
    return tot / iters


def prefill_leg(torch, BL, WL, device, peaks, peak_src, stream, iters=20, M=4096, shapes=None, ffn=True):
    """Prefill: M tokens through the four 2B-class projections (forward =
    quantization + tensor-core GEMM; and the GEMM alone on a pre-quantized
    input) and through the fused FFN block 2560 -> 6912 -> ReLU^2 -> 2560."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    out = {"M": M, "unit": "TOPS", "forward": {}, "forward_rmsnorm": {}, "gemm_only": {}, "ms": {}}
    ws = BL.Workspace(0, device)
    best, best_shape = None, None
    with torch.cuda.stream(stream):
        for shape in (shapes or SHAPE_ORDER):
            K, N = WL.SHAPES_2B[shape]
            W = torch.from_numpy(WL.decode_weights(shape, 0)).to(device)
            packed, s_w = BL.pack(W)
            del W
            X = torch.from_numpy(WL.prefill_activations(M, K, seed=9000 + K + N)).to(device)
            Y = torch.empty((M, N), dtype=torch.float32, device=device)
            act, m = BL.quant_act_tc(X)
            BL.forward(X, packed, s_w, out=Y, workspace=ws)
            BL.forward_tc(act, m, packed, s_w, out=Y, workspace=ws)
            torch.cuda.synchronize()
            ops = 2.0 * M * N * K
            t_fwd = time_each(torch, lambda: BL.forward(X, packed, s_w, out=Y, workspace=ws), iters, stream, flush)
            t_mm = time_each(torch, lambda: BL.forward_tc(act, m, packed, s_w, out=Y, workspace=ws), iters, stream,
                             flush)
            g = torch.from_numpy(WL.norm_gain(K, seed=9200 + K, edge=False)).to(device)
            t_norm = time_each(torch, lambda: BL.forward_rmsnorm(X, packed, s_w, g, out=Y, workspace=ws), iters,
                               stream, flush)
            out["forward"][shape] = round(ops / t_fwd / 1e12, 1)
            out["forward_rmsnorm"][shape] = round(ops / t_norm / 1e12, 1)
            out["gemm_only"][shape] = round(ops / t_mm / 1e12, 1)
            out["ms"][shape] = {"forward": round(t_fwd * 1e3, 4), "forward_rmsnorm": round(t_norm * 1e3, 4),
                                "gemm": round(t_mm * 1e3, 4)}
            if shape == "up" or best is None:
                best, best_shape = (ops, t_mm), shape
            del X, Y, act, m, packed
    if ffn:
        D, F = 2560, 6912
        with torch.cuda.stream(stream):
            up, s_up = BL.pack(torch.from_numpy(WL.decode_weights("up", 1)).to(device))
            down, s_down = BL.pack(torch.from_numpy(WL.decode_weights("down", 1)).to(device))
            X = torch.from_numpy(WL.prefill_activations(M, D, seed=9100)).to(device)
            Yf = torch.empty((M, D), dtype=torch.float32, device=device)
            BL.ffn(X, up, s_up, down, s_down, out=Yf, workspace=ws)
            torch.cuda.synchronize()
            t_ffn = time_each(torch, lambda: BL.ffn(X, up, s_up, down, s_down, out=Yf, workspace=ws), iters,
                              stream, flush)
            gate, s_gate = BL.pack(torch.from_numpy(WL.decode_weights("up", 2)).to(device))
            g_in = torch.from_numpy(WL.norm_gain(D, seed=9300, edge=False)).to(device)
            g_sub = torch.from_numpy(WL.norm_gain(F, seed=9301, edge=False)).to(device)
            t_gated = time_each(torch, lambda: BL.ffn_gated(X, up, s_up, gate, s_gate, down, s_down, out=Yf,
                                                            workspace=ws), iters, stream, flush)
            t_subln = time_each(torch, lambda: BL.ffn_subln(X, up, s_up, down, s_down, g_in=g_in, g_sub=g_sub,
                                                            gate=gate, s_gate=s_gate, out=Yf, workspace=ws),
                                iters, stream, flush)
        out["ffn"] = round(4.0 * M * D * F / t_ffn / 1e12, 1)
        out["ffn_gated"] = round(6.0 * M * D * F / t_gated / 1e12, 1)
        out["ffn_subln_gated"] = round(6.0 * M * D * F / t_subln / 1e12, 1)
        out["ms"]["ffn"] = round(t_ffn * 1e3, 4)
        out["ms"]["ffn_gated"] = round(t_gated * 1e3, 4)
        out["ms"]["ffn_subln_gated"] = round(t_subln * 1e3, 4)
    ops, t_mm = best
    achieved = ops / t_mm / 1e12
    up_name = "FFN up 2560->6912" if best_shape == "up" else best_shape
    peak = peaks["bf16_tflops"]
    out["roofline"] = {"bound": "tensor", "kernel": f"gemm_tc_kernel ({up_name}, M={M})",
                       "achieved": round(achieved, 1), "peak": peak,
                       "peak_source": f"{peak_src} bf16_tflops (burst; fp16 has the same nominal dense rate)",
                       "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                       "alg_ops_per_launch": ops, "avg_launch_us": round(t_mm * 1e6, 2),
                       "how": "one bitlinear_forward_tc launch per timed call (CUDA events on the launching "
                              "stream), L2 flushed between calls"}
    out["how"] = ("integer-valued fp16 operands on tcgen05 kind::f16 (sm_103a has no int8 tcgen05 MMA); "
                  "ops = 2*M*N*K per projection, 4*M*D*F for the FFN, 6*M*D*F gated; forward_rmsnorm and "
                  "ffn_subln_gated include the fused RMSNorm (unit-scale gains)")
    return out


# ------------------------------------------------------------ CPU oracle
def oracle_decode_sample(mats_host, seconds):
    """Times oracle forwards over the packed matrices (round robin) for about
    `seconds`; returns (packed bytes processed, elapsed s, forwards, shapes)."""
    import oracle as O
    done = 0
    nbytes = 0
    t0 = time.perf_counter()
    i = 0
    while True:
        m = mats_host[i % len(mats_host)]
        O.forward_packed(m["X"], m["packed"], m["s_w"])
        nbytes += m["N"] * m["K"] // 4
        done += 1
        i += 1
        if time.perf_counter() - t0 >= seconds and done >= 4:
            break
    return nbytes, time.perf_counter() - t0, done


def host_mats_from_device(mats, limit=8):
    out = []
    for m in mats[:limit]:
        out.append({"K": m["K"], "N": m["N"], "packed": m["packed"].cpu().numpy(),
                    "s_w": np.float32(m["s_w"].cpu().numpy()[0]), "X": m["X"].cpu().numpy()})
    return out


def cpu_baseline(mats, seconds):
    hm = host_mats_from_device(mats, limit=4)
    nbytes, el, n = oracle_decode_sample(hm, seconds)
    return {"value": round(nbytes / el / 1e9, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} oracle forwards (M=1) round-robin over layer 0's four projections, {el:.1f} s"}


def run_reference(args):
    """The CPU oracle as the reference arm: same metric, unit and config."""
    rank, world, _ = rank_info()
    if rank != 0:
        return
    from ternary_weight_linear_06_b300 import workloads as WL
    import oracle as O
    hm = []
    for shape in SHAPE_ORDER:
        K, N = WL.SHAPES_2B[shape]
        W = WL.decode_weights(shape, 0)
        packed, s_w, _ = O.pack_weights(W)
        hm.append({"K": K, "N": N, "packed": packed, "s_w": s_w, "X": WL.decode_activations(shape, 0)})
    per = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_decode_sample(hm, per)
    tot_b = tot_s = 0.0
    tot_n = 0
    for _ in range(args.steps):
        b, s, n = oracle_decode_sample(hm, per)
        tot_b += b
        tot_s += s
        tot_n += n
    value = tot_b / tot_s / 1e9
    out = {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic", "impl": "reference",
           "config": {"workload": f"decode M=1, 2B-class projections (q/o 2560x2560, k/v 2560x640, up 2560x6912, "
                                  f"down 6912x2560) x {args.layers} layers", "M": 1, "layers": args.layers},
           "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": f"each step: {per:.1f} s of oracle forwards over layer 0's four projections "
                                      f"({tot_n} forwards in total)"},
           "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def run_crossover(args):
    """Batched decode: GEMV (dp4a) vs tensor-core GEMM per shape and token count,
    each call timed alone with L2 flushed between calls; the crossover is the
    smallest M from which the GEMM is faster."""
    import torch

    import ternary_weight_linear_06_b300 as BL
    from ternary_weight_linear_06_b300 import workloads as WL
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    ws = BL.Workspace(0, device)
    Ms = [1, 2, 4, 5, 6, 8, 12, 16, 24, 32, 48, 64, 128, 256]
    out = {"what": "batched decode: GEMV vs tensor-core GEMM (us per call, L2 flushed)", "M": Ms, "shapes": {}}
    with torch.cuda.stream(stream):
        for shape in SHAPE_ORDER:
            K, N = WL.SHAPES_2B[shape]
            packed, s_w = BL.pack(torch.from_numpy(WL.decode_weights(shape, 2)).to(device))
            rows = {"gemv_us": [], "gemm_us": [], "crossover_M": None}
            for M in Ms:
                xb = WL.batched_activations_bf16(M, K, seed=700 + M)
                X = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(device)
                q, m = BL.quant_act(X)
                act, m2 = BL.quant_act_tc(X)
                Y1 = torch.empty((M, N), dtype=torch.float32, device=device)
                Y2 = torch.empty((M, N), dtype=torch.float32, device=device)
                prob = [(q, packed, s_w, Y1, None, m)]
                descs = BL.forward_batch(prob, workspace=ws)
                BL.forward_tc(act, m2, packed, s_w, out=Y2, workspace=ws)
                torch.cuda.synchronize()
                assert torch.equal(Y1, Y2), (shape, M)
                t1 = time_each(torch, lambda: BL.forward_batch(prob, workspace=ws, descs=descs), args.prefill_iters,
                               stream, flush)
                t2 = time_each(torch, lambda: BL.forward_tc(act, m2, packed, s_w, out=Y2, workspace=ws),
                               args.prefill_iters, stream, flush)
                rows["gemv_us"].append(round(t1 * 1e6, 2))
                rows["gemm_us"].append(round(t2 * 1e6, 2))
                if rows["crossover_M"] is None and t2 < t1:
                    rows["crossover_M"] = M
            out["shapes"][shape] = rows
    print(json.dumps(out))


def run_large(args):
    """70B-class shapes (hidden 8192, FFN 28672), swept over token counts: each
    forward (quantization + GEMV or GEMM) timed alone with L2 flushed between
    calls; GB/s of packed weights and integer TOPS (2*M*N*K)."""
    import torch

    import ternary_weight_linear_06_b300 as BL
    from ternary_weight_linear_06_b300 import workloads as WL
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    ws = BL.Workspace(0, device)
    peaks, _ = measured_peaks()
    Ms = [1, 8, 64, 512, 2048]
    out = {"what": "70B-class shapes: forward per token count (L2 flushed)", "M": Ms, "shapes": {}}
    with torch.cuda.stream(stream):
        for shape in ("attn", "up", "down"):
            K, N = WL.SHAPES_70B[shape]
            W = torch.from_numpy(WL.large_weights(shape)).to(device)
            packed, s_w = BL.pack(W)
            del W
            rows = {"K": K, "N": N, "us": [], "GBps": [], "TOPS": []}
            for M in Ms:
                X = torch.from_numpy(WL.student_t(M, K, seed=40 + M)).to(device)
                Y = torch.empty((M, N), dtype=torch.float32, device=device)
                BL.forward(X, packed, s_w, out=Y, workspace=ws)
                torch.cuda.synchronize()
                t = time_each(torch, lambda: BL.forward(X, packed, s_w, out=Y, workspace=ws), args.prefill_iters,
                              stream, flush)
                rows["us"].append(round(t * 1e6, 2))
                rows["GBps"].append(round(N * K / 4 / t / 1e9, 1))
                rows["TOPS"].append(round(2.0 * M * N * K / t / 1e12, 1))
                del X, Y
            out["shapes"][shape] = rows
    out["hbm_peak_gbs"] = peaks["hbm_gbs"]
    out["tensor_peak_tflops"] = peaks["bf16_tflops"]
    print(json.dumps(out))


def run_prefill_only(args):
    import torch

    import ternary_weight_linear_06_b300 as BL
    from ternary_weight_linear_06_b300 import workloads as WL
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    peaks, peak_src = measured_peaks()
    stream = torch.cuda.Stream(device)
    shapes = [x for x in args.prefill_shapes.split(",") if x] or None
    out = prefill_leg(torch, BL, WL, device, peaks, peak_src, stream, iters=args.prefill_iters, shapes=shapes,
                      ffn=not args.prefill_no_ffn)
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill (M=4096) leg")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill leg (profiling); prints its JSON object")
    ap.add_argument("--prefill-iters", type=int, default=20)
    ap.add_argument("--prefill-shapes", default="", help="comma-separated subset of qo,kv,up,down")
    ap.add_argument("--prefill-no-ffn", action="store_true")
    ap.add_argument("--large", action="store_true",
                    help="70B-class shapes over token counts (prints its own JSON; not the bench line)")
    ap.add_argument("--crossover", action="store_true",
                    help="batched decode GEMV vs GEMM sweep (prints its own JSON; not the bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill_only:
        run_prefill_only(args)
    elif args.crossover:
        run_crossover(args)
    elif args.large:
        run_large(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
