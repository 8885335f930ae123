"""Benchmark of the MX hot path on GB300.

Headline workload (one JSON line on rank 0): MXFP8 quantize + dequantize of a
bf16 4096 x 4096 activation tensor (blocks of 32 along the last axis, the
seeded synthetic workload with heavy tails, zero / tiny / subnormal blocks and
64 NaN-scale blocks).  One step = mx_quantize (bf16 -> E4M3 codes + E8M0
scales) then mx_dequantize (-> f32).  value = algorithmic bytes of both calls
per step / step time, summed over ranks.

The same line carries the block_matmul workloads (decode 16x14336x4096
E4M3 x E2M1 with its on-the-fly activation quantize, square 8192^3 MXFP8, and
prefill 8192x28672x8192 MXFP4 with its activation quantize) under
``block_matmul``, the dominant kernel's roofline, an end-to-end number through
host buffers, and the CPU oracle's throughput on a bounded sample.

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA
graphs between CUDA events on the launching stream, with a device
synchronize (and a barrier across ranks) on both sides; the maximum time over
ranks is used.  Inputs rotate over enough buffer sets that one rotation
exceeds 3x the L2 size, so no step finds its inputs in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  (N > 1: launch with torch.distributed.run, one rank per GPU; the workload is
  replicated per GPU -- weak scaling, no data-path collective.)
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MX quantize GB/s (% HBM peak); block_matmul TFLOPS (% dense MX tensor peak)"
HEADLINE = "mxfp8_act_4096: bf16 4096x4096 -> MXFP8 (E4M3FN + E8M0) quantize, then dequantize -> f32"
NOMINAL_RATIO = {"fp8": 4.5 / 2.25, "fp4": 13.5 / 2.25}  # dense tensor rates relative to bf16


# ------------------------------------------------------------------ plumbing

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job rate: every rank processed `units_per_rank`; the job took the slowest rank's time."""
    return units_per_rank * world / max_seconds


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.15)
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
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            f = [s.strip() for s in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def l2_bytes() -> int:
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 126 * 2 ** 20


def sets_for(bytes_per_step: int) -> int:
    return max(2, math.ceil(3 * l2_bytes() / bytes_per_step))


def timed_graph_steps(step_fn, nsets: int, steps: int, warmup: int, world: int, dist_replays: int = 20):
    """Run `warmup` eager steps, then exactly `steps` steps replayed from CUDA
    graphs on one stream, between CUDA events on that stream: a graph of up
    to 256 steps (a whole number of rotations) replayed as often as fits, and
    a shorter graph for the remainder.  Afterwards, outside that timed
    region, the main graph is replayed `dist_replays` more times, each between
    its own events, for the spread of the per-step time.  Returns (seconds for
    the `steps` steps, seconds per step of each extra replay).  step_fn(i)
    issues step i."""
    for i in range(warmup):
        step_fn(i % nsets)
    torch.cuda.synchronize()
    n = min(steps, max(nsets, min(steps, 256) // nsets * nsets))
    reps, rem = divmod(steps, n)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step_fn(i % nsets)
        g_rem = None
        if rem:
            g_rem = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_rem, stream=stream):
                for i in range(rem):
                    step_fn(i % nsets)
        torch.cuda.synchronize()
        g.replay()  # upload / first-replay cost kept out of the timed region
        if g_rem is not None:
            g_rem.replay()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(reps):
            g.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(dist_replays + 1)]
        evs[0].record(stream)
        for r in range(dist_replays):
            g.replay()
            evs[r + 1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    per_step = [evs[r].elapsed_time(evs[r + 1]) / 1e3 / n for r in range(dist_replays)]
    return start.elapsed_time(end) / 1e3, per_step


def dist_us(per_step):
    """Median and 10th / 90th percentiles of per-step times, in microseconds
    (one value per graph replay: its time over its steps)."""
    if not per_step:
        return None
    v = sorted(x * 1e6 for x in per_step)
    q = lambda f: v[min(len(v) - 1, max(0, int(round(f * (len(v) - 1)))))]
    return {"median_us": statistics.median(v), "p10_us": q(0.1), "p90_us": q(0.9), "replays": len(v)}


# ------------------------------------------------------------- workloads

def headline_bytes(rows, cols):
    """Algorithmic bytes of quantize (bf16 in, E4M3 codes + scales out) and of
    dequantize (codes + scales in, f32 out)."""
    n = rows * cols
    q = 2 * n + n + n // 32
    d = n + n // 32 + 4 * n
    return q, d


def timed(step_fn, nsets, steps, warmup, world):
    """timed_graph_steps with the maximum over ranks of the total; returns (seconds, distribution)."""
    sec, per = timed_graph_steps(step_fn, nsets, steps, warmup, world)
    return max_over_ranks(sec, world), dist_us(per)


def bench_headline(mx, steps, warmup, world, peaks, device_index):
    """Workload 2: step i quantizes rotation set i and dequantizes the set
    written half a rotation earlier (at least 1.5x L2 of traffic ago), so the
    codes and scales it reads come from HBM like every other counted byte:
    the step's bytes per second is an HBM rate.  Each kernel is also timed on
    its own over the same rotation (the roofline's per-kernel numbers)."""
    w = workloads.make(2)
    rows, cols = w["rows"], w["cols"]
    qb, db = headline_bytes(rows, cols)
    nsets = sets_for(qb + db)
    half = nsets // 2
    x0 = w["x"].cuda()
    sets = []
    for i in range(nsets):
        sets.append({"x": x0.clone(), "codes": mx.alloc_codes(rows, cols, mx.E4M3FN),
                     "scales": mx.alloc_scales(rows, cols), "y": torch.empty(rows, cols, device="cuda")})
    nan_blocks = torch.from_numpy(w["nan_blocks"]).cuda()

    def step(i):
        s = sets[i]
        mx.mx_quantize(s["x"], mx.E4M3FN, s["codes"], s["scales"])
        d = sets[(i + half) % nsets]
        mx.mx_dequantize(d["codes"], d["scales"], rows, cols, mx.E4M3FN, d["y"])

    def deq_only(i):
        s = sets[i]
        mx.mx_dequantize(s["codes"], s["scales"], rows, cols, mx.E4M3FN, s["y"])

    def q_only(i):
        s = sets[i]
        mx.mx_quantize(s["x"], mx.E4M3FN, s["codes"], s["scales"])

    # every set holds codes before a step dequantizes it; correctness of what
    # is timed: the 64 NaN-scale blocks poison their blocks
    for i in range(nsets):
        q_only(i)
    s0 = sets[0]
    s0["scales"][nan_blocks] = 0xFF
    deq_only(0)
    mx.mx_device_status()
    assert int(torch.isnan(s0["y"].view(-1, 32)).all(dim=1).sum()) >= 64
    q_only(0)

    with ClockSampler(device_index) as clk:
        sec, dist = timed(step, nsets, steps, warmup, world)
    value = job_throughput((qb + db) * steps, world, sec) / 1e9
    # per-kernel timing for the roofline (same stream, same rotation)
    k_steps = max(steps, 200)
    sec_d, dist_d = timed(deq_only, nsets, k_steps, 3, world)
    sec_q, dist_q = timed(q_only, nsets, k_steps, 3, world)
    deq_gbs = db * k_steps / sec_d / 1e9
    q_gbs = qb * k_steps / sec_q / 1e9
    mx.mx_device_status()
    return {
        "value": value, "ms_per_step": sec / steps * 1e3, "dist": dist, "clocks": clk.summary(), "nsets": nsets,
        "launches": 2 * steps,
        "quantize": {"gbs": q_gbs, "us": sec_q / k_steps * 1e6, "bytes": qb, "frac": q_gbs / peaks["hbm_gbs"],
                     "dist": dist_q},
        "dequantize": {"gbs": deq_gbs, "us": sec_d / k_steps * 1e6, "bytes": db, "frac": deq_gbs / peaks["hbm_gbs"],
                       "dist": dist_d},
        "dominant": "dequantize" if sec_d >= sec_q else "quantize",
        "x_host": w["x"], "rows": rows, "cols": cols, "bytes": qb + db,
    }


def bench_e2e(mx, hl, steps, world, chunk_options=(2, 4, 8), graph_steps=10):
    """Same metric through the public API with host buffers: per step, copy the
    bf16 input from pinned host memory, quantize, dequantize, copy the f32
    result back to pinned host memory; every copy of every step is inside the
    timed region.  The step is cut into row blocks on three streams (uploads,
    kernels, downloads), so one block's upload, another's kernels and another's
    download overlap, as a caller streaming tensors through the library would
    arrange it, and `graph_steps` such steps are captured in one CUDA graph
    (events between the streams become graph edges), so the host's launch loop
    does not pace the copy engines.  Every block count in chunk_options is
    timed and the best reported; the serial form (one stream, whole tensor, no
    graph) is reported beside it, with the copy rates."""
    rows, cols = hl["rows"], hl["cols"]
    x_host = hl["x_host"].pin_memory()
    y_host = torch.empty(rows, cols, dtype=torch.float32).pin_memory()
    x = torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(rows, cols, device="cuda")
    codes, scales = mx.alloc_codes(rows, cols, mx.E4M3FN), mx.alloc_scales(rows, cols)
    n = max(graph_steps, min(steps, 100) // graph_steps * graph_steps)
    s_in, s_k, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    h2d, d2h = rows * cols * 2, rows * cols * 4

    def serial_step():
        x.copy_(x_host, non_blocking=True)
        mx.mx_quantize(x, mx.E4M3FN, codes, scales)
        mx.mx_dequantize(codes, scales, rows, cols, mx.E4M3FN, y)
        y_host.copy_(y, non_blocking=True)

    def pipelined_step(chunks, ev, first):
        ev_in, ev_k, ev_out = ev
        rc = rows // chunks
        cb, sb = mx.mx_codes_bytes(mx.E4M3FN, rc, cols), mx.mx_scales_bytes(mx.SCALES_ROWMAJOR, rc, cols)
        for c in range(chunks):
            r0, r1 = c * rc, (c + 1) * rc
            with torch.cuda.stream(s_in):
                if not first:
                    s_in.wait_event(ev_k[c])  # the previous step's kernels are done with x[c]
                x[r0:r1].copy_(x_host[r0:r1], non_blocking=True)
                ev_in[c].record(s_in)
            with torch.cuda.stream(s_k):
                s_k.wait_event(ev_in[c])
                if not first:
                    s_k.wait_event(ev_out[c])  # the previous step's download of y[c] is done
                cc, ss = codes[c * cb:(c + 1) * cb], scales[c * sb:(c + 1) * sb]
                mx.mx_quantize(x[r0:r1], mx.E4M3FN, cc, ss, stream=s_k)
                mx.mx_dequantize(cc, ss, rc, cols, mx.E4M3FN, y[r0:r1], stream=s_k)
                ev_k[c].record(s_k)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_k[c])
                y_host[r0:r1].copy_(y[r0:r1], non_blocking=True)
                ev_out[c].record(s_out)

    def capture(chunks):
        ev = tuple([torch.cuda.Event() for _ in range(chunks)] for _ in range(3))
        cap = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            for st in (s_in, s_k, s_out):
                st.wait_stream(cap)
            for i in range(graph_steps):
                pipelined_step(chunks, ev, i == 0)
            for st in (s_in, s_k, s_out):
                cap.wait_stream(st)
        return g, cap

    def timed(fn, stream):
        torch.cuda.synchronize()
        barrier(world)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        fn()
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(start.elapsed_time(end) / 1e3, world)

    for _ in range(3):
        serial_step()
    cur = torch.cuda.current_stream()
    sec_serial = timed(lambda: [serial_step() for _ in range(n)], cur)
    # copy rates alone (pinned host memory), for context
    sec_h2d = timed(lambda: [x.copy_(x_host, non_blocking=True) for _ in range(n)], cur)
    sec_d2h = timed(lambda: [y_host.copy_(y, non_blocking=True) for _ in range(n)], cur)
    best = None
    per_chunks = {}
    for chunks in chunk_options:
        if rows % chunks:
            continue
        g, _ = capture(chunks)
        g.replay()
        torch.cuda.synchronize()
        sec = timed(lambda: [g.replay() for _ in range(n // graph_steps)], cur)  # replays run on the current stream
        per_chunks[chunks] = job_throughput(hl["bytes"] * n, world, sec) / 1e9
        if best is None or sec < best[1]:
            best = (chunks, sec)
        del g
    mx.mx_device_status()
    # the pipelined result is the same tensor: check one step's output against the serial one
    y_ref = y_host.clone()
    serial_step()
    torch.cuda.synchronize()
    assert torch.equal(torch.nan_to_num(y_host).view(torch.int32), torch.nan_to_num(y_ref).view(torch.int32))
    chunks, sec = best
    return {"value": job_throughput(hl["bytes"] * n, world, sec) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "pipeline": f"{chunks} row blocks over upload / kernel / download streams, {graph_steps} steps per "
                        f"CUDA graph", "by_row_blocks": per_chunks,
            "serial_value": job_throughput(hl["bytes"] * n, world, sec_serial) / 1e9,
            "h2d_gbs": h2d * n / sec_h2d / 1e9, "d2h_gbs": d2h * n / sec_d2h / 1e9}


def mma_rates(mx):
    """Measured block-scaled MMA rate per kind (shared-memory operands, no HBM
    traffic): reported beside the recipe-derived tensor peaks."""
    return {"fp8": mx.mx_measure_mma_rate(mx.E4M3FN, 20000), "fp4": mx.mx_measure_mma_rate(mx.E2M1, 20000)}


def tensor_peak(peaks, mma, kind):
    """The GEMM roofline's denominator: the larger of the recipe figure
    (measured bf16 burst x the nominal dense ratio of the format) and this
    GPU's measured block-scaled MMA rate."""
    recipe = peaks["bf16_tflops"] * NOMINAL_RATIO[kind]
    measured = mma[kind] if mma else None
    if measured is not None and measured > recipe:
        return measured, "measured block-scaled MMA rate (mx_measure_mma_rate)"
    return recipe, f"measured bf16 burst x {NOMINAL_RATIO[kind]:g} (nominal dense ratio)"


def bench_gemm(mx, cfg, steps, warmup, world, peaks, scale=1.0, dev_index=0, mma=None, oracle_rows=0):
    """block_matmul workloads.  Weights are quantized before timing; the step
    includes the activation quantize where the workload quantizes on the fly,
    and that quantize is also timed on its own.  oracle_rows > 0: the CPU
    oracle's block_matmul and activation quantize are timed too (rank 0)."""
    w = workloads.make(cfg, scale=scale)
    M, N, K = w["M"], w["N"], w["K"]
    if cfg == 3:
        fa, fb, a_key, b_key, quant_a, kind = mx.E4M3FN, mx.E2M1, "A", "W", True, "fp8"
    elif cfg == 4:
        fa, fb, a_key, b_key, quant_a, kind = mx.E4M3FN, mx.E4M3FN, "A", "Bt", False, "fp8"
    else:
        fa, fb, a_key, b_key, quant_a, kind = mx.E2M1, mx.E2M1, "A", "W", True, "fp4"
    L = mx.SCALES_MMA
    A = torch.as_tensor(w[a_key]).cuda()
    B = torch.as_tensor(w[b_key]).cuda()
    C0 = torch.from_numpy(w["C0"]).cuda()
    bc, bs = mx.alloc_codes(N, K, fb), mx.alloc_scales(N, K, L)
    mx.mx_quantize(B, fb, bc, bs, L)
    del B
    a_bytes_in = A.numel() * A.element_size()
    ca_b, sa_b = mx.mx_codes_bytes(fa, M, K), mx.mx_scales_bytes(L, M, K)
    gemm_bytes = ca_b + sa_b + mx.mx_codes_bytes(fb, N, K) + mx.mx_scales_bytes(L, N, K) + 8 * M * N
    qa_bytes = a_bytes_in + ca_b + sa_b
    step_bytes = gemm_bytes + (qa_bytes if quant_a else 0)
    nsets = sets_for(step_bytes) if step_bytes < 3 * l2_bytes() else 1
    # rotate only what fits; the weight (B) is shared, A and C rotate
    sets = []
    for i in range(nsets):
        ac, as_ = mx.alloc_codes(M, K, fa), mx.alloc_scales(M, K, L)
        if not quant_a:
            mx.mx_quantize(A, fa, ac, as_, L)
        sets.append({"A": A.clone() if (quant_a and i) else A, "ac": ac, "as": as_, "C": C0.clone()})
    if nsets > 1 and cfg == 3:
        # the decode weight (29 MB) would stay in L2 across steps: rotate it too
        for i, s in enumerate(sets):
            if i == 0:
                s["bc"], s["bs"] = bc, bs
            else:
                s["bc"], s["bs"] = bc.clone(), bs.clone()
    for s in sets:
        s.setdefault("bc", bc)
        s.setdefault("bs", bs)

    def step(i):
        s = sets[i]
        if quant_a:
            mx.mx_quantize(s["A"], fa, s["ac"], s["as"], L)
        mx.mx_block_matmul(s["ac"], s["as"], fa, s["bc"], s["bs"], fb, M, N, K, s["C"], L)

    def gemm_only(i):
        s = sets[i]
        mx.mx_block_matmul(s["ac"], s["as"], fa, s["bc"], s["bs"], fb, M, N, K, s["C"], L)

    def q_only(i):
        s = sets[i]
        mx.mx_quantize(s["A"], fa, s["ac"], s["as"], L)

    def fused(i):
        # activations quantized inside the GEMM (one launch; M <= 64 only)
        s = sets[i]
        mx.mx_block_matmul_act(s["A"], fa, s["bc"], s["bs"], fb, N, s["C"])

    step(0)
    mx.mx_device_status()
    sec_f = dist_f = sec_q = dist_q = None
    with ClockSampler(dev_index) as clk:
        sec, dist = timed(step, nsets, steps, warmup, world)
        sec_g, dist_g = timed(gemm_only, nsets, steps, 3, world)
        if quant_a:
            sec_q, dist_q = timed(q_only, nsets, steps, 3, world)
        if quant_a and M <= 64:
            fused(0)
            mx.mx_device_status()
            sec_f, dist_f = timed(fused, nsets, steps, 3, world)
    mx.mx_device_status()
    # the same product with the public row-major scale layout, through the
    # workspace entry point (its two scale relayout launches timed with it)
    rm_bytes = lambda rows: mx.mx_scales_bytes(mx.SCALES_ROWMAJOR, rows, K)
    for s in sets:
        s["as_rm"] = torch.empty(rm_bytes(M), dtype=torch.uint8, device="cuda")
        mx.mx_scales_relayout(s["as"], L, M, K, s["as_rm"], mx.SCALES_ROWMAJOR)
        if "bs_rm" not in s:
            s["bs_rm"] = torch.empty(rm_bytes(N), dtype=torch.uint8, device="cuda")
            mx.mx_scales_relayout(s["bs"], L, N, K, s["bs_rm"], mx.SCALES_ROWMAJOR)
            for t in sets:
                if t["bs"] is s["bs"]:
                    t["bs_rm"] = s["bs_rm"]
    ws = mx.alloc_workspace(M, N, K)

    def gemm_rm(i):
        s = sets[i]
        mx.mx_block_matmul_ws(s["ac"], s["as_rm"], fa, s["bc"], s["bs_rm"], fb, M, N, K, s["C"], ws)

    def gemm_rm_direct(i):
        s = sets[i]
        mx.mx_block_matmul(s["ac"], s["as_rm"], fa, s["bc"], s["bs_rm"], fb, M, N, K, s["C"], mx.SCALES_ROWMAJOR)

    gemm_rm(0)
    mx.mx_device_status()
    sec_rm, dist_rm = timed(gemm_rm, nsets, steps, 3, world)
    gemm_rm_direct(0)
    mx.mx_device_status()
    sec_rmd, dist_rmd = timed(gemm_rm_direct, nsets, steps, 3, world)
    mx.mx_device_status()
    flops = 2.0 * M * N * K
    tf_step = job_throughput(flops * steps, world, sec) / 1e12
    tf_gemm = flops * steps / sec_g / 1e12
    peak_tf, peak_src = tensor_peak(peaks, mma, kind)
    gbs_gemm = gemm_bytes * steps / sec_g / 1e9
    out = {"workload": workloads.NAMES[cfg], "M": M, "N": N, "K": K, "formats": {
        3: "E4M3 x E2M1", 4: "E4M3 x E4M3", 5: "E2M1 x E2M1"}[cfg],
        "step": "quantize A + block_matmul" if quant_a else "block_matmul",
        "tflops_step": tf_step, "us_per_step": sec / steps * 1e6, "step_dist": dist,
        "tflops_gemm": tf_gemm, "us_gemm": sec_g / steps * 1e6, "gemm_dist": dist_g,
        "tensor_peak_tflops": peak_tf, "tensor_peak_source": peak_src, "tensor_frac": tf_gemm / peak_tf,
        "tensor_frac_of_recipe": tf_gemm / (peaks["bf16_tflops"] * NOMINAL_RATIO[kind]),
        "gemm_gbs": gbs_gemm, "hbm_frac": gbs_gemm / peaks["hbm_gbs"], "gemm_bytes": gemm_bytes,
        "launches_per_step": 2 if quant_a else 1, "nsets": nsets, "clocks": clk.summary()}
    if mma is not None:
        out["mma_measured_tflops"] = mma[kind]
        out["tensor_frac_of_mma_measured"] = tf_gemm / mma[kind]
    out["rowmajor_ws"] = {"what": "row-major scales: mx_block_matmul_ws (one scale relayout launch + the product)",
                          "us": sec_rm / steps * 1e6, "dist": dist_rm, "tflops": flops * steps / sec_rm / 1e12,
                          "vs_tensor_core_layout": sec_rm / sec_g, "workspace_bytes": ws.numel() if ws is not None else 0,
                          "launches_per_step": 2}
    out["rowmajor_direct"] = {"what": "row-major scales: mx_block_matmul (scales gathered inside the product)",
                              "us": sec_rmd / steps * 1e6, "dist": dist_rmd, "tflops": flops * steps / sec_rmd / 1e12,
                              "vs_tensor_core_layout": sec_rmd / sec_g, "launches_per_step": 1}
    if sec_q is not None:
        g = qa_bytes * steps / sec_q / 1e9
        out["act_quantize"] = {"what": f"{'bf16' if A.dtype == torch.bfloat16 else 'f32'} {M}x{K} -> "
                                       f"{'MXFP8' if fa == mx.E4M3FN else 'MXFP4'} (tensor-core scale layout)",
                               "us": sec_q / steps * 1e6, "dist": dist_q, "gbs": g,
                               "hbm_frac": g / peaks["hbm_gbs"], "bytes": qa_bytes}
    if sec_f is not None:
        # one launch: activations in (f32/bf16), weight codes and scales, C read and written
        fused_bytes = a_bytes_in + mx.mx_codes_bytes(fb, N, K) + mx.mx_scales_bytes(L, N, K) + 8 * M * N
        out["fused"] = {"step": "block_matmul_act (activations quantized in the GEMM)",
                        "us_per_step": sec_f / steps * 1e6, "dist": dist_f, "tflops": flops * steps / sec_f / 1e12,
                        "gbs": fused_bytes * steps / sec_f / 1e9,
                        "hbm_frac": fused_bytes * steps / sec_f / 1e9 / peaks["hbm_gbs"], "bytes": fused_bytes,
                        "launches_per_step": 1}
    del sets, A, C0, bc, bs, ws
    torch.cuda.empty_cache()
    if oracle_rows > 0:
        out["oracle"] = oracle_gemm_baseline(w, cfg, a_key, b_key, quant_a, oracle_rows)
    return out


FFMA_PER_SM_CLK = 128  # f32 fused multiply-adds per SM per clock (4 partitions x 32 lanes)


def bench_next(mx, steps, warmup, world, peaks, dev_index):
    """The entry points beyond the three core ops, each on its own workload:
    block_matmul with an f32 right operand (workload 6, decode-shaped; the
    activations are quantized before timing), quantize along the first axis
    and dequantize to bf16 (workload 2's tensor), and fold_scale (workload 2's
    scales)."""
    out = {}
    # ---- block_matmul_f32b: C += deq(A) * B, B f32 K x N (235 MB > L2: no rotation needed)
    w = workloads.make(6)
    M, N, K = w["M"], w["N"], w["K"]
    ac, as_ = mx.alloc_codes(M, K, mx.E4M3FN), mx.alloc_scales(M, K)
    mx.mx_quantize(w["A"].cuda(), mx.E4M3FN, ac, as_)
    B = torch.from_numpy(w["B"]).cuda()
    C = torch.from_numpy(w["C0"]).cuda()
    f_bytes = mx.mx_codes_bytes(mx.E4M3FN, M, K) + mx.mx_scales_bytes(mx.SCALES_ROWMAJOR, M, K) + 4 * K * N + 8 * M * N

    def f32b(i):
        mx.mx_block_matmul_f32b(ac, as_, mx.E4M3FN, B, M, C)

    f32b(0)
    mx.mx_device_status()
    with ClockSampler(dev_index) as clk:
        sec, dist = timed(f32b, 1, steps, warmup, world)
    mx.mx_device_status()
    ck = clk.summary()
    flops = 2.0 * M * N * K
    gbs = f_bytes * steps / sec / 1e9
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = ck["sm_max_mhz"] or 2070.0
    alu_peak = sms * FFMA_PER_SM_CLK * 2 * mhz * 1e6 / 1e12
    out["block_matmul_f32b"] = {
        "workload": workloads.NAMES[6], "M": M, "N": N, "K": K, "formats": "E4M3 x f32",
        "us_per_step": sec / steps * 1e6, "dist": dist, "gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
        "bytes": f_bytes,
        "tflops": flops * steps / sec / 1e12, "ffma_peak_tflops": alu_peak,
        "alu_frac": flops * steps / sec / 1e12 / alu_peak, "launches_per_step": 1, "clocks": ck}
    del B, C, ac, as_, w
    torch.cuda.empty_cache()

    # ---- quantize along axis 0, dequantize to bf16, fold_scale: workload 2's tensor
    w = workloads.make(2)
    rows, cols = w["rows"], w["cols"]
    n = rows * cols
    qb = 2 * n + n + n // 32
    db = n + n // 32 + 2 * n
    fb = 2 * (n // 32)
    x0 = w["x"].cuda()
    nsets = sets_for(qb + db)
    sets = [{"x": x0.clone(), "codes": mx.alloc_codes(rows, cols, mx.E4M3FN), "scales": mx.alloc_scales(rows, cols),
             "y": torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")} for _ in range(nsets)]

    def q_axis0(i):
        s = sets[i]
        mx.mx_quantize_axis(s["x"], 0, mx.E4M3FN, s["codes"], s["scales"])

    def deq_bf16(i):
        s = sets[i]
        mx.mx_dequantize_bf16(s["codes"], s["scales"], rows, cols, mx.E4M3FN, s["y"])

    def fold(i):
        s = sets[i]
        mx.mx_fold_scale(s["scales"], rows, cols, 2.0)

    for i in range(nsets):
        q_axis0(i)
    mx.mx_device_status()
    k = max(steps, 200)
    sec_q, dist_q = timed(q_axis0, nsets, k, 3, world)
    sec_d, dist_d = timed(deq_bf16, nsets, k, 3, world)
    sec_f, dist_f = timed(fold, nsets, k, 3, world)
    mx.mx_device_status()
    for name, b, sec_k, dk, what in (
            ("quantize_axis0", qb, sec_q, dist_q, "bf16 4096x4096 -> MXFP8, blocks down the columns"),
            ("dequantize_bf16", db, sec_d, dist_d, "MXFP8 4096x4096 -> bf16"),
            ("fold_scale", fb, sec_f, dist_f, "scale bytes of a 4096x4096 MX tensor, times 2")):
        g = b * k / sec_k / 1e9
        out[name] = {"what": what, "us": sec_k / k * 1e6, "dist": dk, "gbs": g, "hbm_frac": g / peaks["hbm_gbs"],
                     "bytes": b, "nsets": nsets}
    del sets, x0
    torch.cuda.empty_cache()
    return out


TRAFFIC_ROWS = TRAFFIC_COLS = 16384


def traffic_case(mx, launches):
    """The headline kernels on a bf16 16384 x 16384 tensor (seeded N(0,1)):
    the dequantized f32 output (1 GiB) is eight times L2, so the DRAM bytes an
    ncu capture counts for one launch are its steady-state traffic (a launch
    of the 4096 x 4096 workload ends with most of its output still in L2).
    Runs quantize once, then `launches` dequantize and quantize launches in
    turn; the capture picks one of each."""
    torch.manual_seed(0)
    rows, cols = TRAFFIC_ROWS, TRAFFIC_COLS
    x = torch.randn(rows, cols, device="cuda").to(torch.bfloat16)
    codes, scales = mx.alloc_codes(rows, cols, mx.E4M3FN), mx.alloc_scales(rows, cols)
    y = torch.empty(rows, cols, device="cuda")
    for _ in range(max(1, launches)):
        mx.mx_quantize(x, mx.E4M3FN, codes, scales)
        mx.mx_dequantize(codes, scales, rows, cols, mx.E4M3FN, y)
    mx.mx_device_status()
    torch.cuda.synchronize()
    q, d = headline_bytes(rows, cols)
    return {"rows": rows, "cols": cols, "launches": launches, "quantize_algorithmic_bytes": q,
            "dequantize_algorithmic_bytes": d}


def headline_kernel_digest() -> str:
    """sha256 of the source the headline kernels are built from: the sections
    of mx_quant.cu from its top through the dequantize kernel (loads, the
    quantize kernels, the dequantize decoders and kernel), and the device
    headers they include.  Other kernels in the same file do not change it."""
    import hashlib
    csrc = os.path.join(ROOT, "bit_gemm_gb300", "csrc")
    with open(os.path.join(csrc, "mx_quant.cu")) as f:
        text = f.read()
    end = text.index("// ---------------------------------------------------------------- fold_scale")
    h = hashlib.sha256(text[:end].encode())
    for name in ("mx_quant_block.cuh", "mx_device.cuh", "mx_internal.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(key: str):
    """DRAM bytes per launch from the committed ncu capture, or None when the
    headline kernels' source has changed since the counters were taken."""
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(prof):
        return None
    with open(prof) as f:
        d = json.load(f)
    if headline_kernel_digest() != d.get("headline_kernel_sha256"):
        return None
    return d.get(key)


# ---------------------------------------------------------- CPU baseline

def oracle_step_rate(rows_sample: int, x_full: torch.Tensor, reps: int = 1):
    """Oracle quantize + dequantize of `rows_sample` rows of the workload; returns (seconds, bytes)."""
    import oracle
    xs = x_full[:rows_sample].float().numpy()
    cols = xs.shape[1]
    t0 = time.perf_counter()
    for _ in range(reps):
        c, s = oracle.quantize(xs, oracle.E4M3)
        oracle.dequantize(c, s, cols, oracle.E4M3)
    dt = time.perf_counter() - t0
    qb, db = headline_bytes(rows_sample, cols)
    return dt, (qb + db) * reps


class oracle_threads:
    """Run the oracle with n OpenMP threads inside the block."""

    def __init__(self, n):
        self.n = n

    def __enter__(self):
        import oracle
        self.saved = oracle.num_threads()
        oracle.set_threads(self.n)
        return self

    def __exit__(self, *exc):
        import oracle
        oracle.set_threads(self.saved)
        return False


def headline_oracle_rate(x_full: torch.Tensor, target_s: float):
    """Oracle quantize + dequantize of the headline workload: rows sampled and
    passes repeated until about target_s seconds; returns (GB/s, sample text)."""
    dt, _ = oracle_step_rate(8, x_full)
    per_row = max(dt / 8, 1e-6)
    rows = int(min(x_full.shape[0], max(8, target_s / per_row)))
    reps = max(1, min(50, int(round(target_s / (per_row * rows)))))
    dt, nbytes = oracle_step_rate(rows, x_full, reps)
    return nbytes / dt / 1e9, f"{rows} of 4096 rows of the bf16 4096x4096 workload (quantize + dequantize), " \
                              f"{reps} passes, {dt:.1f} s"


def cpu_baseline(x_full: torch.Tensor, target_s: float = 8.0):
    """The oracle, as it stands, on the host cores: quantize + dequantize of a
    sample of the headline workload, on every core and on one core."""
    import oracle
    threads = oracle.num_threads()
    value, sample = headline_oracle_rate(x_full, target_s)
    with oracle_threads(1):
        v1, s1 = headline_oracle_rate(x_full, target_s / 3)
    # workload 1 in full: quantize A and Bt (f32 128 x 256) to MXFP4, dequantize both, the product
    w1 = workloads.make(1)
    t0 = time.perf_counter()
    (ac, as_), (bc, bs) = oracle.quantize(w1["A"], oracle.E2M1), oracle.quantize(w1["Bt"], oracle.E2M1)
    t_q = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.dequantize(ac, as_, w1["K"], oracle.E2M1)
    oracle.dequantize(bc, bs, w1["K"], oracle.E2M1)
    t_d = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.block_matmul(ac, as_, oracle.E2M1, bc, bs, oracle.E2M1, w1["M"], w1["N"], w1["K"], w1["C0"])
    t_g = time.perf_counter() - t0
    return {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
            "one_core": {"value": v1, "unit": "GB/s", "cores": 1, "sample": s1},
            "workload1_full_us": {"quantize_A_and_Bt": t_q * 1e6, "dequantize_both": t_d * 1e6,
                                  "block_matmul": t_g * 1e6}}


def oracle_gemm_baseline(w, cfg, a_key, b_key, quant_a, rows_sample):
    """The oracle's block_matmul (binary64, every element decoded in every
    product) and, where the workload quantizes its activations, the oracle's
    quantize of them, on every host core and on one core.  Operands are
    quantized by the oracle from the workload's host tensors (untimed).  The
    product runs on min(M, rows_sample) rows of A (every column of B) and is
    extrapolated linearly in M; one core runs one row."""
    import oracle
    fmt = {3: (oracle.E4M3, oracle.E2M1), 4: (oracle.E4M3, oracle.E4M3), 5: (oracle.E2M1, oracle.E2M1)}[cfg]
    M, N, K = w["M"], w["N"], w["K"]
    a = w[a_key]
    a = a.float().numpy() if isinstance(a, torch.Tensor) else np.asarray(a, np.float32)
    b = w[b_key]
    b = b.float().numpy() if isinstance(b, torch.Tensor) else np.asarray(b, np.float32)
    out = {"cores": oracle.num_threads()}
    if quant_a:
        in_bytes = M * K * (2 if isinstance(w[a_key], torch.Tensor) and w[a_key].dtype == torch.bfloat16 else 4)
        nbytes = in_bytes + M * (K // 2 if fmt[0] == oracle.E2M1 else K) + M * (K // 32)
        t0 = time.perf_counter()
        oracle.quantize(a, fmt[0])
        dt = time.perf_counter() - t0
        out["act_quantize"] = {"s": dt, "gbs": nbytes / dt / 1e9, "rows": M, "sample": "full activation tensor"}
    bc, bs = oracle.quantize(b, fmt[1])
    r = min(M, rows_sample)
    ac, as_ = oracle.quantize(a[:r], fmt[0])
    c0 = np.ascontiguousarray(w["C0"][:r], np.float32)
    t0 = time.perf_counter()
    oracle.block_matmul(ac, as_, fmt[0], bc, bs, fmt[1], r, N, K, c0)
    dt = time.perf_counter() - t0
    full_s = dt * M / r
    out["block_matmul"] = {"s_sample": dt, "rows": r, "s_full_size": full_s,
                           "tflops": 2.0 * M * N * K / full_s / 1e12,
                           "sample": "full size" if r == M else f"first {r} of {M} rows, extrapolated linearly in M"}
    n1 = min(N, 4096)
    with oracle_threads(1):
        t0 = time.perf_counter()
        oracle.block_matmul(ac[:1], as_[:1], fmt[0], bc[:n1], bs[:n1], fmt[1], 1, n1, K,
                            np.ascontiguousarray(c0[:1, :n1]))
        d1 = time.perf_counter() - t0
    out["block_matmul_one_core"] = {"s_sample": d1, "s_full_size": d1 * M * N / n1,
                                    "tflops": 2.0 * n1 * K / d1 / 1e12,
                                    "sample": f"1 of {M} rows x {n1} of {N} columns on one core, "
                                              f"extrapolated linearly in M and N"}
    return out


# ------------------------------------------------------------------- main

def run_reference(args, world, rank):
    """The oracle as the reference arm: same metric and workload, each step a
    bounded sample of rows, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    w = workloads.make(2)
    x = w["x"]
    dt, _ = oracle_step_rate(8, x)
    per_row = max(dt / 8, 1e-6)
    budget = 120.0
    rows = int(max(1, min(4096, budget / max(1, args.steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        oracle_step_rate(rows, x)
    total_t, total_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_step_rate(rows, x)
        total_t += dt
        total_b += nb
    value = total_b / total_t / 1e9
    sample = f"{rows} of 4096 rows of the bf16 4096x4096 workload per step (quantize + dequantize)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": HEADLINE, "sample_rows_per_step": rows},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def summarize(line):
    """The line's main figures in a few keys (GEMM times in us, fractions of
    their denominators)."""
    r3 = lambda v: None if v is None else round(v, 3)
    out = {"step_hbm_frac": r3(line["hbm_frac"]),
           "quantize_frac": r3(line["kernels"]["quantize"]["frac"]),
           "dequantize_frac": r3(line["kernels"]["dequantize"]["frac"])}
    for g in line["block_matmul"] or []:
        key = g["workload"].split("_")[0]
        out[key] = {"gemm_us": round(g["us_gemm"], 1), "tensor_frac": r3(g["tensor_frac"]),
                    "hbm_frac": r3(g["hbm_frac"]), "step_us": round(g["us_per_step"], 1)}
        if "act_quantize" in g:
            out[key]["act_q_us"] = round(g["act_quantize"]["us"], 1)
            out[key]["act_q_hbm_frac"] = r3(g["act_quantize"]["hbm_frac"])
        if "fused" in g:
            out[key]["fused_us"] = round(g["fused"]["us_per_step"], 1)
        if "rowmajor_ws" in g:
            out[key]["rowmajor_ws_us"] = round(g["rowmajor_ws"]["us"], 1)
        if "rowmajor_direct" in g:
            out[key]["rowmajor_direct_us"] = round(g["rowmajor_direct"]["us"], 1)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--gemm-steps", type=int, default=20)
    ap.add_argument("--no-gemm", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--only", choices=["headline", "decode", "square", "prefill", "next", "traffic"], default=None,
                    help="run one workload only, print its numbers and exit (profiling runs)")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="scale of M and N of the GEMM workloads with --only (1 = full size)")
    ap.add_argument("--oracle-rows", type=int, default=16,
                    help="rows of A in the CPU oracle's timed block_matmul sample (workloads 4 and 5)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    torch.cuda.set_device(local)
    import bit_gemm_gb300 as mx
    peaks = measured_peaks()
    dev_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local

    if args.only is not None:
        if args.only == "headline":
            hl = bench_headline(mx, args.steps, args.warmup, world, peaks, dev_index)
            out = {k: v for k, v in hl.items() if k not in ("x_host",)}
        elif args.only == "next":
            out = bench_next(mx, args.steps, args.warmup, world, peaks, dev_index)
        elif args.only == "traffic":
            out = traffic_case(mx, args.steps)
        else:
            cfg = {"decode": 3, "square": 4, "prefill": 5}[args.only]
            out = bench_gemm(mx, cfg, args.steps, args.warmup, world, peaks, args.scale, dev_index, mma_rates(mx))
        if rank == 0:
            print(json.dumps(out, default=str), flush=True)
        return
    hl = bench_headline(mx, args.steps, args.warmup, world, peaks, dev_index)
    e2e = bench_e2e(mx, hl, args.steps, world)
    gemms = []
    mma = None
    cpu_here = rank == 0 and world == 1 and not args.no_cpu
    if not args.no_gemm:
        mma = mma_rates(mx)
        for cfg in (3, 4, 5):
            # kernels of a few microseconds get 13x the steps, so a timed
            # region is whole graphs of hundreds of launches
            st = args.gemm_steps * (13 if cfg == 3 else 1)
            gemms.append(bench_gemm(mx, cfg, st, max(3, args.warmup), world, peaks, 1.0, dev_index, mma,
                                    args.oracle_rows if cpu_here else 0))
    nxt = None if args.no_gemm else bench_next(mx, args.gemm_steps * 13, max(3, args.warmup), world, peaks, dev_index)
    cpu = None
    if cpu_here:
        cpu = cpu_baseline(hl["x_host"])
        cpu["block_matmul"] = {g["workload"]: g.get("oracle") for g in gemms}

    dom = hl[hl["dominant"]]
    traffic = measured_traffic(f"{hl['dominant']}_mxfp8_4096")
    line = {
        "metric": METRIC, "value": hl["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": hl["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": HEADLINE, "rows": hl["rows"], "cols": hl["cols"],
                   "bytes_per_step": hl["bytes"], "parallelism": f"replicas x{world}",
                   "l2": f"rotating {hl['nsets']} buffer sets (> 3x L2) between steps; each step dequantizes "
                         f"the set quantized half a rotation earlier, so every counted byte crosses HBM",
                   "timing": "CUDA graphs of whole rotations, events on the launch stream; step_dist from 20 "
                             "further replays of the same graph"},
        "hbm_frac": hl["value"] / world / peaks["hbm_gbs"],
        "step_dist": hl["dist"],
        "roofline": {"bound": "hbm", "kernel": hl["dominant"], "achieved": dom["gbs"], "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": dom["frac"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": dom["bytes"], "us_per_launch": dom["us"],
                     "peak_source": f"{peaks['source']} hbm_gbs (MEASURED_PEAKS.json)"},
        "kernels": {"quantize": hl["quantize"], "dequantize": hl["dequantize"]},
        "block_matmul": gemms,
        "tensor_peaks_tflops": {
            "recipe_fp8": peaks["bf16_tflops"] * NOMINAL_RATIO["fp8"],
            "recipe_fp4": peaks["bf16_tflops"] * NOMINAL_RATIO["fp4"],
            "mma_measured_fp8": mma["fp8"] if mma else None, "mma_measured_fp4": mma["fp4"] if mma else None,
            "used": "per format, the larger of the recipe figure and the measured MMA rate"},
        "next": nxt,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": hl["launches"],
        "clocks": hl["clocks"],
    }
    line["summary"] = summarize(line)  # last, so a tail of the output still shows it
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
