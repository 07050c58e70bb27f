"""Benchmark of the Dual-AR decode step on GB300.

One step = one decode frame: a slow-decoder token through 36 layers, the
tied semantic head, and 9 fast-decoder steps of 4 layers (10 codebook ids).
Default workload: the full-size S2-Pro-shaped model with bf16 weights, batch
1, prefill 128 prompt ids, then the 896 decode frames that fill the static
KV cache of 1024 (the schedule of the tuna-fish README speed test
"prefill 128, decode 896").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline]

Prints one JSON line (rank 0).  `value` is frames/s over all ranks with the
weights already resident in HBM, timed with CUDA events on the library's
stream; `e2e` is the same metric through the public C API with host
buffers (prompt upload and every frame's download inside the timed region).
Multi-GPU: independent replicas, one per rank, no collective on the data
path (batch-1 decode is one serial dependency chain).
`--impl reference` times the CPU oracle (float64 NumPy) on a bounded sample
of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from synth import WORKLOADS, tensor_specs  # noqa: E402

METRIC = "Dual-AR decode frames/s at batch 1; achieved HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0
PAGE_LOAD_ELEMENTS = 7_377_351_168   # tuna-fish README, "Inference estimation"
# ncu DRAM bytes (read + write) of one 19456 x 2560 gate/up-shaped k_gemv
# launch, per weight format, from the capture of the kernel as it stands.
GATE_UP_TRAFFIC = {"bf16": 99_670_272 + 3_020_800, "fp8": 49_942_272 + 0}


# ---------------------------------------------------------------- accounting
def linear_bytes(weight_dtype: str, rows: int, cols: int) -> int:
    """Stored bytes of one [rows][cols] linear weight: bf16; e4m3 codes plus a
    float32 scale per row; or 4-bit rows (cols/2 code bytes, cols/16 block
    scales) plus a float32 scale per row."""
    if weight_dtype == "bf16":
        return rows * cols * 2
    if weight_dtype == "fp8":
        return rows * cols + rows * 4
    return rows * (cols // 2 + cols // 16) + rows * 4


def frame_bytes(d, weight_dtype: str, pos: int, batch: int = 1) -> dict:
    """Algorithmic HBM bytes of one decode step whose slow tokens sit at
    position `pos`: every weight streamed once (slow pass + 9 fast passes),
    and for each of the `batch` sequences the valid KV rows read and the new
    KV rows written (embedding rows are part of the weights)."""
    H, F = d.hidden, d.ffn
    lb = lambda r, c: linear_bytes(weight_dtype, r, c)
    layer = lb(d.qkv_dim, H) + lb(H, d.q_dim) + 2 * lb(F, H) + lb(H, F) + 2 * H * 2
    slow_w = d.slow_layers * layer + d.semantic_vocab * H * 2 + H * 2 + H * 2
    fast_w = d.fast_layers * layer + lb(d.codebook_size, H) + H * 2 + H * 2
    kv_row = d.kv_dim * 2                          # one K or V row of one layer, bf16
    kv_read = d.slow_layers * 2 * kv_row * (pos + 1)
    kv_read += sum(d.fast_layers * 2 * kv_row * (j + 1) for j in range(1, d.n_codebooks))
    kv_write = d.slow_layers * 2 * kv_row + d.fast_layers * 2 * kv_row * (d.n_codebooks)
    weights = slow_w + (d.n_codebooks - 1) * fast_w
    kv_read, kv_write = batch * kv_read, batch * kv_write
    return {"weights": weights, "kv_read": kv_read, "kv_write": kv_write,
            "total": weights + kv_read + kv_write}


def schedule_bytes(d, weight_dtype, prefill, frames) -> float:
    return float(np.mean([frame_bytes(d, weight_dtype, p)["total"]
                          for p in range(prefill, prefill + frames)]))


def schedule_plan(prefill: int, cap: int, steps: int, max_segments: int = 8):
    """(start position, frames) segments that time `steps` decode frames
    spread evenly over a schedule of `cap` frames after a `prefill`-id prompt
    (positions prefill .. prefill + cap - 1).  Whole passes over the schedule
    come first when steps >= cap; the rest is split into at most
    max_segments equal segments whose starts are evenly spaced."""
    plan = []
    full, rest = divmod(steps, cap)
    plan += [(prefill, cap)] * full
    if rest:
        n = min(max_segments, rest)
        sizes = [rest // n + (1 if i < rest % n else 0) for i in range(n)]
        for i, k in enumerate(sizes):
            span = cap - k
            start = prefill + (round(i * span / (n - 1)) if n > 1 else 0)
            plan.append((start, k))
    return plan


def workload_config(wl, world: int) -> dict:
    """The workload a bench line measures (both arms print the same dict)."""
    d = wl.dims
    return {"workload": wl.name, "batch": wl.batch, "prefill": wl.prefill,
            "decode_schedule": wl.decode, "max_seq_len": d.max_seq_len,
            "weights": wl.weight_dtype,
            "sampling": "greedy argmax" if not wl.top_k else f"top-k {wl.top_k}, Philox seed 1234",
            "l2": "inputs larger than L2: every frame streams all weights (>= 7 GB)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def max_over_ranks(x: float, device) -> float:
    """The largest x over the ranks of the default process group (x itself
    when there is one rank): a timed region lasts as long as its slowest rank."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the
    max-over-ranks time in milliseconds (replicas do equal work)."""
    return units_per_rank * world / (ms / 1e3)


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j.get("bf16_tflops", 1900.0)),
                "source": "of measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0, "source": "of fallback"}


def prefill_flops(d, P: int) -> float:
    """Algorithmic flops of a P-token prefill through the slow decoder:
    2 * P * (linear weights of the 36 layers) + causal attention
    (scores and weighted values, 2 * 2 * D per query-key pair and head)."""
    lin = d.qkv_dim * d.hidden + d.hidden * d.q_dim + 3 * d.hidden * d.ffn
    attn = 2 * 2 * d.n_heads * d.head_dim * P * (P + 1) / 2
    return d.slow_layers * (2.0 * P * lin + attn)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- inputs
def device_weights(d, seed: int, device):
    """Seeded N(0, 0.02) bf16 weights drawn on the device (torch Philox),
    norms 1.0; returns name -> torch tensor (bf16)."""
    import torch
    out = {}
    for idx, (name, shape, kind) in enumerate(tensor_specs(d)):
        if kind == "norm":
            out[name] = torch.ones(shape, dtype=torch.bfloat16, device=device)
            continue
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1_000_003 + idx)
        out[name] = (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 0.02
                     ).to(torch.bfloat16)
    return out


def host_bits(tensors) -> dict:
    import torch
    return {k: v.view(torch.int16).cpu().numpy().view(np.uint16) for k, v in tensors.items()}


# ---------------------------------------------------------------- oracle leg
def oracle_sample(wl, weights_bits, prompt, budget_s: float = 20.0) -> dict:
    """Oracle frames/s on a bounded sample: prefill (untimed), then decode
    frames until `budget_s` of CPU time has passed (at least one).  Batched
    workloads: one sequence (the oracle has no batching; per-sequence frames
    are the unit) with its prompt cut to 64 ids to bound the untimed part."""
    import oracle
    ref = oracle.DualAROracle(wl.dims, weights_bits, wl.weight_dtype)
    if wl.batch > 1:
        prompt = prompt[:1, :64]
    t0 = time.perf_counter()
    ref.prefill(prompt)
    t_prefill = time.perf_counter() - t0
    n, t0 = 0, time.perf_counter()
    while True:
        ref.decode_frame()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 8:
            break
    return {"value": n / el, "unit": "frames/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{wl.name}: oracle prefill of {prompt.shape[1]} ids ({t_prefill:.1f} s, untimed) "
                      f"then {n} decode frame(s) timed ({el:.1f} s); float64 NumPy, BLAS on all host cores"}


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=896)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--workload", default="full_bf16", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--profile-range", action="store_true",
                    help="mark the timed decode frames as the profiler range (ncu --profile-from-start off)")
    ap.add_argument("--op", default=None, choices=["gemv", "gemm", "skinny", "attn", "attn_prompt",
                                                   "prefill"],
                    help="time one kernel on its own instead of the decode step")
    ap.add_argument("--rows", type=int, default=19456)
    ap.add_argument("--cols", type=int, default=2560)
    ap.add_argument("--fp8", action="store_true")
    ap.add_argument("--nvfp4", action="store_true", help="--op gemv: 4-bit block-scaled rows")
    ap.add_argument("--m", type=int, default=None,
                    help="--op gemm / attn_prompt: prompt rows (1024); --op skinny: activation rows (16)")
    args = ap.parse_args()
    if args.op == "gemv":
        return run_gemv_case(args)
    if args.op == "gemm":
        args.m = args.m or 1024
        return run_gemm_case(args)
    if args.op == "skinny":
        args.m = args.m or 16
        return run_skinny_case(args)
    if args.op == "attn":
        return run_attn_case(args)
    if args.op == "attn_prompt":
        args.m = args.m or 1024
        return run_attn_prompt_case(args)
    if args.op == "prefill":
        return run_prefill_case(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = WORKLOADS[args.workload]
    d = wl.dims
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    if args.impl == "reference":
        return run_reference(args, wl, world, rank)

    import torch
    import torch.distributed as dist
    from dual_ar_decode_gb300 import Decoder
    from synth import make_prompt
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    tensors = device_weights(d, args.seed, device)
    B = wl.batch
    prompt = make_prompt(d, wl.prefill, seed=args.seed + rank * B, batch=B)
    want_cpu = (not args.no_cpu_baseline) and rank == 0 and world == 1
    bits = host_bits(tensors) if want_cpu else None
    dec = Decoder(d, wl.weight_dtype, device=local, max_batch=B)
    dec.load_weights(tensors)
    del tensors
    torch.cuda.empty_cache()
    sampling = {"top_k": wl.top_k, "seed": 1234} if wl.top_k else None
    stream = torch.cuda.ExternalStream(dec.stream(), device=device)

    # warm-up: prefill + W frames (captures the frame graph)
    dec.prefill(prompt, sampling)
    dec.decode_frames(min(args.warmup, wl.decode, d.max_seq_len - wl.prefill), sampling)

    # Timed frames are spread evenly over the decode schedule (positions
    # prefill .. max_seq_len - 1): segment i starts at plan[i][0], reached by
    # untimed decoding after an untimed prefill, and times plan[i][1] frames.
    cap = min(wl.decode, d.max_seq_len - wl.prefill)   # frames of the workload's schedule
    plan = schedule_plan(wl.prefill, cap, args.steps)
    total_ms = 0.0
    clocks = ClockSampler(local)
    positions = []
    clocks.start()
    for start, k in plan:
        dec.prefill(prompt, sampling)                    # untimed: resets position to P
        if start > wl.prefill:
            dec.decode_frames(start - wl.prefill, sampling)   # untimed: walk to the segment
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if args.profile_range:
            torch.cuda.profiler.start()
        dec.decode_frames(k, sampling)
        if args.profile_range:
            torch.cuda.synchronize(device)
            torch.cuda.profiler.stop()
        e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize(device)
        total_ms += e0.elapsed_time(e1)
        positions += list(range(start, start + k))
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, device)
    value = job_rate(args.steps * B, world, total_ms)   # sequence-frames/s
    info = dec.info()

    # dominant kernel, live: the slow gate/up GEMV (batch 1) or skinny
    # tensor-core GEMM (batch > 1) in its in-frame configuration
    prof_ms, prof_bytes = dec.profile_kernel(0 if B == 1 else 4, 4 * d.slow_layers)
    peaks = measured_peaks()
    achieved = prof_bytes / (prof_ms / 1e3) / 1e9

    # e2e through the public API with host buffers
    e2e_frames = min(args.steps, cap)
    torch.cuda.synchronize(device)
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    dec.prefill(prompt, sampling)
    for _ in range(e2e_frames):
        dec.decode_frame(sampling)
    h1.record(stream)
    h1.synchronize()
    e2e_value = job_rate(e2e_frames * B, world, max_over_ranks(h0.elapsed_time(h1), device))

    # prefill throughput (prompt ids uploaded from the host, frame 0 returned)
    pre_ms = []
    for _ in range(3):
        torch.cuda.synchronize(device)
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        dec.prefill(prompt, sampling)
        p1.record(stream)
        p1.synchronize()
        pre_ms.append(p0.elapsed_time(p1))
    pre = float(np.median(pre_ms))
    pre_tflops = B * prefill_flops(d, wl.prefill) / (pre / 1e3) / 1e12

    bytes_avg = float(np.mean([frame_bytes(d, wl.weight_dtype, p, B)["total"] for p in positions]))
    sched_bytes = float(np.mean([frame_bytes(d, wl.weight_dtype, p, B)["total"]
                                 for p in range(wl.prefill, wl.prefill + cap)]))
    frame_gbs = bytes_avg * (value / B) / world / 1e9
    page_gib = PAGE_LOAD_ELEMENTS * {"bf16": 2, "fp8": 1, "nvfp4": 0.5}[wl.weight_dtype] / 2 ** 30
    cpu = oracle_sample(wl, bits, prompt) if want_cpu else None
    dec.close()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "frames/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "fp8": "fp8-e4m3 weights, bf16 KV, f32 accumulate",
                      "nvfp4": "e2m1 + e4m3 block-scale weights, bf16 KV, f32 accumulate"}[wl.weight_dtype],
            "data": "synthetic: seeded N(0, 0.02) random-init weights, uniform prompt ids",
            "config": workload_config(wl, world),
            "timing": {"frames_timed": args.steps, "segments": [list(x) for x in plan],
                       "positions": [min(positions), max(positions)],
                       "bytes_per_frame_timed": round(bytes_avg),
                       "bytes_per_frame_schedule": round(sched_bytes),
                       "note": "segments (start position, frames) spread evenly over the "
                               "decode schedule; each reached by untimed decoding"},
            "tok_s": round(value, 3), "codebook_tok_s": round(10 * value, 3),
            "steps_per_s": round(value / B / world, 3),
            "prefill": {"tokens": wl.prefill * B, "ms": round(pre, 3),
                        "tok_s": round(B * wl.prefill / (pre / 1e3), 1),
                        "tflops": round(pre_tflops, 2), "bf16_peak_tflops": peaks["bf16_tflops"],
                        "frac": round(pre_tflops / peaks["bf16_tflops"], 4),
                        "note": "tcgen05 GEMMs (activations as bf16 hi+lo: tensor work is 2x the "
                                "algorithmic flops) + attention + frame-0 tail"},
            "frame_hbm": {"bytes_per_frame": round(bytes_avg), "achieved_gbs": round(frame_gbs, 1),
                          "peak_gbs": peaks["hbm_gbs"], "frac": round(frame_gbs / peaks["hbm_gbs"], 4),
                          "peak_source": peaks["source"],
                          "page_convention_gib_s": round(value / world * page_gib, 1)},
            "roofline": {"kernel": "k_gemv (slow gate/up, RMSNorm prologue, SwiGLU epilogue)" if B == 1
                         else f"k_umma_skinny (slow gate/up, {B} rows, split-K tcgen05, SwiGLU epilogue)",
                         "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "peak_source": peaks["source"], "bytes_per_launch": prof_bytes,
                         "ms_per_launch": round(prof_ms, 5),
                         # ncu dram__bytes_read.sum + dram__bytes_write.sum of one gate/up
                         # launch of this kernel in its current form (None: not captured)
                         "traffic": GATE_UP_TRAFFIC.get(wl.weight_dtype) if B == 1 else None},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 3), "unit": "frames/s",
                    "h2d_bytes_per_step": round((B * wl.prefill * 4 + 4 * (e2e_frames + 1)) / e2e_frames, 2),
                    "d2h_bytes_per_step": 4 + 40 * B,
                    "note": "tf_prefill (host prompt) + one tf_decode_frame per frame (host frame out)"},
            "gpu_launches": info["graph_nodes"] * args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_gemv_case(args):
    """The decode GEMV alone (tf_op_gemv, no prologue or epilogue) on
    `rows` x `cols` weights, bf16 or e4m3 + row scales: K launches chained
    with PDL, each on a distinct copy of the matrix (about 2.5 GB in all, far
    above L2), after W warm-up passes.  Prints one JSON line."""
    import torch
    from dual_ar_decode_gb300 import op_gemv
    from dual_ar_decode_gb300.binding import TF_DTYPE_BF16, TF_DTYPE_FP8_E4M3
    from dual_ar_decode_gb300.binding import TF_DTYPE_NVFP4
    dev = torch.device("cuda", 0)
    fmt = "nvfp4" if getattr(args, "nvfp4", False) else "fp8" if args.fp8 else "bf16"
    mat = linear_bytes(fmt, args.rows, args.cols) - (0 if fmt == "bf16" else args.rows * 4)
    reps = max(args.steps, int(2.5e9 // mat))
    g = torch.Generator(device=dev).manual_seed(args.seed)
    W = torch.randint(0, 120, (reps * mat,), dtype=torch.uint8, device=dev, generator=g)
    if fmt == "bf16":
        W = (W.view(torch.int16) & 0x3FFF).view(torch.uint8)   # finite bf16
    S = torch.rand(reps * args.rows, device=dev, generator=g) if fmt != "bf16" else None
    x = torch.randn(args.cols, device=dev, generator=g)
    y = torch.empty(args.rows, device=dev)
    dt = {"bf16": TF_DTYPE_BF16, "fp8": TF_DTYPE_FP8_E4M3, "nvfp4": TF_DTYPE_NVFP4}[fmt]
    for _ in range(args.warmup):
        op_gemv(W.data_ptr(), dt, S.data_ptr() if S is not None else None, args.rows, args.cols,
                x.data_ptr(), y.data_ptr(), reps)
    ms = op_gemv(W.data_ptr(), dt, S.data_ptr() if S is not None else None, args.rows, args.cols,
                 x.data_ptr(), y.data_ptr(), reps)
    nbytes = linear_bytes(fmt, args.rows, args.cols) + args.cols * 4 + args.rows * 4
    peaks = measured_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"op": "gemv", "rows": args.rows, "cols": args.cols,
                      "weights": fmt, "launches": reps,
                      "us_per_launch": round(ms * 1e3, 3), "achieved_gbs": round(gbs, 1),
                      "peak_gbs": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4),
                      "peak_source": peaks["source"]}), flush=True)


def run_gemm_case(args):
    """The prompt GEMM alone (tf_op_gemm: tcgen05 tensor cores, activations
    as bf16 hi + lo parts): C[m][rows] = A[m][cols] W[rows][cols]^T, W
    steps times after W warm-up calls.  Prints one JSON line; tflops count
    the algorithmic 2*m*rows*cols once."""
    import torch
    from dual_ar_decode_gb300 import op_gemm
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(args.seed)
    A = torch.randn(args.m, args.cols, device=dev, generator=g)
    W = (torch.randn(args.rows, args.cols, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    C = torch.empty(args.m, args.rows, device=dev)
    for _ in range(args.warmup):
        op_gemm(A.data_ptr(), W.data_ptr(), args.m, args.rows, args.cols, C.data_ptr())
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        op_gemm(A.data_ptr(), W.data_ptr(), args.m, args.rows, args.cols, C.data_ptr())
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    tflops = 2.0 * args.m * args.rows * args.cols / (ms / 1e3) / 1e12
    peaks = measured_peaks()
    print(json.dumps({"op": "gemm", "m": args.m, "rows": args.rows, "cols": args.cols,
                      "ms_per_call": round(ms, 4), "tflops": round(tflops, 2),
                      "bf16_peak_tflops": peaks["bf16_tflops"],
                      "frac": round(tflops / peaks["bf16_tflops"], 4),
                      "note": "per call: hi/lo split + GEMM; tensor work is 2x the algorithmic flops"}),
          flush=True)


def run_skinny_case(args):
    """The batched step's skinny tensor-core GEMMs in their in-frame
    configuration (tf_profile_kernel 4..7: deferred-RMSNorm input, fused
    epilogue, launches chained with PDL and replayed as a graph) over --m
    activation rows, on a full-width model cut to 8 slow layers (1.6 GB of
    distinct bf16 weights per pass, far above L2; --fp8 / --nvfp4: the same
    linears quantised, read as they are).  Prints one JSON line."""
    import torch
    from dual_ar_decode_gb300 import Decoder
    from synth import FULL
    d = FULL.replace(slow_layers=8, fast_layers=1, max_seq_len=64)
    dev = torch.device("cuda", 0)
    w = device_weights(d, args.seed, dev)
    fmt = "nvfp4" if getattr(args, "nvfp4", False) else "fp8" if args.fp8 else "bf16"
    dec = Decoder(d, fmt, max_batch=args.m)
    dec.load_weights(w)
    del w
    peaks = measured_peaks()
    out = {}
    for which, name in ((4, "gate_up_19456x2560"), (5, "qkv_6144x2560"), (6, "o_2560x4096"),
                        (7, "down_2560x9728")):
        for _ in range(args.warmup):
            dec.profile_kernel(which, 16)
        ms, nbytes = dec.profile_kernel(which, 64)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"us_per_launch": round(ms * 1e3, 3), "bytes_per_launch": nbytes,
                     "achieved_gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)}
    dec.close()
    print(json.dumps({"op": "skinny", "rows_m": args.m, "weights": fmt, "shapes": out, "peak_gbs": peaks["hbm_gbs"],
                      "peak_source": peaks["source"]}), flush=True)


def run_attn_case(args):
    """Decode attention alone (tf_op_attention_noalloc: the staged split-key
    kernel, no device allocation per call) for one query row at position
    T - 1 of a full-size KV head layout (32 q / 8 kv heads of 128, T = 1024,
    38 key slices as in the batch-1 frame), cycling over 64 distinct caches
    (268 MB, above L2).  Each call waits for its error word, so the time per
    call includes one host round trip.  Prints one JSON line."""
    import ctypes
    import torch
    from dual_ar_decode_gb300 import binding
    dev = torch.device("cuda", 0)
    T, Hq, Hkv, D, S, ncache = 1024, 32, 8, 128, 38, 64
    g = torch.Generator(device=dev).manual_seed(args.seed)
    K = (torch.randn(ncache, Hkv, T, D, device=dev, generator=g) * 0.5).to(torch.bfloat16)
    V = (torch.randn(ncache, Hkv, T, D, device=dev, generator=g) * 0.5).to(torch.bfloat16)
    q = torch.randn(Hq * D, device=dev, generator=g)
    out = torch.empty(Hq * D, device=dev)
    L = binding.lib()
    stream = torch.cuda.current_stream(dev).cuda_stream

    def call(i):
        st = L.tf_op_attention_noalloc(q.data_ptr(), K[i % ncache].data_ptr(), V[i % ncache].data_ptr(),
                                       T, Hq, Hkv, D, 1, T - 1, S, out.data_ptr(), ctypes.c_void_p(stream))
        if st:
            raise RuntimeError(f"tf_op_attention_noalloc returned {st}")

    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        call(i)
    e1.record()
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    nbytes = 2 * Hkv * T * D * 2 + 2 * Hq * D * 4
    print(json.dumps({"op": "attn", "T": T, "Hq": Hq, "Hkv": Hkv, "D": D, "slices": S,
                      "us_per_call_incl_host_sync": round(us, 3), "kv_bytes": nbytes,
                      "note": "one query row at position T-1; each call syncs for its error word"}),
          flush=True)


def run_attn_prompt_case(args):
    """Causal prompt attention alone (tf_op_attention_prompt: tcgen05, one
    CTA per 128 query rows and head): --m rows at positions m..2m-1 of a
    full-size head layout (32 q / 8 kv heads of 128, T = 2m), so each row
    attends to m + 1 .. 2m keys.  steps calls after W warm-up calls; each call
    splits the queries into bf16 parts and allocates its scratch.  Prints one
    JSON line; tflops count 4 * Hq * D * (keys summed over rows) once."""
    import torch
    from dual_ar_decode_gb300 import op_attention_prompt
    dev = torch.device("cuda", 0)
    m = args.m
    T, Hq, Hkv, D = 2 * m, 32, 8, 128
    g = torch.Generator(device=dev).manual_seed(args.seed)
    q = torch.randn(m, Hq * D, device=dev, generator=g)
    K = torch.randn(Hkv, T, D, device=dev, generator=g).to(torch.bfloat16)
    V = torch.randn(Hkv, T, D, device=dev, generator=g).to(torch.bfloat16)
    out = torch.empty(m, Hq * D, device=dev)
    call = lambda: op_attention_prompt(q.data_ptr(), K.data_ptr(), V.data_ptr(), T, Hq, Hkv, D, m, m,
                                       out.data_ptr())
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    keys = sum(m + r + 1 for r in range(m))
    tflops = 4.0 * Hq * D * keys / (ms / 1e3) / 1e12
    peaks = measured_peaks()
    print(json.dumps({"op": "attn_prompt", "rows": m, "T": T, "Hq": Hq, "Hkv": Hkv, "D": D,
                      "ms_per_call": round(ms, 4), "tflops": round(tflops, 2),
                      "bf16_peak_tflops": peaks["bf16_tflops"], "frac": round(tflops / peaks["bf16_tflops"], 4),
                      "note": "per call: query split + allocation + kernel; tensor work ~4x the "
                              "algorithmic flops (hi + lo parts, whole tiles up to the diagonal)"}),
          flush=True)


def run_prefill_case(args):
    """tf_prefill alone on the workload's model and prompt (--workload):
    W warm-up prefills, then `steps` timed ones (CUDA events on the
    library's stream); with --profile-range the last one is bracketed by the
    profiler range.  Prints one JSON line (ms, prompt tokens/s, algorithmic
    TFLOP/s and their fraction of the measured bf16 burst peak)."""
    import torch
    from dual_ar_decode_gb300 import Decoder
    from synth import make_prompt
    wl = WORKLOADS[args.workload]
    d = wl.dims
    dev = torch.device("cuda", 0)
    tensors = device_weights(d, args.seed, dev)
    dec = Decoder(d, wl.weight_dtype, max_batch=wl.batch)
    dec.load_weights(tensors)
    del tensors
    torch.cuda.empty_cache()
    prompt = make_prompt(d, wl.prefill, seed=args.seed, batch=wl.batch)
    stream = torch.cuda.ExternalStream(dec.stream(), device=dev)
    for _ in range(args.warmup):
        dec.prefill(prompt)
    ts = []
    for i in range(args.steps):
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        last = args.profile_range and i == args.steps - 1
        e0.record(stream)
        if last:
            torch.cuda.profiler.start()
        dec.prefill(prompt)
        if last:
            torch.cuda.synchronize(dev)
            torch.cuda.profiler.stop()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    dec.close()
    ms = float(np.median(ts))
    peaks = measured_peaks()
    tflops = wl.batch * prefill_flops(d, wl.prefill) / (ms / 1e3) / 1e12
    print(json.dumps({"op": "prefill", "workload": wl.name, "tokens": wl.prefill * wl.batch,
                      "ms": round(ms, 3), "tok_s": round(wl.prefill * wl.batch / (ms / 1e3), 1),
                      "tflops": round(tflops, 1), "bf16_peak_tflops": peaks["bf16_tflops"],
                      "frac": round(tflops / peaks["bf16_tflops"], 4), "peak_source": peaks["source"],
                      "note": "prompt ids from the host, frame 0 back to the host; flops: the slow "
                              "decoder's linears and causal attention over the prompt rows"}), flush=True)


def run_reference(args, wl, world, rank):
    """The oracle (float64 NumPy on the host cores) on the same workload:
    untimed prefill and min(W, 8) untimed warm-up frames, then decode frames
    one per step, timed, until `steps` frames or about 90 s of CPU time
    (the line reports the frames actually timed as `steps`).  Batched
    workloads run one sequence with its prompt cut to 64 ids: the oracle has
    no batching, and per-sequence frames are the unit."""
    if rank != 0:
        return
    import oracle
    from synth import make_prompt, make_weights
    d = wl.dims
    w = make_weights(d, args.seed)
    prompt = make_prompt(d, wl.prefill, seed=args.seed, batch=wl.batch)
    if wl.batch > 1:
        prompt = prompt[:1, :64]
    sampling = {"top_k": wl.top_k, "seed": 1234} if wl.top_k else None
    ref = oracle.DualAROracle(d, w, wl.weight_dtype)
    t0 = time.perf_counter()
    ref.prefill(prompt, sampling)
    t_prefill = time.perf_counter() - t0
    warm = min(args.warmup, 8, d.max_seq_len - prompt.shape[1] - 1)
    for _ in range(warm):
        ref.decode_frame(sampling)
    budget_s, n, el = 90.0, 0, 0.0
    limit = min(args.steps, d.max_seq_len - prompt.shape[1] - warm)
    while n < limit:
        t0 = time.perf_counter()
        ref.decode_frame(sampling)
        el += time.perf_counter() - t0
        n += 1
        if el >= budget_s:
            break
    v = n / el
    cores = os.cpu_count()
    sample = (f"{wl.name}: oracle prefill of {prompt.shape[1]} ids ({t_prefill:.1f} s, untimed), "
              f"{warm} untimed warm-up frames, then {n} decode frame(s) timed ({el:.1f} s); "
              f"float64 NumPy, BLAS on all host cores")
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "frames/s",
            "n_gpus": world, "steps": n, "steps_requested": args.steps, "warmup": warm,
            "ms_per_step": round(1e3 / v, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic: seeded N(0, 0.02) random-init "
            "weights, uniform prompt ids",
            "config": workload_config(wl, world),
            "cpu_baseline": {"value": round(v, 5), "unit": "frames/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 5), "unit": "frames/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
