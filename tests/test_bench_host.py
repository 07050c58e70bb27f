"""Host logic of the benchmark, on CPU: the byte accounting behind
`frame_hbm`, and the multi-rank reductions (max over ranks, whole-job
throughput) with two gloo ranks.  Decode does not shard: extra ranks are
replicas, so the only cross-rank step is the timing reduction."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
from synth import FULL, TINY, tensor_specs


def _frame_weight_bytes_from_specs(d, fmt):
    """Weights one decode frame reads, summed from the model's tensor list:
    every slow tensor but the text embedding, plus its semantic slice and one
    embedding row; nine passes over the fast tensors but the codebook tables,
    plus one codebook row each.  Quantised linears: bytes per element (1 for
    e4m3, 1/2 + 1/16 for 4-bit codes and block scales) plus 4 per row."""
    per = {"bf16": 2.0, "fp8": 1.0, "nvfp4": 0.5 + 1.0 / 16}[fmt]
    slow = fast = 0
    for name, shape, kind in tensor_specs(d):
        n = int(np.prod(shape))
        nbytes = n * per + (shape[0] * 4 if fmt != "bf16" else 0) if kind == "linear" else n * 2
        if name.startswith("slow."):
            slow += nbytes
        elif name == "fast.cb_embed":
            fast += d.hidden * 2
        elif name.startswith("fast."):
            fast += nbytes
    slow += d.semantic_vocab * d.hidden * 2 + d.hidden * 2
    return slow + (d.n_codebooks - 1) * fast


@pytest.mark.parametrize("d", [TINY, FULL])
@pytest.mark.parametrize("fmt", ["bf16", "fp8", "nvfp4"])
def test_frame_weight_bytes_match_the_tensor_list(d, fmt):
    fb = bench.frame_bytes(d, fmt, 10)
    assert fb["weights"] == _frame_weight_bytes_from_specs(d, fmt)


def test_frame_bytes_full_size_total_and_batch_scaling():
    # 7,371,909,120 weight elements per frame at full size (slow pass + 9 fast passes)
    assert bench.frame_bytes(FULL, "bf16", 0)["weights"] == 2 * 7_371_909_120
    one = bench.frame_bytes(FULL, "bf16", 600)
    b16 = bench.frame_bytes(FULL, "bf16", 600, 16)
    assert b16["weights"] == one["weights"]                 # weights once per step
    assert b16["kv_read"] == 16 * one["kv_read"]            # KV once per sequence
    assert b16["kv_write"] == 16 * one["kv_write"]
    # slow KV read at position p: 36 layers x (K and V) x (p + 1) rows of 1024 bf16
    slow_kv = 36 * 2 * 1024 * 2 * 601
    fast_kv = sum(4 * 2 * 1024 * 2 * (j + 1) for j in range(1, 10))
    assert one["kv_read"] == slow_kv + fast_kv


def test_job_rate_counts_every_rank():
    assert bench.job_rate(100, 1, 50.0) == pytest.approx(2000.0)
    assert bench.job_rate(100, 4, 50.0) == pytest.approx(8000.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        m = bench.max_over_ranks(ms, torch.device("cpu"))
        out.put((rank, m, bench.job_rate(100, world, m)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 15.0
        assert v == pytest.approx(200 / 0.015)


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(12.5, torch.device("cpu")) == 12.5


def test_reference_arm_is_rank0_only():
    class A:
        seed = 0
        steps = 1
        warmup = 3
    # rank 1 of a torchrun job returns at once without running the oracle
    assert bench.run_reference(A(), bench.WORKLOADS["tiny"], 2, 1) is None


@pytest.mark.parametrize("steps", [1, 5, 20, 64, 895, 896, 897, 2000])
def test_schedule_plan_spreads_timed_frames_over_the_schedule(steps):
    prefill, cap = 128, 896
    plan = bench.schedule_plan(prefill, cap, steps)
    assert sum(k for _, k in plan) == steps
    for start, k in plan:
        assert k >= 1 and prefill <= start and start + k <= prefill + cap
    partial = plan[steps // cap:]
    if len(partial) > 1:
        # the first segment starts the schedule, the last one ends it
        assert partial[0][0] == prefill
        assert partial[-1][0] + partial[-1][1] == prefill + cap
        starts = [s for s, _ in partial]
        assert starts == sorted(starts)


def test_reference_arm_times_what_it_prints(capsys):
    """The oracle arm prints the workload config the GPU arm prints and, as
    `steps`, the number of frames it actually timed."""
    import json

    class A:
        seed = 0
        steps = 3
        warmup = 3
    wl = bench.WORKLOADS["tiny"]
    bench.run_reference(A(), wl, 1, 0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.workload_config(wl, 1)
    assert line["steps"] == 3 and line["warmup"] == 3
    assert line["ms_per_step"] == pytest.approx(1e3 / line["value"], rel=1e-3)
    assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]


@pytest.mark.parametrize("d", [TINY, FULL])
@pytest.mark.parametrize("P", [1, 128, 1024])
def test_prefill_flops_from_the_tensor_list(d, P):
    """The prefill TFLOP/s that `--op prefill` prints: 2 flops per slow-layer
    linear weight element and prompt row (summed from the tensor list, the
    slow head excluded: only the last row reaches it), plus causal attention,
    2 * 2 * head_dim flops per (query, key <= query) pair and query head."""
    lin = sum(int(np.prod(shape)) for name, shape, kind in tensor_specs(d)
              if kind == "linear" and name.startswith("slow.") and name.split(".")[1].isdigit())
    attn = d.slow_layers * d.n_heads * 4 * d.head_dim * (P * (P + 1) // 2)
    assert bench.prefill_flops(d, P) == pytest.approx(2 * P * lin + attn, rel=1e-12)
