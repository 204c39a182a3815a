"""The multi-rank plumbing of bench.py (replicas, barrier, max-over-ranks timing, whole-job
aggregate) on CPU with two gloo ranks; and the reference arm's rank rule."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from mixture_experts_layer_14_gb300.synthetic import WORKLOADS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_env()
    bench.dist_init(w)
    bench.dist_barrier(w)
    ms = 10.0 * (rank + 1)                       # rank 1 is the slower replica
    ms_max = bench.dist_max(ms, w)
    out[rank] = (r, w, ms_max, bench.whole_job_value(w, 4096, 5, ms_max))
    bench.dist_barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_aggregate():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][:3] == (0, 2, 20.0) and res[1][:3] == (1, 2, 20.0)
    # both ranks processed 4096 tokens per step for 5 steps in at most 20 ms
    assert res[0][3] == pytest.approx(2 * 4096 * 5 / 0.020)


def test_single_rank_defaults():
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_max(3.5, 1) == 3.5
    assert bench.whole_job_value(1, 4096, 10, 40.0) == pytest.approx(4096 * 10 / 0.040)


def test_reference_arm_prints_the_contract_line(capsys):
    """`bench.py --impl reference` on the tiny workload (CPU): one JSON line with the contract's
    keys, the oracle as the reference, e2e with no copies, and the cpu_baseline describing the
    run."""
    import json

    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2",
                       "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny"
    # the same workload definition as the GB300 arm's line, key for key
    assert line["config"] == bench.config_of(WORKLOADS["tiny"], 1)
    assert line["metric"] == bench.metric_of(WORKLOADS["tiny"])


def test_work_model_matches_the_stated_algorithmic_bytes():
    """The algorithmic bytes and FLOPs behind the roofline fractions, for the DSV3 forward with
    every expert active: gate/up 15.30 GB (257 weight sets, x once, h written) and 2.17 TFLOP,
    down 8.23 GB, combine 587 MB, gather 529 MB."""

    shape = WORKLOADS["dsv3_bf16_fwd"]
    m, flops, e_act = bench.work_model(shape, [128] * shape.E)
    assert e_act == 256
    assert m["gemm_fwd_gate_up"]["bytes"] == pytest.approx(
        2 * (257 * 2 * 7168 * 2048 + 4096 * 7168 + 9 * 4096 * 2048), rel=1e-12)
    assert m["gemm_fwd_gate_up"]["bytes"] == pytest.approx(15.30e9, rel=2e-3)
    assert m["gemm_fwd_gate_up"]["flops"] == pytest.approx(2.17e12, rel=5e-3)
    assert m["gemm_fwd_down"]["bytes"] == pytest.approx(8.23e9, rel=2e-3)
    assert m["combine"]["bytes"] == pytest.approx(587e6, rel=2e-3)
    assert m["gather"]["bytes"] == pytest.approx(529e6, rel=2e-3)
    # the layer's FLOPs per token: 2 d E + (k + 1) 6 d F
    assert flops == pytest.approx(4096 * (2 * 7168 * 256 + 9 * 6 * 7168 * 2048), rel=1e-12)
