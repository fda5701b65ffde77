"""The multi-GPU path of bench.py on CPU: world size 2 over gloo (no GPU).

The forward pass of a data-parallel replica needs no exchange, so ranks only meet to
time the job: every rank reports its own elapsed time and the job takes as long as the
slowest rank; the throughput counts every rank's replica. The reference arm runs on
rank 0 only; the other ranks exit 0 without work.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms, value = bench.aggregate_timing(10.0 + 5.0 * rank, world, model_flops=2 * 10**12,
                                       steps=4, device="cpu")
    dist.barrier()
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_two_ranks_time_the_slowest_and_count_both_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in res:
        assert ms == 15.0  # the slower rank's time on every rank
        # 2 ranks x 2e12 FLOP x 4 steps in 15 ms
        assert value == pytest.approx(2 * 2e12 * 4 / 0.015 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    ms, value = bench.aggregate_timing(8.0, 1, model_flops=10**12, steps=2, device="cpu")
    assert ms == 8.0 and value == pytest.approx(2e12 / 0.008 / 1e12)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from transformer_block_gb300 import WORKLOADS

    monkeypatch.setenv("RANK", "1")

    def boom(*a, **k):
        raise AssertionError("rank 1 must not run the oracle")

    monkeypatch.setattr(bench, "OracleSample", boom)
    args = bench.argparse.Namespace(gpus=2, steps=1, warmup=0)
    assert bench.run_reference(args, WORKLOADS["tiny"]) == 0
    assert capsys.readouterr().out == ""


def test_mfu_denominators():
    # MFU against the nominal dense peak (2.25 PF), the clock-derived peak (SMs x 8192
    # FLOP/clk/SM x the maximum SM clock) and the measured burst
    sys.path.insert(0, ROOT)
    import bench

    peaks = {"bf16_tflops": 1891.2, "bf16_tflops_sustained": 1692.7, "hbm_gbs": 6788.6}
    m = bench.mfu_of(1800.0, peaks, {"sm_max_mhz": 2070.0}, 152)
    assert abs(m["vs_spec_dense_bf16"] - 1800.0 / 2250.0) < 1e-12
    assert abs(m["clock_derived_tflops"] - 152 * 8192 * 2070e6 / 1e12) < 1e-9
    assert abs(m["vs_clock_derived_bf16"] - 1800.0 / m["clock_derived_tflops"]) < 1e-12
    assert abs(m["vs_measured_bf16"] - 1800.0 / 1891.2) < 1e-12
    # no clock record: the documented maximum clock
    assert bench.mfu_of(1.0, peaks, None, 152)["clock_derived_tflops"] == m["clock_derived_tflops"]
