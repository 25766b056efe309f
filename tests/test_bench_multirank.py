"""bench.py's multi-rank logic on the host: world-size-2 gloo process groups
(one process per rank, as torchrun launches them) check the max-over-ranks
time and the whole-job rate of independent replicas, and that the reference
arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as tmp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 + 5.0 * rank                  # rank 1 is the slow one
        mx = bench.max_over_ranks(ms_local)
        rate, ms = bench.aggregate_rate(1e9, ms_local, world)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{mx} {rate} {ms}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo(tmp_path):
    world = 2
    tmp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"r{r}.txt").read().split() for r in range(world)]
    for mx, rate, ms in rows:
        assert float(mx) == 15.0 and float(ms) == 15.0
        # 2 replicas x 1e9 units in the slowest rank's 15 ms
        assert float(rate) == pytest.approx(2e9 / 15e-3)


def test_max_over_ranks_without_group():
    assert bench.max_over_ranks(3.5) == 3.5
    rate, ms = bench.aggregate_rate(100.0, 2.0, 1)
    assert ms == 2.0 and rate == pytest.approx(5e4)


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, gpus = 1, 3, 2
    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_its_line_on_a_small_workload(monkeypatch, capsys):
    """Rank 0 of the reference arm times the oracle on the selected workload
    and prints one JSON line with the contract's keys."""
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class Args:
        steps, warmup, gpus, workload = 2, 1, 1, "tiny_n256"
    bench.run_reference(Args())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"]["workload"] == "tiny_n256"
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_bench_traffic_table_is_keyed_by_kernel_and_workload():
    """profiles/traffic.json rows are found by (kernel, workload); a workload
    without a row gives None."""
    assert bench.measured_traffic("prefill_kernel", "no_such_workload") is None
    assert bench.prefill_algo_bytes(bench.mi.PREFILL["llama8b_n16k_causal"]) == 200867840


def test_pv_fp4_option_needs_prefill_only():
    """--pv fp4 times the ablation kernel alone: without --only prefill the
    argument check rejects it before any GPU work."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--pv", "fp4"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 2
    assert "--only prefill" in r.stderr


def test_fp4_roofline_is_all_fp4():
    """The ablation's roofline puts both products at the FP4 rate: 6 x the
    bf16 peak, against 3 x for the method's FP4 QK + FP8 PV mix."""
    import mpfa_inputs as mi
    cfg = mi.PREFILL["llama8b_n16k_causal"]
    peaks = {"bf16": 1000.0, "source": "test"}
    r8 = bench.prefill_roofline(cfg, 1.0, peaks)
    r4 = bench.prefill_roofline(cfg, 1.0, peaks, pv4=True)
    assert abs(r8["peak"] - 3000.0) < 1e-6 and abs(r4["peak"] - 6000.0) < 1e-6
    assert r4["traffic"] is None and r4["kernel"].startswith("prefill_kernel<true>")
