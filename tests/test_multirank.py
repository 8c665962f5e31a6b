"""bench.py's N > 1 path on the host: two gloo ranks, no GPU.

Each rank runs its own replica of the workload (independent (batch row, head)
units, no collective on the data path). The job's time is the slowest rank's,
taken with an all-reduce MAX, and its throughput counts every rank's units.
"""
import importlib.util
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    bench = _bench()
    w, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    ms = [3.0, 5.0, 4.0][r]  # this rank's time per step
    slowest = bench.max_over_ranks(ms, w)
    value = bench.job_throughput(w, 1000, slowest)
    dist.barrier()
    dist.destroy_process_group()
    with open(f"{out}.{r}", "w") as f:
        f.write(f"{w} {r} {local} {slowest!r} {value!r}")


def test_two_gloo_ranks_report_the_slowest_rank(tmp_path):
    world = 2
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path / "rank")), nprocs=world, join=True)
    for rank in range(world):
        w, r, local, slowest, value = open(tmp_path / f"rank.{rank}").read().split()
        assert (int(w), int(r), int(local)) == (world, rank, rank)
        assert float(slowest) == 5.0
        assert float(value) == world * 1000 / 5e-3


def test_one_rank_needs_no_process_group():
    bench = _bench()
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_throughput(1, 4194304, 0.893) == 4194304 / 0.893e-3


def test_roofline_bytes_and_profile_lookup():
    """The byte counts behind bench.py's roofline fractions, for the long-context plan the
    library picks on a 148-SM B300 (27 segments of 4864 tokens), and the ncu traffic lookup."""
    import synth
    bench = _bench()
    w = synth.WORKLOADS["linear_long"].with_(b=16)
    assert bench.algorithmic_bytes(w) == 32 * 131072 * 512 + 32 * 64 * 64 * 4 * 2
    affine, combine, readout = bench.kernel_bytes(w, {"seg_count": 27, "seg_len": 4864})
    assert affine == 32 * 26 * 4864 * 256 + 32 * 26 * 2 * 64 * 64 * 4
    assert combine == 32 * 26 * 3 * 64 * 64 * 4 + 32 * 64 * 64 * 4
    assert readout == bench.algorithmic_bytes(w) + 32 * 26 * 64 * 64 * 4
    key = "linear_long B1 H32 T131072 b16"
    for kernel in ("linear_mma_kernel", "linear_seg_affine_wy_kernel"):
        traffic = bench.profiled_traffic(kernel, key)  # None once the kernel's source has changed
        alg = readout if kernel == "linear_mma_kernel" else affine
        assert traffic is None or 0.95 * alg < traffic < 1.02 * alg, (kernel, traffic, alg)
        assert bench.profiled_traffic(kernel, "linear_long B1 H32 T65536 b16") is None


def test_roofline_block_reproduces_a_measured_line():
    """bench.py's roofline block from one B300 run's per-kernel event times (long-context workload,
    b16): the same numbers that run printed, plus the fractions of the nominal 7.7 TB/s."""
    bench = _bench()
    names = ("linear_seg_affine_wy_kernel", "linear_seg_combine_kernel", "linear_mma_kernel")
    r = bench.roofline_summary(names, [0.3671, 0.0376, 0.4853], [1063256064, 41418752, 2162163712], 0.8929,
                               2148532224, 6514.2, "measured", lambda name: None)
    assert r["kernel"] == "linear_mma_kernel" and r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert (r["achieved"], r["frac"], r["peak"]) == (4455.3, 0.6839, 6514.2)
    assert r["kernels"]["linear_seg_affine_wy_kernel"]["frac"] == 0.4446
    assert r["kernels"]["linear_seg_combine_kernel"]["share"] == 0.0421
    assert r["step"]["frac"] == 0.3694
    assert r["frac_of_nominal"] == round(4455.3 / 7700.0, 4) and r["step"]["frac_of_nominal"] == 0.3125
    one_pass = bench.roofline_summary(names, [0.0, 0.0, 3.77], [0, 0, 2162163712], 3.77, 2148532224, 6514.2,
                                      "fallback", lambda name: 7)
    assert list(one_pass["kernels"]) == ["linear_mma_kernel"] and one_pass["traffic"] == 7
    assert one_pass["peak_kind"] == "fallback 6.4 TB/s"


def test_reference_arm_prints_on_rank_zero_only(capsys):
    """bench.py --impl reference: the oracle on a bounded sample of the workload, one JSON line from
    rank 0 with the reference keys (impl, cpu_baseline, e2e with no copies); other ranks print nothing."""
    import argparse
    import json
    bench = _bench()
    bench.REFERENCE_BUDGET_S = 0.5
    args = argparse.Namespace(workload="linear_long", b=16, steps=2, warmup=3)
    bench.bench_reference(args, 2, 1)
    assert capsys.readouterr().out == ""
    bench.bench_reference(args, 2, 0)
    line = json.loads(capsys.readouterr().out)
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0 and line["dtype"] == "f64"
    assert line["unit"] == bench.UNIT and line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "linear_long" and line["warmup"] >= 3
