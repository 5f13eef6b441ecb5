"""bench.py host logic without a GPU: clock-sample parsing, the traffic
record lookup, the cross-rank timing reduction (gloo, world size 2), and the
reference arm (the fp64 oracle on the host cores) end to end."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_clock_sampler_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 1900, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1300.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1800, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage",
    ]
    s = c.summary()
    assert s["sm_mhz"] == 1900 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_samples():
    c = bench.ClockSampler(0)
    c.lines = []
    assert c.summary()["sm_mhz"] is None


def test_recorded_traffic_matches_source_hash(tmp_path, monkeypatch):
    f = tmp_path / "dram_traffic.txt"
    h = bench.kernel_source_hash()
    f.write_text(f"# workload source_hash bytes\nn1024_d64 {h} 104396544\n"
                 f"n4096_d128 deadbeef0000 1\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("n1024_d64") == 104396544.0
    assert bench.recorded_traffic("n4096_d128") is None  # taken on another source


def test_job_throughput_counts_all_ranks():
    assert bench.job_throughput(1, 1e12, 10, 10.0) == pytest.approx(1.0)
    assert bench.job_throughput(4, 1e12, 10, 10.0) == pytest.approx(4.0)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = bench.reduce_max([1.0 + rank, 10.0 - rank], world)
    with open(out + f".{rank}", "w") as f:
        json.dump(vals, f)
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks(tmp_path):
    import socket

    import torch.multiprocessing as mp
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    out = str(tmp_path / "vals")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, start_method="spawn")
    for r in range(2):
        with open(out + f".{r}") as f:
            assert json.load(f) == [2.0, 10.0]


def test_reduce_max_single_rank_is_identity():
    assert bench.reduce_max([3.0, 4.0], 1) == [3.0, 4.0]


def test_reference_arm_prints_one_json_line():
    # The reference arm runs the fp64 oracle on the host: no GPU needed.
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "n256_d64", "--steps", "1", "--warmup", "3"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "n256_d64"


def test_bench_rejects_too_few_warmups():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert res.returncode != 0


def test_flop_counts_of_the_other_workloads():
    from attention_forward_tk_gb300.inputs import (BASED_BY_NAME, BWD_WORKLOADS, BY_NAME,
                                                   GEMM_BY_NAME)
    w = BY_NAME["n4096_d128"]
    assert bench.bwd_flops(w) == 2.5 * 4 * 16 * 16 * 4096 ** 2 * 128
    assert [x.name for x in BWD_WORKLOADS] == ["n4096_d128", "n8192_d128_c"]
    b = BASED_BY_NAME["based_n4096_c"]
    assert b.flops == 16 * 16 * (4096 ** 2 / 2) * 2 * (16 + 64)
    g = GEMM_BY_NAME["gemm_8192"]
    assert g.flops == 2 * 8192 ** 3
    assert g.io_bytes == 3 * 8192 * 8192 * 2


def test_input_generators_are_seeded():
    import torch
    from attention_forward_tk_gb300.inputs import draw_based, draw_gemm, draw_grad
    a1, b1 = draw_gemm(16, 24, 32, 3)
    a2, b2 = draw_gemm(16, 24, 32, 3)
    assert torch.equal(a1, a2) and torch.equal(b1, b2) and not torch.equal(a1[:, :24], b1[:16])
    q1, k1, v1 = draw_based(1, 2, 40, 5)
    q2, k2, v2 = draw_based(1, 2, 40, 5)
    assert torch.equal(q1, q2) and torch.equal(v1, v2) and q1.shape[-1] == 16 and v1.shape[-1] == 64
    g1 = draw_grad((1, 1, 8, 64), 2)
    assert torch.equal(g1, draw_grad((1, 1, 8, 64), 2))
    assert not torch.equal(g1, draw_grad((1, 1, 8, 64), 3))
