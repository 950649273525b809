"""CPU tests of bench.py's host logic: the N > 1 replica path over a real
world-size-2 process group (gloo on CPU, rendezvous on 127.0.0.1), the
reference arm's rank handling, and the roofline / traffic bookkeeping."""
import os
import socket
import json
import types

import pytest
import torch.multiprocessing as mp

import bench
from dense_gemm_13_gb300.inputs import WORKLOADS


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank))
    r, ws, local, dist = bench.dist_setup(2)
    try:
        # per-step times differ per rank; the bench keeps the slowest rank per step
        times = [1.0 + rank, 5.0 - rank, 2.5]
        got = bench.max_over_ranks(times, dist, "cpu")
        bench.barrier(dist)
        out.put((r, ws, local, got))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, ws, lr) for r, ws, lr, _ in res] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, got in res:
        assert got == [2.0, 5.0, 2.5]


def test_single_process_path_has_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.dist_setup(1) == (0, 1, 0, None)
    assert bench.max_over_ranks([3.0, 1.0], None, "cpu") == [3.0, 1.0]
    bench.barrier(None)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = types.SimpleNamespace(workload="sgemm_4096", steps=1, warmup=1, gpus=2)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""


def test_roofline_bounds_and_peaks():
    pk = {"hbm_gbs": 6790.7, "bf16_tflops": 1912.4, "sm_max_mhz": 2070.0}
    r = bench.roofline_for(WORKLOADS["sgemm_4096"], "ffma", 2.5, pk, "measured")
    assert r["bound"] == "alu" and abs(r["peak"] - 152 * 128 * 2 * 2.07e9 / 1e12) < 0.01
    assert abs(r["achieved"] - 2 * 4096 ** 3 / 2.5e-3 / 1e12) < 1e-6
    assert bench.roofline_for(WORKLOADS["bf16_8192"], "tc", 0.6, pk, "measured")["bound"] == "tensor"
    q = bench.roofline_for(WORKLOADS["qkt_bf16"], "tc", 0.03, pk, "measured")
    assert q["bound"] == "hbm" and q["unit"] == "GB/s"
    assert abs(q["achieved"] - WORKLOADS["qkt_bf16"].algorithmic_bytes() / 0.03e-3 / 1e9) < 1e-6
    t = bench.roofline_for(WORKLOADS["sgemm_4096"], "tf32x3", 0.5, pk, "measured")
    assert t["bound"] == "tensor" and abs(t["achieved"] - 3 * 2 * 4096 ** 3 / 0.5e-3 / 1e12) < 1e-6


def test_recorded_traffic_follows_the_source_hash(tmp_path):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({
        "ffma/sgemm_4096": {"dram_bytes_per_launch": 1234, "source_hash": bench.source_hash("ffma")},
        "tc/bf16_8192": {"dram_bytes_per_launch": 99, "source_hash": "0000"}}))
    root = str(tmp_path)
    assert bench.recorded_traffic("ffma", "sgemm_4096", root) == 1234.0
    assert bench.recorded_traffic("tc", "bf16_8192", root) is None          # stale hash
    assert bench.recorded_traffic("ffma", "no_such_workload", root) is None


def test_fp32_peak_follows_the_plan_sm_count():
    pk = {"hbm_gbs": 6790.7, "bf16_tflops": 1912.4, "sm_max_mhz": 2070.0}
    r = bench.roofline_for(WORKLOADS["sgemm_4096"], "ffma", 2.5, pk, "measured", num_sms=148)
    assert abs(r["peak"] - 148 * 128 * 2 * 2.07e9 / 1e12) < 0.01 and "148 SMs" in r["peak_source"]


def test_workload_names_include_sweep_triples():
    w = bench.workload_by_name("sweep:3001,17,4097")
    assert (w.M, w.N, w.K, w.dtype, w.residual, w.alpha) == (3001, 17, 4097, "bf16", True, 0.5)
    assert bench.workload_by_name("ffn2_bf16") is WORKLOADS["ffn2_bf16"]
    with pytest.raises(KeyError):
        bench.workload_by_name("no_such_workload")
