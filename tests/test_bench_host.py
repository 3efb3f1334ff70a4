"""Host logic of bench.py: multi-rank aggregation over gloo (world size 2,
CPU) and the clock-record summary.  No GPU is used."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took (r + 1) seconds for 10 steps of 1e12 flops each
    value, tmax = bench.aggregate(float(rank + 1), 1e12, 10, world, True, torch.device("cpu"))
    out[rank] = (value, tmax)
    dist.destroy_process_group()


def test_aggregate_takes_max_time_over_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        value, tmax = res[r]
        assert tmax == 2.0
        assert value == pytest.approx(1e12 * 10 * world / 2.0 / 1e12)


def test_aggregate_single_rank():
    value, tmax = bench.aggregate(0.5, 2e12, 4, 1, False)
    assert tmax == 0.5 and value == pytest.approx(16.0)


def test_clock_summary_reasons_and_window():
    cs = bench.ClockSampler("0")
    row = lambda sm, thr: ["0", str(sm), "2070", "900.0", "0x0", "Not Active",
                           "Not Active", thr, "Active"]
    cs.samples = [(0.0, row(1000, "Not Active")), (1.0, row(1900, "Not Active")),
                  (1.1, row(1950, "Not Active")), (5.0, row(500, "Active"))]
    s = cs.summary(0.95, 1.2)
    assert s["samples"] == 2 and s["sm_mhz"] == 1925 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    s = cs.summary(4.9, 5.1)
    assert "sw_thermal_slowdown" in s["reasons"]


def test_peaks_fallback_or_measured():
    peak, src, sustained = bench.read_peaks()
    assert peak > 100 and ("fallback" in src or "measured" in src)
    assert sustained is None or 100 < sustained <= peak


def test_backward_pass_flag_and_cpu_baseline():
    import torch
    from exact_headdim_attention_gb300 import workloads as wl
    assert bench.parse_args([]).which == "fwd"
    assert bench.parse_args(["--pass", "bwd"]).which == "bwd"
    w = wl.tiny_d320()
    x = wl.materialize(w)
    dout = torch.randn(x["q"].shape, generator=torch.Generator().manual_seed(3)).to(x["q"].dtype)
    cb = bench.cpu_baseline_bwd(w, x, dout, 0.05)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["rows"] >= cb["cores"]


def test_cpu_model_and_one_core_tiny_timing():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
    assert bench.oracle_tiny_one_core() > 0


def test_kernel_source_hash_ignores_comments_not_code():
    a = "int f(int x) {\n  return x + 1;  // one\n}\n/* block\n comment */\n"
    b = "int f(int x) {   return x + 1; }"
    c = "int f(int x) { return x + 2; }"
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(tmp_path):
    sha = {k: bench.kernel_source_sha(v) for k, v in bench.TRAFFIC_SOURCES.items()}
    rec = {"dram_bytes_per_launch": {"kernel_source_sha": sha["dram_bytes_per_launch"], "w": 123},
           "fp8_dram_bytes_per_launch": {"kernel_source_sha": sha["fp8_dram_bytes_per_launch"], "w": 45},
           "bwd_dram_bytes_per_step": {"kernel_source_sha": sha["bwd_dram_bytes_per_step"],
                                       "w": {"scores": 1, "contract": 5, "gradient_kernels_total": 6}}}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    assert bench.measured_traffic("w", path=str(p)) == 123
    assert bench.measured_traffic("w", path=str(p), key="fp8_dram_bytes_per_launch") == 45
    assert bench.measured_traffic_bwd("w", path=str(p))["gradient_kernels_total"] == 6
    # a record taken on other code is not used; the sections are independent
    rec["dram_bytes_per_launch"]["kernel_source_sha"] = "0" * 16
    rec["bwd_dram_bytes_per_step"]["kernel_source_sha"] = "0" * 16
    p.write_text(json.dumps(rec))
    assert bench.measured_traffic("w", path=str(p)) is None
    assert bench.measured_traffic_bwd("w", path=str(p)) is None
    assert bench.measured_traffic("w", path=str(p), key="fp8_dram_bytes_per_launch") == 45
    # each section hashes its own kernel's files
    assert sha["dram_bytes_per_launch"] != sha["fp8_dram_bytes_per_launch"]


def test_committed_traffic_record_is_consistent():
    with open(bench.TRAFFIC_PATH) as f:
        d = json.load(f)
    for name, tb in d.get("bwd_dram_bytes_per_step", {}).items():
        if name == "kernel_source_sha":
            continue
        assert tb["gradient_kernels_total"] == tb["scores"] + tb["contract"], name
