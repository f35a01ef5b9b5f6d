"""Host-side logic of bench.py (no GPU): flop counting, clock parsing, the
traffic record, the reference arm's JSON line, and the multi-rank aggregation
(max time over ranks, summed work) on two gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_attention_flops_counts_twelve_d_per_pair():
    spec = dict(B=1, H=40, N=32760, d=128)
    assert bench.attention_flops(spec) == 12.0 * 40 * 32760 ** 2 * 128
    assert bench.attention_flops(spec, kv_len=18900) == 12.0 * 40 * 32760 * 18900 * 128


def test_clock_summary_parses_reasons():
    lines = [
        "0, 1995, 2070, 850.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1200.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2040, 2070, 1300.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    s = bench.ClockSampler.summarize(lines)
    assert s["sm_mhz"] == 2040 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3
    assert bench.ClockSampler.summarize([])["sm_mhz"] is None


def test_clock_rejection_rule():
    def summary(rows):
        return bench.ClockSampler.summarize(
            ["0, %d, 2070, 1000.0, 0x0, Not Active, %s, %s, %s" % r for r in rows])

    ok = lambda sm, pcap="Not Active": (sm, "Not Active", "Not Active", pcap)  # noqa: E731
    # full clocks, or the power cap holding them near 1.8 GHz: kept
    assert bench.ClockSampler.rejection(summary([ok(2040)] * 5)) is None
    assert bench.ClockSampler.rejection(summary([ok(1792, "Active")] * 5)) is None
    # the power cap explains a low clock too
    assert bench.ClockSampler.rejection(summary([ok(1200, "Active")] * 5)) is None
    # a thermal reason at a single sample voids the region
    rows = [ok(2040)] * 4 + [(2040, "Active", "Not Active", "Not Active")]
    assert bench.ClockSampler.rejection(summary(rows)) == "hw_thermal_slowdown"
    rows = [ok(2040)] * 4 + [(1900, "Not Active", "Active", "Active")]
    assert bench.ClockSampler.rejection(summary(rows)) == "sw_thermal_slowdown"
    # a low median clock with no reason: a clock lock left behind
    why = bench.ClockSampler.rejection(summary([ok(1200)] * 5))
    assert why is not None and "no reason" in why
    # one idle sample does not move the median
    assert bench.ClockSampler.rejection(summary([ok(345)] + [ok(2040)] * 4)) is None
    # no nvidia-smi samples: nothing to reject
    assert bench.ClockSampler.rejection(bench.ClockSampler.summarize([])) is None


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    monkeypatch.setattr(bench, "KERNEL_SOURCES", (str(src),))
    src.write_text("// kernel\nint f(int a) { return a - -1; }  /* note */\n")
    base = bench.kernel_source_sha()
    src.write_text("// kernel, reworded\n// and one more line\n\nint f(int a)  {\n  return a - -1; }\n")
    assert bench.kernel_source_sha() == base
    src.write_text("// kernel\nint f(int a) { return a - 1; }\n")
    assert bench.kernel_source_sha() != base
    src.write_text("// kernel\nint f(int a) { return a--1; }\n")
    assert bench.kernel_source_sha() != base


def test_oracle_sample_calibration_discounts_start_up(monkeypatch):
    # The CPU baseline's sample is sized to a target time from a timed calibration.  With
    # a fixed start-up cost per call, one row per thread would overstate the cost of a
    # row several times over; the second, larger calibration must not.
    import oracle
    clock = [0.0]

    def fake_oracle(q, k, v, qt, kt, vt, scale, rows=None, nthreads=None):
        clock[0] += 0.05 + 1e-3 * len(rows)  # start-up + 1 ms a row

    monkeypatch.setattr(oracle, "attn_jvp", fake_oracle)
    monkeypatch.setattr(bench.time, "perf_counter", lambda: clock[0])
    n = bench.oracle_rows_for(dict(N=100000, scale=0.1), (None,) * 6, 12.0)
    assert 9000 <= n <= 12000
    assert bench.oracle_rows_for(dict(N=500, scale=0.1), (None,) * 6, 12.0) == 500  # capped at N


def test_traffic_record_tracks_kernel_source(tmp_path, monkeypatch):
    rec = {"k": {"w": {"source_sha": bench.kernel_source_sha(), "heads": 4, "dram_bytes_per_launch": 400.0}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.traffic_per_launch("k", "w", 40) == 4000.0
    rec["k"]["w"]["source_sha"] = "stale"
    path.write_text(json.dumps(rec))
    assert bench.traffic_per_launch("k", "w", 40) is None
    assert bench.traffic_per_launch("other", "w", 40) is None


def test_committed_traffic_record_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        table = json.load(f)
    for kernel, per_workload in table.items():
        for workload, rec in per_workload.items():
            assert rec["dram_bytes_per_launch"] > 0 and rec["heads"] >= 1
            assert len(rec["source_sha"]) == 16


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)

    def rmax(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def rsum(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        return float(t.item())

    dist.barrier()
    t, u = bench.aggregate(local_ms[rank], 1.0e12, world, rmax, rsum)
    q.put((rank, t, u))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    local_ms = [41.0, 57.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u in res:
        assert t == 57.5          # the slowest rank's time
        assert u == 2.0e12        # work of both replicas


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(12.5, 3.0, 1) == (12.5, 3.0)


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
    assert rec["metric"] == bench.METRIC


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_merge_and_tangent_algorithmic_bytes():
    spec = dict(B=1, H=40, N=75600, d=128)
    # four chunks of (O_c, Ot_c, LSE_c, mu_c) read, one merged set written
    rows = 40 * 75600
    assert bench.merge_bytes(spec, 4) == rows * (2 * 128 + 2) * 4 * 5
    assert bench.tangent_bytes(1000) == 12000


def test_clock_normalised_fraction():
    # 152 SMs x 8192 flop/clk at 2000 MHz is 2490.4 TFLOP/s
    full = 152 * 8192 * 2000e6 / 1e12
    assert abs(bench.clock_normalised_frac(full / 2, 152, 2000.0) - 0.5) < 1e-12
    assert bench.clock_normalised_frac(1000.0, 152, None) is None


def test_default_workload_is_the_largest_single_gpu_config():
    from attention_jvp_gb300 import inputs
    args = bench.parse_args([])
    assert args.workload == "long_video" and args.steps >= 1 and args.warmup >= 3
    big = max((w for w in ("image_dit_1k", "video_dit", "long_video", "stress")),
              key=lambda w: bench.attention_flops(inputs.WORKLOADS[w]))
    assert big == args.workload
    assert set(args.also.split(",")) == {"video_dit", "stress", "image_dit_1k"}


def test_backward_executed_flops_count():
    assert bench.backward_executed_flops_per_pair(128) == 14 * 128
    # two CTAs per row tile at 256: S and dP formed twice in each pass
    assert bench.backward_executed_flops_per_pair(256) == (2 * 8 + 4 + 2) * 256


def test_parity_on_rows_metrics():
    import numpy as np
    r = [np.ones((3, 4)), np.full((3, 4), 2.0), np.zeros(3), np.ones(3)]
    g = [r[0] * 1.01, r[1], r[2] + 1e-4, r[3]]
    p = bench.parity_on_rows(g, r)
    assert abs(p["O"]["rel_l2"] - 0.01) < 1e-12 and abs(p["O"]["max_abs_over_rms"] - 0.01) < 1e-12
    assert p["Ot"]["rel_l2"] == 0.0 and abs(p["LSE"]["max_abs"] - 1e-4) < 1e-12
