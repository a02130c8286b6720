"""Host-side logic of bench.py without a GPU: the max-over-ranks timing and
whole-job aggregation over a real 2-rank gloo process group, the reference
arm's JSON line, and rank gating under a multi-rank launch."""

import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, use_cuda=False)
    # rank r "took" 1 + r seconds; the job time is the slowest rank's
    t = bench.reduce_max(dist, 1.0 + rank)
    v = bench.aggregate(2.0e12, world, t)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, v in res:
        assert t == 2.0                       # max over ranks
        assert abs(v - 2.0) < 1e-12           # 2 ranks x 2e12 flops / 2 s = 2 TFLOP/s


def test_reference_arm_prints_one_json_line(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3",
                         "--workload", "tiny_T64_d16_f32_causal"])
    assert rc == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_T64_d16_f32_causal"


def test_reference_arm_other_ranks_do_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--gpus", "2", "--impl", "reference", "--steps", "3", "--warmup", "3",
                         "--workload", "tiny_T64_d16_f32_causal"])
    assert rc == 0 and buf.getvalue().strip() == ""


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_clock_summary_flags_throttling():
    s = bench.ClockSampler(0)
    s.rows = [(10.0, ["t", "1900", "2070", "900", "0x4", "Not Active", "Not Active",
                      "Not Active", "Active"]),
              (10.2, ["t", "1800", "2070", "950", "0x4", "Active", "Not Active",
                      "Not Active", "Active"])]
    out = s.summary(10.0, 10.2)
    assert out["sm_mhz"] == 1850 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_alu_and_exp_peaks_from_measured_rates():
    # SMs x rate per clock per SM x the maximum clock; the rates come from the
    # committed record of `bench.py --measure-pipe-rates`, else the unit
    # counts (128 FP32 lanes, 32 ex2 per clock per SM)
    rates = bench.measured_pipe_rates()
    ffma = max(rates.get("ffma_per_clock_per_sm", 0.0),
               rates.get("ffma2_fma_per_clock_per_sm", 0.0)) or 128.0
    ex2 = rates.get("ex2_per_clock_per_sm", 32.0)
    p = bench.alu_peaks({"sm_max_mhz": 2070.0}, 152)
    assert abs(p["fp32_tflops"] - 152 * ffma * 2 * 2.07e9 / 1e12) < 1e-9
    assert abs(p["exp_per_s"] - 152 * ex2 * 2.07e9) < 1.0
    assert p["source"] == ("measured" if rates else "assumed")
    # without a measured clock the maximum GB300 clock stands in
    assert bench.alu_peaks({}, 152) == p


def test_pipe_rate_record_parses(tmp_path, monkeypatch):
    f = tmp_path / "rates.md"
    f.write_text("# rates\n\n- ex2_per_clock_per_sm = 31.9 (median)\n"
                 "- ffma_per_clock_per_sm = 127.5\nnot a value = x\n")
    monkeypatch.setattr(bench, "PIPE_RATES_FILE", str(f))
    r = bench.measured_pipe_rates()
    assert r == {"ex2_per_clock_per_sm": 31.9, "ffma_per_clock_per_sm": 127.5}
    p = bench.alu_peaks({"sm_max_mhz": 2000.0}, 100)
    assert abs(p["exp_per_s"] - 100 * 31.9 * 2e9) < 1.0
    assert abs(p["fp32_tflops"] - 100 * 127.5 * 2 * 2e9 / 1e12) < 1e-9
