"""Host-side pieces of bench.py: the timing statistics and the bounded oracle
sample (no GPU)."""
import math

import bench


def test_window_stats_mean_cv_and_interval():
    w = [0.010, 0.011, 0.0105, 0.0102, 0.0099, 0.0101, 0.0100]  # seconds per 10-step window
    st = bench.window_stats(w, 10, 70)
    ms = [x / 10 * 1e3 for x in w]
    m = sum(ms) / len(ms)
    sd = math.sqrt(sum((x - m) ** 2 for x in ms) / (len(ms) - 1))
    assert st["windows"] == 7 and abs(st["ms_per_step_mean"] - m) < 1e-12
    assert abs(st["cv"] - sd / m) < 1e-12
    lo, hi = st["ci95_ms_per_step"]
    assert abs((hi - lo) / 2 - 2.447 * sd / math.sqrt(7)) < 1e-12  # Student t, 6 degrees of freedom
    assert st["cv_over_5pct"] is False


def test_window_stats_drop_a_partial_last_window():
    st = bench.window_stats([0.01, 0.01, 0.005], 10, 25)  # the third window held 5 steps
    assert st["windows"] == 2


def test_oracle_sample_is_bounded_and_counts_its_tokens():
    from synth import workloads
    shape = workloads.WORKLOADS["tiny"].shape
    tps, cores, n, dt = bench.oracle_decode_sample(shape, 16, budget_s=0.0, max_tokens=3, warm=False)
    assert n == 3 and cores >= 1 and tps > 0 and abs(tps - n / dt) < 1e-6 * tps
    tps, cores, n, dt = bench.oracle_decode_sample(shape, 16, budget_s=0.0, max_tokens=5)
    assert n == 1  # the warm token sizes the sample to the budget: at least one token


def test_reference_arm_prints_one_contract_line(capsys):
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys."""
    import json
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_traffic_lines_come_only_from_current_captures():
    """The roofline's DRAM traffic is read from profiles/traffic.txt: comment
    lines are skipped, the captures of the dense and MoE GEMVs and of the
    batched 4-bit GEMV are found, an unknown workload has none (the bench
    reports null)."""
    import bench
    assert bench.load_traffic("gemv_swiglu", "dense4b") == 94498560
    assert bench.load_traffic("gemv_in", "moe35b") == 25360128
    assert bench.load_traffic("moe_gateup", "moe35b") == 37838592
    assert bench.load_traffic("gemv_batch", "moe35b-q4-b8") == 68662272
    assert bench.load_traffic("gemv_swiglu", "no-such-workload") is None


def test_other_workloads_trim_lines_and_report_failures(monkeypatch):
    """The default run's `other_workloads`: one child run per workload with the
    parent's steps and warm-up and no CPU baseline; each child's last JSON
    line trimmed to the measurement keys; a failing child gives an error
    entry instead of breaking the line."""
    import json
    import subprocess
    calls = []

    class Done:
        def __init__(self, rc, out, err=""):
            self.returncode, self.stdout, self.stderr = rc, out, err

    def fake_run(cmd, **kw):
        calls.append(cmd)
        wl = cmd[cmd.index("--workload") + 1]
        if wl == "moe35b":
            return Done(1, "", "Traceback\nRuntimeError: no GPU")
        line = {"metric": "m", "value": 1.5, "unit": "tokens/s", "steps": 7, "warmup": 3, "cpu_baseline": None,
                "config": {"workload": wl}, "clocks": {"sm_mhz": 1.0}, "depth_curve": [1, 2]}
        return Done(0, "build log\n" + json.dumps(line) + "\n")

    monkeypatch.setattr(subprocess, "run", fake_run)
    args = bench.parse_args(["--steps", "7", "--warmup", "3"])
    out = bench.other_workloads(args)
    assert list(out) == list(bench.OTHER_WORKLOADS)
    for cmd in calls:
        assert cmd[cmd.index("--steps") + 1] == "7" and cmd[cmd.index("--warmup") + 1] == "3"
        assert "--no-cpu-baseline" in cmd and "--no-other-workloads" in cmd
    ok = out["dense4b-32k"]
    assert ok["value"] == 1.5 and ok["config"]["workload"] == "dense4b-32k" and ok["clocks"] == {"sm_mhz": 1.0}
    assert "depth_curve" not in ok and "cpu_baseline" not in ok and "metric" not in ok
    assert "error" in out["moe35b"] and "no GPU" in out["moe35b"]["error"]
