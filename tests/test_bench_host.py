"""Host-side logic of bench.py, without a GPU: the ncu traffic ratio is used only
while the attention source matches the capture, and clock samples are kept only
inside the timed window (with throttle reasons reported)."""
import hashlib
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_ratio_follows_the_attention_source(tmp_path, monkeypatch):
    src = tmp_path / "tiered_kv_cache_gqa_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "attention.cu").write_bytes(b"kernel v1")
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = hashlib.sha256(b"kernel v1").hexdigest()
    (prof / "a.md").write_text("text\n`traffic_ratio: 7b 1.015 %s`\n" % digest)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic_ratio("7b") == 1.015
    assert bench.ncu_traffic_ratio("14b") is None
    (src / "attention.cu").write_bytes(b"kernel v2")            # changed since the capture
    assert bench.ncu_traffic_ratio("7b") is None


def test_clock_samples_are_filtered_to_the_timed_window(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    cs = bench.ClockSampler(0)
    os.makedirs(os.path.dirname(cs.path), exist_ok=True)
    t0 = time.time()

    def row(t, mhz, thermal="Not Active"):
        stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".%03d" % int((t % 1) * 1000)
        return "%s, 0, %d, 2070, 900.00, 0x0, Not Active, Not Active, %s, Not Active\n" % (stamp, mhz, thermal)

    with open(cs.path, "w") as f:
        f.write(row(t0 - 5, 1000, "Active"))            # before the window: ignored
        f.write(row(t0 + 0.1, 2070))
        f.write(row(t0 + 0.3, 2050, "Active"))          # inside: a throttle reason to report
        f.write(row(t0 + 9, 800))                        # after the window: ignored

    class Done:
        def terminate(self):
            pass

        def wait(self):
            pass

    cs.proc, cs.f = Done(), open(os.devnull, "w")
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    out = cs.stop(t0, t0 + 1.0)
    assert out["samples"] == 2
    assert out["sm_mhz"] == 2060.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_thermal_slowdown"]


def test_reference_arm_runs_on_cpu_and_prints_its_line():
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True


def test_timed_window_holds_a_retier_and_the_delta_step():
    """The timed steps contain a re-tier step (t % 64 == 0) and the delta-prefetch step after it,
    the profiled pass starts right after the second re-tier, and the last timed step ends the
    configuration's sequence."""
    for steps, warmup in ((20, 5), (2, 1), (64, 3), (512, 3)):
        tl = bench.timeline(steps, warmup)
        timed = range(tl["timed0"], tl["last"] + 1)
        assert len(timed) == steps and tl["timed0"] - tl["warm0"] == warmup
        assert tl["prof0"] == bench.PRE_STEPS + 1 and tl["fill0"] == tl["prof0"] + tl["kp"]
        assert tl["warm0"] >= tl["fill0"]
        r = [t for t in timed if t % 64 == 0]
        assert r and r[0] + 1 in timed and tl["retiers_timed"] == r
    for name in ("7b", "14b", "32b", "70b"):
        wl = bench.bench_workload(name, 5, 20)
        assert wl.prefill_len + wl.decode_steps == bench.TARGET_N[name]


def test_both_arms_describe_the_same_config():
    args = bench.parse(["--workload", "70b", "--steps", "20", "--warmup", "5"])
    wl = bench.bench_workload(args.workload, args.warmup, args.steps)
    ref = bench.parse(["--impl", "reference", "--workload", "70b", "--steps", "20", "--warmup", "5"])
    assert bench.run_config(args, wl) == bench.run_config(ref, bench.bench_workload("70b", 5, 20))
    assert bench.run_config(args, wl)["retier_steps_timed"] == [192]


def test_host_link_floor_of_a_step():
    """The link-bound step time: a step's T1 bytes at the measured copy-engine peak."""
    import bench
    assert abs(bench.link_bound_step_ms(211.5e9 * 0.138, {"h2d_ce_gbs": 211.5}) - 138.0) < 1e-9
    assert bench.link_bound_step_ms(0.0, {"h2d_ce_gbs": 211.5}) is None
    assert bench.link_bound_step_ms(1e9, None) is None
    assert bench.link_bound_step_ms(1e9, {"h2d_ce_gbs": 0.0}) is None
