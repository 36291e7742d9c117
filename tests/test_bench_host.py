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
