"""CPU checks of bench.py's reporting helpers and launch rule: the DRAM-traffic figure is
read from the profile summary only while its source digest matches the
kernel sources, and the clock sampler's summary reports the median SM clock
and every throttle reason that was active."""
import os

import bench


def test_profiled_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    good = tmp_path / "good.md"
    good.write_text(f"traffic_bytes_per_launch: 1.25e9\nsource_digest: {bench.source_digest()}\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(good))
    assert bench.profiled_traffic() == 1.25e9
    stale = tmp_path / "stale.md"
    stale.write_text("traffic_bytes_per_launch: 1.25e9\nsource_digest: 0000000000000000\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(stale))
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(tmp_path / "missing.md"))
    assert bench.profiled_traffic() is None


def test_committed_profile_has_a_traffic_figure():
    txt = open(bench.PROFILE_SUMMARY).read()
    assert "traffic_bytes_per_launch:" in txt and "source_digest:" in txt


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _summary(tmp_path, rows):
    s = bench.ClockSampler(None)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    s.fh = open(os.devnull, "w")
    s.proc = _Done()
    return s.stop()


def test_clock_summary_median_and_reasons(tmp_path):
    idle = "Not Active"
    rows = [f"0, {mhz}, 2070, 1000.5, 0x0, {idle}, {idle}, {idle}, {cap}"
            for mhz, cap in ((1500, "Active"), (1480, "Active"), (1520, idle))]
    out = _summary(tmp_path, rows + ["garbage line"])
    assert out["sm_mhz"] == 1500 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    hot = [f"0, 1200, 2070, 900.0, 0x0, Active, {idle}, {idle}, {idle}"]
    assert _summary(tmp_path, hot)["reasons"] == ["hw_slowdown"]


def test_clock_summary_without_samples(tmp_path):
    assert _summary(tmp_path, ["no numbers here"]) is None
    s = bench.ClockSampler(None)
    assert s.stop() is None          # never started


def test_multi_gpu_launch_is_refused():
    """The benchmark is single-GPU: --gpus > 1 and WORLD_SIZE > 1 exit with
    code 2 before touching a device (the cluster GEMMs' TMA multicast stays
    in code that one GPU runs alone)."""
    import subprocess
    import sys
    bench_py = os.path.join(os.path.dirname(bench.__file__), "bench.py")
    r = subprocess.run([sys.executable, bench_py, "--gpus", "2"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "one GPU only" in r.stderr
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    r = subprocess.run([sys.executable, bench_py], capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 2 and r.stdout == ""
