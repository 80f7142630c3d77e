"""Host-side logic of bench.py that needs no GPU: the committed-traffic lookup
(bytes only while the listed kernel sources are unchanged), the clock-record
parser that decides whether a run is kept, and the peak lookup."""
import hashlib
import json
import os

import bench


def _write(path, text):
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write(text)


def test_committed_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    root = str(tmp_path)
    _write(os.path.join(root, "src", "a.cu"), "kernel a\n")
    _write(os.path.join(root, "src", "b.cuh"), "header b\n")
    h = hashlib.sha256()
    for rel in ("src/a.cu", "src/b.cuh"):
        h.update(open(os.path.join(root, rel), "rb").read())
    entry = {"kernel": "k", "bytes_per_launch": 1234, "sources": ["src/a.cu", "src/b.cuh"], "sha256": h.hexdigest()}
    _write(os.path.join(root, "profiles", "traffic.json"), json.dumps({"wl": entry}))
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.committed_traffic("wl") == 1234
    assert bench.committed_traffic("other") is None               # no capture for that workload
    _write(os.path.join(root, "src", "b.cuh"), "header b, edited\n")
    assert bench.committed_traffic("wl") is None                  # kernel changed since the capture
    os.remove(os.path.join(root, "src", "a.cu"))
    assert bench.committed_traffic("wl") is None                  # a listed source is gone


def test_traffic_key_separates_mask_form_and_forced_kernel():
    assert bench.traffic_key("wl", False, 0) == "wl"
    keys = {bench.traffic_key("wl", p, k) for p in (False, True) for k in (0, 1, 2)}
    assert len(keys) == 6


def test_committed_traffic_without_a_capture_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("wl") is None


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    assert d, "no committed traffic captures"
    for name, ent in d.items():
        assert ent["bytes_per_launch"] > 0, name
        for rel in ent["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, rel)), (name, rel)


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(tmp_path, lines):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.fh = open(s.path, "a")
    s.proc = _Proc()
    return s


def test_clock_record_parser_median_max_and_reasons(tmp_path):
    row = "0, {sm}, 2070, {p}, 0x0, Not Active, {th}, Not Active, {cap}"
    lines = [row.format(sm=2070, p=400.0, th="Not Active", cap="Not Active"),
             row.format(sm=2070, p=900.5, th="Not Active", cap="Active"),
             row.format(sm=1900, p=700.0, th="Active", cap="Not Active"),
             "garbage line", "0, [N/A], 2070, 1, 0x0, a, b, c, d"]
    r = _sampler_with(tmp_path, lines).stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["samples"] == 3 and r["power_w_max"] == 900.5
    assert r["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert not os.path.exists(tmp_path / "clocks.csv")           # the temporary record is removed


def test_clock_record_parser_without_samples(tmp_path):
    r = _sampler_with(tmp_path, ["nothing useful"]).stop()
    assert r["sm_mhz"] is None and r["reasons"] == ["no samples"]


def test_clock_sampler_without_nvidia_smi_reports_it():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    assert bench.ClockSampler.stop(s)["reasons"] == ["nvidia-smi unavailable"]


def test_peak_lookup(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (6800.0, "fallback")
    _write(os.path.join(str(tmp_path), "MEASURED_PEAKS.json"), json.dumps({"hbm_gbs": 6696.5}))
    assert bench.load_peaks() == (6696.5, "measured")


def test_bench_refuses_more_than_one_gpu():
    """One GPU per process: --gpus 2, or a multi-rank launch, is an error (exit 2),
    not a silently smaller run.  The refusal comes before any device work."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 2 and "one GPU per process" in r.stderr
    env.update(WORLD_SIZE="2", RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py")], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 2 and "one GPU per process" in r.stderr


def test_reference_arm_other_ranks_exit_without_work():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
