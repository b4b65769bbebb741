"""Host-side bookkeeping of bench.py: the per-kernel DRAM traffic taken from
profiles/traffic.json is reported only while the kernel's sources still hash
to the value the counters were taken with, and the algorithmic byte counts
follow the layouts the kernels move."""
import json
import os

import bench


def _write(tmp_path, kernels):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({"_source": "test", "kernels": kernels}))


def test_traffic_reported_only_for_matching_sources(tmp_path, monkeypatch):
    files = bench.KERNEL_SOURCES["gate_add_kernel"]
    good = bench.sources_hash(files)
    _write(tmp_path, {
        "gate_add_kernel": {"bytes_per_launch": 123, "sources_hash": good},
        "gates_kernel": {"bytes_per_launch": 456, "sources_hash": "0" * 16},   # stale
        "not_a_kernel": {"bytes_per_launch": 789, "sources_hash": good},       # unknown name
    })
    real_hash = bench.sources_hash
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the sources are still read from the repository
    monkeypatch.setattr(bench, "sources_hash", lambda f, read=None: real_hash(
        f, read=lambda n: open(os.path.join(os.path.dirname(os.path.abspath(bench.__file__)),
                                            "hashed_gram_conditional_gb300", "csrc", n), "rb").read()))
    assert bench.profiled_traffic() == {"gate_add_kernel": 123}


def test_no_traffic_file_means_no_figures(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic() == {}


def test_sources_hash_depends_on_every_file_and_its_order():
    data = {"a.cu": b"alpha", "b.h": b"beta"}
    h_ab = bench.sources_hash(["a.cu", "b.h"], read=data.__getitem__)
    assert h_ab == bench.sources_hash(["a.cu", "b.h"], read=data.__getitem__)
    assert h_ab != bench.sources_hash(["b.h", "a.cu"], read=data.__getitem__)
    assert h_ab != bench.sources_hash(["a.cu"], read=data.__getitem__)
    data2 = dict(data, **{"b.h": b"beta!"})
    assert h_ab != bench.sources_hash(["a.cu", "b.h"], read=data2.__getitem__)


def test_every_profiled_kernel_names_existing_sources():
    csrc = os.path.join(os.path.dirname(os.path.abspath(bench.__file__)), "hashed_gram_conditional_gb300", "csrc")
    for name, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (name, f)


def test_algorithmic_bytes_per_token():
    # h read and written (bf16, hc streams), v read once, the partial sums, the mask
    assert bench.GATE_BYTES_PER_TOKEN(4, 5120) == 2 * 4 * 5120 * 2 + 5120 * 2 + 4 * 20 * 16 + 1
    # h read and written, v read once, the gates
    assert bench.CONV_BYTES_PER_TOKEN(4, 5120) == 92_176


def test_clock_sampler_keeps_only_the_timed_region():
    """The clock record counts only nvidia-smi samples taken inside the timed
    region, widening the window in 50 ms steps only while none falls inside."""
    import datetime
    import time

    import bench

    c = bench.ClockSampler("0")
    c.proc = type("Done", (), {"poll": lambda self: 0})()  # no process to stop
    now = time.time()

    def line(dt, mhz, watts, cap):
        stamp = datetime.datetime.fromtimestamp(now + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{stamp}, 0, {mhz}, 2070, {watts}, 0x0, Not Active, Not Active, Not Active, {cap}"

    c.lines = [line(-0.2, 345, 90, "Not Active"), line(0.01, 2070, 900, "Not Active"),
               line(0.03, 1980, 1200, "Active"), line(0.3, 1500, 300, "Not Active")]
    inside = c.stop(now, now + 0.05)
    assert inside["samples"] == 2 and inside["samples_outside_region"] == 2
    assert inside["sm_mhz"] == (2070 + 1980) / 2 and inside["power_w_max"] == 1200
    assert inside["reasons"] == ["sw_power_cap"] and "window_widened_ms" not in inside
    widened = c.stop(now + 0.1, now + 0.12)  # nothing inside: widened until the two samples before it
    assert widened["samples"] == 2 and widened["window_widened_ms"] == 100
