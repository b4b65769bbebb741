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
