"""Host logic of bench.py that decides what a bench line reports.

The DRAM traffic of a workload comes from a committed ncu summary only while
the kernel's sources hash as they did when it was captured, scaled by the
units a launch processes; anything else reports null.
"""
import json

import bench


def _write(tmp_path, entries):
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps({"workloads": entries}))
    return str(p)


def test_traffic_only_for_the_captured_sources(tmp_path, monkeypatch):
    bf16, fp8 = bench.kernel_source_hash(False), bench.kernel_source_hash(True)
    assert bf16 != fp8
    path = _write(tmp_path, {
        "a": {"dram_bytes_per_launch": 1000, "units": 4, "kernel_source_hash": bf16},
        "b": {"dram_bytes_per_launch": 500, "units": 1, "kernel_source_hash": fp8},
        "c": {"dram_bytes_per_launch": 700, "units": 1, "kernel_source_hash": "0" * 16},
    })
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", path)
    assert bench.profiled_traffic("a", 4) == 1000
    assert bench.profiled_traffic("a", 8) == 2000  # scaled by units
    assert bench.profiled_traffic("a", 4, fp8=True) is None  # other kernel
    assert bench.profiled_traffic("b", 1, fp8=True) == 500
    assert bench.profiled_traffic("b", 1) is None
    assert bench.profiled_traffic("c", 1) is None  # sources changed since
    assert bench.profiled_traffic("missing", 1) is None


def test_no_summary_file_means_no_traffic(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "absent.json"))
    assert bench.profiled_traffic("dp16", 1) is None


def test_source_hash_follows_the_kernel_files(tmp_path, monkeypatch):
    """The hash changes when any file it covers changes."""
    import shutil
    root = tmp_path / "r"
    csrc = root / "mla_latent_decode_gb300" / "csrc"
    shutil.copytree(bench.os.path.join(bench.ROOT, "mla_latent_decode_gb300", "csrc"), csrc)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash(False)
    assert h0 == bench.kernel_source_hash(False)
    (csrc / "ptx_sm103.cuh").write_text((csrc / "ptx_sm103.cuh").read_text() + "\n")
    assert bench.kernel_source_hash(False) != h0
