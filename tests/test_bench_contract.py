"""bench.py's host-side helpers (CPU only): profiled DRAM traffic is reported
only while the kernel sources are the ones it was measured on."""

from __future__ import annotations

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_follows_the_kernel_source_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    for f in bench.KERNEL_SOURCES:
        d = tmp_path / os.path.dirname(f)
        d.mkdir(parents=True, exist_ok=True)
        with open(os.path.join(ROOT, f), "rb") as src, open(tmp_path / f, "wb") as dst:
            dst.write(src.read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    (prof / "traffic.json").write_text(json.dumps({"kernel_source_sha256_16": h, "w": 123}))
    assert bench.load_profile_traffic("w") == 123
    assert bench.load_profile_traffic("other") is None
    # any change to a kernel source voids the figure
    with open(tmp_path / bench.KERNEL_SOURCES[0], "ab") as f:
        f.write(b"\n// edited\n")
    assert bench.kernel_source_hash() != h
    assert bench.load_profile_traffic("w") is None

