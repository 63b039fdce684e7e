"""Host-side pieces of the measurement contract, checked without a GPU:

- the bench reports a kernel's DRAM traffic from a committed ncu summary
  only while the summary names the kernel source's current hash, and
  reports none once the source has changed;
- every ncu command recorded under profiles/ leaves the GPU clocks alone
  (`--clock-control none`) and every summary gives the commands it came
  from and the traffic line the bench reads."""

import hashlib
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _write(path, text):
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write(text)


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "k" / "kernel.cu"
    _write(str(src), "__global__ void k() {}\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    summary = ("# k\n\nsource sha256 (first 16 hex): %s\n\n"
               "traffic (DRAM read + write) per launch: 123456 bytes\n" % digest)
    _write(str(tmp_path / "profiles" / "k.md"), summary)
    assert bench.profiled_traffic("k/kernel.cu", "k.md") == 123456
    # a note after the hash (e.g. the capture's own hash) does not hide it
    _write(str(tmp_path / "profiles" / "k2.md"),
           summary.replace(digest + "\n", digest + " (captured at 0123456789abcdef)\n"))
    assert bench.profiled_traffic("k/kernel.cu", "k2.md") == 123456
    # the source changes: no traffic
    _write(str(src), "__global__ void k() { }\n")
    assert bench.profiled_traffic("k/kernel.cu", "k.md") is None
    # missing summary or missing source: no traffic
    assert bench.profiled_traffic("k/kernel.cu", "absent.md") is None
    assert bench.profiled_traffic("k/absent.cu", "k.md") is None


def test_profiled_traffic_needs_both_lines(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "kernel.cu"
    _write(str(src), "x\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    _write(str(tmp_path / "profiles" / "a.md"), "source sha256 (first 16 hex): %s\n" % digest)
    _write(str(tmp_path / "profiles" / "b.md"), "traffic (DRAM read + write) per launch: 5 bytes\n")
    assert bench.profiled_traffic("kernel.cu", "a.md") is None
    assert bench.profiled_traffic("kernel.cu", "b.md") is None


def _summaries():
    return sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


@pytest.mark.parametrize("name", _summaries())
def test_profile_summaries_keep_the_clocks_and_name_their_commands(name):
    text = open(os.path.join(PROFILES, name)).read()
    ncu_lines = [l for l in text.splitlines() if re.match(r"\s*ncu\s", l)]
    assert ncu_lines, f"{name}: no ncu command recorded"
    for l in ncu_lines:
        assert "--clock-control none" in l, f"{name}: ncu without --clock-control none: {l}"
    # the plain run of the same command precedes each capture
    assert "python bench.py" in text, f"{name}: the profiled command is not given"
    assert re.search(r"source sha256 \(first 16 hex\): [0-9a-f]{16}", text), f"{name}: no source hash"
    assert re.search(r"traffic \(DRAM read \+ write\) per launch: \d+ bytes", text), \
        f"{name}: no traffic line"
    # raw ncu reports stay out of the repository
    assert not [f for f in os.listdir(PROFILES) if f.endswith((".ncu-rep", ".nsys-rep", ".qdrep"))]
