"""The DRAM-traffic record behind bench.py's roofline.traffic (host logic, CPU).

bench.py reads the DRAM bytes per launch of its default workload from the ncu
summary under profiles/ and reports them only while the kernel sources hash
to the digest recorded beside them; otherwise traffic is null.  These tests
read the summary as text and never need a GPU or ncu."""
import os
import re
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402

# Q6_K super-block: 256 values in 210 bytes (mlx-native 0.18.0
# src/ops/row_exact_matvec.rs, block constants)
Q6_K_VALUES, Q6_K_BYTES = 256, 210


def _record(workload):
    with open(os.path.join(ROOT, "profiles", f"rem_mv_{workload}.md")) as f:
        text = f.read()
    sha = re.search(r"kernel_sources_sha256: ([0-9a-f]{64})", text)
    traffic = re.search(r"dram_bytes_per_launch: (\d+)", text)
    assert sha and traffic, "the summary records the digest and the bytes per launch"
    return sha.group(1), float(traffic.group(1))


def test_default_profile_traffic_is_one_pass_over_the_weights():
    """The recorded bytes per launch are one read of every weight plus the
    inputs and outputs of an m = 1 call, within 5 % (ECC, page-table and
    output write-back traffic on top); well above that would be re-reads."""
    fmt, n, k, batch, ms = bench.WORKLOADS[bench.DEFAULT][:5]
    assert fmt == "q6_K" and k % Q6_K_VALUES == 0
    _, traffic = _record(bench.DEFAULT)
    m = min(ms)
    algorithmic = batch * n * (k // Q6_K_VALUES) * Q6_K_BYTES + 4 * batch * m * (k + n)
    assert 1.0 <= traffic / algorithmic <= 1.05


def test_traffic_reported_only_for_the_recorded_sources(monkeypatch):
    sha, traffic = _record(bench.DEFAULT)
    monkeypatch.setattr(bench, "kernel_sources_sha256", lambda: sha)
    assert bench.profiled_traffic(bench.DEFAULT) == traffic
    monkeypatch.setattr(bench, "kernel_sources_sha256", lambda: "0" * 64)
    assert bench.profiled_traffic(bench.DEFAULT) is None
    assert bench.profiled_traffic("no_such_workload") is None


@pytest.mark.parametrize("edit", ["quantized_few_row_gb300/csrc/rem_tc.cuh",
                                  "quantized_few_row_gb300/csrc/rem_host.cu", "include/rem.h"])
def test_digest_follows_every_kernel_source(tmp_path, monkeypatch, edit):
    """Any byte changed in a CUDA source, the host planner or the public
    header changes the digest (so a stale record reads as null)."""
    for sub in ("quantized_few_row_gb300/csrc", "include"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = bench.kernel_sources_sha256()
    with open(tmp_path / edit, "ab") as f:
        f.write(b"\n")
    assert bench.kernel_sources_sha256() != before
