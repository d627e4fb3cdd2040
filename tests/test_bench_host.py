"""The benchmark's host-side accounting on CPU: the algorithmic bytes behind
`roofline.achieved` and `cycle`, and the rule that `roofline.traffic` comes
from a committed ncu summary only while the kernel's sources are unchanged."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_drafting_gb300 import synth  # noqa: E402


def test_algorithmic_bytes_at_the_headline_size():
    """U once, W2 once, the W1 rows; the target rows the decisions read; for
    each rejecting request its U_j and P_j rows again plus W2 once more.  The
    sweep's per-launch share counts W2 once per cycle (amortised over gamma)."""
    w = synth.WORKLOADS["headline"]
    R, g, V, r = w.R, w.gamma, w.V, w.r
    n_rej, rows = 235.0, 620.0
    ab = bench.algorithmic_bytes(w, n_rej, rows)
    draft = R * g * V * 4 + r * V * 2 + R * g * r * 2
    verify = rows * V * 4
    resid = n_rej * V * (4 + 4) + r * V * 2
    assert ab["draft"] == draft
    assert ab["verify_rows"] == verify
    assert ab["residual"] == resid
    assert ab["total"] == draft + verify + resid
    assert ab["sweep_per_launch"] == R * V * 4 + r * V * 2 / g + R * r * 2
    assert round(ab["sweep_per_launch"]) == 171271782          # the figure the bench line reports
    # no rejection: the residual pass moves nothing
    assert bench.algorithmic_bytes(w, 0.0, rows)["residual"] == 0


def test_algorithmic_bytes_follow_the_storage_dtypes():
    w = synth.WORKLOADS["longblock"]                              # U, P and W in bf16
    ab = bench.algorithmic_bytes(w, 10.0, 100.0)
    assert ab["draft"] == w.R * w.gamma * w.V * 2 + w.r * w.V * 2 + w.R * w.gamma * w.r * 2
    assert ab["verify_rows"] == 100.0 * w.V * 2
    assert ab["residual"] == 10.0 * w.V * 4 + w.r * w.V * 2


def test_traffic_is_read_only_while_the_sources_match(monkeypatch):
    """Each committed summary records a digest of its kernel's sources; the
    bench reports its DRAM bytes (read + write) only while the digest matches,
    and null once anything it covers has changed."""
    for kernel, (md, cu) in bench.KERNEL_PROFILES.items():
        text = open(os.path.join(ROOT, "profiles", md)).read()
        m = re.search(r"source sha256: ([0-9a-f]{64})", text)
        assert m, md
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
        want = 0.0
        for key in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            v = re.search(re.escape(key) + r" = ([0-9.]+) (byte|Kbyte|Mbyte|Gbyte)", text)
            want += float(v.group(1)) * scale[v.group(2)]
        if m.group(1) == bench.source_digest(cu):
            assert bench.measured_traffic(kernel) == int(want)
        else:
            assert bench.measured_traffic(kernel) is None
    monkeypatch.setattr(bench, "source_digest", lambda cu: "0" * 64)
    for kernel in bench.KERNEL_PROFILES:
        assert bench.measured_traffic(kernel) is None
    assert bench.measured_traffic("no_such_kernel") is None


def test_source_digest_covers_the_kernel_and_every_header(tmp_path, monkeypatch):
    """Changing the kernel's .cu file or any library header changes the digest."""
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    inc = tmp_path / "include"
    inc.mkdir()
    (csrc / "k.cu").write_text("kernel")
    (csrc / "a.cuh").write_text("header a")
    (csrc / "b.h").write_text("header b")
    (inc / "dspark.h").write_text("abi")
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.source_digest("k.cu")
    assert bench.source_digest("k.cu") == d0
    for f in (csrc / "k.cu", csrc / "a.cuh", csrc / "b.h", inc / "dspark.h"):
        old = f.read_text()
        f.write_text(old + " ")
        assert bench.source_digest("k.cu") != d0, f.name
        f.write_text(old)
    assert bench.source_digest("k.cu") == d0
