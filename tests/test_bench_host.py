"""The benchmark's host-side accounting on CPU: the algorithmic bytes behind
`roofline.achieved` and `cycle`, and the rule that `roofline.traffic` comes
from a committed ncu summary only while the kernel's sources are unchanged."""
import os
import re
import sys

import numpy as np
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


def test_flag_accounting_of_the_cpu_leg():
    """count_flags: positions are compared up to a request's first draft
    disagreement; a disagreement counts as flagged only where the oracle's
    margin (draft) or uniform gap (verification) lies inside its band."""
    R, gamma = 4, 3
    od = dict(tokens=np.arange(R * gamma, dtype=np.int32).reshape(R, gamma), margin=np.ones((R, gamma)))
    od["margin"][1, 1] = 5e-5                      # request 1, position 2: inside the Gumbel band
    ov = dict(out_tokens=np.zeros((R, gamma + 1), np.int32), accept_len=np.full(R, 2, np.int32),
              min_gap=np.ones(R))
    ov["min_gap"][2] = 1e-7                        # request 2: a verification decision inside the band
    g_tok = od["tokens"].copy()
    g_tok[1, 1] += 1                               # flagged draft disagreement (position 2 of 3)
    g_tok[3, 0] += 1                               # unflagged draft disagreement at position 1
    g_out = ov["out_tokens"].copy()
    g_out[2, 0] = 9                                # flagged verification disagreement
    g_acc = ov["accept_len"].copy()
    acc = dict(positions=0, flagged=0, flagged_disagreements=0, unflagged_disagreements=0)
    bench.count_flags(od, ov, g_tok, g_out, g_acc, acc)
    assert acc["positions"] == 3 + 2 + 3 + 1
    assert acc["flagged"] == 1 + 1                 # the draft margin and the verification gap
    assert acc["flagged_disagreements"] == 2 and acc["unflagged_disagreements"] == 1


def test_greedy_cycle_has_no_residual_bytes():
    """At T = 0 a mismatch emits the target row's argmax: no U_j / P_j re-read."""
    w = synth.WORKLOADS["greedy"]
    ab = bench.algorithmic_bytes(w, 200.0, 600.0)
    assert ab["residual"] == 0
    assert ab["total"] == ab["draft"] + 600.0 * w.V * 4


def test_device_generator_follows_the_recipe():
    """synth.gen_device draws the gen_all recipe on a torch generator: shapes,
    storage dtypes, the bonus row built from the last U row, and sigmas."""
    import torch
    w = synth.Workload("dev", R=8, gamma=3, V=4096, r=16, T=1.0, u_dtype=synth.BF16, p_dtype=synth.F32)
    x = synth.gen_device(w, "cpu", seed=3)
    assert x["U"].shape == (8, 3, 4096) and x["U"].dtype == torch.bfloat16
    assert x["P"].shape == (8, 4, 4096) and x["P"].dtype == torch.float32
    assert x["W1"].shape == (4096, 16) and x["W2"].shape == (16, 4096) and x["W2"].dtype == torch.bfloat16
    assert int(x["anchor"].min()) >= 0 and int(x["anchor"].max()) < 4096
    noise = x["P"][:, :3].float() - x["U"].float()
    assert abs(float(noise.std()) - w.sigma_pnoise) < 0.05
    assert abs(float(x["U"].float().std()) - w.sigma_u) < 0.05
    assert x["sps"].shape == (8 * 4 + 1,)
    y = synth.gen_device(w, "cpu", seed=3)
    assert torch.equal(x["U"], y["U"]) and torch.equal(x["P"], y["P"])
