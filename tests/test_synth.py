"""The seeded input generator: every array is reproducible, and any subset of
requests can be regenerated on its own (one child stream per request), which
the reference arm and the full-size parity samples rely on."""
import numpy as np

from speculative_decoding_drafting_gb300 import synth


def _small(**kw):
    base = dict(R=6, gamma=3, V=512, r=16, T=1.0, head="rnn", d=8)
    base.update(kw)
    return synth.Workload("t", **base)


def test_generation_is_reproducible_and_seeded():
    a, b = synth.gen_all(_small()), synth.gen_all(_small())
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    c = synth.gen_all(_small(seed=1))
    assert not np.array_equal(a["U"], c["U"]) and not np.array_equal(a["W2"], c["W2"])


def test_a_subset_of_requests_regenerates_identically():
    w = _small()
    full = synth.gen_all(w)
    idx = np.array([1, 4, 5])
    sub = synth.gen_all(w, rows=idx)
    for k in ("U", "P", "anchor", "c", "H"):
        np.testing.assert_array_equal(sub[k], full[k][idx], err_msg=k)
    for k in ("W1", "W2", "Wgco"):
        np.testing.assert_array_equal(sub[k], full[k], err_msg=k)
    np.testing.assert_array_equal(sub["req_ids"], idx.astype(np.uint32))


def test_shapes_and_storage_follow_the_workload():
    w = _small(u_dtype=synth.BF16, p_dtype=synth.BF16)
    x = synth.gen_all(w)
    assert x["U"].shape == (6, 3, 512) and x["U"].dtype == np.uint16
    assert x["P"].shape == (6, 4, 512) and x["P"].dtype == np.uint16
    assert x["W1"].shape == (512, 16) and x["W2"].shape == (16, 512)
    assert x["H"].shape == (6, 3, 8) and x["Wgco"].shape == (2 * 16 + 8, 3 * 16)
    assert ((x["anchor"] >= 0) & (x["anchor"] < 512)).all()
    assert ((x["c"] > 0) & (x["c"] < 1)).all()
