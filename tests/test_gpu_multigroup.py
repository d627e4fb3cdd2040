"""GPU parity with several 128-request M-groups, and at the full headline size.

The tensor-core draft sweep gives each 128-request M-group its own CTAs; the
M-groups that share a column slice run in thread-block clusters of two that
share every W2 stage (when their number is even; no cluster otherwise, and at
four M-groups a slice has two clusters).  These cases cover each cluster shape,
a ragged last M-group, and the full-size launch the benchmark times
(R = 256, gamma = 5, V = 151936, r = 256), where the oracle checks a sample of
requests through their request ids.
"""
import numpy as np
import pytest
import torch

from _parity import Flags, compare_draft, compare_verify, gpu_draft, gpu_verify_on, oracle_draft, oracle_verify_on
from speculative_decoding_drafting_gb300 import binding, synth

pytestmark = pytest.mark.gpu

MULTI = {
    # two M-groups -> clusters of two; ragged last tile and chunk (V = 48 tiles + 8 columns)
    "mg2": synth.Workload("mg2", R=256, gamma=2, V=6152, r=64, T=1.0),
    # three M-groups (the last one 44 requests) -> no cluster
    "mg3": synth.Workload("mg3", R=300, gamma=2, V=4104, r=128, T=0.9),
    # four M-groups -> two clusters of two per slice
    "mg4": synth.Workload("mg4", R=512, gamma=2, V=4104, r=64, T=1.0),
    # greedy with two M-groups
    "mg2_greedy": synth.Workload("mg2_greedy", R=256, gamma=2, V=4104, r=64, T=0.0, sigma_u=2.0),
    # RNN head: f32 codes as three bf16 terms on the tensor cores, two and four M-groups
    "mg2_rnn": synth.Workload("mg2_rnn", R=256, gamma=2, V=4104, r=64, T=1.0, head="rnn", d=96),
    "mg4_rnn": synth.Workload("mg4_rnn", R=512, gamma=2, V=2056, r=128, T=0.8, head="rnn", d=64),
    # RNN head at r = 256: the sweep's codes as two bf16 terms (three would leave
    # tensor memory for one accumulator only); every request compared
    "mg2_rnn256": synth.Workload("mg2_rnn256", R=256, gamma=3, V=4104, r=256, T=1.0, head="rnn", d=96),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


@pytest.mark.parametrize("name", list(MULTI))
def test_draft_parity_multigroup(name):
    w = MULTI[name]
    x = synth.gen_all(w)
    g = gpu_draft(w, x, seed=31)
    o = oracle_draft(w, x, seed=31)
    flags = Flags()
    n, nflag, m = compare_draft(g, o, tag=name, flags=flags)
    assert n >= w.R
    flags.check(name)
    if w.head == "markov":
        np.testing.assert_array_equal(g["code"][m], o["code"][m].astype(np.float32))
    else:
        np.testing.assert_allclose(g["code"][m], o["code"][m], atol=2e-5)


@pytest.mark.parametrize("name,mode", [("mg2", "all"), ("mg3", "all"), ("mg4", "all"), ("mg4", "random"),
                                                ("mg2_rnn", "all"), ("mg4_rnn", "random")])
def test_verify_parity_multigroup(name, mode):
    """The residual pass runs one CTA per 128 rejecting requests and column
    slice, clusters of two M-groups sharing W2; with random verify lengths
    fewer requests reject and the last M-group of a cluster may be empty."""
    w = MULTI[name]
    x = synth.gen_all(w)
    dr = oracle_draft(w, x, 8)
    vl = None if mode == "all" else np.random.default_rng(5).integers(0, w.gamma + 1, w.R).astype(np.int32)
    g = gpu_verify_on(w, x, dr, 8, verify_len=vl)
    o = oracle_verify_on(w, x, dr, 8, verify_len=vl)
    flags = Flags()
    flags.positions += w.R * w.gamma
    n, nflag = compare_verify(g, o, np.ones(w.R, bool), tag=name, flags=flags)
    assert n + nflag == w.R
    flags.check(name)


@pytest.mark.parametrize("name", ["headline", "dspark5", "greedy", "rnn", "longblock"])
def test_full_size_sampled(name):
    """Full-size launches: the benchmark's headline cycle, DSpark-5 at 64
    requests (one M-group, half of its rows empty), the greedy cycle, the RNN
    head (gamma = 8, d = 2048) and the long block (R = 512, gamma = 16, bf16
    storage, T = 0.8).  GPU draft and verify run on every request; the oracle
    recomputes a sample of requests (every M-group, its edges) from the same
    bytes and request ids."""
    w = synth.WORKLOADS[name]
    x = synth.gen_all(w)
    seed = 2024
    g = gpu_draft(w, x, seed)
    gv = gpu_verify_on(w, x, g, seed)
    idx = np.array(sorted(i for i in {0, 1, 126, 127, 128, 200, w.R // 2 + 5, w.R - 129, w.R - 2, w.R - 1}
                          if 0 <= i < w.R))
    xs = {k: (v[idx] if k in ("U", "P", "anchor", "H") else v) for k, v in x.items()}
    o = oracle_draft(w, xs, seed, req_ids=idx.astype(np.uint32))
    gs = {k: v[idx] for k, v in g.items()}
    _, _, m = compare_draft(gs, o, tag=name)
    same = (gs["tokens"] == o["tokens"]).all(axis=1)
    ov = oracle_verify_on(w, xs, o, seed, req_ids=idx.astype(np.uint32))
    gvs = {k: v[idx] for k, v in gv.items()}
    n, _ = compare_verify(gvs, ov, same, tag=name)
    assert n >= len(idx) - 2
