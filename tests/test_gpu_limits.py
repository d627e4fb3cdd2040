"""GPU parity at the documented size limits (include/dspark.h): gamma = 64,
V up to 2^20 (sampled, where the verifier groups residual chunks, and greedy), r = 1024 (the CUDA-core
sweep), the RNN head at r = 512 (tensor-core GRU, CUDA-core sweep), eight
128-request M-groups, and a d = 16384 confidence head.  Comparison rules as in
test_gpu_parity.py."""
import numpy as np
import pytest
import torch

import oracle
from _parity import Flags, compare_draft, compare_verify, dev, gpu_draft, gpu_verify_on, host, oracle_draft, oracle_verify_on
from speculative_decoding_drafting_gb300 import binding, synth

pytestmark = pytest.mark.gpu

F32 = synth.F32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


LIMITS = {
    "gamma64": synth.Workload("gamma64", R=3, gamma=64, V=4104, r=64, T=1.0),
    "v2p18_sampled": synth.Workload("v2p18", R=2, gamma=2, V=1 << 18, r=64, T=1.0),
    "v2p20_greedy": synth.Workload("v2p20", R=2, gamma=2, V=1 << 20, r=32, T=0.0, sigma_u=2.0),
    # more than 1024 residual chunks: the sampler groups them four to a top-tree leaf
    "v2p20_sampled": synth.Workload("v2p20s", R=4, gamma=2, V=(1 << 20) - 8, r=32, T=1.0, sigma_pnoise=2.0),
    "v2p19_sampled": synth.Workload("v2p19s", R=4, gamma=2, V=(1 << 19) + 24, r=32, T=1.0, sigma_pnoise=2.0),
    "r1024": synth.Workload("r1024", R=3, gamma=2, V=2056, r=1024, T=1.0, sigma_w=0.01),
    "rnn_r512": synth.Workload("rnn_r512", R=4, gamma=2, V=4104, r=512, T=1.0, head="rnn", d=128, sigma_w=0.01),
    "mg8": synth.Workload("mg8", R=1024, gamma=2, V=1032, r=64, T=1.0),
}


@pytest.mark.parametrize("name", list(LIMITS))
def test_limits_draft_and_verify(name):
    w = LIMITS[name]
    x = synth.gen_all(w)
    seed = 77
    g = gpu_draft(w, x, seed)
    o = oracle_draft(w, x, seed)
    flags = Flags()
    n, nflag, m = compare_draft(g, o, tag=name, flags=flags)
    assert n >= w.R
    flags.check(name)
    if w.head == "markov":
        np.testing.assert_array_equal(g["code"][m], o["code"][m].astype(np.float32))
    else:
        np.testing.assert_allclose(g["code"][m], o["code"][m], atol=2e-5)
    # verification on the oracle's drafts: identical inputs on both sides
    gv = gpu_verify_on(w, x, o, seed)
    ov = oracle_verify_on(w, x, o, seed)
    nv, nvf = compare_verify(gv, ov, np.ones(w.R, bool), tag=name)
    assert nv + nvf == w.R
    if name.endswith("_sampled"):
        # the residual draw (not only the bonus draw) is exercised
        assert (np.asarray(ov["accept_len"]) < w.gamma).any()


def test_limits_confidence_head_d16384():
    w = synth.Workload("conf_d16k", R=2, gamma=3, V=2056, r=64, T=1.0)
    x = synth.gen_all(w)
    d = 16384
    wc, H = synth.gen_conf_w(w, d), synth.gen_conf_H(w, d)
    out = binding.draft_markov(dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"]), w.T, 5, conf_w=dev(wc),
                               conf_H=dev(H))
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in out.items() if k != "ws"}
    o = oracle.confidence(H, x["W1"], wc, x["anchor"], g["tokens"])
    # error bound of the float32 sum (test_gpu_conf.py) at d + r = 16448 and sum |w x| ~ 210: 1.7e-4
    np.testing.assert_allclose(g["c"], o, rtol=0, atol=2e-4)
