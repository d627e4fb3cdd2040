"""GPU parity of the fused confidence head and of the threshold filter.

Confidence head (DSpark blog, section 4.1 ConfidenceHead): the c that the
draft kernels write against the oracle's sigmoid(w . [h_k, W1[x_{k-1}]]) on
the same bytes and the GPU's own drafted tokens.  Tolerance, from the
arithmetic: the GPU sums the d + r products in float32 (a strided share per
thread of at most ceil((d + r) / 512) terms, then a 32-lane tree and a
16-term sum), so the logit error is below (ceil((d + r)/512) + 5 + 16) u S
with u = 2^-24 and S = sum |w_i x_i|; S < 40 for every case here (d <= 2048,
|w| ~ 0.02-0.3 scaled inputs), i.e. under 6e-5 on the logit and, sigmoid
having slope <= 1/4, under 1.5e-5 on c; expf adds < 1e-6.  The tests use
2e-5.  Turning the head on leaves every other draft output bit-identical.

Threshold filter (blog section 4.3): lengths bit-exact, since both sides
decide on the same float32 prefix product.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import dev, host
from speculative_decoding_drafting_gb300 import binding, synth

pytestmark = pytest.mark.gpu

C_TOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def _draft(w, x, seed, conf_w=None, conf_H=None):
    a = [dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"])]
    cw = None if conf_w is None else dev(conf_w)
    cH = None if conf_H is None else dev(conf_H)
    if w.head == "rnn":
        d = binding.draft_rnn(*a, dev(x["Wgco"]), dev(x["H"]), w.T, seed, conf_w=cw, conf_H=cH)
    else:
        d = binding.draft_markov(*a, w.T, seed, conf_w=cw, conf_H=cH)
    torch.cuda.synchronize()
    assert binding.workspace_status(d["ws"]) == 0
    return {k: host(v) for k, v in d.items() if k != "ws"}


CASES = {
    "markov_bf16": (synth.Workload("cm", R=6, gamma=4, V=20488, r=64, T=1.0), 96),
    "markov_greedy": (synth.Workload("cg", R=5, gamma=3, V=8200, r=128, T=0.0, sigma_u=2.0), 1000),
    "markov_f32_r7": (synth.Workload("cf", R=3, gamma=2, V=1036, r=7, T=1.3, w_dtype=synth.F32, sigma_w=0.3), 33),
    "markov_embedding_only": (synth.Workload("ce", R=4, gamma=3, V=4104, r=64, T=1.0, sigma_w=0.3), 0),
    "markov_multigroup": (synth.Workload("cmg", R=256, gamma=2, V=4104, r=64, T=1.0), 512),
}


@pytest.mark.parametrize("name", list(CASES))
def test_confidence_head_markov(name):
    w, d = CASES[name]
    x = synth.gen_all(w)
    wc = synth.gen_conf_w(w, d)
    H = synth.gen_conf_H(w, d) if d > 0 else None
    plain = _draft(w, x, 11)
    g = _draft(w, x, 11, conf_w=wc, conf_H=H)
    for k in ("tokens", "q_tok", "lse", "code"):
        np.testing.assert_array_equal(g[k], plain[k], err_msg=f"{name}: head changed {k}")
    Hs = H if H is not None else np.zeros((w.R, w.gamma, 0), np.uint16)
    o = oracle.confidence(Hs, x["W1"], wc, x["anchor"], g["tokens"])
    np.testing.assert_allclose(g["c"], o, rtol=0, atol=C_TOL, err_msg=name)
    assert np.all((g["c"] > 0) & (g["c"] < 1))


@pytest.mark.parametrize("own_H", [True, False])
def test_confidence_head_rnn(own_H):
    w = synth.Workload("crnn", R=4, gamma=3, V=8200, r=64, T=1.0, head="rnn", d=96)
    x = synth.gen_all(w)
    dc = w.d if own_H else 200
    wc = synth.gen_conf_w(w, dc)
    H = None if own_H else synth.gen_conf_H(w, dc)
    plain = _draft(w, x, 5)
    g = _draft(w, x, 5, conf_w=wc, conf_H=H)
    for k in ("tokens", "q_tok", "lse", "code", "state"):
        np.testing.assert_array_equal(g[k], plain[k], err_msg=f"head changed {k}")
    o = oracle.confidence(x["H"] if own_H else H, x["W1"], wc, x["anchor"], g["tokens"])
    np.testing.assert_allclose(g["c"], o, rtol=0, atol=C_TOL)


def test_confidence_head_full_size():
    """The benchmark's draft launch (R = 256, gamma = 5, V = 151936, r = 256)
    with a d = 2048 head: every request's c against the oracle."""
    w = synth.WORKLOADS["headline"]
    x = synth.gen_all(w)
    d = 2048
    wc = synth.gen_conf_w(w, d)
    H = synth.gen_conf_H(w, d)
    g = _draft(w, x, 2024, conf_w=wc, conf_H=H)
    o = oracle.confidence(H, x["W1"], wc, x["anchor"], g["tokens"])
    np.testing.assert_allclose(g["c"], o, rtol=0, atol=C_TOL)


def _threshold_inputs(R, gamma, seed):
    rng = np.random.default_rng(seed)
    c = (1 / (1 + np.exp(-rng.normal(1.5, 1.2, (R, gamma))))).astype(np.float32)
    c[rng.random((R, gamma)) < 0.03] = 1.0
    c[rng.random((R, gamma)) < 0.02] = 0.0
    c[rng.random((R, gamma)) < 0.01] = np.nan
    return c


@pytest.mark.parametrize("R,gamma", [(1, 1), (7, 5), (300, 16), (256, 5), (9000, 64)])
@pytest.mark.parametrize("mode", [0, 1])
def test_threshold_filter_parity(R, gamma, mode):
    c = _threshold_inputs(R, gamma, R * 131 + gamma)
    a = oracle.prefix_survival(c)
    # thresholds: a grid, and values that tie exactly with some a or c
    thetas = list(np.linspace(-0.05, 1.05, 12).astype(np.float32))
    finite = a[np.isfinite(a)]
    thetas += [finite[0], finite[len(finite) // 2], np.float32(1.0), np.float32(0.0)]
    cd = dev(c)
    for th in thetas:
        g = host(binding.schedule_threshold(cd, float(th), mode))
        o = oracle.threshold_lengths(c, float(th), mode)
        np.testing.assert_array_equal(g, o, err_msg=f"theta {th} mode {mode}")
