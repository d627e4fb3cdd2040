"""GPU parity of Sequential Temperature Scaling (DSpark blog, section 4.2).

dspark_sts_fit against the oracle's left-to-right grid search.  Which bin a
calibrated prefix survival joins is decided as in double arithmetic on both
sides (the kernel redoes values near a bin edge in double), and the per-bin
sums are exact on the GPU, so the GPU's ECE values differ from the oracle's
only by float32 rounding of the survival values (about 1e-7; the tests allow
1e-6).  The chosen grid index must match wherever the oracle's best and
second-best ECE are 1e-6 or more apart; at a closer position either may be
taken, and when the GPU took the other one the later positions of that set
(which condition on it) are not compared.

dspark_sts_apply and the head's per-position temperatures against the
oracle: float32 logit and sigmoid, 1e-5 absolute for temperatures >= 0.1.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import dev, host
from speculative_decoding_drafting_gb300 import binding, synth

pytestmark = pytest.mark.gpu

ECE_TOL = 1e-6
GAP_FLAG = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def _compare_fit(c, al, grid, M, tag):
    g = binding.sts_fit(dev(c), dev(al), dev(grid), M)
    torch.cuda.synchronize()
    assert binding.workspace_status(g["ws"]) == 0
    g = {k: host(v) for k, v in g.items() if k != "ws"}
    o = oracle.sts_fit(c, al, grid, M)
    gamma = c.shape[1]
    compared = 0
    for k in range(gamma):
        np.testing.assert_allclose(g["ece"][k], o["ece"][k], rtol=0, atol=ECE_TOL, err_msg=f"{tag} ece k={k + 1}")
        if g["g"][k] != o["g"][k]:
            assert o["gap"][k] < GAP_FLAG, (tag, k, g["g"][k], o["g"][k], o["gap"][k])
            break
        assert g["t"][k] == grid[g["g"][k]]
        if np.isfinite(o["gap"][k]):
            assert abs(g["gap"][k] - o["gap"][k]) < 2 * ECE_TOL
        else:
            assert np.isinf(g["gap"][k])
        compared += 1
    return compared


@pytest.mark.parametrize("N,gamma,G,M,tau", [
    (1, 1, 1, 1, 2.0),            # one block, one grid point, one bin
    (7, 3, 5, 4, 2.0),            # fewer samples than bins
    (2048, 4, 64, 15, 2.0),       # exactly one chunk
    (5003, 5, 64, 15, 0.5),       # ragged last chunk, underconfident
    (20000, 5, 128, 10, 2.0),
    (9000, 3, 300, 32, 1.0),      # grid not a multiple of 8, the most bins
])
def test_sts_fit_parity(N, gamma, G, M, tau):
    c, al = synth.gen_sts_set(N, gamma, tau=tau, seed=N + G)
    grid = synth.sts_grid(G, 0.1, 10.0)
    n = _compare_fit(c, al, grid, M, f"N{N}")
    assert n >= 1


def test_sts_fit_degenerate_inputs():
    """Confidences of exactly 0, 1/2 and 1 (fixed by every temperature, so
    every grid point ties and the lowest index wins), outcomes all 0 or all
    gamma, and predictions landing exactly on bin edges."""
    rng = np.random.default_rng(0)
    N, gamma = 3000, 4
    c = rng.choice(np.array([0.0, 0.5, 1.0], np.float32), size=(N, gamma))
    for al in (np.zeros(N, np.int32), np.full(N, gamma, np.int32), rng.integers(0, gamma + 1, N).astype(np.int32)):
        grid = synth.sts_grid(16, 0.5, 2.0)
        g = {k: host(v) for k, v in binding.sts_fit(dev(c), dev(al), dev(grid), 4).items() if k != "ws"}
        o = oracle.sts_fit(c, al, grid, 4)
        np.testing.assert_array_equal(g["g"], o["g"])
        np.testing.assert_array_equal(g["g"], np.zeros(gamma, np.int32))
        np.testing.assert_allclose(g["ece"], o["ece"], rtol=0, atol=1e-12)


def test_sts_fit_benchmark_size():
    """The benchmark's calibration set: 65536 blocks, gamma = 8, 256
    temperatures, 15 bins; the fit recovers the generator's tau = 2."""
    c, al = synth.gen_sts_set(65536, 8, tau=2.0, seed=1)
    grid = synth.sts_grid(256, 0.1, 10.0)
    n = _compare_fit(c, al, grid, 15, "bench")
    assert n >= 1


def test_sts_apply_parity():
    rng = np.random.default_rng(4)
    c = rng.random((1000, 6)).astype(np.float32)
    c[0] = [0.0, 1.0, 0.5, 1e-30, 1 - 2 ** -24, 0.25]
    t = np.array([0.1, 0.5, 1.0, 2.0, 7.5, 10.0])
    g = host(binding.sts_apply(dev(c), dev(t)))
    o = oracle.sts_apply(c, t)
    np.testing.assert_allclose(g, o, rtol=0, atol=1e-5)
    assert g[0, 0] == 0.0 and g[0, 1] == 1.0 and g[0, 2] == 0.5


def test_confidence_head_with_temperatures():
    w = synth.Workload("ct", R=6, gamma=4, V=20488, r=64, T=1.0)
    x = synth.gen_all(w)
    d = 96
    wc, H = synth.gen_conf_w(w, d), synth.gen_conf_H(w, d)
    t = np.array([0.5, 1.0, 2.0, 4.0])
    a = [dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"])]
    out = binding.draft_markov(*a, w.T, 3, conf_w=dev(wc), conf_H=dev(H), conf_t=dev(t))
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in out.items() if k != "ws"}
    o = oracle.confidence(H, x["W1"], wc, x["anchor"], g["tokens"], temps=t)
    np.testing.assert_allclose(g["c"], o, rtol=0, atol=2e-5 / 0.5)
