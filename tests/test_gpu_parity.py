"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Discrete outputs (tokens, accept lengths, verify lengths) must be bit-exact
except at positions the oracle flags as near-ties (Gumbel or argmax margin
below 1e-4, a uniform within 1e-6 of its threshold); q(x), p(x) and the
log-sum-exps agree within 1e-4 relative.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import (compare_draft, compare_verify, dev, gpu_draft, gpu_verify_on, host, oracle_draft,
                     oracle_verify_on)
from speculative_decoding_drafting_gb300 import binding, synth

pytestmark = pytest.mark.gpu

F32, BF16 = synth.F32, synth.BF16

SMALL = {
    "toy": synth.WORKLOADS["toy"],
    "bf16_r64": synth.Workload("bf16_r64", R=6, gamma=4, V=20488, r=64, T=1.0),
    "bf16_storage_T08": synth.Workload("bf16_storage_T08", R=5, gamma=3, V=12296, r=128, T=0.8,
                                       u_dtype=BF16, p_dtype=BF16, sigma_pnoise=1.2),
    "greedy": synth.Workload("greedy", R=5, gamma=4, V=16392, r=64, T=0.0, sigma_u=2.0, sigma_pnoise=0.7),
    "rnn": synth.Workload("rnn", R=4, gamma=3, V=8200, r=64, T=1.0, head="rnn", d=96),
    "f32_r7": synth.Workload("f32_r7", R=3, gamma=2, V=1036, r=7, T=1.3, w_dtype=F32, sigma_w=0.3),
    "tiny": synth.Workload("tiny", R=1, gamma=1, V=8, r=1, T=1.0, w_dtype=F32, sigma_w=0.5),
    # temperature extremes: near-greedy (z spans about 250 nats) and nearly flat
    "cold_T005": synth.Workload("cold_T005", R=5, gamma=4, V=12296, r=64, T=0.05),
    "hot_T8": synth.Workload("hot_T8", R=5, gamma=4, V=12296, r=64, T=8.0, sigma_pnoise=4.0),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("seed", [0, 77])
def test_draft_parity(name, seed):
    w = SMALL[name].scaled(seed=seed)
    x = synth.gen_all(w)
    g = gpu_draft(w, x, seed=1000 + seed)
    o = oracle_draft(w, x, seed=1000 + seed)
    n, nflag, m = compare_draft(g, o, tag=name)
    assert n >= w.R
    # the rank-r code: W1 rows exactly (Markov) / tanh(out) to 1e-5 (RNN)
    if w.head == "markov":
        np.testing.assert_array_equal(g["code"][m], o["code"][m].astype(np.float32))
    else:
        np.testing.assert_allclose(g["code"][m], o["code"][m], atol=2e-5)


@pytest.mark.parametrize("name", [k for k in SMALL if k != "rnn"])
@pytest.mark.parametrize("mode", ["all", "random", "zero"])
def test_verify_parity_on_oracle_drafts(name, mode):
    w = SMALL[name]
    x = synth.gen_all(w)
    seed = 4242
    dr = oracle_draft(w, x, seed)
    rng = np.random.default_rng(3)
    vl = None if mode == "all" else (rng.integers(0, w.gamma + 1, w.R).astype(np.int32) if mode == "random"
                                     else np.zeros(w.R, np.int32))
    g = gpu_verify_on(w, x, dr, seed, verify_len=vl)
    o = oracle_verify_on(w, x, dr, seed, verify_len=vl)
    n, nflag = compare_verify(g, o, np.ones(w.R, bool), tag=name)
    assert n + nflag == w.R


def test_verify_parity_rnn_codes():
    w = SMALL["rnn"]
    x = synth.gen_all(w)
    dr = oracle_draft(w, x, 5)
    g = gpu_verify_on(w, x, dr, 5)
    o = oracle_verify_on(w, x, dr, 5)
    compare_verify(g, o, np.ones(w.R, bool), tag="rnn")


@pytest.mark.parametrize("name", ["toy", "bf16_r64", "greedy", "rnn"])
def test_cycle_end_to_end(name):
    """GPU draft -> GPU verify against oracle draft -> oracle verify."""
    w = SMALL[name]
    x = synth.gen_all(w)
    seed = 99
    g = gpu_draft(w, x, seed)
    o = oracle_draft(w, x, seed)
    _, _, m = compare_draft(g, o, tag=name)
    same = (g["tokens"] == o["tokens"]).all(axis=1)
    gv = gpu_verify_on(w, x, g, seed)
    ov = oracle_verify_on(w, x, o, seed)
    compare_verify(gv, ov, same, tag=name)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_q_equal_to_p_accepts_every_draft(T):
    """Explainer section 05: where the target's distribution equals the
    draft's, nothing is rejected.  W2 = 0 makes q_k = softmax(U_k / T); the
    target rows repeat U (the bonus row repeats the last position), so p = q
    and every block is accepted whole, with its bonus token drawn from
    softmax(U_gamma / T).  The only admissible exception is a uniform within
    the flag band of a ratio that rounding puts a hair below 1."""
    w = synth.Workload("q_eq_p", R=48, gamma=4, V=4104, r=64, T=T)
    x = synth.gen_all(w)
    x["W2"] = synth.f32_to_bf16_bits(np.zeros((w.r, w.V), np.float32))
    x["P"] = np.concatenate([x["U"], x["U"][:, -1:, :]], axis=1)
    seed = 404
    g = gpu_draft(w, x, seed)
    o = oracle_draft(w, x, seed)
    compare_draft(g, o, tag="q_eq_p")
    gv = gpu_verify_on(w, x, g, seed)
    ov = oracle_verify_on(w, x, g, seed)
    assert np.all(ov["accept_len"] == w.gamma)
    ok = ov["min_gap"] >= 1e-6
    assert np.all(gv["accept_len"][ok] == w.gamma) and np.all(gv["n_out"][ok] == w.gamma + 1)
    np.testing.assert_array_equal(gv["out_tokens"][ok, : w.gamma], g["tokens"][ok])
    compare_verify(gv, ov, np.ones(w.R, bool), tag="q_eq_p")


def test_verify_many_requests_statistics():
    """Many requests of a small vocabulary: parity on each request, and the
    empirical first-position acceptance matches 1 - TV of the oracle's p and q."""
    w = synth.Workload("stats", R=512, gamma=3, V=64, r=4, T=1.0, w_dtype=F32, sigma_w=0.2,
                       sigma_pnoise=0.8)
    x = synth.gen_all(w)
    dr = oracle_draft(w, x, 8)
    g = gpu_verify_on(w, x, dr, 8)
    o = oracle_verify_on(w, x, dr, 8)
    compare_verify(g, o, np.ones(w.R, bool), tag="stats")
    # Position 1 is accepted with probability sum_v min(p_1(v), q_1(v)) = 1 - TV
    # (explainer section 05): p_1 = softmax(P_0 / T), q_1 = softmax((U_0 + e_1 W2) / T)
    # with e_1 the draft's first code.  The requests are independent, so the
    # count of accepted first positions has mean sum_r alpha_r and variance
    # sum_r alpha_r (1 - alpha_r): a z-test on the GPU's acceptances.
    from scipy.special import softmax
    z = (x["U"][:, 0, :].astype(np.float64) + dr["code"][:, 0, :] @ x["W2"].astype(np.float64)) / w.T
    q1 = softmax(z, axis=1)
    p1 = softmax(x["P"][:, 0, :].astype(np.float64) / w.T, axis=1)
    alpha = np.minimum(p1, q1).sum(axis=1)
    assert 0.2 < alpha.mean() < 0.95
    acc = (g["accept_len"] >= 1).sum()
    zscore = (acc - alpha.sum()) / np.sqrt((alpha * (1 - alpha)).sum())
    assert abs(zscore) < 4.0, (acc, alpha.sum(), zscore)


@pytest.mark.parametrize("R,gamma,rho", [(1, 1, 0.0), (3, 5, 0.5), (8, 4, 0.0), (5, 16, 0.5), (64, 5, 0.9),
                                         (512, 16, 0.9), (300, 7, 0.1)])
def test_schedule_parity(R, gamma, rho):
    rng = np.random.default_rng(R * 100 + gamma)
    for trial in range(4):
        c = (1 / (1 + np.exp(-rng.normal(1.5, 1.0, (R, gamma))))).astype(np.float32)
        if trial == 3:
            c[:, : max(1, gamma // 2)] = 1.0          # exact ties along requests
            c[0, 0] = 0.0                               # a zero candidate
        sps = synth.gen_sps(R, gamma, rho)
        if trial == 2:
            sps = sps[: R * (1 + gamma) // 2 + 1]       # table shorter than the batch
        out = binding.schedule(dev(c), dev(sps))
        torch.cuda.synchronize()
        L, th, n, gap = oracle.schedule_closed(c, sps)
        L2, th2, n2 = oracle.schedule_loop(c, sps)
        assert np.array_equal(L, L2) and n == n2
        if gap < 1e-12:
            continue                                     # flagged near-tie of Theta
        np.testing.assert_array_equal(host(out["verify_len"]), L)
        assert int(host(out["n_star"])[0]) == n
        np.testing.assert_allclose(host(out["theta"])[0], th, rtol=1e-12)


def test_schedule_toy_workload():
    w = synth.WORKLOADS["toy"]
    c = synth.gen_c(w)
    sps = synth.gen_sps(w.R, w.gamma, w.rho)
    out = binding.schedule(dev(c), dev(sps))
    L, th, n = oracle.schedule_loop(c, sps)
    np.testing.assert_array_equal(host(out["verify_len"]), L)
    assert 0 < n < w.R * w.gamma


def test_bad_anchor_sets_status_not_fault():
    w = SMALL["bf16_r64"]
    x = synth.gen_all(w)
    x["anchor"] = x["anchor"].copy()
    x["anchor"][2] = w.V + 5
    d = binding.draft_markov(dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"]), w.T, 3)
    torch.cuda.synchronize()
    assert binding.workspace_status(d["ws"]) == -6
    assert binding.workspace_status(d["ws"]) == 0          # cleared by the read


def test_bad_draft_token_in_verify_sets_status():
    w = SMALL["bf16_r64"]
    x = synth.gen_all(w)
    dr = oracle_draft(w, x, 1)
    dr["tokens"] = dr["tokens"].copy()
    dr["tokens"][0, 0] = -3
    qx = dr["qx"].astype(np.float32)
    draft = dict(tokens=dev(dr["tokens"]), q_tok=dev(qx), lse=dev(dr["lse"]), code=dev(dr["code"].astype(np.float32)))
    v = binding.verify(dev(x["P"]), dev(x["U"]), dev(x["W2"]), draft, w.T, 1)
    torch.cuda.synchronize()
    assert binding.workspace_status(v["ws"]) == -6


def test_host_argument_errors():
    w = SMALL["bf16_r64"]
    x = synth.gen_all(w)
    with pytest.raises(binding.DsparkError) as e:
        binding.draft_markov(dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"]), -1.0, 0)
    assert e.value.code == -1
    small_ws = torch.zeros(256, dtype=torch.uint8, device="cuda:0")
    with pytest.raises(binding.DsparkError) as e:
        binding.draft_markov(dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"]), 1.0, 0, ws=small_ws)
    assert e.value.code == -8


@pytest.mark.parametrize("R,gamma,rho", [(1, 1, 0.0), (5, 16, 0.5), (64, 5, 0.9), (300, 7, 0.1), (512, 16, 0.5)])
def test_schedule_async_parity(R, gamma, rho):
    """Production-style scheduler (explainer section 04): capacities of none,
    0, the step's own n*, a random value and more than the candidate count;
    lengths and the reported n* exact (unless the oracle's Theta comparison
    is a near-tie), theta within 1e-12."""
    rng = np.random.default_rng(R * 7 + gamma)
    c = (1 / (1 + np.exp(-rng.normal(1.5, 1.0, (R, gamma))))).astype(np.float32)
    c[0, min(1, gamma - 1)] = 0.0
    sps = synth.gen_sps(R, gamma, rho)
    _, _, n0, gap = oracle.schedule_closed(c, sps)
    if gap < 1e-12:
        pytest.skip("near-tie of Theta in this draw")
    for b in (-1, 0, n0, int(rng.integers(0, R * gamma + 1)), R * gamma + 5):
        bud = dev(np.array([b], np.int32))
        out = binding.schedule(dev(c), dev(sps), budget=bud)
        L, th, n, ns = oracle.schedule_budget(c, sps, b)
        np.testing.assert_array_equal(host(out["verify_len"]), L, err_msg=f"budget {b}")
        assert int(host(out["n_star"])[0]) == ns == n0
        np.testing.assert_allclose(host(out["theta"])[0], th, rtol=1e-12)


def test_schedule_async_two_steps_back_ring():
    """Six steps with three n_star buffers in rotation: step t takes the
    n_star of step t - 2 as its capacity (none for the first two), all on the
    device, against the oracle following the same protocol."""
    R, gamma, rho = 64, 5, 0.3
    rng = np.random.default_rng(11)
    ring = [dev(np.array([-1], np.int32)) for _ in range(3)]
    hist = []
    for t in range(6):
        c = (1 / (1 + np.exp(-rng.normal(1.0 + 0.2 * t, 1.2, (R, gamma))))).astype(np.float32)
        sps = synth.gen_sps(R, gamma, rho)
        budget = ring[(t - 2) % 3] if t >= 2 else dev(np.array([-1], np.int32))
        out = dict(verify_len=torch.empty((R,), dtype=torch.int32, device="cuda:0"),
                   theta=torch.empty((1,), dtype=torch.float64, device="cuda:0"), n_star=ring[t % 3])
        binding.schedule(dev(c), dev(sps), budget=budget, out=out)
        b = hist[t - 2] if t >= 2 else -1
        L, th, n, ns = oracle.schedule_budget(c, sps, b)
        hist.append(ns)
        np.testing.assert_array_equal(host(out["verify_len"]), L, err_msg=f"step {t}")
        assert int(host(ring[t % 3])[0]) == ns


def test_verify_reads_host_resident_targets_in_place():
    """P in pinned host memory, read in place through dspark_host_pointer:
    every output equal to the run with P on the device."""
    w = synth.Workload("zc", R=6, gamma=4, V=20488, r=64, T=1.0)
    x = synth.gen_all(w)
    dr = oracle_draft(w, x, 21)
    draft = dict(tokens=dev(dr["tokens"].astype(np.int32)), q_tok=dev(dr["qx"].astype(np.float32)),
                 lse=dev(dr["lse"].astype(np.float64)), code=dev(dr["code"].astype(np.float32)))
    hP = torch.from_numpy(np.ascontiguousarray(x["P"])).pin_memory()
    Pv = binding.host_view(hP, torch.device("cuda:0"))
    a = binding.verify(dev(x["P"]), dev(x["U"]), dev(x["W2"]), draft, w.T, 21)
    b = binding.verify(Pv, dev(x["U"]), dev(x["W2"]), draft, w.T, 21)
    torch.cuda.synchronize()
    for k in ("out_tokens", "accept_len", "n_out", "p_tok", "lse_p"):
        np.testing.assert_array_equal(host(a[k]), host(b[k]), err_msg=k)


@pytest.mark.parametrize("gamma,T,V,pdt", [(4, 1.0, 20488, synth.F32), (16, 0.0, 8200, synth.F32),
                                            (64, 1.0, 4104, synth.F32), (5, 0.8, 8200, synth.BF16)])
def test_verify_staged_host_targets(gamma, T, V, pdt):
    """P read in place from pinned host memory with a device staging buffer
    (one target row per wave, up to gamma + 1 waves): tokens and lengths
    equal to the run with P on the device, p_tok / lse_p equal where the
    decision read them and NaN elsewhere, and the staged rows equal to P
    where verification read them."""
    w = synth.Workload("zcs", R=6, gamma=gamma, V=V, r=64, T=T, p_dtype=pdt)
    x = synth.gen_all(w)
    dr = oracle_draft(w, x, 23)
    draft = dict(tokens=dev(dr["tokens"].astype(np.int32)), q_tok=dev(dr["qx"].astype(np.float32)),
                 lse=dev(dr["lse"].astype(np.float64)), code=dev(dr["code"].astype(np.float32)))
    hP = torch.from_numpy(np.ascontiguousarray(x["P"])).pin_memory()
    if x["P"].dtype == np.uint16:
        hP = hP.view(torch.bfloat16)
    Pv = binding.host_view(hP, torch.device("cuda:0"))
    stage = torch.full(hP.shape, float("nan"), dtype=hP.dtype, device="cuda:0")
    a = binding.verify(dev(x["P"]), dev(x["U"]), dev(x["W2"]), draft, w.T, 23)
    b = binding.verify(Pv, dev(x["U"]), dev(x["W2"]), draft, w.T, 23, p_stage=stage)
    torch.cuda.synchronize()
    for k in ("out_tokens", "accept_len", "n_out"):
        np.testing.assert_array_equal(host(a[k]), host(b[k]), err_msg=k)
    # one row per wave: exactly the rows and positions the decision used
    acc = host(b["accept_len"])
    for r in range(w.R):
        d = int(acc[r])
        np.testing.assert_array_equal(host(b["lse_p"])[r, :d + 1], host(a["lse_p"])[r, :d + 1])
        assert np.isnan(host(b["lse_p"])[r, d + 1:]).all()
        npos = min(d + 1, w.gamma)
        np.testing.assert_array_equal(host(b["p_tok"])[r, :npos], host(a["p_tok"])[r, :npos])
        assert np.isnan(host(b["p_tok"])[r, npos:]).all()
    st = host(stage)
    for r in range(w.R):
        d = int(host(b["accept_len"])[r])
        np.testing.assert_array_equal(st[r, d], x["P"][r, d])     # the decision row was staged


MASKED = {
    "f32_tc": synth.Workload("masked_f32_tc", R=6, gamma=4, V=20488, r=64, T=1.0),
    "bf16_storage_T08": synth.Workload("masked_bf16_T08", R=5, gamma=3, V=12296, r=128, T=0.8,
                                       u_dtype=BF16, p_dtype=BF16, sigma_pnoise=1.2),
    "greedy": synth.Workload("masked_greedy", R=5, gamma=4, V=16392, r=64, T=0.0, sigma_u=2.0, sigma_pnoise=0.7),
    "f32_generic": synth.Workload("masked_f32_r7", R=3, gamma=2, V=5124, r=7, T=1.3, w_dtype=F32, sigma_w=0.3),
}


def _mask(a: np.ndarray, cols: np.ndarray):
    """Set columns `cols` of every row of a (f32 or bf16 bits) to -inf."""
    a[..., cols] = np.uint16(0xFF80) if a.dtype == np.uint16 else np.float32(-np.inf)


@pytest.mark.parametrize("name", list(MASKED))
def test_masked_vocabulary_parity(name):
    """Masked columns (logits of -inf) carry no mass on either side: closed to
    both the draft and the target (one whole 2048-column block, which covers
    two of the target pass's 1024-column chunks and eight of the draft's
    256-column chunks, and a random fifth of the rest), or open to the draft
    and closed to the target, so that such drafts are rejected with p = 0.
    Draft and verification must match the oracle, no column closed to the
    draft may be drafted, and no token may be emitted from a target row that
    closes it."""
    w = MASKED[name]
    x = synth.gen_all(w)
    rng = np.random.default_rng(11)
    both = np.concatenate([np.arange(2048, 4096), rng.choice(np.arange(4096, w.V), (w.V - 4096) // 5, replace=False)])
    open_cols = np.setdiff1d(np.arange(w.V), both)
    p_only = rng.choice(open_cols, w.V // 20, replace=False)
    _mask(x["U"], both)
    _mask(x["P"], both)
    _mask(x["P"], p_only)
    seed = 31
    g = gpu_draft(w, x, seed)
    o = oracle_draft(w, x, seed)
    _, _, m = compare_draft(g, o, tag=name)
    assert not np.isin(g["tokens"], both).any()
    same = (g["tokens"] == o["tokens"]).all(axis=1)
    gv = gpu_verify_on(w, x, g, seed)
    ov = oracle_verify_on(w, x, o, seed)
    compare_verify(gv, ov, same, tag=name)
    # verification of the oracle's drafts, some of them closed to the target:
    # request i (even) finds its draft at position 1 + i // 2 closed in P
    dr = oracle_draft(w, x, 5)
    for i in range(0, w.R, 2):
        k = min(i // 2, w.gamma - 1)
        t = int(dr["tokens"][i, k])
        if x["P"].dtype == np.uint16:
            x["P"][i, k, t] = np.uint16(0xFF80)
        else:
            x["P"][i, k, t] = np.float32(-np.inf)
    gv = gpu_verify_on(w, x, dr, 5)
    ov = oracle_verify_on(w, x, dr, 5)
    n, nflag = compare_verify(gv, ov, np.ones(w.R, bool), tag=name)
    assert n + nflag == w.R
    if w.T > 0:
        # a draft the target has closed is rejected with p(x) = 0 (request 0:
        # position 1 is the one closed)
        assert ov["accept_len"][0] == 0 and gv["accept_len"][0] == 0 and gv["p_tok"][0, 0] == 0.0
    # every emitted token (accepted draft, residual draw, bonus) is open in
    # the target row it was decided on: output slot j comes from row j
    Pf = synth.bf16_bits_to_f32(x["P"]) if x["P"].dtype == np.uint16 else x["P"]
    for i in range(w.R):
        for j in range(int(gv["n_out"][i])):
            t = int(gv["out_tokens"][i, j])
            assert np.isfinite(Pf[i, j, t]), f"{name}: request {i} emitted column {t}, closed in target row {j}"
