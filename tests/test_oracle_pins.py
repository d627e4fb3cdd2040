"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against a value printed on the pages, a closed
form, a library routine, or an exact enumeration -- never against a retyped
copy of the oracle's own formula.
"""
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle
from conftest import GOLDEN, read_golden
from speculative_decoding_drafting_gb300 import synth


# ------------------------------------------------------------------ Philox
def test_philox_known_answers():
    """Salmon et al. SC'11 / Random123 known-answer vectors."""
    n = 0
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            h = [int(t, 16) for t in line.split()]
            out = oracle.philox4x32_10(h[0:4], h[4:6])
            assert [int(x) for x in out] == h[6:10]
            n += 1
    assert n == 3


def test_uniform_range_and_resolution():
    """u = (w + 1/2) 2^-32: strictly inside (0, 1), symmetric, exact in double."""
    lo = oracle.uniform(0)
    hi = oracle.uniform(0xFFFFFFFF)
    assert lo == 2.0 ** -33 and hi == 1.0 - 2.0 ** -33
    rng = np.random.default_rng(1)
    for w in rng.integers(0, 2 ** 32, size=2000, dtype=np.uint64):
        u = oracle.uniform(int(w))
        assert 0.0 < u < 1.0
        assert u + oracle.uniform(int(w) ^ 0xFFFFFFFF) == 1.0      # 1 - u is the complement word


def test_rng_stream_layout():
    """Index v uses counter (v/4, req, pos, stream), word v mod 4."""
    seed = (7 << 32) | 11
    words = oracle.philox4x32_10([5, 3, 2, 0], [11, 7])
    for i in range(4):
        assert oracle.rng_uniform(seed, 3, 2, 0, 20 + i) == oracle.uniform(int(words[i]))


def test_rng_uniformity():
    us = np.array([oracle.rng_uniform(123, r, 1, 0, v) for r in range(8) for v in range(2048)])
    assert stats.kstest(us, "uniform").pvalue > 1e-3


# ------------------------------------------------------------------ section 05 toy
def test_toy_rejection_worked_example():
    g = read_golden("toy_rejection.txt")
    q = np.array(g["q"][0], float)
    p = np.array(g["p"][0], float)
    acc = np.array([qx * oracle.accept_prob(px, qx) for px, qx in zip(p, q)])
    np.testing.assert_allclose(acc, np.array(g["accepted"][0], float), atol=1e-15)
    assert abs(acc.sum() - float(g["accept_total"][0][0])) < 1e-15
    w = oracle.residual_weights(p, q)
    np.testing.assert_allclose(w / w.sum(), np.array(g["residual"][0], float), atol=1e-15)
    law = acc + (1.0 - acc.sum()) * w / w.sum()
    np.testing.assert_allclose(law, p, atol=1e-15)


@pytest.mark.parametrize("V", [2, 3, 4])
def test_enumerated_law_equals_target(V):
    """Exact enumeration over the draft token: P(emit v) = p(v) for random p, q."""
    rng = np.random.default_rng(V)
    for _ in range(200):
        p = rng.dirichlet(np.ones(V) * 0.7)
        q = rng.dirichlet(np.ones(V) * 0.7)
        alpha = np.array([oracle.accept_prob(p[x], q[x]) for x in range(V)])
        w = oracle.residual_weights(p, q)
        rej = 1.0 - float(np.sum(q * alpha))
        law = q * alpha + (rej * w / w.sum() if w.sum() > 0 else 0.0)
        np.testing.assert_allclose(law, p, atol=1e-12)
        # single-step acceptance equals 1 - TV (blog section 4.1)
        assert abs(np.sum(q * alpha) - (1.0 - 0.5 * np.abs(p - q).sum())) < 1e-12


def _one_position_verify(logp, logq, n_req, seed):
    """Full oracle verify of one drafted position with U = log q, W2 = 0, P = log p."""
    V = len(logp)
    R, gamma, r = n_req, 1, 1
    U = np.broadcast_to(np.asarray(logq, np.float32), (R, gamma, V)).copy()
    P = np.broadcast_to(np.asarray(logp, np.float32), (R, gamma + 1, V)).copy()
    W1 = np.zeros((V, r), np.float32)
    W2 = np.zeros((r, V), np.float32)
    anchor = np.zeros(R, np.int32)
    d = oracle.draft_markov(U, anchor, W1, W2, 1.0, seed)
    v = oracle.verify(P, U, W2, d["tokens"], d["qx"], d["lse"], d["code"], 1.0, seed)
    return d, v


def test_toy_monte_carlo_output_law_and_acceptance():
    """Emitted tokens follow p and acceptance is 0.80 for the section 05 toy."""
    g = read_golden("toy_rejection.txt")
    q = np.array(g["q"][0], float)
    p = np.array(g["p"][0], float)
    n = 200_000
    d, v = _one_position_verify(np.log(p), np.log(q), n, seed=2024)
    # draft samples follow q (Gumbel-max)
    cnt_q = np.bincount(d["tokens"][:, 0], minlength=3)
    assert stats.chisquare(cnt_q, n * q / q.sum()).pvalue > 1e-3
    acc = v["accept_len"] == 1
    rate = acc.mean()
    se = math.sqrt(0.8 * 0.2 / n)
    assert abs(rate - 0.8) < 5 * se
    first = v["out_tokens"][:, 0]
    cnt_p = np.bincount(first, minlength=3)
    assert stats.chisquare(cnt_p, n * p).pvalue > 1e-3
    # every request advances at least one token
    assert np.all(v["n_out"] >= 1)


def test_masked_columns_have_no_mass():
    """Logits of -inf (masked columns) carry no probability: the draft follows
    softmax over the open columns (a whole chunk masked included), the
    verification emits the target's law over its open columns, and a draft
    the target has masked is always rejected."""
    rng = np.random.default_rng(23)
    V, n = 700, 200_000
    u = rng.normal(0, 1.0, V)
    p = u + rng.normal(0, 0.7, V)
    u[256:512] = -np.inf                                  # one whole chunk closed to both
    u[rng.choice(V, 120, replace=False)] = -np.inf
    p[np.isinf(u)] = -np.inf
    closed_p = rng.choice(np.nonzero(np.isfinite(u))[0], 40, replace=False)
    p[closed_p] = -np.inf                                 # open to the draft, closed to the target
    u = u.astype(np.float32).astype(np.float64)           # the values as stored
    p = p.astype(np.float32).astype(np.float64)
    U = np.broadcast_to(u.astype(np.float32), (n, 1, V)).copy()
    P = np.broadcast_to(np.stack([p, p]).astype(np.float32), (n, 2, V)).copy()
    W1 = np.zeros((V, 1), np.float32)
    W2 = np.zeros((1, V), np.float32)
    d = oracle.draft_markov(U, np.zeros(n, np.int32), W1, W2, 1.0, 123)
    q = special.softmax(u)
    assert np.all(np.isfinite(u[d["tokens"][:, 0]]))
    open_u = np.isfinite(u)
    cnt = np.bincount(d["tokens"][:, 0], minlength=V)[open_u]
    assert stats.chisquare(cnt, n * q[open_u]).pvalue > 1e-3
    np.testing.assert_allclose(d["lse"][:, 0], special.logsumexp(u), rtol=1e-13)
    v = oracle.verify(P, U, W2, d["tokens"], d["qx"], d["lse"], d["code"], 1.0, 123)
    first = v["out_tokens"][:, 0]
    assert np.all(np.isfinite(p[first]))
    drafted_closed = np.isin(d["tokens"][:, 0], closed_p)
    assert drafted_closed.any() and np.all(v["accept_len"][drafted_closed] == 0)
    np.testing.assert_array_equal(v["px"][drafted_closed, 0], 0.0)
    pt = special.softmax(p)
    open_p = np.isfinite(p)
    assert stats.chisquare(np.bincount(first, minlength=V)[open_p], n * pt[open_p]).pvalue > 1e-3


def test_q_equals_p_accepts_everything():
    """Explainer section 05: if q = p nothing is ever rejected."""
    rng = np.random.default_rng(5)
    R, gamma, V, r = 64, 4, 50, 3
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    P = np.concatenate([U, U[:, -1:, :]], axis=1)
    W1 = rng.normal(0, 0.1, (V, r)).astype(np.float32)
    W2 = np.zeros((r, V), np.float32)
    d = oracle.draft_markov(U, rng.integers(0, V, R), W1, W2, 1.0, 9)
    v = oracle.verify(P, U, W2, d["tokens"], d["qx"], d["lse"], d["code"], 1.0, 9)
    assert np.all(v["accept_len"] == gamma)
    assert np.all(v["n_out"] == gamma + 1)
    np.testing.assert_array_equal(v["out_tokens"][:, :gamma], d["tokens"])


# ------------------------------------------------------------------ drafting
def test_markov_ln9_bias_gives_nine_to_one():
    g = read_golden("markov_bias.txt")
    qexp = np.array(g["q"][0], float)
    R, V, r = 100_000, 2, 1
    U = np.zeros((R, 1, V), np.float32)
    W1 = np.ones((V, r), np.float32)
    W2 = np.array([[math.log(9.0), 0.0]], np.float32)
    d = oracle.draft_markov(U, np.zeros(R, np.int32), W1, W2, 1.0, 77)
    np.testing.assert_allclose(d["lse"], math.log(10.0), rtol=1e-7)
    x = d["tokens"][:, 0]
    np.testing.assert_allclose(d["qx"][:, 0], qexp[x], rtol=1e-7)
    frac = np.mean(x == 0)
    assert abs(frac - 0.9) < 5 * math.sqrt(0.09 / R)


def test_zero_W2_reduces_to_independent_softmax():
    """W2 = 0: the draft is the pure parallel drafter, q_k = softmax(U_k / T)."""
    rng = np.random.default_rng(3)
    R, gamma, V, r, T = 6, 3, 300, 8, 0.7
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.1, (V, r)).astype(np.float32)
    W2 = np.zeros((r, V), np.float32)
    d = oracle.draft_markov(U, rng.integers(0, V, R), W1, W2, T, 4)
    z = U.astype(np.float64) / T
    np.testing.assert_allclose(d["lse"], special.logsumexp(z, axis=2), rtol=1e-13)
    sm = special.softmax(z, axis=2)
    qx = np.take_along_axis(sm, d["tokens"][:, :, None], axis=2)[:, :, 0]
    np.testing.assert_allclose(d["qx"], qx, rtol=1e-12)


def test_two_level_gumbel_draft_law_over_many_chunks():
    """The draft's chunk-then-element Gumbel-max samples softmax(z) exactly:
    chi-square of many independent draws (request ids) over a 5-chunk
    vocabulary against the library softmax."""
    rng = np.random.default_rng(17)
    V, n = 1100, 200_000
    logits = rng.normal(0, 1.0, V).astype(np.float32)
    logits[256:512] += 1.5                       # one heavy chunk
    U = np.broadcast_to(logits, (n, 1, V)).copy()
    W1 = np.zeros((V, 1), np.float32)
    W2 = np.zeros((1, V), np.float32)
    d = oracle.draft_markov(U, np.zeros(n, np.int32), W1, W2, 1.0, 31)
    probs = special.softmax(logits.astype(np.float64))
    cnt = np.bincount(d["tokens"][:, 0], minlength=V).astype(float)
    # pool rare cells so every expected count is at least 5
    order = np.argsort(probs)
    exp_c, obs_c, acc_e, acc_o = [], [], 0.0, 0.0
    for i in order:
        acc_e += n * probs[i]
        acc_o += cnt[i]
        if acc_e >= 5:
            exp_c.append(acc_e)
            obs_c.append(acc_o)
            acc_e = acc_o = 0.0
    exp_c[-1] += acc_e
    obs_c[-1] += acc_o
    assert stats.chisquare(obs_c, exp_c).pvalue > 1e-3
    # chunk frequencies match the chunk masses
    chunk = d["tokens"][:, 0] // 256
    cm = np.array([probs[c * 256:(c + 1) * 256].sum() for c in range(5)])
    assert stats.chisquare(np.bincount(chunk, minlength=5), n * cm).pvalue > 1e-3


def test_single_chunk_draft_is_textbook_gumbel_max():
    """With V <= 256 there is one chunk, so its race is decided and the draft
    is the plain Gumbel-max over the whole vocabulary: x_k = argmax_v z_v + G_v,
    G_v = -ln(-ln u_v), u_v the stream-0 uniform of (request, position k, v),
    z = (U_k + W1[x_{k-1}] W2) / T.  Checked token by token, through an
    independent matmul and the known-answer-pinned generator, with request ids
    that are not the row numbers."""
    rng = np.random.default_rng(41)
    R, gamma, V, r, T, seed = 6, 3, 200, 5, 0.8, (9 << 32) | 1234
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.4, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.4, (r, V)).astype(np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    req = (1000 + 37 * np.arange(R)).astype(np.uint32)
    d = oracle.draft_markov(U, anchor, W1, W2, T, seed, req_ids=req)
    prev = np.concatenate([anchor[:, None], d["tokens"][:, :-1]], axis=1)
    z = (U + np.einsum("rki,iv->rkv", W1.astype(np.float64)[prev], W2.astype(np.float64))) / T
    for i in range(R):
        for k in range(1, gamma + 1):
            u = np.array([oracle.rng_uniform(seed, int(req[i]), k, 0, v) for v in range(V)])
            key = z[i, k - 1] - np.log(-np.log(u))
            assert d["tokens"][i, k - 1] == int(np.argmax(key))
    np.testing.assert_allclose(d["lse"], special.logsumexp(z, axis=2), rtol=1e-12)


def test_two_level_gumbel_draft_never_leaves_the_only_live_chunk():
    V, R = 1024, 64
    U = np.full((R, 2, V), -1.0e4, np.float32)
    U[:, :, 512:768] = np.random.default_rng(3).normal(0, 1, (R, 2, 256))
    W1 = np.zeros((V, 1), np.float32)
    W2 = np.zeros((1, V), np.float32)
    d = oracle.draft_markov(U, np.zeros(R, np.int32), W1, W2, 1.0, 5)
    assert np.all((d["tokens"] >= 512) & (d["tokens"] < 768))


def test_markov_code_is_embedding_of_previous_token():
    rng = np.random.default_rng(8)
    R, gamma, V, r = 5, 4, 64, 6
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    W1 = synth.f32_to_bf16_bits(rng.normal(0, 0.3, (V, r)).astype(np.float32))
    W2 = synth.f32_to_bf16_bits(rng.normal(0, 0.3, (r, V)).astype(np.float32))
    anchor = rng.integers(0, V, R).astype(np.int32)
    d = oracle.draft_markov(U, anchor, W1, W2, 1.0, 6)
    W1f = synth.bf16_bits_to_f32(W1).astype(np.float64)
    prev = np.concatenate([anchor[:, None], d["tokens"][:, :-1]], axis=1)
    np.testing.assert_array_equal(d["code"], W1f[prev])
    # logits of the sampled token through an independent matmul
    W2f = synth.bf16_bits_to_f32(W2).astype(np.float64)
    z = U + np.einsum("rki,iv->rkv", d["code"], W2f)
    np.testing.assert_allclose(d["lse"], special.logsumexp(z, axis=2), rtol=1e-12)


def test_greedy_draft_is_argmax():
    rng = np.random.default_rng(12)
    R, gamma, V, r = 7, 3, 97, 4
    U = rng.normal(0, 2.0, (R, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.5, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.5, (r, V)).astype(np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    d = oracle.draft_markov(U, anchor, W1, W2, 0.0, 0)
    prev = np.concatenate([anchor[:, None], d["tokens"][:, :-1]], axis=1)
    y = U + np.einsum("rki,iv->rkv", W1.astype(np.float64)[prev], W2.astype(np.float64))
    np.testing.assert_array_equal(d["tokens"], np.argmax(y, axis=2))


def test_rnn_zero_weights_match_markov_zero_bias():
    rng = np.random.default_rng(21)
    R, gamma, V, r, dd = 4, 3, 80, 4, 5
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.1, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.1, (r, V)).astype(np.float32)
    H = rng.normal(0, 1, (R, gamma, dd)).astype(np.float32)
    Wgco = np.zeros((2 * r + dd, 3 * r), np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    a = oracle.draft_rnn(U, anchor, W1, W2, Wgco, H, 1.0, 31)
    b = oracle.draft_markov(U, anchor, W1, np.zeros_like(W2), 1.0, 31)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=1e-14)
    assert np.all(a["code"] == 0.0) and np.all(a["state"] == 0.0)


def test_rnn_hand_computed_two_steps():
    """r = 1, d = 1, h = 0, W1 = 1.  Gate/cand/out pre-activations chosen so
    that tanh and sigmoid take closed-form values:
      step 1: z = [0, 1, 0] -> gate 0 (g = 1/2), cand atanh(1/2), out atanh(1/4)
              s1 = 1/2 * 0 + 1/2 * 1/2 = 1/4,  e1 = 1/4
      step 2: z = [1/4, 1, 0] -> gate (1/4)(4 ln 3) = ln 3 (g = 3/4)
              s2 = 3/4 * 1/4 + 1/4 * 1/2 = 5/16,  e2 = 1/4
    """
    a = 0.5 * math.log(3.0)          # tanh(a) = 1/2
    b = 0.5 * math.log(5.0 / 3.0)    # tanh(b) = 1/4
    Wgco = np.array([[4 * math.log(3.0), 0.0, 0.0],    # s input
                     [0.0, a, b],                      # W1[x] input
                     [0.0, 0.0, 0.0]], np.float64)     # h input
    R, gamma, V, r, dd = 1, 2, 3, 1, 1
    U = np.zeros((R, gamma, V), np.float32)
    W1 = np.ones((V, r), np.float32)
    W2 = np.zeros((r, V), np.float32)
    H = np.zeros((R, gamma, dd), np.float32)
    out = oracle.draft_rnn(U, np.zeros(R, np.int32), W1, W2, Wgco.astype(np.float32), H, 1.0, 1)
    np.testing.assert_allclose(out["code"][0, :, 0], [0.25, 0.25], atol=2e-7)
    np.testing.assert_allclose(out["state"][0, 0], 5.0 / 16.0, atol=2e-7)


# ------------------------------------------------------------------ verification
def test_greedy_verify_worked_example():
    """Explainer section 02 (greedy teaching version): the first mismatch is
    replaced by the target's token and the rest is discarded; a fully
    matching block gets a bonus token."""
    V, gamma, r = 8, 3, 1
    P = np.zeros((2, gamma + 1, V), np.float32)
    am = [[3, 5, 2, 6], [3, 5, 7, 1]]
    for i in range(2):
        for k in range(gamma + 1):
            P[i, k, am[i][k]] = 1.0
    tokens = np.array([[3, 5, 7], [3, 5, 7]], np.int32)
    U = np.zeros((2, gamma, V), np.float32)
    W2 = np.zeros((r, V), np.float32)
    v = oracle.verify(P, U, W2, tokens, np.ones((2, gamma)), np.zeros((2, gamma)),
                      np.zeros((2, gamma, r)), 0.0, 0)
    np.testing.assert_array_equal(v["out_tokens"][0], [3, 5, 2, -1])
    np.testing.assert_array_equal(v["out_tokens"][1], [3, 5, 7, 1])
    np.testing.assert_array_equal(v["accept_len"], [2, 3])
    np.testing.assert_array_equal(v["n_out"], [3, 4])


def test_verify_len_zero_draws_from_first_target_row():
    rng = np.random.default_rng(2)
    V = 6
    p = rng.dirichlet(np.ones(V))
    n = 100_000
    R, gamma, r = n, 2, 1
    P = np.broadcast_to(np.log(p).astype(np.float32), (R, gamma + 1, V)).copy()
    P[:, 1:, :] = 0.0
    U = np.zeros((R, gamma, V), np.float32)
    W2 = np.zeros((r, V), np.float32)
    v = oracle.verify(P, U, W2, np.zeros((R, gamma), np.int32), np.full((R, gamma), 1.0 / V),
                      np.full((R, gamma), math.log(V)), np.zeros((R, gamma, r)), 1.0, 3,
                      verify_len=np.zeros(R, np.int32))
    assert np.all(v["accept_len"] == 0) and np.all(v["n_out"] == 1)
    cnt = np.bincount(v["out_tokens"][:, 0], minlength=V)
    assert stats.chisquare(cnt, n * p / p.sum()).pvalue > 1e-3


def test_acceptance_rate_is_one_minus_tv():
    rng = np.random.default_rng(44)
    V = 12
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    n = 200_000
    d, v = _one_position_verify(np.log(p), np.log(q), n, seed=99)
    p32 = special.softmax(np.log(p).astype(np.float32).astype(np.float64))
    q32 = special.softmax(np.log(q).astype(np.float32).astype(np.float64))
    expect = 1.0 - 0.5 * np.abs(p32 - q32).sum()
    rate = np.mean(v["accept_len"] == 1)
    assert abs(rate - expect) < 5 * math.sqrt(expect * (1 - expect) / n)
    cnt = np.bincount(v["out_tokens"][:, 0], minlength=V)
    assert stats.chisquare(cnt, n * p32).pvalue > 1e-3


# ------------------------------------------------------------------ tree sampler
def _residual_pin_case():
    """Position 1 is forced to accept (P_0 = U_0 + e_1 W2, so p_1 = q_1), W2 is
    far from zero and T = 0.7, so the residual at position 2 needs q_2 rebuilt
    from the second code row, the second lse and (U + B) / T together."""
    V, r, T = 6, 3, 0.7
    rng = np.random.default_rng(13)
    W1 = rng.normal(0.0, 1.0, (V, r)).astype(np.float32)
    W2 = rng.normal(0.0, 1.0, (r, V)).astype(np.float32)
    anchor = 0
    U = rng.normal(0.0, 1.0, (2, V)).astype(np.float32)
    P = np.empty((3, V), np.float32)
    P[0] = (U[0].astype(np.float64) + W1[anchor].astype(np.float64) @ W2.astype(np.float64)).astype(np.float32)
    P[1] = rng.normal(0.0, 1.5, V).astype(np.float32)
    P[2] = rng.normal(0.0, 1.5, V).astype(np.float32)
    return V, r, T, W1, W2, anchor, U, P


def _position2_law(V, T, W1, W2, anchor, U, P, rebuild):
    """Law of the token emitted at position 2 when position 1 is accepted,
    by exact enumeration over x_1 ~ q_1 (= p_1) and x_2 ~ q_2(. | x_1), with
    the residual formed from rebuild(x_1) in place of q_2."""
    f64 = lambda a: a.astype(np.float64)  # noqa: E731
    q1 = special.softmax((f64(U[0]) + f64(W1[anchor]) @ f64(W2)) / T)
    p2 = special.softmax(f64(P[1]) / T)
    law = np.zeros(V)
    for x1 in range(V):
        q2 = special.softmax((f64(U[1]) + f64(W1[x1]) @ f64(W2)) / T)
        acc = np.minimum(p2, q2)
        w = np.maximum(p2 - rebuild(x1, q2), 0.0)
        law += q1[x1] * (acc + (1.0 - acc.sum()) * w / w.sum())
    return law, p2


def test_residual_rebuild_gives_the_target_law_at_position_two():
    """Explainer section 05: after a rejection at position j the token comes
    from r(v) = max(p_j - q_j, 0) / Z, with q_j rebuilt from the Markov code
    e_j = W1[x_{j-1}] (blog section 3.2): q_j(v) = exp((U_j + e_j W2)[v] / T - lse_j).
    Exact enumeration gives the target law p_2 = softmax(P_1 / T) for the
    emitted token; the oracle, run on 10^5 request ids, must reproduce it
    (chi-square).  The three plausible slips -- the previous code row, the
    previous position's lse, T dividing U alone -- each move the law far
    enough that the chi-square at this sample size would reject them."""
    V, r, T, W1, W2, anchor, U, P = _residual_pin_case()
    f64 = lambda a: a.astype(np.float64)  # noqa: E731
    law, p2 = _position2_law(V, T, W1, W2, anchor, U, P, lambda x1, q2: q2)
    np.testing.assert_allclose(law, p2, rtol=0, atol=1e-12)

    # the oracle on N independent request ids with identical inputs
    N, seed = 100_000, 424242
    Ur = np.broadcast_to(U, (N, 2, V)).copy()
    Pr = np.broadcast_to(P, (N, 3, V)).copy()
    ids = np.arange(N, dtype=np.uint32)
    d = oracle.draft_markov(Ur, np.full(N, anchor, np.int32), W1, W2, T, seed, req_ids=ids)
    o = oracle.verify(Pr, Ur, W2, d["tokens"], d["qx"], d["lse"], d["code"], T, seed, req_ids=ids)
    reached = o["accept_len"] >= 1
    assert reached.mean() > 0.999                      # p_1 = q_1: position 1 accepted
    rej2 = (o["accept_len"] == 1).mean()
    assert 0.2 < rej2 < 0.9                            # the residual path is taken often (about 0.31)
    counts = np.bincount(o["out_tokens"][reached, 1], minlength=V)
    n = int(reached.sum())
    assert stats.chisquare(counts, n * p2).pvalue > 1e-3

    # power against the slips: the law each would produce, as a chi-square
    # noncentrality at this n (a value of 100 rejects at 1e-3 almost surely)
    lse1 = special.logsumexp((f64(U[0]) + f64(W1[anchor]) @ f64(W2)) / T)
    slips = {
        "previous code row": lambda x1, q2: np.exp(
            (f64(U[1]) + f64(W1[anchor]) @ f64(W2)) / T
            - special.logsumexp((f64(U[1]) + f64(W1[x1]) @ f64(W2)) / T)),
        "previous lse": lambda x1, q2: np.exp((f64(U[1]) + f64(W1[x1]) @ f64(W2)) / T - lse1),
        "T on U alone": lambda x1, q2: np.exp(
            f64(U[1]) / T + f64(W1[x1]) @ f64(W2)
            - special.logsumexp((f64(U[1]) + f64(W1[x1]) @ f64(W2)) / T)),
    }
    for name, reb in slips.items():
        bad, _ = _position2_law(V, T, W1, W2, anchor, U, P, reb)
        lam = n * float(((bad - p2) ** 2 / p2).sum())
        assert lam > 100.0, (name, lam)


def test_tree_sampler_one_hot_and_half_masses():
    for V in (1, 2, 5, 16, 1000):
        for hot in {0, V // 2, V - 1}:
            w = np.zeros(V)
            w[hot] = 0.3
            for req in range(5):
                assert oracle.tree_sample(w, 1, req, 1)[0] == hot


def test_tree_sampler_law():
    rng = np.random.default_rng(10)
    V = 11
    w = rng.random(V)
    w[3] = 0.0
    n = 60_000
    cnt = np.zeros(V)
    for req in range(n):
        cnt[oracle.tree_sample(w, 555, req, 2)[0]] += 1
    assert cnt[3] == 0
    mask = w > 0
    assert stats.chisquare(cnt[mask], n * w[mask] / w.sum()).pvalue > 1e-3


# ------------------------------------------------------------------ scheduler
def test_prefix_survival_worked_value():
    g = read_golden("prefix_survival.txt")
    c = np.array([g["c"][0]], np.float32)
    a = oracle.prefix_survival(c)
    np.testing.assert_allclose(a[0], np.array(g["a"][0], float), rtol=1e-6)
    tau = 1.0 + float(a[0].astype(np.float64).sum())
    assert abs(tau - float(g["tau"][0][0])) < 1e-6


def _brute_force(a, sps, R, gamma):
    """Maximum tau for every total budget n, over all allocations."""
    best_tau = {}
    best_theta = -1.0
    for alloc in np.ndindex(*([gamma + 1] * R)):
        n = sum(alloc)
        tau = R + sum(float(a[i, :alloc[i]].astype(np.float64).sum()) for i in range(R))
        best_tau[n] = max(best_tau.get(n, -1.0), tau)
        B = R + n
        th = tau * (sps[B] if B < len(sps) else 0.0)
        best_theta = max(best_theta, th)
    return best_tau, best_theta


@pytest.mark.parametrize("rho", [0.0, 0.5, 0.9])
def test_scheduler_greedy_is_optimal_for_every_budget(rho):
    rng = np.random.default_rng(int(rho * 10) + 1)
    for trial in range(12):
        R = int(rng.integers(1, 5))
        gamma = int(rng.integers(1, 5))
        c = (1.0 / (1.0 + np.exp(-rng.normal(1.5, 1.0, (R, gamma))))).astype(np.float32)
        sps = synth.gen_sps(R, gamma, rho)
        a = oracle.prefix_survival(c)
        L1, th1, n1 = oracle.schedule_loop(c, sps)
        L2, th2, n2, _ = oracle.schedule_closed(c, sps)
        np.testing.assert_array_equal(L1, L2)
        assert th1 == th2 and n1 == n2 == int(L1.sum())
        bt, btheta = _brute_force(a, sps, R, gamma)
        # greedy tau at its budget is the best tau with that budget
        tau_g = R + sum(float(a[i, :L1[i]].astype(np.float64).sum()) for i in range(R))
        assert abs(tau_g - bt[n1]) < 1e-12
        # Theta along the greedy order: if unimodal, greedy attains the optimum
        srt = np.sort(a.ravel())[::-1]
        thetas = [(R + float(srt[:n].astype(np.float64).sum())) * (sps[R + n] if R + n < len(sps) else 0)
                  for n in range(R * gamma + 1)]
        diffs = np.diff(thetas)
        unimodal = not np.any((diffs[1:] > 0) & (diffs[:-1] <= 0))
        if unimodal:
            assert abs(th1 - btheta) <= 1e-12 * btheta
        # invariants: 0 <= l <= gamma, prefix structure, n* = sum l
        assert np.all((L1 >= 0) & (L1 <= gamma))


def test_scheduler_toy_workload_nondegenerate_and_degenerate():
    w = synth.WORKLOADS["toy"]
    c = synth.gen_c(w)
    L, th, n = oracle.schedule_loop(c, synth.gen_sps(w.R, w.gamma, w.rho))
    assert 0 < n < w.R * w.gamma
    # a large batch under heavy load stops at n = 0 (each extra token costs
    # more Theta through SPS than it adds through tau)
    wl = synth.WORKLOADS["longblock"].scaled(R=64)
    c4 = synth.gen_c(wl)
    L4, th4, n4 = oracle.schedule_loop(c4, synth.gen_sps(wl.R, wl.gamma, wl.rho))
    assert n4 == 0 and np.all(L4 == 0)


def test_scheduler_exact_ties_keep_prefix_order():
    """c = 1 makes a equal along a request; the order (a desc, r asc, j asc)
    never skips a position."""
    c = np.array([[1.0, 1.0, 0.5], [0.9, 1.0, 1.0]], np.float32)
    sps = np.full(2 * 4 + 1, 1.0)      # flat SPS: every candidate helps
    L, th, n = oracle.schedule_loop(c, sps)
    L2, th2, n2, _ = oracle.schedule_closed(c, sps)
    np.testing.assert_array_equal(L, [3, 3])
    np.testing.assert_array_equal(L, L2)
    assert n == 6 and abs(th - (2 + 1 + 1 + 0.5 + 0.9 + 0.9 + 0.9)) < 1e-6


# ------------------------------------------------------------------ confidence head
def _bf16_bits(x):
    """float32 values that bf16 holds exactly -> their bf16 bit patterns."""
    b = np.ascontiguousarray(np.asarray(x, np.float32)).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


@pytest.mark.parametrize("storage", ["f32", "bf16"])
def test_confidence_head_hand_worked_two_steps(storage):
    """Blog section 4.1: c_k = sigmoid(w . [h_k, W1[x_{k-1}]]), no bias.
    d = 2, r = 2, V = 3, every value exact in bf16:
      W1 rows: x=0 -> (3, -1), x=1 -> (1/2, 2), x=2 -> (-2, 1)
      anchor x_0 = 0, drafted x_1 = 1, x_2 = 2
      h_1 = (1, 2), h_2 = (-1, 1/2),  w = (1/2, 1/4 | 1/8, -1/4)
      k = 1: 1/2 + 1/2 + 3/8 + 1/4 = 13/8
      k = 2: -1/2 + 1/8 + 1/16 - 1/2 = -13/16
    (the concatenation [e, h] would give 7/8 at k = 1; the embedding of x_1 at
    k = 1 would give 9/16)."""
    W1 = np.array([[3, -1], [0.5, 2], [-2, 1]], np.float32)
    H = np.array([[[1, 2], [-1, 0.5]]], np.float32)
    w = np.array([0.5, 0.25, 0.125, -0.25], np.float32)
    if storage == "bf16":
        W1, H = _bf16_bits(W1), _bf16_bits(H)
    c = oracle.confidence(H, W1, w, np.array([0], np.int32), np.array([[1, 2]], np.int32))
    np.testing.assert_allclose(c[0], special.expit([13 / 8, -13 / 16]), rtol=0, atol=1e-15)
    # with per-position temperatures (section 4.2): the logits divided by t_k
    ct = oracle.confidence(H, W1, w, np.array([0], np.int32), np.array([[1, 2]], np.int32), temps=[2.0, 0.5])
    np.testing.assert_allclose(ct[0], special.expit([13 / 16, -13 / 8]), rtol=0, atol=1e-15)


def _conf_case(seed, R=6, gamma=4, V=50, d=24, r=8):
    rng = np.random.default_rng(seed)
    H = rng.normal(0, 1, (R, gamma, d)).astype(np.float32)
    W1 = rng.normal(0, 0.5, (V, r)).astype(np.float32)
    w = rng.normal(0, 0.3, d + r).astype(np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    tokens = rng.integers(0, V, (R, gamma)).astype(np.int32)
    return H, W1, w, anchor, tokens


def test_confidence_head_special_cases():
    H, W1, w, anchor, tokens = _conf_case(3)
    d = H.shape[2]
    # w = 0: sigmoid(0) = 1/2 everywhere
    c0 = oracle.confidence(H, W1, np.zeros_like(w), anchor, tokens)
    assert np.all(c0 == 0.5)
    # no bias: negating w gives 1 - c
    c = oracle.confidence(H, W1, w, anchor, tokens)
    cn = oracle.confidence(H, W1, -w, anchor, tokens)
    np.testing.assert_allclose(cn, 1.0 - c, rtol=0, atol=1e-15)
    assert np.all((c > 0) & (c < 1))
    # linear in w: the logits of a split w add up
    wa = np.concatenate([w[:d], np.zeros_like(w[d:])])
    wb = w - wa
    lg = special.logit
    ca = oracle.confidence(H, W1, wa, anchor, tokens)
    cb = oracle.confidence(H, W1, wb, anchor, tokens)
    np.testing.assert_allclose(lg(ca) + lg(cb), lg(c), rtol=0, atol=1e-12)
    # the h part ignores the tokens; the embedding part sees only x_{k-1}
    other = (tokens + 7) % W1.shape[0]
    np.testing.assert_array_equal(ca, oracle.confidence(H, W1, wa, (anchor + 3) % W1.shape[0], other))
    shifted = np.concatenate([anchor[:, None], tokens[:, :-1]], axis=1)      # x_0 .. x_{gamma-1}
    for k in range(tokens.shape[1]):
        for i in range(len(anchor)):
            for j in range(len(anchor)):
                if shifted[i, k] == shifted[j, k]:
                    assert cb[i, k] == cb[j, k]
    same = np.tile(shifted[:1], (len(anchor), 1))
    cb_same = oracle.confidence(H, W1, wb, same[:, 0].copy(), np.concatenate([same[:, 1:], tokens[:, -1:]], 1))
    assert np.all(cb_same == cb_same[:1])


def test_confidence_head_rejects_out_of_range_tokens():
    H, W1, w, anchor, tokens = _conf_case(4)
    tokens[1, 2] = W1.shape[0]
    with pytest.raises(RuntimeError):
        oracle.confidence(H, W1, w, anchor, tokens)


# ------------------------------------------------------------------ threshold filter
def test_threshold_filter_worked_values():
    """The explainer's section 04 numbers: c = 0.8 three times gives
    a = (0.8, 0.64, 0.512).  Prefix-survival mode keeps the positions whose a
    clears theta; per-token mode keeps all three while 0.8 >= theta."""
    g = read_golden("prefix_survival.txt")
    c = np.array([g["c"][0]], np.float32)
    for theta, want in [(0.5, 3), (0.6, 2), (0.7, 1), (0.81, 0)]:
        assert oracle.threshold_lengths(c, theta, 0)[0] == want
    assert oracle.threshold_lengths(c, 0.8, 1)[0] == 3
    assert oracle.threshold_lengths(c, 0.81, 1)[0] == 0


def test_threshold_filter_modes_differ_on_a_dip():
    """c = (0.9, 0.5, 0.95): a = (0.9, 0.45, 0.4275).  A per-token threshold of
    0.6 stops at the dip (length 1) although 0.95 follows; the prefix-survival
    threshold counts a >= theta."""
    c = np.array([[0.9, 0.5, 0.95]], np.float32)
    assert oracle.threshold_lengths(c, 0.6, 1)[0] == 1
    assert oracle.threshold_lengths(c, 0.4, 1)[0] == 3
    for theta, want in [(0.46, 1), (0.44, 2), (0.4, 3), (0.95, 0)]:
        assert oracle.threshold_lengths(c, theta, 0)[0] == want


def test_threshold_filter_invariants():
    w = synth.WORKLOADS["toy"].scaled(R=64)
    c = synth.gen_c(w)
    c[3, 2] = 0.0
    c[5, :] = 1.0
    a = oracle.prefix_survival(c)
    prev0 = prev1 = None
    for theta in np.linspace(-0.1, 1.1, 49).astype(np.float32):
        L0 = oracle.threshold_lengths(c, theta, 0)
        L1 = oracle.threshold_lengths(c, theta, 1)
        assert np.all((L0 >= 0) & (L0 <= w.gamma)) and np.all(L0 <= L1)
        # a is non-increasing along a request, so the kept set is exactly {a >= theta}
        assert L0.sum() == int((a >= theta).sum())
        if prev0 is not None:
            assert np.all(L0 <= prev0) and np.all(L1 <= prev1)
        prev0, prev1 = L0, L1
        if theta <= 0:
            assert np.all(L0 == w.gamma)
        if theta > 1:
            assert np.all(L1 == 0)
    assert oracle.threshold_lengths(c, 0.5, 0)[3] <= 2 and oracle.threshold_lengths(c, 1.0, 0)[5] == w.gamma


# ------------------------------------------------------------------ STS
def test_ece_hand_worked():
    """Guo et al. 2017, section 2, by hand: M = 10, predictions 0.1, 0.1, 0.9,
    0.9 with outcomes 0, 1, 1, 1: bin 1 has accuracy 1/2 and confidence 0.1,
    bin 9 accuracy 1 and confidence 0.9, so ECE = 1/2 (0.4) + 1/2 (0.1) = 0.25."""
    assert abs(oracle.ece([0.1, 0.1, 0.9, 0.9], [0, 1, 1, 1], 10) - 0.25) < 1e-15
    # bin edges, M = 4: p = 0.25 opens bin 1, so 0.25 and 0.24 sit apart
    # (1/2 (0.75) + 1/2 (0.24), not one bin's |1/2 - 0.245|); p = 1 shares
    # bin 3 with 0.75 and 0.8 (|2/3 - 0.85|, not 1/3 + 2/3 |1 - 0.775|)
    assert abs(oracle.ece([0.25, 0.24], [1, 0], 4) - (0.5 * 0.75 + 0.5 * 0.24)) < 1e-15
    assert abs(oracle.ece([1.0, 0.75, 0.8], [0, 1, 1], 4) - abs(2 / 3 - 2.55 / 3)) < 1e-15
    # calibrated in the bins: 30% positives at p = 0.3 gives 0
    assert oracle.ece([0.3] * 10, [1, 1, 1] + [0] * 7, 10) < 1e-15


def test_sts_apply_closed_forms():
    c = np.array([[0.5, special.expit(2.0), 0.0, 1.0]], np.float32)
    out = oracle.sts_apply(c, np.array([3.0, 2.0, 0.5, 0.5]))
    assert out[0, 0] == 0.5                                  # logit 0 is fixed by every t
    # sigmoid(2) stored in float32, then tempered by 2: sigmoid(logit(float32 value) / 2)
    z = math.log(float(c[0, 1])) - math.log1p(-float(c[0, 1]))
    assert abs(out[0, 1] - special.expit(z / 2)) < 1e-15 and abs(out[0, 1] - special.expit(1.0)) < 1e-7
    assert out[0, 2] == 0.0 and out[0, 3] == 1.0
    # t = 1 is the identity; order inside a position is preserved for any t
    cc = np.sort(np.random.default_rng(1).random((50, 1)).astype(np.float32), axis=0)
    np.testing.assert_allclose(oracle.sts_apply(cc, [1.0]), cc.astype(np.float64), rtol=1e-12)
    for t in (0.3, 4.0):
        assert np.all(np.diff(oracle.sts_apply(cc, [t])[:, 0]) >= 0)


@pytest.mark.parametrize("tau", [2.0, 1.0, 0.5])
def test_sts_recovers_a_known_overconfidence(tau):
    """Raw confidences sigmoid(tau u) of events with probability sigmoid(u):
    sigmoid(logit(c) / tau) is exactly calibrated, so the left-to-right search
    should settle near t = tau at every position (sampling noise and the grid
    step of 1.8% aside), and lower the ECE it was given."""
    c, al = synth.gen_sts_set(20000, 5, tau=tau, seed=3)
    grid = synth.sts_grid(256, 0.1, 10.0)
    r = oracle.sts_fit(c, al, grid, 15)
    assert np.all(np.abs(np.log(r["t"] / tau)) < 0.15), r["t"]
    raw = np.cumprod(c.astype(np.float64), axis=1)
    for k in range(5):
        e_raw = oracle.ece(raw[:, k], (al >= k + 1).astype(np.int32), 15)
        assert r["ece"][k] <= e_raw + 1e-12
        if tau != 1.0:
            assert r["ece"][k] < 0.6 * e_raw


def test_sts_is_sequential():
    """Position k's temperature depends only on outcomes up to k: changing
    accept_len among values above k leaves t_1..t_k unchanged; a one-point
    grid returns that point everywhere."""
    c, al = synth.gen_sts_set(3000, 4, tau=2.0, seed=5)
    grid = synth.sts_grid(64, 0.2, 8.0)
    r = oracle.sts_fit(c, al, grid, 10)
    al2 = al.copy()
    al2[al2 >= 3] = 4 - (al2[al2 >= 3] - 3)          # swap 3 <-> 4 above position 2
    r2 = oracle.sts_fit(c, al2, grid, 10)
    np.testing.assert_array_equal(r["g"][:2], r2["g"][:2])
    one = oracle.sts_fit(c, al, np.array([1.7]), 10)
    assert np.all(one["t"] == 1.7) and np.all(np.isinf(one["gap"]))


def test_sts_first_position_is_a_plain_grid_search():
    """At k = 1 nothing is fixed yet: t_1 is the grid point whose tempered
    c_1 has the smallest ECE against accept_len >= 1, found here by
    evaluating every grid point with the ECE pinned above."""
    c, al = synth.gen_sts_set(2000, 3, tau=1.5, seed=9)
    grid = synth.sts_grid(40, 0.3, 5.0)
    r = oracle.sts_fit(c, al, grid, 12)
    y = (al >= 1).astype(np.int32)
    e = [oracle.ece(oracle.sts_apply(c[:, :1], [t])[:, 0], y, 12) for t in grid]
    assert r["g"][0] == int(np.argmin(e)) and abs(r["ece"][0] - min(e)) < 1e-15


# ------------------------------------------------------------------ production-style scheduler
def test_budget_scheduler_fills_the_capacity_in_the_scheduler_order():
    """Explainer section 04: the capacity comes from two steps back and the
    current candidates are ranked into it.  c = (0.9, 0.8), (0.5, 0.99) gives
    a = (0.9, 0.72), (0.5, 0.495): the order is (r0 j1), (r0 j2), (r1 j1),
    (r1 j2), so capacities 1..4 give lengths (1,0), (2,0), (2,1), (2,2); with a
    flat SPS = 1, theta = 2 + the sum of the chosen a."""
    c = np.array([[0.9, 0.8], [0.5, 0.99]], np.float32)
    a = oracle.prefix_survival(c).astype(np.float64)
    sps = np.ones(2 * 3 + 1)
    want = {1: [1, 0], 2: [2, 0], 3: [2, 1], 4: [2, 2], 9: [2, 2]}
    tops = [a[0, 0], a[0, 1], a[1, 0], a[1, 1]]
    for b, L in want.items():
        got, th, n, ns = oracle.schedule_budget(c, sps, b)
        np.testing.assert_array_equal(got, L)
        assert n == min(b, 4) and abs(th - (2 + sum(tops[:n]))) < 1e-12
    got, th, n, _ = oracle.schedule_budget(c, sps, 0)
    assert np.all(got == 0) and n == 0 and th == 2.0


@pytest.mark.parametrize("rho", [0.0, 0.5, 0.9])
def test_budget_scheduler_reduces_to_the_synchronous_one(rho):
    """With its own n* as the capacity (or none) the production-style rule is
    the synchronous scheduler, and the n* it reports is the closed form's."""
    rng = np.random.default_rng(int(rho * 10))
    for R, gamma in [(3, 4), (16, 5), (64, 8)]:
        c = (1 / (1 + np.exp(-rng.normal(1.5, 1.0, (R, gamma))))).astype(np.float32)
        sps = synth.gen_sps(R, gamma, rho)
        L0, th0, n0, _ = oracle.schedule_closed(c, sps)
        for b in (-1, n0):
            L, th, n, ns = oracle.schedule_budget(c, sps, b)
            np.testing.assert_array_equal(L, L0)
            assert n == n0 == ns and abs(th - th0) <= 1e-12 * max(1.0, abs(th0))
