"""Helpers shared by the GPU parity tests: host <-> device conversion and the
comparison rules (bit-exact discrete outputs except flagged near-ties,
1e-4 relative on probabilities and log-sum-exps)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_drafting_gb300 import binding, synth

# parity tolerances for the floating-point outputs and the flagging margins
REL_TOL = 1e-4          # q(x), p(x), logsumexp
GUMBEL_FLAG = 1e-4      # Gumbel-max (or greedy argmax) margin below which a draft token is flagged
UNIFORM_FLAG = 1e-6     # a uniform this close to its threshold is flagged


def dev(a: np.ndarray, device="cuda:0") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(device)


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class Flags:
    """Flag accounting over one or more parity comparisons.

    A decision is flagged when the oracle's own margin lies inside a band the
    kernels' rounding could cross: a Gumbel-max or greedy argmax margin below
    1e-4, a uniform within 1e-6 of its acceptance or tree threshold.  Only
    there may the GPU disagree with the oracle; an unflagged disagreement
    fails the comparison at once.  ``positions`` counts the draft positions
    compared, ``raw`` the flagged decisions among them, ``mismatch`` the
    flagged decisions where the two sides disagreed.  The contract caps the
    flagged disagreements at 1e-4 of the positions."""

    def __init__(self):
        self.positions = 0
        self.raw = 0
        self.mismatch = 0

    def check(self, tag: str = ""):
        assert self.mismatch <= 1e-4 * self.positions, (
            f"{tag} {self.mismatch} flagged disagreements in {self.positions} positions (cap 1e-4)")

    def summary(self) -> dict:
        n = max(1, self.positions)
        return dict(positions=self.positions, flagged=self.raw, flagged_rate=self.raw / n,
                    flagged_disagreements=self.mismatch, disagreement_rate=self.mismatch / n)


def compare_draft(g: dict, o: dict, tag: str = "", flags: Flags = None):
    """GPU draft outputs g (numpy) vs oracle o.

    Tokens must match at every position of a request up to its first flagged
    (margin < 1e-4) mismatch; from there on the request conditions on a
    different prefix and is not compared.  lse and q(x) within 1e-4 relative,
    code exactly (Markov) at compared positions.  Returns (n_compared,
    n_flagged_mismatch, mask of compared positions); ``flags`` (if given)
    adds the compared positions, the flagged ones and the flagged mismatches."""
    tok_g, tok_o = g["tokens"], o["tokens"]
    R, gamma = tok_o.shape
    compared = np.zeros((R, gamma), bool)
    n_flag_mis = 0
    for i in range(R):
        for k in range(gamma):
            compared[i, k] = True
            if tok_g[i, k] != tok_o[i, k]:
                assert o["margin"][i, k] < GUMBEL_FLAG, (
                    f"{tag} draft token mismatch at request {i} position {k + 1}: gpu {tok_g[i, k]} "
                    f"oracle {tok_o[i, k]} margin {o['margin'][i, k]:.3g}")
                n_flag_mis += 1
                break
    m = compared
    # a flagged mismatch ends its request's comparison; q(x) and lse of that
    # position describe different tokens and are not compared
    mv = m.copy()
    for i in range(R):
        k = np.nonzero(tok_g[i] != tok_o[i])[0]
        if k.size:
            mv[i, k[0]] = False
    np.testing.assert_allclose(g["lse"][mv], o["lse"][mv], rtol=REL_TOL, err_msg=f"{tag} lse")
    np.testing.assert_allclose(g["q_tok"][mv], o["qx"][mv], rtol=REL_TOL, err_msg=f"{tag} q(x)")
    if flags is not None:
        flags.positions += int(m.sum())
        flags.raw += int((o["margin"][m] < GUMBEL_FLAG).sum())
        flags.mismatch += n_flag_mis
    return int(m.sum()), n_flag_mis, m


def compare_verify(g: dict, o: dict, rows_ok: np.ndarray, tag: str = "", flags: Flags = None):
    """GPU verify outputs vs oracle on identical inputs.  Requests whose oracle
    decisions came within 1e-6 of a threshold are flagged: they may differ
    (``flags`` counts them and their disagreements), every other request must
    agree.  Returns (requests compared unflagged, flagged requests)."""
    flagged = o["min_gap"] < UNIFORM_FLAG
    sel = rows_ok & ~flagged
    if flags is not None:
        fl = rows_ok & flagged
        differ = (g["out_tokens"] != o["out_tokens"]).any(axis=1) | (g["accept_len"] != o["accept_len"])
        flags.raw += int(fl.sum())
        flags.mismatch += int((fl & differ).sum())
    np.testing.assert_array_equal(g["accept_len"][sel], o["accept_len"][sel], err_msg=f"{tag} accept_len")
    np.testing.assert_array_equal(g["n_out"][sel], o["n_out"][sel], err_msg=f"{tag} n_out")
    bad = np.where((g["out_tokens"][sel] != o["out_tokens"][sel]).any(axis=1))[0]
    assert bad.size == 0, (f"{tag} out_tokens differ for requests {np.where(sel)[0][bad][:8]}: "
                           f"gpu {g['out_tokens'][sel][bad[:2]]} oracle {o['out_tokens'][sel][bad[:2]]} "
                           f"gaps {o['min_gap'][sel][bad[:2]]}")
    assert np.all(g["n_out"] >= 1)
    # probabilities / lse where the oracle evaluated them
    pm = ~np.isnan(o["px"]) & sel[:, None]
    np.testing.assert_allclose(g["p_tok"][pm], o["px"][pm], rtol=REL_TOL, err_msg=f"{tag} p(x)")
    lm = ~np.isnan(o["lse_p"]) & sel[:, None]
    np.testing.assert_allclose(g["lse_p"][lm], o["lse_p"][lm], rtol=REL_TOL, err_msg=f"{tag} lse_p")
    return int(sel.sum()), int(flagged.sum())


def gpu_draft(w: synth.Workload, x: dict, seed: int, req_ids=None):
    if w.head == "rnn":
        d = binding.draft_rnn(dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"]), dev(x["Wgco"]),
                              dev(x["H"]), w.T, seed, req_ids=None if req_ids is None else dev(req_ids))
    else:
        d = binding.draft_markov(dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"]), w.T, seed,
                                 req_ids=None if req_ids is None else dev(req_ids))
    torch.cuda.synchronize()
    assert binding.workspace_status(d["ws"]) == 0
    return {k: host(v) for k, v in d.items() if k != "ws"}


def oracle_draft(w: synth.Workload, x: dict, seed: int, req_ids=None):
    if w.head == "rnn":
        return oracle.draft_rnn(x["U"], x["anchor"], x["W1"], x["W2"], x["Wgco"], x["H"], w.T, seed,
                                req_ids=req_ids)
    return oracle.draft_markov(x["U"], x["anchor"], x["W1"], x["W2"], w.T, seed, req_ids=req_ids)


def gpu_verify_on(w: synth.Workload, x: dict, dr: dict, seed: int, verify_len=None, req_ids=None):
    """GPU verify fed with draft outputs dr (numpy: tokens, qx/q_tok, lse, code)."""
    qx = dr["q_tok"] if "q_tok" in dr else dr["qx"].astype(np.float32)
    draft = dict(tokens=dev(dr["tokens"].astype(np.int32)), q_tok=dev(qx.astype(np.float32)),
                 lse=dev(dr["lse"].astype(np.float64)), code=dev(dr["code"].astype(np.float32)))
    v = binding.verify(dev(x["P"]), dev(x["U"]), dev(x["W2"]), draft, w.T, seed,
                       verify_len=None if verify_len is None else dev(verify_len.astype(np.int32)),
                       req_ids=None if req_ids is None else dev(req_ids))
    torch.cuda.synchronize()
    assert binding.workspace_status(v["ws"]) == 0
    return {k: host(t) for k, t in v.items() if k != "ws"}


def oracle_verify_on(w, x, dr, seed, verify_len=None, req_ids=None):
    qx = (dr["q_tok"] if "q_tok" in dr else dr["qx"]).astype(np.float32).astype(np.float64)
    code = dr["code"].astype(np.float32).astype(np.float64)
    return oracle.verify(x["P"], x["U"], x["W2"], dr["tokens"], qx, dr["lse"], code, w.T, seed,
                         verify_len=verify_len, req_ids=req_ids)
