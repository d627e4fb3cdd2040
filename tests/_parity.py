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


def compare_draft(g: dict, o: dict, tag: str = ""):
    """GPU draft outputs g (numpy) vs oracle o.

    Tokens must match at every position of a request up to its first flagged
    (margin < 1e-4) mismatch; from there on the request conditions on a
    different prefix and is not compared.  lse and q(x) within 1e-4 relative,
    code exactly (Markov) at compared positions.  Returns (n_compared,
    n_flagged_mismatch, mask of compared positions)."""
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
    np.testing.assert_allclose(g["lse"][m], o["lse"][m], rtol=REL_TOL, err_msg=f"{tag} lse")
    np.testing.assert_allclose(g["q_tok"][m], o["qx"][m], rtol=REL_TOL, err_msg=f"{tag} q(x)")
    return int(m.sum()), n_flag_mis, m


def compare_verify(g: dict, o: dict, rows_ok: np.ndarray, tag: str = ""):
    """GPU verify outputs vs oracle on identical inputs.  Requests whose oracle
    decisions came within 1e-6 of a threshold are flagged and skipped."""
    flagged = o["min_gap"] < UNIFORM_FLAG
    sel = rows_ok & ~flagged
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
