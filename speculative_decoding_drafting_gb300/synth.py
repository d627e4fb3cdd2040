"""Seeded synthetic inputs for one DSpark decoding cycle.

This module only draws numbers.  It holds none of the method's arithmetic
(no softmax, no sampling, no verification, no scheduling), so that the CUDA
path and the CPU oracle can both consume exactly the same bytes.

Shapes and value distributions follow the workloads of the DSpark pages:

* base logits ``U[R, gamma, V]`` of the parallel backbone (DSpark blog,
  section 3.1 "Parallel Stage"), normal with the workload's sigma;
* Markov head weights ``W1[V, r]`` (embedding) and ``W2[r, V]`` (rank-r
  projection) (DSpark blog, section 3.2 ``MarkovHead``);
* RNN head weights ``Wgco[2r+d, 3r]`` and backbone states ``h[R, gamma, d]``
  (DSpark blog, section 3.2 ``RNNHead``);
* target logits ``P[R, gamma+1, V]``: ``U`` with its last position repeated
  once more (the bonus row), plus normal noise;
* confidences ``c[R, gamma] = sigmoid(N(mu, s^2))``;
* confidence-head inputs (DSpark blog, section 4.1 ``ConfidenceHead``):
  backbone states ``h[R, gamma, d]`` (bf16, N(0, sigma_h^2)) and the head's
  weight vector ``w[d + r]`` (float32, N(0, sigma_w^2));
* an STS calibration set (DSpark blog, section 4.2): per block n and
  position k a latent acceptance probability ``alpha = sigmoid(u)``,
  ``u ~ N(mu, s^2)``, outcomes drawn position by position (``accept_len`` =
  the leading successes), and raw confidences ``sigmoid(tau u)`` that are
  overconfident by a known factor ``tau``;
* the steps-per-second table ``SPS[B] = 1000 / T(B)`` of the explainer's toy
  cost curve ``T(B) = 20 + (0.05 + 1.15 rho) B + (0.002 + 0.10 rho) B^2`` ms
  (DSpark explainer, section 04 "algorithm details"), tabulated for
  ``B = 0 .. R (1 + gamma)``.

Random numbers come from numpy's PCG64 seeded with the workload seed; every
array has its own child stream so that a subset of requests can be
regenerated cheaply.  bf16 arrays are produced from float32 draws by
round-to-nearest-even and are returned as ``uint16`` bit patterns.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

F32 = 0
BF16 = 1
DTYPE_NAMES = {F32: "f32", BF16: "bf16"}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Sizes and distributions of one synthetic cycle."""

    name: str
    R: int
    gamma: int
    V: int
    r: int
    T: float
    u_dtype: int = F32
    p_dtype: int = F32
    w_dtype: int = BF16
    sigma_u: float = 1.5
    sigma_w: float = 0.02
    sigma_pnoise: float = 1.0
    c_mu: float = 1.5
    c_sigma: float = 1.0
    rho: float = 0.5
    head: str = "markov"          # "markov" or "rnn"
    d: int = 0                    # backbone width (RNN head only)
    sigma_h: float = 1.0
    seed: int = 0
    verify_all: bool = True       # verify every drafted position

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def positions(self) -> int:
        return self.R * self.gamma


# The five workloads of the build plus the headline one.  Sizes are the
# pages' DSpark-5 setting (5-token block, rank 256) on vocabularies of the
# sizes named in the workload list.
WORKLOADS: Dict[str, Workload] = {
    "toy": Workload("toy", R=4, gamma=5, V=4096, r=32, T=1.0, w_dtype=F32,
                    sigma_w=0.05, sigma_pnoise=0.5, rho=0.5, verify_all=False),
    "dspark5": Workload("dspark5", R=64, gamma=5, V=151936, r=256, T=1.0),
    "headline": Workload("headline", R=256, gamma=5, V=151936, r=256, T=1.0),
    "greedy": Workload("greedy", R=256, gamma=5, V=129280, r=256, T=0.0,
                       sigma_u=2.0, sigma_pnoise=0.7),
    "longblock": Workload("longblock", R=512, gamma=16, V=151936, r=256, T=0.8,
                          u_dtype=BF16, p_dtype=BF16, sigma_pnoise=1.2,
                          c_mu=1.0, c_sigma=1.5, rho=0.9, verify_all=False),
    "rnn": Workload("rnn", R=256, gamma=8, V=151936, r=256, T=1.0,
                    head="rnn", d=2048),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _store(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == BF16:
        return f32_to_bf16_bits(x)
    raise ValueError(f"unknown dtype {dtype}")


def _child(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag])))


_TAG = {"anchor": 1, "U": 2, "W1": 3, "W2": 4, "Pnoise": 5, "c": 6, "h": 7, "Wgco": 8, "hconf": 9, "wconf": 10,
        "sts": 11}


def gen_anchor(w: Workload) -> np.ndarray:
    return _child(w.seed, _TAG["anchor"]).integers(0, w.V, size=w.R, dtype=np.int64).astype(np.int32)


def gen_U_f32(w: Workload, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Base logits as float32 draws (before storage rounding), [R, gamma, V].

    Each request has its own stream so a subset ``rows`` can be drawn alone.
    """
    idx = np.arange(w.R) if rows is None else np.asarray(rows)
    out = np.empty((len(idx), w.gamma, w.V), dtype=np.float32)
    for n, i in enumerate(idx):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, _TAG["U"], int(i)])))
        out[n] = g.standard_normal((w.gamma, w.V), dtype=np.float32) * np.float32(w.sigma_u)
    return out


def gen_U(w: Workload, rows=None) -> np.ndarray:
    return _store(gen_U_f32(w, rows), w.u_dtype)


def gen_P(w: Workload, rows=None) -> np.ndarray:
    """Target logits [R, gamma+1, V]: U with its last row repeated, plus noise."""
    idx = np.arange(w.R) if rows is None else np.asarray(rows)
    U = gen_U_f32(w, idx)
    out = np.empty((len(idx), w.gamma + 1, w.V), dtype=np.float32)
    for n, i in enumerate(idx):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, _TAG["Pnoise"], int(i)])))
        noise = g.standard_normal((w.gamma + 1, w.V), dtype=np.float32) * np.float32(w.sigma_pnoise)
        out[n, : w.gamma] = U[n] + noise[: w.gamma]
        out[n, w.gamma] = U[n, w.gamma - 1] + noise[w.gamma]
    return _store(out, w.p_dtype)


def gen_W1(w: Workload) -> np.ndarray:
    g = _child(w.seed, _TAG["W1"])
    return _store(g.standard_normal((w.V, w.r), dtype=np.float32) * np.float32(w.sigma_w), w.w_dtype)


def gen_W2(w: Workload) -> np.ndarray:
    g = _child(w.seed, _TAG["W2"])
    return _store(g.standard_normal((w.r, w.V), dtype=np.float32) * np.float32(w.sigma_w), w.w_dtype)


def gen_H(w: Workload, rows=None) -> np.ndarray:
    """Backbone hidden states [R, gamma, d] (bf16), RNN head only."""
    idx = np.arange(w.R) if rows is None else np.asarray(rows)
    out = np.empty((len(idx), w.gamma, w.d), dtype=np.float32)
    for n, i in enumerate(idx):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, _TAG["h"], int(i)])))
        out[n] = g.standard_normal((w.gamma, w.d), dtype=np.float32) * np.float32(w.sigma_h)
    return f32_to_bf16_bits(out)


def gen_Wgco(w: Workload) -> np.ndarray:
    g = _child(w.seed, _TAG["Wgco"])
    return _store(g.standard_normal((2 * w.r + w.d, 3 * w.r), dtype=np.float32) * np.float32(w.sigma_w), w.w_dtype)


def gen_conf_H(w: Workload, d: int, rows=None) -> np.ndarray:
    """Backbone states [R, gamma, d] (bf16) for the confidence head of a
    Markov-head workload (an RNN-head workload uses its own ``gen_H``)."""
    idx = np.arange(w.R) if rows is None else np.asarray(rows)
    out = np.empty((len(idx), w.gamma, d), dtype=np.float32)
    for n, i in enumerate(idx):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, _TAG["hconf"], int(i)])))
        out[n] = g.standard_normal((w.gamma, d), dtype=np.float32) * np.float32(w.sigma_h)
    return f32_to_bf16_bits(out)


def gen_conf_w(w: Workload, d: int) -> np.ndarray:
    """Confidence-head weights [d + r] (float32): w[:d] meet h_k, w[d:] meet W1[x_{k-1}]."""
    g = _child(w.seed, _TAG["wconf"])
    return g.standard_normal(d + w.r, dtype=np.float32) * np.float32(w.sigma_w)


def gen_c(w: Workload) -> np.ndarray:
    g = _child(w.seed, _TAG["c"])
    x = g.normal(w.c_mu, w.c_sigma, size=(w.R, w.gamma))
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def gen_sts_set(N: int, gamma: int, tau: float = 2.0, mu: float = 1.5, s: float = 1.0, seed: int = 0):
    """STS calibration set: raw confidences c [N, gamma] (float32) and
    accept_len [N] (int32).  u ~ N(mu, s^2); position k of block n is accepted
    with probability sigmoid(u[n, k]) (a uniform below it), accept_len counts
    the leading acceptances, and c = sigmoid(tau u)."""
    g = _child(seed, _TAG["sts"])
    u = g.normal(mu, s, size=(N, gamma))
    v = g.random(size=(N, gamma))
    ok = v < 1.0 / (1.0 + np.exp(-u))
    accept_len = np.where(ok.all(axis=1), gamma, np.argmin(ok, axis=1)).astype(np.int32)
    c = (1.0 / (1.0 + np.exp(-tau * u))).astype(np.float32)
    return c, accept_len


def sts_grid(G: int = 256, lo: float = 0.1, hi: float = 10.0) -> np.ndarray:
    """Candidate temperatures, log-spaced over [lo, hi] (float64)."""
    return np.geomspace(lo, hi, G)


def toy_cost_ms(B: np.ndarray, rho: float) -> np.ndarray:
    """The explainer's toy step-time curve T(B) in milliseconds."""
    B = np.asarray(B, dtype=np.float64)
    return 20.0 + (0.05 + 1.15 * rho) * B + (0.002 + 0.10 * rho) * B * B


def gen_sps(R: int, gamma: int, rho: float) -> np.ndarray:
    """SPS[B] = 1000 / T(B) steps per second, for B = 0 .. R (1 + gamma)."""
    B = np.arange(R * (1 + gamma) + 1, dtype=np.float64)
    return 1000.0 / toy_cost_ms(B, rho)


def gen_all(w: Workload, rows=None) -> Dict[str, np.ndarray]:
    """Every input of one cycle (host arrays)."""
    idx = np.arange(w.R) if rows is None else np.asarray(rows)
    d = {
        "anchor": gen_anchor(w)[idx],
        "U": gen_U(w, idx),
        "P": gen_P(w, idx),
        "W1": gen_W1(w),
        "W2": gen_W2(w),
        "c": gen_c(w)[idx],
        "sps": gen_sps(len(idx), w.gamma, w.rho),
        "req_ids": idx.astype(np.uint32),
    }
    if w.head == "rnn":
        d["H"] = gen_H(w, idx)
        d["Wgco"] = gen_Wgco(w)
    return d


def gen_device(w: Workload, device, seed: int = 0) -> Dict[str, "object"]:
    """The same recipe as gen_all, drawn on the device from a seeded torch
    generator (torch tensors; bf16 by round-to-nearest-even).  The values
    differ from gen_all's (another generator) but the distributions are the
    same; the benchmark uses this for its timing legs at sizes whose numpy
    draw would take minutes (the long block's 2.6 billion normals)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)
    sd = {F32: torch.float32, BF16: torch.bfloat16}

    def normal(shape, sigma):
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma

    U = normal((w.R, w.gamma, w.V), w.sigma_u)
    P = torch.empty((w.R, w.gamma + 1, w.V), dtype=sd[w.p_dtype], device=device)
    P[:, : w.gamma] = (U + normal((w.R, w.gamma, w.V), w.sigma_pnoise)).to(sd[w.p_dtype])
    P[:, w.gamma] = (U[:, w.gamma - 1] + normal((w.R, w.V), w.sigma_pnoise)).to(sd[w.p_dtype])
    d = {
        "anchor": torch.randint(0, w.V, (w.R,), generator=g, device=device, dtype=torch.int32),
        "U": U.to(sd[w.u_dtype]),
        "P": P,
        "W1": normal((w.V, w.r), w.sigma_w).to(sd[w.w_dtype]),
        "W2": normal((w.r, w.V), w.sigma_w).to(sd[w.w_dtype]),
        "c": torch.sigmoid(torch.randn((w.R, w.gamma), generator=g, device=device, dtype=torch.float64)
                           * w.c_sigma + w.c_mu).to(torch.float32),
        "sps": torch.from_numpy(gen_sps(w.R, w.gamma, w.rho)).to(device),
    }
    del U
    return d
