"""CPU oracle of the DSpark cycle: ctypes wrappers around ``dspark_oracle.c``.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path (the
CUDA library and its binding) never does.

Every wrapper takes numpy arrays in their storage type (float32, or bfloat16
as uint16 bit patterns) and returns numpy outputs in double precision.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdspark_oracle.so")
_SRC = [os.path.join(_HERE, "dspark_oracle.c")]
_HDR = [os.path.join(_HERE, "dspark_oracle.h")]
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build``."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(p) for p in _SRC + _HDR)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
           "-pthread", "-o", tmp] + _SRC + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i32, u64, dbl = ctypes.c_int, ctypes.c_uint64, ctypes.c_double
            L.oracle_philox4x32_10.argtypes = [P, P, P]
            L.oracle_uniform.argtypes = [ctypes.c_uint32]
            L.oracle_uniform.restype = dbl
            L.oracle_rng_uniform.argtypes = [u64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
            L.oracle_rng_uniform.restype = dbl
            L.oracle_accept_prob.argtypes = [dbl, dbl]
            L.oracle_accept_prob.restype = dbl
            L.oracle_residual_weights.argtypes = [P, P, i32, P]
            L.oracle_tree_sample.argtypes = [P, i32, u64, ctypes.c_uint32, ctypes.c_uint32, P]
            L.oracle_tree_sample.restype = i32
            L.oracle_draft_markov.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, i32, u64, P, dbl,
                                              P, P, P, P, P, i32]
            L.oracle_draft_markov.restype = i32
            L.oracle_draft_rnn.argtypes = [P, i32, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32,
                                           u64, P, dbl, P, P, P, P, P, P, i32]
            L.oracle_draft_rnn.restype = i32
            L.oracle_verify.argtypes = [P, i32, P, i32, P, i32, P, P, P, P, P, i32, i32, i32, i32,
                                        u64, P, dbl, P, P, P, P, P, P, P, i32]
            L.oracle_verify.restype = i32
            L.oracle_prefix_survival.argtypes = [P, i32, i32, P]
            L.oracle_confidence.argtypes = [P, i32, P, i32, P, P, P, i32, i32, i32, i32, i32, P, P]
            L.oracle_confidence.restype = i32
            L.oracle_threshold_lengths.argtypes = [P, i32, i32, ctypes.c_float, i32, P]
            L.oracle_threshold_lengths.restype = i32
            L.oracle_ece.argtypes = [P, P, i32, i32]
            L.oracle_ece.restype = dbl
            L.oracle_sts_fit.argtypes = [P, P, i32, i32, P, i32, i32, P, P, P, P]
            L.oracle_sts_fit.restype = i32
            L.oracle_sts_apply.argtypes = [P, i32, i32, P, P]
            L.oracle_schedule_loop.argtypes = [P, P, i32, i32, i32, P, P]
            L.oracle_schedule_loop.restype = i32
            L.oracle_schedule_closed.argtypes = [P, P, i32, i32, i32, P, P, P]
            L.oracle_schedule_closed.restype = i32
            L.oracle_schedule_budget.argtypes = [P, P, i32, i32, i32, i32, P, P, P]
            L.oracle_schedule_budget.restype = i32
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"storage dtype must be float32 or uint16 (bf16), got {a.dtype}")


def _c(a, dtype=None):
    return np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------- RNG
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(word: int) -> float:
    return lib().oracle_uniform(int(word) & 0xFFFFFFFF)


def rng_uniform(seed: int, req: int, pos: int, stream: int, v: int) -> float:
    return lib().oracle_rng_uniform(int(seed), int(req), int(pos), int(stream), int(v))


# ---------------------------------------------------------------- section 05 helpers
def accept_prob(px: float, qx: float) -> float:
    return lib().oracle_accept_prob(float(px), float(qx))


def residual_weights(p, q) -> np.ndarray:
    p = _c(p, np.float64)
    q = _c(q, np.float64)
    w = np.zeros_like(p)
    lib().oracle_residual_weights(_ptr(p), _ptr(q), int(p.size), _ptr(w))
    return w


def tree_sample(w, seed: int, req: int, pos: int):
    w = _c(w, np.float64)
    gap = np.zeros(1, dtype=np.float64)
    y = lib().oracle_tree_sample(_ptr(w), int(w.size), int(seed), int(req), int(pos), _ptr(gap))
    return int(y), float(gap[0])


# ---------------------------------------------------------------- draft
def draft_markov(U, anchor, W1, W2, T: float, seed: int, req_ids=None, n_threads=None):
    U = _c(U)
    W1 = _c(W1)
    W2 = _c(W2)
    anchor = _c(anchor, np.int32)
    R, gamma, V = U.shape
    r = W1.shape[1]
    assert W1.shape == (V, r) and W2.shape == (r, V) and anchor.shape == (R,)
    if _dt(W1) != _dt(W2):
        raise TypeError("W1 and W2 must share a storage dtype")
    rid = None if req_ids is None else _c(req_ids, np.uint32)
    out = dict(tokens=np.zeros((R, gamma), np.int32), qx=np.zeros((R, gamma)), lse=np.zeros((R, gamma)),
               code=np.zeros((R, gamma, r)), margin=np.zeros((R, gamma)))
    st = lib().oracle_draft_markov(_ptr(U), _dt(U), _ptr(anchor), _ptr(W1), _ptr(W2), _dt(W1),
                                   R, gamma, V, r, int(seed), _ptr(rid), float(T),
                                   _ptr(out["tokens"]), _ptr(out["qx"]), _ptr(out["lse"]), _ptr(out["code"]),
                                   _ptr(out["margin"]), int(n_threads or default_threads()))
    if st != 0:
        raise RuntimeError(f"oracle_draft_markov failed: {st}")
    return out


def draft_rnn(U, anchor, W1, W2, Wgco, H, T: float, seed: int, req_ids=None, n_threads=None):
    U, W1, W2, Wgco, H = (_c(a) for a in (U, W1, W2, Wgco, H))
    anchor = _c(anchor, np.int32)
    R, gamma, V = U.shape
    r = W1.shape[1]
    d = H.shape[2]
    assert Wgco.shape == (2 * r + d, 3 * r) and H.shape[:2] == (R, gamma)
    if not (_dt(W1) == _dt(W2) == _dt(Wgco)):
        raise TypeError("W1, W2 and Wgco must share a storage dtype")
    rid = None if req_ids is None else _c(req_ids, np.uint32)
    out = dict(tokens=np.zeros((R, gamma), np.int32), qx=np.zeros((R, gamma)), lse=np.zeros((R, gamma)),
               code=np.zeros((R, gamma, r)), margin=np.zeros((R, gamma)), state=np.zeros((R, r)))
    st = lib().oracle_draft_rnn(_ptr(U), _dt(U), _ptr(anchor), _ptr(W1), _ptr(W2), _ptr(Wgco), _dt(W1),
                                _ptr(H), _dt(H), R, gamma, V, r, d, int(seed), _ptr(rid), float(T),
                                _ptr(out["tokens"]), _ptr(out["qx"]), _ptr(out["lse"]), _ptr(out["code"]),
                                _ptr(out["margin"]), _ptr(out["state"]), int(n_threads or default_threads()))
    if st != 0:
        raise RuntimeError(f"oracle_draft_rnn failed: {st}")
    return out


# ---------------------------------------------------------------- verify
def verify(P, U, W2, tokens, qx, lse, code, T: float, seed: int, verify_len=None, req_ids=None,
           n_threads=None):
    P, U, W2 = _c(P), _c(U), _c(W2)
    tokens = _c(tokens, np.int32)
    qx = _c(qx, np.float64)
    lse = _c(lse, np.float64)
    code = _c(code, np.float64)
    R, gamma, V = U.shape
    r = W2.shape[0]
    assert P.shape == (R, gamma + 1, V) and tokens.shape == (R, gamma) and code.shape == (R, gamma, r)
    vl = None if verify_len is None else _c(verify_len, np.int32)
    rid = None if req_ids is None else _c(req_ids, np.uint32)
    out = dict(out_tokens=np.zeros((R, gamma + 1), np.int32), accept_len=np.zeros(R, np.int32),
               n_out=np.zeros(R, np.int32), px=np.zeros((R, gamma)), lse_p=np.zeros((R, gamma + 1)),
               min_gap=np.zeros(R), gap_kind=np.zeros(R, np.int32))
    st = lib().oracle_verify(_ptr(P), _dt(P), _ptr(U), _dt(U), _ptr(W2), _dt(W2),
                             _ptr(tokens), _ptr(qx), _ptr(lse), _ptr(code), _ptr(vl),
                             R, gamma, V, r, int(seed), _ptr(rid), float(T),
                             _ptr(out["out_tokens"]), _ptr(out["accept_len"]), _ptr(out["n_out"]),
                             _ptr(out["px"]), _ptr(out["lse_p"]), _ptr(out["min_gap"]), _ptr(out["gap_kind"]),
                             int(n_threads or default_threads()))
    if st != 0:
        raise RuntimeError(f"oracle_verify failed: {st}")
    return out


# ---------------------------------------------------------------- confidence head
def confidence(H, W1, w, anchor, tokens, temps=None):
    """c [R, gamma] (double) = sigmoid(w . [h_k, W1[x_{k-1}]]) (blog section 4.1).
    H [R, gamma, d] and W1 [V, r] in storage dtype, w [d + r] float32,
    anchor [R] = x_0, tokens [R, gamma] = the drafted x_1..x_gamma; temps
    [gamma] (optional): per-position temperatures, sigmoid(logit / t_k)."""
    H, W1 = _c(H), _c(W1)
    w = _c(w, np.float32)
    anchor = _c(anchor, np.int32)
    tokens = _c(tokens, np.int32)
    R, gamma, d = H.shape
    V, r = W1.shape
    assert w.shape == (d + r,) and anchor.shape == (R,) and tokens.shape == (R, gamma)
    c = np.zeros((R, gamma))
    tt = None if temps is None else _c(temps, np.float64)
    st = lib().oracle_confidence(_ptr(H), _dt(H), _ptr(W1), _dt(W1), _ptr(w), _ptr(anchor), _ptr(tokens),
                                 R, gamma, V, d, r, _ptr(tt), _ptr(c))
    if st != 0:
        raise RuntimeError(f"oracle_confidence failed: {st}")
    return c


# ---------------------------------------------------------------- scheduler
def prefix_survival(c) -> np.ndarray:
    c = _c(c, np.float32)
    a = np.zeros_like(c)
    lib().oracle_prefix_survival(_ptr(c), c.shape[0], c.shape[1], _ptr(a))
    return a


def schedule_loop(c, sps):
    c = _c(c, np.float32)
    sps = _c(sps, np.float64)
    R, gamma = c.shape
    L = np.zeros(R, np.int32)
    th = np.zeros(1)
    n = lib().oracle_schedule_loop(_ptr(c), _ptr(sps), int(sps.size), R, gamma, _ptr(L), _ptr(th))
    if n < 0:
        raise RuntimeError("oracle_schedule_loop failed")
    return L, float(th[0]), int(n)


def schedule_closed(c, sps):
    c = _c(c, np.float32)
    sps = _c(sps, np.float64)
    R, gamma = c.shape
    L = np.zeros(R, np.int32)
    th = np.zeros(1)
    gap = np.zeros(1)
    n = lib().oracle_schedule_closed(_ptr(c), _ptr(sps), int(sps.size), R, gamma, _ptr(L), _ptr(th), _ptr(gap))
    if n < 0:
        raise RuntimeError("oracle_schedule_closed failed")
    return L, float(th[0]), int(n), float(gap[0])


def threshold_lengths(c, theta: float, mode: int = 0):
    """Per-request verify lengths of the threshold filter: the longest prefix
    with a_{r,j} >= theta (mode 0) or c_{r,j} >= theta (mode 1)."""
    c = _c(c, np.float32)
    R, gamma = c.shape
    L = np.zeros(R, np.int32)
    st = lib().oracle_threshold_lengths(_ptr(c), R, gamma, float(np.float32(theta)), int(mode), _ptr(L))
    if st != 0:
        raise RuntimeError(f"oracle_threshold_lengths failed: {st}")
    return L


# ---------------------------------------------------------------- STS
def ece(pred, y, M: int) -> float:
    """Expected calibration error over M equal-width bins (Guo et al. 2017)."""
    pred = _c(pred, np.float64)
    y = _c(y, np.int32)
    return float(lib().oracle_ece(_ptr(pred), _ptr(y), int(pred.size), int(M)))


def sts_fit(c, accept_len, grid, M: int = 15):
    """Sequential Temperature Scaling (blog section 4.2).  c [N, gamma] raw
    confidences (float32), accept_len [N] accepted drafts per block, grid [G]
    candidate temperatures.  Returns dict(t, g, ece, gap), one entry per position."""
    c = _c(c, np.float32)
    al = _c(accept_len, np.int32)
    grid = _c(grid, np.float64)
    N, gamma = c.shape
    out = dict(t=np.zeros(gamma), g=np.zeros(gamma, np.int32), ece=np.zeros(gamma), gap=np.zeros(gamma))
    st = lib().oracle_sts_fit(_ptr(c), _ptr(al), N, gamma, _ptr(grid), int(grid.size), int(M),
                              _ptr(out["t"]), _ptr(out["g"]), _ptr(out["ece"]), _ptr(out["gap"]))
    if st != 0:
        raise RuntimeError(f"oracle_sts_fit failed: {st}")
    return out


def sts_apply(c, t):
    """c'[n, k] = sigmoid(logit(c[n, k]) / t[k])."""
    c = _c(c, np.float32)
    t = _c(t, np.float64)
    out = np.zeros(c.shape)
    lib().oracle_sts_apply(_ptr(c), c.shape[0], c.shape[1], _ptr(t), _ptr(out))
    return out


def schedule_budget(c, sps, budget: int):
    """Production-style scheduler: the capacity (budget) decided two steps
    back, the current candidates ranked into it.  Returns (lengths, theta,
    places filled, this step's synchronous n*)."""
    c = _c(c, np.float32)
    sps = _c(sps, np.float64)
    R, gamma = c.shape
    L = np.zeros(R, np.int32)
    th = np.zeros(1)
    ns = np.zeros(1, np.int32)
    n = lib().oracle_schedule_budget(_ptr(c), _ptr(sps), int(sps.size), R, gamma, int(budget), _ptr(L), _ptr(th),
                                     _ptr(ns))
    if n < 0:
        raise RuntimeError("oracle_schedule_budget failed")
    return L, float(th[0]), int(n), int(ns[0])
