"""Thin Python binding of libdspark.so (ctypes; argument marshalling only).

Every function takes CUDA torch tensors, passes their device pointers and the
current CUDA stream to the C ABI of ``include/dspark.h`` and returns the
output tensors it allocated.  All arithmetic of the cycle runs in the
library's kernels; this module only checks types, allocates outputs and the
workspace, and translates status codes into exceptions.  There is no CPU
fallback: if the library cannot be loaded, importing a function raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

F32 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None

STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported dtype", -3: "unsupported sizes",
          -4: "CUDA runtime error", -5: "bounded device wait ran out", -6: "token id outside [0, V)",
          -7: "not implemented", -8: "workspace null, misaligned or too small"}


class DsparkError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed with status {code} ({STATUS.get(code, 'unknown')})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libdspark.so (building it first if asked); raises if unavailable."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libdspark.so not found at {path}; run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        P, i32, u64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
        L.dspark_strerror.argtypes = [i32]
        L.dspark_strerror.restype = ctypes.c_char_p
        L.dspark_version.restype = ctypes.c_char_p
        L.dspark_workspace_status.argtypes = [P, P]
        L.dspark_host_pointer.argtypes = [P, P]
        L.dspark_host_pointer.restype = i32
        L.dspark_draft_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.dspark_draft_workspace_size.restype = sz
        L.dspark_draft_markov.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, i32, u64, P, f32,
                                          P, P, P, P, P, sz, P]
        L.dspark_draft_rnn.argtypes = [P, i32, P, P, P, P, i32, P, i32, i32, i32, i32, i32, u64, P, f32,
                                       P, P, P, P, P, P, sz, P]
        L.dspark_verify_workspace_size.argtypes = [i32, i32, i32, i32]
        L.dspark_verify_workspace_size.restype = sz
        L.dspark_verify.argtypes = [P, i32, P, i32, P, i32, P, P, P, P, P, i32, i32, i32, i32, u64, P, f32,
                                    P, P, P, P, P, P, sz, P]
        L.dspark_verify_staged.argtypes = [P, i32, P, i32, P, i32, P, P, P, P, P, i32, i32, i32, i32, u64, P, f32,
                                           P, P, P, P, P, P, P, sz, P]
        L.dspark_schedule_workspace_size.argtypes = [i32, i32]
        L.dspark_schedule_workspace_size.restype = sz
        L.dspark_draft_markov_conf.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, i32, u64, P, f32,
                                               P, P, P, P, P, P, sz, P]
        L.dspark_draft_rnn_conf.argtypes = [P, i32, P, P, P, P, i32, P, i32, i32, i32, i32, i32, u64, P, f32,
                                            P, P, P, P, P, P, P, sz, P]
        L.dspark_schedule.argtypes = [P, P, i32, i32, i32, P, P, P, P, sz, P]
        L.dspark_schedule_async.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, sz, P]
        L.dspark_schedule_threshold.argtypes = [P, i32, i32, f32, i32, P, P]
        L.dspark_sts_workspace_size.argtypes = [i32, i32, i32, i32]
        L.dspark_sts_workspace_size.restype = sz
        L.dspark_sts_fit.argtypes = [P, P, i32, i32, P, i32, i32, P, P, P, P, P, sz, P]
        L.dspark_sts_apply.argtypes = [P, i32, i32, P, P, P]
        L.dspark_philox4x32_10.argtypes = [P, P, P, i32, P]
        L.dspark_workspace_set_wait.argtypes = [P, u64, i32, P]
        L.dspark_profile_enable.argtypes = [i32]
        L.dspark_profile_collect.argtypes = [P, P, i32]
        L.dspark_profile_kernel_name.argtypes = [i32]
        L.dspark_profile_kernel_name.restype = ctypes.c_char_p
        for name in ("dspark_draft_markov", "dspark_draft_rnn", "dspark_draft_markov_conf", "dspark_draft_rnn_conf",
                     "dspark_verify", "dspark_verify_staged", "dspark_schedule", "dspark_schedule_async",
                     "dspark_schedule_threshold",
                     "dspark_sts_fit",
                     "dspark_sts_apply", "dspark_philox4x32_10", "dspark_workspace_set_wait",
                     "dspark_workspace_status", "dspark_profile_enable", "dspark_profile_collect"):
            getattr(L, name).restype = i32
        _lib = L
        return _lib


class DeviceView:
    """A device-accessible address with a shape and a dtype, passed where the
    calls take a CUDA tensor: for example a pinned host buffer read in place
    (``host_view``)."""

    is_cuda = True

    def __init__(self, ptr: int, shape, dtype, device, owner=None):
        self.ptr, self.shape, self.dtype, self.device, self.owner = int(ptr), tuple(shape), dtype, device, owner

    def data_ptr(self) -> int:
        return self.ptr

    def is_contiguous(self) -> bool:
        return True

    def numel(self) -> int:
        n = 1
        for d in self.shape:
            n *= d
        return n


def host_view(t: torch.Tensor, device) -> DeviceView:
    """A pinned host tensor as a DeviceView its kernels read in place
    (``dspark_host_pointer``); raises if the memory is not pinned and mapped."""
    if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
        raise ValueError("host_view takes a contiguous pinned host tensor")
    out = ctypes.c_void_p()
    code = load().dspark_host_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(out))
    _check("dspark_host_pointer", code)
    return DeviceView(out.value, t.shape, t.dtype, device, owner=t)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libdspark takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libdspark takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"storage dtype must be float32 or bfloat16, got {t.dtype}")


def _shape(name: str, t, shape, dtype=None):
    """The C ABI takes bare pointers and cannot see sizes: a tensor of the
    wrong shape would be read or written past its end on the device, so the
    binding checks every shape (and the dtype where it is fixed) first."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, code: int):
    if code != 0:
        raise DsparkError(fn, code)


class _Conf(ctypes.Structure):
    """dspark_conf_t: the confidence head's arguments."""
    _fields_ = [("H", ctypes.c_void_p), ("w", ctypes.c_void_p), ("d", ctypes.c_int), ("c", ctypes.c_void_p),
                ("t", ctypes.c_void_p)]


def _conf(conf_w, conf_H, out, R, gamma, dev, conf_t=None):
    """Fill out["c"] and return a dspark_conf_t pointer (None: head off)."""
    if conf_w is None:
        return None, None
    if conf_w.dtype != torch.float32:
        raise TypeError("confidence weights must be float32")
    if conf_H is not None and conf_H.dtype != torch.bfloat16:
        raise TypeError("confidence-head H must be bfloat16")
    if "c" not in out:
        out["c"] = torch.empty((R, gamma), dtype=torch.float32, device=dev)
    if conf_t is not None and conf_t.dtype != torch.float64:
        raise TypeError("per-position temperatures must be float64")
    st = _Conf(_p(conf_H), _p(conf_w), 0 if conf_H is None else conf_H.shape[2], _p(out["c"]), _p(conf_t))
    return st, ctypes.byref(st)


def _workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks; the first
    # word (the device status word) must start at zero.
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def version() -> str:
    return load().dspark_version().decode()


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    return load().dspark_workspace_status(_p(ws), _stream(stream))


def workspace_set_wait(ws: torch.Tensor, limit_cycles: int = 0, test_withhold: int = 0, stream=None) -> None:
    """Bounded-wait limit (SM cycles, 0 = the default 2^32) and the test hook
    of the calls that use workspace ``ws`` (``dspark_workspace_set_wait``)."""
    code = load().dspark_workspace_set_wait(_p(ws), int(limit_cycles), int(test_withhold), _stream(stream))
    _check("dspark_workspace_set_wait", code)


def draft_workspace_bytes(R, gamma, V, r, d=0) -> int:
    return int(load().dspark_draft_workspace_size(R, gamma, V, r, d))


def verify_workspace_bytes(R, gamma, V, r) -> int:
    return int(load().dspark_verify_workspace_size(R, gamma, V, r))


def schedule_workspace_bytes(R, gamma) -> int:
    return int(load().dspark_schedule_workspace_size(R, gamma))


def _draft_shapes(R, gamma, V, r, anchor, W1, W2, req_ids):
    _shape("anchor", anchor, (R,), torch.int32)
    _shape("W1", W1, (V, r))
    _shape("W2", W2, (r, V))
    _shape("req_ids", req_ids, (R,))


def _draft_out_shapes(out, R, gamma, r):
    _shape("tokens", out["tokens"], (R, gamma), torch.int32)
    _shape("q_tok", out["q_tok"], (R, gamma), torch.float32)
    _shape("lse", out["lse"], (R, gamma), torch.float64)
    _shape("code", out["code"], (R, gamma, r), torch.float32)


def draft_markov(U, anchor, W1, W2, temperature: float, seed: int, req_ids=None, ws=None, out=None, stream=None,
                 conf_w=None, conf_H=None, conf_t=None):
    """Markov-head drafting (``dspark_draft_markov``).  Returns a dict of outputs.
    With ``conf_w`` ([d + r] float32) and ``conf_H`` ([R, gamma, d] bfloat16)
    the fused confidence head (``dspark_draft_markov_conf``) adds ``c``."""
    L = load()
    R, gamma, V = U.shape
    r = W1.shape[1]
    dev = U.device
    _draft_shapes(R, gamma, V, r, anchor, W1, W2, req_ids)
    if out is None:
        out = dict(tokens=torch.empty((R, gamma), dtype=torch.int32, device=dev),
                   q_tok=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                   lse=torch.empty((R, gamma), dtype=torch.float64, device=dev),
                   code=torch.empty((R, gamma, r), dtype=torch.float32, device=dev))
    _draft_out_shapes(out, R, gamma, r)
    nbytes = L.dspark_draft_workspace_size(R, gamma, V, r, 0)
    if ws is None:
        ws = _workspace(nbytes, dev)
    keep, cp = _conf(conf_w, conf_H, out, R, gamma, dev, conf_t)
    code = L.dspark_draft_markov_conf(_p(U), _dt(U), _p(anchor), _p(W1), _p(W2), _dt(W1), R, gamma, V, r,
                                      int(seed) & 0xFFFFFFFFFFFFFFFF, _p(req_ids), float(temperature),
                                      _p(out["tokens"]), _p(out["q_tok"]), _p(out["lse"]), _p(out["code"]),
                                      cp, _p(ws), ws.numel(), _stream(stream))
    _check("dspark_draft_markov", code)
    out["ws"] = ws
    return out


def draft_rnn(U, anchor, W1, W2, Wgco, H, temperature: float, seed: int, req_ids=None, ws=None, out=None,
              stream=None, conf_w=None, conf_H=None, conf_t=None):
    """RNN-head drafting (``dspark_draft_rnn``).  With ``conf_w`` the fused
    confidence head adds ``c`` (``conf_H`` None: the head's own H)."""
    L = load()
    R, gamma, V = U.shape
    r = W1.shape[1]
    d = H.shape[2]
    dev = U.device
    if H.dtype != torch.bfloat16:
        raise TypeError("H must be bfloat16")
    _draft_shapes(R, gamma, V, r, anchor, W1, W2, req_ids)
    _shape("Wgco", Wgco, (2 * r + d, 3 * r))
    _shape("H", H, (R, gamma, d))
    if out is None:
        out = dict(tokens=torch.empty((R, gamma), dtype=torch.int32, device=dev),
                   q_tok=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                   lse=torch.empty((R, gamma), dtype=torch.float64, device=dev),
                   code=torch.empty((R, gamma, r), dtype=torch.float32, device=dev),
                   state=torch.empty((R, r), dtype=torch.float32, device=dev))
    _draft_out_shapes(out, R, gamma, r)
    _shape("state", out.get("state"), (R, r), torch.float32)
    nbytes = L.dspark_draft_workspace_size(R, gamma, V, r, d)
    if ws is None:
        ws = _workspace(nbytes, dev)
    keep, cp = _conf(conf_w, conf_H, out, R, gamma, dev, conf_t)
    code = L.dspark_draft_rnn_conf(_p(U), _dt(U), _p(anchor), _p(W1), _p(W2), _p(Wgco), _dt(W1), _p(H), d,
                                   R, gamma, V, r, int(seed) & 0xFFFFFFFFFFFFFFFF, _p(req_ids), float(temperature),
                                   _p(out["tokens"]), _p(out["q_tok"]), _p(out["lse"]), _p(out["code"]),
                                   _p(out.get("state")), cp, _p(ws), ws.numel(), _stream(stream))
    _check("dspark_draft_rnn", code)
    out["ws"] = ws
    return out


def verify(P, U, W2, draft, temperature: float, seed: int, verify_len=None, req_ids=None, ws=None, out=None,
           stream=None, p_stage=None):
    """Rejection-sampling verification (``dspark_verify``); ``draft`` is a draft output dict.
    ``p_stage`` (a device tensor of P's shape and dtype) receives the target
    rows pass 1 reads, for the later passes (``dspark_verify_staged``)."""
    L = load()
    R, G1, V = P.shape
    gamma = G1 - 1
    r = W2.shape[0]
    dev = P.device
    _shape("W2", W2, (r, V))
    if float(temperature) > 0.0:
        _shape("U", U, (R, gamma, V))
    _shape("draft tokens", draft["tokens"], (R, gamma), torch.int32)
    _shape("draft q_tok", draft.get("q_tok"), (R, gamma), torch.float32)
    _shape("draft lse", draft.get("lse"), (R, gamma), torch.float64)
    _shape("draft code", draft.get("code"), (R, gamma, r), torch.float32)
    _shape("verify_len", verify_len, (R,), torch.int32)
    _shape("req_ids", req_ids, (R,))
    if p_stage is not None:
        _shape("p_stage", p_stage, (R, G1, V), P.dtype)
    if out is None:
        out = dict(out_tokens=torch.empty((R, G1), dtype=torch.int32, device=dev),
                   accept_len=torch.empty((R,), dtype=torch.int32, device=dev),
                   n_out=torch.empty((R,), dtype=torch.int32, device=dev),
                   p_tok=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                   lse_p=torch.empty((R, G1), dtype=torch.float64, device=dev))
    _shape("out_tokens", out["out_tokens"], (R, G1), torch.int32)
    _shape("accept_len", out["accept_len"], (R,), torch.int32)
    _shape("n_out", out["n_out"], (R,), torch.int32)
    _shape("p_tok", out.get("p_tok"), (R, gamma), torch.float32)
    _shape("lse_p", out.get("lse_p"), (R, G1), torch.float64)
    nbytes = L.dspark_verify_workspace_size(R, gamma, V, r)
    if ws is None:
        ws = _workspace(nbytes, dev)
    code = L.dspark_verify_staged(_p(P), _dt(P), _p(U), _dt(U), _p(W2), _dt(W2), _p(draft["tokens"]),
                                  _p(draft["q_tok"]), _p(draft["lse"]), _p(draft["code"]), _p(verify_len),
                                  R, gamma, V, r, int(seed) & 0xFFFFFFFFFFFFFFFF, _p(req_ids), float(temperature),
                                  _p(out["out_tokens"]), _p(out["accept_len"]), _p(out["n_out"]),
                                  _p(out.get("p_tok")), _p(out.get("lse_p")), _p(p_stage), _p(ws), ws.numel(),
                                  _stream(stream))
    _check("dspark_verify", code)
    out["ws"] = ws
    return out


def schedule(c, sps, ws=None, out=None, stream=None, budget=None):
    """Confidence scheduler (``dspark_schedule``): verify lengths, Theta*, n*.
    With ``budget`` (an int32 [1] device tensor: the n_star of two steps back)
    the production-style rule (``dspark_schedule_async``)."""
    L = load()
    R, gamma = c.shape
    dev = c.device
    if out is None:
        out = dict(verify_len=torch.empty((R,), dtype=torch.int32, device=dev),
                   theta=torch.empty((1,), dtype=torch.float64, device=dev),
                   n_star=torch.empty((1,), dtype=torch.int32, device=dev))
    if ws is None:
        ws = _workspace(L.dspark_schedule_workspace_size(R, gamma), dev)
    if budget is None:
        code = L.dspark_schedule(_p(c), _p(sps), sps.numel(), R, gamma, _p(out["verify_len"]), _p(out["theta"]),
                                 _p(out["n_star"]), _p(ws), ws.numel(), _stream(stream))
        _check("dspark_schedule", code)
    else:
        if budget.dtype != torch.int32:
            raise TypeError("budget must be int32")
        code = L.dspark_schedule_async(_p(c), _p(sps), sps.numel(), R, gamma, _p(budget), _p(out["verify_len"]),
                                       _p(out["theta"]), _p(out["n_star"]), _p(ws), ws.numel(), _stream(stream))
        _check("dspark_schedule_async", code)
    out["ws"] = ws
    return out


def schedule_threshold(c, theta: float, mode: int = 0, out=None, stream=None):
    """Threshold filter (``dspark_schedule_threshold``): per-request verify
    lengths, the longest prefix with a_{r,j} >= theta (mode 0) or
    c_{r,j} >= theta (mode 1)."""
    L = load()
    R, gamma = c.shape
    if out is None:
        out = torch.empty((R,), dtype=torch.int32, device=c.device)
    code = L.dspark_schedule_threshold(_p(c), R, gamma, float(theta), int(mode), _p(out), _stream(stream))
    _check("dspark_schedule_threshold", code)
    return out


def sts_fit(c, accept_len, grid, M: int = 15, ws=None, out=None, stream=None):
    """Sequential Temperature Scaling (``dspark_sts_fit``): per-position
    temperatures t, grid indices g, minimum ECE and the gap to the second."""
    L = load()
    N, gamma = c.shape
    G = grid.numel()
    dev = c.device
    if grid.dtype != torch.float64 or accept_len.dtype != torch.int32:
        raise TypeError("grid must be float64 and accept_len int32")
    if out is None:
        out = dict(t=torch.empty((gamma,), dtype=torch.float64, device=dev),
                   g=torch.empty((gamma,), dtype=torch.int32, device=dev),
                   ece=torch.empty((gamma,), dtype=torch.float64, device=dev),
                   gap=torch.empty((gamma,), dtype=torch.float64, device=dev))
    if ws is None:
        ws = _workspace(L.dspark_sts_workspace_size(N, gamma, G, M), dev)
    code = L.dspark_sts_fit(_p(c), _p(accept_len), N, gamma, _p(grid), G, M, _p(out["t"]), _p(out["g"]),
                            _p(out["ece"]), _p(out["gap"]), _p(ws), ws.numel(), _stream(stream))
    _check("dspark_sts_fit", code)
    out["ws"] = ws
    return out


def sts_apply(c, t, out=None, stream=None):
    """out = sigmoid(logit(c) / t[k]) per position (``dspark_sts_apply``)."""
    L = load()
    N, gamma = c.shape
    if out is None:
        out = torch.empty_like(c)
    code = L.dspark_sts_apply(_p(c), N, gamma, _p(t), _p(out), _stream(stream))
    _check("dspark_sts_apply", code)
    return out


def philox4x32_10(ctr, key, out=None, stream=None):
    """The device's Philox4x32-10 block function on n counters ``ctr`` [n, 4]
    and keys ``key`` [n, 2] (uint32 values in int32 CUDA tensors, bit for
    bit); returns out [n, 4] (``dspark_philox4x32_10``)."""
    L = load()
    n = ctr.shape[0]
    _shape("ctr", ctr, (n, 4), torch.int32)
    _shape("key", key, (n, 2), torch.int32)
    if out is None:
        out = torch.empty((n, 4), dtype=torch.int32, device=ctr.device)
    _shape("out", out, (n, 4), torch.int32)
    code = L.dspark_philox4x32_10(_p(ctr), _p(key), _p(out), n, _stream(stream))
    _check("dspark_philox4x32_10", code)
    return out


def profile_enable(on: bool = True) -> None:
    """Bracket every library launch with CUDA events (benchmark timing)."""
    load().dspark_profile_enable(1 if on else 0)


def profile_collect(cap: int = 1 << 16):
    """Per launch since the last collect: list of (kernel name, milliseconds)."""
    import numpy as np
    L = load()
    ids = np.zeros(cap, np.int32)
    ms = np.zeros(cap, np.float32)
    n = L.dspark_profile_collect(ctypes.c_void_p(ids.ctypes.data), ctypes.c_void_p(ms.ctypes.data), cap)
    if n < 0:
        raise DsparkError("dspark_profile_collect", n)
    n = min(n, cap)
    return [(L.dspark_profile_kernel_name(int(i)).decode(), float(t)) for i, t in zip(ids[:n], ms[:n])]
