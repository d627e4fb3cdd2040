"""The C ABI library builds, loads and exports every entry point that
include/dspark.h declares; host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest

from speculative_decoding_drafting_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "dspark.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_calls():
    syms = declared_symbols()
    for name in ("dspark_draft_markov", "dspark_draft_rnn", "dspark_verify", "dspark_schedule"):
        assert name in syms


def test_library_exports_every_declared_symbol():
    path = _build.build()
    lib = ctypes.CDLL(path)
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_host_only_calls():
    L = binding.load()
    assert b"sm_103a" in L.dspark_version()
    assert L.dspark_strerror(-6) == b"token id outside [0, V)"
    assert binding.draft_workspace_bytes(256, 5, 151936, 256) > 0
    assert binding.draft_workspace_bytes(0, 5, 151936, 256) == 0
    assert binding.verify_workspace_bytes(256, 5, 151936, 256) > 0
    assert binding.schedule_workspace_bytes(512, 16) > 0
    assert binding.schedule_workspace_bytes(1024, 16) == 0          # R * gamma above 8192


def test_invalid_arguments_rejected_before_any_device_work():
    L = binding.load()
    null = None
    # null inputs
    st = L.dspark_draft_markov(null, 0, null, null, null, 1, 4, 5, 4096, 32, 0, null, 1.0,
                               null, null, null, null, null, 0, null)
    assert st == -1
    # unsupported dtype / sizes
    assert L.dspark_draft_markov(null, 7, null, null, null, 1, 4, 5, 4096, 32, 0, null, 1.0,
                                 null, null, null, null, null, 0, null) == -2
    assert L.dspark_draft_markov(null, 0, null, null, null, 1, 4, 5, 4099, 32, 0, null, 1.0,
                                 null, null, null, null, null, 0, null) == -3
    assert L.dspark_verify(null, 0, null, 0, null, 1, null, null, null, null, null, 4, 0, 4096, 32, 0, null,
                           1.0, null, null, null, null, null, null, 0, null) == -3
    # the vocabulary stays within 2^20, sampled or greedy
    big = (1 << 20) + 8
    for t in (1.0, 0.0):
        assert L.dspark_verify(null, 0, null, 0, null, 1, null, null, null, null, null, 4, 5, big, 32, 0, null,
                               t, null, null, null, null, null, null, 0, null) == -3
        assert L.dspark_verify(null, 0, null, 0, null, 1, null, null, null, null, null, 4, 5, 1 << 20, 32, 0,
                               null, t, null, null, null, null, null, null, 0, null) == -1
    assert L.dspark_schedule(null, null, 10, 4, 5, null, null, null, null, 0, null) == -1
    assert L.dspark_schedule(null, null, 10, 1000, 16, null, null, null, null, 0, null) == -3


def test_confidence_head_and_threshold_arguments_rejected_on_the_host():
    L = binding.load()
    null = None
    fake = ctypes.c_void_p(4096)   # never dereferenced: every call below fails its host checks

    def markov_conf(conf):
        return L.dspark_draft_markov_conf(null, 0, null, null, null, 1, 4, 5, 4096, 32, 0, null, 1.0,
                                          null, null, null, null, conf, null, 0, null)

    # null weights or output
    assert markov_conf(ctypes.byref(binding._Conf(fake, None, 8, fake))) == -1
    assert markov_conf(ctypes.byref(binding._Conf(fake, fake, 8, None))) == -1
    # d out of range; Markov head without H but d > 0
    assert markov_conf(ctypes.byref(binding._Conf(fake, fake, 16385, fake))) == -3
    assert markov_conf(ctypes.byref(binding._Conf(None, fake, 8, fake))) == -1
    # a valid head still needs the draft's own inputs
    assert markov_conf(ctypes.byref(binding._Conf(fake, fake, 8, fake))) == -1
    assert markov_conf(None) == -1
    st = L.dspark_draft_rnn_conf(null, 0, null, null, null, null, 1, null, 16, 4, 5, 4096, 32, 0, null, 1.0,
                                 null, null, null, null, null, ctypes.byref(binding._Conf(None, None, 0, fake)),
                                 null, 0, null)
    assert st == -1
    # threshold filter: mode, sizes, null pointers
    assert L.dspark_schedule_threshold(fake, 4, 5, ctypes.c_float(0.5), 2, fake, null) == -1
    assert L.dspark_schedule_threshold(fake, 4, 65, ctypes.c_float(0.5), 0, fake, null) == -3
    assert L.dspark_schedule_threshold(fake, 0, 5, ctypes.c_float(0.5), 0, fake, null) == -3
    assert L.dspark_schedule_threshold(null, 4, 5, ctypes.c_float(0.5), 0, fake, null) == -1


def test_sts_arguments_rejected_on_the_host():
    L = binding.load()
    null = None
    fake = ctypes.c_void_p(4096)   # never dereferenced: every call below fails its host checks
    assert L.dspark_sts_workspace_size(65536, 8, 256, 15) > 0
    for bad in [(0, 8, 256, 15), (10, 0, 256, 15), (10, 65, 256, 15), (10, 8, 0, 15), (10, 8, 4097, 15),
                (10, 8, 256, 0), (10, 8, 256, 33), ((1 << 24) + 1, 8, 256, 15)]:
        assert L.dspark_sts_workspace_size(*bad) == 0
    fit = lambda c, al, N, g, grid, G, M, out, ws, wsb: L.dspark_sts_fit(  # noqa: E731
        c, al, N, g, grid, G, M, out, out, out, out, ws, wsb, null)
    assert fit(fake, fake, 10, 8, fake, 256, 33, fake, fake, 1 << 20) == -3
    assert fit(null, fake, 10, 8, fake, 256, 15, fake, fake, 1 << 20) == -1
    assert fit(fake, fake, 10, 8, fake, 256, 15, null, fake, 1 << 20) == -1
    assert fit(fake, fake, 10, 8, fake, 256, 15, fake, null, 1 << 20) == -8
    assert fit(fake, fake, 10, 8, fake, 256, 15, fake, ctypes.c_void_p(4096 + 8), 1 << 20) == -8   # misaligned
    assert fit(fake, fake, 10, 8, fake, 256, 15, fake, fake, 64) == -8                            # too small
    assert L.dspark_sts_apply(fake, 0, 8, fake, fake, null) == -3
    assert L.dspark_sts_apply(fake, 10, 65, fake, fake, null) == -3
    assert L.dspark_sts_apply(null, 10, 8, fake, fake, null) == -1


def test_schedule_async_arguments_rejected_on_the_host():
    L = binding.load()
    null = None
    fake = ctypes.c_void_p(4096)
    assert L.dspark_schedule_async(fake, fake, 10, 4, 5, null, fake, fake, fake, fake, 1 << 12, null) == -1
    assert L.dspark_schedule_async(fake, fake, 10, 1000, 16, fake, fake, fake, fake, fake, 1 << 12, null) == -3
    assert L.dspark_schedule_async(fake, fake, 10, 4, 5, fake, fake, fake, fake, null, 1 << 12, null) == -8


def test_misaligned_streamed_arrays_rejected_on_the_host():
    """U, P, the staging buffer, W2 and Wgco feed 16-byte loads and tensor-map
    copies: a pointer off a 16-byte boundary fails before anything runs."""
    L = binding.load()
    null = None
    ok = ctypes.c_void_p(1 << 20)            # 16- and 256-byte aligned; never dereferenced
    off = ctypes.c_void_p((1 << 20) + 4)

    def verify(P, U, W2, T, stage=None):
        return L.dspark_verify_staged(P, 0, U, 0, W2, 1, ok, ok, ok, ok, null, 4, 5, 4096, 32, 0, null, T,
                                      ok, ok, ok, null, null, stage, ok, 1 << 30, null)

    assert verify(off, ok, ok, 1.0) == -1                      # P
    assert verify(ok, ok, ok, 1.0, stage=off) == -1            # staging buffer
    assert verify(ok, off, ok, 1.0) == -1                      # U (sampled verification reads it)
    assert verify(ok, ok, off, 1.0) == -1                      # W2
    assert verify(off, null, null, 0.0) == -1                  # greedy: P only

    def markov(U, W2):
        return L.dspark_draft_markov(U, 0, ok, ok, W2, 1, 4, 5, 4096, 32, 0, null, 1.0,
                                     ok, ok, ok, ok, ok, 1 << 30, null)

    assert markov(off, ok) == -1
    assert markov(ok, off) == -1


def test_foreign_memory_refused_on_the_host():
    """U and W2 must be device memory of the current device (tensor maps,
    and W2 tiles shared by multicast within a cluster): an address that is
    not (here: no allocation at all, and on a machine without a GPU no
    current device) fails with INVALID_ARG before any kernel is enqueued."""
    L = binding.load()
    null = None
    ok = ctypes.c_void_p(1 << 20)            # 16- and 256-byte aligned; never dereferenced
    st = L.dspark_draft_markov(ok, 0, ok, ok, ok, 1, 4, 5, 4096, 32, 0, null, 1.0,
                               ok, ok, ok, ok, ok, 1 << 30, null)
    assert st == -1
    st = L.dspark_verify_staged(ok, 0, ok, 0, ok, 1, ok, ok, ok, ok, null, 4, 5, 4096, 32, 0, null, 1.0,
                                ok, ok, ok, null, null, null, ok, 1 << 30, null)
    assert st == -1


def test_binding_checks_shapes_before_any_launch():
    """The C ABI cannot see sizes, so the binding rejects a tensor of the
    wrong shape or dtype before passing any pointer (CPU tensors suffice:
    the check comes first)."""
    import torch
    R, gamma, V, r = 3, 4, 64, 8
    P = torch.zeros((R, gamma + 1, V))
    U = torch.zeros((R, gamma, V))
    W2 = torch.zeros((r, V), dtype=torch.bfloat16)
    draft = dict(tokens=torch.zeros((R, gamma), dtype=torch.int32),
                 q_tok=torch.zeros((R, gamma)), lse=torch.zeros((R, gamma), dtype=torch.float64),
                 code=torch.zeros((R, gamma, r)))
    with pytest.raises(ValueError, match="p_stage"):
        binding.verify(P, U, W2, draft, 1.0, 0, p_stage=torch.zeros((R, gamma, V)))
    with pytest.raises(TypeError, match="p_stage"):
        binding.verify(P, U, W2, draft, 1.0, 0, p_stage=torch.zeros((R, gamma + 1, V), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="U"):
        binding.verify(P, U[:, :2], W2, draft, 1.0, 0)
    with pytest.raises(ValueError, match="draft code"):
        binding.verify(P, U, W2, dict(draft, code=torch.zeros((R, gamma, r + 1))), 1.0, 0)
    with pytest.raises(ValueError, match="verify_len"):
        binding.verify(P, U, W2, draft, 1.0, 0, verify_len=torch.zeros((R + 1,), dtype=torch.int32))
    W1 = torch.zeros((V, r), dtype=torch.bfloat16)
    anchor = torch.zeros((R,), dtype=torch.int32)
    with pytest.raises(ValueError, match="W2"):
        binding.draft_markov(U, anchor, W1, W2[:, :V - 8], 1.0, 0)
    with pytest.raises(ValueError, match="anchor"):
        binding.draft_markov(U, anchor[:2], W1, W2, 1.0, 0)
    # correct shapes reach the pointer marshalling, which wants CUDA tensors
    with pytest.raises(ValueError, match="CUDA"):
        binding.verify(P, U, W2, draft, 1.0, 0, p_stage=torch.zeros((R, gamma + 1, V)))


def test_status_codes_agree_between_header_library_and_binding():
    """Every DSPARK_ERR_* value in the header has a dspark_strerror text and
    the binding's message table covers exactly the same codes."""
    with open(os.path.join(ROOT, "include", "dspark.h")) as f:
        text = f.read()
    codes = {name: int(v) for name, v in re.findall(r"\b(DSPARK_(?:OK|ERR_[A-Z_]+))\s*=\s*(-?\d+)", text)}
    assert codes.get("DSPARK_OK") == 0 and len(codes) >= 8
    L = binding.load()
    for name, v in codes.items():
        msg = L.dspark_strerror(v)
        assert msg and msg != b"unknown status", name
        assert binding.STATUS.get(v), name
    assert set(binding.STATUS) == set(codes.values())
