"""dspark_verify_noalloc against dspark_verify.

The no-allocation entry point serves callers that are given only their input
and output buffers (a plugin, an engine that owns all device memory, a path
that must not allocate), so it takes no workspace and uses a scratch array
built into the library instead.  It must give the same results as the
regular entry point, call after call, although every call reuses the same
array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_drafting_gb300 import binding, synth

pytestmark = pytest.mark.gpu

F32, BF16 = synth.F32, synth.BF16


def _dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to("cuda:0")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dt(t):
    return F32 if t.dtype == torch.float32 else BF16


def _noalloc(L, P, U, W2, d, T, seed, verify_len, R, gamma, V, r):
    out = dict(out_tokens=torch.full((R, gamma + 1), -7, dtype=torch.int32, device="cuda:0"),
               accept_len=torch.full((R,), -7, dtype=torch.int32, device="cuda:0"),
               n_out=torch.full((R,), -7, dtype=torch.int32, device="cuda:0"),
               p_tok=torch.zeros((R, gamma), dtype=torch.float32, device="cuda:0"),
               lse_p=torch.zeros((R, gamma + 1), dtype=torch.float64, device="cuda:0"))
    P_, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    fn = L.dspark_verify_noalloc
    fn.argtypes = [P_, i32, P_, i32, P_, i32, P_, P_, P_, P_, P_, i32, i32, i32, i32, u64, P_, f32,
                   P_, P_, P_, P_, P_, P_]
    fn.restype = i32
    st = fn(_p(P), _dt(P), _p(U), _dt(U), _p(W2), _dt(W2), _p(d["tokens"]), _p(d["q_tok"]), _p(d["lse"]),
            _p(d["code"]), _p(verify_len), R, gamma, V, r, seed, None, float(T),
            _p(out["out_tokens"]), _p(out["accept_len"]), _p(out["n_out"]), _p(out["p_tok"]), _p(out["lse_p"]),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, f"dspark_verify_noalloc returned {st}"
    return out


@pytest.mark.parametrize("w", [
    synth.Workload("noalloc_tc", R=9, gamma=4, V=20488, r=64, T=1.0),
    synth.Workload("noalloc_generic", R=5, gamma=3, V=4096, r=32, T=1.0, w_dtype=F32, sigma_w=0.05),
])
def test_noalloc_matches_regular_entry_point_twice(w):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = binding.load()
    x = synth.gen_all(w)
    U, P, W1, W2 = _dev(x["U"]), _dev(x["P"]), _dev(x["W1"]), _dev(x["W2"])
    d = binding.draft_markov(U, _dev(x["anchor"]), W1, W2, w.T, 11)
    vl = torch.tensor(np.random.default_rng(1).integers(0, w.gamma + 1, w.R), dtype=torch.int32, device="cuda:0")
    for call, (seed, lens) in enumerate([(21, None), (22, vl)]):
        ref = binding.verify(P, U, W2, d, w.T, seed, verify_len=lens)
        got = _noalloc(L, P, U, W2, d, w.T, seed, lens, w.R, w.gamma, w.V, w.r)
        torch.cuda.synchronize()
        for k in ("out_tokens", "accept_len", "n_out"):
            assert torch.equal(ref[k], got[k]), f"call {call}: {k} differs"
        for k in ("p_tok", "lse_p"):
            a, b = ref[k].cpu().numpy(), got[k].cpu().numpy()
            assert np.array_equal(np.isnan(a), np.isnan(b))
            np.testing.assert_allclose(b[~np.isnan(b)], a[~np.isnan(a)], rtol=1e-4)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = binding.load()
    fn = L.dspark_verify_noalloc
    fn.restype = ctypes.c_int
    # 512 requests x 17 rows x 149 chunks of partials alone exceed 8 MiB
    st = fn(None, 0, None, 0, None, 1, None, None, None, None, None, 512, 16, 151936, 256, ctypes.c_uint64(0),
            None, ctypes.c_float(1.0), None, None, None, None, None, None)
    assert st == -3
