"""GPU checks of the C ABI's contract that token parity alone would not pin.

- The device's Philox4x32-10 block function, through ``dspark_philox4x32_10``,
  against the published known-answer vectors (Salmon et al., SC'11, Random123)
  and against the oracle's copy on random counters and keys.
- U and W2 must be device memory of the current device: the tensor-core
  kernels build tensor maps over them and share W2 tiles among the CTAs of a
  cluster, which is defined for this GPU's own memory only.  A mapped pinned
  host buffer is refused with DSPARK_ERR_INVALID_ARG before anything runs,
  and the next normal call is unaffected.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_drafting_gb300 import binding, synth

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def _as_i32(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.uint32)).view(np.int32)).cuda()


def test_device_philox_known_answers():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append([int(t, 16) for t in line.split()])
    assert len(rows) == 3
    h = np.array(rows, dtype=np.uint64)
    out = binding.philox4x32_10(_as_i32(h[:, 0:4]), _as_i32(h[:, 4:6]))
    got = out.cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got, h[:, 6:10].astype(np.uint32))


def test_device_philox_matches_the_oracle_on_random_blocks():
    rng = np.random.default_rng(3)
    n = 1000 + 37                               # several CTAs and a ragged last one
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64)
    key = rng.integers(0, 2 ** 32, size=(n, 2), dtype=np.uint64)
    got = binding.philox4x32_10(_as_i32(ctr), _as_i32(key)).cpu().numpy().view(np.uint32)
    for i in range(0, n, 7):
        want = oracle.philox4x32_10([int(v) for v in ctr[i]], [int(v) for v in key[i]])
        assert [int(x) for x in got[i]] == [int(x) for x in want], i


def test_philox_entry_point_checks_arguments():
    L = binding.load()
    buf = torch.zeros((4, 4), dtype=torch.int32, device="cuda")
    p = binding._p(buf)
    assert L.dspark_philox4x32_10(p, p, p, 0, None) == -3
    assert L.dspark_philox4x32_10(None, p, p, 4, None) == -1


def _small():
    w = synth.Workload("resid", R=4, gamma=2, V=1024, r=64, T=1.0)
    return w, synth.gen_all(w)


def _dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def test_host_mapped_W2_and_U_are_refused_before_any_launch():
    w, x = _small()
    U, A, W1, W2 = _dev(x["U"]), _dev(x["anchor"]), _dev(x["W1"]), _dev(x["W2"])
    hW2 = torch.from_numpy(x["W2"].view(np.int16)).pin_memory().view(torch.bfloat16)
    hU = torch.from_numpy(x["U"]).pin_memory()
    vW2 = binding.host_view(hW2, U.device)
    vU = binding.host_view(hU, U.device)
    for args in ((U, A, W1, vW2), (vU, A, W1, W2)):
        with pytest.raises(binding.DsparkError) as ei:
            binding.draft_markov(*args, w.T, 1)
        assert ei.value.code == -1
    # a good draft, then verification with a host-mapped W2 or U is refused too
    d = binding.draft_markov(U, A, W1, W2, w.T, 1)
    P = _dev(x["P"])
    for u_, w2_ in ((U, vW2), (vU, W2)):
        with pytest.raises(binding.DsparkError) as ei:
            binding.verify(P, u_, w2_, d, w.T, 1)
        assert ei.value.code == -1
    # P itself may be read in place from mapped host memory
    hP = torch.from_numpy(x["P"]).pin_memory()
    v1 = binding.verify(binding.host_view(hP, U.device), U, W2, d, w.T, 1)
    v2 = binding.verify(P, U, W2, d, w.T, 1)
    torch.cuda.synchronize()
    assert torch.equal(v1["out_tokens"], v2["out_tokens"])
    assert binding.workspace_status(v2["ws"]) == 0
