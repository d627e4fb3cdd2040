"""A bounded device wait that runs out, on the GPU, without faulting it.

Every wait of the tensor-core kernels on another thread's progress gives up
after a limit of SM cycles, records DSPARK_ERR_TIMEOUT in the workspace's
status word and winds the kernel down (copies in flight land, the tensor
memory is freed, no CTA of a cluster leaves while a peer may still write into
it).  Here the limit is lowered to about a millisecond and the test hook of
dspark_workspace_set_wait makes the draft sweep's U producer withhold the
first stage of the first step: no copy is issued for it, so the epilogue's
wait on it runs out with nothing in flight on that stage, in every CTA of the
sweep (two M-groups, clusters of two sharing W2 by multicast).  The call must
report DSPARK_ERR_TIMEOUT, and the very next normal call on the same
workspace and GPU must pass parity with the oracle.
"""
import numpy as np
import pytest
import torch

from _parity import Flags, compare_draft, compare_verify, dev, gpu_verify_on, host, oracle_draft, oracle_verify_on
from speculative_decoding_drafting_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def test_withheld_stage_times_out_then_the_next_call_passes_parity():
    w = synth.Workload("timeout", R=256, gamma=2, V=4104, r=64, T=1.0)
    x = synth.gen_all(w)
    U, A, W1, W2 = dev(x["U"]), dev(x["anchor"]), dev(x["W1"]), dev(x["W2"])
    d = binding.draft_markov(U, A, W1, W2, w.T, 3)
    torch.cuda.synchronize()
    assert binding.workspace_status(d["ws"]) == 0
    # about 1 ms at 2 GHz: far above any wait of a normal step, far below the default
    binding.workspace_set_wait(d["ws"], 1 << 21, test_withhold=1)
    d = binding.draft_markov(U, A, W1, W2, w.T, 3, ws=d["ws"], out=d)
    torch.cuda.synchronize()
    assert binding.workspace_status(d["ws"]) == -5          # DSPARK_ERR_TIMEOUT
    # the hook off and the default limit back: a normal call on the same GPU
    binding.workspace_set_wait(d["ws"], 0, test_withhold=0)
    d = binding.draft_markov(U, A, W1, W2, w.T, 3, ws=d["ws"], out=d)
    torch.cuda.synchronize()
    assert binding.workspace_status(d["ws"]) == 0
    g = {k: host(v) for k, v in d.items() if k != "ws"}
    o = oracle_draft(w, x, 3)
    flags = Flags()
    compare_draft(g, o, tag="after timeout", flags=flags)
    np.testing.assert_array_equal(g["code"], o["code"].astype(np.float32))
    flags.check("after timeout")
    gv = gpu_verify_on(w, x, o, 3)
    ov = oracle_verify_on(w, x, o, 3)
    n, nf = compare_verify(gv, ov, np.ones(w.R, bool), tag="after timeout")
    assert n + nf == w.R


def test_set_wait_checks_its_arguments():
    L = binding.load()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert L.dspark_workspace_set_wait(None, 0, 0, None) == -1
    assert L.dspark_workspace_set_wait(binding._p(ws), 0, 2, None) == -1
    assert L.dspark_workspace_set_wait(binding._p(ws), 1 << 20, 0, None) == 0
    assert int(ws[4:16].view(torch.int32)[1].item()) == 1 << 20
