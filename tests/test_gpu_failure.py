"""Device-side failure detection without a GPU fault.

A tiny kernel waits, with the bounded wait that every GEMM role uses, on an
mbarrier that nothing arrives on. The wait must give up after about a second,
record GRPO_ERR_DEVICE_TIMEOUT in the workspace status word and return; the
context must stay usable, and the next call must start from a clean status.
"""

import time

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def clp():
    import __graft_entry__

    __graft_entry__.build()
    import chunked_log_prob_gb300 as m

    return m


def test_bounded_wait_runs_out_and_reports(clp):
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    t0 = time.perf_counter()
    st = clp.grpo_selftest_bounded_wait(ws)
    dt = time.perf_counter() - t0
    assert st == -7  # GRPO_ERR_DEVICE_TIMEOUT
    assert 0.3 < dt < 10.0  # gave up after about a second, did not hang
    assert int(ws[4:8].view(torch.int32).item()) == 1  # the wait reported failure


def test_context_usable_after_timeout(clp):
    ws0 = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    assert clp.grpo_selftest_bounded_wait(ws0) == -7
    p = synth.make_problem("tiny", seed=80)
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    old, ref = p.old_ref(torch.from_numpy(base))
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, device=DEV)
    ws[:64] = 0xFF  # a stale status from an earlier call must not leak into this one
    loss, logp, dH = clp.grpo_loss_fwd_bwd(
        p.hidden.to(DEV), p.weight.to(DEV), p.ids.to(DEV), p.mask.to(DEV), old.to(DEV),
        ref.to(DEV), p.adv.to(DEV), p.seq_len, workspace=ws)
    assert clp.grpo_read_device_status(ws) == 0
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len)
    assert np.abs(logp.cpu().double().numpy() - want["logp"]).max() <= 1e-2
    assert abs(loss.item() - want["L"]) <= 1e-3 * abs(want["L"])
