"""GPU: the library's opt-in per-launch timing (grpo_launch_timing_enable /
grpo_launch_timing_read). It must record every launch of a call on the
calling thread only, give positive device times, and leave results unchanged.
"""

import threading

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
STORED = 1


@pytest.fixture(scope="module")
def clp():
    import __graft_entry__

    __graft_entry__.build()
    import chunked_log_prob_gb300 as m

    return m


def _problem(D, n=4096, V=3000):
    p = synth.make_problem("tiny", seed=D, prompts=n // 1024, G=4, T=256, D=D, V=V,
                           lengths=(128, 256))
    old = torch.full((p.n_tokens,), -7.5)
    return p, old


def _call(clp, p, old, params, ws):
    to = lambda t: t.to(DEV)  # noqa: E731
    loss, logp, dH = clp.grpo_loss_fwd_bwd(to(p.hidden), to(p.weight), to(p.ids), to(p.mask),
                                           to(old), to(old), to(p.adv), p.seq_len,
                                           params=params, workspace=ws)
    torch.cuda.synchronize()
    return loss.item(), logp.cpu(), dH.cpu()


@pytest.mark.parametrize("D, V, want_g", [(2304, 3000, "finalize_gform_kernel"),
                                          (1536, 3000, "finalize_rows_kernel"),
                                          (1536, 9000, "tail_fixup_kernel")])
def test_timing_records_every_launch_of_a_call(clp, D, V, want_g):
    # V = 9000: a vocabulary loop long enough for the tail split, so the fused
    # dH launch (at most 8 pair row units x 3 hidden tiles, fewer than the SM
    # pairs) is followed by its fixup pass.
    p, old = _problem(D, V=V)
    params = clp.make_params(flags=STORED)
    ws = clp.alloc_workspace(p.n_tokens, D, p.vocab, p.seq_len, params, DEV)
    plan = clp.grpo_get_plan(p.n_tokens, D, p.vocab, p.seq_len, params)
    ref = _call(clp, p, old, params, ws)  # untimed
    assert clp.grpo_launch_timing_read() == []  # off by default: nothing recorded

    calls = 3
    clp.grpo_launch_timing_enable(True)
    try:
        outs = [_call(clp, p, old, params, ws) for _ in range(calls)]
    finally:
        clp.grpo_launch_timing_enable(False)
    times = clp.grpo_launch_timing_read()
    print(times)
    names = {k["name"] for k in times}
    gemm_dh = "tc_gemm_kernel<2, 2>" if want_g == "finalize_gform_kernel" \
        else "tc_gemm_kernel<5, 2>"
    assert {"row_plan_kernel", "tc_gemm_kernel<3, 2>", want_g, gemm_dh,
            "finish_loss_kernel"} <= names
    assert sum(k["launches"] for k in times) == calls * plan["launches_loss"]
    for k in times:
        assert k["launches"] % calls == 0, k
        assert k["total_ms"] > 0.0, k
    # The GEMMs take most of the device time.
    top = max(times, key=lambda k: k["total_ms"])
    assert top["name"].startswith("tc_gemm_kernel")
    # The record was emptied by the read; results are those of the untimed call.
    assert clp.grpo_launch_timing_read() == []
    for L, logp, dH in outs:
        assert L == ref[0]
        assert torch.equal(logp, ref[1]) and torch.equal(dH, ref[2])


def test_timing_is_per_host_thread(clp):
    p, old = _problem(2304, n=1024)
    params = clp.make_params(flags=STORED)
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, DEV)
    got = {}

    def worker():
        torch.cuda.set_device(0)
        clp.grpo_launch_timing_enable(True)
        _call(clp, p, old, params, ws)
        clp.grpo_launch_timing_enable(False)
        got["worker"] = clp.grpo_launch_timing_read()

    clp.grpo_launch_timing_enable(True)
    try:
        t = threading.Thread(target=worker)
        t.start()
        t.join()
    finally:
        clp.grpo_launch_timing_enable(False)
    # The worker's launches are the worker's; this thread launched nothing.
    assert clp.grpo_launch_timing_read() == []
    plan = clp.grpo_get_plan(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params)
    assert sum(k["launches"] for k in got["worker"]) == plan["launches_loss"]


def test_timing_of_the_forward_call(clp):
    p, _ = _problem(2304, n=2048)
    params = clp.make_params()
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, DEV)
    logp0, _ = clp.grpo_logp_fwd(p.hidden.to(DEV), p.weight.to(DEV), p.ids.to(DEV),
                                 params=params, workspace=ws)
    clp.grpo_launch_timing_enable(True)
    try:
        logp1, _ = clp.grpo_logp_fwd(p.hidden.to(DEV), p.weight.to(DEV), p.ids.to(DEV),
                                     params=params, workspace=ws)
    finally:
        clp.grpo_launch_timing_enable(False)
    times = {k["name"]: k for k in clp.grpo_launch_timing_read()}
    gemm = [n for n in times if n.startswith("tc_gemm_kernel<0, ")]
    assert len(gemm) == 1 and times[gemm[0]]["launches"] == 1
    assert times["finalize_kernel"]["launches"] == 1
    assert np.array_equal(logp0.cpu().numpy(), logp1.cpu().numpy())
