"""The workspace-free forward, grpo_logp_fwd_noalloc.

Some callers cannot allocate device memory: a plugin inside a host framework
that owns all device memory through its own pool, or a latency-critical caller
that cannot take cudaMalloc's implicit synchronisation. For them the library
keeps the forward's scratch in a static device array. These tests call that
entry point through the C ABI and check that it gives what the workspace
version (grpo_logp_fwd) gives, within the parity tolerance used everywhere
else, on two calls in a row with different shapes (the second call must not
see the first call's leftovers).
"""

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

LOGP_TOL = 1e-2
DEV = "cuda:0"


@pytest.fixture(scope="module")
def clp():
    import __graft_entry__

    __graft_entry__.build()
    import chunked_log_prob_gb300 as m

    return m


def _problem(seed, **kw):
    p = synth.make_problem("tiny", seed=seed, **kw)
    return p.hidden.to(DEV), p.weight.to(DEV), p.ids.to(DEV)


def test_noalloc_matches_workspace_forward_on_two_calls(clp):
    a = _problem(0)                                   # 256 x 256 x 4096
    b = _problem(1, T=75, prompts=1, G=4, D=200, V=1000)  # ragged in every dim
    want = []
    for h, W, ids in (a, b):
        lp, lse = clp.grpo_logp_fwd(h, W, ids, want_lse=True)
        want.append((lp.clone(), lse.clone()))
    torch.cuda.synchronize()

    got = []
    for h, W, ids in (a, b):  # two calls in a row, no synchronisation between them
        lp = torch.full((h.shape[0],), float("nan"), device=DEV)
        lse = torch.full((h.shape[0],), float("nan"), device=DEV)
        clp.grpo_logp_fwd_noalloc(h, W, ids, lp, lse)
        got.append((lp, lse))
    torch.cuda.synchronize()

    for (wl, wz), (gl, gz) in zip(want, got):
        dl = (gl - wl).abs().max().item()
        dz = (gz - wz).abs().max().item()
        assert np.isfinite(dl) and dl <= LOGP_TOL
        assert np.isfinite(dz) and dz <= LOGP_TOL


def test_noalloc_rejects_more_than_its_static_scratch(clp):
    n = clp.NOALLOC_MAX_TOKENS + 1
    h = torch.zeros(n, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(16, 64, dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros(n, dtype=torch.int32, device=DEV)
    lp = torch.zeros(n, dtype=torch.float32, device=DEV)
    with pytest.raises(clp.GrpoError) as e:
        clp.grpo_logp_fwd_noalloc(h, W, ids, lp)
    assert e.value.code == -3
