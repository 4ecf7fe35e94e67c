"""The workspace-free forward, grpo_logp_fwd_noalloc.

Some callers cannot allocate device memory: a plugin inside a host framework
that owns all device memory through its own pool, or a latency-critical caller
that cannot take cudaMalloc's implicit synchronisation. For them the library
keeps the forward's scratch in a static device array. These tests call that
entry point through the C ABI and check that it gives what the workspace
version (grpo_logp_fwd) gives - the same kernels with the same plan, so the
results must be bitwise equal, which is tighter than the 1e-2 logp tolerance
of the other parity tests - on several calls in a row with no synchronisation
between them. The calls go from the largest batch the array allows down to
smaller ones, so that a later call finds the earlier call's rows and partials
still in the array past its own. The largest call is also checked against the
fp64 oracle: at 8192 tokens the forward's scratch nearly fills the array.
"""

import numpy as np
import pytest
import torch

import oracle
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


def _cases(clp):
    n_max = clp.NOALLOC_MAX_TOKENS
    return [
        _problem(2, T=n_max // 4, prompts=1, G=4),      # 8192 x 256 x 4096: the limit
        _problem(1, T=75, prompts=1, G=4, D=200, V=1000),  # 300 rows, ragged in every dim
        _problem(0),                                    # 256 x 256 x 4096
        # a large vocabulary: the workspace's backward part (tail-split slots,
        # logit block) is far beyond the scratch, the forward's part is not
        _problem(3, T=128, prompts=1, G=4, D=256, V=128256),
    ]


def test_noalloc_matches_workspace_forward_on_calls_in_a_row(clp):
    cases = _cases(clp)
    assert cases[0][0].shape[0] == clp.NOALLOC_MAX_TOKENS
    want = []
    for h, W, ids in cases:
        lp, lse = clp.grpo_logp_fwd(h, W, ids, want_lse=True)
        want.append((lp.clone(), lse.clone()))
    torch.cuda.synchronize()

    got = []
    for h, W, ids in cases:  # calls in a row, no synchronisation between them
        lp = torch.full((h.shape[0],), float("nan"), device=DEV)
        lse = torch.full((h.shape[0],), float("nan"), device=DEV)
        clp.grpo_logp_fwd_noalloc(h, W, ids, lp, lse)
        got.append((lp, lse))
    torch.cuda.synchronize()

    for i, ((wl, wz), (gl, gz)) in enumerate(zip(want, got)):
        dl = (gl - wl).abs().max().item()
        print(f"call {i}: N={wl.shape[0]} max|dlogp| vs workspace forward = {dl:.3e}")
        assert torch.isfinite(gl).all() and torch.isfinite(gz).all()
        assert torch.equal(gl, wl) and torch.equal(gz, wz)


def test_noalloc_at_its_limit_matches_the_oracle(clp):
    h, W, ids = _cases(clp)[0]
    lp = torch.empty(h.shape[0], dtype=torch.float32, device=DEV)
    clp.grpo_logp_fwd_noalloc(h, W, ids, lp)
    want, _ = oracle.selective_logp(h.cpu(), W.cpu(), ids.cpu().numpy())
    d = np.abs(lp.cpu().double().numpy() - want)
    print(f"noalloc N={h.shape[0]}: max|dlogp|={d.max():.3e} rms={np.sqrt((d ** 2).mean()):.3e}")
    assert d.max() <= LOGP_TOL


def test_noalloc_rejects_more_than_its_static_scratch(clp):
    n = clp.NOALLOC_MAX_TOKENS + 1
    h = torch.zeros(n, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(16, 64, dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros(n, dtype=torch.int32, device=DEV)
    lp = torch.zeros(n, dtype=torch.float32, device=DEV)
    with pytest.raises(clp.GrpoError) as e:
        clp.grpo_logp_fwd_noalloc(h, W, ids, lp)
    assert e.value.code == -3
